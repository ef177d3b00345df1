"""Benchmark of the Muon step on GB300 (one JSON line on rank 0).

Workload (default ``gpt2``): the GPT-2-124M hidden-matrix bank -- 12 layers of
q, k, v, o (768x768), c_fc (3072x768), c_proj (768x3072): 72 matrices, 84.93 M
fp32 parameters, bf16 gradients, fp32 momentum buffers -- with fresh seeded
gradients every step (three gradient sets, used in turn).  One step = one full
Muon step over the bank: momentum, normalisation, 5 quintic Newton-Schulz
steps, parameter update (18 kernel launches through the C ABI).

  value      matrices per second, device-timed with CUDA events on the
             launching stream, inputs resident in HBM (the bank's 0.85 GB of
             inputs exceed the 129 MB L2, so no flush between steps)
  e2e        the same metric through the public API with host buffers: each
             step copies that step's gradients host->device from pinned memory
             and reads the updated parameters back device->host
  roofline   the dominant kernel (largest share of device time), its
             algorithmic FLOPs (or bytes) per launch over its live average
             launch time, against MEASURED_PEAKS.json
  cpu_baseline  the CPU oracle (bf16-emulating mode) timed on the host cores
             on a bounded sample of the bank's matrices

``--impl reference`` times the CPU oracle as the reference arm (rank 0 only).
Multi-GPU (torchrun, N ranks): the data-parallel step of sharded.ShardedBank.
The bank is repeated N times (weak scaling: one bank's Newton-Schulz work per
GPU) and every rank holds all of it; matrices are owned by the library's
work-balanced partition (muon_partition).  Per size group: a reduce-scatter
of the bf16 gradients, the owners' muon_step, an asynchronous all-gather of
the parameters.  value = matrices of the whole bank / max time over ranks.
``--sharded`` runs the same path on one rank.  The Adam and FP8 workloads run
one independent copy per rank.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LR, MU, NS_STEPS = 0.02, 0.95, 5
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ workloads
def workload_shapes(name):
    from newton_schulz_08_gb300 import inputs
    if name == "fp8":
        return [FP8_SHAPE]
    if name == "adam":
        return inputs.adam_bank_shapes()
    return {
        "gpt2": inputs.gpt2_shapes(),
        "gpt1p5b": inputs.gpt1p5b_shapes(),
        "rect": inputs.rect_shapes(),
        "single": [inputs.SINGLE["shape"]],
        "spectra": inputs.spectra_shapes(),
    }[name]


NS5_ONLY = {"spectra"}
ADAM_WORKLOADS = {"adam"}
ADAM_HP = {"lr": 3e-3, "beta1": 0.9, "beta2": 0.95, "eps": 1e-10, "weight_decay": 0.05, "cautious": True}


WORKLOAD_DESC = {
    "gpt2": "GPT-2-124M hidden-matrix bank: 12 x {4 x 768x768, 3072x768, 768x3072}, 72 matrices, "
            "84.93M fp32 params, bf16 grads (fresh each step), fp32 momentum",
    "gpt1p5b": "1.5B-shaped bank: 48 x {4 x 1600x1600, 6400x1600, 1600x6400}, 288 matrices, "
               "1.4746B fp32 params, bf16 grads, fp32 momentum",
    "rect": "rectangular bank: 8 each of 1024x4096, 4096x1024, 768x3072, 2048x8192, bf16 grads",
    "single": "single 128x512 matrix, fp32 grad",
    "spectra": "spectra sweep, Newton-Schulz only (ns5_bank): 64 x 1024x1024 and 16 x 4096x4096 bf16 "
               "G = U diag(s) V^T, s log-uniform in [1e-4, 1]",
    "adam": "Adam step with cautious weight decay on an embedding-type bank: 4 tables of 50304x768, "
            "154.53M fp32 params, bf16 grads, fp32 moments, step 10 of training",
    "fp8": "FP8 scaled product (forward of the page's FP8 matmul): x 65536x768 bf16 (64 x 1024 tokens of "
           "GPT-2-124M), w 3072x768 bf16 (its MLP input projection), E4M3 operands, bf16 out",
}
FP8_SHAPE = (65536, 3072, 768)  # M (tokens), N (outputs), K (inputs)


def ns_flops(shapes, steps=NS_STEPS):
    """Algorithmic FLOPs per kernel kind for one step over the bank."""
    f = {"gram": 0.0, "poly": 0.0, "update": 0.0}
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        f["gram"] += float(m) * (m + 1) * n
        f["poly"] += float(m) * m * (m + 1)
        f["update"] += 2.0 * m * m * n
    return {k: v * steps for k, v in f.items()}


def ns_flops_issued(shapes, steps=NS_STEPS):
    """FLOPs the tensor cores execute for one step over the bank: whole
    256 x 256 tiles (Gram / poly: the tiles on and above the diagonal),
    K padded to 64."""
    f = {"gram": 0.0, "poly": 0.0, "update": 0.0}
    t, kb = 256, 64
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        tm, tn = -(-m // t), -(-n // t)
        upper = tm * (tm + 1) // 2
        f["gram"] += 2.0 * upper * t * t * (-(-n // kb) * kb)
        f["poly"] += 2.0 * upper * t * t * (-(-m // kb) * kb)
        f["update"] += 2.0 * tm * tn * t * t * (-(-m // kb) * kb)
    return {k: v * steps for k, v in f.items()}


def ns_flops_dense(shapes, steps=NS_STEPS):
    """Dense-equivalent FLOPs (X X^T, A A and B X as plain GEMMs): 4 m^2 n + 2 m^3."""
    return steps * sum(4.0 * min(r, c) ** 2 * max(r, c) + 2.0 * min(r, c) ** 3 for r, c in shapes)


def hbm_bytes(shapes, gbytes, ns5_only=False):
    """Algorithmic bytes of the elementwise passes for one step over the bank."""
    e = float(sum(r * c for r, c in shapes))
    if ns5_only:
        return {"momentum_cast": e * (gbytes + 2),       # G r, Xraw w
                "normalise": e * 4,                      # Xraw r, X0 w
                "apply": e * (2 + 2)}                    # X r, O w
    b_bytes = float(sum(2 * min(r, c) ** 2 for r, c in shapes))
    return {"momentum_cast": e * (gbytes + 4 + 4 + 2),  # g, buf r/w, Xraw
            "normalise": e * 4,                          # Xraw r, X0 w
            "apply": e * (2 + 4 + 4),                    # X r, p r/w
            # the Muon step's last update: X and B read, p read and written
            "update_apply": e * (2 + 4 + 4) + b_bytes}


def kernel_report(ktimes, steps, flops, issued_flops, gbytes, peaks):
    """Per kernel kind: mean launch time, launches per step, achieved rate on
    the algorithmic work of the launches timed under that kind, fraction of
    the measured peak and share of the summed kernel time.  ktimes:
    {kind: (total_ms, launches)} over `steps` steps; flops / issued_flops:
    FLOPs per step of the GEMM kinds (all NS_STEPS iterations); gbytes:
    algorithmic bytes per step of the HBM-bound kinds.  When the Muon step's
    last update is timed as its own kind (update_apply, which also applies
    p -= lr O), the update kind holds NS_STEPS - 1 of the iterations."""
    kflops, kissued = dict(flops), dict(issued_flops)
    if ktimes.get("update_apply", (0, 0))[1]:
        for f in (kflops, kissued):
            f["update"] *= (NS_STEPS - 1) / NS_STEPS
    kern = {}
    for kind, (tot_ms, cnt) in ktimes.items():
        if cnt == 0:
            continue
        avg = tot_ms / cnt
        per_step = cnt / steps
        if kind in kflops:
            work = kflops[kind] / per_step  # per launch
            ach = work / (avg * 1e-3) / 1e12
            issued = kissued[kind] / per_step / (avg * 1e-3) / 1e12
            kern[kind] = {"avg_ms": avg, "launches_per_step": per_step, "share": None,
                          "achieved": ach, "unit": "TFLOP/s", "bound": "tensor",
                          "peak": peaks["bf16_tflops"], "frac": ach / peaks["bf16_tflops"],
                          "work_per_launch": work, "issued_tflops": issued,
                          "issued_frac": issued / peaks["bf16_tflops"]}
        else:
            work = gbytes[kind] / per_step
            ach = work / (avg * 1e-3) / 1e9
            kern[kind] = {"avg_ms": avg, "launches_per_step": per_step, "share": None,
                          "achieved": ach, "unit": "GB/s", "bound": "hbm",
                          "peak": peaks["hbm_gbs"], "frac": ach / peaks["hbm_gbs"],
                          "work_per_launch": work}
    tot = sum(v["avg_ms"] * v["launches_per_step"] for v in kern.values())
    for v in kern.values():
        v["share"] = v["avg_ms"] * v["launches_per_step"] / tot
    return kern


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle
def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_sample(shapes, budget_s, min_mats=1, mode="bf16"):
    """Time the oracle's Muon step on matrices of the bank taken in order
    (wrapping around) until `budget_s` seconds have passed."""
    import oracle
    from newton_schulz_08_gb300 import inputs
    done, t_total, i = 0, 0.0, 0
    while done < min_mats or t_total < budget_s:
        shape = shapes[i % len(shapes)]
        p = inputs.param(shape, i)
        g = oracle.round_to_bf16(inputs.grad(shape, i)).astype(np.float32)
        b = inputs.buffer(shape, i)
        t0 = time.perf_counter()
        oracle.muon_step(p, g, b, LR, MU, True, NS_STEPS, mode)
        t_total += time.perf_counter() - t0
        done += 1
        i += 1
    return done, t_total


def adam_oracle_sample(shapes, budget_s, min_tensors=1):
    """Time the oracle's float32 Adam step on whole tensors of the bank taken
    in order (wrapping around) until `budget_s` seconds have passed; returns
    (parameters done, seconds)."""
    import oracle
    from newton_schulz_08_gb300 import inputs
    done, n_params, t_total, i = 0, 0, 0.0, 0
    hp = dict(ADAM_HP)
    while done < min_tensors or t_total < budget_s:
        shape = shapes[i % len(shapes)]
        p, m, v, g = inputs.adam_state(shape, i)
        g = oracle.round_to_bf16(g)
        t0 = time.perf_counter()
        oracle.adam_step(p, g, m, v, inputs.ADAM_STEP, lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"],
                         eps=hp["eps"], wd=hp["weight_decay"], cautious=hp["cautious"], mode="fp32")
        t_total += time.perf_counter() - t0
        done += 1
        n_params += int(np.prod(shape))
        i += 1
    return n_params, t_total


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    shapes = workload_shapes(args.workload)
    if args.workload == "fp8":
        # each step: the oracle's product on a row sample sized to ~1 s
        budget = max(0.2, 60.0 / max(1, args.steps + args.warmup))
        for _ in range(args.warmup):
            fp8_oracle_sample(budget)
        total_f, total_t = 0.0, 0.0
        for _ in range(args.steps):
            f, t = fp8_oracle_sample(budget)
            total_f += f
            total_t += t
        value = total_f / total_t / 1e12
        line = {
            "impl": "reference", "metric": "fp8_mm_tflops", "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * total_t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (E4M3-emulating)", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC[args.workload]},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": "leading rows of x against all of w per step (FP8 oracle)"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return
    if args.workload in ADAM_WORKLOADS:
        for _ in range(args.warmup):
            adam_oracle_sample(shapes, 0.0)
        total, total_t = 0, 0.0
        for _ in range(args.steps):
            n, t = adam_oracle_sample(shapes, 0.0)
            total += n
            total_t += t
        value = total / total_t
        line = {
            "impl": "reference", "metric": "adam_step_params_per_s", "value": value, "unit": "params/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * total_t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC[args.workload]},
            "cpu_baseline": {"value": value, "unit": "params/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": "one 50304x768 table of the bank per step (float32 oracle)"},
            "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return
    # size each step so the whole run stays within about two minutes (the
    # cost per matrix from one pass over the bank's first six, which cover
    # every shape of a layer)
    n0, t0 = oracle_sample(shapes, 0.0, min_mats=min(6, len(shapes)))
    per_mat = t0 / n0
    per_step_budget = max(per_mat, 120.0 / max(1, args.steps + args.warmup))
    mats_per_step = max(1, int(per_step_budget / per_mat))
    for _ in range(args.warmup):
        oracle_sample(shapes, 0.0, min_mats=mats_per_step)
    total_mats, total_t = 0, 0.0
    for _ in range(args.steps):
        n, t = oracle_sample(shapes, 0.0, min_mats=mats_per_step)
        total_mats += n
        total_t += t
    value = total_mats / total_t
    sample = f"{mats_per_step} matrices of the bank per step (bf16-emulating oracle, taken in bank order)"
    line = {
        "impl": "reference", "metric": "muon_step_matrices_per_s", "value": value,
        "unit": "matrices/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (bf16-emulating)",
        "data": "synthetic", "config": {"workload": WORKLOAD_DESC[args.workload]},
        "cpu_baseline": {"value": value, "unit": "matrices/s", "cores": cpu_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "matrices/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ranks
def rank_bank(shapes, world, rank):
    """The matrices `rank` of `world` processes owns: the bank repeated `world`
    times (matrix g is shapes[g % len(shapes)]), split by muon.partition.
    Returns (global ids, shapes); the ids seed each matrix's inputs."""
    from newton_schulz_08_gb300 import muon
    full = [shapes[g % len(shapes)] for g in range(len(shapes) * world)]
    owner = muon.partition(full, world) if world > 1 else [0] * len(full)
    ids = [g for g, o in enumerate(owner) if o == rank]
    return ids, [full[g] for g in ids]


def max_over_ranks(x, world, device=None):
    """Largest value of `x` over all ranks (every rank gets it)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def e2e_pipelined(stream, device, n_steps, in_bufs, in_host, step_fn, out_dev, out_host):
    """End-to-end timing with host copies: every step uploads its inputs from
    pinned host memory and reads its result back to pinned host memory.  The
    copies run on two copy streams and overlap the compute: step k+1's inputs
    go into the second of two device input buffers while step k runs, and
    step k's result is snapshotted on the device (into the second of two
    snapshot buffers, so that the snapshot waits only for the read-back of
    step k-2) and read back while step k+1 runs.  in_bufs: two lists of
    device input tensors; in_host: lists of pinned host tensors (cycled);
    step_fn(j) runs one step on in_bufs[j]; out_dev / out_host: lists of
    device result tensors and pinned host buffers.  Returns milliseconds per
    step (CUDA events on `stream`)."""
    import torch
    h2d, d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    snap = [[torch.empty_like(t) for t in out_dev] for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer j landed
    ev_used = [torch.cuda.Event() for _ in range(2)]  # the step reading buffer j finished
    ev_snap = [torch.cuda.Event() for _ in range(2)]  # snapshot j taken
    ev_out = [torch.cuda.Event() for _ in range(2)]   # snapshot j read back
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in ev_used + ev_out:
        e.record(stream)

    def upload(k, j):
        h2d.wait_event(ev_used[j])
        with torch.cuda.stream(h2d):
            for dst, src in zip(in_bufs[j], in_host[k % len(in_host)]):
                dst.copy_(src, non_blocking=True)
        ev_in[j].record(h2d)

    e0.record(stream)
    upload(0, 0)
    for k in range(n_steps):
        j = k % 2
        if k + 1 < n_steps:
            upload(k + 1, 1 - j)
        stream.wait_event(ev_in[j])
        step_fn(j)
        ev_used[j].record(stream)
        stream.wait_event(ev_out[j])  # snapshot j (step k-2) has been read back
        with torch.cuda.stream(stream):
            for dst, src in zip(snap[j], out_dev):
                dst.copy_(src, non_blocking=True)
        ev_snap[j].record(stream)
        d2h.wait_event(ev_snap[j])
        with torch.cuda.stream(d2h):
            for dst, src in zip(out_host, snap[j]):
                dst.copy_(src, non_blocking=True)
        ev_out[j].record(d2h)
    for e in ev_out:
        stream.wait_event(e)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / n_steps


E2E_NOTE = ("every step uploads its inputs from pinned host memory and reads its result back to pinned host "
            "memory; the copies run on two copy streams overlapped with compute (next step's inputs into a "
            "second device buffer; this step's result snapshotted on the device into one of two buffers, then "
            "read back)")


# ------------------------------------------------------------------ GPU arm
def build_bank(shapes, device, grad_sets, ids=None):
    """Device tensors of the bank: params, bufs, grad sets (flat + views).
    Matrix k's inputs are seeded by ids[k] (default: k)."""
    import torch
    from newton_schulz_08_gb300 import inputs
    ids = list(range(len(shapes))) if ids is None else ids
    sizes = [r * c for r, c in shapes]
    total = sum(sizes)
    P = torch.empty(total, dtype=torch.float32, device=device)
    Bf = torch.empty(total, dtype=torch.float32, device=device)
    Gs_host = [torch.empty(total, dtype=torch.bfloat16).pin_memory() for _ in range(grad_sets)]
    off = 0
    for i, shape, sz in zip(ids, shapes, sizes):
        P[off:off + sz].copy_(torch.from_numpy(inputs.param(shape, i).ravel()))
        Bf[off:off + sz].copy_(torch.from_numpy(inputs.buffer(shape, i).ravel()))
        for k in range(grad_sets):
            Gs_host[k][off:off + sz].copy_(torch.from_numpy(inputs.grad(shape, i, step=k).ravel()))
        off += sz
    Gs = [g.to(device) for g in Gs_host]
    return P, Bf, Gs, Gs_host


def views(flat, shapes):
    out, off = [], 0
    for r, c in shapes:
        out.append(flat[off:off + r * c].view(r, c))
        off += r * c
    return out


def secondary_spectra(device, steps=5, warmup=3):
    """A short spectra sweep (ns5_bank over 64 x 1024^2 + 16 x 4096^2 bf16,
    5 Newton-Schulz steps) timed in the same process as the headline line:
    ms per sweep, per-kernel fractions of the measured peaks and the clocks
    seen meanwhile.  It puts the 4096-wide kernels' rate into the record."""
    import ctypes

    import torch

    from newton_schulz_08_gb300 import inputs, muon
    L = muon.lib()
    shapes = inputs.spectra_shapes()
    n = len(shapes)
    total = sum(r * c for r, c in shapes)
    G = torch.empty(total, dtype=torch.bfloat16, device=device)
    off = 0
    for i, (r, c) in enumerate(shapes):
        G[off:off + r * c].copy_(inputs.spectra_matrix_device(r, i, device, torch.bfloat16).reshape(-1))
        off += r * c
    O = torch.empty_like(G)
    gp = (ctypes.c_void_p * n)(*[g.data_ptr() for g in views(G, shapes)])
    op = (ctypes.c_void_p * n)(*[o.data_ptr() for o in views(O, shapes)])
    dt = (ctypes.c_int32 * n)(*([muon.MUON_BF16] * n))
    rows = (ctypes.c_int64 * n)(*[r for r, _ in shapes])
    cols = (ctypes.c_int64 * n)(*[c for _, c in shapes])
    ws = muon.new_workspace(L.ns5_bank_workspace_size(rows, cols, n), device)
    stream = torch.cuda.current_stream(device)
    sptr = ctypes.c_void_p(stream.cuda_stream)

    def sweep():
        st = L.ns5_bank(gp, dt, op, rows, cols, n, NS_STEPS, ctypes.c_void_p(ws.data_ptr()), ws.numel(), sptr)
        if st != 0:
            raise muon.MuonError(st, "ns5_bank")

    for _ in range(max(warmup, 3)):
        sweep()
    torch.cuda.synchronize(device)
    clocks = ClockSampler(device.index or 0)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        sweep()
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    muon.muon_set_debug("record_kernel_events", 1)
    muon.muon_kernel_times()
    for _ in range(steps):
        sweep()
    torch.cuda.synchronize(device)
    kt = muon.muon_kernel_times()
    muon.muon_set_debug("record_kernel_events", 0)
    clk = clocks.stop()
    if muon.muon_device_status(ws) != 0:
        raise RuntimeError("device status after the spectra sweep")
    peaks, src = load_peaks()
    kern = kernel_report(kt, steps, ns_flops(shapes), ns_flops_issued(shapes), hbm_bytes(shapes, 2, True), peaks)
    flops = sum(ns_flops(shapes).values())
    return {
        "workload": WORKLOAD_DESC["spectra"], "steps": steps, "ms_per_sweep": ms,
        "matrices_per_s": n / (ms * 1e-3), "ns5_tflops": flops / (ms * 1e-3) / 1e12,
        "kernels": {k: {"avg_ms": v["avg_ms"], "frac": v["frac"], "issued_frac": v.get("issued_frac"),
                        "unit": v["unit"], "achieved": v["achieved"]} for k, v in kern.items()},
        "peak_source": src, "clocks": clk,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gpt2", choices=sorted(WORKLOAD_DESC))
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of CPU oracle work")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true", help="skip the spectra sweep of the gpt2 line")
    ap.add_argument("--sharded", action="store_true",
                    help="time the sharded data-parallel step (the default when more than one rank runs)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import ctypes

    import torch
    import torch.distributed as dist

    from newton_schulz_08_gb300 import muon

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    if args.workload in ADAM_WORKLOADS:
        run_adam(args, rank, world, device)
        return
    if args.workload == "fp8":
        run_fp8(args, rank, world, device)
        return
    if (world > 1 or args.sharded) and args.workload not in NS5_ONLY:
        run_sharded(args, rank, world, device)
        return

    L = muon.lib()
    ids, shapes = rank_bank(workload_shapes(args.workload), world, rank)
    n_mats = len(shapes)
    n_total = len(workload_shapes(args.workload)) * world
    ns5_only = args.workload in NS5_ONLY
    stream = torch.cuda.current_stream(device)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    if not ns5_only:
        grad_sets = 3
        P, Bf, Gs, Gs_host = build_bank(shapes, device, grad_sets, ids)
        Pv, Bv = views(P, shapes), views(Bf, shapes)
        descs = []
        for k in range(grad_sets):
            arr, n = muon._descs(Pv, views(Gs[k], shapes), Bv)
            descs.append(arr)
        ws = muon.new_workspace(L.muon_workspace_size(descs[0], n_mats), device)
        ws_ptr, ws_bytes = ctypes.c_void_p(ws.data_ptr()), ws.numel()

        def step(k, arr=None):
            st = L.muon_step(descs[k % grad_sets] if arr is None else arr, n_mats, LR, MU, 1, NS_STEPS,
                             ws_ptr, ws_bytes, sptr)
            if st != 0:
                raise muon.MuonError(st, "muon_step")

        # e2e: each step's gradients in (device sets 1 and 2 as the two input
        # buffers), the updated parameters out
        e2e_in = [[Gs[1]], [Gs[2]]]
        e2e_host = [[g] for g in Gs_host]
        e2e_out = [P]

        def e2e_step(j):
            step(0, descs[1 + j])
        gbytes = 2
    else:
        from newton_schulz_08_gb300 import inputs
        total = sum(r * c for r, c in shapes)
        Gflat = torch.empty(total, dtype=torch.bfloat16, device=device)
        off = 0
        for i, (r, c) in zip(ids, shapes):
            Gflat[off:off + r * c].copy_(inputs.spectra_matrix_device(r, i, device, torch.bfloat16).reshape(-1))
            off += r * c
        Oflat = torch.empty_like(Gflat)
        Gv, Ov = views(Gflat, shapes), views(Oflat, shapes)
        gp = (ctypes.c_void_p * n_mats)(*[g.data_ptr() for g in Gv])
        op = (ctypes.c_void_p * n_mats)(*[o.data_ptr() for o in Ov])
        dt = (ctypes.c_int32 * n_mats)(*([muon.MUON_BF16] * n_mats))
        rows = (ctypes.c_int64 * n_mats)(*[r for r, _ in shapes])
        cols = (ctypes.c_int64 * n_mats)(*[c for _, c in shapes])
        ws = muon.new_workspace(L.ns5_bank_workspace_size(rows, cols, n_mats), device)
        ws_ptr, ws_bytes = ctypes.c_void_p(ws.data_ptr()), ws.numel()
        Gflat2 = torch.empty_like(Gflat)
        gp2 = (ctypes.c_void_p * n_mats)(*[g.data_ptr() for g in views(Gflat2, shapes)])

        def step(k, arr=None):
            st = L.ns5_bank(gp if arr is None else arr, dt, op, rows, cols, n_mats, NS_STEPS, ws_ptr, ws_bytes,
                            sptr)
            if st != 0:
                raise muon.MuonError(st, "ns5_bank")

        e2e_in = [[Gflat], [Gflat2]]
        e2e_host = [[Gflat.cpu().pin_memory()]]
        e2e_out = [Oflat]

        def e2e_step(j):
            step(0, (gp, gp2)[j])
        gbytes = 2

    def barrier():
        torch.cuda.synchronize(device)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(device)

    for k in range(args.warmup):
        step(k)
    barrier()
    st = muon.muon_device_status(ws)
    if st != 0:
        raise muon.MuonError(st, "device status after warm-up")

    # -------------------------------------------------------------- timed
    clocks = ClockSampler(local)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for k in range(args.steps):
        step(k)
    e1.record(stream)
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)

    # ---------------------------------------------- per-kernel live timing
    muon.muon_set_debug("record_kernel_events", 1)
    muon.muon_kernel_times()
    for k in range(args.steps):
        step(k)
    barrier()
    ktimes = muon.muon_kernel_times()
    muon.muon_set_debug("record_kernel_events", 0)

    # ------------------------------------------------------------- e2e
    out_host = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in e2e_out]
    e_steps = max(10, args.steps // 2)
    barrier()
    e2e_ms = e2e_pipelined(stream, device, e_steps, e2e_in, e2e_host, e2e_step, e2e_out, out_host)
    barrier()
    clk = clocks.stop()
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    st = muon.muon_device_status(ws)
    if st != 0:
        raise muon.MuonError(st, "device status after timing")

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # ------------------------------------------------------------- report
    peaks, peak_src = load_peaks()
    flops = ns_flops(shapes)
    gbytes = hbm_bytes(shapes, gbytes, ns5_only)
    kern = kernel_report(ktimes, args.steps, flops, ns_flops_issued(shapes), gbytes, peaks)
    dom = max(kern, key=lambda k: kern[k]["share"])
    d = kern[dom]
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            traffic = json.load(f).get(args.workload, {}).get(dom)

    value = n_total / (ms * 1e-3)
    total_flops = sum(flops.values())
    line = {
        "metric": "muon_step_matrices_per_s", "value": value, "unit": "matrices/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.workload], "matrices": n_total,
                   "params": int(sum(r * c for r, c in workload_shapes(args.workload))) * world, "ns_steps": NS_STEPS,
                   "lr": LR, "momentum": MU, "nesterov": True,
                   "l2": "no flush: inputs (params, bufs, grads) exceed the 129 MB L2",
                   "parallelism": (f"{world} ranks, each owning a work-balanced share of {world} banks "
                                   "(no data exchanged)" if world > 1 else "1 GPU")},
        "ns5_tflops": total_flops / (ms * 1e-3) / 1e12,
        "ns5_tflops_note": "algorithmic NS FLOPs of the whole step / step time",
        "ns5_tflops_issued": sum(ns_flops_issued(shapes).values()) / (ms * 1e-3) / 1e12,
        "ns5_tflops_dense_equivalent": ns_flops_dense(shapes) / (ms * 1e-3) / 1e12,
        "update_gbs": (gbytes["momentum_cast"] + gbytes["apply"]) / (ms * 1e-3) / 1e9,
        "roofline": {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"],
                     "unit": d["unit"], "frac": d["frac"], "traffic": traffic,
                     "peak_source": f"{peak_src} ({'bf16_tflops burst' if d['unit'] == 'TFLOP/s' else 'hbm_gbs'})"},
        "kernels": kern,
        "e2e": {"value": n_total / (e2e_ms * 1e-3), "unit": "matrices/s",
                "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in e2e_in[0])),
                "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in e2e_out)),
                "method": E2E_NOTE},
        "gpu_launches": int(sum(c for _, c in ktimes.values())),
        "gpu_launches_note": "kernels launched in the per-kernel timing pass (same count as the main timed loop)",
        "clocks": clk,
    }
    if world == 1 and args.workload == "gpt2" and not args.no_secondary:
        line["secondary"] = secondary_spectra(device)
    if world == 1 and not args.no_cpu_baseline and not ns5_only:
        n_cpu, t_cpu = oracle_sample(shapes, args.cpu_budget)
        n64, t64 = oracle_sample(shapes, args.cpu_budget / 2, mode="fp64")
        per_bank = len(shapes)
        line["cpu_baseline"] = {
            "value": n_cpu / t_cpu, "unit": "matrices/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": f"{n_cpu} matrices of the bank in order, full Muon step, bf16-emulating oracle, "
                      f"{t_cpu:.1f} s (capped; a full {per_bank}-matrix step extrapolates to "
                      f"{per_bank * t_cpu / n_cpu:.1f} s)",
            "fp64": {"value": n64 / t64, "unit": "matrices/s",
                     "sample": f"{n64} matrices in order, fp64 oracle, {t64:.1f} s (capped; a full step "
                               f"extrapolates to {per_bank * t64 / n64:.1f} s)"}}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_sharded(args, rank, world, device):
    """The data-parallel Muon step (sharded.ShardedBank) over `world` ranks:
    the bank repeated `world` times (weak scaling: one bank's Newton-Schulz
    work per GPU, while the exchange covers the whole world-sized bank),
    every rank holding all parameters and its own gradients for all of them;
    per size group one reduce-scatter of the bf16 gradients, the owners'
    muon_step, one asynchronous all-gather of the parameters."""
    import torch
    import torch.distributed as dist

    from newton_schulz_08_gb300 import inputs, muon, sharded

    if not dist.is_initialized():
        # one rank (--sharded): a process group of its own, so that the same
        # collectives run (as copies)
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        store = dist.TCPStore("127.0.0.1", port, 1, True)
        dist.init_process_group("nccl", store=store, rank=0, world_size=1, device_id=device)
    base = workload_shapes(args.workload)
    shapes = [base[g % len(base)] for g in range(len(base) * world)]
    bank = sharded.ShardedBank(shapes, device)
    for i, s in enumerate(shapes):
        bank.params[i].copy_(torch.from_numpy(inputs.param(s, i)))
        bank.grads[i].copy_(torch.from_numpy(inputs.grad(s, i, step=rank)))
    for i in bank.owned():
        bank.bufs[i].copy_(torch.from_numpy(inputs.buffer(shapes[i], i)))
    stream = torch.cuda.current_stream(device)

    def step():
        bank.step(lr=LR, momentum=MU, nesterov=True, ns_steps=NS_STEPS)

    def barrier():
        torch.cuda.synchronize(device)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(device)

    for _ in range(args.warmup):
        step()
    barrier()
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
    muon.muon_set_debug("record_kernel_events", 1)
    muon.muon_kernel_times()
    for _ in range(args.steps):
        step()
    barrier()
    ktimes = muon.muon_kernel_times()
    muon.muon_set_debug("record_kernel_events", 0)
    # e2e: this rank's gradients in from pinned host memory, the gathered
    # parameters out, every step (serialised with the step)
    g_host = [f.cpu().pin_memory() for f in bank.grad_flat]
    p_host = [torch.empty(f.shape, dtype=f.dtype).pin_memory() for f in bank.param_flat]
    e_steps = max(10, args.steps // 2)
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(e_steps):
        for dst, src in zip(bank.grad_flat, g_host):
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in zip(p_host, bank.param_flat):
            dst.copy_(src, non_blocking=True)
    f1.record(stream)
    barrier()
    clk = clocks.stop()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / e_steps, world, device)
    if bank.workspace is not None and muon.muon_device_status(bank.workspace) != 0:
        raise RuntimeError("device status after the sharded step")
    if rank != 0:
        dist.destroy_process_group()
        return
    dist.destroy_process_group()
    peaks, peak_src = load_peaks()
    mine = [shapes[i] for i in bank.owned()]
    kern = kernel_report(ktimes, args.steps, ns_flops(mine), ns_flops_issued(mine), hbm_bytes(mine, 2), peaks)
    dom = max(kern, key=lambda k: kern[k]["share"])
    d = kern[dom]
    n_total = len(shapes)
    line = {
        "metric": "muon_step_matrices_per_s", "value": n_total / (ms * 1e-3), "unit": "matrices/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.workload], "matrices": n_total,
                   "params": int(sum(r * c for r, c in shapes)), "ns_steps": NS_STEPS, "lr": LR, "momentum": MU,
                   "nesterov": True, "l2": "no flush: the bank's state exceeds the 129 MB L2",
                   "parallelism": f"data-parallel over {world} ranks: {world} copies of the bank, matrices owned by "
                                  "work-balanced partition; per size group a bf16 reduce-scatter of the gradients, "
                                  "the owners' Muon steps, an asynchronous all-gather of the parameters",
                   "exchange_bytes_per_rank_per_step": bank.exchange_bytes()},
        "roofline": {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"],
                     "unit": d["unit"], "frac": d["frac"], "traffic": None,
                     "peak_source": f"{peak_src} ({'bf16_tflops burst' if d['unit'] == 'TFLOP/s' else 'hbm_gbs'})"},
        "kernels": kern,
        "e2e": {"value": n_total / (e2e_ms * 1e-3), "unit": "matrices/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": int(sum(f.numel() * f.element_size() for f in bank.grad_flat)),
                "d2h_bytes_per_step": int(sum(f.numel() * f.element_size() for f in bank.param_flat)),
                "method": "every step uploads this rank's gradients from pinned host memory and reads the gathered "
                          "parameters back, serialised with the step"},
        "gpu_launches": int(sum(c for _, c in ktimes.values())),
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_adam(args, rank, world, device):
    """The Adam step with cautious weight decay on the embedding-type bank:
    one adam_step call (one kernel launch) per step."""
    import torch
    import torch.distributed as dist

    from newton_schulz_08_gb300 import inputs, muon

    ids, shapes = rank_bank(workload_shapes(args.workload), world, rank)
    n_total = sum(int(np.prod(s)) for s in workload_shapes(args.workload)) * world
    n_local = sum(int(np.prod(s)) for s in shapes)
    P, M, V, G = [], [], [], []
    for i, shp in zip(ids, shapes):
        p, m, v, g = inputs.adam_state(shp, i)
        P.append(torch.from_numpy(p).to(device))
        M.append(torch.from_numpy(m).to(device))
        V.append(torch.from_numpy(v).to(device))
        G.append(torch.from_numpy(g).to(device).to(torch.bfloat16))
    hp = dict(ADAM_HP)
    stream = torch.cuda.current_stream(device)

    def step(k):
        muon.adam_step(P, G, M, V, inputs.ADAM_STEP + k, lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"],
                       eps=hp["eps"], weight_decay=hp["weight_decay"], cautious=hp["cautious"], stream=stream)

    def barrier():
        torch.cuda.synchronize(device)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(device)

    launches_per_step = (len(shapes) + 63) // 64
    for k in range(args.warmup):
        step(k)
    barrier()
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for k in range(args.steps):
        step(args.warmup + k)
    e1.record(stream)
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)

    # e2e: each step's gradients in from pinned host memory (two device
    # gradient buffers), the updated parameters out
    g_host = [[g.cpu().pin_memory() for g in G]]
    p_host = [torch.empty(p.shape, dtype=p.dtype).pin_memory() for p in P]
    G2 = [torch.empty_like(g) for g in G]
    Gsets = [G, G2]
    e_steps = max(10, args.steps // 2)
    k0 = args.warmup + args.steps

    def e2e_step(j):
        muon.adam_step(P, Gsets[j], M, V, inputs.ADAM_STEP + k0, lr=hp["lr"], beta1=hp["beta1"],
                       beta2=hp["beta2"], eps=hp["eps"], weight_decay=hp["weight_decay"],
                       cautious=hp["cautious"], stream=stream)
    barrier()
    e2e_ms = e2e_pipelined(stream, device, e_steps, Gsets, g_host, e2e_step, P, p_host)
    barrier()
    clk = clocks.stop()
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    bytes_per_step = 26.0 * n_local  # p, m, v read + written (fp32), g read (bf16)
    achieved = bytes_per_step / (ms * 1e-3) / 1e9
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            traffic = json.load(f).get(args.workload, {}).get("adam")
    line = {
        "metric": "adam_step_params_per_s", "value": n_total / (ms * 1e-3), "unit": "params/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.workload], "tensors": len(shapes) * world,
                   "params": n_total, "hyper_parameters": hp,
                   "l2": "no flush: the bank's 2.2 GB of state exceeds the 129 MB L2",
                   "parallelism": (f"{world} ranks, each owning a share of {world} banks (no data exchanged)"
                                   if world > 1 else "1 GPU")},
        "roofline": {"kernel": "adam", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "peak_source": f"{peak_src} (hbm_gbs)"},
        "e2e": {"value": n_total / (e2e_ms * 1e-3), "unit": "params/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": int(sum(g.numel() * g.element_size() for g in G)),
                "d2h_bytes_per_step": int(sum(p.numel() * p.element_size() for p in P)),
                "method": E2E_NOTE},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        n_cpu, t_cpu = adam_oracle_sample(shapes, args.cpu_budget)
        line["cpu_baseline"] = {"value": n_cpu / t_cpu, "unit": "params/s", "cores": cpu_threads(),
                                "kind": "oracle",
                                "sample": f"{n_cpu} params (whole tables in bank order), float32 oracle, "
                                          f"{t_cpu:.1f} s"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def fp8_operands(seed=0):
    """Seeded bf16 operands of the FP8 workload and per-tensor scales that
    fill E4M3 (largest |x| / x_s = 448 / 1.05)."""
    M, N, K = FP8_SHAPE
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x_s = float(np.abs(x).max() / 448.0 * 1.05)
    w_s = float(np.abs(w).max() / 448.0 * 1.05)
    return x, w, x_s, w_s


def fp8_oracle_sample(budget_s):
    """The oracle's FP8 product on the first rows of x, doubling the rows
    until the budget is spent; returns (FLOPs, seconds)."""
    import oracle
    x, w, x_s, w_s = fp8_operands()
    xb, wb = oracle.round_to_bf16(x), oracle.round_to_bf16(w)
    N, K = w.shape
    rows, flops, t = 16, 0.0, 0.0
    while True:  # at least one chunk
        t0 = time.perf_counter()
        oracle.fp8_mm(xb[:rows], wb, x_s, w_s)
        t += time.perf_counter() - t0
        flops += 2.0 * rows * N * K
        rows *= 2
        if t >= budget_s or rows > x.shape[0]:
            return flops, t


def run_fp8(args, rank, world, device):
    """The FP8 scaled product (fp8_mm: quantise pass + tcgen05 kind::f8f6f4
    product) on one GPT-2-124M MLP projection's worth of tokens; each rank
    runs its own copy (weak scaling)."""
    import torch
    import torch.distributed as dist

    from newton_schulz_08_gb300 import muon

    M, N, K = FP8_SHAPE
    x, w, x_s, w_s = fp8_operands(rank)
    X = torch.from_numpy(x).to(device).to(torch.bfloat16)
    W = torch.from_numpy(w).to(device).to(torch.bfloat16)
    O = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    XQ = torch.empty((M, K), dtype=torch.uint8, device=device)
    WQ = torch.empty((N, K), dtype=torch.uint8, device=device)
    ws = muon.new_workspace(256, device)
    stream = torch.cuda.current_stream(device)

    def step(Xi=X, Wi=W):
        muon.fp8_mm(Xi, Wi, x_s, w_s, out=O, x_f8=XQ, w_f8=WQ, workspace=ws, stream=stream)

    def barrier():
        torch.cuda.synchronize(device)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(device)

    for _ in range(args.warmup):
        step()
    barrier()
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
    muon.muon_set_debug("record_kernel_events", 1)
    muon.muon_kernel_times()
    for _ in range(args.steps):
        step()
    barrier()
    kt = muon.muon_kernel_times()
    muon.muon_set_debug("record_kernel_events", 0)
    # backward (fp8_mm_backward): a seeded bf16 output gradient of M x N,
    # the forward's E4M3 operands, grad_s filling E5M2
    gen = torch.Generator(device=device).manual_seed(1234 + rank)
    Gd = (torch.randn((M, N), generator=gen, device=device) * 1e-3).to(torch.bfloat16)
    grad_s = float(Gd.abs().max().float().item() / 57344.0 * 1.05)
    GX = torch.empty((M, K), dtype=torch.bfloat16, device=device)
    GW = torch.empty((N, K), dtype=torch.bfloat16, device=device)
    GQ = torch.empty((M, N), dtype=torch.uint8, device=device)
    bws = muon.new_workspace(muon.fp8_mm_backward_workspace_size(M, N, K), device)

    def bstep():
        muon.fp8_mm_backward(Gd, XQ, WQ, x_s, w_s, grad_s, grad_x=GX, grad_w=GW, g_f8=GQ, workspace=bws,
                             stream=stream)

    for _ in range(args.warmup):
        bstep()
    barrier()
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(args.steps):
        bstep()
    b1.record(stream)
    barrier()
    bms = max_over_ranks(b0.elapsed_time(b1) / args.steps, world, device)
    muon.muon_set_debug("record_kernel_events", 1)
    muon.muon_kernel_times()
    for _ in range(args.steps):
        bstep()
    barrier()
    bkt = muon.muon_kernel_times()
    muon.muon_set_debug("record_kernel_events", 0)
    if muon.muon_device_status(bws) != 0:
        raise RuntimeError("device status after the FP8 backward")
    del Gd, GX, GW, GQ, bws

    # e2e: x and w in from pinned host memory, out back
    in_host = [[X.cpu().pin_memory(), W.cpu().pin_memory()]]
    bufs = [[X, W], [torch.empty_like(X), torch.empty_like(W)]]
    o_host = [torch.empty(O.shape, dtype=O.dtype).pin_memory()]
    barrier()
    e2e_ms = e2e_pipelined(stream, device, max(10, args.steps // 2), bufs, in_host,
                           lambda j: step(bufs[j][0], bufs[j][1]), [O], o_host)
    barrier()
    clk = clocks.stop()
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    st = muon.muon_device_status(ws)
    if st != 0:
        raise muon.MuonError(st, "device status after timing")
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    flops = 2.0 * M * N * K
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # nominal dense FP8 : BF16 rate = 4.5 : 2.25
    fp8_traffic = {}
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            fp8_traffic = json.load(f).get("fp8", {})
    g_ms, g_n = kt["fp8_mm"]
    q_ms, q_n = kt["fp8_quantize"]
    g_avg, q_avg = g_ms / g_n, q_ms / q_n
    ach = flops / (g_avg * 1e-3) / 1e12
    q_bytes = 3.0 * (M + N) * K  # bf16 in, E4M3 out
    line = {
        "metric": "fp8_mm_tflops", "value": flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC["fp8"], "M": M, "N": N, "K": K, "x_s": x_s, "w_s": w_s,
                   "l2": "no flush: x (101 MB bf16) and out (403 MB bf16) exceed the 129 MB L2",
                   "parallelism": f"{world} ranks, one product each" if world > 1 else "1 GPU"},
        "roofline": {"kernel": "fp8_mm", "bound": "tensor", "achieved": ach, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": ach / fp8_peak, "traffic": fp8_traffic.get("fp8_mm"),
                     "peak_source": f"{peak_src} bf16_tflops burst x 2 (nominal FP8 : BF16 dense rate)"},
        "kernels": {"fp8_quantize": {"avg_ms": q_avg, "achieved": q_bytes / (q_avg * 1e-3) / 1e9, "unit": "GB/s",
                                     "bound": "hbm", "peak": peaks["hbm_gbs"],
                                     "frac": q_bytes / (q_avg * 1e-3) / 1e9 / peaks["hbm_gbs"]},
                    "fp8_mm": {"avg_ms": g_avg, "achieved": ach, "unit": "TFLOP/s", "bound": "tensor",
                               "peak": fp8_peak, "frac": ach / fp8_peak}},
        "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": int(X.numel() * 2 + W.numel() * 2),
                "d2h_bytes_per_step": int(O.numel() * 2), "method": E2E_NOTE},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }
    bflops = 4.0 * M * N * K  # grad_x and grad_w
    t_ms, t_n = bkt["fp8_transpose"]
    g_ms2, g_n2 = bkt["fp8_mm_bwd"]
    r_ms, r_n = bkt["fp8_reduce"]
    t_bytes = 4.0 * M * N + 2.0 * M * K + 2.0 * N * K  # g r (2) + g_f8 w + g_f8^T w; x_f8, w_f8 r + copies w
    bk = {"fp8_transpose": {"avg_ms": t_ms / t_n, "achieved": t_bytes / (t_ms / t_n * 1e-3) / 1e9, "unit": "GB/s",
                            "bound": "hbm", "peak": peaks["hbm_gbs"],
                            "frac": t_bytes / (t_ms / t_n * 1e-3) / 1e9 / peaks["hbm_gbs"],
                            "work_per_launch": t_bytes, "traffic": fp8_traffic.get("fp8_transpose")},
          "fp8_mm_bwd": {"avg_ms": g_ms2 / g_n2, "achieved": bflops / (g_ms2 / g_n2 * 1e-3) / 1e12,
                         "unit": "TFLOP/s", "bound": "tensor", "peak": fp8_peak,
                         "frac": bflops / (g_ms2 / g_n2 * 1e-3) / 1e12 / fp8_peak, "work_per_launch": bflops}}
    if r_n:
        r_bytes = 4.0 * N * K * 2 + 2.0 * N * K  # two fp32 slices read, bf16 written
        bk["fp8_reduce"] = {"avg_ms": r_ms / r_n, "achieved": r_bytes / (r_ms / r_n * 1e-3) / 1e9, "unit": "GB/s",
                            "bound": "hbm", "peak": peaks["hbm_gbs"],
                            "frac": r_bytes / (r_ms / r_n * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    line["backward"] = {"what": "fp8_mm_backward: g 65536x3072 bf16 -> E5M2, grad_x = g_f8 . w_f8 and "
                                "grad_w = g_f8^T . x_f8 on the tensor cores (E5M2 x E4M3), bf16 out",
                        "ms_per_call": bms, "tflops": bflops * world / (bms * 1e-3) / 1e12, "grad_s": grad_s,
                        "kernels": bk, "gpu_launches_per_call": 2 + (1 if r_n else 0)}
    if world == 1 and not args.no_cpu_baseline:
        f_cpu, t_cpu = fp8_oracle_sample(args.cpu_budget)
        line["cpu_baseline"] = {"value": f_cpu / t_cpu / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(),
                                "kind": "oracle",
                                "sample": f"{f_cpu / 2 / N / K:.0f} rows of x against all of w, FP8 oracle "
                                          f"(float64 matmul), {t_cpu:.1f} s"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
