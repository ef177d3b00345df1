"""Where the Newton-Schulz kernels' time goes, per role, on one bank.

Diagnostic tool over the library's ``wait_profile_buffer`` debug hook: every
CTA of the Gram, polynomial and update kernels adds clock64 cycles per role
into a device array while ``--steps`` Muon steps run (after three untimed
ones).  Printed per phase, averaged over CTAs and over the phase's launches:

  prod_empty     TMA producer waiting for a free stage
  mma_full       MMA issuer waiting for operands (leader CTAs; others 0)
  mma_tempty     MMA issuer waiting for a drained accumulator (leader CTAs)
  epi_tfull      epilogue waiting for an accumulator
  epi_busy       epilogue working on its tiles
  kernel         whole kernel (thread 0), including the wait for the
                 previous kernel
  tiles          tiles per CTA
  mma_loop       MMA issuer's whole loop (leader CTAs)

The Muon step's last update also applies p -= lr O, so its update average
mixes four plain launches with that one; --ns5 profiles ns5_bank on the same
bank instead, whose updates are all plain.

Usage: python -m newton_schulz_08_gb300.wait_profile [gpt2|gpt1p5b|rect] [--steps N] [--ns5]
"""

import argparse
import json

import numpy as np
import torch

from . import inputs, muon

COUNTERS = ["prod_empty", "mma_full", "mma_tempty", "epi_tfull", "epi_busy", "kernel", "tiles", "mma_loop"]
PHASES = ["gram", "poly", "update"]
MAX_CTAS = 256
LEADER_ONLY = {"mma_full", "mma_tempty", "mma_loop"}


def bank(name):
    return {"gpt2": inputs.gpt2_shapes, "gpt1p5b": inputs.gpt1p5b_shapes, "rect": inputs.rect_shapes}[name]()


def profile(shapes, steps=5, ns_steps=5, device="cuda", ns5=False):
    dev = torch.device(device)
    P = [torch.from_numpy(inputs.param(s, i)).to(dev) for i, s in enumerate(shapes)]
    B = [torch.from_numpy(inputs.buffer(s, i)).to(dev) for i, s in enumerate(shapes)]
    G = [torch.from_numpy(inputs.grad(s, i)).to(dev).to(torch.bfloat16) for i, s in enumerate(shapes)]
    if ns5:
        ws = muon.new_workspace(muon.ns5_bank_workspace_size(shapes), dev)
        run = lambda: muon.ns5_bank(G, ns_steps, workspace=ws)
    else:
        ws = muon.muon_step(P, G, B, ns_steps=ns_steps)
        run = lambda: muon.muon_step(P, G, B, ns_steps=ns_steps, workspace=ws)
    for _ in range(3):
        run()
    torch.cuda.synchronize(dev)
    counts = torch.zeros(len(PHASES) * MAX_CTAS * len(COUNTERS), dtype=torch.int64, device=dev)
    muon.muon_set_debug("wait_profile_buffer", counts.data_ptr())
    try:
        for _ in range(steps):
            run()
        torch.cuda.synchronize(dev)
    finally:
        muon.muon_set_debug("wait_profile_buffer", 0)
    c = counts.view(len(PHASES), MAX_CTAS, len(COUNTERS)).cpu().numpy().astype(np.float64)
    launches = steps * ns_steps
    out = {}
    for k, phase in enumerate(PHASES):
        used = np.nonzero(c[k][:, COUNTERS.index("tiles")] > 0)[0]
        rows = c[k][used]
        leaders = c[k][used[used % 2 == 0]]  # CTA pairs: the even CTA issues the MMAs
        d = {}
        for i, name in enumerate(COUNTERS):
            src = leaders if name in LEADER_ONLY else rows
            d[name] = float(src[:, i].mean() / launches) if len(src) else 0.0
        d["ctas"] = int(len(rows))
        out[phase] = d
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("bank", nargs="?", default="gpt2", choices=["gpt2", "gpt1p5b", "rect"])
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--ns5", action="store_true", help="profile ns5_bank (no parameter update)")
    args = ap.parse_args()
    for phase, d in profile(bank(args.bank), args.steps, ns5=args.ns5).items():
        print(phase, json.dumps({k: round(v, 1) for k, v in d.items()}))


if __name__ == "__main__":
    main()
