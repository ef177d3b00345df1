"""The Muon step sharded over data-parallel ranks (one process per GPU).

Every rank holds the whole bank of parameters and computes gradients for all
of it.  Each matrix's step depends on that matrix alone, so ownership splits
the work (muon_partition: heaviest first, identical shapes together,
least-loaded rank).  The exchange around the local step follows the page
"深入解析KellerJordan/modded-nanogpt中的训练架构与优化技术" (reposource.net),
section "Muon优化器：动量正交化技术" (parameters grouped by size; each rank
orthogonalises its share of a group; the updated parameters are gathered
with an asynchronous all_gather_into_tensor, the next group's work
overlapping it), with a reduce-scatter of the gradients in front, as the
energy-efficiency page (bxzpzcl.cn) describes for the gradients:

  per size group g (largest matrices first):
    1. reduce_scatter_tensor of the group's gradients, in their own dtype:
       each rank receives the sum over ranks of the gradients of the
       matrices it owns, and divides it by the world size (the average);
    2. muon_step (the CUDA path) on the rank's matrices of the group; their
       momentum buffers live on the owner only;
    3. all_gather_into_tensor of the group's updated parameters, issued
       asynchronously so that it overlaps the next group's steps 1-2.

Layout (what makes the exchange copy-free): for every group the parameters
and the gradients live in one flat buffer each, ordered by owner rank, every
rank's segment padded to the group's longest segment.  A rank's segment of
the gradient buffer is exactly the reduce-scatter's input chunk for that
rank, and its segment of the parameter buffer is its all-gather input.
``ShardedBank.params`` and ``ShardedBank.grads`` are views into these
buffers, in bank order, for the training code to read and write.
"""

import torch
import torch.distributed as dist

from . import muon


def owners(shapes, world):
    """Owner rank of each matrix (muon_partition)."""
    return muon.partition([tuple(s) for s in shapes], world)


def size_groups(shapes):
    """Matrix indices grouped by element count, largest first (the page
    groups its parameters by size); bank order within a group."""
    by = {}
    for i, (r, c) in enumerate(shapes):
        by.setdefault(r * c, []).append(i)
    return [by[k] for k in sorted(by, reverse=True)]


class _Group:
    """One size group's owner-ordered layout on one rank."""

    def __init__(self, idx, shapes, owner, world):
        self.idx = idx
        self.numel = shapes[idx[0]][0] * shapes[idx[0]][1]
        self.members = [[i for i in idx if owner[i] == r] for r in range(world)]
        self.seg = self.numel * max(len(m) for m in self.members)  # elements per rank segment
        # element offset of each matrix in the flat buffer
        self.offset = {}
        for r, mem in enumerate(self.members):
            for k, i in enumerate(mem):
                self.offset[i] = r * self.seg + k * self.numel


class ShardedBank:
    """A bank of 2-D matrices stepped with Muon over `world` data-parallel
    ranks.

    shapes      (rows, cols) of every matrix, identical on every rank;
    device      where the buffers live (CUDA for the real step; the CPU
                tests use gloo on CPU tensors);
    grad_dtype  dtype of the gradients and of the reduce-scatter
                (bfloat16 by default, as the training computes them).

    params (fp32) and grads are lists of views in bank order.  bufs holds a
    zero-initialised fp32 momentum buffer for each matrix this rank owns
    (None for the others).  step() runs the exchange and the local steps;
    `local_step(params, grads, bufs, lr, momentum, nesterov, ns_steps,
    workspace)` defaults to the CUDA muon_step."""

    def __init__(self, shapes, device, group=None, grad_dtype=torch.bfloat16):
        self.shapes = [tuple(int(x) for x in s) for s in shapes]
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.device = torch.device(device)
        self.owner = owners(self.shapes, self.world)
        self.groups = [_Group(idx, self.shapes, self.owner, self.world) for idx in size_groups(self.shapes)]
        self.param_flat = [torch.zeros(self.world * g.seg, dtype=torch.float32, device=self.device)
                           for g in self.groups]
        self.grad_flat = [torch.zeros(self.world * g.seg, dtype=grad_dtype, device=self.device) for g in self.groups]
        # the reduce-scatter's output: this rank's summed (then averaged) gradients
        self.grad_mine = [torch.empty(g.seg, dtype=grad_dtype, device=self.device) for g in self.groups]
        self.params = [None] * len(self.shapes)
        self.grads = [None] * len(self.shapes)
        self.bufs = [None] * len(self.shapes)
        self._mine = []  # per group: (index, param view, averaged-gradient view, buffer)
        for g, pf, gf, gm in zip(self.groups, self.param_flat, self.grad_flat, self.grad_mine):
            mine = []
            for i in g.idx:
                r, c = self.shapes[i]
                o = g.offset[i]
                self.params[i] = pf[o:o + r * c].view(r, c)
                self.grads[i] = gf[o:o + r * c].view(r, c)
                if self.owner[i] == self.rank:
                    lo = o - self.rank * g.seg
                    self.bufs[i] = torch.zeros((r, c), dtype=torch.float32, device=self.device)
                    mine.append((i, self.params[i], gm[lo:lo + r * c].view(r, c), self.bufs[i]))
            self._mine.append(mine)
        self.workspace = None

    def owned(self):
        """Indices of the matrices this rank owns."""
        return [i for i, o in enumerate(self.owner) if o == self.rank]

    def exchange_bytes(self):
        """Bytes this rank sends per step: its reduce-scatter input minus its
        own segment, and its all-gather segment to every other rank (both
        per group, padding included)."""
        out = 0
        for g, gf, pf in zip(self.groups, self.grad_flat, self.param_flat):
            out += (self.world - 1) * g.seg * (gf.element_size() + pf.element_size())
        return out

    def step(self, lr=0.02, momentum=0.95, nesterov=True, ns_steps=5, local_step=None, stream=None):
        """One data-parallel Muon step over the bank (in place)."""
        if local_step is None:
            local_step = self._cuda_step
        pending = []
        # every group's reduce-scatter is issued up front; each group then
        # waits for its own before stepping
        rs = [dist.reduce_scatter_tensor(gm, gf, op=dist.ReduceOp.SUM, group=self.group, async_op=True)
              for gm, gf in zip(self.grad_mine, self.grad_flat)]
        for g, mine, work, gm, pf in zip(self.groups, self._mine, rs, self.grad_mine, self.param_flat):
            work.wait()
            if mine:
                gm.div_(self.world)
                local_step([m[1] for m in mine], [m[2] for m in mine], [m[3] for m in mine], lr, momentum,
                           nesterov, ns_steps, stream)
            seg = pf[self.rank * g.seg:(self.rank + 1) * g.seg]
            pending.append(dist.all_gather_into_tensor(pf, seg, group=self.group, async_op=True))
        for w in pending:
            w.wait()

    def _cuda_step(self, params, grads, bufs, lr, momentum, nesterov, ns_steps, stream):
        # one workspace, sized for the largest group, reused by every group's
        # call (stream-ordered)
        need = muon.muon_workspace_size([tuple(p.shape) for p in params])
        if self.workspace is None or self.workspace.numel() < need:
            self.workspace = muon.new_workspace(max(need, max(
                muon.muon_workspace_size([tuple(self.shapes[m[0]]) for m in mine]) for mine in self._mine if mine)),
                self.device)
        muon.muon_step(params, grads, bufs, lr=lr, momentum=momentum, nesterov=nesterov, ns_steps=ns_steps,
                       workspace=self.workspace, stream=stream)
