"""The Muon step sharded over data-parallel ranks (one process per GPU).

Every rank holds the whole bank of parameters and its own gradients.  Each
matrix's step depends on that matrix alone, so ownership splits the work
(muon_partition: heaviest first, identical shapes together, least-loaded
rank):

  1. the gradients of each matrix are averaged onto its owner rank (one
     packed fp32 reduce per owner);
  2. every rank runs the Muon step (muon_step, the CUDA path) on the matrices
     it owns; momentum buffers live on the owner only;
  3. every owner broadcasts its updated parameters (one packed broadcast per
     owner), so all ranks end with the same parameters.

This is the exchange around the step in the page "深入解析KellerJordan/
modded-nanogpt中的训练架构与优化技术" (reposource.net), section "Muon优化器：
动量正交化技术": each rank orthogonalises its share of the parameters and
the updates are then gathered on all ranks.  The collectives use
torch.distributed (NCCL for CUDA tensors).
"""

import torch
import torch.distributed as dist

from . import muon


def owners(shapes, world):
    """Owner rank of each matrix (muon_partition)."""
    return muon.partition([tuple(s) for s in shapes], world)


def _packed(tensors, dtype):
    return torch.cat([t.reshape(-1).to(dtype) for t in tensors]) if tensors else None


def _unpack_into(flat, tensors):
    off = 0
    for t in tensors:
        n = t.numel()
        t.copy_(flat[off:off + n].view(t.shape).to(t.dtype))
        off += n


def reduce_grads_to_owners(grads, owner, rank, world, group=None):
    """Averages every matrix's gradient over the ranks onto its owner.
    Returns {matrix index: averaged fp32 gradient} for the matrices `rank`
    owns (new tensors; `grads` is not modified)."""
    out = {}
    for r in range(world):
        idx = [i for i, o in enumerate(owner) if o == r]
        if not idx:
            continue
        flat = _packed([grads[i] for i in idx], torch.float32)
        dist.reduce(flat, dst=r, op=dist.ReduceOp.SUM, group=group)
        if r == rank:
            flat.div_(world)
            off = 0
            for i in idx:
                n = grads[i].numel()
                out[i] = flat[off:off + n].view(grads[i].shape)
                off += n
    return out


def broadcast_params_from_owners(params, owner, world, group=None):
    """Every owner sends its matrices' parameters to all ranks (in place)."""
    for r in range(world):
        idx = [i for i, o in enumerate(owner) if o == r]
        if not idx:
            continue
        flat = _packed([params[i] for i in idx], params[idx[0]].dtype)
        dist.broadcast(flat, src=r, group=group)
        _unpack_into(flat, [params[i] for i in idx])


def sharded_muon_step(params, grads, bufs, lr=0.02, momentum=0.95, nesterov=True, ns_steps=5, group=None,
                      workspace=None, stream=None):
    """One data-parallel Muon step.  params, grads, bufs: lists of 2-D CUDA
    tensors of the whole bank (fp32 params and buffers; bufs are used and
    updated only for the matrices this rank owns).  Returns the workspace
    used for the local step (reuse it across steps), or None when this rank
    owns no matrix."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    owner = owners([p.shape for p in params], world)
    mine = reduce_grads_to_owners(grads, owner, rank, world, group)
    if mine:
        idx = sorted(mine)
        workspace = muon.muon_step([params[i] for i in idx], [mine[i] for i in idx], [bufs[i] for i in idx],
                                   lr=lr, momentum=momentum, nesterov=nesterov, ns_steps=ns_steps,
                                   workspace=workspace, stream=stream)
    broadcast_params_from_owners(params, owner, world, group)
    return workspace if mine else None
