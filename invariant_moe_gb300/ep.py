"""Expert-parallel MoE layer: the experts split over R ranks, every output bit
the single-GPU layer's.

Source: "Batch-invariance generation with vLLM fused-MoE backend at improved
performance", sections "Summary" (the batch-invariant fused-MoE run with
expert parallelism over 8 GPUs) and "Usage" (the token dispatcher).  The
pages run that topology without stating how bits survive it; the rule kept
here is the plain one: a token's k contributions are computed by the same
kernels (same K order) on whichever rank owns each expert, travel back to the
token's home rank unchanged (fp32 rows), and are summed there in slot order,
so the sum is the single-GPU combine's.

Rank r owns experts [r*E/R, (r+1)*E/R) (E divisible by R).  One call:

  home rank   route      bi_moe_permute groups the (token, slot) pairs by
                         expert -- hence by destination rank, each rank's
                         pairs a contiguous range of positions;
                         bi_moe_gather copies the token rows in that order
                         and bi_moe_gather_routing their local expert index
                         and probability
  exchange 1             rows, local expert ids and probabilities, one
                         all-to-all each (split sizes from the offsets)
  owning rank experts    the expert GEMMs on the rows received, top_k = 1,
                         a row's pair id = its index in the received order:
                         fp32 contribution rows in that order
  exchange 2             the contribution rows back, splits reversed: each
                         home rank gets its rows in its own permuted order
  home rank   combine    bi_moe_scatter_contrib puts them back at row
                         token*top_k + slot, bi_moe_combine sums the slots
                         in order (fp32) and rounds once to bf16

Only the split sizes cross to the host (one small device-to-host read per
call): the all-to-all needs them.  The data path stays on the device; the
collectives are torch.distributed's (NCCL between GPUs).  Slots whose expert
id is invalid are skipped by the permutation and add +0 (the home rank's
contribution buffer starts zeroed); a slot-order sum that adds +0 for them
equals the sum over the valid slots.

The protocol is written against two small interfaces so that its host logic
can be tested on CPU ranks (gloo) with a test-side implementation of the
ops: `ops` (the per-rank data steps; `CudaOps` calls the library's kernels
and nothing else) and `comm` (split sizes and the all-to-all;
`TorchComm` over torch.distributed).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass
class Dispatch:
    """What the home rank keeps between sending its rows and combining."""
    M: int
    top_k: int
    E: int
    offsets: torch.Tensor      # [E+1] int32: positions of each expert's pairs
    perm: torch.Tensor         # [M*top_k] int32: pair id at each position
    send_counts: list          # rows sent to each rank
    rows: torch.Tensor         # [sum(send_counts), H] token rows, permuted order
    lid: torch.Tensor          # [sum(send_counts)] int32 expert index on its rank
    pw: torch.Tensor           # [sum(send_counts)] fp32 routing probability


def split_counts(offsets_host, E, world):
    """Pairs sent to each rank: rank d owns experts [d*E/R, (d+1)*E/R), whose
    pairs occupy positions [offsets[d*E/R], offsets[(d+1)*E/R])."""
    if E % world:
        raise ValueError(f"E={E} is not divisible by the {world} ranks")
    el = E // world
    return [int(offsets_host[(d + 1) * el]) - int(offsets_host[d * el]) for d in range(world)]


def dispatch(ops, x, ids, wts, E, world):
    """Home-rank step 1: group the pairs by expert (and so by destination)
    and gather what travels with them."""
    M, top_k = ids.shape
    offsets, perm = ops.permute(ids, E)
    counts = split_counts(ops.to_host(offsets), E, world)
    n = sum(counts)
    rows = ops.gather_rows(x, offsets, perm, top_k)[:n]
    lid, pw = ops.gather_routing(ids, wts, offsets, perm, E // world)
    return Dispatch(M, top_k, E, offsets, perm, counts, rows, lid[:n], pw[:n])


def experts(ops, rows, lid, pw, w13_local, w2_local):
    """Owning-rank step: the expert GEMMs on the received rows; returns their
    fp32 contribution rows in the received order."""
    return ops.experts(rows, lid, pw, w13_local, w2_local)


def combine_home(ops, d, back):
    """Home-rank step 2: contribution rows (back, in the permuted order) to
    (token, slot) order, then the slot-order sum."""
    contrib = ops.scatter_contrib(back, d.offsets, d.perm, d.M, d.top_k)
    return ops.combine(contrib, d.M, d.top_k)


def ep_moe_forward(x, ids, wts, w13_local, w2_local, E, comm, ops=None):
    """out [M, H] for this rank's M tokens, with this rank's experts
    w13_local [E/R, 2I, H], w2_local [E/R, H, I] and the ranks of `comm`."""
    ops = ops if ops is not None else CudaOps()
    d = dispatch(ops, x, ids, wts, E, comm.world)
    recv_counts = comm.exchange_counts(d.send_counts, x.device)
    rows = comm.all_to_all(d.rows, d.send_counts, recv_counts)
    lid = comm.all_to_all(d.lid, d.send_counts, recv_counts)
    pw = comm.all_to_all(d.pw, d.send_counts, recv_counts)
    contrib_rows = experts(ops, rows, lid, pw, w13_local, w2_local)
    back = comm.all_to_all(contrib_rows, recv_counts, d.send_counts)
    return combine_home(ops, d, back)


class TorchComm:
    """Split sizes and all-to-all over a torch.distributed process group
    (NCCL for CUDA tensors, gloo for CPU tensors)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)

    def exchange_counts(self, send_counts, device):
        s = torch.tensor(send_counts, dtype=torch.int64, device=device)
        r = torch.empty_like(s)
        self.dist.all_to_all_single(r, s, group=self.group)
        return [int(v) for v in r.tolist()]

    def all_to_all(self, send, send_counts, recv_counts):
        out = torch.empty((sum(recv_counts),) + tuple(send.shape[1:]), dtype=send.dtype, device=send.device)
        self.dist.all_to_all_single(out, send.contiguous(), output_split_sizes=list(recv_counts),
                                    input_split_sizes=list(send_counts), group=self.group)
        return out


class CudaOps:
    """The per-rank data steps, each one of the library's kernels (no other
    arithmetic).  Tensors live on the current CUDA device."""

    def __init__(self):
        from invariant_moe_gb300 import load_library
        load_library()  # fails loudly when the CUDA library is missing

    @staticmethod
    def to_host(t):
        return t.cpu().tolist()

    @staticmethod
    def permute(ids, E):
        import invariant_moe_gb300 as bm
        return bm.bi_moe_permute(ids, E)

    @staticmethod
    def gather_rows(x, offsets, perm, top_k):
        import invariant_moe_gb300 as bm
        return bm.bi_moe_gather(x, offsets, perm, top_k)

    @staticmethod
    def gather_routing(ids, wts, offsets, perm, experts_per_rank):
        import invariant_moe_gb300 as bm
        return bm.bi_moe_gather_routing(ids, wts, offsets, perm, experts_per_rank)

    @staticmethod
    def experts(rows, lid, pw, w13_local, w2_local):
        import invariant_moe_gb300 as bm
        R, H = rows.shape
        if R == 0:
            return torch.empty(0, H, dtype=torch.float32, device=rows.device)
        el = w13_local.shape[0]
        off, perm = bm.bi_moe_permute(lid.view(R, 1), el)
        xp = bm.bi_moe_gather(rows, off, perm, 1)
        act = bm.bi_moe_gate_up(xp, off, perm, pw.view(R, 1), w13_local, 1)
        return bm.bi_moe_down(act, off, perm, w2_local, R, 1)

    @staticmethod
    def scatter_contrib(back, offsets, perm, M, top_k):
        import invariant_moe_gb300 as bm
        H = back.shape[-1]
        contrib = torch.zeros(M * top_k, H, dtype=torch.float32, device=back.device)
        if back.shape[0]:
            bm.bi_moe_scatter_contrib(back, offsets, perm, M, top_k, contrib=contrib)
        return contrib

    @staticmethod
    def combine(contrib, M, top_k):
        import invariant_moe_gb300 as bm
        return bm.bi_moe_combine(contrib, M, top_k)
