"""Test-side implementation of the expert-parallel protocol's per-rank data
steps on CPU tensors, so the protocol's host logic (split sizes, the order
rows travel in and come back in, the return to (token, slot) order, the slot
order of the sum) runs on gloo ranks without a GPU.  The expert arithmetic is
the fp64 oracle's, rounded to fp32 contributions; the slot-order sum is fp32.
Test infrastructure only: the library's own path is
invariant_moe_gb300.ep.CudaOps."""
from __future__ import annotations

import numpy as np
import torch

from tests import synthetic as syn


class HostOps:
    def __init__(self, oracle_mod):
        self.oracle = oracle_mod

    @staticmethod
    def to_host(t):
        return t.tolist()

    def permute(self, ids, E):
        off, perm = self.oracle.permute(ids.numpy(), E)
        return torch.from_numpy(off), torch.from_numpy(perm)

    @staticmethod
    def gather_rows(x, offsets, perm, top_k):
        n = int(offsets[-1])
        return x[perm[:n].long() // top_k].contiguous()

    @staticmethod
    def gather_routing(ids, wts, offsets, perm, experts_per_rank):
        n = int(offsets[-1])
        p = perm[:n].long()
        return (ids.flatten()[p] % experts_per_rank).to(torch.int32), wts.flatten()[p].contiguous()

    def experts(self, rows, lid, pw, w13_local, w2_local):
        R, H = rows.shape
        out = torch.zeros(R, H, dtype=torch.float32)
        el, twoI, _ = w13_local.shape
        w13b, w2b = syn.bf16_bits(w13_local), syn.bf16_bits(w2_local)
        xb = syn.bf16_bits(rows)
        for r in range(R):
            c = self.oracle.moe(xb[r:r + 1], np.array([[int(lid[r])]], np.int32),
                                np.array([[float(pw[r])]], np.float32), w13b, w2b, el, twoI // 2)
            out[r] = torch.from_numpy(c[0].astype(np.float32))
        return out

    @staticmethod
    def scatter_contrib(back, offsets, perm, M, top_k):
        contrib = torch.zeros(M * top_k, back.shape[-1], dtype=torch.float32)
        n = back.shape[0]
        contrib[perm[:n].long()] = back
        return contrib

    @staticmethod
    def combine(contrib, M, top_k):
        c = contrib.view(M, top_k, -1).numpy()
        s = c[:, 0].copy()
        for t in range(1, top_k):
            s = (s + c[:, t]).astype(np.float32)   # fp32 adds in slot order
        return torch.from_numpy(s)


class LocalComm:
    """One rank alone: the exchange is the identity."""
    world, rank = 1, 0

    @staticmethod
    def exchange_counts(send_counts, device):
        return list(send_counts)

    @staticmethod
    def all_to_all(send, send_counts, recv_counts):
        return send
