"""Expert-parallel layer (invariant_moe_gb300.ep) through the library's
kernels on one GPU.

One GPU runs the ranks one after another in this process (no kernel waits on
another rank): each emulated rank dispatches its tokens, the test moves the
chunks between the ranks as the two all-to-alls would, each rank runs the
expert GEMMs on what it received with its own slice of the experts, and each
home rank combines.  Every rank's output must have the bits of
bi_moe_forward on that rank's tokens with all experts.  A one-rank NCCL
process group runs the same protocol through torch.distributed."""
import os
import socket

import pytest
import torch

from tests import synthetic as syn

pytestmark = pytest.mark.gpu


def _chunk(t, counts, i):
    s = sum(counts[:i])
    return t[s:s + counts[i]]


def emulate_ranks(ops, xs, idss, wtss, w13, w2, E):
    from invariant_moe_gb300 import ep
    R = len(xs)
    el = E // R
    ds = [ep.dispatch(ops, xs[r], idss[r], wtss[r], E, R) for r in range(R)]
    contrib = []
    for d in range(R):  # rank d: rows from every source rank, in source order
        rows = torch.cat([_chunk(ds[r].rows, ds[r].send_counts, d) for r in range(R)])
        lid = torch.cat([_chunk(ds[r].lid, ds[r].send_counts, d) for r in range(R)])
        pw = torch.cat([_chunk(ds[r].pw, ds[r].send_counts, d) for r in range(R)])
        contrib.append(ep.experts(ops, rows, lid, pw, w13[d * el:(d + 1) * el], w2[d * el:(d + 1) * el]))
    outs = []
    for r in range(R):  # home rank r: its rows back from every owning rank
        back = torch.cat([_chunk(contrib[d], [ds[s].send_counts[d] for s in range(R)], r) for d in range(R)])
        outs.append(ep.combine_home(ops, ds[r], back))
    return outs, ds


@pytest.mark.parametrize("R,kind", [(2, "rand"), (4, "rand"), (4, "skew")])
def test_emulated_ranks_match_single_gpu_layer(cuda, R, kind):
    import invariant_moe_gb300 as bm
    from invariant_moe_gb300 import ep
    H, E, I, k = syn.QWEN_SHAPE["H"], syn.QWEN_SHAPE["E"], syn.QWEN_SHAPE["I"], syn.QWEN_SHAPE["top_k"]
    w = syn.moe_weights(H, E, I, seed=31, device="cuda")
    f = syn.random_routing if kind == "rand" else syn.skewed_routing
    xs, idss, wtss = [], [], []
    for r in range(R):
        M = 50 + 113 * r
        xs.append(syn.moe_tokens(M, H, seed=40 + r).to(cuda))
        ids, wts = f(M, E, k, seed=50 + r)
        idss.append(ids.to(cuda))
        wtss.append(wts.to(cuda))
    outs, ds = emulate_ranks(ep.CudaOps(), xs, idss, wtss, w.w13, w.w2, E)
    torch.cuda.synchronize()
    for r in range(R):
        ref = bm.bi_moe_forward(xs[r], idss[r], wtss[r], w.w13, w.w2)
        torch.cuda.synchronize()
        assert torch.equal(outs[r], ref), f"rank {r}: differs from the single-GPU layer"
        assert sum(ds[r].send_counts) == xs[r].shape[0] * k


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_one_rank_nccl_group(cuda):
    """The protocol through torch.distributed (NCCL, one rank): the
    all-to-alls carry the rows, the routing and the contributions."""
    import torch.distributed as dist

    import invariant_moe_gb300 as bm
    from invariant_moe_gb300 import ep
    if dist.is_initialized():
        pytest.skip("a process group already exists in this process")
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1,
                            device_id=cuda)
    try:
        H, E, I, k, M = 1024, 32, 256, 4, 300
        w = syn.moe_weights(H, E, I, seed=61, unit=True, device="cuda")
        x = syn.moe_tokens(M, H, seed=62, unit=True).to(cuda)
        ids, wts = syn.random_routing(M, E, k, seed=63)
        ids, wts = ids.to(cuda), wts.to(cuda)
        out = ep.ep_moe_forward(x, ids, wts, w.w13, w.w2, E, ep.TorchComm())
        ref = bm.bi_moe_forward(x, ids, wts, w.w13, w.w2)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    finally:
        dist.destroy_process_group()
