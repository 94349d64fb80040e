"""Router + top-k in one call (bi_router_topk) on the GPU.

With schedule 10 the call is one kernel (a cluster owns all N scores of up
to 4 rows and selects from distributed shared memory); otherwise the
selection grid runs as a programmatic dependent of the router grid.  Either
way the call must reproduce the two separate calls bit for bit: the same scores as
bi_router_gemm under every schedule, and the same ids, wts and probs as
bi_topk on those scores (which a missed dependency would break).  Against the oracle it is pinned through
that equality plus a direct check of the selection on rows without near-ties,
the oracle computing its own fp64 scores from the host inputs."""
import numpy as np
import pytest
import torch

from tests import synthetic as syn

pytestmark = pytest.mark.gpu

MS = (1, 2, 3, 4, 5, 8, 17, 64, 100, 383, 384, 1000, 4096)


def two_launch(bm, x, w, b, k, schedule):
    y = bm.bi_router_gemm(x, w, b, schedule=schedule)
    ids, wts, probs = bm.bi_topk(y, k, want_probs=True)
    return y, ids, wts, probs


@pytest.fixture(scope="module")
def dsv4(cuda):
    inp = syn.router_inputs()
    return inp, inp.x.to(cuda), inp.w.to(cuda), inp.b.to(cuda)


@pytest.mark.parametrize("schedule", [0, 1, 2, 3, 4, 7, 9])
def test_fused_equals_two_launch_dsv4(cuda, dsv4, schedule):
    import invariant_moe_gb300 as bm
    _, x, w, b = dsv4
    for M in MS:
        if schedule == 1 and M > 1000:
            continue  # the rows schedule at M=4096 is slow and adds nothing
        xm = x[:M].contiguous()
        y1, i1, w1, p1 = two_launch(bm, xm, w, b, 8, schedule)
        y2, i2, w2, p2 = bm.bi_router_topk(xm, w, 8, bias=b, want_probs=True, schedule=schedule)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2), f"scores M={M}"
        assert torch.equal(i1, i2), f"ids M={M}"
        assert torch.equal(w1, w2), f"wts M={M}"
        assert torch.equal(p1, p2), f"probs M={M}"
    assert bm.device_error() == 0


@pytest.mark.parametrize("k", [1, 8, 16])
def test_fused_equals_two_launch_qwen_shape(cuda, k):
    """K=2048, N=128, no bias (the Qwen3-30B-A3B-shaped router)."""
    import invariant_moe_gb300 as bm
    g = syn.gen(71)
    x = torch.randn(1500, 2048, generator=g).to(cuda)
    w = (torch.randn(128, 2048, generator=g) * 0.02).to(cuda)
    for M, sched in ((1, 0), (4, 0), (9, 0), (300, 0), (1500, 0), (33, 9), (1500, 9)):
        xm = x[:M].contiguous()
        y1, i1, w1, _ = two_launch(bm, xm, w, None, k, sched)
        y2, i2, w2, _ = bm.bi_router_topk(xm, w, k, schedule=sched)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2) and torch.equal(i1, i2) and torch.equal(w1, w2), f"M={M}"


@pytest.mark.parametrize("shape", ["dsv4", "qwen", "n64"])
@pytest.mark.parametrize("xdtype", [torch.float32, torch.bfloat16])
def test_one_kernel_equals_two_launch(cuda, shape, xdtype):
    """The one-kernel path (forced: schedule 10) against bi_router_gemm +
    bi_topk: scores, ids, wts and probs bit for bit, for every batch size it
    takes (1..4), fp32 and bf16 tokens, with and without bias, top_k 1..16,
    and the cluster sizes 16 (N=256), 8 (N=128) and 4 (N=64)."""
    import invariant_moe_gb300 as bm
    K, N = {"dsv4": (4096, 256), "qwen": (2048, 128), "n64": (3072, 64)}[shape]
    g = syn.gen(81 + N)
    x = torch.randn(4, K, generator=g).to(xdtype).to(cuda)
    w = (torch.randn(N, K, generator=g) / K ** 0.5).to(cuda)
    b = (torch.randn(N, generator=g) * 0.01).to(cuda)
    for M in (1, 2, 3, 4):
        for bias in (b, None):
            for k in (1, 8, 16):
                xm = x[:M].contiguous()
                y1 = bm.bi_router_gemm(xm, w, bias)
                i1, w1, p1 = bm.bi_topk(y1, k, want_probs=True)
                y2, i2, w2, p2 = bm.bi_router_topk(xm, w, k, bias=bias, want_probs=True, schedule=10)
                torch.cuda.synchronize()
                tag = f"{shape} M={M} k={k} bias={bias is not None} x={xdtype}"
                assert torch.equal(y1, y2), "scores " + tag
                assert torch.equal(i1, i2), "ids " + tag
                assert torch.equal(w1, w2), "wts " + tag
                assert torch.equal(p1, p2), "probs " + tag
    assert bm.device_error() == 0


def test_one_kernel_ties_and_rows(cuda):
    """Exact plateaus (duplicated W rows, x on multiples of 1/8) through the
    one-kernel path: the same ids as the separate selection, and each row's
    result is the same alone or beside up to three other rows."""
    import invariant_moe_gb300 as bm
    inp, rows = syn.router_tie_inputs(M=64)
    x, w, b = inp.x.to(cuda), inp.w.to(cuda), inp.b.to(cuda)
    tied = torch.nonzero(rows).flatten()[:4].tolist() + [0, 1, 2, 3]
    for r0 in tied:
        alone = bm.bi_router_topk(x[r0:r0 + 1].contiguous(), w, 8, bias=b, schedule=10)
        y1 = bm.bi_router_gemm(x[r0:r0 + 1].contiguous(), w, b)
        i1, w1, _ = bm.bi_topk(y1, 8)
        torch.cuda.synchronize()
        assert torch.equal(alone[1], i1) and torch.equal(alone[2], w1)
        for M in (2, 3, 4):
            xb = x[60 - M:60].clone()
            xb[M - 1] = x[r0]
            got = bm.bi_router_topk(xb, w, 8, bias=b, schedule=10)
            torch.cuda.synchronize()
            for t in range(3):
                assert torch.equal(got[t][M - 1], alone[t][0]), f"row {r0} beside {M - 1} others"


def test_one_kernel_rejects_shapes_it_does_not_take(cuda):
    """Schedule 10 on a shape the one-kernel path does not take is an error,
    not a silent fallback: N not a multiple of 16, more than 4 rows, K not a
    multiple of 1024."""
    import invariant_moe_gb300 as bm
    g = syn.gen(5)
    for M, K, N in ((1, 4096, 200), (5, 4096, 256), (2, 640, 128)):
        x = torch.randn(M, K, generator=g).to(cuda)
        w = torch.randn(N, K, generator=g).to(cuda)
        with pytest.raises(RuntimeError, match="BI_ERR_UNSUPPORTED"):
            bm.bi_router_topk(x, w, 8, schedule=10)


def test_fused_ties_and_invariance(cuda):
    """Duplicated W rows give exact plateaus; the fused selection breaks them
    by index exactly as the separate top-k, and every row's ids are the same
    whatever the batch size."""
    import invariant_moe_gb300 as bm
    inp, _ = syn.router_tie_inputs(M=4096)
    x, w, b = inp.x.to(cuda), inp.w.to(cuda), inp.b.to(cuda)
    _, ref_ids, ref_w, _ = bm.bi_router_topk(x, w, 8, bias=b)
    _, i1, _, _ = two_launch(bm, x, w, b, 8, 0)
    torch.cuda.synchronize()
    assert torch.equal(ref_ids, i1)
    for M in syn.batch_sizes(4096):
        _, ids, wts, _ = bm.bi_router_topk(x[:M].contiguous(), w, 8, bias=b)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids[:M]) and torch.equal(wts, ref_w[:M]), f"M={M}"


def test_fused_against_oracle(oracle_mod, cuda, dsv4):
    """Scores within the router tolerance of the fp64 oracle; ids equal to
    the oracle's own selection on rows whose top-k+1 ordering has no
    near-tie below 1e-4; wts within fp32 rounding of sigmoid(oracle score)."""
    import invariant_moe_gb300 as bm
    inp, x, w, b = dsv4
    M = 512
    y, ids, wts, _ = bm.bi_router_topk(x[:M].contiguous(), w, 8, bias=b)
    torch.cuda.synchronize()
    r = oracle_mod.router(inp.x[:M].numpy(), inp.w.numpy(), inp.b.numpy())
    yg = y.cpu().numpy()
    assert np.all(np.abs(yg - r) <= 2e-3 + 1e-4 * np.abs(r))
    ok = syn.unambiguous_rows(r, 8)
    assert len(ok) >= 0.9 * M
    ids_o, wts_o = oracle_mod.topk(r.astype(np.float32), 8)
    assert np.array_equal(ids.cpu().numpy()[ok], ids_o[ok])
    assert np.all(np.abs(wts.cpu().numpy()[ok] - wts_o[ok]) <= 2e-3)


def test_fused_repeatable_and_stream_ordered(cuda, dsv4):
    """Back-to-back calls at different M, and a call whose scores buffer was
    just overwritten by another kernel, give the same bits: the selection
    always reads the router output of its own call."""
    import invariant_moe_gb300 as bm
    _, x, w, b = dsv4
    y = torch.empty(4096, 256, dtype=torch.float32, device=cuda)
    outs = []
    for M in (4096, 1, 37, 4096):
        y.fill_(float("nan"))
        _, ids, wts, _ = bm.bi_router_topk(x[:M].contiguous(), w, 8, bias=b, out=y[:M])
        outs.append((ids.clone(), wts.clone()))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[3][0]) and torch.equal(outs[0][1], outs[3][1])
    assert torch.equal(outs[1][0], outs[0][0][:1])
    assert torch.equal(outs[2][0], outs[0][0][:37])


def test_fused_empty_batch(cuda, dsv4):
    import invariant_moe_gb300 as bm
    _, x, w, b = dsv4
    y, ids, wts, _ = bm.bi_router_topk(x[:0], w, 8, bias=b)
    assert ids.shape == (0, 8) and y.shape == (0, 256)
