"""The layer captured once in a CUDA graph and replayed with new tokens
copied into the captured input: every replay gives the bits of an eager call
on those tokens (scores, ids, wts, out).  Replays run back to back on one
stream, so the decode path's per-token completion counters and the
workspace's routing must be rebuilt by each replay, not left from the last."""
import pytest
import torch

from tests import synthetic as syn

pytestmark = pytest.mark.gpu

SHAPES = {"qwen": (2048, 128, 768, 8), "dsv4": (4096, 256, 2048, 8), "small": (384, 8, 256, 2),
          "mid": (1024, 16, 512, 4)}


# qwen 1 and mid 4: the decode layer's one-launch expert path, whose arrival
# count each replay's router kernel zeroes again
@pytest.mark.parametrize("shape,M", [("qwen", 1), ("qwen", 3), ("dsv4", 1), ("dsv4", 4), ("mid", 4),
                                     ("qwen", 300), ("small", 1000)])
def test_layer_graph_replays_same_bits_as_eager(cuda, shape, M):
    import invariant_moe_gb300 as bm
    H, E, I, k = SHAPES[shape]
    w = syn.moe_weights(H, E, I, seed=M + 201, unit=True, device="cuda")
    b = syn.normal((E,), 0.01, M + 202).to(cuda)
    xs = [syn.moe_tokens(M, H, seed=M + 203 + i, unit=True).to(cuda) for i in range(4)]
    eager = []
    for x in xs:
        eager.append([t.clone() for t in bm.bi_moe_layer(x, w.w_router, w.w13, w.w2, k, bias=b)])
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(cuda)
    x_in = xs[0].clone()
    out = torch.empty(M, H, dtype=torch.bfloat16, device=cuda)
    scores = torch.empty(M, E, dtype=torch.float32, device=cuda)
    ids = torch.empty(M, k, dtype=torch.int32, device=cuda)
    wts = torch.empty(M, k, dtype=torch.float32, device=cuda)
    ws = bm.moe_workspace(M, H, E, k, I, cuda)

    def call():
        bm.bi_moe_layer(x_in, w.w_router, w.w13, w.w2, k, bias=b, out=out, scores=scores, ids=ids, wts=wts,
                        workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        call()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()
        for order in ((1, 2, 3, 0), (3, 3, 1)):
            for i in order:
                x_in.copy_(xs[i])
                g.replay()
                stream.synchronize()
                for got, ref, name in zip((out, scores, ids, wts), eager[i], ("out", "scores", "ids", "wts")):
                    assert torch.equal(got, ref), f"replay of tokens {i}: {name}"
        # back-to-back replays with no host wait between them
        for i in (2, 0, 1):
            x_in.copy_(xs[i])
            g.replay()
        stream.synchronize()
        assert torch.equal(out, eager[1][0])
    assert bm.device_error() == 0


@pytest.mark.parametrize("M", [1, 200])
def test_forward_graph_replays_same_bits_as_eager(cuda, M):
    """bi_moe_forward alone (routing given), captured and replayed with new
    tokens and new routing."""
    import invariant_moe_gb300 as bm
    H, E, I, k = SHAPES["qwen"]
    w = syn.moe_weights(H, E, I, seed=M + 211, unit=True, device="cuda")
    cases = []
    for i in range(3):
        x = syn.moe_tokens(M, H, seed=M + 212 + i, unit=True).to(cuda)
        ids, wts = syn.random_routing(M, E, k, seed=M + 215 + i)
        cases.append((x, ids.to(cuda), wts.to(cuda)))
    eager = [bm.bi_moe_forward(x, ids, wts, w.w13, w.w2).clone() for x, ids, wts in cases]
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(cuda)
    x_in, ids_in, wts_in = (t.clone() for t in cases[0])
    out = torch.empty(M, H, dtype=torch.bfloat16, device=cuda)
    ws = bm.moe_workspace(M, H, E, k, I, cuda)

    def call():
        bm.bi_moe_forward(x_in, ids_in, wts_in, w.w13, w.w2, out=out, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        call()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()
        for i in (2, 1, 0, 2):
            x_in.copy_(cases[i][0])
            ids_in.copy_(cases[i][1])
            wts_in.copy_(cases[i][2])
            g.replay()
            stream.synchronize()
            assert torch.equal(out, eager[i]), f"replay of case {i}"
    assert bm.device_error() == 0
