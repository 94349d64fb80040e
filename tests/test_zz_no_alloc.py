"""bi_moe_forward_noalloc: the MoE forward for callers that cannot allocate
device memory (code running inside an allocator callback, runtimes that own
all device memory).  Its scratch space is a fixed array inside the library
instead of a caller workspace.  Called through the C ABI, it must give the
same output as bi_moe_forward with a caller-provided workspace, on two calls
in a row (the second one finds the first one's leftovers in the array).

This file sorts last so that a run stopping at the first failure has run
every other test first."""
import ctypes

import pytest
import torch

from tests import synthetic as syn

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, x, ids, wts, w13, w2, out):
    M, H = x.shape
    E, twoI, _ = w13.shape
    return lib.bi_moe_forward_noalloc(_p(x), _p(ids), _p(wts), _p(w13), _p(w2), _p(out), M, H, E,
                                      ids.shape[1], twoI // 2,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_forward(cuda):
    import invariant_moe_gb300 as bm
    lib = bm.load_library()
    H, E, I, k = 2048, 128, 768, 8
    w = syn.moe_weights(H, E, I, seed=71, unit=True)
    w13, w2 = w.w13.to(cuda), w.w2.to(cuda)
    for call, (M, seed) in enumerate(((300, 72), (77, 74))):
        x = syn.moe_tokens(M, H, seed=seed, unit=True).to(cuda)
        ids, wts = syn.random_routing(M, E, k, seed=seed + 1)
        ids, wts = ids.to(cuda), wts.to(cuda)
        ref = bm.bi_moe_forward(x, ids, wts, w13, w2)
        out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=cuda)
        st = _noalloc(lib, x, ids, wts, w13, w2, out)
        assert st == 0, lib.bi_last_error_message()
        torch.cuda.synchronize()
        # the tests' tolerance for this layer is met trivially: same bits
        assert torch.equal(out, ref), f"call {call}: outputs differ"


def test_noalloc_three_launch_permutation_after_larger_call(cuda):
    """Small shapes with more than 1024 tokens take the three-launch
    permutation, whose per-block counts and offsets live in the scratch array.
    A larger call first leaves its leftovers there; the next calls must still
    give bi_moe_forward's bits."""
    import invariant_moe_gb300 as bm
    lib = bm.load_library()
    H, E, I, k = 256, 16, 128, 4
    w = syn.moe_weights(H, E, I, seed=75, unit=True)
    w13, w2 = w.w13.to(cuda), w.w2.to(cuda)
    for call, (M, seed) in enumerate(((3000, 76), (2048, 78), (1100, 80))):
        assert lib.bi_moe_workspace_bytes(M, H, E, k, I) <= 64 << 20
        x = syn.moe_tokens(M, H, seed=seed, unit=True).to(cuda)
        ids, wts = syn.random_routing(M, E, k, seed=seed + 1)
        ids, wts = ids.to(cuda), wts.to(cuda)
        ref = bm.bi_moe_forward(x, ids, wts, w13, w2)
        out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=cuda)
        st = _noalloc(lib, x, ids, wts, w13, w2, out)
        assert st == 0, lib.bi_last_error_message()
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call} (M={M}): outputs differ"


def test_noalloc_python_wrapper(cuda):
    """The binding's wrapper gives the same bits as bi_moe_forward."""
    import invariant_moe_gb300 as bm
    H, E, I, k, M = 512, 32, 256, 8, 200
    w = syn.moe_weights(H, E, I, seed=81, unit=True)
    x = syn.moe_tokens(M, H, seed=82, unit=True).to(cuda)
    ids, wts = syn.random_routing(M, E, k, seed=83)
    ids, wts = ids.to(cuda), wts.to(cuda)
    w13, w2 = w.w13.to(cuda), w.w2.to(cuda)
    ref = bm.bi_moe_forward(x, ids, wts, w13, w2)
    for _ in range(2):
        got = bm.bi_moe_forward_noalloc(x, ids, wts, w13, w2)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)


def test_noalloc_rejects_sizes_beyond_its_array(cuda):
    import invariant_moe_gb300 as bm
    lib = bm.load_library()
    H, E, I, k, M = 2048, 128, 768, 8, 4096   # needs ~453 MB of scratch
    assert lib.bi_moe_workspace_bytes(M, H, E, k, I) > 64 << 20
    x = torch.zeros(M, H, dtype=torch.bfloat16, device=cuda)
    ids, wts = syn.random_routing(M, E, k, seed=3)
    w13 = torch.zeros(E, 2 * I, H, dtype=torch.bfloat16, device=cuda)
    w2 = torch.zeros(E, H, I, dtype=torch.bfloat16, device=cuda)
    out = torch.zeros(M, H, dtype=torch.bfloat16, device=cuda)
    st = _noalloc(lib, x, ids.to(cuda), wts.to(cuda), w13, w2, out)
    assert st == 3  # BI_ERR_WORKSPACE
    assert b"scratch" in lib.bi_last_error_message()
