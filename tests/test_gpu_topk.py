"""Top-k selection on the GPU.  Both sides select on the same fp32 scores, so
the expert ids must match the oracle bit for bit (score descending, ties to
the lowest index); routing weights sigmoid(score) match the fp64 sigmoid to
fp32 rounding."""
import struct

import numpy as np
import pytest
import torch

from tests import synthetic as syn

pytestmark = pytest.mark.gpu


def gpu_topk(scores, k, cuda, want_probs=False):
    import invariant_moe_gb300 as bm
    ids, wts, probs = bm.bi_topk(scores.to(cuda).contiguous(), k, want_probs=want_probs)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), wts.cpu().numpy(), (probs.cpu().numpy() if probs is not None else None)


def check(oracle_mod, scores, k, cuda):
    ids, wts, probs = gpu_topk(scores, k, cuda, want_probs=True)
    ids_o, wts_o = oracle_mod.topk(scores.numpy(), k)
    assert np.array_equal(ids, ids_o)
    fin = np.isfinite(wts_o)
    assert np.all(np.abs(wts[fin] - wts_o[fin]) <= 4e-7 * np.abs(wts_o[fin]) + 1e-30)
    p_o = oracle_mod.sigmoid(scores.numpy())
    pf = np.isfinite(p_o)
    assert np.all(np.abs(probs[pf] - p_o[pf]) <= 4e-7 * np.abs(p_o[pf]) + 1e-30)
    return ids


@pytest.mark.parametrize("E,k", [(256, 8), (128, 8), (100, 3), (512, 16), (33, 1), (8, 8)])
def test_quantised_tie_plateaus(oracle_mod, cuda, E, k):
    s, rows = syn.quantised_scores(M=2048, E=E, frac=0.3, seed=E + k)
    check(oracle_mod, s, k, cuda)


def test_router_tie_construction(oracle_mod, cuda):
    """Duplicated W rows give exact ties in every row (the GEMM computes every
    column with the same arithmetic); both sides must break them by index.
    The oracle selects on its own fp64 scores (from the host inputs) rounded
    to fp32; rows with a near-tie closer than 1e-4 are left out of the id
    comparison (exact ties stay in)."""
    import invariant_moe_gb300 as bm
    inp, _ = syn.router_tie_inputs(M=4096)
    y = bm.bi_router_gemm(inp.x.to(cuda), inp.w.to(cuda), inp.b.to(cuda))
    ids, _, _ = bm.bi_topk(y, 8)
    torch.cuda.synchronize()
    ids = ids.cpu().numpy()
    rows = torch.randperm(4096, generator=syn.gen(6))[:512].numpy()
    r = oracle_mod.router(inp.x[rows].numpy(), inp.w.numpy(), inp.b.numpy())
    ok = syn.unambiguous_rows(r, 8)
    assert len(ok) >= 0.9 * len(rows)
    ids_o, _ = oracle_mod.topk(r.astype(np.float32), 8)
    assert np.array_equal(ids[rows][ok], ids_o[ok])
    # the plateaus are real: duplicated experts score exactly alike
    assert (r[:, None, :] == r[:, :, None]).sum() > len(rows) * 256
    # invariance of the selection over batch sizes
    for M in syn.batch_sizes(4096):
        y_m = bm.bi_router_gemm(inp.x[:M].contiguous().to(cuda), inp.w.to(cuda), inp.b.to(cuda))
        ids_m, _, _ = bm.bi_topk(y_m, 8)
        torch.cuda.synchronize()
        assert np.array_equal(ids_m.cpu().numpy(), ids[:M]), f"M={M}"


def f32(bits):
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def test_special_rows(oracle_mod, cuda):
    E, k = 64, 8
    rows = [
        np.full(E, 0.25, np.float32),
        np.full(E, -np.inf, np.float32),
        np.array([(-0.0 if i % 3 else 0.0) for i in range(E)], np.float32),
        np.arange(E, dtype=np.float32),
        -np.arange(E, dtype=np.float32),
        np.array([f32(1) if i % 2 else f32(0x007FFFFF) for i in range(E)], np.float32),  # denormals
    ]
    nan_row = np.zeros(E, np.float32)
    nan_bits = [0x7FC00000, 0xFFC00000, 0xFFFFFFFF, 0xFFFFFFFE, 0x7F800001, 0x7F800000, 0xFF800000]
    for i, bb in enumerate(nan_bits):
        nan_row[5 * i] = f32(bb)
    rows.append(nan_row)
    s = torch.from_numpy(np.stack(rows))
    ids, _, _ = gpu_topk(s, k, cuda)
    ids_o, _ = oracle_mod.topk(s.numpy(), k)
    assert np.array_equal(ids, ids_o)
    assert list(ids[0]) == list(range(k))
    assert list(ids[1]) == list(range(k))
    assert list(ids[2]) == list(range(k))  # -0.0 ties +0.0


def test_invariance_over_position(cuda):
    g = syn.gen(8)
    E, k = 256, 8
    base, _ = syn.quantised_scores(M=4096, E=E, frac=0.5, seed=9)
    ref, _, _ = gpu_topk(base, k, cuda)
    for B in (1, 17, 300, 4096):
        idx = torch.randperm(4096, generator=g)[:B]
        got, _, _ = gpu_topk(base[idx], k, cuda)
        assert np.array_equal(got, ref[idx.numpy()])


def test_empty(cuda):
    import invariant_moe_gb300 as bm
    ids, wts, _ = bm.bi_topk(torch.empty(0, 256, device=cuda), 8)
    assert ids.shape == (0, 8)
