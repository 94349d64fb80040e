"""Windowed per-row top-k (bi_topk_window) on the GPU, bit-exact against the
oracle (integer work: every emitted index must match)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

KS = (512, 1024, 2048)


def f32_bits(bits):
    return np.array(bits, dtype=np.uint32).view(np.float32)


def run(bm, cuda, scores, k, rs=None, re=None, num_cols=None):
    s = torch.from_numpy(np.ascontiguousarray(scores)).to(cuda)
    if num_cols is not None:
        s = s[:, :num_cols] if s.shape[1] > num_cols else s
    rs_t = None if rs is None else torch.tensor(rs, dtype=torch.int64, device=cuda)
    re_t = None if re is None else torch.tensor(re, dtype=torch.int64, device=cuda)
    out = bm.bi_topk_window(s, k, rs_t, re_t, num_cols=num_cols)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def random_rows(rng, n, width, kind):
    x = rng.normal(size=(n, width)).astype(np.float32)
    if kind == "quant":
        x = np.round(x * 4) / 4
    elif kind == "relu":   # DSA-style relu(q.k) scores: exact-zero plateaus of both signs
        x = np.maximum(x, 0) * np.where(rng.random((n, width)) < 0.5, -1, 1).astype(np.float32)
    elif kind == "denorm":
        x = (x * 1e-39).astype(np.float32)
    elif kind == "ninf":
        x[rng.random((n, width)) < 0.3] = -np.inf
    return x


@pytest.mark.parametrize("k", KS)
@pytest.mark.parametrize("kind", ["normal", "quant", "relu", "denorm", "ninf"])
def test_random_rows_and_windows(oracle_mod, cuda, k, kind):
    import invariant_moe_gb300 as bm
    rng = np.random.default_rng(k + len(kind))
    n, width = 64, 8192
    x = random_rows(rng, n, width, kind)
    rs = rng.integers(0, width, size=n)
    re = rs + rng.integers(0, width, size=n)
    rs[:4] = [0, 0, 100, 8000]            # full row, full row, interior, narrow tail window
    re[:4] = [width, width + 5, 100 + k - 1, 8192]
    got = run(bm, cuda, x, k, rs.tolist(), re.tolist())
    ref = oracle_mod.topk_window(x, k, rs, re)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("k", KS)
def test_bit_pattern_classes(oracle_mod, cuda, k):
    """Signed zeros, infinities, quiet and signalling NaNs of both signs, the
    smallest and largest denormals and the two sentinel-adjacent negative NaNs,
    in three window shapes, with the selection truncating inside each class."""
    import invariant_moe_gb300 as bm
    classes = [0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000,
               0x7F800001, 0xFF800001, 0x00000001, 0x807FFFFF, 0x007FFFFF, 0x80000001,
               0xFFFFFFFF, 0xFFFFFFFE, 0x3F800000, 0xBF800000]
    rng = np.random.default_rng(k)
    rows, rss, res = [], [], []
    for shape in ("window<k", "wide", "truncating"):
        for cls in range(len(classes)):
            bits = rng.choice(classes, size=8192)
            bits[rng.random(8192) < 0.5] = classes[cls]   # a plateau of one class
            rows.append(bits)
            if shape == "window<k":
                rss.append(1); res.append(31)
            elif shape == "wide":
                rss.append(3); res.append(8190)
            else:
                rss.append(100); res.append(100 + 2600)
    x = f32_bits(np.stack(rows))
    got = run(bm, cuda, x, k, rss, res)
    ref = oracle_mod.topk_window(x, k, rss, res)
    assert np.array_equal(got, ref)


def test_negative_nan_plateau_and_validity_first(oracle_mod, cuda):
    """600 in-window negative NaNs (0xffffffff, the lowest key) at row_start=1
    give 512 indices; out-of-window lanes (+inf) never take a slot."""
    import invariant_moe_gb300 as bm
    x = np.full((1, 1024), np.inf, np.float32)
    x[0, 1:601] = f32_bits([0xFFFFFFFF] * 600)
    got = run(bm, cuda, x, 512, [1], [601])
    assert np.array_equal(got[0], np.arange(512))
    x2 = np.full((1, 630), np.inf, np.float32)
    x2[0, 100:130] = f32_bits([0xFFFFFFFF, 0xFFFFFFFE] * 15)
    got2 = run(bm, cuda, x2, 512, [100], [130])
    assert np.array_equal(got2, oracle_mod.topk_window(x2, 512, [100], [130]))
    assert np.array_equal(got2[0, :30], np.arange(30)) and np.all(got2[0, 30:] == -1)


def test_shift_invariance(cuda):
    """The same logical row at six window offsets selects the same local
    indices (the masked-lane fix), whatever surrounds the window."""
    import invariant_moe_gb300 as bm
    rng = np.random.default_rng(3)
    logical = np.round(rng.normal(size=3000) * 2).astype(np.float32) / 2
    outs = []
    for off in (0, 1, 17, 100, 511, 5000):
        buf = np.full((1, 8192), np.inf, np.float32)
        buf[0, off:off + 3000] = logical
        outs.append(run(bm, cuda, buf, 1024, [off], [off + 3000])[0])
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_strided_rows_and_int64_bounds(oracle_mod, cuda):
    """Row stride wider than num_cols (padding columns hold +inf and are never
    chosen); bounds beyond the int32 range clamp to [0, num_cols]."""
    import invariant_moe_gb300 as bm
    rng = np.random.default_rng(4)
    buf = rng.normal(size=(5, 7000)).astype(np.float32)
    buf[:, 6000:] = np.inf
    rs = [-(2 ** 40), 0, 10, 2 ** 33, -5]
    re = [2 ** 41, 6000, 2 ** 40, 2 ** 34, 3]
    got = run(bm, cuda, buf, 512, rs, re, num_cols=6000)
    ref = oracle_mod.topk_window(buf, 512, rs, re, num_cols=6000)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("num_cols", [1, 511, 512, 513, 8191, 8192])
def test_column_count_edges(oracle_mod, cuda, num_cols):
    import invariant_moe_gb300 as bm
    rng = np.random.default_rng(num_cols)
    x = np.round(rng.normal(size=(3, num_cols)) * 3).astype(np.float32)
    for k in (1, 512, 2048):
        got = run(bm, cuda, x, k)
        assert np.array_equal(got, oracle_mod.topk_window(x, k)), k


def test_rows_invariant_over_batch(cuda):
    """A row's output does not depend on the other rows of the launch."""
    import invariant_moe_gb300 as bm
    rng = np.random.default_rng(6)
    x = random_rows(rng, 64, 8192, "relu")
    rs = rng.integers(0, 4000, size=64)
    re = rs + 3000
    full = run(bm, cuda, x, 2048, rs.tolist(), re.tolist())
    for i in (0, 17, 63):
        solo = run(bm, cuda, x[i:i + 1], 2048, [int(rs[i])], [int(re[i])])
        assert np.array_equal(solo[0], full[i])


def test_empty_batch_and_whole_rows(cuda):
    import invariant_moe_gb300 as bm
    out = bm.bi_topk_window(torch.empty(0, 100, device=cuda), 512)
    assert out.shape == (0, 512)
