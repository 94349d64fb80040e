"""Pins for the fp64 CPU oracle (no GPU).

Each test checks the oracle against something other than itself: exact
integer arithmetic, closed forms, a hand-worked example, brute force on tiny
inputs, library routines (numpy matmul / sort) for special cases, and
invariants of the definition.  A dropped term, a wrong sign or index, a
transposed operand or a swapped gate/up half fails at least one of them.
"""
import itertools
import json
import math
import os
import struct

import numpy as np
import pytest
import torch

from tests import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_from_bits(u):
    return struct.unpack("<f", struct.pack("<I", u))[0]


def bf16(a):
    """bf16 bit patterns of a float array (round to nearest even)."""
    return syn.bf16_bits(torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16))


def bf16_val(bits):
    return syn.bits_to_bf16(bits).to(torch.float64).numpy()


# ------------------------------------------------------------------ router --
def test_router_exact_integer_case(oracle_mod):
    """x in multiples of 1/8 (|x|<=2), W in multiples of 1/64 (|W|<=1), b in
    multiples of 1/64: every partial sum is exact in fp64, so the oracle must
    equal the int64 sum bit for bit.  Non-square shapes catch a transposed W."""
    rng = np.random.default_rng(0)
    M, K, N = 5, 4096, 7
    xi = rng.integers(-16, 17, size=(M, K))
    wi = rng.integers(-64, 65, size=(N, K))
    bi = rng.integers(-64, 65, size=N)
    x = (xi / 8.0).astype(np.float32)
    w = (wi / 64.0).astype(np.float32)
    b = (bi / 64.0).astype(np.float32)
    r = oracle_mod.router(x, w, b)
    exact = (xi.astype(np.int64) @ wi.T.astype(np.int64) + 8 * bi[None, :]) / 512.0
    assert np.array_equal(r, exact)
    r0 = oracle_mod.router(x, w, None)
    assert np.array_equal(r0, (xi.astype(np.int64) @ wi.T.astype(np.int64)) / 512.0)


def test_router_one_hot_closed_form(oracle_mod):
    """x = e_j gives y = W[:, j] + b exactly."""
    K, N = 96, 11
    rng = np.random.default_rng(1)
    w = rng.standard_normal((N, K)).astype(np.float32)
    b = rng.standard_normal(N).astype(np.float32)
    for j in (0, 5, K - 1):
        x = np.zeros((1, K), np.float32)
        x[0, j] = 1.0
        r = oracle_mod.router(x, w, b)
        assert np.array_equal(r[0], w[:, j].astype(np.float64) + b.astype(np.float64))


def test_router_invariants(oracle_mod):
    rng = np.random.default_rng(2)
    M, K, N = 9, 256, 13
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = rng.standard_normal((N, K)).astype(np.float32)
    r = oracle_mod.router(x, w)
    # row permutation permutes rows, exactly
    p = rng.permutation(M)
    assert np.array_equal(oracle_mod.router(x[p], w), r[p])
    # duplicated W rows give bit-equal columns
    w2 = w.copy()
    w2[3] = w2[7]
    r2 = oracle_mod.router(x, w2)
    assert np.array_equal(r2[:, 3], r2[:, 7])
    # scaling x by 2 scales y by 2 exactly (no bias)
    assert np.array_equal(oracle_mod.router(2 * x, w), 2 * r)
    # agrees with a library fp64 matmul to fp64 rounding
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    bound = 1e-13 * (np.abs(x).astype(np.float64) @ np.abs(w).astype(np.float64).T)
    assert np.all(np.abs(r - ref) <= bound)


def test_router_within_bound_of_correctly_rounded_sum(oracle_mod):
    """Against math.fsum of the exact products (fp32 x fp32 is exact in fp64):
    the oracle's fp64 sum in increasing k, bias last, stays within the
    recursive-summation bound (K+1) u sum|terms| of the correctly rounded
    sum, at the router's K = 4096."""
    rng = np.random.default_rng(21)
    M, K, N = 3, 4096, 5
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) / 64).astype(np.float32)
    b = (rng.standard_normal(N) * 0.01).astype(np.float32)
    r = oracle_mod.router(x, w, b)
    u = 2.0 ** -53
    for i in range(M):
        for n in range(N):
            terms = [float(x[i, k]) * float(w[n, k]) for k in range(K)] + [float(b[n])]
            exact = math.fsum(terms)
            mag = math.fsum(abs(t) for t in terms)
            assert abs(r[i, n] - exact) <= (K + 1) * u * mag


def test_sigmoid_closed_forms(oracle_mod):
    assert oracle_mod.sigmoid(np.array([0.0]))[0] == 0.5
    v = np.array([-3.5, -1.0, 0.25, 1.0, 2.0, 7.0], np.float32)
    s = oracle_mod.sigmoid(v)
    for vi, si in zip(v, s):
        assert abs(si - 1.0 / (1.0 + math.exp(-float(vi)))) <= 1e-16
    # symmetry sigma(-v) = 1 - sigma(v)
    assert np.allclose(oracle_mod.sigmoid(-v), 1.0 - s, rtol=0, atol=1e-15)


# ------------------------------------------------------------------- top-k --
def test_score_key_page_values(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "topk_key.json")))
    for bits, key in g["bits_to_key"]:
        assert oracle_mod.score_key(f32_from_bits(int(bits, 16))) == key
    for a, b in g["equal_keys"]:
        assert oracle_mod.score_key(f32_from_bits(int(a, 16))) == oracle_mod.score_key(f32_from_bits(int(b, 16)))


def test_score_key_monotone(oracle_mod):
    vals = [-math.inf, -3e38, -1.5, -1e-40, -0.0, 0.0, 1e-45, 1e-40, 1.0, 2.0, 3e38, math.inf]
    keys = [oracle_mod.score_key(v) for v in vals]
    for (va, ka), (vb, kb) in zip(zip(vals, keys), zip(vals[1:], keys[1:])):
        if va == vb:
            assert ka == kb
        else:
            assert ka < kb
    assert oracle_mod.score_key(f32_from_bits(0x7FC00000)) > oracle_mod.score_key(math.inf)
    assert oracle_mod.score_key(f32_from_bits(0xFFC00000)) < oracle_mod.score_key(-math.inf)


def _rank_brute(row, k):
    """Rank of each expert = number of experts that beat it ((value, index)
    order); the selection is the experts of rank < k.  Values only (no NaN)."""
    E = len(row)
    v = [0.0 if x == 0 else x for x in row]
    rank = [sum(1 for f in range(E) if v[f] > v[e] or (v[f] == v[e] and f < e)) for e in range(E)]
    return [e for r in range(k) for e in range(E) if rank[e] == r]


@pytest.mark.parametrize("E,k", [(2, 1), (5, 2), (7, 3), (10, 3), (10, 1)])
def test_topk_brute_force(oracle_mod, E, k):
    rng = np.random.default_rng(E * 10 + k)
    rows = []
    for _ in range(60):
        r = rng.integers(-3, 4, size=E).astype(np.float32) / 2  # many exact ties
        rows.append(r)
    rows.append(np.zeros(E, np.float32))
    rows.append(np.array([(-0.0 if i % 2 else 0.0) for i in range(E)], np.float32))
    rows.append(np.arange(E, dtype=np.float32))
    s = np.stack(rows)
    ids, wts = oracle_mod.topk(s, k)
    for m in range(s.shape[0]):
        exp = _rank_brute(list(s[m]), k)
        assert list(ids[m]) == exp
        # library sort with the (value desc, index asc) order
        srt = sorted(range(E), key=lambda e: (-(0.0 if s[m, e] == 0 else s[m, e]), e))[:k]
        assert list(ids[m]) == srt
        for t in range(k):
            assert wts[m, t] == pytest.approx(1 / (1 + math.exp(-float(s[m, ids[m, t]]))), rel=1e-15)


def test_topk_special_rows(oracle_mod):
    E, k = 256, 8
    ids, _ = oracle_mod.topk(np.full((1, E), 0.3, np.float32), k)
    assert list(ids[0]) == list(range(k))
    ids, _ = oracle_mod.topk(np.arange(E, dtype=np.float32)[None], k)
    assert list(ids[0]) == list(range(E - 1, E - 1 - k, -1))
    ids, _ = oracle_mod.topk(np.full((1, E), -np.inf, np.float32), k)
    assert list(ids[0]) == list(range(k))


def test_topk_relabelling(oracle_mod):
    """Relabelling experts by a permutation pi maps the selection through pi
    when the row has no ties."""
    rng = np.random.default_rng(3)
    E, k = 64, 8
    s = rng.standard_normal((20, E)).astype(np.float32)
    pi = rng.permutation(E)
    s2 = np.empty_like(s)
    s2[:, pi] = s
    a, _ = oracle_mod.topk(s, k)
    b, _ = oracle_mod.topk(s2, k)
    assert np.array_equal(pi[a], b)


# ----------------------------------------------------------------- permute --
def test_permute_matches_stable_sort(oracle_mod):
    M, E, k = 37, 16, 4
    ids, _ = syn.random_routing(M, E, k, seed=5)
    ids = ids.numpy()
    off, perm = oracle_mod.permute(ids, E)
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")
    assert np.array_equal(perm, order.astype(np.int32))
    cnt = np.bincount(flat, minlength=E)
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32))
    with pytest.raises(ValueError):
        oracle_mod.permute(np.array([[0, E]], np.int32), E)


# --------------------------------------------------------------------- MoE --
def test_moe_hand_worked_example(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "moe_two_expert.json")))
    x = np.array([g["x"]], np.float32)
    rw = np.array(g["router_w"], np.float32)
    r = oracle_mod.router(x, rw)
    assert list(r[0]) == g["scores"]
    w13 = bf16(np.array(g["w13"], np.float32))
    w2 = bf16(np.array(g["w2"], np.float32))
    xb = bf16(x)
    for key, k in (("top1", 1), ("top2", 2)):
        ids, wts = oracle_mod.topk(r.astype(np.float32), k)
        assert list(ids[0]) == g[key]["ids"]
        assert wts[0, 0] == pytest.approx(g["probs"]["s2"], rel=1e-15)
        # the router's probability is fp32 on the CUDA path; feed the fp32 value
        out = oracle_mod.moe(xb, ids, wts.astype(np.float32), w13, w2, 2, 1)
        exp = np.array(g[key]["out"])
        # fp32 rounding of the probabilities: relative 2^-24 per factor
        assert np.allclose(out[0], exp, rtol=2e-7, atol=0)
        # with exact fp64 probabilities the closed form holds to fp64 rounding
    # exactness of the formula itself: p = 1 exactly (no rounding anywhere)
    ids = np.array([[1, 0]], np.int32)
    ones = np.ones((1, 2), np.float32)
    out = oracle_mod.moe(xb, ids, ones, w13, w2, 2, 1)
    # expert 1: g=2,u=1 -> a = 2*s2 ; expert 0: g=1,u=2 -> a = 2*s1
    s1, s2 = g["probs"]["s1"], g["probs"]["s2"]
    assert out[0, 0] == pytest.approx(2 * (2 * s2) + (2 * s1), rel=1e-15)
    assert out[0, 1] == pytest.approx((2 * s2) - (2 * s1), rel=1e-15)


def _dense_swiglu(x, wg, wu, wd, p):
    g = x @ wg.T
    u = x @ wu.T
    a = g / (1 + np.exp(-g)) * u * p
    return a @ wd.T


def test_moe_reduces_to_dense_swiglu(oracle_mod):
    """E=1, k=1, p=1 is a dense SwiGLU MLP; checked against numpy fp64 matmuls
    with H != I so transposed or swapped operands fail."""
    rng = np.random.default_rng(4)
    M, H, I = 6, 24, 16
    x = bf16(rng.standard_normal((M, H)))
    w13 = bf16(rng.standard_normal((1, 2 * I, H)) * 0.3)
    w2 = bf16(rng.standard_normal((1, H, I)) * 0.3)
    ids = np.zeros((M, 1), np.int32)
    wts = np.ones((M, 1), np.float32)
    out = oracle_mod.moe(x, ids, wts, w13, w2, 1, I)
    xv, w13v, w2v = bf16_val(x), bf16_val(w13)[0], bf16_val(w2)[0]
    ref = _dense_swiglu(xv, w13v[:I], w13v[I:], w2v, 1.0)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    # the gate half is rows [0,I): swapping halves gives a different answer
    bad = _dense_swiglu(xv, w13v[I:], w13v[:I], w2v, 1.0)
    assert not np.allclose(out, bad, rtol=1e-3, atol=1e-3)


def _small_moe(seed=6, M=7, H=32, E=5, I=16, k=3):
    rng = np.random.default_rng(seed)
    x = bf16(rng.standard_normal((M, H)))
    w13 = bf16(rng.standard_normal((E, 2 * I, H)) * 0.2)
    w2 = bf16(rng.standard_normal((E, H, I)) * 0.2)
    ids, wts = syn.random_routing(M, E, k, seed=seed)
    return x, ids.numpy(), wts.numpy(), w13, w2, E, I


def test_moe_invariants(oracle_mod):
    x, ids, wts, w13, w2, E, I = _small_moe()
    out = oracle_mod.moe(x, ids, wts, w13, w2, E, I)
    # linear in p, exactly (power-of-two scaling)
    assert np.array_equal(oracle_mod.moe(x, ids, 2 * wts, w13, w2, E, I), 2 * out)
    # zero down weights give zero
    assert not np.any(oracle_mod.moe(x, ids, wts, w13, np.zeros_like(w2), E, I))
    # consistent relabelling of experts leaves the output unchanged
    pi = np.random.default_rng(9).permutation(E)
    w13p = np.empty_like(w13)
    w2p = np.empty_like(w2)
    w13p[pi] = w13
    w2p[pi] = w2
    assert np.array_equal(oracle_mod.moe(x, pi[ids].astype(np.int32), wts, w13p, w2p, E, I), out)
    # token permutation permutes the rows
    q = np.random.default_rng(10).permutation(x.shape[0])
    assert np.array_equal(oracle_mod.moe(x[q], ids[q], wts[q], w13, w2, E, I), out[q])
    # each slot contributes: the sum over single-slot layers equals the layer
    parts = sum(oracle_mod.moe(x, ids[:, t:t + 1], wts[:, t:t + 1], w13, w2, E, I)
                for t in range(ids.shape[1]))
    assert np.allclose(parts, out, rtol=1e-13, atol=1e-15)


def test_stage_oracles_compose(oracle_mod):
    """permute -> gate_up -> down -> combine equals the full layer (up to the
    bf16/fp32 storage of the intermediate activations and contributions)."""
    x, ids, wts, w13, w2, E, I = _small_moe(seed=8, M=11)
    M, H = x.shape
    k = ids.shape[1]
    off, perm = oracle_mod.permute(ids, E)
    act = oracle_mod.gate_up(x, off, perm, wts, w13, E, k, I)
    # gate_up agrees with per-pair dense evaluation
    xv, w13v = bf16_val(x), bf16_val(w13)
    for p in range(off[E]):
        e = int(np.searchsorted(off, p, side="right") - 1)
        pair = perm[p]
        g = xv[pair // k] @ w13v[e, :I].T
        u = xv[pair // k] @ w13v[e, I:].T
        assert np.allclose(act[p], g / (1 + np.exp(-g)) * u * wts.reshape(-1)[pair], rtol=1e-12, atol=1e-14)
    contrib = oracle_mod.down(bf16(act), off, perm, w2, M, H, E, k, I)
    out = oracle_mod.combine(contrib.astype(np.float32), k)
    ref = oracle_mod.moe(x, ids, wts, w13, w2, E, I)
    # contributions land at row token*k + slot
    c_direct = np.zeros_like(contrib)
    c_abs = np.zeros_like(contrib)
    w2v = bf16_val(w2)
    av = bf16_val(bf16(act))
    for p in range(off[E]):
        e = int(np.searchsorted(off, p, side="right") - 1)
        c_direct[perm[p]] = av[p] @ w2v[e].T
        c_abs[perm[p]] = np.abs(act[p]) @ np.abs(w2v[e]).T
    assert np.allclose(contrib, c_direct, rtol=1e-12, atol=1e-15)
    # bf16 storage of act (relative 2^-9) and fp32 storage of contrib
    # (relative 2^-24) bound the difference term by term
    bound = 2.0 ** -9 * c_abs.reshape(M, k, H).sum(1) + 2.0 ** -23 * np.abs(c_direct).reshape(M, k, H).sum(1)
    assert np.all(np.abs(out - ref) <= bound * 1.0001)


def test_combine_is_slot_sum(oracle_mod):
    rng = np.random.default_rng(12)
    M, k, H = 4, 8, 10
    c = rng.standard_normal((M * k, H)).astype(np.float32)
    out = oracle_mod.combine(c, k)
    assert np.allclose(out, c.astype(np.float64).reshape(M, k, H).sum(axis=1), rtol=1e-14, atol=1e-14)


# ------------------------------------------------------- windowed top-k --
# The sparse-MLA indexer's per-row top-k ("[BI][DSv4] Pin sparse-MLA decode
# and prefill scheduling under batch invariance", commit log).  For rows with
# no NaN the rank (key desc, column asc) is numpy's stable argsort of the
# negated values, since the monotone key orders non-NaN floats numerically
# and makes -0.0 equal to +0.0.
def f32_bits(bits):
    return np.array(bits, dtype=np.uint32).view(np.float32)


def stable_topk_ref(row, k):
    """Chosen columns, ascending, by numpy's stable sort of -value."""
    order = np.argsort(-row.astype(np.float64), kind="stable")[:k]
    return np.sort(order)


@pytest.mark.parametrize("k", [1, 7, 512])
def test_topk_window_matches_stable_sort(oracle_mod, k):
    rng = np.random.default_rng(k)
    for trial in range(40):
        width = int(rng.integers(1, 1400))
        row = rng.normal(size=width).astype(np.float32)
        if trial % 2:   # quantised values: tie plateaus at the cutoff
            row = np.round(row * 4) / 4
        if trial % 3 == 0:   # relu plateaus of exact zeros, both signs
            row = np.maximum(row, 0) * np.where(rng.random(width) < 0.5, -1, 1).astype(np.float32)
        rs = int(rng.integers(0, width))
        re = int(rng.integers(rs, width + 1))
        got = oracle_mod.topk_window(row[None], k, [rs], [re])[0]
        ref = stable_topk_ref(row[rs:re], k)
        assert np.array_equal(got[: len(ref)], ref)
        assert np.all(got[len(ref):] == -1)


def test_topk_window_closed_forms(oracle_mod):
    k = 512
    # all-equal and all -inf rows: the first k columns of the window
    for v in (0.5, -np.inf, 0.0):
        out = oracle_mod.topk_window(np.full((1, 3000), v, np.float32), k, [100], [2900])[0]
        assert np.array_equal(out, np.arange(k))
    # window narrower than k: all of it, then -1
    out = oracle_mod.topk_window(np.random.default_rng(1).normal(size=(1, 630)).astype(np.float32),
                                 k, [5], [35])[0]
    assert np.array_equal(out[:30], np.arange(30)) and np.all(out[30:] == -1)
    # empty windows
    for rs, re in ((10, 10), (20, 3), (700, 800)):
        out = oracle_mod.topk_window(np.ones((1, 630), np.float32), 4, [rs], [re])[0]
        assert np.all(out == -1)


def test_topk_window_shift_invariance(oracle_mod):
    """The same logical row at six window offsets selects the same local
    indices, whatever the masked lanes around it hold (the masked-lane fix)."""
    rng = np.random.default_rng(5)
    logical = np.round(rng.normal(size=600) * 2).astype(np.float32) / 2
    logical[::7] = -np.inf
    base = None
    for off in (0, 1, 17, 100, 511, 1400):
        buf = np.full((1, 2100), np.inf, np.float32)   # out-of-window lanes would win on score
        buf[0, off:off + 600] = logical
        out = oracle_mod.topk_window(buf, 512, [off], [off + 600])[0]
        base = out if base is None else base
        assert np.array_equal(out, base), off
    assert np.array_equal(base, stable_topk_ref(logical, 512))


def test_topk_window_signed_zero_and_nan_patterns(oracle_mod):
    # -0.0 ties +0.0: the lower column wins
    row = np.array([-0.0, 0.0, -1.0], np.float32)
    assert list(oracle_mod.topk_window(row[None], 1)[0]) == [0]
    row = np.array([-1.0, 0.0, -0.0], np.float32)
    assert list(oracle_mod.topk_window(row[None], 1)[0]) == [1]
    # the two sentinel-adjacent negative NaNs are distinct keys: 0xfffffffe
    # (INT32_MIN + 1) ranks above 0xffffffff (INT32_MIN)
    row = f32_bits([0xFFFFFFFF, 0xFFFFFFFE, 0xFFFFFFFF])
    assert list(oracle_mod.topk_window(row[None], 1)[0]) == [1]
    # validity first: a window of 30 negative NaNs inside a wider row never
    # gives up a slot to an out-of-window lane, whatever that lane holds
    row = np.concatenate([np.full(300, np.inf, np.float32), f32_bits([0xFFFFFFFF] * 30),
                          np.full(300, np.inf, np.float32)])
    out = oracle_mod.topk_window(row[None], 512, [300], [330])[0]
    assert np.array_equal(out[:30], np.arange(30)) and np.all(out[30:] == -1)
    # the class ladder: +NaN > +inf > max > min denormal > +0 = -0 > -min denormal > -inf > -NaN
    ladder = f32_bits([0xFF800000, 0x00000001, 0x7FC00000, 0x80000000, 0x7F800000,
                       0x80000001, 0xFFC00000, 0x7F7FFFFF, 0x00000000])
    ranked = [int(c) for c in oracle_mod.topk_window(ladder[None], 9)[0]]
    assert ranked == list(range(9))   # all chosen, ascending
    # top-1 is +NaN (col 2), top-2 adds +inf (col 4), top-3 adds max normal (col 7)
    assert [oracle_mod.topk_window(ladder[None], j)[0].tolist() for j in (1, 2, 3)] == \
        [[2], [2, 4], [2, 4, 7]]


def test_topk_window_bounds_and_stride(oracle_mod):
    rng = np.random.default_rng(9)
    buf = rng.normal(size=(3, 1000)).astype(np.float32)
    # bounds clamp to [0, num_cols]: negative start, end past the end, past int32
    out = oracle_mod.topk_window(buf, 8, [-50, 0, -(2 ** 40)], [2000, 2 ** 40, 2 ** 41], num_cols=900)
    for i in range(3):
        assert np.array_equal(out[i], stable_topk_ref(buf[i, :900], 8))
    # columns past num_cols (row padding) are never chosen even if they would win
    buf[:, 900:] = np.inf
    out2 = oracle_mod.topk_window(buf, 8, None, None, num_cols=900)
    assert np.array_equal(out2, out)
