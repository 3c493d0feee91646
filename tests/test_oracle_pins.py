"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: hand-derived
bytes, closed forms, invariants, brute force, or a library routine (numpy /
torch float64) on inputs where the method reduces to it.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle as orc
from conftest import parse_golden

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_hand.txt")
CASES = parse_golden(GOLDEN)


def f32_bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


# ---------------------------------------------------------------------------
# quantiser: hand-derived bytes (quant_int4_grouped, section 权重转换)

@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_quant_hand_vectors(case):
    w = np.array(case["w"], np.float32)
    assert w.shape[1] == case["cols"]
    packed, scales = orc.quant_i4g(w)
    assert packed.tolist() == case["bytes"]
    assert f32_bits(scales).tolist() == case["scales"]


def test_quant_f32_division_differs_from_f64():
    # The f32_division fixture only pins something if an f64 division would give
    # other bytes: check that premise with exact rational arithmetic.
    from fractions import Fraction
    s = np.float32(3.0) / np.float32(7.0)
    exact = Fraction(1.5) / Fraction(float(s))
    assert exact < Fraction(7, 2)           # exact quotient is below 3.5 ...
    assert np.float32(1.5) / s == np.float32(3.5)  # ... but rounds to 3.5 in f32


def _random_weights(rows, cols, seed, outliers=True):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    if outliers:
        pos = rng.choice(w.size, max(1, w.size // 100), replace=False)
        w.reshape(-1)[pos] *= 20
    # bf16 values, widened exactly (the workloads' weight dtype)
    return torch.from_numpy(w).to(torch.bfloat16).float().numpy()


def _nibbles(packed, cols):
    lo = packed & 0x0F
    hi = packed >> 4
    u = np.empty((packed.shape[0], packed.shape[1] * 2), np.int64)
    u[:, 0::2] = lo
    u[:, 1::2] = hi
    return u[:, :cols]


@pytest.mark.parametrize("rows,cols", [(3, 64), (5, 200), (7, 333), (16, 1024)])
def test_quant_invariants(rows, cols):
    w = _random_weights(rows, cols, seed=rows * 1000 + cols)
    w[0, :min(cols, 64)] = 0.0                   # one all-zero group
    packed, scales = orc.quant_i4g(w)
    u = _nibbles(packed, cols)
    ng = (cols + 63) // 64
    s_full = np.repeat(scales, 64, axis=1)[:, :cols].astype(np.float64)
    # u in [1, 15]: with s = max|w|/7 the clip at -8 never fires
    assert u.min() >= 1 and u.max() <= 15
    # |w - s (u - 8)| <= s/2 (1 + 2^-19): rint error plus one f32 rounding of w/s
    err = np.abs(w.astype(np.float64) - s_full * (u - 8))
    assert np.all(err <= s_full / 2 * (1 + 2.0 ** -19))
    for r in range(rows):
        for g in range(ng):
            seg = u[r, 64 * g:64 * (g + 1)]
            m = np.abs(w[r, 64 * g:64 * (g + 1)]).max()
            if m == 0:
                assert scales[r, g] == 0 and np.all(seg == 8)
            else:
                # the element(s) holding the max reach |q| = 7
                assert np.abs(seg - 8).max() == 7
                assert scales[r, g] == np.float32(m) / np.float32(7)
    if cols % 2:
        assert np.all(packed[:, -1] >> 4 == 0)


def _on_grid(rows, cols, seed):
    """Weights w = s q with s a power of two and q in [-7, 7], |q| = 7 in every group.

    For these the quantiser is exactly invertible: s' = 7s/7 = s and w/s = q.
    """
    rng = np.random.default_rng(seed)
    ng = (cols + 63) // 64
    q = rng.integers(-7, 8, size=(rows, cols))
    for g in range(ng):
        c = 64 * g + rng.integers(0, min(64, cols - 64 * g), size=rows)
        q[np.arange(rows), c] = rng.choice([-7, 7], size=rows)
    e = rng.integers(-9, -3, size=(rows, ng))
    s = np.ldexp(1.0, e)
    w = (np.repeat(s, 64, axis=1)[:, :cols] * q).astype(np.float32)
    return w


@pytest.mark.parametrize("rows,cols", [(4, 64), (9, 192), (6, 130)])
def test_dequant_matvec_on_grid(rows, cols):
    w = _on_grid(rows, cols, seed=rows + cols)
    packed, scales = orc.quant_i4g(w)
    wd = orc.dequant_i4g(packed, scales, cols)
    assert np.array_equal(wd, w.astype(np.float64))
    x = np.random.default_rng(1).standard_normal(cols)
    y = orc.matvec_i4g(packed, scales, cols, x)
    ref = w.astype(np.float64) @ x                 # library routine
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# router and top-k

def test_router_logits_matmul():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 40))
    wr = rng.standard_normal((6, 40))
    np.testing.assert_allclose(orc.router_logits(x, wr), x @ wr.T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("E,k", [(8, 2), (16, 5), (12, 12), (64, 8)])
def test_topk_brute_force(E, k):
    rng = np.random.default_rng(E * 31 + k)
    for _ in range(20):
        logits = rng.standard_normal(E) * 2
        idx, gates, nan = orc.topk(logits, k)
        assert not nan
        order = sorted(range(E), key=lambda e: (-logits[e], e))[:k]
        assert idx.tolist() == order
        p = np.exp(logits - logits.max())
        p /= p.sum()                                  # softmax over all E ...
        ref = p[order] / p[order].sum()               # ... renormalised over the k
        np.testing.assert_allclose(gates, ref, rtol=1e-12)
        assert abs(gates.sum() - 1) < 1e-12
        assert np.all(np.diff(gates) <= 0)


def test_topk_ties_lower_id_first():
    logits = np.array([0.5, 1.0, 1.0, 0.5, 1.0, -3.0])
    idx, gates, _ = orc.topk(logits, 4)
    assert idx.tolist() == [1, 2, 4, 0]
    np.testing.assert_allclose(gates[:3], gates[0])


def test_topk_equal_logits_k_equals_E():
    idx, gates, _ = orc.topk(np.zeros(8), 8)
    assert idx.tolist() == list(range(8))
    np.testing.assert_allclose(gates, 1 / 8)


def test_topk_nan_rules():
    # every logit NaN: slot j takes expert j, gates 1/k (rt_router_pick fallback)
    idx, gates, nan = orc.topk(np.full(6, np.nan), 3)
    assert nan and idx.tolist() == [0, 1, 2]
    np.testing.assert_allclose(gates, 1 / 3)
    # some NaN: they rank below every number and get gate 0 if picked
    lg = np.array([np.nan, 0.2, np.nan, 1.0])
    idx, gates, nan = orc.topk(lg, 3)
    assert nan and idx.tolist() == [3, 1, 0]
    assert gates[2] == 0
    np.testing.assert_allclose(gates[:2].sum(), 1.0)


# ---------------------------------------------------------------------------
# expert FFN and the layer

def _expert_grid(H, F, seed):
    wg = _on_grid(F, H, seed)
    wu = _on_grid(F, H, seed + 1)
    wd = _on_grid(H, F, seed + 2)
    parts = [orc.quant_i4g(m) for m in (wg, wu, wd)]
    packed = np.concatenate([p.reshape(-1) for p, _ in parts])
    scales = np.concatenate([s.reshape(-1) for _, s in parts])
    assert packed.size == orc.expert_packed_bytes(H, F)
    assert scales.size == orc.expert_scales(H, F)
    return packed, scales, (wg, wu, wd)


def _torch_expert(mats, x):
    wg, wu, wd = (torch.from_numpy(m.astype(np.float64)) for m in mats)
    xt = torch.from_numpy(np.asarray(x, np.float64))
    return (wd @ (Fn.silu(wg @ xt) * (wu @ xt))).numpy()


@pytest.mark.parametrize("H,F", [(64, 128), (192, 64), (128, 320)])
def test_expert_swiglu_on_grid(H, F):
    packed, scales, mats = _expert_grid(H, F, seed=H + F)
    x = np.random.default_rng(2).standard_normal(H)
    y = orc.expert(packed, scales, H, F, x)
    np.testing.assert_allclose(y, _torch_expert(mats, x), rtol=1e-10, atol=1e-12)


def _layer(H, F, E, S, seed):
    ps, ss, mats = [], [], []
    for e in range(E + S):
        p, s, m = _expert_grid(H, F, seed + 10 * e)
        ps.append(p)
        ss.append(s)
        mats.append(m)
    return np.concatenate(ps), np.concatenate(ss), mats


@pytest.mark.parametrize("E,S,k", [(8, 1, 2), (6, 0, 3), (5, 2, 1)])
def test_moe_dense_masked(E, S, k):
    H, F, T = 64, 128, 5
    packed, scales, mats = _layer(H, F, E, S, seed=E * 7 + k)
    rng = np.random.default_rng(11)
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) / 8
    counts = np.zeros(E, np.uint32)
    out, idx, gates, nan = orc.moe_forward(x, wr, packed, scales, H, F, E, S, k, counts)
    assert nan == 0
    # dense reference: every expert on every token, masked by the brute-force top-k
    logits = x @ wr.T
    ref = np.zeros((T, H))
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        p = np.exp(logits[t] - logits[t].max())
        w = np.zeros(E)
        w[order] = p[order] / p[order].sum()
        for e in range(E):
            ref[t] += w[e] * _torch_expert(mats[e], x[t])
        for s in range(S):
            ref[t] += _torch_expert(mats[E + s], x[t])
        assert idx[t].tolist() == order
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-10)
    hist = np.bincount(idx.reshape(-1), minlength=E)
    assert counts.tolist() == hist.tolist() and counts.sum() == T * k


def test_moe_k1_single_ffn_and_counts_accumulate():
    H, F, E, T = 64, 64, 4, 3
    packed, scales, mats = _layer(H, F, E, 0, seed=5)
    x = np.random.default_rng(4).standard_normal((T, H))
    wr = np.random.default_rng(5).standard_normal((E, H))
    counts = np.zeros(E, np.uint32)
    out, idx, gates, _ = orc.moe_forward(x, wr, packed, scales, H, F, E, 0, 1, counts)
    assert np.all(gates == 1.0)
    for t in range(T):
        np.testing.assert_allclose(out[t], _torch_expert(mats[idx[t, 0]], x[t]), rtol=1e-10)
    orc.moe_forward(x, wr, packed, scales, H, F, E, 0, 1, counts)
    assert counts.sum() == 2 * T                      # counts accumulate across calls


def test_moe_k_equals_E_equal_logits_is_mean():
    H, F, E = 64, 64, 4
    packed, scales, mats = _layer(H, F, E, 0, seed=9)
    x = np.random.default_rng(6).standard_normal((2, H))
    out, idx, gates, _ = orc.moe_forward(x, np.zeros((E, H)), packed, scales, H, F, E, 0, E)
    for t in range(2):
        mean = np.mean([_torch_expert(mats[e], x[t]) for e in range(E)], axis=0)
        np.testing.assert_allclose(out[t], mean, rtol=1e-10, atol=1e-12)


def test_stack_residual_chain():
    H, F, E, k = 64, 64, 4, 2
    layers = []
    for l in range(2):
        p, s, _ = _layer(H, F, E, 1, seed=100 + 50 * l)
        layers.append((np.random.default_rng(l).standard_normal((E, H)) / 8, p, s))
    x0 = np.random.default_rng(7).standard_normal((1, H))
    counts = np.zeros((2, E), np.uint32)
    xL, outs, idxs = orc.moe_stack_forward(x0, layers, H, F, E, 1, k, counts)
    o0, _, _, _ = orc.moe_forward(x0, *layers[0], H, F, E, 1, k)
    o1, _, _, _ = orc.moe_forward(x0 + o0, *layers[1], H, F, E, 1, k)
    np.testing.assert_array_equal(xL, x0 + o0 + o1)
    assert counts.sum() == 2 * k


# ---------------------------------------------------------------------------
# the GLM router: sigmoid scores, selection-only bias, normalised gates

def test_topk_sigmoid_hand_example():
    # logits 0, ln 3, -ln 3, ln 9 have sigmoid scores 1/2, 3/4, 1/4, 9/10 exactly
    lg = np.array([0.0, np.log(3.0), -np.log(3.0), np.log(9.0)])
    # no bias: the two largest scores, 9/10 and 3/4; gates 0.9/1.65 = 6/11, 5/11
    idx, gates, nan = orc.topk_sigmoid(lg, 2)
    assert not nan and idx.tolist() == [3, 1]
    np.testing.assert_allclose(gates, [6 / 11, 5 / 11], rtol=1e-14)
    # a bias of 0.8 on expert 2 lifts its key to 1.05 (first) and pushes expert
    # 1 out; the gates still use the scores alone: 1/4 and 9/10 over 23/20
    idx, gates, nan = orc.topk_sigmoid(lg, 2, np.array([0.0, 0.0, 0.8, 0.0]))
    assert idx.tolist() == [2, 3]
    np.testing.assert_allclose(gates, [5 / 23, 18 / 23], rtol=1e-14)


def test_topk_sigmoid_zero_bias_picks_like_softmax():
    # the sigmoid is increasing: without bias the picks equal the softmax ones
    rng = np.random.default_rng(21)
    for E, k in ((8, 2), (64, 8), (256, 8)):
        for _ in range(5):
            lg = rng.standard_normal(E) * 2
            i_soft, _, _ = orc.topk(lg, k)
            i_sig, g_sig, _ = orc.topk_sigmoid(lg, k)
            assert i_sig.tolist() == i_soft.tolist()
            assert abs(g_sig.sum() - 1) < 1e-12 and np.all(g_sig > 0)


def test_topk_sigmoid_common_bias_shift_changes_nothing():
    rng = np.random.default_rng(22)
    lg = rng.standard_normal(32)
    b = rng.standard_normal(32) * 0.1
    i0, g0, _ = orc.topk_sigmoid(lg, 4, b)
    i1, g1, _ = orc.topk_sigmoid(lg, 4, b + 0.25)
    assert i0.tolist() == i1.tolist()
    np.testing.assert_allclose(g0, g1, rtol=1e-14)


def test_topk_sigmoid_brute_force():
    rng = np.random.default_rng(23)
    for E, k in ((8, 3), (48, 6)):
        for _ in range(10):
            lg = rng.standard_normal(E) * 2
            b = rng.standard_normal(E) * 0.2
            s = 1 / (1 + np.exp(-lg))
            order = sorted(range(E), key=lambda e: (-np.float32(s[e] + b[e]), e))[:k]
            idx, gates, _ = orc.topk_sigmoid(lg, k, b)
            assert idx.tolist() == order
            np.testing.assert_allclose(gates, s[order] / s[order].sum(), rtol=1e-12)


def test_topk_sigmoid_nan_rules():
    idx, gates, nan = orc.topk_sigmoid(np.full(5, np.nan), 2, np.zeros(5))
    assert nan and idx.tolist() == [0, 1]
    np.testing.assert_allclose(gates, 0.5)
    lg = np.array([np.nan, 0.0, 1.0])
    idx, gates, nan = orc.topk_sigmoid(lg, 3)
    assert nan and idx.tolist() == [2, 1, 0] and gates[2] == 0
    np.testing.assert_allclose(gates[:2].sum(), 1.0)


def test_moe_sigmoid_router_dense_masked():
    H, F, E, S, k, T = 64, 64, 6, 1, 2, 4
    packed, scales, mats = _layer(H, F, E, S, seed=77)
    rng = np.random.default_rng(12)
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) / 8
    b = rng.standard_normal(E) * 0.3
    out, idx, gates, nan = orc.moe_forward(x, wr, packed, scales, H, F, E, S, k,
                                           router="sigmoid", bias=b)
    assert nan == 0
    logits = x @ wr.T
    for t in range(T):
        s = 1 / (1 + np.exp(-logits[t]))
        order = sorted(range(E), key=lambda e: (-np.float32(s[e] + b[e]), e))[:k]
        assert idx[t].tolist() == order
        ref = sum(s[e] / s[order].sum() * _torch_expert(mats[e], x[t]) for e in order)
        ref = ref + _torch_expert(mats[E], x[t])
        np.testing.assert_allclose(out[t], ref, rtol=1e-10, atol=1e-10)


# ---------------------------------------------------------------------------
# the OpenMP build of the oracle (the benchmark's multi-core leg, large test
# cases) must give the single-threaded build's bits


def test_openmp_build_gives_the_same_bits():
    rng = np.random.default_rng(11)
    H, F, E, S, k, T = 128, 192, 6, 1, 2, 9
    w = (rng.standard_normal((37, 320)) * 0.02).astype(np.float32)
    mats = [(rng.standard_normal(s) * 0.02).astype(np.float32)
            for _ in range(E + S) for s in ((F, H), (F, H), (H, F))]
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) / np.sqrt(H)

    def run():
        p, s = orc.quant_i4g(w)
        qs = [orc.quant_i4g(m) for m in mats]
        packed = np.concatenate([q[0].reshape(-1) for q in qs])
        scales = np.concatenate([q[1].reshape(-1) for q in qs])
        counts = np.zeros(E, np.uint32)
        out, idx, gates, _ = orc.moe_forward(x, wr, packed, scales, H, F, E, S, k, counts)
        return p, s, out, idx, gates, counts

    prev = orc.set_threads(1)
    try:
        serial = run()
        orc.set_threads(4)
        par = run()
    finally:
        orc.set_threads(prev)
    for a, b in zip(serial, par):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))
