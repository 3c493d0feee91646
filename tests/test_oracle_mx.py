"""Pins of the oracle's MXFP4 container (fmt 7 of the engine's format
registry) against the OCP Microscaling definition: hand-derived bytes, the
E2M1 value table, round trips of on-grid weights, error bounds, and the layer
reduced to a textbook SwiGLU on the decoded weights."""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle as orc
from conftest import parse_golden

CASES = parse_golden(os.path.join(os.path.dirname(__file__), "golden", "mxfp4_hand.txt"))
MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_hand_vectors(case):
    w = np.array(case["w"], np.float32)
    assert w.shape[1] == case["cols"]
    p, s = orc.quant_mxfp4(w)
    assert p.tolist() == case["bytes"]
    assert s.tolist() == case["scales"]


def test_e2m1_table():
    # E2M1: bias 1; exponent 0 is subnormal (0, 0.5); sign in bit 3
    for c in range(16):
        e, m = (c >> 1) & 3, c & 1
        mag = m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
        assert orc.e2m1_value(c) == (-mag if c & 8 else mag)
    assert [orc.e2m1_value(c) for c in range(8)] == MAGS


def test_on_grid_round_trip():
    # every block: an element at +-6 * X fixes the shared exponent, the rest on
    # the E2M1 grid of that X; quantise -> the same values exactly
    rng = np.random.default_rng(3)
    rows, cols = 16, 96
    se = rng.integers(-20, 10, size=(rows, cols // 32))
    codes = rng.integers(0, 16, size=(rows, cols))
    codes[:, ::32] = 7                       # 6 X in each block
    vals = np.array([orc.e2m1_value(c) for c in range(16)])[codes]
    w = (vals * np.exp2(np.repeat(se, 32, axis=1))).astype(np.float32)
    p, s = orc.quant_mxfp4(w)
    assert np.array_equal(s.astype(int) - 127, se)
    assert np.array_equal(orc.dequant_mxfp4(p, s, cols), w.astype(np.float64))


def test_error_bound_and_saturation():
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((32, 128)) * 0.02).astype(np.float32)
    p, s = orc.quant_mxfp4(w)
    d = orc.dequant_mxfp4(p, s, 128)
    X = np.repeat(np.exp2(s.astype(np.float64) - 127), 32, axis=1)
    q = np.abs(w) / X                             # in [0, 8)
    assert q.max() < 8
    # below 6 the error is at most half the grid step at that magnitude
    step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    inside = q <= 6
    assert np.all(np.abs(d - w)[inside] <= (step / 2 * X)[inside] * (1 + 1e-12))
    # above 6: saturated to 6 X with the sign
    out = ~inside
    assert np.all(np.abs(d[out]) == 6 * X[out]) and np.all(np.sign(d[out]) == np.sign(w[out]))


def test_expert_and_layer_reduce_to_swiglu():
    rng = np.random.default_rng(5)
    H, F, E, S, k, T = 64, 96, 4, 1, 2, 3
    mats = [(rng.standard_normal(sh) * 0.05).astype(np.float32)
            for _ in range(E + S) for sh in ((F, H), (F, H), (H, F))]
    qs = [orc.quant_mxfp4(m) for m in mats]
    packed = np.concatenate([q[0].reshape(-1) for q in qs])
    scales = np.concatenate([q[1].reshape(-1) for q in qs])
    assert packed.size == (E + S) * orc.fmt_expert_bytes(orc.FMT_MXFP4, H, F)
    assert scales.size == (E + S) * orc.fmt_expert_scale_bytes(orc.FMT_MXFP4, H, F)
    deq = [torch.from_numpy(orc.dequant_mxfp4(q[0], q[1], m.shape[1])) for q, m in zip(qs, mats)]
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) / 8
    counts = np.zeros(E, np.uint32)
    out, idx, gates, _ = orc.moe_forward_fmt(orc.FMT_MXFP4, x, wr, packed, scales, H, F, E, S, k,
                                             counts)
    xt = torch.from_numpy(x)
    ref = torch.zeros((T, H), dtype=torch.float64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            g, u, d = deq[3 * e], deq[3 * e + 1], deq[3 * e + 2]
            ref[t] += gates[t, j] * (d @ (Fn.silu(g @ xt[t]) * (u @ xt[t])))
        g, u, d = deq[3 * E], deq[3 * E + 1], deq[3 * E + 2]
        ref[t] += d @ (Fn.silu(g @ xt[t]) * (u @ xt[t]))
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    # routing is the int4 layer's (same logits, same top-k)
    o4, idx4, _, _ = orc.moe_forward(x, wr, np.zeros((E + S) * orc.expert_packed_bytes(H, F), np.uint8),
                                     np.zeros((E + S) * orc.expert_scales(H, F), np.float32),
                                     H, F, E, S, k)
    assert np.array_equal(idx, idx4)
    assert counts.sum() == T * k
