"""Pins of the oracle's fp8-e4m3-b128 container (fmt 8 of the engine's format
registry) against the OCP E4M3 definition: hand-derived codes, the value table
of all 256 codes, on-grid round trips, the half-step error bound with
saturation, and the layer reduced to a float64 SwiGLU on decoded weights."""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle as orc
from conftest import parse_golden

CASES = parse_golden(os.path.join(os.path.dirname(__file__), "golden", "fp8_hand.txt"))


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_hand_vectors(case):
    w = np.array(case["w"], np.float32)
    p, s = orc.quant_fp8b128(w)
    assert p.tolist() == case["bytes"]
    assert s.view(np.uint32).tolist() == case["scales"]


def test_e4m3_table():
    finite = []
    for c in range(256):
        sgn, e, m = c >> 7, (c >> 3) & 15, c & 7
        v = orc.e4m3_value(c)
        if e == 15 and m == 7:
            assert math.isnan(v)
            continue
        mag = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        assert v == (-mag if sgn else mag)
        finite.append(v)
    assert max(finite) == 448 and min(finite) == -448
    assert sorted(set(abs(v) for v in finite))[1] == 2.0 ** -9


def test_on_grid_round_trip():
    # blocks whose max is 448 s (s a power of two) and whose other elements are
    # E4M3 values times s quantise back to the same codes and scale
    rng = np.random.default_rng(6)
    rows, cols = 8, 256
    s = np.exp2(rng.integers(-12, 2, size=(rows, cols // 128))).astype(np.float32)
    codes = rng.integers(0, 0x7F, size=(rows, cols))
    codes |= rng.integers(0, 2, size=(rows, cols)) << 7
    codes[:, ::128] = 0x7E                      # 448 in every block
    vals = np.array([orc.e4m3_value(c) for c in range(256)])[codes]
    w = (vals * np.repeat(s, 128, axis=1)).astype(np.float32)
    p, sc = orc.quant_fp8b128(w)
    assert np.array_equal(sc, s)
    assert np.array_equal(orc.dequant_fp8b128(p, sc), w.astype(np.float64))


def test_error_bound():
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((16, 384)) * 0.02).astype(np.float32)
    p, s = orc.quant_fp8b128(w)
    d = orc.dequant_fp8b128(p, s)
    S = np.repeat(s.astype(np.float64), 128, axis=1)
    q = np.abs(w) / S
    assert q.max() <= 448 * (1 + 1e-6)
    # the grid step at |q|: 2^(floor(log2 q) - 3) for normals, 2^-9 below 2^-6
    step = np.where(q < 2.0 ** -6, 2.0 ** -9, np.exp2(np.floor(np.log2(np.maximum(q, 1e-30))) - 3))
    assert np.all(np.abs(d - w) <= step / 2 * S * (1 + 1e-6) + 1e-30)


def test_layer_reduces_to_swiglu():
    rng = np.random.default_rng(8)
    H, F, E, S, k, T = 128, 256, 4, 1, 2, 3
    mats = [(rng.standard_normal(sh) * 0.05).astype(np.float32)
            for _ in range(E + S) for sh in ((F, H), (F, H), (H, F))]
    qs = [orc.quant_fp8b128(m) for m in mats]
    packed = np.concatenate([q[0].reshape(-1) for q in qs])
    scales = np.concatenate([q[1].reshape(-1) for q in qs])
    assert packed.size == (E + S) * orc.fmt_expert_bytes(orc.FMT_FP8, H, F)
    assert scales.size * 4 == (E + S) * orc.fmt_expert_scale_bytes(orc.FMT_FP8, H, F)
    deq = [torch.from_numpy(orc.dequant_fp8b128(*q)) for q in qs]
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) / 8
    out, idx, gates, _ = orc.moe_forward_fmt(orc.FMT_FP8, x, wr, packed, scales, H, F, E, S, k)
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
