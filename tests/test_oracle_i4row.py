"""Pins of the oracle's int4-row container (fmt 2 of the engine's format
registry): hand-derived bytes, equality with int4-grouped when a row is one
group (at most 64 columns), the half-step error bound, on-grid round trips,
and the layer reduced to a float64 SwiGLU on the decoded weights."""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle as orc
from conftest import parse_golden

CASES = parse_golden(os.path.join(os.path.dirname(__file__), "golden", "i4row_hand.txt"))


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_hand_vectors(case):
    w = np.array(case["w"], np.float32)
    p, s = orc.quant_i4row(w)
    assert p.tolist() == case["bytes"]
    assert s.view(np.uint32).tolist() == case["scales"]


@pytest.mark.parametrize("cols", [1, 7, 33, 64])
def test_equals_grouped_for_one_group(cols):
    rng = np.random.default_rng(cols)
    w = (rng.standard_normal((9, cols)) * 0.05).astype(np.float32)
    w[0] = 0
    pr, sr = orc.quant_i4row(w)
    pg, sg = orc.quant_i4g(w)
    assert np.array_equal(pr, pg)
    assert np.array_equal(sr.view(np.uint32), sg.view(np.uint32))


def test_error_bound_and_range():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((24, 777)) * 0.02).astype(np.float32)
    w[5, 100] = 0.9                           # an outlier widens its row's step
    p, s = orc.quant_i4row(w)
    d = orc.dequant_i4row(p, s, 777)
    step = s.astype(np.float64)
    assert np.all(np.abs(d - w) <= step / 2 * (1 + 1e-6))
    u = np.stack([p & 15, p >> 4], axis=2).reshape(24, -1)[:, :777]
    assert u.min() >= 1 and u.max() <= 15     # q in [-7, 7]: the clip at -8 never fires
    assert np.all((np.abs(u.astype(int) - 8) == 7).any(axis=1))


def test_on_grid_round_trip():
    rng = np.random.default_rng(4)
    q = rng.integers(-7, 8, size=(6, 300))
    q[:, 0] = 7
    s = np.exp2(rng.integers(-9, 1, size=(6, 1))).astype(np.float32)
    w = (q * s).astype(np.float32)
    p, sc = orc.quant_i4row(w)
    assert np.array_equal(sc, s)
    assert np.array_equal(orc.dequant_i4row(p, sc, 300), w.astype(np.float64))


def test_layer_reduces_to_swiglu():
    rng = np.random.default_rng(5)
    H, F, E, S, k, T = 128, 192, 5, 1, 2, 3
    mats = [(rng.standard_normal(sh) * 0.05).astype(np.float32)
            for _ in range(E + S) for sh in ((F, H), (F, H), (H, F))]
    qs = [orc.quant_i4row(m) for m in mats]
    packed = np.concatenate([q[0].reshape(-1) for q in qs])
    scales = np.concatenate([q[1].reshape(-1) for q in qs])
    assert packed.size == (E + S) * orc.fmt_expert_bytes(orc.FMT_I4ROW, H, F)
    assert scales.size * 4 == (E + S) * orc.fmt_expert_scale_bytes(orc.FMT_I4ROW, H, F)
    deq = [torch.from_numpy(orc.dequant_i4row(q[0], q[1], m.shape[1])) for q, m in zip(qs, mats)]
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) / 8
    out, idx, gates, _ = orc.moe_forward_fmt(orc.FMT_I4ROW, x, wr, packed, scales, H, F, E, S, k)
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
