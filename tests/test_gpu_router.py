"""GPU router (coli_router_topk) against the oracle: bit-exact indices and counts,
gates within f32 rounding, NaN and tie rules."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_ffn_gb300 import synth
from helpers import coli, tokens_without_ties

pytestmark = pytest.mark.gpu


def run_router(shape, x, wr, k=None, counts=None):
    c = coli()
    k = k or shape.top_k
    T = x.shape[0]
    desc = c.MoEDesc(shape.hidden, shape.ffn, shape.experts, shape.shared, T,
                     c.COLI_F32 if x.dtype == torch.float32 else c.COLI_BF16,
                     c.COLI_F32 if wr.dtype == torch.float32 else c.COLI_BF16)
    ws = c.new_workspace(desc, k)
    idx, gates = c.coli_router_topk(desc, k, x.cuda(), wr.cuda(), ws, route_counts=counts)
    flags = c.coli_moe_check(ws)
    return idx.cpu().numpy(), gates.cpu().numpy(), flags


def oracle_router(x, wr, k):
    lg = orc.router_logits(x.double().numpy(), wr.double().numpy())
    res = [orc.topk(l, k) for l in lg]
    return np.stack([r[0] for r in res]), np.stack([r[1] for r in res]), any(r[2] for r in res)


SHAPES = [
    (synth.TINY, 4),
    (synth.OLMOE_DECODE, 1),
    (synth.OLMOE_DECODE, 16),
    (synth.GLM_DECODE_B8, 8),
    (synth.GLM_DECODE_B1, 37),     # several 16-token passes, ragged tail
]


@pytest.mark.parametrize("shape,T", SHAPES, ids=["%s-T%d" % (s.name, t) for s, t in SHAPES])
def test_router_parity(shape, T):
    shape = dataclasses.replace(shape, tokens=T)
    wr = synth.router_weights(shape, 0)
    x = tokens_without_ties(shape, wr.double().numpy())
    counts = torch.zeros(shape.experts, dtype=torch.int32, device="cuda")
    idx, gates, flags = run_router(shape, x, wr, counts=counts)
    oi, og, _ = oracle_router(x, wr, shape.top_k)
    assert np.array_equal(idx, oi)
    np.testing.assert_allclose(gates, og, rtol=2e-5, atol=1e-7)
    hist = np.bincount(oi.reshape(-1), minlength=shape.experts)
    assert np.array_equal(counts.cpu().numpy(), hist)
    assert flags == 0


@pytest.mark.parametrize("E,k", [(8, 1), (8, 8), (64, 33), (64, 64), (256, 8), (1000, 5)])
def test_router_k_and_E_range(E, k):
    shape = dataclasses.replace(synth.TINY, experts=E, top_k=k, tokens=5, hidden=128)
    wr = synth.router_weights(shape, 1)
    x = tokens_without_ties(shape, wr.double().numpy())
    idx, gates, _ = run_router(shape, x, wr, k=k)
    oi, og, _ = oracle_router(x, wr, k)
    assert np.array_equal(idx, oi)
    np.testing.assert_allclose(gates, og, rtol=2e-5, atol=1e-7)


def test_router_equal_logits_lower_id_first():
    shape = dataclasses.replace(synth.TINY, tokens=3)
    wr = synth.router_weights(shape, 0)
    wr[5] = wr[1]          # identical rows -> identical f32 logits
    wr[6] = wr[1]
    x = synth.tokens(shape)
    idx, gates, _ = run_router(shape, x, wr, k=8)
    for t in range(3):
        pos = [list(idx[t]).index(e) for e in (1, 5, 6)]
        assert pos == sorted(pos)
        assert gates[t][pos[0]] == gates[t][pos[1]] == gates[t][pos[2]]
    # zero router: every logit 0 -> experts 0..k-1, gates 1/k
    idx, gates, _ = run_router(shape, x, torch.zeros_like(wr), k=3)
    assert (idx == np.arange(3)).all()
    np.testing.assert_allclose(gates, 1 / 3, rtol=1e-6)


def test_router_nan_rules():
    shape = dataclasses.replace(synth.TINY, tokens=3)
    wr = synth.router_weights(shape, 0)
    x = synth.tokens(shape).clone()
    x[1, 7] = float("nan")          # token 1: every logit NaN
    wr[2, 3] = float("nan")         # expert 2: NaN logit for every token
    counts = torch.zeros(shape.experts, dtype=torch.int32, device="cuda")
    idx, gates, flags = run_router(shape, x, wr, k=8, counts=counts)
    assert flags & coli().COLI_FLAG_NAN_LOGITS
    assert idx[1].tolist() == list(range(8))
    np.testing.assert_allclose(gates[1], 1 / 8)
    for t in (0, 2):
        assert idx[t][-1] == 2 and gates[t][-1] == 0     # NaN ranks last, gate 0
        np.testing.assert_allclose(gates[t].sum(), 1.0, rtol=1e-6)
    oi, og, onan = oracle_router(x, wr, 8)
    assert onan and np.array_equal(idx, oi)
    np.testing.assert_allclose(gates, og, rtol=2e-5, atol=1e-7)
    assert counts.cpu().numpy().sum() == 3 * 8


def test_router_counts_accumulate():
    shape = dataclasses.replace(synth.OLMOE_DECODE, tokens=4)
    wr = synth.router_weights(shape, 3)
    x = tokens_without_ties(shape, wr.double().numpy())
    counts = torch.zeros(shape.experts, dtype=torch.int32, device="cuda")
    for _ in range(3):
        idx, _, _ = run_router(shape, x, wr, counts=counts)
    hist = np.bincount(idx.reshape(-1), minlength=shape.experts)
    assert np.array_equal(counts.cpu().numpy(), 3 * hist)
