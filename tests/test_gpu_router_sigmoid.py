"""The GLM router variant (sigmoid scores, selection-only bias, normalised gates)
on the GPU against the oracle: the router-only call, the decode layer at one
and several tokens (fixed-point routing in the gate/up CTAs, and the ticket
path when T * E is large), the stack with per-layer biases, and the batched
path.  Indices and counts bit-exact, gates and outputs within tolerance."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_ffn_gb300 import synth
from helpers import Layer, REL_TOL, coli, rel_err, tokens_without_ties

pytestmark = pytest.mark.gpu


def desc_for(shape, T, bias, x_dtype=torch.float32):
    c = coli()
    return c.MoEDesc(shape.hidden, shape.ffn, shape.experts, shape.shared, T,
                     c.COLI_F32 if x_dtype == torch.float32 else c.COLI_BF16,
                     c.COLI_F32 if shape.router_dtype == "f32" else c.COLI_BF16,
                     c.COLI_ROUTER_SIGMOID_BIAS, bias)


ROUTER_SHAPES = [
    (synth.TINY, 4),
    (synth.OLMOE_DECODE, 1),
    (synth.GLM_DECODE_B8, 8),
    (synth.GLM_DECODE_B1, 37),     # 16-token passes: T * E above the fixed-point limit
]


@pytest.mark.parametrize("shape,T", ROUTER_SHAPES,
                         ids=["%s-T%d" % (s.name, t) for s, t in ROUTER_SHAPES])
def test_sigmoid_router_parity(shape, T):
    shape = dataclasses.replace(shape, tokens=T)
    wr = synth.router_weights(shape, 0)
    bias = synth.router_bias(shape, 0)
    x = tokens_without_ties(shape, wr.double().numpy(), bias=bias.double().numpy())
    c = coli()
    desc = desc_for(shape, T, bias.cuda())
    ws = c.new_workspace(desc, shape.top_k)
    counts = torch.zeros(shape.experts, dtype=torch.int32, device="cuda")
    idx, gates = c.coli_router_topk(desc, shape.top_k, x.cuda(), wr.cuda(), ws,
                                    route_counts=counts)
    assert c.coli_moe_check(ws) == 0
    lg = orc.router_logits(x.double().numpy(), wr.double().numpy())
    res = [orc.topk_sigmoid(l, shape.top_k, bias.double().numpy()) for l in lg]
    oi = np.stack([r[0] for r in res])
    og = np.stack([r[1] for r in res])
    assert np.array_equal(idx.cpu().numpy(), oi)
    np.testing.assert_allclose(gates.cpu().numpy(), og, rtol=2e-5, atol=1e-7)
    assert np.array_equal(counts.cpu().numpy(), np.bincount(oi.reshape(-1), minlength=shape.experts))


def test_sigmoid_router_null_bias_is_zero_bias():
    shape = dataclasses.replace(synth.OLMOE_DECODE, tokens=3)
    wr = synth.router_weights(shape, 0)
    x = tokens_without_ties(shape, wr.double().numpy(), bias=np.zeros(shape.experts))
    c = coli()
    desc = desc_for(shape, 3, None)
    ws = c.new_workspace(desc, shape.top_k)
    idx, gates = c.coli_router_topk(desc, shape.top_k, x.cuda(), wr.cuda(), ws)
    lg = orc.router_logits(x.double().numpy(), wr.double().numpy())
    for t in range(3):
        oi, og, _ = orc.topk_sigmoid(lg[t], shape.top_k)
        assert idx[t].cpu().numpy().tolist() == oi.tolist()
        np.testing.assert_allclose(gates[t].cpu().numpy(), og, rtol=2e-5, atol=1e-7)


def check_layer(shape, T, n_layers=1):
    shape = dataclasses.replace(shape, tokens=T, layers=n_layers)
    layers = [Layer(shape, l, 0) for l in range(n_layers)]
    biases = [synth.router_bias(shape, l) for l in range(n_layers)]
    gp = [ly.gpu() for ly in layers]
    ol = [ly.oracle() for ly in layers]
    x = tokens_without_ties(shape, ol[0][2], bias=biases[0].double().numpy())
    c = coli()
    bias_dev = torch.cat(biases).cuda()
    desc = desc_for(shape, T, bias_dev)
    ws = c.new_workspace(desc, shape.top_k)
    counts = torch.zeros((n_layers, shape.experts), dtype=torch.int32, device="cuda")
    ocounts = np.zeros((n_layers, shape.experts), np.uint32)
    if n_layers == 1:
        out = c.coli_moe_forward(desc, shape.top_k, x.cuda(), gp[0][2], gp[0][0], gp[0][1], ws,
                                 route_counts=counts[0])
        ref, _, _, _ = orc.moe_forward(x.double().numpy(), ol[0][2], ol[0][0], ol[0][1],
                                       shape.hidden, shape.ffn, shape.experts, shape.shared,
                                       shape.top_k, ocounts[0], router="sigmoid",
                                       bias=biases[0].double().numpy())
    else:
        packed = torch.cat([g[0] for g in gp])
        scales = torch.cat([g[1] for g in gp])
        wr = torch.cat([g[2] for g in gp])
        out = c.coli_moe_stack_forward(desc, shape.top_k, n_layers, x.cuda(), wr, packed, scales,
                                       ws, route_counts=counts)
        ref, _, _ = orc.moe_stack_forward(x.double().numpy(), [(w, p, s) for p, s, w in ol],
                                          shape.hidden, shape.ffn, shape.experts, shape.shared,
                                          shape.top_k, ocounts, router="sigmoid",
                                          biases=[b.double().numpy() for b in biases])
    torch.cuda.synchronize()
    assert c.coli_moe_check(ws) == 0
    err = rel_err(out.cpu().numpy(), ref)
    assert err.max() <= REL_TOL, "max rel err %.3g" % err.max()
    assert np.array_equal(counts.cpu().numpy(), ocounts)


LAYER_CASES = [
    # (hidden, ffn, experts, shared, top_k, tokens, layers)
    (256, 512, 8, 1, 2, 4, 1),       # several tokens
    (2048, 1024, 64, 1, 8, 1, 1),    # one token
    (2048, 1024, 64, 1, 8, 8, 1),
    (512, 256, 256, 1, 8, 16, 1),    # T * E = 4096: routed by the last CTA
    (256, 512, 16, 1, 4, 1, 3),      # stack, one token, per-layer biases
    (256, 512, 16, 0, 4, 5, 3),      # stack, several tokens
    (512, 256, 256, 1, 8, 12, 2),    # stack above the fixed-point limit
]


@pytest.mark.parametrize("H,F,E,S,k,T,L", LAYER_CASES)
def test_sigmoid_layer(H, F, E, S, k, T, L):
    shape = synth.MoEShape("s", L, H, F, E, S, k, T, "bf16", "f32")
    check_layer(shape, T, L)


def test_sigmoid_prefill_layer():
    """The batched path (T >= 64) routes with the same function."""
    check_layer(synth.MoEShape("sp", 1, 256, 128, 8, 1, 2, 100, "bf16", "f32"), 100)
