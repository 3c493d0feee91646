"""One-token calls on the GEMV kernels: the first layer's gate/up CTAs form
its router logits themselves (each CTA the whole logits of the experts it
owns, published as nonzero words that every CTA waits for) instead of a
router launch before them.  Against the oracle: f32 and bf16 inputs and
routers, the sigmoid router, stacks (layer 0 routed this way, later layers
from the previous down kernel's partials), calls back to back on one
workspace (the down kernel leaves the words zero), graph replay, and the
bounded wait for the words running out (flagged, then a correct call)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_ffn_gb300 import synth
from helpers import Layer, REL_TOL, coli, rel_err, tokens_without_ties

pytestmark = pytest.mark.gpu


def make(H, F, E, S, k, rdt="bf16", xdt="f32", L=1, seed=0):
    shape = synth.MoEShape("gr", L, H, F, E, S, k, 1, rdt, xdt)
    layers = [Layer(shape, l, seed) for l in range(L)]
    return shape, layers


def desc(shape, x_dtype, bias=None):
    c = coli()
    args = [shape.hidden, shape.ffn, shape.experts, shape.shared, 1,
            c.COLI_F32 if x_dtype == torch.float32 else c.COLI_BF16,
            c.COLI_F32 if shape.router_dtype == "f32" else c.COLI_BF16]
    if bias is not None:
        args += [c.COLI_ROUTER_SIGMOID_BIAS, bias]
    return c.MoEDesc(*args)


# H not a multiple of 1024: the gate/up and down GEMV kernels (not the one-token layer kernel)
@pytest.mark.parametrize("xdt,rdt", [(torch.float32, "bf16"), (torch.bfloat16, "f32"),
                                     (torch.float32, "f32"), (torch.bfloat16, "bf16")])
def test_first_layer_router_in_gateup(xdt, rdt):
    shape, (layer,) = make(1536, 512, 64, 1, 6, rdt=rdt)
    packed, scales, wr = layer.gpu()
    op, os_, owr = layer.oracle()
    c = coli()
    d = desc(shape, xdt)
    ws = c.new_workspace(d, shape.top_k)
    counts = torch.zeros(shape.experts, dtype=torch.int32, device="cuda")
    ocounts = np.zeros(shape.experts, np.uint32)
    for step in range(4):                     # back to back on one workspace
        x = tokens_without_ties(shape, owr, seed=3, step=step, dtype=xdt)
        out = c.coli_moe_forward(d, shape.top_k, x.cuda(), wr, packed, scales, ws,
                                 route_counts=counts)
        torch.cuda.synchronize()
        assert c.coli_moe_check(ws) == 0
        ref, _, _, _ = orc.moe_forward(x.double().numpy(), owr, op, os_, shape.hidden, shape.ffn,
                                       shape.experts, shape.shared, shape.top_k, ocounts)
        assert rel_err(out.cpu().numpy(), ref).max() <= REL_TOL, step
    assert np.array_equal(counts.cpu().numpy(), ocounts)


def test_sigmoid_router_and_graph_replay():
    shape, (layer,) = make(3072, 1536, 96, 1, 8)
    packed, scales, wr = layer.gpu()
    op, os_, owr = layer.oracle()
    bias = synth.router_bias(shape, 0, 5)
    c = coli()
    d = desc(shape, torch.float32, bias=bias.cuda())
    ws = c.new_workspace(d, shape.top_k)
    xs = [tokens_without_ties(shape, owr, seed=5, step=s, bias=bias.double().numpy())
          for s in range(3)]
    xin = torch.empty((1, shape.hidden), device="cuda")
    out = torch.empty((1, shape.hidden), device="cuda")
    stream = torch.cuda.Stream()
    xin.copy_(xs[0].cuda())
    with torch.cuda.stream(stream):
        c.coli_moe_forward(d, shape.top_k, xin, wr, packed, scales, ws, out=out, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        c.coli_moe_forward(d, shape.top_k, xin, wr, packed, scales, ws, out=out, stream=stream)
    for x in xs:
        xin.copy_(x.cuda())
        g.replay()
        torch.cuda.synchronize()
        ref, _, _, _ = orc.moe_forward(x.double().numpy(), owr, op, os_, shape.hidden, shape.ffn,
                                       shape.experts, shape.shared, shape.top_k,
                                       router="sigmoid", bias=bias.double().numpy())
        assert rel_err(out.cpu().numpy(), ref).max() <= REL_TOL
    assert c.coli_moe_check(ws) == 0


def test_stack_first_layer_router_in_gateup():
    shape, layers = make(1536, 1024, 32, 1, 4, L=3, seed=2)
    gp = [ly.gpu() for ly in layers]
    ol = [ly.oracle() for ly in layers]
    c = coli()
    d = desc(shape, torch.float32)
    ws = c.new_workspace(d, shape.top_k)
    for step in range(2):
        x = synth.tokens(shape, 2, step)
        counts = torch.zeros((3, shape.experts), dtype=torch.int32, device="cuda")
        layer_out = torch.empty((3, 1, shape.hidden), device="cuda")
        xo = c.coli_moe_stack_forward(d, shape.top_k, 3, x.cuda(),
                                      torch.cat([g[2] for g in gp]), torch.cat([g[0] for g in gp]),
                                      torch.cat([g[1] for g in gp]), ws, layer_out=layer_out,
                                      route_counts=counts)
        ocounts = np.zeros((3, shape.experts), np.uint32)
        xL, outs, _ = orc.moe_stack_forward(x.double().numpy(), [(w, p, s) for p, s, w in ol],
                                            shape.hidden, shape.ffn, shape.experts, shape.shared,
                                            shape.top_k, ocounts)
        torch.cuda.synchronize()
        assert np.array_equal(counts.cpu().numpy(), ocounts), step
        for l in range(3):
            assert rel_err(layer_out[l].cpu().numpy(), outs[l]).max() <= REL_TOL, (step, l)
        assert rel_err(xo.cpu().numpy(), xL).max() <= REL_TOL


def test_router_wait_runs_out_then_recovers():
    """A workspace control word shortens the bounded wait for the published
    logit words to one clock cycle: CTAs that read a word before its owner
    wrote it give up, the call flags COLI_FLAG_TIMEOUT; with the word cleared
    the next call on the same workspace is correct."""
    shape, (layer,) = make(1536, 512, 64, 1, 6)
    packed, scales, wr = layer.gpu()
    op, os_, owr = layer.oracle()
    c = coli()
    d = desc(shape, torch.float32)
    ws = c.new_workspace(d, shape.top_k)
    x = tokens_without_ties(shape, owr, seed=8)
    words = ws[:256].view(torch.int32)
    WAIT_LIMIT = 5                                  # control word index (coli_internal.cuh)
    words[WAIT_LIMIT] = 1
    c.coli_moe_forward(d, shape.top_k, x.cuda(), wr, packed, scales, ws)
    torch.cuda.synchronize()
    assert c.coli_moe_check(ws) & c.COLI_FLAG_TIMEOUT
    words[WAIT_LIMIT] = 0
    out = c.coli_moe_forward(d, shape.top_k, x.cuda(), wr, packed, scales, ws)
    torch.cuda.synchronize()
    assert c.coli_moe_check(ws) == 0
    ref, _, _, _ = orc.moe_forward(x.double().numpy(), owr, op, os_, shape.hidden, shape.ffn,
                                   shape.experts, shape.shared, shape.top_k)
    assert rel_err(out.cpu().numpy(), ref).max() <= REL_TOL
