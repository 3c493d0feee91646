"""The one-token layer kernel (one launch per layer: routing, gate/up, down,
combine, next layer's router partials) against the oracle.  It is taken at
one token when hidden and ffn are whole multiples of 1024 and the used
experts come to at most 512 KB per SM (wider layers run the gate/up and down
GEMV kernels, covered by the other decode tests); these cases span
the slot geometry (down stages of 8, 16 and 24 rows, hidden below and above
ffn), shared experts 0..8, k up to 40, f32 and bf16 routers and inputs, the
sigmoid router, chained stacks (residual and fixed-point logits alternating
between layers), the NaN rule, kernel bracketing, and the bounded grid-barrier
wait running out (flagged, then a correct call)."""
import os

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_ffn_gb300 import synth
from helpers import Layer, REL_TOL, coli, rel_err, tokens_without_ties

pytestmark = pytest.mark.gpu


def desc(shape, x_dtype=torch.float32, bias=None):
    c = coli()
    args = [shape.hidden, shape.ffn, shape.experts, shape.shared, shape.tokens,
            c.COLI_F32 if x_dtype == torch.float32 else c.COLI_BF16,
            c.COLI_F32 if shape.router_dtype == "f32" else c.COLI_BF16]
    if bias is not None:
        args += [c.COLI_ROUTER_SIGMOID_BIAS, bias]
    return c.MoEDesc(*args)


CASES = [
    # (hidden, ffn, experts, shared, top_k, router dtype)
    (1024, 1024, 8, 1, 2, "f32"),       # down stages of 8 rows
    (2048, 1024, 64, 0, 8, "bf16"),     # 16-row down stages, no shared expert
    (3072, 1024, 32, 1, 6, "bf16"),     # 24-row down stages
    (1024, 2048, 16, 2, 4, "bf16"),     # ffn above hidden
    (1024, 1024, 24, 8, 3, "f32"),      # the most shared experts
    (1024, 1024, 128, 0, 40, "bf16"),   # k = 40 > 32: the rank top-k, 40 down experts per CTA
    (6144, 2048, 12, 1, 2, "bf16"),     # the GLM-like widths (k = 2 keeps it on this kernel)
]


@pytest.fixture(autouse=True, scope="module")
def oracle_threads():
    prev = orc.set_threads(os.cpu_count() or 1)
    yield
    orc.set_threads(prev)


@pytest.mark.parametrize("H,F,E,S,k,rdt", CASES)
def test_one_token_layer(H, F, E, S, k, rdt):
    shape = synth.MoEShape("l1", 1, H, F, E, S, k, 1, rdt, "f32")
    layer = Layer(shape, 0, seed=5)
    packed, scales, wr = layer.gpu()
    op, os_, owr = layer.oracle()
    x = tokens_without_ties(shape, owr, seed=5)
    c = coli()
    d = desc(shape)
    ws = c.new_workspace(d, k)
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(2):
        outs.append(c.coli_moe_forward(d, k, x.cuda(), wr, packed, scales, ws,
                                       route_counts=counts).clone())
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]), "not deterministic"
    assert c.coli_moe_check(ws) == 0
    ocounts = np.zeros(E, np.uint32)
    ref, _, _, _ = orc.moe_forward(x.double().numpy(), owr, op, os_, H, F, E, S, k, ocounts)
    err = rel_err(outs[0].cpu().numpy(), ref)
    assert err.max() <= REL_TOL, "max rel err %.3g" % err.max()
    assert np.array_equal(counts.cpu().numpy(), 2 * ocounts)


def test_bf16_input_one_token():
    shape = synth.MoEShape("l1b", 1, 2048, 1024, 32, 1, 4, 1, "bf16", "bf16")
    layer = Layer(shape, 0, seed=6)
    packed, scales, wr = layer.gpu()
    op, os_, owr = layer.oracle()
    x = tokens_without_ties(shape, owr, seed=6, dtype=torch.bfloat16)
    c = coli()
    d = desc(shape, torch.bfloat16)
    ws = c.new_workspace(d, 4)
    out = c.coli_moe_forward(d, 4, x.cuda(), wr, packed, scales, ws)
    ref, _, _, _ = orc.moe_forward(x.double().numpy(), owr, op, os_, 2048, 1024, 32, 1, 4)
    assert rel_err(out.cpu().numpy(), ref).max() <= REL_TOL


@pytest.mark.parametrize("S", [0, 1])
def test_one_token_stack(S):
    """Four chained layers: each kernel adds the next layer's router partials and
    the residual; the fixed-point buffers alternate."""
    L, H, F, E, k = 4, 1024, 1024, 16, 4
    shape = synth.MoEShape("l1s", L, H, F, E, S, k, 1, "bf16", "f32")
    layers = [Layer(shape, l, 2) for l in range(L)]
    gp = [ly.gpu() for ly in layers]
    ol = [ly.oracle() for ly in layers]
    packed = torch.cat([g[0] for g in gp])
    scales = torch.cat([g[1] for g in gp])
    wr = torch.cat([g[2] for g in gp])
    c = coli()
    d = desc(shape)
    ws = c.new_workspace(d, k)
    for step in range(3):
        x = synth.tokens(shape, 2, step)
        counts = torch.zeros((L, E), dtype=torch.int32, device="cuda")
        layer_out = torch.empty((L, 1, H), device="cuda")
        xo = c.coli_moe_stack_forward(d, k, L, x.cuda(), wr, packed, scales, ws,
                                      layer_out=layer_out, route_counts=counts)
        ocounts = np.zeros((L, E), np.uint32)
        xL, outs, _ = orc.moe_stack_forward(x.double().numpy(), [(w, p, s) for p, s, w in ol],
                                            H, F, E, S, k, ocounts)
        torch.cuda.synchronize()
        assert np.array_equal(counts.cpu().numpy(), ocounts), "step %d counts" % step
        for l in range(L):
            assert rel_err(layer_out[l].cpu().numpy(), outs[l]).max() <= REL_TOL, (step, l)
        assert rel_err(xo.cpu().numpy(), xL).max() <= REL_TOL


def test_sigmoid_router_one_token_stack():
    L, H, F, E, S, k = 3, 2048, 1024, 64, 1, 8
    shape = synth.MoEShape("l1g", L, H, F, E, S, k, 1, "bf16", "f32")
    layers = [Layer(shape, l, 4) for l in range(L)]
    biases = [synth.router_bias(shape, l, 4) for l in range(L)]
    gp = [ly.gpu() for ly in layers]
    ol = [ly.oracle() for ly in layers]
    x = tokens_without_ties(shape, ol[0][2], seed=4, bias=biases[0].double().numpy())
    c = coli()
    d = desc(shape, bias=torch.cat(biases).cuda())
    ws = c.new_workspace(d, k)
    counts = torch.zeros((L, E), dtype=torch.int32, device="cuda")
    xo = c.coli_moe_stack_forward(d, k, L, x.cuda(), torch.cat([g[2] for g in gp]),
                                  torch.cat([g[0] for g in gp]), torch.cat([g[1] for g in gp]),
                                  ws, route_counts=counts)
    ocounts = np.zeros((L, E), np.uint32)
    ref, _, _ = orc.moe_stack_forward(x.double().numpy(), [(w, p, s) for p, s, w in ol], H, F, E,
                                      S, k, ocounts, router="sigmoid",
                                      biases=[b.double().numpy() for b in biases])
    torch.cuda.synchronize()
    assert rel_err(xo.cpu().numpy(), ref).max() <= REL_TOL
    assert np.array_equal(counts.cpu().numpy(), ocounts)


def test_nan_token_falls_back_and_flags():
    shape = synth.MoEShape("l1n", 1, 1024, 1024, 16, 1, 4, 1, "f32", "f32")
    layer = Layer(shape, 0, seed=7)
    packed, scales, wr = layer.gpu()
    x = synth.tokens(shape, 7).cuda()
    x[0, 3] = float("nan")
    c = coli()
    d = desc(shape)
    ws = c.new_workspace(d, 4)
    counts = torch.zeros(16, dtype=torch.int32, device="cuda")
    c.coli_moe_forward(d, 4, x, wr, packed, scales, ws, route_counts=counts)
    assert c.coli_moe_check(ws) & c.COLI_FLAG_NAN_LOGITS
    # every logit NaN: experts 0..k-1, one route each
    assert counts.cpu().numpy().tolist() == [1, 1, 1, 1] + [0] * 12


def test_profile_events_bracket_the_layer_kernel():
    shape = synth.MoEShape("l1p", 3, 1024, 1024, 16, 1, 4, 1, "bf16", "f32")
    layers = [Layer(shape, l, 0) for l in range(3)]
    gp = [ly.gpu() for ly in layers]
    packed = torch.cat([g[0] for g in gp])
    scales = torch.cat([g[1] for g in gp])
    wr = torch.cat([g[2] for g in gp])
    x = synth.tokens(shape).cuda()
    c = coli()
    d = desc(shape)
    ws = c.new_workspace(d, 4)
    ref = c.coli_moe_stack_forward(d, 4, 3, x, wr, packed, scales, ws).clone()
    stream = torch.cuda.Stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record(stream)
    torch.cuda.synchronize()
    c.coli_profile_events(c.COLI_KERNEL_LAYER, ev[:3], ev[3:])
    try:
        g = torch.cuda.CUDAGraph()
        out = torch.empty_like(ref)
        with torch.cuda.graph(g, stream=stream):
            c.coli_moe_stack_forward(d, 4, 3, x, wr, packed, scales, ws, x_out=out, stream=stream)
    finally:
        got = c.coli_profile_events(c.COLI_KERNEL_LAYER, [], [])
    assert got == 3
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert all(0.0 < b.elapsed_time(a) < 1000.0 for b, a in zip(ev[:3], ev[3:]))


def test_grid_barrier_wait_runs_out_then_recovers():
    """A workspace control word shortens the grid barrier's bounded wait to one
    clock cycle: CTAs that arrive early give up, the call flags
    COLI_FLAG_TIMEOUT (coli_moe_check returns COLI_ETIMEOUT); with the word
    cleared the next call on the same workspace is correct."""
    shape = synth.MoEShape("l1t", 1, 2048, 1024, 64, 1, 8, 1, "bf16", "f32")
    layer = Layer(shape, 0, seed=8)
    packed, scales, wr = layer.gpu()
    op, os_, owr = layer.oracle()
    x = tokens_without_ties(shape, owr, seed=8).cuda()
    c = coli()
    d = desc(shape)
    ws = c.new_workspace(d, 8)
    words = ws[:256].view(torch.int32)
    WAIT_LIMIT = 5                                  # control word index (coli_internal.cuh)
    words[WAIT_LIMIT] = 1
    c.coli_moe_forward(d, 8, x, wr, packed, scales, ws)
    torch.cuda.synchronize()
    flags = c.coli_moe_check(ws)                    # reads and clears the flag word
    assert flags & c.COLI_FLAG_TIMEOUT
    words[WAIT_LIMIT] = 0
    out = c.coli_moe_forward(d, 8, x, wr, packed, scales, ws)
    torch.cuda.synchronize()
    assert c.coli_moe_check(ws) == 0
    ref, _, _, _ = orc.moe_forward(x.double().cpu().numpy(), owr, op, os_, 2048, 1024, 64, 1, 8)
    assert rel_err(out.cpu().numpy(), ref).max() <= REL_TOL
