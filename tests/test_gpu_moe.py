"""GPU routed-MoE layer / stack (coli_moe_forward, coli_moe_stack_forward) against
the oracle: outputs within 2e-3 relative error per token, route counts bit-exact."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_ffn_gb300 import synth
from helpers import Layer, REL_TOL, coli, rel_err, tokens_without_ties

pytestmark = pytest.mark.gpu


def desc_for(shape, T, x_dtype=torch.float32):
    c = coli()
    return c.MoEDesc(shape.hidden, shape.ffn, shape.experts, shape.shared, T,
                     c.COLI_F32 if x_dtype == torch.float32 else c.COLI_BF16,
                     c.COLI_F32 if shape.router_dtype == "f32" else c.COLI_BF16)


def check_layer(shape, T, x_dtype=torch.float32, seed=0, repeat=1):
    shape = dataclasses.replace(shape, tokens=T)
    layer = Layer(shape, 0, seed)
    packed, scales, wr = layer.gpu()
    op, os_, owr = layer.oracle()
    assert np.array_equal(packed.cpu().numpy(), op), "GPU and oracle packing differ"
    x = tokens_without_ties(shape, owr, seed, dtype=x_dtype)
    c = coli()
    desc = desc_for(shape, T, x_dtype)
    ws = c.new_workspace(desc, shape.top_k)
    counts = torch.zeros(shape.experts, dtype=torch.int32, device="cuda")
    for _ in range(repeat):
        out = c.coli_moe_forward(desc, shape.top_k, x.cuda(), wr, packed, scales, ws,
                                 route_counts=counts)
    torch.cuda.synchronize()
    ocounts = np.zeros(shape.experts, np.uint32)
    ref, idx, gates, _ = orc.moe_forward(x.double().numpy(), owr, op, os_, shape.hidden,
                                         shape.ffn, shape.experts, shape.shared, shape.top_k,
                                         ocounts)
    err = rel_err(out.cpu().numpy(), ref)
    assert err.max() <= REL_TOL, "max rel err %.3g" % err.max()
    assert np.array_equal(counts.cpu().numpy(), repeat * ocounts)
    return err


def test_tiny_config():
    err = check_layer(synth.TINY, 4)
    assert err.max() < 5e-4      # 15-bit activations: far inside the 2e-3 bound


SMALL = [
    # (hidden, ffn, experts, shared, top_k, tokens)
    (128, 192, 5, 0, 2, 3),
    (320, 64, 12, 2, 3, 16),
    (64, 64, 4, 1, 4, 1),        # k = E
    (1088, 1088, 9, 1, 2, 5),    # not a multiple of 1024: ragged chunk
    (256, 512, 8, 1, 2, 37),     # three 16-token passes, ragged tail
    (2048, 1024, 64, 0, 8, 8),
    (16384, 64, 4, 1, 2, 1),     # the largest hidden size: 16 chunks per gate/up row
    (64, 16384, 3, 0, 1, 2),     # the largest FFN width: 16 chunks per down row
    (256, 256, 1, 0, 1, 3),      # a single routed expert
    (128, 128, 4, 8, 2, 2),      # the most shared experts
    (64, 64, 64, 0, 64, 1),      # k = 64 (the largest top-k): the rank top-k in the routing
    (192, 128, 40, 1, 33, 4),    # k = 33 > 32, several tokens
]


@pytest.mark.parametrize("H,F,E,S,k,T", SMALL)
def test_layer_shapes(H, F, E, S, k, T):
    shape = synth.MoEShape("t", 1, H, F, E, S, k, T, "bf16", "f32")
    check_layer(shape, T)


def test_bf16_activations_and_f32_router():
    shape = dataclasses.replace(synth.TINY, x_dtype="bf16")
    check_layer(shape, 6, x_dtype=torch.bfloat16)


def test_counts_accumulate_and_deterministic():
    shape = dataclasses.replace(synth.TINY, tokens=4)
    check_layer(shape, 4, repeat=3)
    # identical inputs -> bit-identical outputs
    layer = Layer(shape, 0, 1)
    packed, scales, wr = layer.gpu()
    x = synth.tokens(shape).cuda()
    c = coli()
    desc = desc_for(shape, 4)
    ws = c.new_workspace(desc, shape.top_k)
    a = c.coli_moe_forward(desc, shape.top_k, x, wr, packed, scales, ws)
    b = c.coli_moe_forward(desc, shape.top_k, x, wr, packed, scales, ws)
    assert torch.equal(a, b)


def test_zero_tokens_is_noop():
    c = coli()
    shape = synth.TINY
    desc = desc_for(shape, 0)
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    out = torch.full((1, shape.hidden), 7.0, device="cuda")
    st = c.lib.coli_moe_forward(__import__("ctypes").byref(desc.c()), 2, None, None, None, None,
                                out.data_ptr(), None, ws.data_ptr(), ws.numel(), None)
    assert st == c.COLI_OK
    assert (out == 7).all()


def test_stack_tiny_chain():
    """Residual chain over 3 layers: x_{l+1} = x_l + MoE_l(x_l), per-layer outputs."""
    shape = dataclasses.replace(synth.TINY, layers=3, tokens=2)
    layers = [Layer(shape, l, 0) for l in range(3)]
    gp = [ly.gpu() for ly in layers]
    packed = torch.cat([g[0] for g in gp])
    scales = torch.cat([g[1] for g in gp])
    wr = torch.cat([g[2] for g in gp])
    ol = [ly.oracle() for ly in layers]
    x = synth.tokens(shape)
    c = coli()
    desc = desc_for(shape, 2)
    ws = c.new_workspace(desc, shape.top_k)
    counts = torch.zeros((3, shape.experts), dtype=torch.int32, device="cuda")
    layer_out = torch.empty((3, 2, shape.hidden), device="cuda")
    xo = c.coli_moe_stack_forward(desc, shape.top_k, 3, x.cuda(), wr, packed, scales, ws,
                                  layer_out=layer_out, route_counts=counts)
    ocounts = np.zeros((3, shape.experts), np.uint32)
    xL, outs, _ = orc.moe_stack_forward(x.double().numpy(), [(w, p, s) for p, s, w in ol],
                                        shape.hidden, shape.ffn, shape.experts, shape.shared,
                                        shape.top_k, ocounts)
    assert rel_err(xo.cpu().numpy(), xL).max() <= REL_TOL
    for l in range(3):
        assert rel_err(layer_out[l].cpu().numpy(), outs[l]).max() <= REL_TOL
    assert np.array_equal(counts.cpu().numpy(), ocounts)


@pytest.mark.parametrize("graph", [False, True])
def test_profile_events_bracket_each_kernel(graph):
    """coli_profile_events brackets exactly the selected kernel's launches, in
    eager mode and inside a captured graph, without changing the results."""
    shape = dataclasses.replace(synth.TINY, layers=3, tokens=2)
    layers = [Layer(shape, l, 0) for l in range(3)]
    gp = [ly.gpu() for ly in layers]
    packed = torch.cat([g[0] for g in gp])
    scales = torch.cat([g[1] for g in gp])
    wr = torch.cat([g[2] for g in gp])
    x = synth.tokens(shape).cuda()
    c = coli()
    desc = desc_for(shape, 2)
    ws = c.new_workspace(desc, shape.top_k)
    ref = c.coli_moe_stack_forward(desc, shape.top_k, 3, x, wr, packed, scales, ws).clone()
    stream = torch.cuda.Stream()
    for kernel, n in ((c.COLI_KERNEL_ROUTE, 1), (c.COLI_KERNEL_GATEUP, 3), (c.COLI_KERNEL_DOWN, 3)):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
        for e in ev:
            e.record(stream)
        out = torch.empty_like(ref)
        torch.cuda.synchronize()
        c.coli_profile_events(kernel, ev[:n], ev[n:])
        try:
            if graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    c.coli_moe_stack_forward(desc, shape.top_k, 3, x, wr, packed, scales, ws,
                                             x_out=out, stream=stream)
            else:
                with torch.cuda.stream(stream):
                    c.coli_moe_stack_forward(desc, shape.top_k, 3, x, wr, packed, scales, ws,
                                             x_out=out, stream=stream)
        finally:
            got = c.coli_profile_events(kernel, [], [])
        assert got == n
        if graph:
            g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        times = [b.elapsed_time(a) for b, a in zip(ev[:n], ev[n:])]
        assert all(0.0 < t < 1000.0 for t in times), times
