"""int4-row container (COLI_FMT_I4ROW) on the GPU against the oracle: the
quantiser bit for bit (hand vectors, random rows with outliers, ragged and
odd column counts, NaN, -0 and all-zero rows, bf16 and f32), and int4-row
layers -- on the tensor-core grouped GEMM at every token count -- within the
tolerance of the other tests, route counts exact, including the sigmoid
router, shared experts and a chained stack."""
import os

import numpy as np
import pytest
import torch

import oracle as orc
from conftest import parse_golden
from int4_expert_ffn_gb300 import synth
from helpers import REL_TOL, FmtLayer, coli, fmt_desc, rel_err, tokens_without_ties

pytestmark = pytest.mark.gpu

GOLDEN = parse_golden(os.path.join(os.path.dirname(__file__), "golden", "i4row_hand.txt"))


def gpu_quant(w):
    p, s = coli().coli_quant_i4row(w.cuda())
    torch.cuda.synchronize()
    return p.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("case", GOLDEN, ids=[c["name"] for c in GOLDEN])
def test_quant_hand_vectors(case, dtype):
    w = torch.tensor(case["w"], dtype=torch.float32).to(dtype)
    if dtype == torch.bfloat16 and not torch.equal(w.float(), torch.tensor(case["w"])):
        pytest.skip("values not exact in bf16")
    p, s = gpu_quant(w.reshape(1, -1))
    assert p.reshape(-1).tolist() == case["bytes"][0]
    assert s.view(np.uint32).reshape(-1).tolist() == case["scales"][0]


@pytest.mark.parametrize("rows,cols", [(1, 64), (64, 64), (100, 6144), (37, 2048), (33, 200),
                                       (7, 333), (5, 1), (3, 16384), (300, 129)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quant_random_with_outliers(rows, cols, dtype):
    w = synth.matrix(rows, cols, 0.02, 13, rows, cols, dtype=dtype, outliers=0.01)
    w[0] = 0                                  # an all-zero row
    if rows > 2 and cols > 40:
        w[1, 5] = float("nan")
        w[2, 3] = -0.0
    p, s = gpu_quant(w)
    op, os_ = orc.quant_i4row(w.float().cpu().numpy())
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32))
    bad = np.argwhere(p != op)
    assert bad.size == 0, "%d bytes differ, first %s" % (len(bad), bad[:3].tolist())


SHAPES = [
    # (hidden, ffn, experts, shared, top_k, tokens)
    (256, 128, 8, 1, 2, 1),
    (512, 256, 16, 2, 4, 17),
    (256, 256, 8, 0, 3, 64),
    (512, 128, 12, 1, 2, 200),
    (6144, 2048, 6, 1, 2, 5),      # the GLM-like widths
]


@pytest.mark.parametrize("H,F,E,S,k,T", SHAPES)
def test_i4row_layer(H, F, E, S, k, T):
    c = coli()
    shape = synth.MoEShape("i4r", 1, H, F, E, S, k, T, "bf16", "f32")
    prev = orc.set_threads(os.cpu_count() or 1)
    try:
        ly = FmtLayer(shape, c.COLI_FMT_I4ROW, 0, seed=9)
        x = tokens_without_ties(shape, ly.wr.double().numpy(), seed=9)
        d = fmt_desc(shape, T, c.COLI_FMT_I4ROW)
        ws = c.new_workspace(d, k)
        counts = torch.zeros(E, dtype=torch.int32, device="cuda")
        out = c.coli_moe_forward(d, k, x.cuda(), ly.wr.cuda(), ly.packed, ly.scales, ws,
                                 route_counts=counts)
        out2 = c.coli_moe_forward(d, k, x.cuda(), ly.wr.cuda(), ly.packed, ly.scales, ws)
        torch.cuda.synchronize()
        assert torch.equal(out, out2), "not deterministic"
        ocounts = np.zeros(E, np.uint32)
        ref, _, _, _ = orc.moe_forward_fmt(orc.FMT_I4ROW, x.double().numpy(),
                                           ly.wr.double().numpy(), ly.o_packed, ly.o_scales,
                                           H, F, E, S, k, ocounts)
    finally:
        orc.set_threads(prev)
    err = rel_err(out.cpu().numpy(), ref)
    assert err.max() <= REL_TOL, "max rel err %.3g" % err.max()
    assert np.array_equal(counts.cpu().numpy().astype(np.uint32), ocounts)


def test_i4row_sigmoid_router_and_stack():
    c = coli()
    shape = synth.MoEShape("i4rs", 2, 512, 256, 16, 1, 4, 6, "bf16", "f32")
    layers = [FmtLayer(shape, c.COLI_FMT_I4ROW, l, seed=10) for l in range(2)]
    biases = [synth.router_bias(shape, l, 10) for l in range(2)]
    x = tokens_without_ties(shape, layers[0].wr.double().numpy(), seed=10,
                            bias=biases[0].double().numpy())
    d = fmt_desc(shape, 6, c.COLI_FMT_I4ROW, bias=torch.cat(biases).cuda())
    ws = c.new_workspace(d, 4)
    counts = torch.zeros((2, 16), dtype=torch.int32, device="cuda")
    xo = c.coli_moe_stack_forward(d, 4, 2, x.cuda(), torch.cat([ly.wr for ly in layers]).cuda(),
                                  torch.cat([ly.packed for ly in layers]),
                                  torch.cat([ly.scales for ly in layers]), ws,
                                  route_counts=counts)
    torch.cuda.synchronize()
    xr = x.double().numpy()
    ocounts = np.zeros((2, 16), np.uint32)
    for l, ly in enumerate(layers):
        o, _, _, _ = orc.moe_forward_fmt(orc.FMT_I4ROW, xr, ly.wr.double().numpy(), ly.o_packed,
                                         ly.o_scales, 512, 256, 16, 1, 4, ocounts[l],
                                         router="sigmoid", bias=biases[l].double().numpy())
        xr = xr + o
    assert rel_err(xo.cpu().numpy(), xr).max() <= REL_TOL
    assert np.array_equal(counts.cpu().numpy().astype(np.uint32), ocounts)
