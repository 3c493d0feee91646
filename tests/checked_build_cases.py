"""Run by tests/test_gpu_checked_build.py in a child process with
COLI_LIBRARY=check: layer calls over the paths whose indices come from data
(routing, union lists, the batched grouping, the one-token layer kernel, the
other containers, a chained stack), each compared with the oracle and each
required to leave no flag in the workspace (COLI_FLAG_BOUNDS in particular).
Prints one line per case; exits non-zero on the first failure."""
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import oracle as orc  # noqa: E402
from int4_expert_ffn_gb300 import synth  # noqa: E402
from helpers import REL_TOL, FmtLayer, Layer, coli, fmt_desc, rel_err, tokens_without_ties  # noqa: E402


def check_layer(name, H, F, E, S, k, T, xdt="f32", rdt="bf16"):
    c = coli()
    assert c.LIB_PATH.endswith("libcoli_check.so"), c.LIB_PATH
    shape = synth.MoEShape(name, 1, H, F, E, S, k, T, rdt, xdt)
    layer = Layer(shape, 0, 3)
    packed, scales, wr = layer.gpu()
    op, os_, owr = layer.oracle()
    x = tokens_without_ties(shape, owr, 3)
    d = c.MoEDesc(H, F, E, S, T, c.COLI_BF16 if xdt == "bf16" else c.COLI_F32,
                  c.COLI_BF16 if rdt == "bf16" else c.COLI_F32)
    ws = c.new_workspace(d, k)
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    out = c.coli_moe_forward(d, k, x.cuda(), wr, packed, scales, ws, route_counts=counts)
    torch.cuda.synchronize()
    flags = c.coli_moe_check(ws)
    assert flags == 0, "%s: flags %#x" % (name, flags)
    ocounts = np.zeros(E, np.uint32)
    ref, _, _, _ = orc.moe_forward(x.double().numpy(), owr, op, os_, H, F, E, S, k, ocounts)
    assert np.array_equal(counts.cpu().numpy(), ocounts), name
    err = rel_err(out.cpu().numpy(), ref).max()
    assert err <= REL_TOL, "%s: rel err %.3g" % (name, err)
    print("ok", name, "%.2e" % err, flush=True)


def check_fmt(name, fmt, H, F, E, S, k, T):
    c = coli()
    shape = synth.MoEShape(name, 1, H, F, E, S, k, T, "bf16", "f32")
    ly = FmtLayer(shape, fmt, 0, seed=4)
    x = tokens_without_ties(shape, ly.wr.double().numpy(), seed=4)
    d = fmt_desc(shape, T, fmt)
    ws = c.new_workspace(d, k)
    out = c.coli_moe_forward(d, k, x.cuda(), ly.wr.cuda(), ly.packed, ly.scales, ws)
    torch.cuda.synchronize()
    flags = c.coli_moe_check(ws)
    assert flags == 0, "%s: flags %#x" % (name, flags)
    ofmt = {c.COLI_FMT_MXFP4: orc.FMT_MXFP4, c.COLI_FMT_FP8: orc.FMT_FP8,
            c.COLI_FMT_I4ROW: orc.FMT_I4ROW}[fmt]
    ref, _, _, _ = orc.moe_forward_fmt(ofmt, x.double().numpy(), ly.wr.double().numpy(),
                                       ly.o_packed, ly.o_scales, H, F, E, S, k)
    err = rel_err(out.cpu().numpy(), ref).max()
    assert err <= REL_TOL, "%s: rel err %.3g" % (name, err)
    print("ok", name, "%.2e" % err, flush=True)


def check_stack(name, L, H, F, E, S, k, T):
    c = coli()
    shape = synth.MoEShape(name, L, H, F, E, S, k, T, "bf16", "f32")
    layers = [Layer(shape, l, 2) for l in range(L)]
    gp = [ly.gpu() for ly in layers]
    ol = [ly.oracle() for ly in layers]
    x = synth.tokens(shape, 2, 0)
    d = c.MoEDesc(H, F, E, S, T, c.COLI_F32, c.COLI_BF16)
    ws = c.new_workspace(d, k)
    xo = c.coli_moe_stack_forward(d, k, L, x.cuda(), torch.cat([g[2] for g in gp]),
                                  torch.cat([g[0] for g in gp]), torch.cat([g[1] for g in gp]), ws)
    torch.cuda.synchronize()
    flags = c.coli_moe_check(ws)
    assert flags == 0, "%s: flags %#x" % (name, flags)
    xL, _, _ = orc.moe_stack_forward(x.double().numpy(), [(w, p, s) for p, s, w in ol],
                                     H, F, E, S, k)
    err = rel_err(xo.cpu().numpy(), xL).max()
    assert err <= REL_TOL, "%s: rel err %.3g" % (name, err)
    print("ok", name, "%.2e" % err, flush=True)


def main():
    c = coli()
    check_layer("gemv_one_token", 1536, 512, 64, 1, 6, 1)            # first-layer router in k_gateup
    check_layer("layer_kernel_one_token", 1024, 1024, 16, 1, 4, 1)   # one fused kernel per layer
    check_layer("gemv_several_tokens", 512, 256, 32, 2, 4, 9)
    check_layer("gemv_passes", 256, 512, 8, 1, 2, 37)                # 16-token passes, ragged tail
    check_layer("ticket_routing", 256, 256, 300, 0, 8, 9)            # T * E > 2048: partials + ticket
    check_layer("batched", 512, 256, 16, 1, 4, 200, xdt="bf16")      # grouped GEMMs, tensor-core logits
    check_layer("batched_f32", 768, 256, 32, 1, 8, 130)
    check_fmt("mxfp4_one_token", c.COLI_FMT_MXFP4, 512, 256, 16, 1, 4, 1)
    check_fmt("fp8_batched", c.COLI_FMT_FP8, 512, 256, 16, 1, 4, 70)
    check_fmt("i4row", c.COLI_FMT_I4ROW, 256, 128, 8, 1, 2, 5)
    check_stack("stack_one_token", 3, 1536, 1024, 32, 1, 4, 1)
    check_stack("stack_layer_kernel", 3, 1024, 1024, 16, 0, 4, 1)
    print("all cases passed", flush=True)


if __name__ == "__main__":
    main()
