"""coli_moe_forward_noalloc: the layer forward for callers that cannot allocate
device memory (hosts that pre-budget every byte of the device, loops that must
never reach cudaMalloc).  It must give exactly what coli_moe_forward gives, call
after call, while using only the library's fixed scratch array, and match the
oracle within the tolerance of the other parity tests.

This file is collected last on purpose: it also has to pass after every other
GPU test has run in the same process, and alone in a fresh one.
"""
import ctypes as C
import dataclasses

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_ffn_gb300 import synth
from helpers import Layer, REL_TOL, coli, rel_err, tokens_without_ties

pytestmark = pytest.mark.gpu

CASES = [
    dataclasses.replace(synth.TINY, tokens=4),
    dataclasses.replace(synth.OLMOE_DECODE, tokens=1),
    synth.MoEShape("ragged", 1, 320, 192, 12, 2, 3, 21, "bf16", "f32"),
    # 64 tokens at hidden 256: the batched (tensor-core) path, whose workspace
    # also fits in the fixed array
    dataclasses.replace(synth.TINY, name="tiny_batched", tokens=64),
]


def _noalloc(c, d, k, x, wr, packed, scales, out, counts):
    return c.lib.coli_moe_forward_noalloc(
        C.byref(d), k, x.data_ptr(), wr.data_ptr(), packed.data_ptr(), scales.data_ptr(),
        out.data_ptr(), counts.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape", CASES, ids=[s.name for s in CASES])
def test_noalloc_matches_workspace_entry_point(shape):
    c = coli()
    layer = Layer(shape, 0, seed=3)
    packed, scales, wr = layer.gpu()
    x = tokens_without_ties(shape, layer.wr.double().numpy(), seed=3).cuda()
    desc = c.MoEDesc(shape.hidden, shape.ffn, shape.experts, shape.shared, shape.tokens,
                     c.COLI_F32, c.COLI_F32 if shape.router_dtype == "f32" else c.COLI_BF16)
    assert c.coli_moe_workspace_size(desc, shape.top_k) <= (4 << 20)
    ws = c.new_workspace(desc, shape.top_k)
    counts_ref = torch.zeros(shape.experts, dtype=torch.int32, device="cuda")
    ref = c.coli_moe_forward(desc, shape.top_k, x, wr, packed, scales, ws,
                             route_counts=counts_ref)
    torch.cuda.synchronize()
    # the oracle on the same tokens (its own quantisation of the same weights)
    o_packed, o_scales, o_wr = layer.oracle()
    o_counts = np.zeros(shape.experts, np.uint32)
    o_out, _, _, _ = orc.moe_forward(x.double().cpu().numpy(), o_wr, o_packed, o_scales,
                                     shape.hidden, shape.ffn, shape.experts, shape.shared,
                                     shape.top_k, o_counts)
    counts = torch.zeros(shape.experts, dtype=torch.int32, device="cuda")
    d = desc.c()
    for call in range(2):                 # two calls in a row share the scratch
        out = torch.full((shape.tokens, shape.hidden), float("nan"), device="cuda")
        st = _noalloc(c, d, shape.top_k, x, wr, packed, scales, out, counts)
        assert st == c.COLI_OK, c.lib.coli_status_str(st)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: bit-identical to the workspace call
        assert torch.equal(out, ref), "call %d differs from coli_moe_forward" % call
        err = rel_err(out.cpu().numpy(), o_out)
        assert err.max() <= REL_TOL, "call %d: rel err %.3g vs the oracle" % (call, err.max())
        assert np.array_equal(counts.cpu().numpy(), (call + 1) * counts_ref.cpu().numpy())
    assert np.array_equal(counts_ref.cpu().numpy().astype(np.uint32), o_counts)


def test_noalloc_rejects_oversized_scratch():
    c = coli()
    # 16 tokens x (8 + 8) slots x F=16384 f32 intermediates: far above 4 MiB
    desc = c.MoEDesc(1024, 16384, 64, 8, 16, c.COLI_F32, c.COLI_BF16)
    assert c.coli_moe_workspace_size(desc, 8) > (4 << 20)
    d = desc.c()
    fake = C.c_void_p(0x1000)   # never touched: the size check comes first
    st = c.lib.coli_moe_forward_noalloc(C.byref(d), 8, fake, fake, fake, fake, fake, None, None)
    assert st == c.COLI_ENOMEM
