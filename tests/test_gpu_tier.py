"""Tiered expert store on the GPU: an HBM pool of expert slots plus the full
store in pinned host memory, read over the host link when an expert is not
resident.

  - placement never changes the result: every call equals coli_moe_forward on
    the all-in-HBM store bit for bit (same kernels, same arithmetic), and the
    oracle within the tolerance of the other tests;
  - the LFRU policy tick on the GPU matches the plain-Python policy oracle
    exactly (slots, heat, last use, clock, the uploads of each tick), and the
    pool holds, after every tick, the records of the experts its table names;
  - the batched path (64 tokens) reads the same store the same way;
  - a store that is not pinned host memory is refused before any launch.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle as orc
from oracle import tier as OT
from int4_expert_ffn_gb300 import synth
from helpers import Layer, REL_TOL, coli, rel_err, tokens_without_ties

pytestmark = pytest.mark.gpu


def make(shape, seed, owners, max_uploads=2):
    c = coli()
    H, F, E, S = shape.hidden, shape.ffn, shape.experts, shape.shared
    layer = Layer(shape, 0, seed, router_row_std=synth.skewed_router_std(E, H, gamma=1.0))
    packed, scales, wr = layer.gpu()
    host_p = packed.cpu().pin_memory()
    host_s = scales.cpu().pin_memory()
    desc = c.MoEDesc(H, F, E, S, shape.tokens, c.COLI_F32, c.COLI_BF16)
    tier = c.Tier(desc, owners, max_uploads=max_uploads)
    c.coli_tier_place(desc, host_p, host_s, tier)
    return layer, packed, scales, wr, host_p, host_s, desc, tier


def check_pool(c, tier, packed, scales, shape):
    eb = c.coli_expert_packed_bytes(shape.hidden, shape.ffn)
    es = c.coli_expert_scale_count(shape.hidden, shape.ffn)
    owners = tier.slot_owner.cpu().tolist()
    for sl, e in enumerate(owners):
        if e < 0:
            continue
        assert torch.equal(tier.pool_packed[sl * eb:(sl + 1) * eb], packed[e * eb:(e + 1) * eb])
        assert torch.equal(tier.pool_scales[sl * es:(sl + 1) * es], scales[e * es:(e + 1) * es])


def test_tiered_forward_and_policy_match():
    c = coli()
    shape = synth.MoEShape("tier", 1, 512, 512, 16, 1, 4, 2, "bf16", "f32")
    E = shape.experts
    owners = [E, 3, 5, -1, -1, -1]                 # the shared expert, two routed, three free
    layer, packed, scales, wr, host_p, host_s, desc, tier = make(shape, 21, owners)
    torch.cuda.synchronize()
    check_pool(c, tier, packed, scales, shape)
    ws = c.new_workspace(desc, shape.top_k)
    ws2 = c.new_workspace(desc, shape.top_k)
    o_packed, o_scales, o_wr = layer.oracle()
    pol = OT.TierState(E, shape.shared, owners)
    n_up = 0
    for tick in range(16):
        x = tokens_without_ties(shape, o_wr, seed=21, step=tick).cuda()
        counts = torch.zeros(E, dtype=torch.int32, device="cuda")
        out = c.coli_moe_forward_tiered(desc, shape.top_k, x, wr, host_p, host_s, tier, ws,
                                        route_counts=counts)
        ref = c.coli_moe_forward(desc, shape.top_k, x, wr, packed, scales, ws2)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), "tick %d: placement changed the result" % tick
        cnt = counts.cpu().numpy().astype(np.uint32)
        if tick % 4 == 0:
            ocounts = np.zeros(E, np.uint32)
            oref, _, _, _ = orc.moe_forward(x.double().cpu().numpy(), o_wr, o_packed, o_scales,
                                            shape.hidden, shape.ffn, E, shape.shared,
                                            shape.top_k, ocounts)
            assert rel_err(out.cpu().numpy(), oref).max() <= REL_TOL
            assert np.array_equal(cnt, ocounts)
        c.coli_tier_update(desc, counts, host_p, host_s, tier)
        want = pol.tick(cnt.tolist(), tier.max_uploads)
        torch.cuda.synchronize()
        up = tier.uploads.cpu().numpy().view(np.uint32)
        got = [(int(up[1 + 2 * i]), int(up[2 + 2 * i])) for i in range(int(up[0]))]
        assert got == want, "tick %d uploads %s vs %s" % (tick, got, want)
        assert tier.slot_owner.cpu().tolist() == pol.owner
        assert tier.slot_of.cpu().tolist() == pol.slot_of
        assert tier.heat.cpu().numpy().view(np.uint32).tolist() == pol.heat
        assert tier.last.cpu().numpy().view(np.uint32).tolist() == pol.last
        assert int(tier.clock.cpu().numpy().view(np.uint32)[0]) == pol.clock
        check_pool(c, tier, packed, scales, shape)
        n_up += len(got)
    assert n_up >= 2, "no expert earned a slot in 16 ticks"


def test_tiered_batched_path_reads_the_same_store():
    c = coli()
    shape = synth.MoEShape("tierb", 1, 512, 256, 12, 1, 3, 64, "bf16", "f32")
    E = shape.experts
    layer, packed, scales, wr, host_p, host_s, desc, tier = make(shape, 22, [E, 0, 4, 7, -1])
    x = synth.tokens(shape, 22).cuda()
    ws = c.new_workspace(desc, shape.top_k)
    out = c.coli_moe_forward_tiered(desc, shape.top_k, x, wr, host_p, host_s, tier, ws)
    ref = c.coli_moe_forward(desc, shape.top_k, x, wr, packed, scales, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_tiered_store_must_be_pinned_host_memory():
    c = coli()
    shape = synth.MoEShape("tierv", 1, 512, 512, 8, 1, 2, 1, "bf16", "f32")
    layer, packed, scales, wr, host_p, host_s, desc, tier = make(shape, 23, [-1, -1])
    ws = c.new_workspace(desc, 2)
    x = synth.tokens(shape, 23).cuda()
    out = torch.empty((1, 512), device="cuda")
    d, t = desc.c(), tier.c()
    # device memory given as the host store: refused before any launch
    st = c.lib.coli_moe_forward_tiered(C.byref(d), 2, x.data_ptr(), wr.data_ptr(),
                                       packed.data_ptr(), scales.data_ptr(), C.byref(t),
                                       out.data_ptr(), None, ws.data_ptr(), ws.numel(), None)
    assert st == c.COLI_EINVAL
