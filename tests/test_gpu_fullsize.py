"""Parity at the decode workloads' full sizes, in the launch configuration the
benchmark times (one stack call per step for chained stacks, one layer call
per layer otherwise):

  - the 16-layer OLMoE-like stack (hidden 2048, 64 experts of width 1024,
    top-8, no shared expert, bf16 router) at batch 1;
  - GLM-like layers (hidden 6144, 256 experts of width 2048, top-8, one shared
    expert, bf16 router) at batch 1 and batch 8: layer calls on independent
    inputs (as the benchmark runs them), and the stack entry point two deep.

Weights are drawn on the device by the seeded generator and quantised there by
the library.  The oracle quantises, from the same bf16 values, only the experts
its own routing selects (plus one rank of margin); the other experts' bytes stay
zero in its copy.  Outputs are compared per token within 2e-3 relative error,
route counts bit-exact.  Tokens are drawn (by attempt index) until the oracle's
own chain has no near-tie in any layer's top-k, so that the 15-bit activation
rounding of the GPU path cannot flip a selection.  Each GPU call runs three
times and must give bit-identical results.
"""
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_ffn_gb300 import synth
from helpers import REL_TOL, coli, layer_geometry, min_topk_gap, quant_gpu_into, quant_oracle, rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

CHAIN_GAP = 2e-3     # min top-k gap along the oracle chain (>> GPU logit error ~1e-4)
SEED = 0


class DeviceStack:
    """Quantised experts and routers of a stack, resident on the GPU."""

    def __init__(self, shape, seed=SEED):
        c = coli()
        L, H, F, E, S = shape.layers, shape.hidden, shape.ffn, shape.experts, shape.shared
        eb, es = layer_geometry(H, F)
        self.packed = torch.empty(L * (E + S) * eb, dtype=torch.uint8, device="cuda")
        self.scales = torch.empty(L * (E + S) * es, dtype=torch.float32, device="cuda")
        for l in range(L):
            p0, s0 = l * (E + S) * eb, l * (E + S) * es
            for e in range(E + S):
                mats = [synth.expert_matrix(shape, l, e, m, seed, device="cuda") for m in range(3)]
                p0, s0 = quant_gpu_into(mats, self.packed, self.scales, p0, s0)
        self.router = torch.stack([synth.router_weights(shape, l, seed, device="cuda")
                                   for l in range(L)]).contiguous()
        torch.cuda.synchronize()


class OracleLayer:
    """One layer for the oracle: its router in float64, and experts quantised on
    demand from the same device-drawn bf16 values."""

    def __init__(self, shape, layer, router_dev, seed=SEED):
        H, F, E, S = shape.hidden, shape.ffn, shape.experts, shape.shared
        self.shape, self.layer, self.seed = shape, layer, seed
        self.eb, self.es = layer_geometry(H, F)
        self.packed = np.zeros((E + S) * self.eb, np.uint8)     # pages stay untouched
        self.scales = np.zeros((E + S) * self.es, np.float32)
        self.wr = router_dev.double().cpu().numpy()
        self.done = set()
        self.need(range(E, E + S))

    def need(self, experts):
        for e in experts:
            e = int(e)
            if e in self.done:
                continue
            mats = [synth.expert_matrix(self.shape, self.layer, e, m, self.seed, device="cuda")
                    for m in range(3)]
            p, s = quant_oracle(mats)
            self.packed[e * self.eb:(e + 1) * self.eb] = p
            self.scales[e * self.es:(e + 1) * self.es] = s
            self.done.add(e)


def oracle_chain(shape, layers, x0):
    """x_{l+1} = x_l + MoE_l(x_l) in the oracle; None if some layer has a near-tie."""
    H, F, E, S, k = shape.hidden, shape.ffn, shape.experts, shape.shared, shape.top_k
    x = np.asarray(x0, np.float64)
    outs, counts = [], np.zeros((len(layers), E), np.uint32)
    for l, ol in enumerate(layers):
        lg = orc.router_logits(x, ol.wr)
        if min_topk_gap(lg, k) < CHAIN_GAP:
            return None
        ol.need(np.unique(np.argsort(-lg, axis=1)[:, :k + 1]))
        out, _, _, _ = orc.moe_forward(x, ol.wr, ol.packed, ol.scales, H, F, E, S, k, counts[l])
        outs.append(out)
        x = x + out
    return x, outs, counts


def check_stack(shape, n_steps):
    c = coli()
    dev_stack = DeviceStack(shape)
    layers = [OracleLayer(shape, l, dev_stack.router[l]) for l in range(shape.layers)]
    T, L, H, E = shape.tokens, shape.layers, shape.hidden, shape.experts
    desc = c.MoEDesc(H, shape.ffn, E, shape.shared, T, c.COLI_F32,
                     c.COLI_BF16 if shape.router_dtype == "bf16" else c.COLI_F32)
    ws = c.new_workspace(desc, shape.top_k)
    checked = 0
    for step in range(n_steps):
        for attempt in range(40):
            x = synth.tokens(shape, SEED, step, attempt=attempt)
            ref = oracle_chain(shape, layers, x.double().numpy())
            if ref is not None:
                break
        else:
            raise RuntimeError("no tie-free token chain found")
        x_ref, outs_ref, counts_ref = ref
        results = []
        for _ in range(3):
            counts = torch.zeros((L, E), dtype=torch.int32, device="cuda")
            layer_out = torch.empty((L, T, H), dtype=torch.float32, device="cuda")
            xo = c.coli_moe_stack_forward(desc, shape.top_k, L, x.cuda(), dev_stack.router,
                                          dev_stack.packed, dev_stack.scales, ws,
                                          layer_out=layer_out, route_counts=counts)
            torch.cuda.synchronize()
            results.append((xo.cpu(), layer_out.cpu(), counts.cpu()))
        for r in results[1:]:
            assert all(torch.equal(a, b) for a, b in zip(r, results[0])), "not deterministic"
        xo, layer_out, counts = results[0]
        assert np.array_equal(counts.numpy().astype(np.uint32), counts_ref), "route counts differ"
        for l in range(L):
            err = rel_err(layer_out[l].numpy(), outs_ref[l])
            assert err.max() <= REL_TOL, "layer %d: max rel err %.3g" % (l, err.max())
        assert rel_err(xo.numpy(), x_ref).max() <= REL_TOL
        checked += 1
    assert checked == n_steps


def check_layers(shape, n_layers):
    """Unchained stacks: every layer call on its own tie-free input, against
    the oracle layer by layer (coli_moe_forward, as the benchmark calls it)."""
    c = coli()
    shape = dataclasses.replace(shape, layers=n_layers)
    dev_stack = DeviceStack(shape)
    T, H, F, E, S, k = shape.tokens, shape.hidden, shape.ffn, shape.experts, shape.shared, shape.top_k
    eb, es = layer_geometry(H, F)
    desc = c.MoEDesc(H, F, E, S, T, c.COLI_F32, c.COLI_BF16)
    ws = c.new_workspace(desc, k)
    for l in range(n_layers):
        ol = OracleLayer(shape, l, dev_stack.router[l])
        for attempt in range(40):
            x = synth.tokens(shape, SEED, 0, attempt=attempt, layer=l)
            lg = orc.router_logits(x.double().numpy(), ol.wr)
            if min_topk_gap(lg, k) >= CHAIN_GAP:
                break
        else:
            raise RuntimeError("no tie-free input found")
        ol.need(np.unique(np.argsort(-lg, axis=1)[:, :k + 1]))
        ocounts = np.zeros(E, np.uint32)
        ref, _, _, _ = orc.moe_forward(x.double().numpy(), ol.wr, ol.packed, ol.scales, H, F, E,
                                       S, k, ocounts)
        packed = dev_stack.packed[l * (E + S) * eb:(l + 1) * (E + S) * eb]
        scales = dev_stack.scales[l * (E + S) * es:(l + 1) * (E + S) * es]
        results = []
        for _ in range(3):
            counts = torch.zeros(E, dtype=torch.int32, device="cuda")
            out = c.coli_moe_forward(desc, k, x.cuda(), dev_stack.router[l], packed, scales, ws,
                                     route_counts=counts)
            torch.cuda.synchronize()
            results.append((out.cpu(), counts.cpu()))
        for r in results[1:]:
            assert all(torch.equal(a, b) for a, b in zip(r, results[0])), "not deterministic"
        out, counts = results[0]
        assert np.array_equal(counts.numpy().astype(np.uint32), ocounts)
        err = rel_err(out.numpy(), ref)
        assert err.max() <= REL_TOL, "layer %d: max rel err %.3g" % (l, err.max())


def test_olmoe_stack_batch1():
    check_stack(synth.OLMOE_DECODE, n_steps=3)


@pytest.mark.parametrize("shape", [synth.GLM_DECODE_B1, synth.GLM_DECODE_B8],
                         ids=lambda s: s.name)
def test_glm_layer_calls(shape):
    check_layers(shape, n_layers=2)


@pytest.mark.parametrize("T", [1, 8])
def test_glm_stack_two_deep(T):
    """The stack entry point at the GLM-like layer shape (two layers stay far
    from the overflow a longer unnormalised chain of these layers reaches)."""
    shape = dataclasses.replace(synth.GLM_DECODE_B1, layers=2, tokens=T, chained=True)
    check_stack(shape, n_steps=1)


def prefill_tokens_without_ties(shape, wr64, seed=SEED, step=0, gap=1e-4, max_attempts=40):
    """The prefill batch with every near-tie token redrawn on its own: token t is
    row t of the attempt-a_t draw, a_t the first attempt whose top-(k+1) f32
    logits of that token have adjacent gaps above ``gap``."""
    k = shape.top_k
    x = synth.tokens(shape, seed, step)                  # attempt 0, host bf16 [T, H]
    lg = orc.router_logits(x.double().numpy(), wr64)
    todo = np.array([t for t in range(x.shape[0]) if min_topk_gap(lg[t:t + 1], k) <= gap])
    for attempt in range(1, max_attempts):
        if todo.size == 0:
            return x, lg
        xa = synth.tokens(shape, seed, step, attempt=attempt)[todo]
        la = orc.router_logits(xa.double().numpy(), wr64)
        ok = np.array([min_topk_gap(la[i:i + 1], k) > gap for i in range(len(todo))])
        x[todo[ok]] = xa[ok]
        lg[todo[ok]] = la[ok]
        todo = todo[~ok]
    raise RuntimeError("%d tokens kept a near-tie" % todo.size)


def test_glm_prefill_tie_free():
    """The batched path at the prefill workload: one GLM-like layer, 4096 bf16
    tokens, a router skewed so that 32 experts take about half of the routes,
    every token redrawn until its top-(k+1) logits are tie-free (gap > 1e-4).
    Route counts must equal the oracle's bit for bit.  Outputs are compared with
    the oracle on at least 512 tokens that include, for every expert with
    routes, the token of its first route (its first 128-route m-tile) and the
    token of its last route (its last, partial m-tile)."""
    c = coli()
    shape = synth.GLM_PREFILL
    T, H, F, E, S, k = shape.tokens, shape.hidden, shape.ffn, shape.experts, shape.shared, shape.top_k
    eb, es = layer_geometry(H, F)
    packed = torch.empty((E + S) * eb, dtype=torch.uint8, device="cuda")
    scales = torch.empty((E + S) * es, dtype=torch.float32, device="cuda")
    p0 = s0 = 0
    for e in range(E + S):
        mats = [synth.expert_matrix(shape, 0, e, m, SEED, device="cuda") for m in range(3)]
        p0, s0 = quant_gpu_into(mats, packed, scales, p0, s0)
    wr = synth.router_weights(shape, 0, SEED, device="cuda",
                              row_std=synth.skewed_router_std(E, H))
    prev = orc.set_threads(os.cpu_count() or 1)
    try:
        ol = OracleLayer(shape, 0, wr)
        x, lg = prefill_tokens_without_ties(shape, ol.wr)
        desc = c.MoEDesc(H, F, E, S, T, c.COLI_BF16, c.COLI_BF16)
        ws = c.new_workspace(desc, k)
        counts = torch.zeros(E, dtype=torch.int32, device="cuda")
        out = c.coli_moe_forward(desc, k, x.cuda(), wr, packed, scales, ws, route_counts=counts)
        out2 = c.coli_moe_forward(desc, k, x.cuda(), wr, packed, scales, ws)
        torch.cuda.synchronize()
        assert torch.equal(out, out2), "not deterministic"
        # routing of all 4096 tokens: the oracle's top-k, counted
        idx = np.stack([orc.topk(lg[t], k)[0] for t in range(T)])
        ocounts = np.bincount(idx.reshape(-1), minlength=E)
        assert np.array_equal(counts.cpu().numpy().astype(np.int64), ocounts), "route counts differ"
        assert np.sort(ocounts)[::-1][:32].sum() > 0.4 * T * k, "router not skewed"
        # tokens to compare: first and last route of every routed expert, then
        # random tokens up to 512
        sample = set()
        for e in range(E):
            toks = np.nonzero((idx == e).any(axis=1))[0]
            if toks.size:
                sample.update((int(toks[0]), int(toks[-1])))
        sample.update((0, T - 1))                        # the shared expert's first and last tile
        for t in np.random.default_rng(1).permutation(T):
            if len(sample) >= 512:
                break
            sample.add(int(t))
        sample = np.array(sorted(sample))
        ol.need(np.unique(idx[sample]))
        ref, ridx, _, _ = orc.moe_forward(x.double().numpy()[sample], ol.wr, ol.packed, ol.scales,
                                          H, F, E, S, k)
        assert np.array_equal(ridx, idx[sample])
        err = rel_err(out.cpu().numpy()[sample], ref)
        assert err.max() <= REL_TOL, "max rel err %.3g (token %d)" % (err.max(),
                                                                  sample[int(np.argmax(err))])
    finally:
        orc.set_threads(prev)
