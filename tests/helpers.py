"""Shared helpers for the GPU parity tests: build a layer's weights once, quantise
them with the library (GPU) and independently with the oracle (CPU), draw token
inputs without routing near-ties, and compare outputs."""
import numpy as np
import torch

import oracle as orc
from int4_expert_ffn_gb300 import synth

REL_TOL = 2e-3          # max relative error per token, ||y - r||_inf / ||r||_inf
TIE_GAP = 1e-4          # min gap between adjacent sorted logits over ranks 0..k


def coli():
    import int4_expert_ffn_gb300 as pkg
    return pkg.binding


def layer_geometry(H, F):
    c = coli()
    return c.coli_expert_packed_bytes(H, F), c.coli_expert_scale_count(H, F)


def quant_gpu_into(mats, packed, scales, p0=0, s0=0):
    """Quantise a list of matrices (device) with the library, appending them to
    the flat packed/scales buffers at byte/element offsets p0/s0."""
    c = coli()
    for m in mats:
        rows, cols = m.shape
        nb, ns = rows * c.coli_packed_row_bytes(cols), rows * c.coli_scales_per_row(cols)
        c.coli_quant_i4g(m, packed[p0:p0 + nb].view(rows, -1), scales[s0:s0 + ns].view(rows, -1))
        p0 += nb
        s0 += ns
    return p0, s0


def quant_oracle(mats):
    """Oracle quantisation of host matrices -> flat numpy arrays in record order."""
    ps, ss = [], []
    for m in mats:
        p, s = orc.quant_i4g(m.float().cpu().numpy())
        ps.append(p.reshape(-1))
        ss.append(s.reshape(-1))
    return np.concatenate(ps), np.concatenate(ss)


class Layer:
    """One MoE layer's inputs drawn on the host (small shapes)."""

    def __init__(self, shape, layer=0, seed=0, router_row_std=None):
        self.shape = shape
        E, S = shape.experts, shape.shared
        self.mats = [[synth.expert_matrix(shape, layer, e, m, seed) for m in range(3)]
                     for e in range(E + S)]
        self.wr = synth.router_weights(shape, layer, seed, row_std=router_row_std)

    def flat_mats(self):
        return [m for ms in self.mats for m in ms]

    def gpu(self, dev="cuda"):
        H, F = self.shape.hidden, self.shape.ffn
        n = self.shape.experts + self.shape.shared
        eb, es = layer_geometry(H, F)
        packed = torch.empty(n * eb, dtype=torch.uint8, device=dev)
        scales = torch.empty(n * es, dtype=torch.float32, device=dev)
        quant_gpu_into([m.to(dev) for m in self.flat_mats()], packed, scales)
        return packed, scales, self.wr.to(dev)

    def oracle(self):
        p, s = quant_oracle(self.flat_mats())
        return p, s, self.wr.double().numpy()


class FmtLayer:
    """One MoE layer in another container (COLI_FMT_MXFP4, COLI_FMT_FP8 or
    COLI_FMT_I4ROW): quantised on the GPU and, independently, by the oracle;
    the two records must agree byte for byte."""

    def __init__(self, shape, fmt, layer=0, seed=0):
        c = coli()
        H, F, E, S = shape.hidden, shape.ffn, shape.experts, shape.shared
        gpu_q, orc_q, sdt = {
            c.COLI_FMT_MXFP4: (c.coli_quant_mxfp4, orc.quant_mxfp4, torch.uint8),
            c.COLI_FMT_FP8: (c.coli_quant_fp8b128, orc.quant_fp8b128, torch.float32),
            c.COLI_FMT_I4ROW: (c.coli_quant_i4row, orc.quant_i4row, torch.float32),
        }[fmt]
        self.shape, self.fmt = shape, fmt
        mats = [synth.expert_matrix(shape, layer, e, m, seed) for e in range(E + S)
                for m in range(3)]
        esz = torch.tensor([], dtype=sdt).element_size()
        eb = c.coli_fmt_expert_bytes(fmt, H, F)
        es = c.coli_fmt_expert_scale_bytes(fmt, H, F) // esz
        self.packed = torch.empty((E + S) * eb, dtype=torch.uint8, device="cuda")
        self.scales = torch.empty((E + S) * es, dtype=sdt, device="cuda")
        p0 = s0 = 0
        ops, oss = [], []
        for m in mats:
            rows, cols = m.shape
            nb = rows * c.lib.coli_fmt_row_bytes(fmt, cols)
            ns = rows * c.lib.coli_fmt_scale_bytes(fmt, cols) // esz
            gpu_q(m.cuda(), self.packed[p0:p0 + nb].view(rows, -1),
                  self.scales[s0:s0 + ns].view(rows, -1))
            p0, s0 = p0 + nb, s0 + ns
            a, b = orc_q(m.float().numpy())
            ops.append(a.reshape(-1))
            oss.append(b.reshape(-1))
        self.o_packed, self.o_scales = np.concatenate(ops), np.concatenate(oss)
        self.wr = synth.router_weights(shape, layer, seed)
        torch.cuda.synchronize()
        assert np.array_equal(self.packed.cpu().numpy(), self.o_packed)
        assert np.array_equal(self.scales.cpu().numpy().view(np.uint8),
                              self.o_scales.view(np.uint8))


def fmt_desc(shape, T, fmt, bias=None, x_dtype=None):
    """Layer descriptor for weights in container fmt (softmax router unless a
    sigmoid-router bias is given)."""
    c = coli()
    args = [shape.hidden, shape.ffn, shape.experts, shape.shared, T,
            c.COLI_F32 if (x_dtype or torch.float32) == torch.float32 else c.COLI_BF16,
            c.COLI_F32 if shape.router_dtype == "f32" else c.COLI_BF16]
    if bias is not None:
        args += [c.COLI_ROUTER_SIGMOID_BIAS, bias]
    else:
        args += [c.COLI_ROUTER_SOFTMAX, None]
    return c.MoEDesc(*args, weight_fmt=fmt)


def min_topk_gap(logits, k):
    """Smallest adjacent gap among the k+1 largest logits of each row (f32 ranking)."""
    lg = np.sort(logits.astype(np.float32), axis=1)[:, ::-1]
    kk = min(k + 1, lg.shape[1])
    if kk < 2:
        return np.inf
    return float(np.min(lg[:, :kk - 1] - lg[:, 1:kk]))


def selection_keys(logits, bias):
    """Ranking keys of the sigmoid router: sigmoid(logit) + bias (f64)."""
    return 1.0 / (1.0 + np.exp(-logits)) + np.asarray(bias, np.float64)[None, :]


def tokens_without_ties(shape, wr64, seed=0, step=0, T=None, dtype=None, bias=None):
    """Layer input drawn with the next attempt index until no near-tie (of the
    logits, or with ``bias`` of the sigmoid router's keys)."""
    for attempt in range(50):
        x = synth.tokens(shape, seed, step, attempt=attempt)
        if T is not None:
            x = x[:T]
        if dtype is not None:
            x = x.to(dtype)
        lg = orc.router_logits(x.double().numpy(), wr64)
        keys = lg if bias is None else selection_keys(lg, bias)
        if min_topk_gap(keys, shape.top_k) > TIE_GAP:
            return x
    raise RuntimeError("could not draw tie-free tokens")


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(got - ref).max(axis=-1) / np.abs(ref).max(axis=-1)
