"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module draws random numbers and lays them out; it holds none of the
method's arithmetic (no quantisation, routing or expert math).  Every draw is
keyed by (seed, sub-keys) so that any single tensor -- one expert's matrix of
one layer, say -- can be regenerated on its own.

Host draws use numpy's PCG64; device draws (used for the multi-GB workloads
that would take minutes to draw on the host) use torch's CUDA generator.  A
given tensor is always drawn on one side and copied to the other, so both the
CUDA path and the oracle see the same values.
"""
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

# ---------------------------------------------------------------------------
# Workload shapes (the pages' model families, scaled as stated).


@dataclass(frozen=True)
class MoEShape:
    name: str
    layers: int
    hidden: int
    ffn: int
    experts: int
    shared: int
    top_k: int
    tokens: int
    router_dtype: str  # "f32" | "bf16"
    x_dtype: str       # "f32" | "bf16"
    steps: int = 1     # sequential decode steps (fresh input each)
    # decode stacks: layer l > 0 takes x_l + MoE_l(x_l) of the layer before
    # (True), or its own fresh N(0, 1) draw for the step (False)
    chained: bool = True


TINY = MoEShape("tiny", 1, 256, 512, 8, 1, 2, 4, "f32", "f32")
OLMOE_DECODE = MoEShape("olmoe_decode", 16, 2048, 1024, 64, 0, 8, 1, "bf16", "f32", steps=256)
# Without the normalisation a real model applies before each MoE layer, a
# residual chain of these wide SwiGLU layers grows without bound (the FFN is
# quadratic in its input) and overflows f32 within eight layers, so each layer
# of a step gets its own unit-variance input.
GLM_DECODE_B1 = MoEShape("glm_decode_b1", 8, 6144, 2048, 256, 1, 8, 1, "bf16", "f32",
                         chained=False)
GLM_DECODE_B8 = MoEShape("glm_decode_b8", 8, 6144, 2048, 256, 1, 8, 8, "bf16", "f32",
                         chained=False)
GLM_PREFILL = MoEShape("glm_prefill", 1, 6144, 2048, 256, 1, 8, 4096, "bf16", "bf16")

SHAPES = {s.name: s for s in (TINY, OLMOE_DECODE, GLM_DECODE_B1, GLM_DECODE_B8, GLM_PREFILL)}

EXPERT_STD = 0.02  # expert weights N(0, 0.02)

# sub-key tags
_T_X, _T_ROUTER, _T_EXPERT, _T_OUTLIER, _T_BIAS = 1, 2, 3, 4, 5
MAT_GATE, MAT_UP, MAT_DOWN = 0, 1, 2


def _seq(seed, *keys):
    return np.random.SeedSequence([int(seed)] + [int(k) for k in keys])


def host_rng(seed, *keys) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(_seq(seed, *keys)))


def _device_gen(device, seed, *keys) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(_seq(seed, *keys).generate_state(1, np.uint64)[0] & 0x7FFF_FFFF_FFFF_FFFF))
    return g


def normal(shape, std, dtype, seed, *keys, device="cpu"):
    """N(0, std^2) tensor of ``dtype`` (torch dtype) drawn on ``device``.

    On the host the values come from PCG64 in float32 and are rounded once to
    ``dtype``; on a CUDA device they come from torch's generator.
    """
    if torch.device(device).type == "cpu":
        a = host_rng(seed, *keys).standard_normal(size=shape, dtype=np.float32)
        a *= np.float32(std)
        return torch.from_numpy(a).to(dtype)
    g = _device_gen(device, seed, *keys)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, float(std), generator=g)
    return t.to(dtype)


def _tdt(name):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def tokens(shape: MoEShape, seed=0, step=0, device="cpu", attempt=0, layer=0):
    """Input activations [T, H], N(0, 1), of the shape's x dtype, for layer 0
    (or, for stacks that are not chained, for the given layer) of a step."""
    keys = (_T_X, step, attempt) if layer == 0 else (_T_X, step, attempt, layer)
    return normal((shape.tokens, shape.hidden), 1.0, _tdt(shape.x_dtype), seed, *keys,
                  device=device)


# Exponent of the skewed router: with top-8 over 256 experts and N(0, 1)
# tokens, the 32 most-used experts take about half of all routes.
PREFILL_SKEW = 0.28


def skewed_router_std(E, H, gamma=PREFILL_SKEW):
    """Per-expert router row std that falls as a power of the expert's rank,
    (e + 1) ** -gamma, normalised to mean 1 / sqrt(H): the larger a row's
    scale, the more often its expert is among a token's top-k."""
    w = (np.arange(E, dtype=np.float64) + 1.0) ** (-gamma)
    return (w / w.mean() / np.sqrt(H)).astype(np.float32)


def router_weights(shape: MoEShape, layer, seed=0, device="cpu", row_std=None):
    """Router matrix [E, H], N(0, 1/H) of the shape's router dtype.

    ``row_std`` (length E) replaces the common std 1/sqrt(H) per expert row;
    the skewed prefill workload uses it to concentrate routes on a few experts.
    """
    H, E = shape.hidden, shape.experts
    base = normal((E, H), 1.0, torch.float32, seed, _T_ROUTER, layer, device=device)
    std = torch.full((E, 1), 1.0 / np.sqrt(H), dtype=torch.float32, device=base.device)
    if row_std is not None:
        std = torch.as_tensor(np.asarray(row_std, np.float32).reshape(E, 1), device=base.device)
    return (base * std).to(_tdt(shape.router_dtype))


def router_bias(shape: MoEShape, layer, seed=0, device="cpu", std=0.1):
    """Selection bias [E] of the sigmoid router, N(0, std^2) f32 (the pages give
    no values; trained biases of this kind are small next to the scores' 0..1)."""
    return normal((shape.experts,), std, torch.float32, seed, _T_BIAS, layer, device=device)


def expert_matrix(shape: MoEShape, layer, expert, mat, seed=0, device="cpu",
                  dtype=torch.bfloat16):
    """One expert matrix, N(0, 0.02) bf16: gate/up are [F, H], down is [H, F].

    Experts E..E+S-1 are the shared experts.
    """
    H, F = shape.hidden, shape.ffn
    rows, cols = (F, H) if mat in (MAT_GATE, MAT_UP) else (H, F)
    return normal((rows, cols), EXPERT_STD, dtype, seed, _T_EXPERT, layer, expert, mat,
                  device=device)


def with_outliers(w: torch.Tensor, seed, *keys, frac=0.01, factor=20.0):
    """Scale a seeded ``frac`` of the elements of ``w`` by ``factor`` (in place)."""
    n = w.numel()
    m = int(round(n * frac))
    if m == 0:
        return w
    if w.device.type == "cpu":
        pos = torch.from_numpy(host_rng(seed, _T_OUTLIER, *keys).choice(n, m, replace=False))
    else:
        g = _device_gen(w.device, seed, _T_OUTLIER, *keys)
        pos = torch.randperm(n, generator=g, device=w.device)[:m]
    flat = w.view(-1)
    flat[pos] = (flat[pos].float() * factor).to(w.dtype)
    return w


def matrix(rows, cols, std, seed, *keys, device="cpu", dtype=torch.bfloat16,
           outliers: Optional[float] = None):
    """A generic seeded weight matrix (used by quantiser tests and workloads)."""
    w = normal((rows, cols), std, dtype, seed, *keys, device=device)
    if outliers:
        with_outliers(w, seed, *keys, frac=outliers)
    return w
