"""ctypes shim over the plain-C oracle (``coli_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Takes and returns numpy
arrays; all conversions here are exact widenings (bf16/f32 -> f32/f64).
"""
import ctypes as C

import numpy as np

from .build import build_oracle, build_oracle_omp

__all__ = [
    "GROUP", "packed_row_bytes", "scales_per_row", "expert_packed_bytes",
    "expert_scales", "quant_i4g", "dequant_i4g", "matvec_i4g", "router_logits",
    "topk", "topk_sigmoid", "expert", "moe_forward", "moe_stack_forward", "lib",
    "set_threads", "threads", "quant_mxfp4", "dequant_mxfp4", "e2m1_value", "fmt_expert_bytes",
    "fmt_expert_scale_bytes", "moe_forward_fmt", "FMT_I4G", "FMT_MXFP4", "FMT_FP8",
    "quant_fp8b128", "dequant_fp8b128", "e4m3_value", "FMT_I4ROW", "quant_i4row",
    "dequant_i4row",
]

FMT_I4ROW, FMT_I4G, FMT_MXFP4, FMT_FP8 = 2, 4, 7, 8

GROUP = 64
_libs = {}
_threads = 1


def set_threads(n):
    """Run the following oracle calls on n threads (the OpenMP build of the same
    source; every sum keeps its order, so results do not depend on n).  n = 1
    selects the single-threaded build.  Returns the previous setting."""
    global _threads
    prev, _threads = _threads, max(1, int(n))
    if _threads > 1:
        L = lib()
        L.omp_set_num_threads(_threads)
    return prev


def threads():
    return _threads


def lib():
    key = "omp" if _threads > 1 else "serial"
    if key not in _libs:
        L = C.CDLL(build_oracle_omp() if key == "omp" else build_oracle())
        if key == "omp":
            L.omp_set_num_threads.argtypes = [C.c_int]
            L.omp_set_num_threads.restype = None
        i64, f32p, f64p = C.c_int64, C.POINTER(C.c_float), C.POINTER(C.c_double)
        u8p, i32p, u32p = C.POINTER(C.c_uint8), C.POINTER(C.c_int32), C.POINTER(C.c_uint32)
        L.orc_packed_row_bytes.argtypes = [i64]
        L.orc_packed_row_bytes.restype = i64
        L.orc_scales_per_row.argtypes = [i64]
        L.orc_scales_per_row.restype = i64
        L.orc_expert_packed_bytes.argtypes = [i64, i64]
        L.orc_expert_packed_bytes.restype = i64
        L.orc_expert_scales.argtypes = [i64, i64]
        L.orc_expert_scales.restype = i64
        L.orc_quant_i4g.argtypes = [f32p, i64, i64, u8p, f32p]
        L.orc_quant_i4g.restype = None
        L.orc_dequant_i4g.argtypes = [u8p, f32p, i64, i64, f64p]
        L.orc_dequant_i4g.restype = None
        L.orc_matvec_i4g.argtypes = [u8p, f32p, i64, i64, f64p, f64p]
        L.orc_matvec_i4g.restype = None
        L.orc_router_logits.argtypes = [f64p, f64p, i64, i64, i64, f64p]
        L.orc_router_logits.restype = None
        L.orc_topk.argtypes = [f64p, i64, C.c_int, i32p, f64p]
        L.orc_topk.restype = C.c_int
        L.orc_expert.argtypes = [u8p, f32p, i64, i64, f64p, f64p]
        L.orc_expert.restype = None
        L.orc_moe_forward.argtypes = [f64p, i64, i64, i64, i64, i64, f64p, u8p, f32p,
                                      C.c_int, f64p, i32p, f64p, u32p]
        L.orc_moe_forward.restype = C.c_int
        L.orc_topk_sigmoid.argtypes = [f64p, f64p, i64, C.c_int, i32p, f64p]
        L.orc_topk_sigmoid.restype = C.c_int
        L.orc_moe_forward_router.argtypes = [f64p, i64, i64, i64, i64, i64, f64p, C.c_int, f64p,
                                             u8p, f32p, C.c_int, f64p, i32p, f64p, u32p]
        L.orc_moe_forward_router.restype = C.c_int
        u8 = C.POINTER(C.c_uint8)
        L.orc_quant_mxfp4.argtypes = [f32p, i64, i64, u8, u8]
        L.orc_quant_mxfp4.restype = None
        L.orc_dequant_mxfp4.argtypes = [u8, u8, i64, i64, f64p]
        L.orc_dequant_mxfp4.restype = None
        L.orc_e2m1_value.argtypes = [C.c_int]
        L.orc_e2m1_value.restype = C.c_double
        for f in ("orc_fmt_expert_bytes", "orc_fmt_expert_scale_bytes"):
            getattr(L, f).argtypes = [C.c_int, i64, i64]
            getattr(L, f).restype = i64
        L.orc_moe_forward_fmt.argtypes = [C.c_int, f64p, i64, i64, i64, i64, i64, f64p, C.c_int,
                                          f64p, u8, u8, C.c_int, f64p, i32p, f64p, u32p]
        L.orc_moe_forward_fmt.restype = C.c_int
        L.orc_quant_fp8b128.argtypes = [f32p, i64, i64, u8, f32p]
        L.orc_quant_fp8b128.restype = None
        L.orc_dequant_fp8b128.argtypes = [u8, f32p, i64, i64, f64p]
        L.orc_dequant_fp8b128.restype = None
        L.orc_e4m3_value.argtypes = [C.c_int]
        L.orc_e4m3_value.restype = C.c_double
        L.orc_quant_i4row.argtypes = [f32p, i64, i64, u8, f32p]
        L.orc_quant_i4row.restype = None
        L.orc_dequant_i4row.argtypes = [u8, f32p, i64, i64, f64p]
        L.orc_dequant_i4row.restype = None
        _libs[key] = L
    return _libs[key]


def _p(a, ctype):
    return a.ctypes.data_as(C.POINTER(ctype))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def packed_row_bytes(cols):
    return int(lib().orc_packed_row_bytes(cols))


def scales_per_row(cols):
    return int(lib().orc_scales_per_row(cols))


def expert_packed_bytes(H, F):
    return int(lib().orc_expert_packed_bytes(H, F))


def expert_scales(H, F):
    return int(lib().orc_expert_scales(H, F))


def quant_i4g(w):
    """w: [rows, cols] float32 (bf16 widened exactly).  -> (packed u8, scales f32)."""
    w = _c(w, np.float32)
    rows, cols = w.shape
    packed = np.zeros((rows, packed_row_bytes(cols)), np.uint8)
    scales = np.zeros((rows, scales_per_row(cols)), np.float32)
    lib().orc_quant_i4g(_p(w, C.c_float), rows, cols, _p(packed, C.c_uint8),
                        _p(scales, C.c_float))
    return packed, scales


def dequant_i4g(packed, scales, cols):
    packed, scales = _c(packed, np.uint8), _c(scales, np.float32)
    rows = packed.shape[0]
    w = np.zeros((rows, cols), np.float64)
    lib().orc_dequant_i4g(_p(packed, C.c_uint8), _p(scales, C.c_float), rows, cols,
                          _p(w, C.c_double))
    return w


def matvec_i4g(packed, scales, cols, x):
    packed, scales, x = _c(packed, np.uint8), _c(scales, np.float32), _c(x, np.float64)
    rows = packed.shape[0]
    y = np.zeros(rows, np.float64)
    lib().orc_matvec_i4g(_p(packed, C.c_uint8), _p(scales, C.c_float), rows, cols,
                         _p(x, C.c_double), _p(y, C.c_double))
    return y


def router_logits(x, wr):
    """x [T, H], wr [E, H] -> logits [T, E] (float64)."""
    x, wr = _c(x, np.float64), _c(wr, np.float64)
    T, H = x.shape
    E = wr.shape[0]
    out = np.zeros((T, E), np.float64)
    lib().orc_router_logits(_p(x, C.c_double), _p(wr, C.c_double), T, H, E,
                            _p(out, C.c_double))
    return out


def topk(logits, k):
    """logits [E] (float64) -> (idx int32 [k], gates float64 [k], any_nan)."""
    logits = _c(logits, np.float64)
    idx = np.zeros(k, np.int32)
    gates = np.zeros(k, np.float64)
    nan = lib().orc_topk(_p(logits, C.c_double), logits.shape[0], k,
                         _p(idx, C.c_int32), _p(gates, C.c_double))
    return idx, gates, bool(nan)


def topk_sigmoid(logits, k, bias=None):
    """GLM router for one token: logits [E], bias [E] or None ->
    (idx int32 [k], gates float64 [k], any_nan)."""
    logits = _c(logits, np.float64)
    idx = np.zeros(k, np.int32)
    gates = np.zeros(k, np.float64)
    b64 = None if bias is None else _c(bias, np.float64)   # kept alive for the call
    bp = None if b64 is None else _p(b64, C.c_double)
    nan = lib().orc_topk_sigmoid(_p(logits, C.c_double), bp, logits.shape[0], k,
                                 _p(idx, C.c_int32), _p(gates, C.c_double))
    return idx, gates, bool(nan)


def expert(packed_e, scales_e, H, F, x):
    packed_e, scales_e, x = _c(packed_e, np.uint8), _c(scales_e, np.float32), _c(x, np.float64)
    y = np.zeros(H, np.float64)
    lib().orc_expert(_p(packed_e, C.c_uint8), _p(scales_e, C.c_float), H, F,
                     _p(x, C.c_double), _p(y, C.c_double))
    return y


def moe_forward(x, wr, packed, scales, H, F, E, n_shared, k, counts=None, router="softmax",
                bias=None):
    """One routed-MoE layer.

    x [T, H]; wr [E, H]; packed / scales: flat arrays holding experts 0..E+S-1
    in the library layout.  Returns (out [T,H] f64, idx [T,k] i32, gates [T,k]
    f64, nan_tokens).  ``counts`` (uint32 [E]) is accumulated in place.
    ``router``: "softmax" or "sigmoid" (scores with the selection ``bias`` [E]).
    """
    x, wr = _c(x, np.float64), _c(wr, np.float64)
    packed, scales = _c(packed.reshape(-1), np.uint8), _c(scales.reshape(-1), np.float32)
    T = x.shape[0]
    out = np.zeros((T, H), np.float64)
    idx = np.zeros((T, k), np.int32)
    gates = np.zeros((T, k), np.float64)
    cp = None
    if counts is not None:
        assert counts.dtype == np.uint32 and counts.flags.c_contiguous
        cp = _p(counts, C.c_uint32)
    fn = {"softmax": 0, "sigmoid": 1}[router]
    b64 = None if bias is None else _c(bias, np.float64)   # kept alive for the call
    bp = None if b64 is None else _p(b64, C.c_double)
    nan = lib().orc_moe_forward_router(_p(x, C.c_double), T, H, F, E, n_shared,
                                       _p(wr, C.c_double), fn, bp, _p(packed, C.c_uint8),
                                       _p(scales, C.c_float), k, _p(out, C.c_double),
                                       _p(idx, C.c_int32), _p(gates, C.c_double), cp)
    return out, idx, gates, int(nan)


def moe_stack_forward(x0, layers, H, F, E, n_shared, k, counts=None, router="softmax",
                      biases=None):
    """Decode stack: x_{l+1} = x_l + MoE_l(x_l) (residual chain, no attention or norm).

    ``layers`` is a list of (wr, packed, scales) per layer; ``biases`` the
    per-layer selection bias of the sigmoid router.  Returns (x_L, per-layer
    outputs, per-layer idx).  ``counts`` is uint32 [L, E].
    """
    x = np.asarray(x0, np.float64)
    outs, idxs = [], []
    for l, (wr, packed, scales) in enumerate(layers):
        c = None if counts is None else counts[l]
        b = None if biases is None else biases[l]
        out, idx, _, _ = moe_forward(x, wr, packed, scales, H, F, E, n_shared, k, c,
                                     router=router, bias=b)
        outs.append(out)
        idxs.append(idx)
        x = x + out
    return x, outs, idxs


# ---------------------------------------------------------------------------
# other container formats (MXFP4)


def quant_mxfp4(w):
    """w: [rows, cols] float32 -> (packed u8 [rows, ceil(cols/2)], E8M0 scales u8
    [rows, ceil(cols/32)])."""
    w = _c(w, np.float32)
    rows, cols = w.shape
    packed = np.zeros((rows, (cols + 1) // 2), np.uint8)
    scales = np.zeros((rows, (cols + 31) // 32), np.uint8)
    lib().orc_quant_mxfp4(_p(w, C.c_float), rows, cols, _p(packed, C.c_uint8),
                          _p(scales, C.c_uint8))
    return packed, scales


def dequant_mxfp4(packed, scales, cols):
    packed, scales = _c(packed, np.uint8), _c(scales, np.uint8)
    rows = packed.shape[0]
    w = np.zeros((rows, cols), np.float64)
    lib().orc_dequant_mxfp4(_p(packed, C.c_uint8), _p(scales, C.c_uint8), rows, cols,
                            _p(w, C.c_double))
    return w


def e2m1_value(code):
    return float(lib().orc_e2m1_value(int(code)))


def fmt_expert_bytes(fmt, H, F):
    return int(lib().orc_fmt_expert_bytes(fmt, H, F))


def fmt_expert_scale_bytes(fmt, H, F):
    return int(lib().orc_fmt_expert_scale_bytes(fmt, H, F))


def moe_forward_fmt(fmt, x, wr, packed, scales, H, F, E, n_shared, k, counts=None,
                    router="softmax", bias=None):
    """moe_forward over the container `fmt` (FMT_I4G: scales f32; FMT_MXFP4:
    scales are E8M0 bytes), experts 0..E+S-1 in the record layout."""
    x, wr = _c(x, np.float64), _c(wr, np.float64)
    packed = _c(packed.reshape(-1), np.uint8)
    scales = _c(np.asarray(scales).reshape(-1).view(np.uint8), np.uint8)
    T = x.shape[0]
    out = np.zeros((T, H), np.float64)
    idx = np.zeros((T, k), np.int32)
    gates = np.zeros((T, k), np.float64)
    cp = None
    if counts is not None:
        assert counts.dtype == np.uint32 and counts.flags.c_contiguous
        cp = _p(counts, C.c_uint32)
    fn = {"softmax": 0, "sigmoid": 1}[router]
    b64 = None if bias is None else _c(bias, np.float64)
    bp = None if b64 is None else _p(b64, C.c_double)
    nan = lib().orc_moe_forward_fmt(fmt, _p(x, C.c_double), T, H, F, E, n_shared,
                                    _p(wr, C.c_double), fn, bp, _p(packed, C.c_uint8),
                                    _p(scales, C.c_uint8), k, _p(out, C.c_double),
                                    _p(idx, C.c_int32), _p(gates, C.c_double), cp)
    return out, idx, gates, int(nan)


# ---------------------------------------------------------------------------
# fp8-e4m3-b128


def quant_fp8b128(w):
    """w: [rows, cols] float32 -> (E4M3 codes u8 [rows, cols], f32 scales
    [rows, ceil(cols/128)])."""
    w = _c(w, np.float32)
    rows, cols = w.shape
    packed = np.zeros((rows, cols), np.uint8)
    scales = np.zeros((rows, (cols + 127) // 128), np.float32)
    lib().orc_quant_fp8b128(_p(w, C.c_float), rows, cols, _p(packed, C.c_uint8),
                            _p(scales, C.c_float))
    return packed, scales


def dequant_fp8b128(packed, scales):
    packed, scales = _c(packed, np.uint8), _c(scales, np.float32)
    rows, cols = packed.shape
    w = np.zeros((rows, cols), np.float64)
    lib().orc_dequant_fp8b128(_p(packed, C.c_uint8), _p(scales, C.c_float), rows, cols,
                              _p(w, C.c_double))
    return w


def e4m3_value(code):
    return float(lib().orc_e4m3_value(int(code)))


def quant_i4row(w):
    """w: [rows, cols] float32 -> (packed u8 [rows, ceil(cols/2)], f32 scales [rows, 1])."""
    w = _c(w, np.float32)
    rows, cols = w.shape
    packed = np.zeros((rows, (cols + 1) // 2), np.uint8)
    scales = np.zeros((rows, 1), np.float32)
    lib().orc_quant_i4row(_p(w, C.c_float), rows, cols, _p(packed, C.c_uint8),
                          _p(scales, C.c_float))
    return packed, scales


def dequant_i4row(packed, scales, cols):
    packed, scales = _c(packed, np.uint8), _c(scales, np.float32)
    rows = packed.shape[0]
    w = np.zeros((rows, cols), np.float64)
    lib().orc_dequant_i4row(_p(packed, C.c_uint8), _p(scales, C.c_float), rows, cols,
                            _p(w, C.c_double))
    return w
