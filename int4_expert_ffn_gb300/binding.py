"""Python binding of libcoli, the GB300 routed-MoE forward over int4-grouped experts.

Argument marshalling only: every function forwards torch tensors' device
pointers and the current CUDA stream to the C ABI in ``include/coli.h`` under
the same name.  All computation runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback -- importing this package fails loudly when
``libcoli.so`` is missing, and calls fail when no GPU is present.
"""
import ctypes as C
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# COLI_LIBRARY=check loads the diagnostic bounds-checked build (libcoli_check.so,
# built by build(variant="check")); otherwise the library itself
LIB_PATH = os.path.join(_PKG, "libcoli_check.so" if os.environ.get("COLI_LIBRARY") == "check"
                        else "libcoli.so")

COLI_OK, COLI_EINVAL, COLI_EALIGN, COLI_ECUDA, COLI_ETIMEOUT, COLI_ENOMEM, COLI_EUNSUPPORTED = (
    0, -1, -2, -3, -4, -5, -6)
COLI_EIO, COLI_EREFUSED, COLI_ERANGE, COLI_EBOUNDS = -7, -8, -9, -10
COLI_F32, COLI_BF16 = 0, 1
COLI_ROUTER_SOFTMAX, COLI_ROUTER_SIGMOID_BIAS = 0, 1
COLI_FLAG_NAN_LOGITS, COLI_FLAG_TIMEOUT, COLI_FLAG_RANGE, COLI_FLAG_BOUNDS = 0x1, 0x2, 0x4, 0x8
COLI_KERNEL_ROUTE, COLI_KERNEL_GATEUP, COLI_KERNEL_DOWN = 0, 1, 2
COLI_KERNEL_PREFILL_GATEUP, COLI_KERNEL_PREFILL_DOWN = 3, 4
COLI_KERNEL_LAYER = 5
COLI_FMT_I4ROW, COLI_FMT_I4G, COLI_FMT_MXFP4, COLI_FMT_FP8 = 2, 4, 7, 8
GROUP = 64

# every symbol include/coli.h declares
EXPORTS = (
    "coli_status_str", "coli_last_error", "coli_packed_row_bytes", "coli_scales_per_row",
    "coli_expert_packed_bytes", "coli_expert_scale_count", "coli_quant_i4g",
    "coli_router_workspace_size", "coli_moe_workspace_size", "coli_router_topk",
    "coli_moe_forward", "coli_moe_forward_noalloc", "coli_moe_stack_forward",
    "coli_profile_events", "coli_moe_check", "coli_usage_engine_id", "coli_usage_save",
    "coli_usage_load", "coli_moe_forward_tiered", "coli_tier_place", "coli_tier_update",
    "coli_quant_mxfp4", "coli_fmt_row_bytes", "coli_fmt_scale_bytes", "coli_fmt_expert_bytes",
    "coli_fmt_expert_scale_bytes", "coli_quant_fp8b128", "coli_quant_i4row",
)


class ColiError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = "%s failed: %s (%d)" % (fn, _status_str(status), status)
        if status == COLI_ECUDA:
            msg += ": " + coli_last_error()
        super().__init__(msg)


class coli_moe_desc(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("ffn", C.c_int32), ("n_experts", C.c_int32),
                ("n_shared", C.c_int32), ("n_tokens", C.c_int32), ("x_dtype", C.c_int),
                ("router_dtype", C.c_int), ("router_fn", C.c_int32),
                ("router_bias", C.c_void_p), ("weight_fmt", C.c_int32)]


class coli_tier(C.Structure):
    _fields_ = [("n_slots", C.c_int32), ("max_uploads", C.c_int32), ("slot_of", C.c_void_p),
                ("slot_owner", C.c_void_p), ("pool_packed", C.c_void_p),
                ("pool_scales", C.c_void_p), ("heat", C.c_void_p), ("last", C.c_void_p),
                ("clock", C.c_void_p), ("uploads", C.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libcoli.so is not built (expected at %s); run "
            "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
    L = C.CDLL(LIB_PATH)
    vp, i64, sz = C.c_void_p, C.c_int64, C.c_size_t
    dp = C.POINTER(coli_moe_desc)
    L.coli_status_str.argtypes = [C.c_int]
    L.coli_status_str.restype = C.c_char_p
    L.coli_last_error.argtypes = []
    L.coli_last_error.restype = C.c_char_p
    for f in ("coli_packed_row_bytes", "coli_scales_per_row"):
        getattr(L, f).argtypes = [i64]
        getattr(L, f).restype = i64
    for f in ("coli_expert_packed_bytes", "coli_expert_scale_count"):
        getattr(L, f).argtypes = [i64, i64]
        getattr(L, f).restype = i64
    L.coli_quant_i4g.argtypes = [vp, C.c_int, i64, i64, vp, vp, vp]
    L.coli_quant_i4g.restype = C.c_int
    L.coli_quant_mxfp4.argtypes = [vp, C.c_int, i64, i64, vp, vp, vp]
    L.coli_quant_mxfp4.restype = C.c_int
    L.coli_quant_fp8b128.argtypes = [vp, C.c_int, i64, i64, vp, vp, vp]
    L.coli_quant_fp8b128.restype = C.c_int
    L.coli_quant_i4row.argtypes = [vp, C.c_int, i64, i64, vp, vp, vp]
    L.coli_quant_i4row.restype = C.c_int
    for f in ("coli_fmt_row_bytes", "coli_fmt_scale_bytes"):
        getattr(L, f).argtypes = [C.c_int32, i64]
        getattr(L, f).restype = i64
    for f in ("coli_fmt_expert_bytes", "coli_fmt_expert_scale_bytes"):
        getattr(L, f).argtypes = [C.c_int32, i64, i64]
        getattr(L, f).restype = i64
    for f in ("coli_router_workspace_size", "coli_moe_workspace_size"):
        getattr(L, f).argtypes = [dp, C.c_int]
        getattr(L, f).restype = sz
    L.coli_router_topk.argtypes = [dp, C.c_int, vp, vp, vp, vp, vp, vp, sz, vp]
    L.coli_router_topk.restype = C.c_int
    L.coli_moe_forward.argtypes = [dp, C.c_int, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.coli_moe_forward.restype = C.c_int
    L.coli_moe_forward_noalloc.argtypes = [dp, C.c_int, vp, vp, vp, vp, vp, vp, vp]
    L.coli_moe_forward_noalloc.restype = C.c_int
    L.coli_moe_stack_forward.argtypes = [dp, C.c_int, C.c_int, vp, vp, vp, vp, vp, vp, vp,
                                         vp, sz, vp]
    L.coli_moe_stack_forward.restype = C.c_int
    L.coli_profile_events.argtypes = [C.c_int, C.POINTER(vp), C.POINTER(vp), C.c_int]
    L.coli_profile_events.restype = C.c_int
    L.coli_moe_check.argtypes = [vp, C.c_int, C.POINTER(C.c_uint32), vp]
    L.coli_moe_check.restype = C.c_int
    L.coli_usage_engine_id.argtypes = [C.c_char_p]
    L.coli_usage_engine_id.restype = C.c_uint32
    L.coli_usage_save.argtypes = [C.c_char_p, vp, C.c_int32, C.c_int32, C.c_char_p, C.c_float]
    L.coli_usage_save.restype = C.c_int
    L.coli_usage_load.argtypes = [C.c_char_p, vp, C.c_int32, C.c_int32, C.c_char_p, C.c_int,
                                  C.POINTER(C.c_int64)]
    L.coli_usage_load.restype = C.c_int
    tp = C.POINTER(coli_tier)
    L.coli_moe_forward_tiered.argtypes = [dp, C.c_int, vp, vp, vp, vp, tp, vp, vp, vp, sz, vp]
    L.coli_moe_forward_tiered.restype = C.c_int
    L.coli_tier_place.argtypes = [dp, vp, vp, tp, vp]
    L.coli_tier_place.restype = C.c_int
    L.coli_tier_update.argtypes = [dp, vp, vp, vp, tp, vp]
    L.coli_tier_update.restype = C.c_int
    return L


lib = _load()


def _status_str(status):
    return lib.coli_status_str(status).decode()


def coli_last_error():
    """Message of the last CUDA error a call on this thread returned as COLI_ECUDA."""
    return lib.coli_last_error().decode()


def _check(fn, status):
    if status != COLI_OK:
        raise ColiError(fn, status)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dt(t):
    if t.dtype == torch.float32:
        return COLI_F32
    if t.dtype == torch.bfloat16:
        return COLI_BF16
    raise TypeError("expected float32 or bfloat16, got %s" % t.dtype)


def _cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


@dataclass(frozen=True)
class MoEDesc:
    hidden: int
    ffn: int
    n_experts: int
    n_shared: int
    n_tokens: int
    x_dtype: int = COLI_F32
    router_dtype: int = COLI_BF16
    router_fn: int = COLI_ROUTER_SOFTMAX
    router_bias: object = None    # f32 CUDA tensor [E] (or [n_layers, E]), or None
    weight_fmt: int = 0           # COLI_FMT_I4G (0 also), _I4ROW, _MXFP4 or _FP8

    def c(self):
        b = self.router_bias
        if b is not None:
            if not (b.is_cuda and b.is_contiguous() and b.dtype == torch.float32):
                raise ValueError("router_bias must be a contiguous float32 CUDA tensor")
        return coli_moe_desc(self.hidden, self.ffn, self.n_experts, self.n_shared,
                             self.n_tokens, self.x_dtype, self.router_dtype, self.router_fn,
                             None if b is None else b.data_ptr(), self.weight_fmt)


def coli_packed_row_bytes(cols):
    return lib.coli_packed_row_bytes(cols)


def coli_scales_per_row(cols):
    return lib.coli_scales_per_row(cols)


def coli_expert_packed_bytes(H, F):
    return lib.coli_expert_packed_bytes(H, F)


def coli_expert_scale_count(H, F):
    return lib.coli_expert_scale_count(H, F)


def coli_quant_i4g(w, packed=None, scales=None, stream=None):
    """Quantise w [rows, cols] (bf16 or f32, CUDA) -> (packed u8, scales f32)."""
    _cuda(w)
    rows, cols = w.shape
    if packed is None:
        packed = torch.empty((rows, coli_packed_row_bytes(cols)), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((rows, coli_scales_per_row(cols)), dtype=torch.float32, device=w.device)
    _cuda(packed, scales)
    _check("coli_quant_i4g", lib.coli_quant_i4g(_ptr(w), _dt(w), rows, cols, _ptr(packed),
                                                 _ptr(scales), _stream(stream)))
    return packed, scales


def coli_quant_mxfp4(w, packed=None, scales=None, stream=None):
    """Quantise w [rows, cols] (bf16 or f32, CUDA) to MXFP4 -> (packed u8
    [rows, ceil(cols/2)], E8M0 scales u8 [rows, ceil(cols/32)])."""
    _cuda(w)
    rows, cols = w.shape
    if packed is None:
        packed = torch.empty((rows, (cols + 1) // 2), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((rows, (cols + 31) // 32), dtype=torch.uint8, device=w.device)
    _cuda(packed, scales)
    _check("coli_quant_mxfp4", lib.coli_quant_mxfp4(_ptr(w), _dt(w), rows, cols, _ptr(packed),
                                                     _ptr(scales), _stream(stream)))
    return packed, scales


def coli_quant_i4row(w, packed=None, scales=None, stream=None):
    """Quantise w [rows, cols] (bf16 or f32, CUDA) to int4-row -> (packed u8
    [rows, ceil(cols/2)], scales f32 [rows, 1])."""
    _cuda(w)
    rows, cols = w.shape
    if packed is None:
        packed = torch.empty((rows, (cols + 1) // 2), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((rows, 1), dtype=torch.float32, device=w.device)
    _cuda(packed, scales)
    _check("coli_quant_i4row", lib.coli_quant_i4row(_ptr(w), _dt(w), rows, cols, _ptr(packed),
                                                     _ptr(scales), _stream(stream)))
    return packed, scales


def coli_quant_fp8b128(w, packed=None, scales=None, stream=None):
    """Quantise w [rows, cols] (bf16 or f32, CUDA) to fp8-e4m3-b128 -> (packed
    u8 [rows, cols] E4M3 codes, scales f32 [rows, ceil(cols/128)])."""
    _cuda(w)
    rows, cols = w.shape
    if packed is None:
        packed = torch.empty((rows, cols), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((rows, (cols + 127) // 128), dtype=torch.float32, device=w.device)
    _cuda(packed, scales)
    _check("coli_quant_fp8b128", lib.coli_quant_fp8b128(_ptr(w), _dt(w), rows, cols,
                                                         _ptr(packed), _ptr(scales),
                                                         _stream(stream)))
    return packed, scales


def coli_fmt_expert_bytes(fmt, H, F):
    return lib.coli_fmt_expert_bytes(fmt, H, F)


def coli_fmt_expert_scale_bytes(fmt, H, F):
    return lib.coli_fmt_expert_scale_bytes(fmt, H, F)


def coli_moe_workspace_size(desc: MoEDesc, top_k):
    d = desc.c()
    return lib.coli_moe_workspace_size(C.byref(d), top_k)


def coli_router_workspace_size(desc: MoEDesc, top_k):
    d = desc.c()
    return lib.coli_router_workspace_size(C.byref(d), top_k)


def new_workspace(desc: MoEDesc, top_k, device="cuda"):
    """Zero-filled workspace of the size the library asks for."""
    n = coli_moe_workspace_size(desc, top_k)
    if n == 0:
        raise ColiError("coli_moe_workspace_size", COLI_EINVAL)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def coli_router_topk(desc: MoEDesc, top_k, x, router_w, workspace, idx=None, gates=None,
                     route_counts=None, stream=None):
    _cuda(x, router_w, workspace, route_counts)
    T = desc.n_tokens
    if idx is None:
        idx = torch.empty((T, top_k), dtype=torch.int32, device=x.device)
    if gates is None:
        gates = torch.empty((T, top_k), dtype=torch.float32, device=x.device)
    d = desc.c()
    _check("coli_router_topk", lib.coli_router_topk(
        C.byref(d), top_k, _ptr(x), _ptr(router_w), _ptr(idx), _ptr(gates),
        _ptr(route_counts), _ptr(workspace), workspace.numel(), _stream(stream)))
    return idx, gates


def coli_moe_forward(desc: MoEDesc, top_k, x, router_w, packed_experts, scales, workspace,
                     out=None, route_counts=None, stream=None):
    _cuda(x, router_w, packed_experts, scales, workspace, out, route_counts)
    if out is None:
        out = torch.empty((desc.n_tokens, desc.hidden), dtype=torch.float32, device=x.device)
    d = desc.c()
    _check("coli_moe_forward", lib.coli_moe_forward(
        C.byref(d), top_k, _ptr(x), _ptr(router_w), _ptr(packed_experts), _ptr(scales),
        _ptr(out), _ptr(route_counts), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def coli_moe_forward_noalloc(desc: MoEDesc, top_k, x, router_w, packed_experts, scales,
                             out=None, route_counts=None, stream=None):
    """coli_moe_forward with the library's fixed device scratch instead of a
    workspace, for callers that cannot allocate device memory (see coli.h)."""
    _cuda(x, router_w, packed_experts, scales, out, route_counts)
    if out is None:
        out = torch.empty((desc.n_tokens, desc.hidden), dtype=torch.float32, device=x.device)
    d = desc.c()
    _check("coli_moe_forward_noalloc", lib.coli_moe_forward_noalloc(
        C.byref(d), top_k, _ptr(x), _ptr(router_w), _ptr(packed_experts), _ptr(scales),
        _ptr(out), _ptr(route_counts), _stream(stream)))
    return out


def coli_moe_stack_forward(desc: MoEDesc, top_k, n_layers, x, router_w, packed_experts, scales,
                           workspace, x_out=None, layer_out=None, route_counts=None,
                           stream=None):
    _cuda(x, router_w, packed_experts, scales, workspace, x_out, layer_out, route_counts)
    if x_out is None:
        x_out = torch.empty((desc.n_tokens, desc.hidden), dtype=torch.float32, device=x.device)
    d = desc.c()
    _check("coli_moe_stack_forward", lib.coli_moe_stack_forward(
        C.byref(d), top_k, n_layers, _ptr(x), _ptr(router_w), _ptr(packed_experts),
        _ptr(scales), _ptr(x_out), _ptr(layer_out), _ptr(route_counts), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return x_out


def coli_profile_events(kernel, before, after):
    """Bracket the next len(before) launches of `kernel` (COLI_KERNEL_*) with
    the given torch.cuda.Event pairs (diagnostic, see coli.h); empty lists turn
    recording off.  Returns the launches bracketed under the previous setting."""
    n = len(before)
    if len(after) != n:
        raise ValueError("before/after lengths differ")
    arr_b = (C.c_void_p * max(n, 1))(*[e.cuda_event for e in before])
    arr_a = (C.c_void_p * max(n, 1))(*[e.cuda_event for e in after])
    st = lib.coli_profile_events(kernel, arr_b, arr_a, n)
    if st < 0:
        raise ColiError("coli_profile_events", st)
    return st


def coli_moe_check(workspace, clear=True, stream=None):
    """Return the device-side flag word (COLI_FLAG_*) of a workspace; clears it by default."""
    flags = C.c_uint32(0)
    st = lib.coli_moe_check(_ptr(workspace), 1 if clear else 0, C.byref(flags), _stream(stream))
    if st not in (COLI_OK, COLI_ETIMEOUT, COLI_ERANGE, COLI_EBOUNDS):
        raise ColiError("coli_moe_check", st)
    return flags.value


class Tier:
    """Device state of a tiered expert store (coli_tier in coli.h): a pool of
    n_slots expert records in HBM and the LFRU policy state.  ``owners`` is the
    initial expert of each slot (-1 free); the pool itself is filled by
    coli_tier_place from the host store."""

    def __init__(self, desc: MoEDesc, owners, max_uploads=8, device="cuda"):
        E, S = desc.n_experts, desc.n_shared
        n = len(owners)
        eb = coli_expert_packed_bytes(desc.hidden, desc.ffn)
        es = coli_expert_scale_count(desc.hidden, desc.ffn)
        slot_of = [-1] * (E + S)
        for sl, e in enumerate(owners):
            if e >= 0:
                slot_of[e] = sl
        self.n_slots, self.max_uploads = n, max_uploads
        self.slot_of = torch.tensor(slot_of, dtype=torch.int32, device=device)
        self.slot_owner = torch.tensor(list(owners) or [0], dtype=torch.int32, device=device)[:n]
        self.pool_packed = torch.empty(max(n, 1) * eb, dtype=torch.uint8, device=device)
        self.pool_scales = torch.empty(max(n, 1) * es, dtype=torch.float32, device=device)
        self.heat = torch.zeros(E, dtype=torch.int32, device=device)
        self.last = torch.zeros(E, dtype=torch.int32, device=device)
        self.clock = torch.zeros(1, dtype=torch.int32, device=device)
        self.uploads = torch.zeros(1 + 2 * max(max_uploads, 1), dtype=torch.int32, device=device)

    def c(self):
        return coli_tier(self.n_slots, self.max_uploads, self.slot_of.data_ptr(),
                         self.slot_owner.data_ptr(), self.pool_packed.data_ptr(),
                         self.pool_scales.data_ptr(), self.heat.data_ptr(), self.last.data_ptr(),
                         self.clock.data_ptr(), self.uploads.data_ptr())


def _pinned(*ts):
    for t in ts:
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError("the host store must be contiguous pinned host tensors")


def coli_moe_forward_tiered(desc: MoEDesc, top_k, x, router_w, host_packed, host_scales,
                            tier: Tier, workspace, out=None, route_counts=None, stream=None):
    """coli_moe_forward over a tiered store: experts from their HBM slots when
    resident, else from the pinned host store."""
    _cuda(x, router_w, workspace, out, route_counts)
    _pinned(host_packed, host_scales)
    if out is None:
        out = torch.empty((desc.n_tokens, desc.hidden), dtype=torch.float32, device=x.device)
    d, t = desc.c(), tier.c()
    _check("coli_moe_forward_tiered", lib.coli_moe_forward_tiered(
        C.byref(d), top_k, _ptr(x), _ptr(router_w), _ptr(host_packed), _ptr(host_scales),
        C.byref(t), _ptr(out), _ptr(route_counts), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out


def coli_tier_place(desc: MoEDesc, host_packed, host_scales, tier: Tier, stream=None):
    _pinned(host_packed, host_scales)
    d, t = desc.c(), tier.c()
    _check("coli_tier_place", lib.coli_tier_place(C.byref(d), _ptr(host_packed),
                                                   _ptr(host_scales), C.byref(t),
                                                   _stream(stream)))


def coli_tier_update(desc: MoEDesc, call_counts, host_packed, host_scales, tier: Tier,
                     stream=None):
    """One LFRU policy tick from a call's route counts, then its uploads."""
    _cuda(call_counts)
    _pinned(host_packed, host_scales)
    d, t = desc.c(), tier.c()
    _check("coli_tier_update", lib.coli_tier_update(C.byref(d), _ptr(call_counts),
                                                     _ptr(host_packed), _ptr(host_scales),
                                                     C.byref(t), _stream(stream)))


def coli_usage_engine_id(engine):
    """32-bit FNV-1a hash of an engine name (the usage history's identity field)."""
    return int(lib.coli_usage_engine_id(engine.encode()))


def _host_counts(counts):
    import numpy as np
    a = counts.detach().cpu().numpy() if isinstance(counts, torch.Tensor) else counts
    return np.ascontiguousarray(a, dtype=np.uint32)


def coli_usage_save(path, counts, engine, decay=1.0):
    """Write route counts [n_layers, n_experts] (torch or numpy, any device) as a
    usage history file; see coli.h."""
    a = _host_counts(counts)
    L, E = a.shape
    _check("coli_usage_save", lib.coli_usage_save(os.fsencode(path), a.ctypes.data, L, E,
                                                  engine.encode(), decay))


def coli_usage_load(path, n_layers, n_experts, engine, trusted=False, counts=None):
    """Read a usage history into counts (uint32 numpy [n_layers, n_experts], added to
    ``counts`` if given).  Returns (counts, records added); raises ColiError if refused."""
    import numpy as np
    a = np.zeros((n_layers, n_experts), np.uint32) if counts is None else counts
    assert a.dtype == np.uint32 and a.flags.c_contiguous and a.shape == (n_layers, n_experts)
    n = C.c_int64(0)
    _check("coli_usage_load", lib.coli_usage_load(os.fsencode(path), a.ctypes.data, n_layers,
                                                  n_experts, engine.encode(), int(trusted),
                                                  C.byref(n)))
    return a, n.value
