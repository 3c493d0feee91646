"""The C-ABI library loads, exports every symbol include/coli.h declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def coli():
    from int4_expert_ffn_gb300 import build as b
    b.build()
    import int4_expert_ffn_gb300 as pkg
    return pkg.binding


def header_functions():
    src = open(os.path.join(ROOT, "include", "coli.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(coli_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree(coli):
    assert header_functions() == sorted(coli.EXPORTS)


def test_library_exports_every_declared_symbol(coli):
    lib = C.CDLL(coli.LIB_PATH)
    for name in header_functions():
        assert hasattr(lib, name), name


def test_status_strings(coli):
    for st in range(0, -11, -1):
        assert coli.lib.coli_status_str(st) != b"unknown status", st
    assert coli.lib.coli_status_str(-99) == b"unknown status"


def test_size_helpers(coli):
    assert coli.coli_packed_row_bytes(5) == 3
    assert coli.coli_scales_per_row(65) == 2
    H, F = 6144, 2048
    assert coli.coli_expert_packed_bytes(H, F) == 3 * H * F // 2
    assert coli.coli_expert_scale_count(H, F) == 3 * H * F // 64
    # bytes per GLM-like expert with scales: 21 233 664
    assert coli.coli_expert_packed_bytes(H, F) + 4 * coli.coli_expert_scale_count(H, F) == 21233664


def _desc(coli, **kw):
    base = dict(hidden=256, ffn=512, n_experts=8, n_shared=1, n_tokens=4,
                x_dtype=coli.COLI_F32, router_dtype=coli.COLI_F32)
    base.update(kw)
    return coli.MoEDesc(**base)


@pytest.mark.parametrize("bad", [
    dict(hidden=100), dict(hidden=0), dict(ffn=96), dict(n_experts=0), dict(n_experts=2048),
    dict(n_shared=-1), dict(n_shared=9), dict(n_tokens=-1), dict(x_dtype=7),
])
def test_workspace_size_rejects_bad_desc(coli, bad):
    assert coli.coli_moe_workspace_size(_desc(coli, **bad), 2) == 0


def test_router_fn_validated(coli):
    # unknown routing function -> rejected before any launch or allocation size
    assert coli.coli_moe_workspace_size(_desc(coli, router_fn=2), 2) == 0
    assert coli.coli_moe_workspace_size(_desc(coli, router_fn=-1), 2) == 0
    # the sigmoid router with no bias (zero bias) is a valid descriptor
    assert coli.coli_moe_workspace_size(_desc(coli, router_fn=coli.COLI_ROUTER_SIGMOID_BIAS), 2) > 0


def test_desc_layout_matches_header(coli):
    # the ctypes mirror of coli_moe_desc: 8 int32-sized fields, the bias pointer,
    # then the weight format
    D = coli.coli_moe_desc
    assert D.router_fn.offset == 28 and D.router_bias.offset == 32
    assert D.weight_fmt.offset == 40 and C.sizeof(D) == 48
    text = open(os.path.join(ROOT, "include", "coli.h")).read()
    assert "COLI_ROUTER_SIGMOID_BIAS = 1" in text and "const float *router_bias;" in text
    assert "int32_t weight_fmt;" in text and "COLI_FMT_MXFP4 = 7" in text
    assert "COLI_FMT_FP8 = 8" in text and "COLI_FMT_I4ROW = 2" in text


def test_workspace_size_bad_topk(coli):
    d = _desc(coli)
    assert coli.coli_moe_workspace_size(d, 0) == 0
    assert coli.coli_moe_workspace_size(d, 9) == 0     # k > E
    assert coli.coli_moe_workspace_size(d, 2) > 0


def test_entry_points_validate_before_launch(coli):
    lib = coli.lib
    bad = _desc(coli, hidden=100).c()
    good = _desc(coli).c()
    fake = C.c_void_p(0x1000)   # never dereferenced: validation fails first
    assert lib.coli_moe_forward(C.byref(bad), 2, fake, fake, fake, fake, fake, None, fake,
                                1 << 20, None) == coli.COLI_EINVAL
    assert lib.coli_moe_forward(C.byref(good), 2, None, fake, fake, fake, fake, None, fake,
                                1 << 20, None) == coli.COLI_EINVAL
    assert lib.coli_moe_forward(C.byref(good), 2, C.c_void_p(0x1004), fake, fake, fake, fake,
                                None, fake, 1 << 20, None) == coli.COLI_EALIGN
    assert lib.coli_moe_forward(C.byref(good), 2, fake, fake, fake, fake, fake, None, fake,
                                16, None) == coli.COLI_ENOMEM
    assert lib.coli_router_topk(C.byref(good), 3000, fake, fake, fake, fake, None, fake,
                                1 << 20, None) == coli.COLI_EINVAL
    assert lib.coli_moe_stack_forward(C.byref(good), 2, 0, fake, fake, fake, fake, fake, None,
                                      None, fake, 1 << 20, None) == coli.COLI_EINVAL
    assert lib.coli_quant_i4g(fake, coli.COLI_BF16, -1, 64, fake, fake, None) == coli.COLI_EINVAL
    assert lib.coli_quant_i4g(fake, 5, 1, 64, fake, fake, None) == coli.COLI_EINVAL
    assert lib.coli_quant_i4g(None, coli.COLI_BF16, 2, 64, fake, fake, None) == coli.COLI_EINVAL
    # empty inputs are valid no-ops
    empty = _desc(coli, n_tokens=0).c()
    assert lib.coli_moe_forward(C.byref(empty), 2, None, None, None, None, None, None, None,
                                0, None) == coli.COLI_OK
    assert lib.coli_quant_i4g(None, coli.COLI_BF16, 0, 64, None, None, None) == coli.COLI_OK


def header_defines():
    src = open(os.path.join(ROOT, "include", "coli.h")).read()
    return {m.group(1): int(m.group(2), 0)
            for m in re.finditer(r"#define\s+(COLI_[A-Z0-9_]+)\s+(0x[0-9a-fA-F]+|\d+)u?", src)}


def test_header_constants_match_binding(coli):
    defs = header_defines()
    assert {"COLI_FLAG_NAN_LOGITS", "COLI_FLAG_TIMEOUT", "COLI_KERNEL_ROUTE",
            "COLI_KERNEL_GATEUP", "COLI_KERNEL_DOWN"} <= set(defs)
    for name, value in defs.items():
        assert getattr(coli, name) == value, name


def test_profile_events_validation(coli):
    lib = coli.lib
    arr = (C.c_void_p * 1)()
    assert lib.coli_profile_events(coli.COLI_KERNEL_GATEUP, arr, arr, -1) == coli.COLI_EINVAL
    assert lib.coli_profile_events(7, arr, arr, 1) == coli.COLI_EINVAL
    assert lib.coli_profile_events(coli.COLI_KERNEL_GATEUP, None, None, 1) == coli.COLI_EINVAL
    # turning recording off is always valid and reports no bracketed launches
    assert lib.coli_profile_events(coli.COLI_KERNEL_GATEUP, None, None, 0) == 0


def test_last_error_before_any_failure(coli):
    assert coli.coli_last_error() == "no error"


def test_weight_format_rules(coli):
    # MXFP4 runs on the grouped GEMM: hidden % 256 == 0, ffn % 128 == 0
    d = coli.MoEDesc(320, 128, 8, 1, 4, coli.COLI_F32, coli.COLI_BF16,
                     weight_fmt=coli.COLI_FMT_MXFP4)
    assert coli.coli_moe_workspace_size(d, 2) == 0
    d = coli.MoEDesc(256, 128, 8, 1, 4, coli.COLI_F32, coli.COLI_BF16,
                     weight_fmt=coli.COLI_FMT_MXFP4)
    assert coli.coli_moe_workspace_size(d, 2) > 0
    d = coli.MoEDesc(256, 128, 8, 1, 4, coli.COLI_F32, coli.COLI_BF16, weight_fmt=5)
    assert coli.coli_moe_workspace_size(d, 2) == 0
    # sizes: MXFP4 rows are the int4 rows; one scale byte per 32 columns
    assert coli.lib.coli_fmt_row_bytes(coli.COLI_FMT_MXFP4, 333) == 167
    assert coli.lib.coli_fmt_scale_bytes(coli.COLI_FMT_MXFP4, 333) == 11
    assert coli.lib.coli_fmt_scale_bytes(coli.COLI_FMT_I4G, 333) == 4 * 6
    assert coli.coli_fmt_expert_bytes(coli.COLI_FMT_MXFP4, 256, 128) == coli.coli_expert_packed_bytes(256, 128)
    assert coli.coli_fmt_expert_scale_bytes(coli.COLI_FMT_MXFP4, 256, 128) == 3 * 256 * 128 // 32
    assert coli.lib.coli_fmt_row_bytes(9, 64) == 0
    # fp8-e4m3-b128: one byte per element, one f32 scale per 128 columns; same shape rules
    d = coli.MoEDesc(256, 64, 8, 1, 4, coli.COLI_F32, coli.COLI_BF16, weight_fmt=coli.COLI_FMT_FP8)
    assert coli.coli_moe_workspace_size(d, 2) == 0
    d = coli.MoEDesc(256, 128, 8, 1, 4, coli.COLI_F32, coli.COLI_BF16, weight_fmt=coli.COLI_FMT_FP8)
    assert coli.coli_moe_workspace_size(d, 2) > 0
    assert coli.lib.coli_fmt_row_bytes(coli.COLI_FMT_FP8, 333) == 333
    assert coli.lib.coli_fmt_scale_bytes(coli.COLI_FMT_FP8, 333) == 4 * 3
    assert coli.coli_fmt_expert_bytes(coli.COLI_FMT_FP8, 256, 128) == 3 * 256 * 128
    assert coli.coli_fmt_expert_scale_bytes(coli.COLI_FMT_FP8, 256, 128) == 4 * (2 * 128 * 2 + 256 * 1)
    # int4-row: int4 nibbles, one f32 scale per row
    d = coli.MoEDesc(256, 128, 8, 1, 4, coli.COLI_F32, coli.COLI_BF16, weight_fmt=coli.COLI_FMT_I4ROW)
    assert coli.coli_moe_workspace_size(d, 2) > 0
    assert coli.lib.coli_fmt_row_bytes(coli.COLI_FMT_I4ROW, 333) == 167
    assert coli.lib.coli_fmt_scale_bytes(coli.COLI_FMT_I4ROW, 333) == 4
    assert coli.coli_fmt_expert_scale_bytes(coli.COLI_FMT_I4ROW, 256, 128) == 4 * (2 * 128 + 256)
