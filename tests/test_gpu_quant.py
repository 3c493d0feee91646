"""GPU quantiser (coli_quant_i4g) against the oracle: bit-exact packing and scales."""
import os

import numpy as np
import pytest
import torch

import oracle as orc
from conftest import parse_golden
from int4_expert_ffn_gb300 import synth
from helpers import coli

pytestmark = pytest.mark.gpu

GOLDEN = parse_golden(os.path.join(os.path.dirname(__file__), "golden", "quant_hand.txt"))


def gpu_quant(w):
    packed, scales = coli().coli_quant_i4g(w.cuda())
    torch.cuda.synchronize()
    return packed.cpu().numpy(), scales.cpu().numpy()


def assert_same(w, tag=""):
    gp, gs = gpu_quant(w)
    op, os_ = orc.quant_i4g(w.float().cpu().numpy())
    bad = np.argwhere(gp != op)
    assert bad.size == 0, "%s: %d bytes differ, first %s" % (tag, len(bad), bad[:3].tolist())
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32)), tag


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("case", GOLDEN, ids=[c["name"] for c in GOLDEN])
def test_hand_vectors(case, dtype):
    w = torch.tensor(case["w"], dtype=torch.float32).to(dtype)
    gp, gs = gpu_quant(w)
    assert gp.tolist() == case["bytes"]
    assert gs.view(np.uint32).tolist() == case["scales"]


@pytest.mark.parametrize("rows,cols", [(1, 64), (64, 64), (100, 6144), (2048, 1024), (37, 2048),
                                       (33, 200), (7, 333), (5, 1), (3, 65)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_random_with_outliers(rows, cols, dtype):
    w = synth.matrix(rows, cols, 0.02, 7, rows, cols, dtype=dtype, outliers=0.01)
    w[0, : min(cols, 64)] = 0           # an all-zero group
    assert_same(w, "%dx%d" % (rows, cols))


def test_misaligned_input_takes_general_path():
    base = synth.matrix(17, 6145, 0.02, 3, dtype=torch.bfloat16).cuda()
    w = base.view(-1)[1:1 + 17 * 6144].view(17, 6144)   # 2-byte offset
    assert w.data_ptr() % 16 != 0
    assert_same(w.cpu(), "offset")
    gp, gs = coli().coli_quant_i4g(w)
    op, os_ = orc.quant_i4g(w.float().cpu().numpy())
    assert np.array_equal(gp.cpu().numpy(), op)


def test_half_integer_quotients_f32():
    # Quotients that land within a few f32 ulps of n + 0.5: the fast
    # reciprocal path must hand them to the exact division.
    rng = np.random.default_rng(5)
    rows, cols = 256, 128
    m = rng.uniform(0.5, 4.0, size=(rows, cols // 64)).astype(np.float32)
    s = m / np.float32(7)
    n = rng.integers(-7, 7, size=(rows, cols))
    w = np.repeat(s, 64, axis=1) * (n + np.float32(0.5))
    w = w.astype(np.float32)
    ulp = rng.integers(-3, 4, size=w.shape)
    w = np.nextafter(w, np.where(ulp > 0, np.inf, -np.inf).astype(np.float32))
    w[:, ::64] = np.repeat(m, 1, axis=1)          # each group's max is m
    assert_same(torch.from_numpy(w), "half-integer")


def test_nan_and_zero_rows():
    w = synth.matrix(4, 128, 0.02, 9, dtype=torch.float32)
    w[1] = 0
    w[2, 5] = float("nan")
    w[3, 70] = float("nan")
    w[3, 71] = 1.0
    assert_same(w, "nan")


def test_empty_rows():
    c = coli()
    w = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    p, s = c.coli_quant_i4g(w)
    assert p.shape == (0, 32) and s.shape == (0, 1)


def test_full_size_all_elements():
    """Quantiser workload: 256 experts x {gate, up [2048, 6144], down [6144, 2048]}
    bf16 N(0, 0.02) with 1% outliers x 20 (9.66 G elements).  The whole workload
    is quantised on the GPU in one call per matrix kind, as the benchmark runs
    it; then every element's nibble and every scale is compared with the
    oracle, 16 experts at a time (the oracle's OpenMP build over the rows)."""
    c = coli()
    E, F, H = 256, 2048, 6144
    chunk = 16
    prev = orc.set_threads(os.cpu_count() or 1)
    try:
        for mat, (rows, cols) in enumerate([(F, H), (F, H), (H, F)]):
            w = torch.empty((E * rows, cols), dtype=torch.bfloat16, device="cuda")
            for e in range(E):
                w[e * rows:(e + 1) * rows] = synth.matrix(rows, cols, 0.02, 0, 5, e, mat,
                                                          device="cuda", outliers=0.01)
            packed, scales = c.coli_quant_i4g(w)
            torch.cuda.synchronize()
            for e0 in range(0, E, chunk):
                r0, r1 = e0 * rows, (e0 + chunk) * rows
                op, os_ = orc.quant_i4g(w[r0:r1].float().cpu().numpy())
                gp = packed[r0:r1].cpu().numpy()
                gs = scales[r0:r1].cpu().numpy()
                bad = np.argwhere(gp != op)
                assert bad.size == 0, "matrix %d experts %d..%d: %d bytes differ, first %s" % (
                    mat, e0, e0 + chunk - 1, len(bad), bad[:3].tolist())
                assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32)), (mat, e0)
            del w, packed, scales
            torch.cuda.empty_cache()
    finally:
        orc.set_threads(prev)
