"""Route-count history file (.coli_usage) through the C ABI, on the host (no GPU).

Page: "colibrì 路由遥测全解析..." §历史文件 (three numeric fields per record, -1
geometry and -2 version/engine-hash headers, nonzero counts only, temporary file
and rename, 0-byte empty history), §编辑格式前必须知道的两个后果 (the hash is the
third field; glm_moe_dsa hashes to 3815245270), §可信读取 (trust relaxes identity
only), and the COLI_USAGE_DECAY entry (multiplier in (0, 1], count-1 experts kept).
"""
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "usage_glm_small.txt")


@pytest.fixture(scope="module")
def coli():
    from int4_expert_ffn_gb300 import build as b
    b.build()
    import int4_expert_ffn_gb300 as pkg
    return pkg.binding


SMALL = np.array([[0, 3, 0, 1], [5, 0, 0, 0]], np.uint32)


def old_reader(path, n_layers, n_experts):
    """A reader that predates the header records: takes triples of integers while
    three can be parsed, keeps those with 0 <= layer < n_layers (and expert in
    range), skips the rest."""
    toks = open(path).read().split()
    out = []
    for i in range(0, len(toks) - 2, 3):
        l, e, c = int(toks[i]), int(toks[i + 1]), int(toks[i + 2])
        if 0 <= l < n_layers and 0 <= e < n_experts:
            out.append((l, e, c))
    return out


def test_engine_id_is_the_pages_hash(coli):
    # the page prints the identity of the GLM engine: glm_moe_dsa -> 3815245270
    assert coli.coli_usage_engine_id("glm_moe_dsa") == 3815245270
    assert coli.coli_usage_engine_id("glm_moe_dsa") > 2 ** 31 - 1   # why it is the third field


def test_save_matches_golden_file(coli, tmp_path):
    p = tmp_path / ".coli_usage"
    coli.coli_usage_save(str(p), SMALL, "glm_moe_dsa")
    assert p.read_bytes() == open(GOLDEN, "rb").read()
    assert not (tmp_path / ".coli_usage.tmp").exists()


def test_every_record_has_three_fields(coli, tmp_path):
    p = tmp_path / "u"
    rng = np.random.default_rng(0)
    counts = (rng.random((3, 16)) < 0.4) * rng.integers(1, 1000, (3, 16))
    coli.coli_usage_save(str(p), counts.astype(np.uint32), "x")
    for line in p.read_text().splitlines():
        assert len(line.split()) == 3 and all(f.lstrip("-").isdigit() for f in line.split())


def test_empty_history_is_a_zero_byte_file(coli, tmp_path):
    p = tmp_path / "u"
    p.write_text("stale\n")
    coli.coli_usage_save(str(p), np.zeros((2, 4), np.uint32), "glm_moe_dsa")
    assert p.stat().st_size == 0
    counts, n = coli.coli_usage_load(str(p), 2, 4, "glm_moe_dsa")
    assert n == 0 and counts.sum() == 0


def test_old_reader_sees_exactly_the_data_records(coli, tmp_path):
    p = tmp_path / "u"
    coli.coli_usage_save(str(p), SMALL, "glm_moe_dsa")
    assert old_reader(str(p), 2, 4) == [(0, 1, 3), (0, 3, 1), (1, 0, 5)]


def test_roundtrip_adds_into_counts(coli, tmp_path):
    p = tmp_path / "u"
    coli.coli_usage_save(str(p), SMALL, "e1")
    counts, n = coli.coli_usage_load(str(p), 2, 4, "e1")
    assert n == 3 and np.array_equal(counts, SMALL)
    counts, n = coli.coli_usage_load(str(p), 2, 4, "e1", counts=counts)
    assert np.array_equal(counts, 2 * SMALL)


def _status(coli, fn, *args):
    with pytest.raises(coli.ColiError) as ei:
        fn(*args)
    return ei.value.status


def test_refusals_and_trust(coli, tmp_path):
    p = tmp_path / "u"
    coli.coli_usage_save(str(p), SMALL, "kimi_k3")
    # another engine's history: refused, unless the caller trusts the file
    assert _status(coli, coli.coli_usage_load, str(p), 2, 4, "glm_moe_dsa") == coli.COLI_EREFUSED
    counts, n = coli.coli_usage_load(str(p), 2, 4, "glm_moe_dsa", trusted=True)
    assert n == 3 and np.array_equal(counts, SMALL)
    # another geometry: refused even when trusted
    assert _status(coli, coli.coli_usage_load, str(p), 3, 4, "kimi_k3", True) == coli.COLI_EREFUSED
    # a later format version: refused even when trusted
    q = tmp_path / "v2"
    q.write_text("-1 2 4\n-2 2 %d\n0 0 1\n" % coli.coli_usage_engine_id("kimi_k3"))
    assert _status(coli, coli.coli_usage_load, str(q), 2, 4, "kimi_k3", True) == coli.COLI_EREFUSED
    # the dense binary layout of another engine
    d = tmp_path / "dense"
    d.write_bytes(b"IKU1" + np.array([2, 4] + [1] * 8, np.uint32).tobytes())
    assert _status(coli, coli.coli_usage_load, str(d), 2, 4, "kimi_k3", True) == coli.COLI_EREFUSED
    # a refused load adds nothing
    base = np.ones((2, 4), np.uint32)
    assert _status(coli, coli.coli_usage_load, str(p), 2, 4, "other", False, base) == \
        coli.COLI_EREFUSED
    assert np.array_equal(base, np.ones((2, 4), np.uint32))


def test_out_of_range_records_discarded_and_not_counted(coli, tmp_path):
    p = tmp_path / "u"
    p.write_text("0 0 2\n2 1 9\n1 4 9\n1 3 7\n-3 7 12\n99 0 1\n")
    counts, n = coli.coli_usage_load(str(p), 2, 4, "any")   # no header: the older layout
    assert n == 2
    assert counts[0, 0] == 2 and counts[1, 3] == 7 and counts.sum() == 9


def test_decay(coli, tmp_path):
    p = tmp_path / "u"
    counts = np.array([[10, 3, 1, 0, 2]], np.uint32)
    coli.coli_usage_save(str(p), counts, "e", decay=0.5)
    got, _ = coli.coli_usage_load(str(p), 1, 5, "e")
    # round(c/2), but an expert routed at all keeps a count of at least 1
    assert got.tolist() == [[5, 2, 1, 0, 1]]
    ref = tmp_path / "ref"
    coli.coli_usage_save(str(ref), counts, "e")
    for d in (1.0, 1.5, 0.0, -0.5):   # outside (0, 1): no decay, byte for byte
        coli.coli_usage_save(str(p), counts, "e", decay=d)
        assert p.read_bytes() == ref.read_bytes()


def test_replaces_existing_file_and_refuses_long_paths(coli, tmp_path):
    p = tmp_path / "u"
    p.write_text("0 0 1000\n")
    coli.coli_usage_save(str(p), SMALL, "glm_moe_dsa")
    assert p.read_bytes() == open(GOLDEN, "rb").read()
    long = str(tmp_path / ("x" * 4200))
    st = coli.lib.coli_usage_save(os.fsencode(long), SMALL.ctypes.data, 2, 4, b"e", 1.0)
    assert st == coli.COLI_EINVAL
    assert os.listdir(tmp_path) == ["u"]


def test_bad_arguments_and_missing_file(coli, tmp_path):
    lib = coli.lib
    assert lib.coli_usage_save(None, SMALL.ctypes.data, 2, 4, b"e", 1.0) == coli.COLI_EINVAL
    assert lib.coli_usage_save(b"x", SMALL.ctypes.data, 0, 4, b"e", 1.0) == coli.COLI_EINVAL
    out = np.zeros((2, 4), np.uint32)
    assert lib.coli_usage_load(os.fsencode(str(tmp_path / "none")), out.ctypes.data, 2, 4, b"e",
                               0, None) == coli.COLI_EIO
    assert coli._status_str(coli.COLI_EREFUSED).startswith("usage history")


@pytest.mark.gpu
def test_route_counts_of_a_stack_roundtrip(coli, tmp_path):
    """The per-(layer, expert) counts of a GPU stack call, kept in a history file."""
    import dataclasses
    import torch
    from int4_expert_ffn_gb300 import synth
    from helpers import Layer
    shape = dataclasses.replace(synth.TINY, layers=2, tokens=3)
    layers = [Layer(shape, l, 0) for l in range(2)]
    gp = [ly.gpu() for ly in layers]
    c = coli
    desc = c.MoEDesc(shape.hidden, shape.ffn, shape.experts, shape.shared, 3, c.COLI_F32,
                     c.COLI_F32)
    ws = c.new_workspace(desc, shape.top_k)
    counts = torch.zeros((2, shape.experts), dtype=torch.int32, device="cuda")
    c.coli_moe_stack_forward(desc, shape.top_k, 2, synth.tokens(shape).cuda(),
                             torch.cat([g[2] for g in gp]), torch.cat([g[0] for g in gp]),
                             torch.cat([g[1] for g in gp]), ws, route_counts=counts)
    host = counts.cpu().numpy().astype(np.uint32)
    assert host.sum() == 2 * 3 * shape.top_k
    p = tmp_path / ".coli_usage"
    c.coli_usage_save(str(p), counts, "int4_expert_ffn_gb300")
    back, n = c.coli_usage_load(str(p), 2, shape.experts, "int4_expert_ffn_gb300")
    assert np.array_equal(back, host) and n == int((host > 0).sum())
