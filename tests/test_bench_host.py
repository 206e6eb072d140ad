"""Host-side arithmetic of bench.py (no GPU): the algorithmic work it divides
by, the roofline of a Cayley-Neumann point, and the traffic table lookup."""
import os

import pytest

import bench
from orthogonal_equivalence_neumann_b300 import inputs

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 1500.0}


def test_step_flops_of_the_square_layer():
    # fwd: W0 GEMM 2 T d^2 + two block applies 2 T d b each; bwd: the same plus the dQ sums
    c = inputs.SQUARE_2048
    T, d, b = c.T, c.d_in, c.b_in
    fwd = 2 * T * d * d + 2 * 2 * T * d * b
    assert bench.step_flops(c) == pytest.approx(fwd + fwd + 2 * 2 * T * d * b)
    assert bench.step_flops(c) == pytest.approx(189.0e9, rel=1e-3)


def test_cnp_roofline_point_bounds():
    # b = 256, bf16 out: 4096 blocks of n = 3 products are tensor-bound at these peaks
    sec = 1e-3
    p = bench.cnp_roofline_point(256, 2, 3, 4096, sec, PEAKS)
    byts = 4096 * (4 * 256 * 255 // 2 + 2 * 256 * 256)
    flops = 4096 * 2.0 * 3 * 256 ** 3
    assert p["bound"] == "tensor"
    assert p["frac"] == pytest.approx(flops / 1.5e15 / sec, rel=1e-3)
    assert p["hbm_frac"] == pytest.approx(byts / 6e12 / sec, rel=1e-3)
    # b = 32: HBM-bound (for either output type)
    q = bench.cnp_roofline_point(32, 2, 3, 4096, sec, PEAKS)
    assert q["bound"] == "hbm" and q["frac"] == q["hbm_frac"]
    r = bench.cnp_roofline_point(32, 4, 3, 4096, sec, PEAKS)
    assert r["bound"] == "hbm" and r["hbm_frac"] > q["hbm_frac"]
    # fp32 Q at b = 128 runs three bf16 MMA chains per product: a third of the bf16 peak
    f = bench.cnp_roofline_point(128, 4, 6, 4096, sec, PEAKS)
    t_split = 4096 * 2.0 * 6 * 128 ** 3 / (1.5e15 / 3)
    assert f["bound"] == "tensor_split3" and f["frac"] == pytest.approx(t_split / sec, rel=1e-3)
    # fp32 Q at b = 256 also runs the three-term split on the tensor cores
    a = bench.cnp_roofline_point(256, 4, 3, 4096, sec, PEAKS)
    assert a["bound"] == "tensor_split3"
    assert a["frac"] == pytest.approx(flops / (1.5e15 / 3) / sec, rel=1e-3)


def test_traffic_entries_follow_their_sources(tmp_path, monkeypatch):
    # an entry counts only while the hash of all its sources matches
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.sources_sha("k.cu")
    (tmp_path / "profiles" / "traffic.txt").write_text("# c\nk k.cu %s 123\n" % sha)
    assert bench.read_traffic("k") == 123.0
    assert bench.read_traffic("other") is None
    src.write_text("kernel v2")
    assert bench.read_traffic("k") is None


def test_committed_traffic_table_matches_the_sources():
    # every committed entry names existing sources; its hash is checked by the bench at run time
    path = os.path.join(bench.ROOT, "profiles", "traffic.txt")
    for line in open(path):
        parts = line.split("#", 1)[0].split()
        if len(parts) == 4:
            assert bench.sources_sha(parts[1]) is not None, parts[1]
            assert float(parts[3]) > 0
