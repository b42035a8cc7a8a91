"""bench.py's host-side bookkeeping, on the CPU: the DRAM-traffic figure is
taken from a committed JSON record only while the kernel source it was
measured on is unchanged, and the visible-pair counts behind the FLOP totals
match brute force."""
import hashlib
import json
import os

import numpy as np

import bench


def test_traffic_follows_the_profiled_source(tmp_path, monkeypatch):
    csrc = tmp_path / "chunked_prefill_causal_cp_gb300" / "csrc"
    prof = tmp_path / "profiles"
    csrc.mkdir(parents=True)
    prof.mkdir()
    src = csrc / "kern.cu"
    src.write_text("// kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    (prof / "kern.json").write_text(json.dumps({"kernel_source": "kern.cu", "source_sha256": sha,
                                                "dram_bytes_per_launch": 12345}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("kern.json") == 12345.0
    src.write_text("// kernel v2\n")  # the kernel changed since the capture
    assert bench.kernel_traffic("kern.json") is None
    assert bench.kernel_traffic("missing.json") is None


def test_committed_profiles_name_current_sources():
    """Every committed traffic record names a kernel source that exists and
    carries a positive byte count."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    names = [n for n in os.listdir(os.path.join(root, "profiles")) if n.endswith(".json")]
    assert "decode_split_paged.json" in names
    for name in names:
        rec = json.load(open(os.path.join(root, "profiles", name)))
        assert len(rec["source_sha256"]) == 64 and rec["dram_bytes_per_launch"] > 0
        assert os.path.exists(os.path.join(root, "chunked_prefill_causal_cp_gb300", "csrc", rec["kernel_source"]))


def test_visible_pairs_brute_force():
    for past in (0, 1, 37, 512):
        for rows in (1, 5, 128):
            mask = np.zeros((rows, past + rows), dtype=bool)
            for i in range(rows):
                mask[i, :past + i + 1] = True
            assert bench.visible_pairs(past, rows) == int(mask.sum())


def test_rolling_visible_pairs_match_the_oracle_mask():
    """The rolling workload's FLOP count uses visible pairs of real rows; the
    oracle's printed-form mask (0 = visible, -32768 = masked) gives the same
    count chunk by chunk."""
    import oracle

    for L, c, C, lp in ((2048, 256, 1024, 48), (768, 256, 1024, 68), (96, 16, 40, 5)):
        total = 0
        for k in range(L // c):
            m = oracle.rolling_mask(c, C, k, lp)
            total += int((m == 0).sum())
        assert bench.rolling_visible_pairs(L, c, C, lp) == total, (L, c, C, lp)


def test_mixed_rooflines_bracket_each_step():
    """T* takes each step's larger term and the serial time their sum, so
    T* <= serial <= 2 T*, with equality cases at the ends."""
    steps = [{"flops": 2e12, "bytes": 1e9}, {"flops": 0.0, "bytes": 5e9}, {"flops": 4e12, "bytes": 0.0}]
    tc, hbm = 2000.0, 5000.0  # TFLOP/s, GB/s
    t_star, t_serial = bench.mixed_rooflines(steps, tc, hbm)
    assert abs(t_star - (1.0 + 1.0 + 2.0)) < 1e-9          # ms: max(1, 0.2), max(0, 1), max(2, 0)
    assert abs(t_serial - (1.2 + 1.0 + 2.0)) < 1e-9
    assert t_star <= t_serial <= 2 * t_star


def test_oracle_config_samples_cover_every_other_workload():
    """The CPU baseline's bounded oracle samples name the configs they stand for
    and return positive rates (a tiny budget: one prompt, one rolling run)."""
    from oracle import cpp
    cpp.build()
    r = bench.oracle_config_samples(budget_s=0.01, ladder_groups=1)
    assert set(r) == {"fp32_example", "padding_ladder", "rolling", "mixed_budget8192_step1", "threads"}
    for name in ("fp32_example", "padding_ladder", "rolling"):
        assert r[name]["tokens_per_s"] > 0 and r[name]["sample"]
    assert r["mixed_budget8192_step1"]["rows_per_s"] > 0
    assert r["threads"] >= 1
