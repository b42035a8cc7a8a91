"""bench.py's host-side bookkeeping, on the CPU: the DRAM-traffic figure is
taken from a committed profile summary only while the kernel source it was
measured on is unchanged, and the visible-pair counts behind the FLOP totals
match brute force."""
import hashlib
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
    (prof / "kern.md").write_text(f"# kern\n\nsource_sha256: {sha} (kern.cu)\ndram_bytes_per_launch: 12345\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("kern.cu", "kern.md") == 12345.0
    src.write_text("// kernel v2\n")  # the kernel changed since the capture
    assert bench.kernel_traffic("kern.cu", "kern.md") is None
    assert bench.kernel_traffic("kern.cu", "missing.md") is None


def test_committed_profiles_name_current_sources():
    """Every committed summary that carries a traffic figure names a source
    file that exists, and the figure is read back for it."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for name, src in (("attn_tc_gqa_prefill.md", "attn_tc.cu"), ("decode_split_paged.md", "decode.cu")):
        text = open(os.path.join(root, "profiles", name)).read()
        assert "source_sha256:" in text and "dram_bytes_per_launch:" in text
        assert os.path.exists(os.path.join(root, "chunked_prefill_causal_cp_gb300", "csrc", src))


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
