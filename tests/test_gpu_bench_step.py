"""The exact step the benchmark times, checked against the oracle.

bench.py's default workload is one captured CUDA graph per step: the device
widening of the 416-row last chunk to its 512-row tier (cp_pad_chunk) and one
cp_prefill_chunk call per chunk of the 4000-token GQA prompt (32/8 heads x
128, bf16, chunk 512, cache capacity 8192).  This test replays that very graph
once and compares its results with the oracle: sampled output rows of every
chunk one by one, and the whole cache bit for bit, including the 96 pad slots
after position 4000 (ONNX GenAI Wiki "Chunked Prefill" §四: the pad rows'
K/V are written past the valid length and hold the last real row)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import BF16_TOL, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def step():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()
    import bench
    wl = bench.GqaPrefill(torch.device("cuda", 0))
    wl.capture()
    # poison everything the step must write, then replay the captured graph once
    wl.out.fill_(float("nan"))
    wl.kc.zero_()
    wl.vc.zero_()
    wl.graph.replay()
    torch.cuda.synchronize()
    return wl


def test_bench_step_state(step):
    wl = step
    assert wl.sizes == [512] * 7 + [416] and wl.widths == [512] * 8
    assert int(wl.lens.item()) == wl.N
    assert int(wl.status.item()) == 0
    k, v = wl.host_k, wl.host_v
    kc, vc = wl.kc[0].cpu(), wl.vc[0].cpu()
    # positions [0, 4000): the prompt's K/V, byte for byte
    assert torch.equal(kc[:, :wl.N], k.permute(1, 0, 2))
    assert torch.equal(vc[:, :wl.N], v.permute(1, 0, 2))
    # the 96 pad slots of the widened last chunk repeat the last real row
    pad = wl.widths[-1] - wl.sizes[-1]
    kp = oracle.pad_rows(f64(k[-wl.sizes[-1]:]), wl.widths[-1])[-pad:]
    vp = oracle.pad_rows(f64(v[-wl.sizes[-1]:]), wl.widths[-1])[-pad:]
    assert np.array_equal(f64(kc[:, wl.N:wl.N + pad]), kp.transpose(1, 0, 2))
    assert np.array_equal(f64(vc[:, wl.N:wl.N + pad]), vp.transpose(1, 0, 2))
    # nothing past the widened chunk is touched
    assert not kc[:, wl.N + pad:].any() and not vc[:, wl.N + pad:].any()


def test_bench_step_outputs_match_oracle(step):
    """Each chunk's first and last real rows and 24 seeded rows per chunk match
    the oracle's attention of that row over keys [0, pos] within 2e-2."""
    wl = step
    q, k, v = f64(wl.host_q), f64(wl.host_k), f64(wl.host_v)
    out = f64(wl.out[:wl.N])
    rng = np.random.default_rng(2024)
    past, worst = 0, 0.0
    for r in wl.sizes:
        rows = {past, past + r - 1} | set(int(x) for x in rng.integers(past, past + r, 24))
        for p in sorted(rows):
            ref = oracle.attention_row(q[p], k[:p + 1], v[:p + 1], p)
            worst = max(worst, float(np.abs(out[p] - ref).max()))
        past += r
    assert worst < BF16_TOL, worst
    assert np.isfinite(out).all()
