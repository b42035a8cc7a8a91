"""GPU parity of the device-side widening cp_pad_chunk (the query-width ladder's
pad rows, ONNX GenAI Wiki "Chunked Prefill" §四: the extra rows of a widened
chunk repeat the last real token) against the oracle's pad_rows, bit for bit,
through the C ABI."""
import numpy as np
import pytest
import torch

import chunked_prefill_causal_cp_gb300 as cp
import oracle
import synth_inputs as SI

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()


def _bits(t):
    """Raw bytes of a tensor as a numpy array (bit-exact comparison, NaN-safe)."""
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def _oracle_widened(x_real_rows: torch.Tensor, rows_padded: int) -> np.ndarray:
    """oracle.pad_rows applied to each sequence's real rows, on the raw bytes."""
    b = x_real_rows.detach().cpu().contiguous().view(torch.uint8).numpy()
    return np.stack([oracle.pad_rows(b[i], rows_padded) for i in range(b.shape[0])])


@pytest.mark.parametrize("real_rows", [1, 100, 171, 172, 300, 343, 416, 511])
@pytest.mark.parametrize("dtype,hq,hkv,d", [(torch.bfloat16, 32, 8, 128), (torch.float16, 16, 16, 64),
                                            (torch.float32, 8, 2, 64)])
def test_pad_chunk_matches_oracle_every_tier(real_rows, dtype, hq, hkv, d):
    """Chunk width 512: every ladder tier (171, 342, 512) for a batch of 3
    sequences.  Rows [real_rows, R) of q, k_new and v_new become copies of row
    real_rows - 1, byte for byte; rows below real_rows are not touched."""
    W, B = 512, 3
    R = cp.cp_query_width(real_rows, W)
    assert R == oracle.query_width(real_rows, W)
    q = SI.normal((B, R, hq, d), seed=real_rows, dtype=dtype).cuda()
    k = SI.normal((B, R, hkv, d), seed=real_rows + 1, dtype=dtype).cuda()
    v = SI.normal((B, R, hkv, d), seed=real_rows + 2, dtype=dtype).cuda()
    before = [_bits(t) for t in (q, k, v)]
    desc = cp.layer_desc(dtype, B, hq, hkv, d, cp.CP_CACHE_CONTIG, capacity=1024)
    cp.cp_pad_chunk(desc, q, k, v, real_rows, R)
    torch.cuda.synchronize()
    for t, b0 in zip((q, k, v), before):
        got = _bits(t)
        ref = _oracle_widened(t[:, :real_rows], R)
        assert np.array_equal(got, ref)
        assert np.array_equal(got[:, :real_rows], b0[:, :real_rows])


def test_pad_chunk_null_tensor_is_skipped():
    """A NULL tensor is skipped; the others are widened."""
    dtype, B, hq, hkv, d, r, R = torch.bfloat16, 2, 32, 8, 128, 200, 342
    q = SI.normal((B, R, hq, d), seed=5, dtype=dtype).cuda()
    k = SI.normal((B, R, hkv, d), seed=6, dtype=dtype).cuda()
    q0 = q.clone()
    desc = cp.layer_desc(dtype, B, hq, hkv, d, cp.CP_CACHE_CONTIG, capacity=1024)
    cp.cp_pad_chunk(desc, None, k, None, r, R)
    torch.cuda.synchronize()
    assert torch.equal(q, q0)
    assert np.array_equal(_bits(k), _oracle_widened(k[:, :r], R))


def test_pad_chunk_full_width_is_a_no_op():
    dtype, B, hq, hkv, d, R = torch.bfloat16, 1, 32, 8, 128, 512
    q = SI.normal((B, R, hq, d), seed=7, dtype=dtype).cuda()
    q0 = q.clone()
    desc = cp.layer_desc(dtype, B, hq, hkv, d, cp.CP_CACHE_CONTIG, capacity=1024)
    cp.cp_pad_chunk(desc, q, None, None, R, R)
    torch.cuda.synchronize()
    assert torch.equal(q, q0)
