"""The C ABI from C: tests/capi_example.c, built with gcc against
include/cp_api.h and libcp.so, calls the host-side helpers (no GPU) and
prints results the pages fix (the 7 x 512 + 416 plan, the {171, 342, 512}
ladder, the 10-step budget-8192 schedule whose first step is 64 decodes plus
8128 prompt rows)."""
import os
import subprocess

import numpy as np
import pytest
import torch

import chunked_prefill_causal_cp_gb300 as cp
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_c_program_links_and_calls_the_host_helpers(tmp_path):
    cp.lib()  # the library is built
    libdir = os.path.dirname(os.path.abspath(cp.LIB_PATH))
    exe = os.path.join(tmp_path, "capi_example")
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           os.path.join(HERE, "capi_example.c"), "-L", libdir, "-l:libcp.so",
                           "-Wl,-rpath," + libdir, "-o", exe])
    out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.splitlines()
    assert out[0] == f"abi {cp.cp_abi_version()}"
    assert out[1] == "plan 8: 512 512 512 512 512 512 512 416"
    assert out[2] == "ladder 3: 171 342 512"
    assert out[3] == "width416 512"
    assert out[4] == "aligned 2048"
    assert out[5].startswith("schedule ") and out[5].endswith(", 10 steps, step 0 rows 8192")
    ws = cp.cp_workspace_size(cp.layer_desc(1, 1, 32, 8, 128, cp.CP_CACHE_CONTIG, capacity=8192), 512, 8192, 1)
    assert out[6] == f"workspace {ws}"
    assert out[7] == f"rows past the chunk: {cp.lib().cp_status_string(cp.CP_ERR_INVALID_ARG).decode()}"



@pytest.mark.gpu
def test_c_program_runs_a_chunked_prefill_on_the_gpu(tmp_path):
    """tests/capi_gpu_example.c: cudaMalloc, cp_prefill_chunk per chunk; the
    inputs and outputs it writes out are compared with the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from chunked_prefill_causal_cp_gb300 import _build
    _build.build()
    libdir = os.path.dirname(os.path.abspath(cp.LIB_PATH))
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = os.path.join(tmp_path, "capi_gpu_example")
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           "-I", os.path.join(cuda, "include"), os.path.join(HERE, "capi_gpu_example.c"),
                           "-L", libdir, "-l:libcp.so", "-L", os.path.join(cuda, "lib64"), "-lcudart",
                           "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", exe])
    dump = os.path.join(tmp_path, "tensors.bin")
    r = subprocess.run([exe, dump], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("chunks 3 seqlens_k 300 status 0")
    n, hq, hkv, d = 300, 8, 2, 64
    raw = np.fromfile(dump, dtype=np.uint16)
    sizes = [n * hq * d, n * hkv * d, n * hkv * d, n * hq * d]
    parts = np.split(raw, np.cumsum(sizes)[:-1])
    q, k, v, out = (torch.from_numpy(p.astype(np.int16)).view(torch.bfloat16).double().numpy()
                    .reshape(n, -1, d) for p in parts)
    ref, _, _ = oracle.chunked_prefill(q, k, v, 128)
    assert np.abs(out - ref).max() < 2e-2
