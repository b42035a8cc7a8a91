"""Plant plausible mistakes in the C++ oracle and check that at least one pin
fails for each.  Each mutant is a copy of ``oracle/cp_oracle.cpp`` with one
textual change (the text it replaces must occur exactly once), compiled with
g++ into a temporary library on the CPU and driven through the same Python
interface as the real one.  Every change keeps its reads and writes inside
the buffers the real code touches, so a mutant can be wrong but cannot crash
the test process."""
import concurrent.futures as cf
import os
import subprocess

import numpy as np
import pytest

import oracle.cpp as C
import oracle_pins
from oracle_pins import ALL_PINS

MUTANTS = {
    # the causal diagonal dropped: row i sees keys [0, past + i)
    "diag_dropped": ("    const int m = past + i + 1;\n", "    const int m = past + i;\n"),
    # query head h read from KV head h mod Hkv instead of h / G
    "gqa_modulo": ("    const int g = h / group;\n", "    const int g = h % hkv;\n"),
    # softmax scale 1/D instead of 1/sqrt(D)
    "scale_1_over_d": ("double default_scale(int d) { return 1.0 / std::sqrt((double)d); }",
                       "double default_scale(int d) { return 1.0 / (double)d; }"),
    # the weighted sum left unnormalised (the excluding form)
    "no_normalisation": ("    for (int t = 0; t < d; ++t) out[t] += w * v[j * stride + t];\n  }\n"
                         "  for (int t = 0; t < d; ++t) out[t] /= z;\n}\n\n// [Horizon] §4",
                         "    for (int t = 0; t < d; ++t) out[t] += w * v[j * stride + t];\n  }\n"
                         "  (void)z;\n}\n\n// [Horizon] §4"),
    # the chunk's rows appended in reverse order
    "append_reversed": ("(((int64_t)b * hkv + g) * cap + past[b] + t) * d,",
                        "(((int64_t)b * hkv + g) * cap + past[b] + (r - 1 - t)) * d,"),
    # the rolling update keeps the oldest rows and drops the new ones
    "rolling_keeps_oldest": ("      const int src = j + c;\n", "      const int src = j;\n"),
    # the rolling mask lets the next position through
    "rolling_mask_future": ("(a >= 0 && a >= left_pad && a <= p) ? 0.0 : -32768.0",
                            "(a >= 0 && a >= left_pad && a <= p + 1) ? 0.0 : -32768.0"),
    # the rolling mask admits the last left-pad position
    "rolling_mask_pad": ("(a >= 0 && a >= left_pad && a <= p) ? 0.0 : -32768.0",
                         "(a >= 0 && a >= left_pad - 1 && a <= p) ? 0.0 : -32768.0"),
    # the ladder step rounded down
    "ladder_floor": ("  const int step = (w + 2) / 3;\n", "  const int step = std::max(1, w / 3);\n"),
    # the remainder chunk put first
    "remainder_first": ("if (count < cap) sizes[count] = std::min(w, n - start);",
                        "if (count < cap) sizes[count] = (count == 0 && n % w) ? n % w : w;"),
    # the scores taken against V instead of K
    "scores_from_v": ("    if (!visible[j]) continue;\n    double dot = 0.0;\n    for (int t = 0; t < d; ++t) dot += q[t] * k[j * stride + t];",
                      "    if (!visible[j]) continue;\n    double dot = 0.0;\n    for (int t = 0; t < d; ++t) dot += q[t] * v[j * stride + t];"),
    # the additive rolling mask left out of the scores
    "additive_mask_dropped": ("    s[j] = scale * dot + mask[j];\n", "    s[j] = scale * dot;\n"),
    # the token budget not charged for the decode rows
    "budget_ignores_decodes": ("    int left = budget - (int)decodes.size();\n", "    int left = budget;\n"),
    # pad rows filled with zeros instead of the last real row
    "pad_with_zeros": ("  for (int t = r; t < rp; ++t) std::memcpy(out + t * e, x + (int64_t)(r - 1) * e, "
                       "sizeof(double) * e);\n",
                       "  for (int t = r; t < rp; ++t) std::memset(out + t * e, 0, sizeof(double) * e);\n"),
}
# page index and in-page offset swapped, in the write and in the gather alike
PAGED_SWAP = [
    ("  const int pg = table_row[pos / page];\n", "  const int pg = table_row[pos % page];\n"),
    ("(((int64_t)pg * hkv + g) * page + pos % page) * d, row", "(((int64_t)pg * hkv + g) * page + pos / page % page) * d, row"),
    ("    const int pg = table_row[a / page];\n", "    const int pg = table_row[a % page];\n"),
    ("(((int64_t)pg * hkv + g) * page + a % page) * d,", "(((int64_t)pg * hkv + g) * page + a / page % page) * d,"),
]


def _mutate(src, changes):
    for old, new in changes:
        assert src.count(old) == 1, f"mutation site not found exactly once: {old[:60]!r}"
        src = src.replace(old, new)
    return src


@pytest.fixture(scope="module")
def mutant_libs(tmp_path_factory):
    """Compile every mutant once (in parallel) into a temporary directory."""
    src = open(C.SRC).read()
    d = tmp_path_factory.mktemp("cpo_mutants")
    jobs = {name: [change] for name, change in MUTANTS.items()}
    jobs["paged_swap"] = PAGED_SWAP

    def build(item):
        name, changes = item
        cpp = os.path.join(d, f"{name}.cpp")
        with open(cpp, "w") as f:
            f.write(_mutate(src, changes))
        so = os.path.join(d, f"lib_{name}.so")
        subprocess.check_call(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", cpp, "-o", so])
        return name, so

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        return dict(ex.map(build, jobs.items()))


def _failing_pins(lib, monkeypatch):
    monkeypatch.setattr(C, "_lib", lib)
    monkeypatch.setattr(oracle_pins, "O", C)
    failed = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except Exception as e:  # an assertion, a shape error or an invalid-argument error all count
            failed.append((pin.__name__, type(e).__name__))
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS) + ["paged_swap"])
def test_cpp_mutant_is_caught(name, mutant_libs, monkeypatch):
    failed = _failing_pins(C.load(mutant_libs[name]), monkeypatch)
    assert failed, f"no pin caught the C++ oracle mutant {name}"


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    """The same build route with no change: every pin passes (so the mutants
    fail because of their change, not because of the route)."""
    cpp = os.path.join(tmp_path, "same.cpp")
    with open(cpp, "w") as f:
        f.write(open(C.SRC).read())
    so = os.path.join(tmp_path, "lib_same.so")
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", cpp, "-o", so])
    assert _failing_pins(C.load(so), monkeypatch) == []
