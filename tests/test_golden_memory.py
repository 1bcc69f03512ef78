"""The pages' printed memory figures (tests/golden/page_memory_figures.json, each
with its page and section) against the shapes they state, and the library's
workspace against the chunked budgets the pages give. The worked example's
figures reproduce with 8 bytes per logit, in MiB: its profiling script ("Step 2:
Verification and Memory Profiling") counts an fp32 logit plus an fp32 gradient
(4 + 4 bytes) per element, for the whole batch and for one 512-row chunk."""
import ctypes
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FIG = json.load(open(os.path.join(ROOT, "tests", "golden", "page_memory_figures.json")))["figures"]
UNIT = {"GB": 1e9, "MiB": 2.0 ** 20, "MB": 1e6}


def _fig(i):
    return next(f for f in FIG if f["id"] == i)


@pytest.mark.parametrize("f", FIG, ids=[f["id"] for f in FIG])
def test_printed_figure_follows_from_the_stated_shape(f):
    value = f["rows"] * f["V"] * f["bytes_per_element"] / UNIT[f["unit"]]
    assert round(value, f["printed_decimals"]) == pytest.approx(f["printed"]), value


def test_worked_example_chunked_figure_and_savings():
    f = _fig("worked_example_2048_tokens")
    chunked = f["chunk"] * f["V"] * f["bytes_per_element"] / UNIT[f["unit"]]
    assert round(chunked, 2) == f["chunked_printed"]
    assert round(100 * (1 - chunked / f["printed"]), 1) == f["savings_pct_printed"]


def test_logits_and_gradient_exceed_the_printed_total():
    f = _fig("logits_bf16_llama3_16384_tokens")
    assert 2 * f["rows"] * f["V"] * f["bytes_per_element"] / 1e9 >= f["with_gradient_printed_at_least"]


@pytest.fixture(scope="module")
def L():
    import linear_cross_entropy_chunked_gb300 as pkg
    try:
        pkg.build()
    except RuntimeError as e:   # no nvcc here
        pytest.skip(str(e))
    return pkg.lib()


LOW_MEMORY = 16   # LCE_LOW_MEMORY: one chunk buffer


def _ws(L, N, D, V, chunk, flags=0):
    out = ctypes.c_size_t(0)
    assert L.lce_workspace_size_opt(N, D, V, chunk, flags, ctypes.byref(out)) == 0
    return out.value


def test_library_workspace_within_the_pages_chunked_budgets(L):
    """The library's whole extra memory (its workspace; the outputs are needed
    anyway) with one chunk's logits at a time, as the pages hold them
    (LCE_LOW_MEMORY): below the exercise's chunked peak (chunks of 128 tokens, D
    4096 assumed: the exercise gives none), below the worked example's chunked
    figure, and a small fraction of the Llama-3 logits. The default workspace holds
    a second chunk buffer (chunks go in pairs with one dW contraction per pair) and
    the pair's H^T and dH parts: a little over twice that, still O(chunk * V)."""
    ex = _fig("exercise_fp16_batch4_seq2048")
    assert _ws(L, ex["rows"], 4096, ex["V"], ex["chunk"], LOW_MEMORY) < \
        ex["chunked_peak_below_mb"] * 1e6
    we = _fig("worked_example_2048_tokens")
    assert _ws(L, we["rows"], we["D"], we["V"], we["chunk"], LOW_MEMORY) < \
        we["chunked_printed"] * 2 ** 20
    l3 = _fig("logits_bf16_llama3_16384_tokens")
    low = _ws(L, l3["rows"], 4096, l3["V"], 1024, LOW_MEMORY)
    assert low < 0.07 * l3["printed"] * 1e9
    default = _ws(L, l3["rows"], 4096, l3["V"], 1024)
    assert low < default <= 2.2 * low
    assert default < 0.15 * l3["printed"] * 1e9
