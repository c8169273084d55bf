"""The oracle's pins are sensitive to the mistakes it could plausibly contain.

Each entry below plants one slip in a copy of the oracle's C++ source (a wrong
exponent bias, a dropped scale or ReLU, a swapped nibble, a reversed operand,
a wrong tie order, a value read from the wrong offset, a missing
normalisation, ...), compiles the copy on the CPU, swaps it in for the real
library, and runs every pin of tests/test_oracle_pins.py against it: at least
one pin must fail.  The two schedule functions written in Python (the
IndexCache / MLI layer sources and the prefill chunk plan) get the same
treatment through patched copies of their source.  The oracle itself is never
modified.  Every planted slip keeps the copy's memory accesses inside the
buffers the pins pass in."""
from __future__ import annotations

import concurrent.futures as cf
import ctypes
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins


def _nth_after(marker: str, old: str, new: str):
    """A patch of the first `old` after `marker` in the source."""
    def patch(src: str) -> str:
        start = src.index(marker)
        i = src.index(old, start)
        return src[:i] + new + src[i + len(old):]
    return patch


def _first(old: str, new: str):
    def patch(src: str) -> str:
        assert old in src, old
        return src.replace(old, new, 1)
    return patch


MUTANTS = {
    # decoders
    "e4m3 exponent bias 6": _first("mag = std::ldexp(8.0 + m, e - 7 - 3);",
                                   "mag = std::ldexp(8.0 + m, e - 6 - 3);"),
    "e4m3 subnormal step 2^-10": _first("mag = std::ldexp(static_cast<double>(m), -9);",
                                        "mag = std::ldexp(static_cast<double>(m), -10);"),
    "e2m1 subnormal 0.25": _first("mag = 0.5 * m;", "mag = 0.25 * m;"),
    "e2m1 nibble order (decoder)": _first("out[i] = dec_e2m1((i & 1) ? (byte >> 4) : (byte & 0xF));",
                                          "out[i] = dec_e2m1((i & 1) ? (byte & 0xF) : (byte >> 4));"),
    "ue8m0 bias 126": _first("static_cast<int>(e) - 127", "static_cast<int>(e) - 126"),
    "bf16 shift 15": _first("uint32_t u = static_cast<uint32_t>(h) << 16;",
                            "uint32_t u = static_cast<uint32_t>(h) << 15;"),
    # rows of a request
    "row length one short": _nth_after("int64_t row_len(", "(next_n - 1 - j)", "(next_n - j)"),
    # dense indexer, Eq. (1)
    "indexer without q scale": _nth_after(
        "int orc_indexer_logits(", "qd[h * D + d] = static_cast<double>(q_scale[r * H + h]) *",
        "qd[h * D + d] = 1.0 *"),
    "indexer without key scale": _first("kd[d] = s * dec_e4m3(kp[d], &bad);",
                                        "kd[d] = dec_e4m3(kp[d], &bad);"),
    "indexer without ReLU": _nth_after("int orc_indexer_logits(",
                                       "const double relu = dot > 0.0 ? dot : 0.0;",
                                       "const double relu = dot;"),
    "indexer |w| for w": _nth_after("int orc_indexer_logits(", "I += wh * relu;",
                                    "I += std::fabs(wh) * relu;"),
    "indexer key dims reversed": _nth_after("int orc_indexer_logits(",
                                            "dot += qd[h * D + d] * kd[d];",
                                            "dot += qd[h * D + d] * kd[D - 1 - d];"),
    # candidate path
    "expansion unsorted": _first("std::sort(ids.begin(), ids.end());", ""),
    "expansion end counts tok == L": _first("if (tok >= 0 && tok < L) ++cnt;",
                                            "if (tok >= 0 && tok <= L) ++cnt;"),
    "candidate nibble order": _nth_after("int orc_candidate_logits(",
                                         "(d & 1) ? (byte >> 4) : (byte & 0xF)",
                                         "(d & 1) ? (byte & 0xF) : (byte >> 4)"),
    "candidate scale group 64": _first("sp[d / 32]", "sp[d / 64]"),
    "candidate without ReLU": _nth_after("int orc_candidate_logits(",
                                         "const double relu = dot > 0.0 ? dot : 0.0;",
                                         "const double relu = dot;"),
    # top-k
    "top-k ascending": _first("if (s[a] != s[b]) return s[a] > s[b];",
                              "if (s[a] != s[b]) return s[a] < s[b];"),
    "top-k ties to the higher column": _first("return a < b;", "return a > b;"),
    "top-k pads with 0": _first("int64_t v = -1;", "int64_t v = 0;"),
    "top-k column map c / bs": _nth_after("int orc_topk(", "v % bs;", "v / bs;"),
    # sparse MLA, Eq. (2)
    "mla without softmax scale": _first("z[j] = scale * dot;", "z[j] = dot;"),
    "mla query dims reversed": _first("dot += dec_bf16(qg[d]) * c[j * Dqk + d];",
                                      "dot += dec_bf16(qg[Dqk - 1 - d]) * c[j * Dqk + d];"),
    "mla value from the last Dv elements": _first("o[d] += p * c[j * Dqk + d];",
                                                  "o[d] += p * c[j * Dqk + d + (Dqk - Dv)];"),
    "mla weights not normalised": _first("const double p = std::exp(z[j] - m) / sum;",
                                         "const double p = std::exp(z[j] - m);"),
    "mla lse without log": _first("m + std::log(sum);", "m + sum;"),
}


def _code_lines(src: str):
    return [l.split("//")[0].strip() for l in src.splitlines() if l.split("//")[0].strip()]


def _compile(item):
    name, patch, out_dir = item
    orig = open(oracle._SRC).read()
    src = patch(orig)
    assert _code_lines(src) != _code_lines(orig), f"{name}: the patch changes no code"
    so = os.path.join(out_dir, name.replace(" ", "_").replace("/", "_").replace("|", "abs")
                      .replace("=", "eq") + ".so")
    r = subprocess.run(["g++", "-std=c++17", "-O1", "-fPIC", "-shared", "-pthread",
                        "-fno-fast-math", "-ffp-contract=off", "-x", "c++", "-", "-o", so],
                       input=src, text=True, capture_output=True)
    assert r.returncode == 0, f"{name}: the planted copy does not compile:\n{r.stderr}"
    return name, so


@pytest.fixture(scope="module")
def mutant_libs(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("oracle_mutants"))
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        return dict(ex.map(_compile, [(n, p, out) for n, p in MUTANTS.items()]))


def _failing_pins(golden_dir):
    failed = []
    for name, fn in sorted(vars(pins).items()):
        if not name.startswith("test_") or not callable(fn):
            continue
        kwargs = {"golden_dir": golden_dir} if "golden_dir" in inspect.signature(fn).parameters else {}
        try:
            fn(**kwargs)
        except Exception:  # an assertion (or a value the pin cannot use) rejects the copy
            failed.append(name)
    return failed


# Slips in the oracle's Python schedule functions: (function, old, new).
PY_MUTANTS = {
    "layer 0 attends nothing under MLI": ("layer_sources", "if mli and layer > 0:", "if mli:"),
    "kept layers attend the previous one without MLI": (
        "layer_sources", "out.append(layer if kept else latest)", "out.append(latest)"),
    "every layer counts as an indexer layer": (
        "layer_sources", "        if kept:\n            latest = layer", "        latest = layer"),
    "chunk width not rounded to 4": (
        "prefill_chunk_plan", "w = (max(int(c), int(min_cols)) + 3) // 4 * 4",
        "w = max(int(c), int(min_cols))"),
    "chunk width ignores min_cols": (
        "prefill_chunk_plan", "w = (max(int(c), int(min_cols)) + 3) // 4 * 4",
        "w = (int(c) + 3) // 4 * 4"),
    "chunk budget exclusive": ("prefill_chunk_plan", "* 4 > budget_bytes:", "* 4 >= budget_bytes:"),
    "new row's width left out of the budget": (
        "prefill_chunk_plan", "(rows + 1) * max(width, w) * 4", "(rows + 1) * width * 4"),
}


def test_pins_pass_on_the_oracle(golden_dir):
    assert _failing_pins(golden_dir) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_slip(name, mutant_libs, golden_dir, monkeypatch):
    monkeypatch.setattr(oracle, "_lib", ctypes.CDLL(mutant_libs[name]))
    assert _failing_pins(golden_dir), f"no pin rejects the oracle with '{name}' planted"


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_pins_reject_planted_schedule_slip(name, golden_dir, monkeypatch):
    fn_name, old, new = PY_MUTANTS[name]
    src = inspect.getsource(getattr(oracle, fn_name))
    assert src.count(old) == 1, (name, old)
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), oracle.__file__, "exec"), ns)
    monkeypatch.setattr(oracle, fn_name, ns[fn_name])
    assert _failing_pins(golden_dir), f"no pin rejects the oracle with '{name}' planted"
