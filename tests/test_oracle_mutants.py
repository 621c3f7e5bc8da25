"""Each plausible mistake planted in a copy of the C oracle (on the CPU) must
be caught by at least one pin.  The real oracle source is never modified."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attention_oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("mask_off_by_one", "int64_t last = i + (int64_t)(Tk - Tq);",
     "int64_t last = i + (int64_t)(Tk - Tq) - 1;"),
    ("mask_ignored", "if (job->causal) {", "if (0 && job->causal) {"),
    ("mask_tq_aligned", "int64_t last = i + (int64_t)(Tk - Tq);", "int64_t last = i;"),
    ("scale_dropped", "s[j] = job->scale * acc;", "s[j] = acc;"),
    ("scale_squared", "s[j] = job->scale * acc;", "s[j] = job->scale * job->scale * acc;"),
    ("lse_without_max", "*lse_out = n_vis > j0 ? m + log(z)", "*lse_out = n_vis > j0 ? log(z)"),
    ("window_one_key_short", "int64_t first = last - (int64_t)job->window + 1;",
     "int64_t first = last - (int64_t)job->window + 2;"),
    ("window_one_key_long", "int64_t first = last - (int64_t)job->window + 1;",
     "int64_t first = last - (int64_t)job->window;"),
    ("window_ignored", "if (job->window > 0) {", "if (0) {"),
    ("window_from_row_index", "int64_t first = last - (int64_t)job->window + 1;",
     "int64_t first = i - (int64_t)job->window + 1;"),
    ("window_sum_from_zero", "for (int64_t j = j0; j < n_vis; ++j) {\n        s[j] = exp(s[j] - m);",
     "for (int64_t j = 0; j < n_vis; ++j) {\n        s[j] = exp(s[j] - m);"),
    ("scores_use_v", "acc += (double)qrow[d] * (double)kh[j * D + d];",
     "acc += (double)qrow[d] * (double)vh[j * D + d];"),
    ("gqa_modulo_map", "const int64_t hkv = hq / group;", "const int64_t hkv = hq % job->Hkv;"),
    ("softmax_not_normalised", "for (int64_t j = j0; j < n_vis; ++j) s[j] /= z;", ""),
    ("o_transposed_index", "o_out[d] += p * (double)vr[d];", "o_out[d] += p * (double)vh[d * D + j % D];"),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC, encoding="utf-8").read()
    assert old in src, f"mutation site for {name} not found in the oracle source"
    c = tmp_path / f"{name}.c"
    c.write_text(src.replace(old, new, 1), encoding="utf-8")
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-o", str(so), str(c), "-lm"], check=True)
    return oracle.OracleLib(str(so)).attention_f64


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    attn = _build_mutant(tmp_path, name, old, new)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            with np.errstate(invalid="ignore", divide="ignore"):  # a mutant may yield inf - inf
                pin(attn)
        except Exception:  # AssertionError, or NaN-driven errors
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
