"""Plant plausible mistakes in a COPY of the oracle source and check that the
pins catch every one of them (CPU only; the real oracle file is never touched).

Each mutant is compiled from a text-edited copy of ``oracle/mla_oracle.c`` into a
temporary directory and run against the brute-force pin in all three
evaluation orders, and, where the fixture can see the mistake, against the
hand-worked call of tests/golden.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle.oracle import _SRC, load_variant
from tests.test_oracle import brute_force, run_oracle
from mla_speculative_verify_gb300 import inputs

MUTANTS = {
    "rope_dropped": ("for (int d = 0; d < D_QK; ++d) s += bf16_to_double(qv[d]) * k[d];",
                     "for (int d = 0; d < D_V; ++d) s += bf16_to_double(qv[d]) * k[d];"),
    "causal_off_by_one_direct": ("int n_i = ctx - q + i + 1;\n    attend_range",
                                 "int n_i = ctx - q + i + 2;\n    attend_range"),
    "causal_off_by_one_fold": ("if (j >= ctx - q + i + 1) continue;", "if (j >= ctx - q + i) continue;"),
    "kv_scale_missing": ("return p->kv_scale * mla_oracle_e4m3_to_double(", "return mla_oracle_e4m3_to_double("),
    "page_offset_reversed": ("return (int64_t)page * p->page_size + j % p->page_size;",
                             "return (int64_t)page * p->page_size + (p->page_size - 1 - j % p->page_size);"),
    "softmax_sign": ("double w = exp(s[j - j0] - m);", "double w = exp(m - s[j - j0]);"),
    "value_columns_shifted": ("for (int d = 0; d < D_V; ++d) o[d] += w * k[d];",
                              "for (int d = 0; d < D_V; ++d) o[d] += w * k[d + 64];"),
    "lse_log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "merge_weight": ("double w = exp(pl[slot] - L);", "double w = exp(pl[slot] - mx);"),
    "fold_rescale_dropped": ("l[r] = l[r] * a + w;", "l[r] = l[r] + w;"),
    "e4m3_bias": ("else v = ldexp(1.0 + (double)m / 8.0, e - 7);", "else v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "head_index": ("int64_t qrow = (tok0 + f) * H + (r % H);\n      double s", "int64_t qrow = (tok0 + f) * H + (H - 1 - r % H);\n      double s"),
}


def _cases():
    return [
        inputs.make_problem(3, [7, 4, 9], [1, 4, 2], inputs.KV_BF16, seed=12, page_size=2),
        inputs.make_problem(2, [6, 11], [2, 3], inputs.KV_FP8, seed=13, page_size=4),
        inputs.make_problem(5, [70, 130], [4, 1], inputs.KV_BF16, seed=14, page_size=64),
    ]


def _bounds(prob):
    return [[0, int(c) // 3, int(c) // 3, int(c) - 1, int(c)] for c in prob.seq_lens]


def pins_hold(lib) -> bool:
    for prob in _cases():
        o_ref, l_ref = brute_force(prob)
        for mode in (oracle.MODE_DIRECT, oracle.MODE_FOLDED, oracle.MODE_SPLIT):
            o, l = run_oracle(prob, mode, _bounds(prob) if mode == oracle.MODE_SPLIT else None, lib=lib)
            if not (np.allclose(o, o_ref, rtol=1e-11, atol=1e-12, equal_nan=False)
                    and np.allclose(l, l_ref, rtol=1e-11, atol=1e-12)):
                return False
    return True


def test_unmutated_copy_passes(tmp_path):
    path = str(tmp_path / "liborig.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", path, "-lm"], check=True)
    assert pins_hold(load_variant(path))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(_SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / f"{name}.c"
    mutated.write_text(src.replace(old, new))
    path = str(tmp_path / f"lib{name}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(mutated), "-o", path, "-lm"],
                   check=True)
    assert not pins_hold(load_variant(path)), f"pins did not catch mutant {name}"


# The hand-worked fixture of tests/golden must catch the mutants it can see (one head, a
# bf16 cache: the head-index, e4m3-bias and kv_scale mutants are out of its reach).
GOLDEN_REACH = ["rope_dropped", "causal_off_by_one_direct", "causal_off_by_one_fold", "page_offset_reversed",
                "softmax_sign", "value_columns_shifted", "lse_log2", "merge_weight", "fold_rescale_dropped"]


def golden_holds(lib) -> bool:
    import torch
    from tests import golden_fixture

    g = golden_fixture.load("closed_form_h1_q2_ctx3.json", page_size=2, page_order=[2, 0])
    qb = g["q"].view(torch.int16).numpy().view(np.uint16)
    kb = g["kv"].view(torch.int16).numpy().view(np.uint16)
    for mode in (oracle.MODE_DIRECT, oracle.MODE_FOLDED, oracle.MODE_SPLIT):
        o, l = oracle.decode(qb, kb, oracle.KV_BF16, 1.0, g["page_table"], 2, g["seq_lens"], g["q_lens"], g["H"],
                             g["sm_scale"], mode=mode, split_bounds=[[0, 1, 3]] if mode == oracle.MODE_SPLIT else None,
                             lib=lib)
        if not (np.allclose(o, g["out"], rtol=0, atol=1e-12) and np.allclose(l, g["lse"], rtol=0, atol=1e-12)):
            return False
    return True


def test_golden_unmutated_copy_passes(tmp_path):
    path = str(tmp_path / "liborig.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", path, "-lm"], check=True)
    assert golden_holds(load_variant(path))


@pytest.mark.parametrize("name", GOLDEN_REACH)
def test_golden_catches_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    mutated = tmp_path / f"{name}.c"
    mutated.write_text(open(_SRC).read().replace(old, new))
    path = str(tmp_path / f"lib{name}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(mutated), "-o", path, "-lm"],
                   check=True)
    assert not golden_holds(load_variant(path)), f"the golden fixture did not catch mutant {name}"
