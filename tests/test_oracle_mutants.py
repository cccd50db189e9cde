"""Each plausible mistake planted in a copy of the oracle fails some pin.

The mistakes are planted in the oracle's C source on the CPU (never in the
CUDA path): a dropped scale, a wrong sign, an off-by-one causal mask, a
reversed operand index, a missing normalisation or max term, a wrong paged
gather.  A mutant that passed every check would mean the pins cannot tell a
correct oracle from a broken one.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = [
    ("dropped_scale", "scores[j] = scale * acc;", "scores[j] = acc;"),
    ("exp_sign_flipped", "scores[j] = exp(scores[j] - m);", "scores[j] = exp(m - scores[j]);"),
    ("min_instead_of_max", "if (scores[j] > m) m = scores[j];", "if (scores[j] < m) m = scores[j];"),
    ("causal_off_by_one", "const long n_keys = causal ? i + 1 : N;\n                attend_row",
     "const long n_keys = causal ? i : N;\n                attend_row"),
    ("value_rows_reversed", "const double *vj = vv + j * d;",
     "const double *vj = vv + (n_keys - 1 - j) * d;"),
    ("key_dims_shifted", "acc += qi[c] * kj[c];", "acc += qi[c] * kj[(c + 1) % d];"),
    ("no_normalisation", "const double pj = scores[j] / l;", "const double pj = scores[j];"),
    ("lse_without_max", "*lse_i = m + log(l);", "*lse_i = log(l);"),
    ("key_gather_token_major",
     "K[tok * D + c] = kb[((c / x) * block_size + off) * x + (c % x)];",
     "K[tok * D + c] = kb[(off * (D / x) + c / x) * x + (c % x)];"),
    ("value_gather_transposed", "V[tok * D + c] = vb[c * block_size + off];",
     "V[tok * D + c] = vb[off * D + c];"),
    ("block_table_index_mod", "block_tables[s * max_blocks + tok / block_size]",
     "block_tables[s * max_blocks + tok % block_size]"),
]


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, find, repl):
    src = oracle.source_text()
    assert src.count(find) == 1, f"mutation site for {name} not unique"
    lib = oracle.compile_variant(src.replace(find, repl), os.path.join(tmp_path, f"{name}.so"))
    failed = []
    with oracle.use_library(lib):
        for check in oracle_pins.ALL_CHECKS:
            try:
                check()
            except (AssertionError, ValueError):
                failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
