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
    ("mask_inverted", "if (mrow[j] != 0) {", "if (mrow[j] == 0) {"),
    ("mask_transposed", "const unsigned char *mrow = mask + bh * mask_bh_stride + i * N;\n                long n_vis = 0;\n                for (long j = 0; j < N; ++j) {\n                    if (mrow[j] != 0) {",
     "const unsigned char *mrow = mask + bh * mask_bh_stride + i;\n                long n_vis = 0;\n                for (long j = 0; j < N; ++j) {\n                    if (mrow[j * N] != 0) {"),
    ("gqa_heads_interleaved", "const long kvh = h / group;", "const long kvh = h % num_kv_heads;"),
    ("bwd_D_sign", "const double ds = p[j] * (dp[j] - D);", "const double ds = p[j] * (dp[j] + D);"),
    ("bwd_dq_no_scale", "dqh[i * d + c] += scale * ds * kh[j * d + c];",
     "dqh[i * d + c] += ds * kh[j * d + c];"),
    ("bwd_dk_uses_k", "dkh[j * d + c] += scale * ds * qi[c];",
     "dkh[j * d + c] += scale * ds * kh[j * d + c];"),
    ("bwd_dv_without_p", "dvh[j * d + c] += p[j] * doi[c];", "dvh[j * d + c] += doi[c];"),
    ("bwd_dp_uses_k", "for (long c = 0; c < d; ++c) acc += doi[c] * vh[j * d + c];",
     "for (long c = 0; c < d; ++c) acc += doi[c] * kh[j * d + c];"),
    ("bwd_unnormalised_p", "for (long j = 0; j < n_keys; ++j) p[j] /= l;",
     "for (long j = 0; j < n_keys; ++j) p[j] /= 1.0;"),
    ("bwd_causal_off_by_one", "const long n_keys = causal ? i + 1 : N;\n                    const double *qi",
     "const long n_keys = causal ? i : N;\n                    const double *qi"),
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
