"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
each one trips at least one pin.  This is what makes the pins worth trusting:
a dropped term, a wrong sign, a wrong or transposed index, an off-by-one mask
or a missing rescale anywhere in the oracle must not go unnoticed.

Each mutant is a textual edit of oracle/attn_oracle.c compiled into a temp
directory; the real oracle is never modified.
"""
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (id, exact text in attn_oracle.c, replacement)
MUTANTS = [
    ("dropped_scale", "s[j] = scale * dot;", "s[j] = dot;"),
    ("exp_sign", "s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    ("max_not_subtracted_lse", "*lse_out = m + log(z);", "*lse_out = log(z);"),
    ("k_index_transposed", "const double* kj = kh + j * D;", "const double* kj = kh + j;"),
    ("q_row_index", "const double* qi = qh + i * D;", "const double* qi = qh;"),
    ("dot_wrong_operand", "dot += qi[d] * kj[d];", "dot += qi[d] * kj[0];"),
    ("causal_off_by_one", "int64_t nvis = causal ? (i + 1) : N; /* keys",
     "int64_t nvis = causal ? i : N; /* keys"),
    ("causal_sees_one_more", "int64_t nvis = causal ? (i + 1) : N; /* keys",
     "int64_t nvis = causal ? (i + 2) : N; /* keys"),
    ("no_normalisation", "double p = s[j] / z;", "double p = s[j];"),
    ("v_reversed", "const double* vj = vh + j * D;", "const double* vj = vh + (nvis - 1 - j) * D;"),
    ("v_uses_k", "const double* vj = vh + j * D;", "const double* vj = kh + j * D;"),
    ("pv_wrong_column", "o_row[c] += p * vj[c];", "o_row[c] += p * vj[0];"),
    ("probs_bad_norm", "for (int64_t j = 0; j < nvis; ++j) row[j] /= z;",
     "for (int64_t j = 0; j < nvis; ++j) row[j] /= (z + 1.0);"),
    ("probs_causal_off_by_one", "int64_t nvis = causal ? (i + 1) : N;\n        const double* qi",
     "int64_t nvis = causal ? i : N;\n        const double* qi"),
    ("online_no_rescale", "double corr = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - m_new);",
     "double corr = 1.0;"),
    ("online_diag_test", "int diag = jb->causal && (kv_start + Bc - 1 > q_start);",
     "int diag = jb->causal && (kv_start > q_start);"),
    ("online_skips_diagonal_tile", "kv_limit = (q_start + Br < N) ? q_start + Br : N;",
     "kv_limit = (q_start < N) ? q_start : N;"),
    ("online_drops_ragged_tile", "int64_t Tc = (kv_limit + Bc - 1) / Bc;", "int64_t Tc = kv_limit / Bc;"),
    ("online_mask_row_vs_block", "(diag && key > row)", "(diag && key > q_start)"),
    ("online_l_not_rescaled", "l[r] = corr * l[r] + lsum;", "l[r] = l[r] + lsum;"),
    ("gqa_interleaved_heads", "const int64_t kvh = b * jb->Hkv + h / (jb->H / jb->Hkv);",
     "const int64_t kvh = b * jb->Hkv + h % jb->Hkv;"),
    ("bwd_dk_dropped_scale", "dk_row[c] += scale * ds * qi[c];", "dk_row[c] += ds * qi[c];"),
    ("bwd_dq_wrong_operand", "dq_row[c] += scale * ds * kj[c];", "dq_row[c] += scale * ds * qi[c];"),
    ("bwd_ds_sign", "const double ds = p * (dp - delta_h[i]);", "const double ds = p * (delta_h[i] - dp);"),
    ("bwd_dq_delta_dropped", "const double ds = p * (dp - delta_i);", "const double ds = p * dp;"),
    ("bwd_delta_unweighted", "delta += exp(s[j] - lse) * dp;", "delta += dp;"),
    ("bwd_lse_without_max", "const double lse = m + log(z);", "const double lse = log(z);"),
    ("bwd_dv_uses_ds", "dv_row[c] += p * doi[c];", "dv_row[c] += ds * doi[c];"),
    ("bwd_dkdv_causal_skips_diagonal", "for (int64_t i = causal ? j : 0; i < N; ++i) {",
     "for (int64_t i = causal ? j + 1 : 0; i < N; ++i) {"),
    ("bwd_dq_ignores_causal", "int64_t nvis = causal ? (i + 1) : N;\n    if (nvis > N) nvis = N;\n    for (int64_t c = 0; c < D; ++c) dq_row[c] = 0.0;",
     "int64_t nvis = N;\n    if (nvis > N) nvis = N;\n    for (int64_t c = 0; c < D; ++c) dq_row[c] = 0.0;"),
    ("bwd_dp_wrong_row", "for (int64_t c = 0; c < D; ++c) dp += doi[c] * vj[c];\n        const double p = exp(scale * dot - lse_i);",
     "for (int64_t c = 0; c < D; ++c) dp += doh[c] * vj[c];\n        const double p = exp(scale * dot - lse_i);"),
    ("bwd_gqa_first_head_only", "for (int64_t g = 0; g < G; ++g) {\n        const int64_t bh = b * c->H + hk * G + g;",
     "for (int64_t g = 0; g < 1; ++g) {\n        const int64_t bh = b * c->H + hk * G + g;"),
    ("bwd_gqa_interleaved_heads", "const int64_t bh = b * c->H + hk * G + g;", "const int64_t bh = b * c->H + g * c->Hkv + hk;"),
    ("bwd_gqa_kv_head_mod", "return b * c->Hkv + h / (c->H / c->Hkv);", "return b * c->Hkv + h % c->Hkv;"),
    ("gqa_no_batch_offset", "const int64_t kvh = b * jb->Hkv + h / (jb->H / jb->Hkv);",
     "const int64_t kvh = h / (jb->H / jb->Hkv) + 0 * b;"),
]


def _compile(text, tmp_path, name):
    src = tmp_path / (name + ".c")
    src.write_text(text)
    hdr = os.path.join(os.path.dirname(SRC), "attn_oracle.h")
    (tmp_path / "attn_oracle.h").write_text(open(hdr).read())
    lib = tmp_path / ("lib" + name + ".so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o",
                    str(lib), str(src), "-lm"], check=True, capture_output=True)
    return str(lib)


@pytest.mark.parametrize("mid,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(mid, old, new, tmp_path):
    text = open(SRC).read()
    assert text.count(old) >= 1, "mutation anchor vanished: %r" % old
    mutated = text.replace(old, new, 1)
    orc = oracle.OracleLib(_compile(mutated, tmp_path, mid))
    tripped = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            tripped.append(pin.__name__)
    assert tripped, "mutant %s passed every pin" % mid


def test_unmutated_copy_passes(tmp_path):
    orc = oracle.OracleLib(_compile(open(SRC).read(), tmp_path, "clean"))
    for pin in oracle_pins.ALL_PINS:
        pin(orc)
