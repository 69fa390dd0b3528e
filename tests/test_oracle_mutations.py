"""The oracle's pins must fail on plausible mistakes planted in the oracle.

Each case writes a copy of oracle.c with one planted mistake into a temporary
directory, compiles it with gcc (CPU only) and runs the pin suite against it
through the CF_ORACLE_LIB override; the suite must fail.  The committed
oracle itself is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "eps_outside_sqrt": ("sqrt(sum_sq / (double)H + eps)", "(sqrt(sum_sq / (double)H) + eps)"),
    "sum_not_mean": ("sum_sq / (double)H + eps", "sum_sq + eps"),
    "drop_ln_weight": ("n[i] = (x[i] / rms) * g[i];", "n[i] = (x[i] / rms);"),
    "rope_sign_first": ("u[i] = a * c - b * s;", "u[i] = a * c + b * s;"),
    "rope_sign_second": ("u[i + half] = b * c + a * s;", "u[i + half] = b * c - a * s;"),
    "rope_frequency": ("pow(theta, -2.0 * (double)i / (double)d)",
                       "pow(theta, -1.0 * (double)i / (double)d)"),
    "no_score_scale": ("const double scale = 1.0 / sqrt((double)d);\n  double* s =",
                       "const double scale = 1.0;\n  double* s ="),
    "gqa_modulo_grouping": ("const int j = h / group;", "const int j = h % nkv;"),
    "drop_new_token": ("orc_attention(d, pos + 1,", "orc_attention(d, pos,"),
    "drop_residual": ("out[i] = x[i] + proj[i];", "out[i] = proj[i];"),
    "q_from_wrong_columns": ("double* q = y;", "double* q = y + (size_t)nkv * d;"),
    "no_rope_on_q": ("for (int h = 0; h < nq; ++h) orc_rope(", "for (int h = 0; h < 0; ++h) orc_rope("),
    "no_rope_on_k": ("for (int j = 0; j < nkv; ++j) orc_rope(", "for (int j = 0; j < 0; ++j) orc_rope("),
    "split_without_rescale": ("double r = exp(mc[c] - m);", "double r = 1.0;"),
    "ffn_silu_on_up": ("a[i] = orc_silu(gs) * us;", "a[i] = gs * orc_silu(us);"),
    "ffn_silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "ffn_drop_residual": ("out[j] = h[j] + proj[j];", "out[j] = proj[j];"),
    "ffn_up_from_gate_rows": ("us += urow[k] * n[k];", "us += grow[k] * n[k];"),
    "ffn_norm_weight_dropped": ("orc_rmsnorm(H, h, g2, eps, n);", "orc_rmsnorm(H, h, h, eps, n);"),
    "ffn_gate_row_read_as_column": ("gs += grow[k] * n[k];",
                                    "gs += wg[(size_t)k * (size_t)I + (size_t)i % (size_t)I] * n[k];"),
    "ffn_down_transposed": ("orc_matvec(I, H, a, wd, proj);",
                            "for (int j = 0; j < H; ++j) {\n    proj[j] = 0.0;\n    "
                            "for (int i = 0; i < I; ++i) proj[j] += a[i] * wd[(size_t)j * (size_t)I + i];\n  }"),
    "mla_value_from_key_columns": ("const double* wvv = wk + dn;", "const double* wvv = wk;"),
    "mla_scale_without_rope_dims": ("const double scale = 1.0 / sqrt((double)dq);",
                                    "const double scale = 1.0 / sqrt((double)dn);"),
    "mla_no_latent_norm": ("orc_rmsnorm(dc, a, g_kv, c->rms_eps, a);", ""),
    "mla_rope_on_nope_part": ("orc_rope(dr, c->rope_theta, pos, q + (size_t)h * dq + dn);",
                              "orc_rope(dr, c->rope_theta, pos, q + (size_t)h * dq);"),
    "mla_no_rope_on_shared_key": ("orc_rope(dr, c->rope_theta, pos, a + dc);", ""),
    "mla_drop_new_token": ("const int dq = dn + dr, dl = dc + dr, ntok = pos + 1;",
                           "const int dq = dn + dr, dl = dc + dr, ntok = pos;"),
    "mla_head_stride_without_value": ("const double* wk = wukv + (size_t)h * (dn + dv);",
                                      "const double* wk = wukv + (size_t)h * dn;"),
    "mla_key_rope_part_from_latent_head": ("for (int j = 0; j < dr; ++j) kt[dn + j] = lt[dc + j];",
                                           "for (int j = 0; j < dr; ++j) kt[dn + j] = lt[j];"),
    "mla_drop_residual": ("for (int i = 0; i < H; ++i) out[i] = x[i] + proj[i];\n\n  if (dbg_q)",
                          "for (int i = 0; i < H; ++i) out[i] = proj[i];\n\n  if (dbg_q)"),
    "transposed_weight": (
        "const double* row = W + (size_t)i * (size_t)N;\n    for (int j = 0; j < N; ++j) y[j] += xi * row[j];",
        "for (int j = 0; j < N; ++j) y[j] += xi * W[(size_t)j * (size_t)K + i];"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(SRC).read()
    old, new = MUTATIONS[name]
    assert old in src, f"mutation anchor for {name} no longer present"
    cpath = tmp_path / f"{name}.c"
    cpath.write_text(src.replace(old, new, 1))
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-I", os.path.dirname(SRC), "-fPIC",
                           "-shared", str(cpath), "-o", str(so), "-lm"])
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=dict(os.environ, CF_ORACLE_LIB=str(so)),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"pins did not catch '{name}':\n{r.stdout[-2000:]}"
