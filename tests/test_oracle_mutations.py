"""The pins have teeth: plausible mistakes planted in copies of the oracle are caught.

Each mutation edits one line of ``oracle/mla_oracle.c`` in a temporary copy, builds
it, and runs the pin suite against that build in a subprocess; the suite must fail.
Nothing here touches the committed oracle or the GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mla_oracle.c")

MUTATIONS = {
    "rope_sign": ("y[t] = x0 * c - x1 * s;", "y[t] = x0 * c + x1 * s;"),
    "rope_theta": ("pow(base, -2.0 * (double)t / (double)d)", "pow(base, -1.0 * (double)t / (double)d)"),
    "rms_eps_outside_sqrt": ("1.0 / sqrt(ss / (double)d + eps)", "1.0 / (sqrt(ss / (double)d) + eps)"),
    "dropped_rope_score_term": ("sc[j] = scale * (dot(qn, kn + j * Dn, Dn) +",
                                "sc[j] = scale * (dot(qn, kn + j * Dn, Dn) + 0.0 *"),
    "k_from_v_rows": ("kn[j * Dn + d] = dot(wk + (size_t)d * Dk, cj, Dk);",
                      "kn[j * Dn + d] = dot(wk + (size_t)(d + 1) * Dk, cj, Dk);"),
    "causal_off_by_one": ("long n = pos + 1;", "long n = pos;"),
    "combine_weight": ("acc += exp(part_lse[(size_t)s * rows + r] - l) *",
                       "acc += exp(part_lse[(size_t)s * rows + r] - m) *"),
    "bwd_softmax_no_D": ("const double ds = p * (dot(dO, vv + j * Dv, Dv) - Di);",
                         "const double ds = p * dot(dO, vv + j * Dv, Dv);"),
    "bwd_rope_transpose_sign": ("rope_row(dqr, -(double)pos, Dr, base, dq_pe + qrow * Dr);",
                                "rope_row(dqr, (double)pos, Dr, base, dq_pe + qrow * Dr);"),
    "bwd_rms_dropped_term": ("dx[k] = dy[k] * rms_w[k] / r - x[k] * g / ((double)Dk * r * r * r);",
                             "dx[k] = dy[k] * rms_w[k] / r;"),
    "tpla_rope_band_dropped": ("sc[j] = scale * (dot(qa + k0, cb + j * Dk + k0, ds) + dot(qr, kb + j * Dr, Dr));",
                               "sc[j] = scale * dot(qa + k0, cb + j * Dk + k0, ds);"),
    "tpla_wv_shard_offset": ("out[row * Dv + d] += dot(wv + (size_t)d * Dk + k0, ol + k0, ds);",
                             "out[row * Dv + d] += dot(wv + (size_t)d * Dk, ol + k0, ds);"),
    "tpla_norm_weight_slice": ("rmsnorm_row(c_raw + r * Dk + (size_t)i * ds, rms_w + (size_t)i * ds, ds, eps,",
                               "rmsnorm_row(c_raw + r * Dk + (size_t)i * ds, rms_w, ds, eps,"),
    "rms_weight_dropped": ("y[k] = x[k] * inv * w[k];", "y[k] = x[k] * inv;"),
    "head_offset_ignored": ("int h = head_begin + hl;", "int h = hl;"),
    "decode_query_position": ("(double)(kv_len - 1)", "(double)kv_len"),
    "split_chunk_rounded_down": ("((long)kv_len + n_splits - 1) / n_splits", "(long)kv_len / n_splits"),
    "unabsorb_reads_k_rows": ("                const double *wv = wk + (size_t)Dn * Dk;\n                double *qa",
                              "                const double *wv = wk;\n                double *qa"),
    "absorb_transposed": ("acc += qn[d] * wk[(size_t)d * Dk + k];\n                    qa[k] = acc;",
                          "acc += qn[d] * wk[(size_t)k * Dn + d];\n                    qa[k] = acc;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: " + name
    mutated = tmp_path / "mla_oracle_mut.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = tmp_path / "libmla_oracle_mut.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-ffp-contract=off", str(mutated), "-o", str(lib), "-lm"])
    env = dict(os.environ, MLA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    # caught = a test FAILED (pytest exit code 1), not a collection error or a crash
    tail = r.stdout.strip().splitlines()[-1] if r.stdout.strip() else ""
    assert r.returncode == 1, "pins did not catch mutation %s (rc %d):\n%s" % (name, r.returncode, r.stdout[-2000:])
    assert " failed" in tail and "error" not in tail, "mutation %s: %s" % (name, tail)
