"""Mutation check of the oracle pins (CPU only).

Each case plants one plausible mistake in a private copy of the C oracle
(a dropped term, a wrong sign, a wrong or transposed index), builds it, and
runs the pin suite against it in a subprocess: every mutant must make at
least one pin fail.  The real oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "attnres_oracle.c")

MUTANTS = {
    "mean_square_not_divided_by_n": [("    ms /= (double)n;\n", "")],
    "eps_outside_sqrt": [("sqrt(ms + eps)", "(sqrt(ms) + eps)")],
    "softmax_sign": [("alpha[i] = exp(s[i] - m)", "alpha[i] = exp(m - s[i])")],
    "first_source_dropped_from_sum": [
        ("for (int64_t i = 0; i < n_src; ++i) acc += a[i] * rows[i][c];",
         "for (int64_t i = 1; i < n_src; ++i) acc += a[i] * rows[i][c];")],
    "gain_ignored": [("double gc = g ? g[c] : 1.0;", "double gc = 1.0;")],
    "lse_drops_max": [("return m + log(l);", "return log(l);")],
    "merge_sign": [("double a = exp(lse[t] - M), b = exp(sp - M);", "double a = exp(lse[t] - M), b = exp(M - sp);")],
    "mhar_phase2_merge_sign": [("double a = exp(l - M), b = exp(sp - M);\n            for (int64_t c = 0; c < dh; ++c)",
                                "double a = exp(l - M), b = exp(M - sp);\n            for (int64_t c = 0; c < dh; ++c)")],
    "first_layer_reads_partial": [("if (li >= 1) { rows[N]", "if (li >= 0) { rows[N]")],
    "mhar_query_transposed": [("queries + (q * H + hd) * dh", "queries + (hd * n_q + q) * dh")],
    "bwd_softmax_mean_dropped": [("ds[q * n_src + i] = a[q * n_src + i] * (ds[q * n_src + i] - mean + (dlse",
                                  "ds[q * n_src + i] = a[q * n_src + i] * (ds[q * n_src + i] + (dlse")],
    "bwd_lse_gradient_sign": [("- mean + (dlse ? dlse[q * T + t] : 0.0));", "- mean - (dlse ? dlse[q * T + t] : 0.0));")],
    "merge_bwd_dlse_without_b": [("dlse[t] = a * b * hdiff;", "dlse[t] = a * hdiff;")],
    "merge_bwd_value_path_weight": [("double dp = b * ht[c];", "double dp = a * ht[c];")],
    "merge_bwd_rms_term_sign": [("dp += dsp * (gc * query[c] / r - pt[c] * wgp", "dp += dsp * (gc * query[c] / r + pt[c] * wgp")],
    "bwd_rms_term_sign": [("dv[c] += gc * dk[c] / r[i] - v[c] * gdkv", "dv[c] += gc * dk[c] / r[i] + v[c] * gdkv")],
    "bwd_gain_grad_not_normalised": [("dg[c] += dk[c] * v[c] / r[i];", "dg[c] += dk[c] * v[c];")],
    "bwd_value_path_first_query_weights": [("dv[c] += a[q * n_src + i] * dh[c];", "dv[c] += a[i] * dh[c];")],
    "mhar_bwd_gain_not_sliced": [("for (int64_t c = 0; c < dh; ++c) g_h[c] = gain ? gain[c0 + c] : 1.0;",
                                  "for (int64_t c = 0; c < dh; ++c) g_h[c] = gain ? gain[c] : 1.0;")],
    "mhar_bwd_dout_of_first_head": [("do_h[(q * T + t) * dh + c] = dout[(q * T + t) * d + c0 + c];",
                                     "do_h[(q * T + t) * dh + c] = dout[(q * T + t) * d + c];")],
    "mhar_bwd_query_grad_unsliced": [("dq[q * d + c0 + c] = dq_h[q * dh + c];", "dq[q * d + c] = dq_h[q * dh + c];")],
    "msar_phase1_layer_stream_transposed": [("queries + (sl * m + r) * d, gain, eps,",
                                             "queries + (r * S + sl) * d, gain, eps,")],
    "msar_phase2_merge_sign": [("double a = exp(l - M), b = exp(sp - M);\n            for (int64_t c = 0; c < d; ++c) zr[c]",
                                "double a = exp(l - M), b = exp(M - sp);\n            for (int64_t c = 0; c < d; ++c) zr[c]")],
    "msar_phase2_partial_identity_streams": [("if (rc == 0 && partial) rc = msar_expand(partial, T, d, m, ksizes, conv_w, up);",
                                              "if (rc == 0 && partial) rc = msar_expand(partial, T, d, 1, ksizes, conv_w, up);\n    for (int64_t r = 1; r < m && up; ++r) memcpy(up + (size_t)r * per, partial, sizeof(double) * per);")],
    "msar_phase2_lse_of_stream_zero": [("const double l = lse[r * T + t];\n            double sp = score(",
                                        "const double l = lse[t];\n            double sp = score(")],
    "msar_ps_first_source_kernels": [("conv_w + i * conv_src_stride,", "conv_w,")],
    "msar_bwd_sigmoid_derivative": [("dl[o] = dc * c[o] * (1.0 - c[o]);", "dl[o] = dc * c[o];")],
    "msar_bwd_mixer_rms_sign": [("/ nu - zf[kk] * s / ((double)md * nu * nu * nu);", "/ nu + zf[kk] * s / ((double)md * nu * nu * nu);")],
    "msar_bwd_conv_transpose_unshifted": [("dv[(t - j) * d + k] += cw[k * kr + j] * dui[t * d + k];",
                                           "dv[t * d + k] += cw[k * kr + j] * dui[t * d + k];")],
    "msar_bwd_kernel_grad_unshifted": [("dcw[k * kr + j] += dui[t * d + k] * v[(t - j) * d + k];",
                                        "dcw[k * kr + j] += dui[t * d + k] * v[t * d + k];")],
    "msar_ps_bwd_shared_kernel_in_transpose": [("const double *cw = conv_w + i * conv_src_stride + off;",
                                                "const double *cw = conv_w + off;")],
    "msar_ps_bwd_kernel_grad_not_per_source": [("double *dcw = dconv_w + i * conv_src_stride + off;",
                                                "double *dcw = dconv_w + off;")],
    "msar_phase1_bwd_drops_dlse": [("rc = oracle_read_bwd_lse(ur, n_src, T, d, qr, S, gain, eps, dor, dlr, du, dqr, dgr);",
                                    "rc = oracle_read_bwd_lse(ur, n_src, T, d, qr, S, gain, eps, dor, NULL, du, dqr, dgr);")],
    "msar_phase2_bwd_drops_partial_identity_stream": [("for (size_t k = 0; k < per; ++k) d_partial[k] += dup[k];", "")],
    "msar_phase2_bwd_query_of_stream_zero": [("query + r * d, gain, eps, dZ + (size_t)r * per, d_o + (size_t)r * per,",
                                              "query, gain, eps, dZ + (size_t)r * per, d_o + (size_t)r * per,")],
    "msar_phase1_bwd_queries_stream_major": [("memcpy(qr + sl * d, queries + (sl * m + r) * d,",
                                              "memcpy(qr + sl * d, queries + (r * S + sl) * d,")],
    "msar_mix_bwd_gain_grad_missing_nu": [("if (nu > 0.0) dmix_gain[k] += acc * zf[k] / nu;",
                                           "if (nu > 0.0) dmix_gain[k] += acc * zf[k];")],
    "update_drops_old_partial": [("p_out[t * d + c] = (p ? p[t * d + c] : 0.0) + f[t * d + c];",
                                  "p_out[t * d + c] = f[t * d + c];")],
    "mhar_phase2_lse_transposed": [("const double l = lse[hd * T + t];", "const double l = lse[t * H + hd];")],
    "mhar_phase2_gain_not_sliced": [("double sp = score(query + hd * dh, ph, gain ? gain + hd * dh : NULL, dh, eps, tmp);",
                                     "double sp = score(query + hd * dh, ph, gain, dh, eps, tmp);")],
    "conv_kernel_reversed": [("acc += cw[c * k + j] * v[(t - j) * d + c];",
                              "acc += cw[c * k + (k - 1 - j)] * v[(t - j) * d + c];")],
    "conv_anticausal": [("if (t - j >= 0) acc += cw[c * k + j] * v[(t - j) * d + c];",
                         "if (t + j < T) acc += cw[c * k + j] * v[(t + j) * d + c];")],
    "flatten_channel_major": [("acc += zf[k] * mix_w[k * m + o];",
                               "acc += zf[k] * mix_w[((k % d) * m + k / d) * m + o];")],
    "sigmoid_sign": [("logit[o] = 1.0 / (1.0 + exp(-acc));", "logit[o] = 1.0 / (1.0 + exp(acc));")],
    "mixer_wrong_stream_weight": [("acc += logit[r] * Z[r * d + c];",
                                   "acc += logit[0] * Z[r * d + c];")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    c = tmp_path / "mutant.c"
    c.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                           "-o", str(so), str(c), "-lm"])
    env = dict(os.environ, ATTNRES_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
