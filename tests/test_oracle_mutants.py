"""Planted mistakes in a copy of the oracle must fail at least one pin (no GPU).

Each mutant is a one-line edit of ``oracle/attn_oracle.c`` of the kind a careful
author could still make: a dropped scale, a transposed operand, a flipped or
off-by-one mask, a wrong stride or head offset, a missing normalisation or log.
It is compiled into a temporary directory and the pins of ``oracle_pins.py`` run
against it in a child process (so an out-of-range read in a mutant cannot take
the test runner down). The real oracle source is never modified.
"""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

MUTANTS = {
    "scale_dropped": ("s[j] = p->scale * dot;", "s[j] = dot;"),
    "k_transposed": ("elem(p->q, p->dtype, qoff + t) * elem(p->k, p->dtype, koff + (long long)j * p->d_k + t)",
                     "elem(p->q, p->dtype, qoff + t) * elem(p->k, p->dtype, koff + (long long)t * p->n_k + j)"),
    "causal_flipped": ("&& j > i) return 0;", "&& j < i) return 0;"),
    "causal_off_by_one": ("&& j > i) return 0;", "&& j >= i) return 0;"),
    "padding_off_by_one": ("j >= p->key_lens[b]", "j > p->key_lens[b]"),
    "padding_wrong_batch": ("int b = bh / p->H;", "int b = bh % p->B;"),
    "mask_ignored": ("if (!legal(p, b, i, j)) {", "if (0) {"),
    "exp_sign": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "not_normalised": ("s[j] = s[j] / l;", "s[j] = s[j];"),
    "lse_missing_log": ("? m + log(l) :", "? m + l :"),
    "v_row_stride": ("o[t] += s[j] * elem(p->v, p->dtype, voff + (long long)j * p->d_v + t)",
                     "o[t] += s[j] * elem(p->v, p->dtype, voff + (long long)j * p->d_k + t)"),
    "k_head_offset": ("long long koff = (long long)bh * p->n_k * p->d_k;",
                      "long long koff = (long long)(bh / p->H) * p->n_k * p->d_k;"),
    "v_head_offset": ("long long voff = (long long)bh * p->n_k * p->d_v;",
                      "long long voff = (long long)(bh / p->H) * p->n_k * p->d_v;"),
    "q_row_reversed": ("((long long)bh * p->n_q + i) * p->d_k", "((long long)bh * p->n_q + (p->n_q - 1 - i)) * p->d_k"),
    "bf16_widening": ("<< 16;", "<< 15;"),
    "decode_off_by_one": ("j > p->key_lens[b] - p->n_q + i", "j >= p->key_lens[b] - p->n_q + i"),
    "decode_start_aligned": ("j > p->key_lens[b] - p->n_q + i", "j > i"),
    "window_one_sided": ("(j > i + p->window || j < i - p->window)", "(j > i + p->window)"),
    "bwd_no_jacobian_correction": ("const double ds = w[j] * (dp[j] - sum_pdp);", "const double ds = w[j] * dp[j];"),
    "bwd_jacobian_sign": ("const double ds = w[j] * (dp[j] - sum_pdp);", "const double ds = w[j] * (sum_pdp - dp[j]);"),
    "bwd_dk_unscaled": ("dk[koff + (long long)j * p->d_k + t] += p->scale * ds *", "dk[koff + (long long)j * p->d_k + t] += ds *"),
    "bwd_dq_uses_q": ("dq[qoff + (long long)i * p->d_k + t] += p->scale * ds * elem(p->k, p->dtype, koff + (long long)j * p->d_k + t);",
                      "dq[qoff + (long long)i * p->d_k + t] += p->scale * ds * elem(p->q, p->dtype, qoff + (long long)i * p->d_k + t);"),
    "bwd_dv_unweighted": ("dv[voff + (long long)j * p->d_v + t] += w[j] *", "dv[voff + (long long)j * p->d_v + t] += (w[j] > 0.0) *"),
    "window_off_by_one": ("(j > i + p->window || j < i - p->window)", "(j >= i + p->window || j <= i - p->window)"),
    # multi-head attention: projections, head split, concatenation, output projection
    "mha_q_from_kv_source": ("project_heads(x_q, w_q, b_q,", "project_heads(x_kv, w_q, b_q,"),
    "mha_heads_interleaved": ("const long long col = (long long)h * d + t;", "const long long col = (long long)t * H + h;"),
    "mha_projection_bias_dropped": ("double acc = bias ? elem(bias, dtype, col) : 0.0;", "double acc = 0.0;"),
    "mha_output_bias_dropped": ("double acc = b_o ? elem(b_o, dtype, c) : 0.0;", "double acc = 0.0;"),
    "mha_w_o_transposed": ("elem(w_o, dtype, ((long long)h * d_v + t) * d_model + c)",
                           "elem(w_o, dtype, (long long)c * H * d_v + (long long)h * d_v + t)"),
    # linear projection
    "linear_w_transposed": ("elem(w, dtype, (long long)k * N + n)", "elem(w, dtype, (long long)n * K + k)"),
    "linear_bias_dropped": ("double acc = bias ? elem(bias, dtype, n) : 0.0;", "double acc = 0.0;"),
    "linear_x_row_stride": ("elem(x, dtype, (long long)m * K + k)", "elem(x, dtype, (long long)m * N + k)"),
    "mha_concat_batch_head_swapped": ("oh[(((long long)b * H + h) * n_q + i) * d_v + t]",
                                      "oh[(((long long)h * B + b) * n_q + i) * d_v + t]"),
}

_CHILD = r"""
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle
from oracle_pins import PINS
orc = oracle.Oracle({lib!r})
failed = []
for pin in PINS:
    try:
        pin(orc)
    except Exception as e:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    with open(oracle.SRC) as f:
        src = f.read()
    before, after = MUTANTS[name]
    assert src.count(before) == 1, f"mutation site for {name!r} not found exactly once in the oracle source"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    tests = os.path.dirname(os.path.abspath(__file__))
    with tempfile.TemporaryDirectory() as tmp:
        src_path = os.path.join(tmp, "attn_oracle.c")
        with open(src_path, "w") as f:
            f.write(src.replace(before, after))
        lib = oracle.build(src_path, os.path.join(tmp, "liboracle_mutant.so"))
        code = _CHILD.format(root=root, tests=tests, lib=lib)
        res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    caught = [ln for ln in res.stdout.splitlines() if ln.startswith("FAILED:")]
    # a crash of the child also counts as caught; a clean run with no failed pin does not
    assert res.returncode != 0 or (caught and caught[-1] != "FAILED:"), f"mutant {name!r} passed every pin"
