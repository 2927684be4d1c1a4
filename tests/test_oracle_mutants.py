"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that the pins catch each.

Every entry replaces one exact piece of ``oracle/onebit_oracle.c``: a dropped term, a wrong sign, a
transposed operand or index, a wrong convention.  The mutated copy is compiled into a temporary
directory and every pin of ``oracle_pins.py`` is run against it; at least one must fail.
"""
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "onebit_oracle.c")

MUTANTS = {
    "worker_error_sign": ("err[e] = (c[e] >= 0.0f) ? c[e] - s : c[e] + s;",
                          "err[e] = (c[e] >= 0.0f) ? s - c[e] : -s - c[e];"),
    "worker_error_zero_sign": ("err[e] = (c[e] >= 0.0f) ? c[e] - s : c[e] + s;",
                               "err[e] = (c[e] > 0.0f) ? c[e] - s : c[e] + s;"),
    "error_not_added": ("c[(int64_t)i * D + p] = mi + delta[(int64_t)i * D + p];",
                        "c[(int64_t)i * D + p] = mi;"),
    "momentum_operands_swapped": ("const float mi = b1 * m[p] + omb1 * ora_grad_value(g, cfg->grad_dtype, e);",
                                  "const float mi = omb1 * m[p] + b1 * ora_grad_value(g, cfg->grad_dtype, e);"),
    "server_sum_not_averaged": ("a[off + e] = acc / (float)n + eps_srv[off + e];",
                                "a[off + e] = acc + eps_srv[off + e];"),
    "server_error_subtracted": ("a[off + e] = acc / (float)n + eps_srv[off + e];",
                                "a[off + e] = acc / (float)n - eps_srv[off + e];"),
    "rms_without_len": ("return (float)sqrt((sum + comp) / (double)len);", "return (float)sqrt(sum + comp);"),
    "rms_without_sqrt": ("return (float)sqrt((sum + comp) / (double)len);",
                         "return (float)((sum + comp) / (double)len);"),
    "shard_not_word_aligned": ("int64_t per = 32 * ((len + 32 * (int64_t)n - 1) / (32 * (int64_t)n));",
                               "int64_t per = (len + (int64_t)n - 1) / (int64_t)n;"),
    "sign_of_zero": ("if (v[e] >= 0.0f) words[e / 32] |= 1u << (e % 32);",
                     "if (v[e] > 0.0f) words[e / 32] |= 1u << (e % 32);"),
    "bit_order_reversed": ("if (v[e] >= 0.0f) words[e / 32] |= 1u << (e % 32);",
                           "if (v[e] >= 0.0f) words[e / 32] |= 1u << (31 - e % 32);"),
    "update_sign": ("x[p] = x[p] - cfg->lr * (m[p] / den[p]);", "x[p] = x[p] + cfg->lr * (m[p] / den[p]);"),
    "variance_not_decayed": ("*v = b2 * *v + omb2 * (g * g);", "*v = *v + omb2 * (g * g);"),
    "eps_inside_sqrt": ("den[p] = sqrtf(vu) + cfg->eps;", "den[p] = sqrtf(vu + cfg->eps);"),
    "bias_correction_inverted": ("mh = mh / bc1;", "mh = mh * bc1;"),
    "broadcast_uncompressed": ("bcast[p] = bit ? S : -S;", "bcast[p] = a[p];"),
    "half_exponent_bias": ("mag = ldexpf((float)(1024 + frac), expo - 25);",
                           "mag = ldexpf((float)(1024 + frac), expo - 24);"),
    "bf16_shift": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    "server_error_dropped": ("eps_srv[p] = bit ? a[p] - S : a[p] + S;", "eps_srv[p] = 0.0f;"),
    "server_sign_of_zero": ("const int bit = a[p] >= 0.0f;", "const int bit = a[p] > 0.0f;"),
    "worker_scale_index_transposed": ("const float s = wscale[(int64_t)i * T + k];",
                                      "const float s = wscale[(int64_t)k * n + i];"),
    "warmup_sum_not_averaged": ("const float g = acc / (float)n;", "const float g = acc;"),
    "norm2_without_sqrt": ("  return sqrt(sum + comp);\n}", "  return sum + comp;\n}"),
    "ec_adam_compresses_momentum": (
        "c[(int64_t)i * D + p] = ora_grad_value(g, cfg->grad_dtype, e) + delta[(int64_t)i * D + p];",
        "c[(int64_t)i * D + p] = cfg->beta1 * m[p] + (1.0f - cfg->beta1) * ora_grad_value(g, cfg->grad_dtype, e)"
        " + delta[(int64_t)i * D + p];"),
    "ec_adam_update_from_local_gradient": (
        "for (int64_t p = 0; p < D; ++p) adam_element(cfg, bc1, bc2, bcast[p], &m[p], &v[p], &x[p]);",
        "for (int64_t p = 0; p < D; ++p) adam_element(cfg, bc1, bc2, c[p], &m[p], &v[p], &x[p]);"),
    "warmup_reads_one_worker": ("acc = acc + ora_grad_value(grads[(int64_t)i * T + k], cfg->grad_dtype, e);",
                                "acc = acc + ora_grad_value(grads[k], cfg->grad_dtype, e);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique or missing: {old}"
    mut_src = tmp_path / "onebit_oracle.c"
    mut_src.write_text(src.replace(old, new))
    so = oracle.build(force=True, src=str(mut_src), out=str(tmp_path / "libmutant.so"))
    # run the pins in a child process, so that a mutant that corrupts memory cannot take the test
    # session down with it
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import oracle, oracle_pins\n"
        "lib = oracle.OracleLib(%r)\n"
        "for pin in oracle_pins.ALL_PINS:\n"
        "    try:\n"
        "        pin(lib)\n"
        "    except Exception as e:\n"
        "        print('CAUGHT', pin.__name__, type(e).__name__); sys.exit(0)\n"
        "print('MISSED')\n"
    ) % (here, os.path.dirname(here), so)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert "MISSED" not in r.stdout, f"no pin catches mutation {name}"
    assert "CAUGHT" in r.stdout or r.returncode != 0, r.stdout + r.stderr
