"""The oracle's pins must catch a planted mistake (no GPU).

Each mutant below is a copy of the oracle with one plausible slip planted in
it -- a wrong sign, a dropped term or factor, an off-by-one, a wrong index or
grouping, a transposed operand. The copy is built in a temporary directory
together with a copy of ``test_oracle.py`` and its golden fixtures, and that
pin suite is run against it in a fresh interpreter; it must fail. The
unmodified copy must pass in the same harness, so a broken harness cannot
pass for a caught mutant.

The mistakes are planted in the oracle only, on the CPU; the repository's own
oracle is never modified.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (id, file under oracle/, text to find (must occur exactly once), replacement)
MUTANTS = [
    # RoPE ("Core Layers -- Deep Reference", RoPE): rotation and frequencies
    ("rope_sign", "oracle.c", "x[i] = a * cs - b * sn;", "x[i] = a * cs + b * sn;"),
    ("rope_second_half_swapped", "oracle.c", "x[i + half] = a * sn + b * cs;",
     "x[i + half] = b * sn + a * cs;"),
    ("rope_interleaved_pairs", "oracle.c",
     "double a = x[i], b = x[i + half];\n        x[i] = a * cs - b * sn;\n"
     "        x[i + half] = a * sn + b * cs;",
     "double a = x[2 * i], b = x[2 * i + 1];\n        x[2 * i] = a * cs - b * sn;\n"
     "        x[2 * i + 1] = a * sn + b * cs;"),
    ("freq_exponent_over_D", "oracle.c", "-(2.0 * i) / (double)R)", "-(2.0 * i) / (double)c->D)"),
    ("freq_exponent_drops_two", "oracle.c", "-(2.0 * i) / (double)R)", "-(1.0 * i) / (double)R)"),
    ("angle_uses_position_plus_one", "oracle.c", "double ang = (double)p * inv[i];",
     "double ang = (double)(p + 1) * inv[i];"),
    ("linear_scaling_multiplies", "oracle.c",
     "if (c->scaling_type == 1) {\n            f = f / c->factor;",
     "if (c->scaling_type == 1) {\n            f = f * c->factor;"),
    ("llama3_long_branch_not_divided", "oracle.c",
     "} else if (wavelength > long_wl) {\n                f = f / c->factor;",
     "} else if (wavelength > long_wl) {\n                f = f;"),
    ("llama3_ramp_weights_swapped", "oracle.c", "f = (1.0 - s) * f / c->factor + s * f;",
     "f = s * f / c->factor + (1.0 - s) * f;"),
    ("llama3_ramp_high_low_swapped", "oracle.c",
     "(c->high_freq_factor - c->low_freq_factor)", "(c->low_freq_factor - c->high_freq_factor)"),
    ("llama3_ramp_blends_wavelengths", "oracle.c", "f = (1.0 - s) * f / c->factor + s * f;",
     "f = 1.0 / ((1.0 - s) * c->factor / f + s / f);"),
    ("llama3_ramp_blends_log_frequency", "oracle.c", "f = (1.0 - s) * f / c->factor + s * f;",
     "f = exp((1.0 - s) * log(f / c->factor) + s * log(f));"),
    ("llama3_ramp_s_linear_in_wavelength", "oracle.c",
     "double s = (c->original_max_positions / wavelength - c->low_freq_factor) /\n"
     "                           (c->high_freq_factor - c->low_freq_factor);",
     "double s = (long_wl - wavelength) / (long_wl - short_wl);"),
    ("llama3_short_and_long_swapped", "oracle.c",
     "double short_wl = c->original_max_positions / c->high_freq_factor;",
     "double short_wl = c->original_max_positions / c->low_freq_factor;"),
    # RMSNorm ("Core Layers -- Deep Reference", RMSNorm) and its place before RoPE
    ("rmsnorm_drops_eps", "oracle.c", "double rms = sqrt(ss / D + eps);",
     "double rms = sqrt(ss / D);"),
    ("rmsnorm_sum_not_mean", "oracle.c", "double rms = sqrt(ss / D + eps);",
     "double rms = sqrt(ss + eps);"),
    ("rmsnorm_offset_weight", "oracle.c", "y[i] = x[i] / rms * w[i];",
     "y[i] = x[i] / rms * (1.0 + w[i]);"),
    ("norm_after_rope", "oracle.c",
     "if (norm_w) rmsnorm(xr, norm_w, D, c->norm_eps, yr);\n"
     "        else memcpy(yr, xr, sizeof(double) * D);\n"
     "        if (R > 0) rope_vec(yr, R, inv, (long)start[b] + l);",
     "memcpy(yr, xr, sizeof(double) * D);\n"
     "        if (R > 0) rope_vec(yr, R, inv, (long)start[b] + l);\n"
     "        if (norm_w) { double t[4096]; memcpy(t, yr, sizeof(double) * D);\n"
     "                      rmsnorm(t, norm_w, D, c->norm_eps, yr); }"),
    ("position_ignores_start", "oracle.c", "rope_vec(yr, R, inv, (long)start[b] + l);",
     "rope_vec(yr, R, inv, (long)l);"),
    # scores, mask and softmax ("Core Layers -- Deep Reference", MHA and GQA, sliding window)
    ("scale_over_rope_dim", "oracle.c", "1.0 / sqrt((double)c->D)", "1.0 / sqrt((double)c->rope_dim)"),
    ("scale_dropped", "oracle.c", "        s *= sc;\n", "\n"),
    ("scores_read_values", "oracle.c", "s += q[d] * keys[j][d];", "s += q[d] * vals[j][d];"),
    ("output_weighs_keys", "oracle.c", "out[d] += w * vals[j][d];", "out[d] += w * keys[j][d];"),
    ("softcap_drops_outer_factor", "oracle.c", "s = c->softcap * tanh(s / c->softcap);",
     "s = tanh(s / c->softcap);"),
    ("softcap_before_scale", "oracle.c",
     "s *= sc;\n        if (c->softcap > 0.0) s = c->softcap * tanh(s / c->softcap);",
     "if (c->softcap > 0.0) s = c->softcap * tanh(s / c->softcap);\n        s *= sc;"),
    ("not_normalised", "oracle.c", "for (int d = 0; d < D; ++d) out[d] /= den;", ""),
    ("window_admits_w_plus_one", "oracle.c", "if (W > 0 && m < p - W + 1) return 0;",
     "if (W > 0 && m < p - W) return 0;"),
    ("window_admits_w_minus_one", "oracle.c", "if (W > 0 && m < p - W + 1) return 0;",
     "if (W > 0 && m < p - W + 2) return 0;"),
    ("causal_sees_next_key", "oracle.c", "if (m > p) return 0;", "if (m > p + 1) return 0;"),
    ("gqa_interleaved_groups", "oracle.c", "int G = H / Hkv, hk = h / G;",
     "int G = H / Hkv, hk = h % Hkv; (void)G;"),
    ("prefill_key_positions_ignore_start", "oracle.c", "pos[j] = (long)start[b] + j;",
     "pos[j] = j;"),
    # cache slots and decode ("mojolearn.transformer", TransformerState and step)
    ("ring_slot_shifted", "oracle.c", "return W > 0 ? m % W : m;",
     "return W > 0 ? (m + 1) % W : m;"),
    ("decode_query_one_position_early", "oracle.c",
     "attend(c, qr + r * D, kp, vp, pos, n, p, out + r * D, scratch);",
     "attend(c, qr + r * D, kp, vp, pos, n, p - 1, out + r * D, scratch);"),
    ("decode_positions_are_slots", "oracle.c", "pos[n] = m;", "pos[n] = slot_of(m, W);"),
    ("decode_interleaved_groups", "oracle.c", "int b = (int)(r / H), h = (int)(r % H), hk = h / G;",
     "int b = (int)(r / H), h = (int)(r % H), hk = h % Hkv; (void)G;"),
    ("sampled_rows_head_and_position_swapped", "oracle.c",
     "rows[3 * i], rows[3 * i + 1], rows[3 * i + 2]",
     "rows[3 * i], rows[3 * i + 2], rows[3 * i + 1]"),
    ("rotate_rows_position_index", "oracle.c",
     "int l = (int)(r % L);\n        const double* xr",
     "int l = (int)((r / L) % L);\n        const double* xr"),
    ("rotate_rows_first_batch_start", "oracle.c", "int b = (int)(r / ((long)NH * L));",
     "int b = 0; (void)NH;"),
    ("append_values_from_keys", "oracle.c", "memcpy(vc + dst, v + src, sizeof(double) * D);",
     "memcpy(vc + dst, kr + src, sizeof(double) * D);"),
    ("append_records_the_slot", "oracle.c",
     "written[((long)b * Hkv + hk) * capacity + s] = m;",
     "written[((long)b * Hkv + hk) * capacity + s] = s;"),
    ("decode_values_from_key_cache", "oracle.c", "vp[n] = vc + off;", "vp[n] = kc + off;"),
    ("decode_rows_share_the_first_length", "oracle.c", "long p = (long)cache_len[b] - 1;",
     "long p = (long)cache_len[0] - 1;"),
    # the ragged batch and the decoder block (numpy, oracle/__init__.py)
    ("ragged_padding_keeps_full_length_rows", "__init__.py",
     "        out[b, :, :n] = o[0]\n",
     "        out[b, :, :n] = o[0]\n"
     "        out[b, :, n:] = prefill(q[b:b + 1], k[b:b + 1], v[b:b + 1], [0], "
     "Cfg(**{**cfg.__dict__, 'B': 1}), q_norm_w, k_norm_w)[0][0][:, n:]\n"),
    ("silu_sign", "__init__.py", "act = gate / (1.0 + np.exp(-gate)) * up",
     "act = gate / (1.0 + np.exp(gate)) * up"),
    ("mlp_gate_and_up_swapped", "__init__.py", "act = gate / (1.0 + np.exp(-gate)) * up",
     "act = up / (1.0 + np.exp(-up)) * gate"),
    ("attention_residual_dropped", "__init__.py",
     "h = x + attn.transpose(0, 2, 1, 3)", "h = attn.transpose(0, 2, 1, 3)"),
    ("mlp_residual_dropped", "__init__.py", "return h + act @ W[\"down_proj.weight\"].T",
     "return act @ W[\"down_proj.weight\"].T"),
    ("heads_split_token_major", "__init__.py",
     "return y.reshape(B, L, nh, D).transpose(0, 2, 1, 3)", "return y.reshape(B, nh, L, D)"),
    ("post_norm_reads_input", "__init__.py",
     "n2 = rmsnorm(h, W[\"post_attention_layernorm.weight\"]",
     "n2 = rmsnorm(x, W[\"post_attention_layernorm.weight\"]"),
    ("offset_norm_ignored", "__init__.py", "scale = (1.0 + _f64(w)) if offset else _f64(w)",
     "scale = _f64(w)"),
]


def _make_copy(dst, mutant):
    """A self-contained copy of the oracle and its pin suite, with one mistake planted."""
    os.makedirs(os.path.join(dst, "oracle"))
    for name in ("oracle.c", "__init__.py"):
        shutil.copy(os.path.join(ROOT, "oracle", name), os.path.join(dst, "oracle", name))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    for name in ("conftest.py", "test_oracle.py"):
        shutil.copy(os.path.join(ROOT, "tests", name), os.path.join(dst, "tests", name))
    if mutant is not None:
        _, fname, find, repl = mutant
        path = os.path.join(dst, "oracle", fname)
        with open(path) as f:
            text = f.read()
        assert text.count(find) == 1, f"{mutant[0]}: pattern occurs {text.count(find)} times"
        with open(path, "w") as f:
            f.write(text.replace(find, repl))


def _run_pins(dst):
    env = {k: v for k, v in os.environ.items() if k != "PYTHONPATH"}
    env["OMP_NUM_THREADS"] = "1"
    proc = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
         os.path.join("tests", "test_oracle.py")],
        cwd=dst, env=env, capture_output=True, text=True, timeout=600)
    return proc.returncode, proc.stdout[-3000:] + proc.stderr[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    base = tmp_path_factory.mktemp("oracle_mutants")
    jobs = [("unmodified", None)] + [(m[0], m) for m in MUTANTS]
    for name, m in jobs:
        _make_copy(str(base / name), m)
    with ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
        results = list(ex.map(lambda j: _run_pins(str(base / j[0])), jobs))
    return {name: r for (name, _), r in zip(jobs, results)}


def test_mutant_ids_are_unique():
    ids = [m[0] for m in MUTANTS]
    assert len(ids) == len(set(ids))


def test_unmodified_copy_passes_its_pins(outcomes):
    rc, log = outcomes["unmodified"]
    assert rc == 0, log


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(outcomes, mutant):
    rc, log = outcomes[mutant[0]]
    assert rc == 1, f"mistake {mutant[0]!r} planted in oracle/{mutant[1]} was not caught " \
                    f"(pytest exit {rc}):\n{log}"
