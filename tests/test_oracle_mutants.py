"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle's C source (a flipped sign, a
transposed operand, a dropped term, a wrong index, a reversed tie-break ...), builds it, and runs the
pin suite against that build in a subprocess.  The numpy parts of the oracle (the log-sum-exp merge,
the basis fit, the predictor's gradient and Adam, the attention mass and the eviction plan) get the
same treatment through a temporary copy of the oracle package that the subprocess imports first.  The
suite must fail for every mutant.  Nothing here touches the real oracle build or a GPU.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "lowram_oracle.c")

MUTANTS = {
    "rope_sign": ("y[i + h] = b * c + a * s;", "y[i + h] = b * c - a * s;"),
    "rope_frequency": ("double w = pow(theta, -2.0 * i / d);\n        double c = cos",
                       "double w = pow(theta, -1.0 * i / d);\n        double c = cos"),
    "mlp_w1_transposed": ("acc += w1[(int64_t)j * d + i] * k_pre[i];", "acc += w1[(int64_t)i * m + j] * k_pre[i];"),
    "mlp_b2_dropped": ("double acc = b2 ? b2[i] : 0.0;", "double acc = 0.0;"),
    "mlp_no_silu": ("hidden_scratch[j] = silu(acc);", "hidden_scratch[j] = acc;"),
    "residual_not_added": ("v[(int64_t)j * d + i] += rv[i];", "v[(int64_t)j * d + i] += 0.0 * rv[i];"),
    "gqa_interleaved": ("q + ((int64_t)b * Hq + h * g + jq) * d;", "q + ((int64_t)b * Hq + jq * Hkv + h) * d;"),
    "tie_break_reversed": ("return (a->t > b->t) - (a->t < b->t);", "return (a->t < b->t) - (a->t > b->t);"),
    "selects_smallest": ("if (a->v > b->v) return -1;\n    if (a->v < b->v) return 1;",
                         "if (a->v < b->v) return -1;\n    if (a->v > b->v) return 1;"),
    "selection_ignored": ("top_n_ascending(T, kv, S_eff, chosen);",
                          "top_n_ascending(T, kv, S_eff, chosen); for (int j = 0; j < S_eff; ++j) chosen[j] = j;"),
    "softmax_not_normalised": ("for (int i = 0; i < d; ++i) o[i] /= den;\n                if (lse)",
                               "for (int i = 0; i < d; ++i) o[i] /= 1.0;\n                if (lse)"),
    "scale_wrong": ("return D->sm_scale > 0 ? D->sm_scale : 1.0 / sqrt((double)D->d);",
                    "return D->sm_scale > 0 ? D->sm_scale : 1.0 / (double)D->d;"),
    "key_sum_not_max": ("if (dot * scale > best) best = dot * scale;", "best = (jq == 0 ? 0.0 : best) + dot * scale;"),
    "error_squared": ("e[t] = sqrt(ss);", "e[t] = ss;"),
    "residual_sign": ("rr[i] = vt[i] - vhat[(int64_t)t * d + i];", "rr[i] = vhat[(int64_t)t * d + i] - vt[i];"),
    "projection_transposed": ("acc += proj[k * N + n] * kp[n];", "acc += proj[(n % r) * N + (k % N)] * kp[n];"),
    "basis_row_offset": ("basis + ((int64_t)h * D->d + i) * D->r;", "basis + ((int64_t)i * D->H_kv + h) * D->r;"),
    "unrotate_not_inverse": ("if (keys_post_rope) lro_rope(d, theta, p, kr + off, kp + off, 1);",
                             "if (keys_post_rope) lro_rope(d, theta, p, kr + off, kp + off, 0);"),
    "position_ignored": ("double p = pos ? (double)pos[(int64_t)b * T + t] : (double)t;\n                rebuild_key",
                         "double p = (double)t;\n                rebuild_key"),
    "int4_nibbles_swapped": ("(uint8_t)((lo & 0xF) | ((hi & 0xF) << 4));", "(uint8_t)((hi & 0xF) | ((lo & 0xF) << 4));"),
    "int4_round_half_away": ("double c = nearbyint(x / scale);", "double c = round(x / scale);"),
    "bf16_nine_bits": ("return round_to_format(x, 8, -126,", "return round_to_format(x, 9, -126,"),
    "f16_scale_unrounded": ("double s = lro_round_f16_scalar(amax / 7.0);", "double s = amax / 7.0;"),
}


def _run_mutant(name, find, repl, tmp):
    src = open(SRC).read()
    assert src.count(find) >= 1, f"mutation site of {name} not found"
    mut = src.replace(find, repl, 1)
    c_path = os.path.join(tmp, f"{name}.c")
    so_path = os.path.join(tmp, f"{name}.so")
    open(c_path, "w").write(mut)
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", so_path, c_path, "-lm"])
    env = dict(os.environ, LOWRAM_ORACLE_LIB=so_path, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
            results = list(ex.map(lambda kv: _run_mutant(kv[0], *kv[1], tmp), MUTANTS.items()))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, "mutants not caught by any pin: " + ", ".join(n for n, _ in survivors)


PY_SRC = os.path.join(ROOT, "oracle", "oracle.py")

PY_MUTANTS = {
    "merge_weight_sign": ("b = np.where(empty, 0.0, np.exp(lb - Wf))", "b = np.where(empty, 0.0, np.exp(Wf - lb))"),
    "merge_lse_without_max": ("lse = np.where(empty, -np.inf, Wf + np.log(", "lse = np.where(empty, -np.inf, np.log("),
    "basis_smallest_eigenvectors": ("order = np.argsort(w)[::-1][:r]", "order = np.argsort(w)[:r]"),
    "basis_rope_not_inverted": ("K = rope_rows(K, np.broadcast_to(np.asarray(P)[:, :, None, None], (B, T, G, H_kv)), "
                                "theta, inverse=True)",
                                "K = rope_rows(K, np.broadcast_to(np.asarray(P)[:, :, None, None], (B, T, G, H_kv)), "
                                "theta, inverse=False)"),
    "basis_layer_blocks_reversed": ("[U[l * H_kv * d:(l + 1) * H_kv * d].copy() for l in range(G)]",
                                    "[U[(G - 1 - l) * H_kv * d:(G - l) * H_kv * d].copy() for l in range(G)]"),
    "grad_silu_derivative": ("dZ = (dV @ W2) * (S + Z * S * (1.0 - S))", "dZ = (dV @ W2) * (S * (1.0 - S))"),
    "grad_factor_two_dropped": ("dV = 2.0 * E / (N * d)", "dV = E / (N * d)"),
    "grad_b2_from_hidden": ("g_b2 = dV.sum(axis=0)", "g_b2 = dV.sum(axis=0) + H.sum(axis=0)[:d] * 0.0 + dV.mean(axis=0)"),
    "adam_no_bias_correction": ("mh = m / (1.0 - beta1 ** step)", "mh = m"),
    "adam_second_moment_unsquared": ("v = beta2 * v + (1.0 - beta2) * g * g", "v = beta2 * v + (1.0 - beta2) * np.abs(g)"),
    "mass_interleaved_heads": ("s = (Q[b, :, hq] @ K[b, :, hq // g].T) * scale", "s = (Q[b, :, hq] @ K[b, :, hq % H_kv].T) * scale"),
    "mass_softmax_over_window": ("mass[b] += (p / p.sum(axis=1, keepdims=True)).sum(axis=0)",
                                 "mass[b] += (p / p.sum(axis=0, keepdims=True)).sum(axis=0)"),
    "evict_ties_to_higher_index": ("key=lambda t: (-M[b, t], t))", "key=lambda t: (-M[b, t], -t))"),
    "evict_recents_shifted": ("set(range(max(0, T - n_recent), T))", "set(range(max(0, T - n_recent - 1), T - 1))"),
}


def _run_py_mutant(name, find, repl, tmp, oracle_so):
    src = open(PY_SRC).read()
    assert src.count(find) == 1, f"mutation site of {name} not found once"
    pkg = os.path.join(tmp, name, "oracle")
    shutil.copytree(os.path.join(ROOT, "oracle"), pkg, ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    open(os.path.join(pkg, "oracle.py"), "w").write(src.replace(find, repl))
    env = dict(os.environ, LOWRAM_ORACLE_LIB=oracle_so, OMP_NUM_THREADS="1",
               PYTHONPATH=os.pathsep.join([os.path.dirname(pkg), ROOT]))
    # run from the copy's folder, so that `import oracle` finds the mutant before the real package
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")], cwd=os.path.dirname(pkg), env=env,
                       capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def test_every_planted_mistake_in_the_numpy_oracle_fails_a_pin():
    import oracle
    so = oracle.build()
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
            results = list(ex.map(lambda kv: _run_py_mutant(kv[0], *kv[1], tmp, so), PY_MUTANTS.items()))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, "mutants not caught by any pin: " + ", ".join(n for n, _ in survivors)
