"""Mutation check of the oracle's pins (CPU only).

Each case below plants one plausible mistake in a copy of the oracle's C
source -- a wrong head map, a dropped scale, an off-by-one window, a
transposed operand, a wrong LSE slot, a missed clamp -- compiles it into a
temporary directory and runs every pin against it in a child process (a
mutant may read out of bounds, so it must not share the test's process).
The real oracle passes every pin; each mutant must fail at least one.
"""
import concurrent.futures
import json
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "attn_oracle.c")

# (name, text to replace, replacement, replace every occurrence?)
MUTANTS = [
    ("gqa_modulo", "const int g = h / gs;", "const int g = h % G;", True),
    ("gqa_wrong_divisor", "const int g = h / gs;", "const int g = (h / G) % G;", True),
    ("scale_dropped", "s[t] = dot * scale;", "s[t] = dot;", False),
    ("scale_without_sqrt", "1.0 / sqrt((double)D)", "1.0 / (double)D", True),
    ("causal_window_short", "(size_t)pos + 1 : (size_t)kv_seq", "(size_t)pos : (size_t)kv_seq", False),
    ("causal_treated_as_full", "(mask == 0) ?", "(mask == 1) ?", False),
    ("lse_slot1_is_total", "*logl_out = log(l);", "*logl_out = m + log(l);", False),
    ("max_not_subtracted", "s[t] = exp(s[t] - m);", "s[t] = exp(s[t]);", False),
    ("max_sign_flipped", "s[t] = exp(s[t] - m);", "s[t] = exp(s[t] + m);", False),
    ("k_transposed", "(double)q[d] * (double)kt[d]", "(double)q[d] * (double)k[d * kv_stride + t]", False),
    ("v_read_from_k", "(double)v[t * kv_stride + d]", "(double)k[t * kv_stride + d]", False),
    ("not_normalised", "out[d] = acc / l;", "out[d] = acc;", False),
    ("empty_lse_zero", "#define ORACLE_EMPTY_LSE (-1e30)", "#define ORACLE_EMPTY_LSE (0.0)", False),
    ("empty_out_ones", "out[d] = 0.0;", "out[d] = 1.0;", False),
    ("prefill_drops_q_base", "size_t n = (size_t)start_pos + q_global + 1;",
     "size_t n = (size_t)start_pos + (size_t)i + 1;", False),
    ("prefill_no_clamp", "if (n > (size_t)max_seq) n = (size_t)max_seq;\n                    const int g",
     "const int g", False),
    ("window_one_short", "return (window > 0 && n > (size_t)window) ? n - (size_t)window : 0;",
     "return (window > 0 && n > (size_t)window) ? n - (size_t)window + 1 : 0;", False),
    ("window_ignored", "return (window > 0 && n > (size_t)window) ? n - (size_t)window : 0;", "return 0;", False),
    ("window_from_start", "attend_row(q + qo, k + lo * kv_dim + (size_t)g * D, v + lo * kv_dim + (size_t)g * D, kv_dim,\n                               n - lo,",
     "attend_row(q + qo, k + (size_t)g * D, v + (size_t)g * D, kv_dim,\n                               n - lo,", False),
    ("decode_no_clamp", "if (n > (size_t)max_seq) n = (size_t)max_seq;\n    double *s", "double *s", False),
    ("decode_window_short", "size_t n = (size_t)kv_pos + 1;", "size_t n = (size_t)kv_pos;", False),
    ("prefill_out_uses_q_stride", "out_batch + q_global * out_stride", "out_batch + q_global * q_stride", False),
    ("prefill_scale_ignored", "const double sc = (double)scale;", "const double sc = 1.0 / sqrt((double)D);", False),
    ("forward_kv_head_offset_dropped", "attend_row(q + qo, k + lo * kv_dim + (size_t)g * D, v + lo * kv_dim + (size_t)g * D,",
     "attend_row(q + qo, k + lo * kv_dim, v + lo * kv_dim,", False),
    ("query_head_is_kv_head", "(size_t)pos * H * D + (size_t)h * D;", "(size_t)pos * H * D + (size_t)(h / gs) * D;", False),
    ("first_key_skipped", "for (size_t t = 0; t < n; ++t) {\n        const float *kt",
     "for (size_t t = 1; t < n; ++t) {\n        const float *kt", False),
    ("dot_in_fp32", "double dot = 0.0;", "float dot = 0.0f;", False),
    ("sum_in_fp32", "double l = 0.0;", "float l = 0.0f;", False),
    # backward
    ("bwd_mean_dropped", "const double ds = p[t] * (dp[t] - mean);", "const double ds = p[t] * dp[t];", False),
    ("bwd_dk_unscaled", "dkt[d] += scale * ds * (double)qr[d];", "dkt[d] += ds * (double)qr[d];", False),
    ("bwd_dq_reads_v", "dqr[d] += scale * ds * (double)kt[d];",
     "dqr[d] += scale * ds * (double)v[t * kv_dim + (size_t)g * D + d];", False),
    ("bwd_dv_unweighted", "dvt[d] += p[t] * (double)dor[d];", "dvt[d] += (double)dor[d];", False),
    ("bwd_p_not_normalised", "for (size_t t = lo; t < n; ++t) p[t] /= l;", "", False),
    ("bwd_dp_reads_k", "(double)dor[d] * (double)vt[d]", "(double)dor[d] * (double)k[t * kv_dim + (size_t)g * D + d]",
     False),
    ("bwd_window_ignored", "const size_t lo = window_start(n, window);\n                        if (n == lo)",
     "const size_t lo = 0;\n                        if (n == lo)", False),
    ("bwd_causal_short", "const size_t n = (mask == 0) ? (size_t)pos + 1", "const size_t n = (mask == 0) ? (size_t)pos",
     False),
    # RoPE forward
    ("rope_sign_flipped", "y[d] = (double)x[d] * c - (double)x[d + half] * s;",
     "y[d] = (double)x[d] * c + (double)x[d + half] * s;", False),
    ("rope_pairs_interleaved", "y[d + half] = (double)x[d + half] * c + (double)x[d] * s;",
     "y[d + half] = (double)x[d + half] * c + (double)x[d] * s; if (D > 2 && d < half) { y[d] = (double)x[d] * c - (double)x[d ^ 1] * s; }",
     False),
    ("rope_exponent_halved", "pow(base, -2.0 * (double)d / (double)D)", "pow(base, -1.0 * (double)d / (double)D)", False),
    ("rope_key_position_shifted", "D, t,\n                                               rope_base);",
     "D, t + 1,\n                                               rope_base);", False),
    ("rope_query_unrotated", "rope_rotate(q + qo, qr, D, (size_t)pos, rope_base);",
     "rope_rotate(q + qo, qr, D, 0, rope_base);", False),
    ("rope_bwd_not_turned_back", "x[d] = x0 * c + x1 * s;", "x[d] = x0 * c - x1 * s;", False),
    ("bwd_head_map_interleaved", "const int h = g * gs + hh;", "const int h = hh * G + g;", False),
]

RUNNER = r"""
import json, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle, pins
orc = oracle.Oracle({lib!r})
failed = []
for pin in pins.ALL_PINS:
    try:
        pin(orc)
    except Exception as e:
        failed.append(pin.__name__)
print(json.dumps(failed))
"""


def _run_mutant(name, old, new, every, tmp):
    src = open(SRC).read()
    assert old in src, "mutation site not found: " + name
    mutated = src.replace(old, new) if every else src.replace(old, new, 1)
    cfile = os.path.join(tmp, name + ".c")
    lib = os.path.join(tmp, "lib" + name + ".so")
    with open(cfile, "w") as f:
        f.write(mutated)
    r = subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", cfile, "-o", lib, "-lm"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if p.returncode != 0:
        return ["<crashed: %d>" % p.returncode]
    return json.loads(p.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def mutant_results():
    with tempfile.TemporaryDirectory() as tmp:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            futs = {m[0]: ex.submit(_run_mutant, *m, tmp) for m in MUTANTS}
            return {k: f.result() for k, f in futs.items()}


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_is_caught(mutant_results, name):
    assert mutant_results[name], "no pin caught the planted mistake " + name


# The paged oracle is a numpy gather (oracle/__init__.py), outside the C file:
# its plausible mistakes are planted by swapping the gather for a wrong one.
def _gather_identity(pool, table, page_rows):          # table ignored
    n = len(table) * page_rows
    return np.ascontiguousarray(np.asarray(pool, np.float32)[:n])


def _gather_inverse(pool, table, page_rows):           # table read backwards (pool page -> logical page)
    pool = np.asarray(pool, np.float32)
    pages = pool.reshape(-1, page_rows, pool.shape[1])
    inv = np.argsort(np.asarray(table, np.int64))
    inv = inv[inv < pages.shape[0]][:len(table)]
    return np.ascontiguousarray(pages[inv].reshape(-1, pool.shape[1]))


def _gather_rows_transposed(pool, table, page_rows):   # rows within a page reversed
    pool = np.asarray(pool, np.float32)
    pages = pool.reshape(-1, page_rows, pool.shape[1])
    return np.ascontiguousarray(pages[np.asarray(table, np.int64)][:, ::-1].reshape(-1, pool.shape[1]))


@pytest.mark.parametrize("wrong", [_gather_identity, _gather_inverse, _gather_rows_transposed])
def test_paged_gather_mistake_is_caught(wrong, monkeypatch):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    import pins
    orc = oracle.default()
    monkeypatch.setattr(oracle.Oracle, "gather_pages", staticmethod(wrong))
    failed = 0
    for pin in (pins.pin_paged_decode_equals_contiguous, pins.pin_paged_prefill_equals_contiguous,
                pins.pin_paged_shared_page):
        try:
            pin(orc)
        except Exception:
            failed += 1
    assert failed > 0
