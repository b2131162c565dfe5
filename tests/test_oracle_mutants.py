"""The oracle's pins catch plausible mistakes: each mistake below is planted,
one at a time, in a copy of the oracle's C source (built into its own
directory), and the pins of that part of the oracle are run against it in a
separate process. The unmodified copy must pass every pin; every mutant must
fail at least one. CPU only; nothing here touches the CUDA path.

The mistakes are the kind a transcription of the recurrences could make: a
term dropped, an operand transposed, a gate or state taken at the wrong step,
a branch run the wrong way.
"""

import json
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORK = os.path.join(ROOT, "tests", "_mutants")

# (family, mutant name, original text, replacement); every original occurs
# exactly once in oracle.c
MUTANTS = [
    # scalar form
    ("scalar", "fwd_drops_h0",
     "      double state = h0 ? h0[h0_index(cu, s, r, C)] : 0.0;\n      if (!reverse) {",
     "      double state = 0.0;\n      if (!reverse) {"),
    ("scalar", "fwd_reverse_runs_forwards",
     "        for (int64_t t = end - 1; t >= beg; --t) {\n          state = ar[t] * state + xr[t];\n"
     "          hr[t] = state;",
     "        for (int64_t t = beg; t < end; ++t) {\n          state = ar[t] * state + xr[t];\n"
     "          hr[t] = state;"),
    ("scalar", "bwd_gate_not_shifted",
     "const double shifted_gate = (t + 1 < end) ? ar[t + 1] : 0.0;",
     "const double shifted_gate = ar[t];"),
    ("scalar", "bwd_state_not_shifted",
     "const double shifted_state = (t > beg) ? hs[t - 1] : init;",
     "const double shifted_state = hs[t];"),
    ("scalar", "bwd_no_h0_at_sequence_start",
     "const double shifted_state = (t > beg) ? hs[t - 1] : init;",
     "const double shifted_state = (t > beg) ? hs[t - 1] : 0.0;"),
    ("scalar", "bwd_dh0_without_gate",
     "if (end > beg) d_init = ar[beg] * dxr[beg];",
     "if (end > beg) d_init = dxr[beg];"),
    ("scalar", "bwd_reverse_gate_wrong_side",
     "const double shifted_gate = (t - 1 >= beg) ? ar[t - 1] : 0.0;",
     "const double shifted_gate = (t + 1 < end) ? ar[t + 1] : 0.0;"),
    ("scalar", "bwd_reverse_state_wrong_side",
     "const double shifted_state = (t + 1 < end) ? hs[t + 1] : init;",
     "const double shifted_state = (t > beg) ? hs[t - 1] : init;"),
    ("scalar", "bwd_reverse_dh0_wrong_end",
     "if (end > beg) d_init = ar[end - 1] * dxr[end - 1];",
     "if (end > beg) d_init = ar[beg] * dxr[beg];"),
    # log space
    ("log", "fwd_drops_gate",
     "          l = log_add_exp(l + la[t], lx[t]);\n          hr[t] = exp(l);\n        }\n      } else {",
     "          l = log_add_exp(l, lx[t]);\n          hr[t] = exp(l);\n        }\n      } else {"),
    ("log", "fwd_swaps_a_and_x",
     "          l = log_add_exp(l + la[t], lx[t]);\n          hr[t] = exp(l);\n        }\n      } else {",
     "          l = log_add_exp(l + lx[t], la[t]);\n          hr[t] = exp(l);\n        }\n      } else {"),
    ("log", "fwd_reverse_runs_forwards",
     "      if (!reverse) {\n        for (int64_t t = beg; t < end; ++t) {\n          l = log_add_exp",
     "      if (1) {\n        for (int64_t t = beg; t < end; ++t) {\n          l = log_add_exp"),
    ("log", "fwd_drops_h0",
     "double l = log_h0 ? log_h0[h0_index(cu, s, r, C)] : -INFINITY;",
     "double l = -INFINITY;"),
    ("log", "bwd_dlog_a_scaled_by_x", "    dlog_a[i] *= a[i];", "    dlog_a[i] *= x[i];"),
    ("log", "bwd_dlog_x_unscaled", "    dlog_x[i] *= x[i];", "    dlog_x[i] *= 1.0;"),
    ("log", "bwd_dlog_h0_unscaled", "dlog_h0[i] = h0 ? dh0[i] * h0[i] : 0.0;",
     "dlog_h0[i] = h0 ? dh0[i] : 0.0;"),
    # block form
    ("affine", "fwd_A_transposed", "acc += At[i * k + l] * state[l * v + j];",
     "acc += At[l * k + i] * state[l * v + j];"),
    ("affine", "fwd_drops_h0", "        state[e] = h0 ? h0[(b * N + n) * kv + e] : 0.0;",
     "        state[e] = 0.0;"),
    ("affine", "fwd_drops_B", "next[i * v + j] = acc + Bt[i * v + j];", "next[i * v + j] = acc;"),
    ("affine", "bwd_A_t_instead_of_A_t1", "const double* An = A + ((b * T + t + 1) * N + n) * kk;",
     "const double* An = A + ((b * T + t) * N + n) * kk;"),
    ("affine", "bwd_A_not_transposed", "acc += An[l * k + i] * g[l * v + j];",
     "acc += An[i * k + l] * g[l * v + j];"),
    ("affine", "bwd_dA_uses_H_t",
     "        const double* prev = t > 0 ? hs + (t - 1) * kv : init;\n        double* dAt",
     "        const double* prev = hs + t * kv;\n        double* dAt"),
    ("affine", "bwd_dA_transposed", "dAt[i * k + l] = acc;", "dAt[l * k + i] = acc;"),
    ("affine", "bwd_dh0_A_not_transposed", "acc += A0[l * k + i] * g[l * v + j];",
     "acc += A0[i * k + l] * g[l * v + j];"),
    ("affine", "bwd_states_A_transposed", "acc += At[i * k + l] * prev[l * v + j];",
     "acc += At[l * k + i] * prev[l * v + j];"),
    # scalar-gated outer-product state
    ("gdn", "fwd_drops_h0",
     "for (int64_t i = 0; i < S * D; ++i) h[i] = h0 ? h0[bh * S * D + i] : 0.0;",
     "for (int64_t i = 0; i < S * D; ++i) h[i] = 0.0;"),
    ("gdn", "fwd_gate_of_previous_step", "const double al = alpha[st];",
     "const double al = alpha[st > bh * T ? st - 1 : st];"),
    ("gdn", "fwd_read_sign", "for (int64_t s = 0; s < S; ++s) acc += c[st * S + s] * h[s * D + d];",
     "for (int64_t s = 0; s < S; ++s) acc -= c[st * S + s] * h[s * D + d];"),
    ("gdn", "fwd_drops_decay",
     "h[s * D + d] = al * h[s * D + d] + b[st * S + s] * v[st * D + d];",
     "h[s * D + d] = h[s * D + d] + b[st * S + s] * v[st * D + d];"),
    ("gdn", "bwd_gate_at_t_not_t1", "const double an = (t + 1 < T) ? alpha[st + 1] : 0.0;",
     "const double an = alpha[st];"),
    ("gdn", "bwd_dalpha_uses_h_t", "for (int64_t i = 0; i < SD; ++i) acc_a += dh[i] * hp[i];",
     "for (int64_t i = 0; i < SD; ++i) acc_a += dh[i] * ht[i];"),
    ("gdn", "bwd_dh0_without_gate", "dh0[bh * SD + i] = (T > 0 ? alpha[bh * T] : 0.0) * dh[i];",
     "dh0[bh * SD + i] = dh[i];"),
    ("gdn", "bwd_dc_uses_h_prev", "acc_c += ht[s * D + d] * dout[st * D + d];",
     "acc_c += hp[s * D + d] * dout[st * D + d];"),
    ("gdn", "bwd_db_uses_dout", "acc_b += dh[s * D + d] * v[st * D + d];",
     "acc_b += dh[s * D + d] * dout[st * D + d];"),
    ("gdn", "bwd_dv_uses_c", "for (int64_t s = 0; s < S; ++s) acc += b[st * S + s] * dh[s * D + d];",
     "for (int64_t s = 0; s < S; ++s) acc += c[st * S + s] * dh[s * D + d];"),
    ("gdn", "bwd_read_injected_only_at_last_step",
     "dh[s * D + d] = c[st * S + s] * dout[st * D + d] + an * dh[s * D + d];",
     "dh[s * D + d] = an * dh[s * D + d] + (t == T - 1 ? c[st * S + s] * dout[st * D + d] : 0.0);"),
    # RG-LRU gate preparation
    ("rglru", "scale_4", "#define RG_SCALE 8.0", "#define RG_SCALE 4.0"),
    ("rglru", "fwd_log_sigmoid_sign",
     "const double ls = rg_log_sigmoid(a_param[c]);\n      double state",
     "const double ls = rg_log_sigmoid(-a_param[c]);\n      double state"),
    ("rglru", "fwd_no_multiplier",
     "write = sqrt(-expm1(2.0 * log_a)) * in_gate * x[e];\n        }\n        state = a * state + write;",
     "write = in_gate * x[e];\n        }\n        state = a * state + write;"),
    ("rglru", "fwd_reset_keeps_gate", "a = 0.0;\n          write = in_gate * x[e];",
     "a = exp(RG_SCALE * rg_sigmoid(gate_a[e]) * ls);\n          write = in_gate * x[e];"),
    ("rglru", "fwd_reset_keeps_multiplier", "write = in_gate * x[e];\n        } else {",
     "write = sqrt(-expm1(2.0 * RG_SCALE * rg_sigmoid(gate_a[e]) * ls)) * in_gate * x[e];\n"
     "        } else {"),
    ("rglru", "fwd_segment_pos_ignores_batch",
     "if (segment_pos && segment_pos[b * T + t] == 0) {\n          a = 0.0;\n          write",
     "if (segment_pos && segment_pos[t] == 0) {\n          a = 0.0;\n          write"),
    ("rglru", "bwd_adjoint_drops_gate", "g = dh[e] + a_next * g; /* dL/dh_t */",
     "g = dh[e] + g; /* dL/dh_t */"),
    ("rglru", "bwd_da_uses_h_t", "const double d_a = g * hs[t] + ",
     "const double d_a = g * hs[t + 1] + "),
    ("rglru", "bwd_drops_multiplier_term", "d_mult * dmult_du * (-2.0 * a)",
     "0.0 * dmult_du * (-2.0 * a)"),
    ("rglru", "bwd_da_param_without_sigmoid", "da_param[c] = d_ls * rg_sigmoid(-a_param[c]);",
     "da_param[c] = d_ls;"),
    ("rglru", "bwd_dh0_without_gate", "dh0[b * C + c] = (T > 0 ? a_next : 0.0) * g;",
     "dh0[b * C + c] = g;"),
    ("rglru", "bwd_dgate_x_without_sigmoid_derivative",
     "dgate_x[e] = d_in * in_gate * (1.0 - in_gate);", "dgate_x[e] = d_in;"),
    ("rglru", "bwd_dgate_a_without_sigmoid_derivative",
     "dgate_a[e] = d_log_a * RG_SCALE * ls * r * (1.0 - r);",
     "dgate_a[e] = d_log_a * RG_SCALE * ls * r;"),
]

PINS = {
    "scalar": ["test_fwd_matches_exact_closed_form",
               "test_fwd_reverse_matches_closed_form_on_flipped_input",
               "test_constant_gate_geometric_series", "test_reset_erases_prefix_exactly",
               "test_packed_sequences_do_not_leak", "test_stream_continuation",
               "test_bwd_central_differences", "test_bwd_dx_matches_exact_closed_form",
               "test_bwd_adjoint_identity", "test_bwd_packed_central_differences_and_boundaries"],
    "log": ["test_log_matches_linear_scan", "test_log_matches_logcumsumexp_closed_form",
            "test_log_reset_and_packed", "test_log_bwd_central_differences"],
    "affine": ["test_affine_k1_is_scalar_scan", "test_affine_diagonal_is_independent_scalar_scans",
               "test_affine_identity_is_cumsum", "test_affine_explicit_products_and_order",
               "test_affine_bwd_central_differences",
               "test_affine_coefficient_prefix_is_the_product_of_gates"],
    "gdn": ["test_gdn_forward_exact_closed_form",
            "test_gdn_with_one_by_one_state_is_the_scalar_scan",
            "test_gdn_backward_central_differences"],
    "rglru": ["test_rglru_transition_and_multiplier", "test_rglru_frozen_and_open_gates",
              "test_rglru_is_the_scan_of_its_step_maps", "test_rglru_reset_erases_the_prefix",
              "test_rglru_backward_central_differences"],
}

# Runs the named pins against the oracle copy in argv[1] and prints, as JSON,
# "pass" or why each failed. Parametrised pins run over all their cases.
RUNNER = r'''
import importlib.util, json, sys
sys.path.insert(0, sys.argv[1])
import oracle
assert oracle.__file__.startswith(sys.argv[1]), oracle.__file__
oracle.build()
spec = importlib.util.spec_from_file_location("pins", sys.argv[2])
pins = importlib.util.module_from_spec(spec)
spec.loader.exec_module(pins)
res = {}
for name in sys.argv[3:]:
    fn = getattr(pins, name)
    calls = [{}]
    for m in getattr(fn, "pytestmark", []):
        if m.name != "parametrize":
            continue
        names = [s.strip() for s in m.args[0].split(",")]
        calls = [dict(c, **dict(zip(names, v if len(names) > 1 else (v,))))
                 for c in calls for v in m.args[1]]
    try:
        for kw in calls:
            fn(**kw)
        res[name] = "pass"
    except AssertionError:
        res[name] = "fail"
    except Exception as e:
        res[name] = "error " + type(e).__name__
print(json.dumps(res))
'''


def _run(tag, src):
    d = os.path.join(WORK, tag)
    shutil.rmtree(d, ignore_errors=True)
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(d, "oracle"),
                    ignore=shutil.ignore_patterns("*.so", "*.so.tmp*", "__pycache__"))
    with open(os.path.join(d, "oracle", "oracle.c"), "w") as f:
        f.write(src)
    family = tag.split(".")[0]
    r = subprocess.run([sys.executable, "-c", RUNNER, d,
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")] + PINS[family],
                       capture_output=True, text=True, cwd=d, timeout=600)
    assert r.returncode == 0, (tag, r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_every_planted_mistake_fails_a_pin():
    with open(os.path.join(ROOT, "oracle", "oracle.c")) as f:
        src = f.read()
    jobs = [(f"{fam}.unmodified", src) for fam in PINS]
    for fam, name, old, new in MUTANTS:
        assert src.count(old) == 1, (fam, name, src.count(old))
        jobs.append((f"{fam}.{name}", src.replace(old, new)))
    os.makedirs(WORK, exist_ok=True)
    try:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            results = dict(zip((t for t, _ in jobs), ex.map(lambda j: _run(*j), jobs)))
    finally:
        shutil.rmtree(WORK, ignore_errors=True)
    for tag, res in results.items():
        if tag.endswith(".unmodified"):
            assert all(v == "pass" for v in res.values()), (tag, res)
        else:
            assert any(v == "fail" for v in res.values()), (tag, res)
            assert not any(v.startswith("error") for v in res.values()), (tag, res)
