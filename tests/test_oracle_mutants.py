"""Planted mistakes in the oracle, on the CPU.

Each mutant is a copy of the oracle's C sources with one plausible slip -- a
dropped term, a wrong sign, a swapped index or operand, an off-by-one bound --
compiled into its own library. The pin tests then run against that library in
a child process and must fail. The regression fixture is left out of those
runs: it was written by the oracle itself, so only the pins, which rest on
closed forms, brute force and library routines, count here. A mutant that
passed would mark a part of the oracle that nothing independent checks.
"""
import importlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

oracle_build = importlib.import_module("oracle.build")  # the module (the package re-exports its build())

PINS = ["test_oracle_pins.py", "test_oracle_spec_pins.py", "test_oracle_replay2_pins.py",
        "test_oracle_prefill_pins.py", "test_oracle_mamba2_pins.py"]

# (name, source file, text, replacement); the text occurs exactly once unless the name says "first"
MUTANTS = [
    # gating and normalisation
    ("softplus_without_log1p", "gdn_oracle.c", "x > 20.0 ? x : log1p(exp(x))", "x > 20.0 ? x : exp(x)"),
    ("sigmoid_sign", "gdn_oracle.c", "*beta = 1.0 / (1.0 + exp(-b));", "*beta = 1.0 / (1.0 + exp(b));"),
    ("decay_without_inner_exp", "gdn_oracle.c", "*alpha = exp(-exp(A_log) * softplus(a + dt_bias));",
     "*alpha = exp(-A_log * softplus(a + dt_bias));"),
    ("l2norm_eps_outside_sqrt", "gdn_oracle.c", "1.0 / sqrt(ss + 1e-6)", "1.0 / (sqrt(ss) + 1e-6)"),
    ("query_scale_dropped_first", "gdn_oracle.c", "orc_l2norm(dk, qr, 1.0 / sqrt((double)dk), qn);",
     "orc_l2norm(dk, qr, 1.0, qn);"),
    # the rule
    ("prediction_without_decay", "gdn_oracle.c", "beta * kn[i] * (v[j] - alpha * u);",
     "beta * kn[i] * (v[j] - u);"),
    ("correction_sign", "gdn_oracle.c", "beta * kn[i] * (v[j] - alpha * u);",
     "beta * kn[i] * (v[j] + alpha * u);"),
    ("state_not_decayed", "gdn_oracle.c", "col[i] = alpha * col[i] + beta", "col[i] = col[i] + beta"),
    ("readout_before_update_first", "gdn_oracle.c",
     "rule_step(dk, dv, Sd, kn, vv, alpha, beta);\n    readout(dk, dv, Sd, qn, out);",
     "readout(dk, dv, Sd, qn, out);\n    rule_step(dk, dv, Sd, kn, vv, alpha, beta);"),
    ("key_head_modulo", "gdn_oracle.c",
     "int bi = (int)(u / Hv), h = (int)(u % Hv), kh = h / group;\n        double* o = out + u * dv;",
     "int bi = (int)(u / Hv), h = (int)(u % Hv), kh = h % Hk;\n        double* o = out + u * dv;"),
    ("key_gets_query_scale_first", "gdn_oracle.c", "orc_l2norm(dk, kr, 1.0, kn);",
     "orc_l2norm(dk, kr, 1.0 / sqrt((double)dk), kn);"),
    ("bad_count_of_padding_first", "gdn_oracle.c", "if (slot >= num_slots) bad += 1;", "if (slot < 0) bad += 1;"),
    # storage formats
    ("bf16_load_shift", "gdn_oracle.c", "uint32_t u = ((uint32_t)h) << 16;", "uint32_t u = ((uint32_t)h) << 15;"),
    ("f16_subnormal_scale", "gdn_oracle.c", "v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    ("rounding_truncates", "gdn_oracle.c", "nearbyint(ax / quantum)", "trunc(ax / quantum)"),
    ("no_gradual_underflow", "gdn_oracle.c", "if (e < emin) e = emin;", "if (e < emin) return copysign(0.0, x);"),
    # ReplaySSM
    ("fold_one_entry_early", "gdn_oracle.c",
     "if (meta[0] + T > L) fold(dk, dv, S0, sdt, ek, ev, idt, ealpha, ebeta, meta);",
     "if (meta[0] + T >= L) fold(dk, dv, S0, sdt, ek, ev, idt, ealpha, ebeta, meta);"),
    ("window_output_one_token_behind", "gdn_oracle.c", "rebuild(dk, dv, S0, sdt, c + t + 1,",
     "rebuild(dk, dv, S0, sdt, c + t,"),
    ("rollback_drops_one_more", "gdn_oracle.c", "int r = T - 1 - accepted;", "int r = T - accepted;"),
    ("fold_runs_from_the_read_copy", "gdn_oracle.c", "rebuild(dk, dv, M, mdt, meta[0],",
     "rebuild(dk, dv, Rd, rdt, meta[0],"),
    # speculative step and prefill
    ("spec_copies_negated", "gdn_oracle.c",
     "if (write[t])\n            for (int64_t i = 0; i < n; ++i) orc_store(S_out,",
     "if (!write[t])\n            for (int64_t i = 0; i < n; ++i) orc_store(S_out,"),
    ("prefill_write_back_off_by_one", "gdn_oracle.c", "if ((t + 1) % interval == 0 || t == T - 1)",
     "if (t % interval == 0 || t == T - 1)"),
    ("prefill_continues_unrounded", "gdn_oracle.c",
     "for (int64_t i = 0; i < n; ++i) orc_store(S, i, sdt, Sd[i]);\n            load_vec(S, 0, (int)n, sdt, Sd);",
     "for (int64_t i = 0; i < n; ++i) orc_store(S, i, sdt, Sd[i]);"),
    ("flush_ignores_force", "gdn_oracle.c",
     "if (force ? meta[0] > 0 : meta[0] == L) fold(dk, dv, S0, sdt,", "if (meta[0] == L) fold(dk, dv, S0, sdt,"),
    ("rollback_past_checkpoint", "gdn_oracle.c", "if (meta[0] - r < 0) return -2;\n", ""),
    ("gates_swapped_first", "gdn_oracle.c", "orc_load(a, u, idt), orc_load(b, u, idt)",
     "orc_load(b, u, idt), orc_load(a, u, idt)"),
    ("prefill_value_row_of_key_head", "gdn_oracle.c", "elem_ptr(v, (tok * Hv + h) * dv, idt)",
     "elem_ptr(v, (tok * Hv + kh) * dv, idt)"),
    ("prefill_gates_of_local_token", "gdn_oracle.c",
     "orc_load(a, tok * Hv + h, idt), orc_load(b, tok * Hv + h, idt)",
     "orc_load(a, t * Hv + h, idt), orc_load(b, t * Hv + h, idt)"),
    ("prefill_outputs_at_sequence_local_rows", "gdn_oracle.c",
     "for (int j = 0; j < dv; ++j) out[((int64_t)(t0 + t) * Hv + h) * dv + j] = o[(int64_t)t * dv + j];",
     "for (int j = 0; j < dv; ++j) out[((int64_t)t * Hv + h) * dv + j] = o[(int64_t)t * dv + j];"),
    ("spec_copies_to_first_destination", "gdn_oracle.c",
     "memcpy((char*)pool + ((int64_t)dst_slots[(int64_t)bi * T + t] * Hv + h) * n * esz,",
     "memcpy((char*)pool + ((int64_t)dst_slots[(int64_t)bi * T] * Hv + h) * n * esz,"),
    ("read_copy_rounds_unrounded_master", "gdn_oracle.c", "orc_store(Rd, i, rdt, m);", "orc_store(Rd, i, rdt, Sm[i]);"),
    ("fold2_master_not_stored", "gdn_oracle.c", "orc_store(M, i, mdt, m);", ""),
    ("spec_continues_from_rounded_copy", "gdn_oracle.c",
     "for (int64_t i = 0; i < n; ++i) orc_store(S_out, (int64_t)t * n + i, sdt, Sd[i]);",
     "for (int64_t i = 0; i < n; ++i) orc_store(S_out, (int64_t)t * n + i, sdt, Sd[i]);\n"
     "        if (write[t]) load_vec(S_out, (int64_t)t * n, (int)n, sdt, Sd);"),
    ("decode_reads_out_the_rounded_state", "gdn_oracle.c",
     "    readout(dk, dv, Sd, qn, out);\n    for (int64_t i = 0; i < n; ++i) orc_store(S, i, sdt, Sd[i]);",
     "    for (int64_t i = 0; i < n; ++i) orc_store(S, i, sdt, Sd[i]);\n"
     "    load_vec(S, 0, (int)n, sdt, Sd);\n    readout(dk, dv, Sd, qn, out);"),
    ("prefill_final_state_not_stored", "gdn_oracle.c", "if ((t + 1) % interval == 0 || t == T - 1)",
     "if ((t + 1) % interval == 0)"),
    ("window_gates_in_one_entry", "gdn_oracle.c",
     "orc_gating(A_log, dt_bias, a[t], b[t], &ealpha[c + t], &ebeta[c + t]);",
     "orc_gating(A_log, dt_bias, a[t], b[t], &ealpha[c], &ebeta[c]);"),
    ("dt_bias_outside_softplus", "gdn_oracle.c", "*alpha = exp(-exp(A_log) * softplus(a + dt_bias));",
     "*alpha = exp(-exp(A_log) * (softplus(a) + dt_bias));"),
    ("softplus_cut_over_at_2", "gdn_oracle.c", "x > 20.0 ? x : log1p(exp(x))", "x > 2.0 ? x : log1p(exp(x))"),
    ("l1_norm_for_l2", "gdn_oracle.c", "ss += x[i] * x[i];", "ss += fabs(x[i]);"),
    ("no_overflow_to_inf", "gdn_oracle.c", "if (r > maxfin) r = INFINITY;", ""),
    ("decode_state_at_key_head_stride_first", "gdn_oracle.c",
     "void* S = (char*)pool + ((int64_t)slot * Hv + h) * (int64_t)dv * dk * orc_dtype_size(sdt);",
     "void* S = (char*)pool + ((int64_t)slot * Hk + h) * (int64_t)dv * dk * orc_dtype_size(sdt);"),
    ("replay_query_unscaled", "gdn_oracle.c", "orc_l2norm(dk, qv, 1.0 / sqrt((double)dk), qv + dk);",
     "orc_l2norm(dk, qv, 1.0, qv + dk);"),
    ("replay_keys_unnormalised", "gdn_oracle.c", "rule_step(dk, dv, S, kn, vv, ea[e], eb[e]);",
     "rule_step(dk, dv, S, kr, vv, ea[e], eb[e]);"),
    # Mamba2
    ("m2_softplus_cut_over_at_2", "mamba2_oracle.c", "x > 20.0 ? x : log1p(exp(x))", "x > 2.0 ? x : log1p(exp(x))"),
    ("m2_dt_bias_dropped", "mamba2_oracle.c", "*delta = softplus_m2(dt + dt_bias);", "*delta = softplus_m2(dt);"),
    ("m2_flush_ignores_force", "mamba2_oracle.c", "if (meta[0] == L || (force && meta[0] > 0)) m2_fold(",
     "if (meta[0] == L) m2_fold("),
    ("m2_skip_term_dropped", "mamba2_oracle.c", "y[p] = acc + D * x[p];", "y[p] = acc;"),
    ("m2_step_size_dropped", "mamba2_oracle.c", "+ delta * x[p] * Bv[i];", "+ x[p] * Bv[i];"),
    ("m2_group_modulo", "mamba2_oracle.c", "g = h / per_group;", "g = h % G;"),
    ("m2_update_reads_C", "mamba2_oracle.c", "m2_update(N, P, Sd, bv, xv, alpha, delta);",
     "m2_update(N, P, Sd, cv, xv, alpha, delta);"),
    ("m2_readout_before_update", "mamba2_oracle.c",
     "m2_update(N, P, Sd, bv, xv, alpha, delta);\n    m2_readout(N, P, Sd, cv, xv, D, out);",
     "m2_readout(N, P, Sd, cv, xv, D, out);\n    m2_update(N, P, Sd, bv, xv, alpha, delta);"),
    ("m2_decay_without_inner_exp", "mamba2_oracle.c", "*alpha = exp(-exp(A_log) * *delta);",
     "*alpha = exp(-A_log * *delta);"),
    ("m2_window_output_one_token_behind", "mamba2_oracle.c", "m2_rebuild(N, P, S0, sdt, c + t + 1,",
     "m2_rebuild(N, P, S0, sdt, c + t,"),
]


def _mutate(tmp, name, src, text, repl) -> str:
    """Copy the oracle sources into tmp, plant the slip (none when src is None), build the copy."""
    for f in oracle_build.SOURCES + oracle_build.HEADERS:
        shutil.copy(os.path.join(oracle_build.HERE, f), tmp)
    if src is not None:
        path = os.path.join(tmp, src)
        with open(path) as fh:
            code = fh.read()
        count = code.count(text)
        assert count == 1 or (name.endswith("_first") and count > 1), f"{name}: text found {count} times"
        with open(path, "w") as fh:
            fh.write(code.replace(text, repl, 1))
    return oracle_build.build(force=True, src_dir=tmp, out=os.path.join(tmp, "lib", "liboracle.so"))


def _run_pins(lib):
    env = dict(os.environ, ORACLE_LIBRARY=lib)
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-k",
                           "not regression_fixture", *[os.path.join(ROOT, "tests", p) for p in PINS]],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_unaltered_copy_passes_the_pins(tmp_path):
    """The control: the same harness on an unaltered copy passes, so a failing mutant run means the slip."""
    run = _run_pins(_mutate(str(tmp_path), "control", None, None, None))
    assert run.returncode == 0, run.stdout[-3000:]


def test_pins_catch_every_planted_mistake(tmp_path):
    """Every mutant, built and checked in parallel (each in its own directory and child process)."""

    def check(i):
        name, src, text, repl = MUTANTS[i]
        d = tmp_path / f"m{i}"
        d.mkdir()
        run = _run_pins(_mutate(str(d), name, src, text, repl))
        return name, run.returncode, run.stdout[-1500:]

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(check, range(len(MUTANTS))))
    survivors = [(name, code, out) for name, code, out in results if code != 1]
    assert not survivors, "mutants the pins did not catch:\n" + "\n".join(
        f"{name} (exit {code})\n{out}" for name, code, out in survivors)
