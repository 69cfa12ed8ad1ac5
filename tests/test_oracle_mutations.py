"""Planted mistakes: every plausible slip in the oracle must fail at least one pin.

Each case copies the oracle's C source, applies one textual mutation (a dropped
term, an off-by-one mask, a wrong index, ...), compiles the copy on the CPU and
runs the pins of ``test_oracle.py`` against it. A mutant that passes every pin
would mean the pins could not tell that mistake from the definition.
"""
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTATIONS = {
    "mask_keeps_diagonal_out": ("for (int64_t j = i + 1; j < N; ++j)", "for (int64_t j = i; j < N; ++j)"),
    "mask_lets_next_key_in": ("for (int64_t j = i + 1; j < N; ++j)", "for (int64_t j = i + 2; j < N; ++j)"),
    "scale_dropped": ("s[j] = scale * acc;", "s[j] = acc;"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "lse_log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "no_normalisation": ("s[j] /= l;", "s[j] /= (l > 1.0 ? 1.0 : 1.0);"),
    "value_row_of_query": ("const uint16_t *vj = Vh + j * d;", "const uint16_t *vj = Vh + i * d;"),
    "key_row_of_query": ("const uint16_t *kj = Kh + j * d;", "const uint16_t *kj = Kh + i * d;"),
    "no_max_subtraction": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    "head_offset_dropped_for_kv": ("job->Q + head + i * job->d, job->K + head, job->V + head,",
                                   "job->Q + head + i * job->d, job->K, job->V,"),
    "bf16_decoded_as_low_half": ("uint32_t u = ((uint32_t)bits) << 16;", "uint32_t u = ((uint32_t)bits) << 15;"),
    "max_ignores_first_key": ("for (int64_t j = 0; j < N; ++j)\n        if (s[j] > m) m = s[j];",
                              "for (int64_t j = 1; j < N; ++j)\n        if (s[j] > m) m = s[j];"),
}


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_") or "oracle_mod" not in inspect.signature(fn).parameters:
            continue
        marks = getattr(fn, "pytestmark", [])
        grid = [{}]
        for m in marks:
            if m.name == "parametrize":
                names = [n.strip() for n in m.args[0].split(",")] if isinstance(m.args[0], str) else m.args[0]
                new = []
                for g in grid:
                    for val in m.args[1]:
                        vals = val if len(names) > 1 else (val,)
                        new.append({**g, **dict(zip(names, vals))})
                grid = new
        for kw in grid:
            out.append((name, fn, kw))
    return out


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, mutation):
    old, new = MUTATIONS[mutation]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new, 1))  # the first occurrence: the bf16 forward
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    str(mutant_c), "-o", str(lib), "-lm"], check=True)
    mutant = oracle.OracleBuild(str(lib))
    caught = []
    for name, fn, kw in _pin_functions():
        try:
            fn(mutant, **kw)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(name)
    assert caught, f"no pin caught mutation {mutation}"


BWD_MUTATIONS = {
    "bwd_drops_D": ("const double dSij = p[j] * (dPij - Di);", "const double dSij = p[j] * dPij;"),
    "bwd_dq_without_scale": ("dqi[c] += jb->scale * dSij * kj[c];", "dqi[c] += dSij * kj[c];"),
    "bwd_dk_uses_key": ("dkj[c] += jb->scale * dSij * qi[c];", "dkj[c] += jb->scale * dSij * kj[c];"),
    "bwd_dv_uses_dS": ("dvj[c] += p[j] * doi[c];", "dvj[c] += dSij * doi[c];"),
    "bwd_dP_uses_key": ("dPij += doi[c] * vj[c];", "dPij += doi[c] * kj[c];"),
    "bwd_D_uses_value": ("Di += doi[c] * o[c];", "Di += doi[c] * doi[c];"),
}


def _bwd_pins():
    import test_oracle_bwd as bp

    out = []
    for name, fn in inspect.getmembers(bp, inspect.isfunction):
        if not name.startswith("test_") or "oracle_mod" not in inspect.signature(fn).parameters:
            continue
        grid = [{}]
        for m in getattr(fn, "pytestmark", []):
            if m.name == "parametrize":
                names = [n.strip() for n in m.args[0].split(",")]
                grid = [{**g, **dict(zip(names, val if len(names) > 1 else (val,)))} for g in grid for val in m.args[1]]
        out += [(name, fn, kw) for kw in grid]
    return out


@pytest.mark.parametrize("mutation", sorted(BWD_MUTATIONS))
def test_backward_pins_catch_planted_mistake(tmp_path, mutation):
    old, new = BWD_MUTATIONS[mutation]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    str(mutant_c), "-o", str(lib), "-lm"], check=True)
    mutant = oracle.OracleBuild(str(lib))
    caught = []
    for name, fn, kw in _bwd_pins():
        try:
            fn(mutant, **kw)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(name)
    assert caught, f"no backward pin caught mutation {mutation}"


FP8_MUTATIONS = {
    "e4m3_bias_8": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_no_implicit_one": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp((double)m / 8.0, e - 7);"),
    "e4m3_subnormal_exponent": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    "e4m3_sign_dropped": ("return sign ? -v : v;", "return v;"),
    "e4m3_nan_not_decoded": ("if (e == 15 && m == 7)\n        return NAN;", "if (e == 16)\n        return NAN;"),
    "e4m3_scale_dropped": ("dst[i] = scale * e4m3_to_double(src[i]);", "dst[i] = e4m3_to_double(src[i]);"),
}


def _module_pins(modname):
    import importlib

    mod = importlib.import_module(modname)
    out = []
    for name, fn in inspect.getmembers(mod, inspect.isfunction):
        if not name.startswith("test_") or "oracle_mod" not in inspect.signature(fn).parameters:
            continue
        grid = [{}]
        for m in getattr(fn, "pytestmark", []):
            if m.name == "parametrize":
                names = [n.strip() for n in m.args[0].split(",")]
                grid = [{**g, **dict(zip(names, val if len(names) > 1 else (val,)))} for g in grid for val in m.args[1]]
        out += [(name, fn, kw) for kw in grid]
    return out


@pytest.mark.parametrize("mutation", sorted(FP8_MUTATIONS))
def test_fp8_pins_catch_planted_mistake(tmp_path, mutation):
    old, new = FP8_MUTATIONS[mutation]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    str(mutant_c), "-o", str(lib), "-lm"], check=True)
    mutant = oracle.OracleBuild(str(lib))
    caught = []
    for name, fn, kw in _module_pins("test_oracle_fp8"):
        try:
            fn(mutant, **kw)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(name)
    assert caught, f"no FP8 pin caught mutation {mutation}"


ROWWISE_MUTATIONS = {
    "softmax_no_max_subtraction": ("            y[j] = exp(x[j] - m);\n            l += y[j];",
                                   "            y[j] = exp(x[j]);\n            l += y[j];"),
    "softmax_not_normalised": ("        for (int64_t j = 0; j < N; ++j)\n            y[j] /= l;\n    }\n    return 0;\n}\n\n/* Layer",
                               "        for (int64_t j = 0; j < N; ++j)\n            y[j] /= 1.0;\n    }\n    return 0;\n}\n\n/* Layer"),
    "layernorm_unbiased_variance": ("        var /= (double)N;", "        var /= (double)(N > 1 ? N - 1 : 1);"),
    "layernorm_eps_outside_sqrt": ("const double rstd = 1.0 / sqrt(var + eps);", "const double rstd = 1.0 / (sqrt(var) + eps);"),
    "layernorm_gamma_beta_swapped": ("y[j] = (x[j] - mean) * rstd * gamma[j] + beta[j];",
                                     "y[j] = (x[j] - mean) * rstd * beta[j] + gamma[j];"),
    "layernorm_mean_not_removed": ("y[j] = (x[j] - mean) * rstd * gamma[j] + beta[j];", "y[j] = x[j] * rstd * gamma[j] + beta[j];"),
}


@pytest.mark.parametrize("mutation", sorted(ROWWISE_MUTATIONS))
def test_rowwise_pins_catch_planted_mistake(tmp_path, mutation):
    old, new = ROWWISE_MUTATIONS[mutation]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    str(mutant_c), "-o", str(lib), "-lm"], check=True)
    mutant = oracle.OracleBuild(str(lib))
    caught = []
    for name, fn, kw in _module_pins("test_oracle_rowwise"):
        try:
            fn(mutant, **kw)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(name)
    assert caught, f"no row-operation pin caught mutation {mutation}"
