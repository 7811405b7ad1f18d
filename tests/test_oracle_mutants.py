"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle's C source to a temporary directory, plants one
mistake (a dropped term, a wrong sign or index, a transposed operand), compiles
it, and runs every pin in test_oracle_pins.py against the mutant.  At least one
pin must fail for every mutant.  Everything runs on the CPU; the real oracle is
untouched.
"""
import inspect
import json
import os
import subprocess
import ctypes

import numpy as np
import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gattn_oracle.c")

MUTANTS = {
    "gqa_strided_mapping": ("int g = h / r;", "int g = h % G;"),
    "scale_by_d_not_sqrt_d": ("double scale = 1.0 / sqrt((double)d);", "double scale = 1.0 / (double)d;"),
    "no_scale": ("double scale = 1.0 / sqrt((double)d);", "double scale = 1.0;"),
    "rope_sign_flip": ("y[i] = a * c - b * s;", "y[i] = a * c + b * s;"),
    "rope_exponent_over_d": ("pow(base, -2.0 * (double)i / (double)rd)", "pow(base, -2.0 * (double)i / (double)d)"),
    "rope_adjacent_pairs": ("double a = x[i], b = x[i + half];", "double a = x[2 * i], b = x[2 * i + 1];"),
    "causal_excludes_diagonal": ("attend_row(qt, kb, (int64_t)G * d, vb, (int64_t)G * d, t + 1,",
                                 "attend_row(qt, kb, (int64_t)G * d, vb, (int64_t)G * d, t > 0 ? t : 1,"),
    "gate_negated": ("double s = oracle_sigmoid(z);", "double s = oracle_sigmoid(-z);"),
    "gate_transposed_dim": ("layout == ORACLE_GATE_HEADWISE ? z[0] : z[e], act);",
                            "layout == ORACLE_GATE_HEADWISE ? z[0] : z[d - 1 - e], act);"),
    "rmsnorm_sum_not_mean": ("double inv = 1.0 / sqrt(ss / (double)d + eps);", "double inv = 1.0 / sqrt(ss + eps);"),
    "rmsnorm_eps_outside": ("double inv = 1.0 / sqrt(ss / (double)d + eps);",
                            "double inv = 1.0 / (sqrt(ss / (double)d) + eps);"),
    "rmsnorm_drops_weight": ("y[r * d + e] = xr[e] * inv * w[e];", "y[r * d + e] = xr[e] * inv;"),
    "softmax_not_normalised": ("double wj = scratch[j] / z;", "double wj = scratch[j];"),
    "values_from_keys": ("o[e] += wj * v[j * val_stride + e];", "o[e] += wj * kr[j * key_stride + e];"),
    "decode_position_off_by_one": ("rope_row(tmp, (double)(L - 1), d, rd, base, qr);",
                                   "rope_row(tmp, (double)L, d, rd, base, qr);"),
    "prefill_k_uses_q_weight": ("prologue_head(k + (int64_t)b * S * G * d, knorm_w, posb, S, G, g,",
                                "prologue_head(k + (int64_t)b * S * G * d, qnorm_w, posb, S, G, g,"),
    "headwise_gate_index": ("case ORACLE_GATE_HEADWISE: return gate + bt * H + h;",
                            "case ORACLE_GATE_HEADWISE: return gate + bt * H;"),
    "ns_sigmoid_without_offset": ("return 0.5 + 0.5 * s;", "return 0.5 * s;"),
    "silu_is_sigmoid": ("return z * s;", "return s;"),
    "additive_multiplies": ("o[e] = additive ? o[e] + g : o[e] * g;", "o[e] = o[e] * g;"),
    "append_at_seqlen": ("double* kdst = kcache + (((int64_t)b * G + g) * Lmax + (L - 1)) * d;",
                         "double* kdst = kcache + (((int64_t)b * G + g) * Lmax + (L > 1 ? L - 2 : 0)) * d;"),
    "append_normed_with_q_weight": ("oracle_rmsnorm(kn, knorm_w, 1, d, eps, tmp);",
                                    "oracle_rmsnorm(kn, qnorm_w, 1, d, eps, tmp);"),
    "append_rotated_at_seqlen": ("rope_row(tmp, (double)(L - 1), d, rd, base, kdst);",
                                 "rope_row(tmp, (double)L, d, rd, base, kdst);"),
    "head_shared_previous_token": ("case ORACLE_GATE_HEAD_SHARED: return gate + bt * d;",
                                   "case ORACLE_GATE_HEAD_SHARED: return gate + (bt > 0 ? bt - 1 : 0) * d;"),
}


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_") or name == "test_kv_cache_byte_accounting":
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argnames, values = params[0].args
            names = [a.strip() for a in argnames.split(",")]
            for vals in values:
                out.append((name, fn, dict(zip(names, vals if isinstance(vals, tuple) else (vals,)))))
        else:
            out.append((name, fn, {}))
    return out


def _golden(name):
    with open(os.path.join(os.path.dirname(pins.__file__), "golden", name)) as f:
        return json.load(f)


def _compile_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: " + old
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(path), "-o", str(lib), "-lm"],
                   check=True)
    return str(lib)


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_mutant(mutant, tmp_path):
    old, new = MUTANTS[mutant]
    libpath = _compile_mutant(tmp_path, old, new)
    real = oracle._load()
    mutant_lib = ctypes.CDLL(libpath)
    for fname in ("oracle_sigmoid", "oracle_gate_act", "oracle_rmsnorm", "oracle_rope", "oracle_gate", "oracle_sdpa_gate",
                  "oracle_prefill", "oracle_prefill_rows", "oracle_decode", "oracle_decode_append"):
        getattr(mutant_lib, fname).argtypes = getattr(real, fname).argtypes
        getattr(mutant_lib, fname).restype = getattr(real, fname).restype
    caught = []
    oracle._lib = mutant_lib
    try:
        for name, fn, kwargs in _pin_functions():
            args = {}
            if "golden" in inspect.signature(fn).parameters:
                args["golden"] = _golden
            try:
                fn(**args, **kwargs)
            except AssertionError:
                caught.append(name)
    finally:
        oracle._lib = real
    assert caught, "no pin caught mutant " + mutant


# The packed-sequence oracle is a Python wrapper over the batched one: plausible
# mistakes in it, planted in a copy of the wrapper, must fail a pin too.
def _varlen_mutant(kind):
    def mutant(q, k, v, gate_logits, qnorm_w, knorm_w, pos, cu_seqlens, rotary_dim, rope_base, eps, gate_mode):
        q, k, v = np.asarray(q, np.float64), np.asarray(k, np.float64), np.asarray(v, np.float64)
        T, H, d = q.shape
        cu = [int(x) for x in np.asarray(cu_seqlens)]
        z = None if gate_logits is None else np.asarray(gate_logits, np.float64)
        p = None if pos is None else np.asarray(pos, np.float64)
        out = np.zeros((T, H * d))
        for i in range(len(cu) - 1):
            s, e = cu[i], cu[i + 1]
            if e <= s:
                continue
            ps = p[s:e] if p is not None else None
            if kind == "positions_continue" and p is None:
                ps = np.arange(s, e, dtype=np.float64)  # positions run on across sequences
            lo = s
            if kind == "keys_leak_from_previous" and i > 0:
                lo = cu[i - 1]  # the previous sequence's tokens are visible too
                if ps is not None:
                    ps = np.concatenate([np.arange(s - lo, dtype=np.float64), ps])
            zs = None if z is None else z[lo:e]
            if kind == "gate_of_previous_sequence" and z is not None and i > 0 and cu[i] - cu[i - 1] >= e - s:
                zs = z[cu[i - 1]:cu[i - 1] + (e - s)]
            res = oracle.prefill(q[None, lo:e], k[None, lo:e], v[None, lo:e], None if zs is None else zs[None],
                                 qnorm_w, knorm_w, None if ps is None else ps[None], rotary_dim, rope_base, eps,
                                 gate_mode)[0]
            out[s:e] = res[s - lo:]
        return out
    return mutant


@pytest.mark.parametrize("kind", ["positions_continue", "keys_leak_from_previous", "gate_of_previous_sequence"])
def test_pins_catch_varlen_mutant(kind, monkeypatch):
    monkeypatch.setattr(oracle, "prefill_varlen", _varlen_mutant(kind))
    with pytest.raises(AssertionError):
        pins.test_varlen_sequences_are_independent_batches()


def test_varlen_mutant_harness_is_faithful(monkeypatch):
    """With no mistake planted the copied wrapper passes the pin (so the mutants
    above fail for their mistake, not for the copy)."""
    monkeypatch.setattr(oracle, "prefill_varlen", _varlen_mutant("none"))
    pins.test_varlen_sequences_are_independent_batches()
