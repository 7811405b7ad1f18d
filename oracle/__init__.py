"""fp64 CPU oracle for the gated softmax attention core -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The GPU library never uses it: there is no CPU
fallback in the product path.

The arithmetic lives in ``gattn_oracle.c`` (plain double-precision loops, each
step citing the page it follows); this module only marshals numpy arrays into
that library with ctypes.  Every function takes and returns float64 numpy
arrays in the layouts documented there.

Pinned by ``tests/test_oracle_pins.py`` against the pages' worked examples, the
mathematics' closed forms and library special cases.  The RoPE frequency and
pairing convention is a reading (the pages do not print ``apply_rope``): it is
pinned to closed forms of that reading, not to a printed value.
"""
import ctypes
import os

import numpy as np

from . import build as _build

# gate_mode = layout | activation << 4 | ADDITIVE (the encoding of gattn_oracle.c)
GATE_NONE, GATE_ELEMENTWISE, GATE_HEADWISE, GATE_HEAD_SHARED = 0, 1, 2, 3
_GATE_MODES = {"none": GATE_NONE, "elementwise": GATE_ELEMENTWISE, "headwise": GATE_HEADWISE,
               "head_shared": GATE_HEAD_SHARED}
_GATE_ACTS = {"sigmoid": 0, "ns_sigmoid": 1, "silu": 2}
GATE_ADDITIVE = 256


def gate_code(layout, act="sigmoid", additive=False):
    """The oracle's gate_mode for a layout name, an activation name and the
    additive flag (Y + act(z) instead of Y * act(z))."""
    return _GATE_MODES[layout] | (_GATE_ACTS[act] << 4) | (GATE_ADDITIVE if additive else 0)

_lib = None
_D = ctypes.POINTER(ctypes.c_double)
_I32 = ctypes.POINTER(ctypes.c_int32)
_int, _dbl = ctypes.c_int, ctypes.c_double


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.oracle_sigmoid.restype = ctypes.c_double
        lib.oracle_sigmoid.argtypes = [_dbl]
        lib.oracle_gate_act.restype = ctypes.c_double
        lib.oracle_gate_act.argtypes = [_dbl, _int]
        lib.oracle_rmsnorm.argtypes = [_D, _D, ctypes.c_int64, _int, _dbl, _D]
        lib.oracle_rope.argtypes = [_D, _D, ctypes.c_int64, _int, _int, _dbl, _D]
        lib.oracle_gate.argtypes = [_D, _D, _int, _int, _int, _D]
        lib.oracle_sdpa_gate.argtypes = [_D, _D, _D, _D, _int, _int, _int, _int, _int, _int, _D, _D]
        lib.oracle_prefill.argtypes = [_D, _D, _D, _D, _D, _D, _D, _int, _int, _int, _int, _int, _int, _dbl,
                                       _dbl, _int, _D]
        lib.oracle_prefill_rows.argtypes = [_D, _D, _D, _D, _D, _D, _D, _int, _int, _int, _int, _int, _int,
                                            _dbl, _dbl, _int, _I32, _I32, _int, _D]
        lib.oracle_decode.argtypes = [_D, _D, _D, _I32, _D, _D, _int, _int, _int, _int, _int, _int, _dbl, _dbl,
                                      _int, _D]
        lib.oracle_decode_append.argtypes = [_D, _D, _D, _D, _D, _I32, _D, _D, _D, _int, _int, _int, _int, _int,
                                             _int, _dbl, _dbl, _int, _D]
        _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


def _gate_mode(mode):
    return _GATE_MODES[mode] if isinstance(mode, str) else int(mode)


def sigmoid(z: float) -> float:
    return _load().oracle_sigmoid(float(z))


def gate_act(z: float, act) -> float:
    """The gate activation of one logit (act: "sigmoid", "ns_sigmoid", "silu")."""
    return _load().oracle_gate_act(float(z), _GATE_ACTS[act] if isinstance(act, str) else int(act))


def rmsnorm(x, w, eps):
    x, w = _f64(x), _f64(w)
    d = x.shape[-1]
    y = np.empty_like(x)
    _load().oracle_rmsnorm(_p(x), _p(w), x.size // d, d, float(eps), _p(y))
    return y


def rope(x, pos, rotary_dim, base):
    """x [..., d]; pos broadcastable to x.shape[:-1] (one position per row)."""
    x = _f64(x)
    d = x.shape[-1]
    pos = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.float64), x.shape[:-1]))
    y = np.empty_like(x)
    _load().oracle_rope(_p(x), _p(pos), x.size // d, d, int(rotary_dim), float(base), _p(y))
    return y


def gate(y, z, gate_mode):
    """y [n_heads, d]; z [n_heads, d] (elementwise), [n_heads] (headwise) or [d]
    (head-shared)."""
    y = _f64(y)
    n_heads, d = y.shape
    mode = _gate_mode(gate_mode)
    z = _f64(z) if z is not None else np.zeros(1)
    out = np.empty_like(y)
    _load().oracle_gate(_p(y), _p(z), n_heads, d, mode, _p(out))
    return out


def sdpa_gate(q, k, v, gate_logits, gate_mode, want_attn=False):
    """Causal GQA attention + gate on q [B,S,H,d], k,v [B,S,G,d] that are already
    normed and rotated.  Returns out [B,S,H*d] (and attn [B,H,S,S])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, H, d = q.shape
    G = k.shape[2]
    mode = _gate_mode(gate_mode)
    z = _f64(gate_logits) if (mode & 15) != GATE_NONE else np.zeros(1)
    out = np.empty((B, S, H * d))
    attn = np.empty((B, H, S, S)) if want_attn else None
    _load().oracle_sdpa_gate(_p(q), _p(k), _p(v), _p(z), B, S, H, G, d, mode, _p(out), _p(attn))
    return (out, attn) if want_attn else out


def o_proj(x, w_o):
    """The output projection that follows the gated attention: the concatenated,
    gated heads x [..., K] (K = H*d) times the o_proj weight w_o [N, K] transposed,
    y[..., n] = sum_k x[..., k] w_o[n, k], in fp64 ("Transformer by Hand, ch. 6",
    section "The code: qwen/attention.py": o_proj after the gate; the weight is a
    linear layer's, applied as x W^T)."""
    x, w = _f64(x), _f64(w_o)
    return x @ w.T


def prefill(q, k, v, gate_logits, qnorm_w, knorm_w, pos, rotary_dim, rope_base, eps, gate_mode):
    """Full prefill on raw q [B,S,H,d], k,v [B,S,G,d]; pos [B,S] or None."""
    q, k, v, qw, kw = _f64(q), _f64(k), _f64(v), _f64(qnorm_w), _f64(knorm_w)
    B, S, H, d = q.shape
    G = k.shape[2]
    mode = _gate_mode(gate_mode)
    z = _f64(gate_logits) if (mode & 15) != GATE_NONE else np.zeros(1)
    p = _f64(pos)
    out = np.empty((B, S, H * d))
    _load().oracle_prefill(_p(q), _p(k), _p(v), _p(z), _p(qw), _p(kw), _p(p), B, S, H, G, d, int(rotary_dim),
                           float(rope_base), float(eps), mode, _p(out))
    return out


def prefill_varlen(q, k, v, gate_logits, qnorm_w, knorm_w, pos, cu_seqlens, rotary_dim, rope_base, eps,
                   gate_mode):
    """Packed variable-length prefill: sequences i = [cu_seqlens[i], cu_seqlens[i+1])
    of q [T,H,d], k,v [T,G,d], gate [T,H,d] / [T,H] / [T,d]; pos [T] or None
    (positions then restart at 0 in every sequence).  Each sequence is a batch
    of one, attending only to its own keys.  Returns out [T, H*d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, d = q.shape
    cu = [int(x) for x in np.asarray(cu_seqlens if not hasattr(cu_seqlens, "cpu") else cu_seqlens.cpu())]
    mode = _gate_mode(gate_mode)
    z = _f64(gate_logits) if (mode & 15) != GATE_NONE else None
    p = _f64(pos)
    out = np.zeros((T, H * d))
    for i in range(len(cu) - 1):
        s, e = cu[i], cu[i + 1]
        if e <= s:
            continue
        out[s:e] = prefill(q[None, s:e], k[None, s:e], v[None, s:e], None if z is None else z[None, s:e], qnorm_w,
                           knorm_w, None if p is None else p[None, s:e], rotary_dim, rope_base, eps, mode)[0]
    return out


def prefill_rows(q, k, v, gate_logits, qnorm_w, knorm_w, pos, rotary_dim, rope_base, eps, gate_mode, row_b,
                 row_t):
    """Prefill output for the selected tokens (row_b[i], row_t[i]) only: [n, H*d]."""
    q, k, v, qw, kw = _f64(q), _f64(k), _f64(v), _f64(qnorm_w), _f64(knorm_w)
    B, S, H, d = q.shape
    G = k.shape[2]
    mode = _gate_mode(gate_mode)
    z = _f64(gate_logits) if (mode & 15) != GATE_NONE else np.zeros(1)
    p = _f64(pos)
    rb = np.ascontiguousarray(row_b, dtype=np.int32)
    rt = np.ascontiguousarray(row_t, dtype=np.int32)
    out = np.empty((rb.size, H * d))
    _load().oracle_prefill_rows(_p(q), _p(k), _p(v), _p(z), _p(qw), _p(kw), _p(p), B, S, H, G, d,
                                int(rotary_dim), float(rope_base), float(eps), mode, rb.ctypes.data_as(_I32),
                                rt.ctypes.data_as(_I32), rb.size, _p(out))
    return out


def decode(q_new, kcache, vcache, seqlens, gate_logits, qnorm_w, rotary_dim, rope_base, eps, gate_mode):
    """Decode: q_new [B,H,d] raw; kcache, vcache [B,G,Lmax,d]; seqlens [B]."""
    q, kc, vc, qw = _f64(q_new), _f64(kcache), _f64(vcache), _f64(qnorm_w)
    B, H, d = q.shape
    G, Lmax = kc.shape[1], kc.shape[2]
    mode = _gate_mode(gate_mode)
    z = _f64(gate_logits) if (mode & 15) != GATE_NONE else np.zeros(1)
    sl = np.ascontiguousarray(np.asarray(seqlens if not hasattr(seqlens, "cpu") else seqlens.cpu().numpy()),
                              dtype=np.int32)
    out = np.empty((B, H * d))
    _load().oracle_decode(_p(q), _p(kc), _p(vc), sl.ctypes.data_as(_I32), _p(z), _p(qw), B, H, G, d, Lmax,
                          int(rotary_dim), float(rope_base), float(eps), mode, _p(out))
    return out


def decode_append(q_new, k_new, v_new, kcache, vcache, seqlens, gate_logits, qnorm_w, knorm_w, rotary_dim,
                  rope_base, eps, gate_mode):
    """Decode after appending the new token: k_new, v_new [B,G,d] raw; kcache,
    vcache [B,G,Lmax,d] (copied, not modified).  Returns (out [B,H*d], kcache,
    vcache) with the caches as updated."""
    q, kn, vn, qw, kw = _f64(q_new), _f64(k_new), _f64(v_new), _f64(qnorm_w), _f64(knorm_w)
    kc, vc = _f64(kcache).copy(), _f64(vcache).copy()
    B, H, d = q.shape
    G, Lmax = kc.shape[1], kc.shape[2]
    mode = _gate_mode(gate_mode)
    z = _f64(gate_logits) if (mode & 15) != GATE_NONE else np.zeros(1)
    sl = np.ascontiguousarray(np.asarray(seqlens if not hasattr(seqlens, "cpu") else seqlens.cpu().numpy()),
                              dtype=np.int32)
    out = np.empty((B, H * d))
    _load().oracle_decode_append(_p(q), _p(kn), _p(vn), _p(kc), _p(vc), sl.ctypes.data_as(_I32), _p(z), _p(qw),
                                 _p(kw), B, H, G, d, Lmax, int(rotary_dim), float(rope_base), float(eps), mode,
                                 _p(out))
    return out, kc, vc


def threads_used() -> int:
    """OpenMP threads the oracle runs with (OMP_NUM_THREADS, else all cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    return int(env) if env else (os.cpu_count() or 1)
