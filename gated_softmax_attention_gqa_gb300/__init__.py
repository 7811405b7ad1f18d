"""GB300-native gated softmax attention with GQA (libgattn).

The Python names mirror the C ABI in include/gattn.h.  Each call hands raw
device pointers, sizes and the current CUDA stream to libgattn.so; every step of
the computation runs in the library's CUDA kernels.  PyTorch only supplies
device memory and streams.  If the library is not built, calls raise: there is
no CPU fallback.

    out = gattn_prefill(q, k, v, gate, qnorm_w, knorm_w, rotary_dim=64, rope_base=1e7)
    out = gattn_decode(q_new, kv_cache, seqlens, gate, qnorm_w, rotary_dim=64, rope_base=1e7)
"""
import ctypes

import torch

from . import _lib
from ._lib import GattnError, check

# gate_mode = layout | activation | additive (the bit fields of gattn_gate_mode in gattn.h)
GATE_MODES = {"none": 0, "elementwise": 1, "headwise": 2, "head_shared": 3}
GATE_ACTS = {"sigmoid": 0x00, "ns_sigmoid": 0x10, "silu": 0x20}
GATE_ADDITIVE = 0x100
DTYPES = {torch.bfloat16: 0, torch.float32: 1}

__all__ = ["gattn_prefill", "gattn_prefill_varlen", "gattn_decode", "gattn_decode_append", "gattn_decode_paged", "gattn_decode_noalloc", "gattn_prefill_workspace_size", "gattn_prefill_varlen_workspace_size", "gattn_decode_workspace_size",
           "gattn_get_device_status", "gattn_set_profile_events", "gattn_selftest_wait_timeout", "gattn_o_proj", "gattn_strerror", "GattnError", "GATE_MODES",
           "GATE_ACTS", "GATE_ADDITIVE"]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _mode(gate_mode, gate_act="sigmoid", gate_additive=False):
    """The C gate_mode for a layout name, an activation name and the additive flag
    (an int is passed through unchanged)."""
    if not isinstance(gate_mode, str):
        return int(gate_mode)
    m = GATE_MODES[gate_mode]
    if m == 0:
        if gate_act != "sigmoid" or gate_additive:
            raise ValueError("gate_act / gate_additive need a gate")
        return 0
    return m | GATE_ACTS[gate_act] | (GATE_ADDITIVE if gate_additive else 0)


def gattn_strerror(status: int) -> str:
    return _lib.strerror(status)


def gattn_prefill_workspace_size(B, S, H, G, d, dtype=torch.bfloat16) -> int:
    return _lib.load().gattn_prefill_workspace_size(B, S, H, G, d, DTYPES[dtype])


def gattn_prefill_varlen_workspace_size(T, nseq, H, G, d, dtype=torch.bfloat16) -> int:
    return _lib.load().gattn_prefill_varlen_workspace_size(T, nseq, H, G, d, DTYPES[dtype])


def gattn_decode_workspace_size(B, H, G, d, Lmax) -> int:
    return _lib.load().gattn_decode_workspace_size(B, H, G, d, Lmax)


def gattn_set_profile_events(start=None, stop=None):
    """Record `start`/`stop` (torch.cuda.Event) around the main attention kernel of
    every later call; None, None switches it off."""
    for e in (start, stop):
        if e is not None and e.cuda_event == 0:
            e.record()  # torch creates the underlying cudaEvent lazily, on first record
    _lib.load().gattn_set_profile_events(ctypes.c_void_p(start.cuda_event) if start is not None else None,
                                         ctypes.c_void_p(stop.cuda_event) if stop is not None else None)


def gattn_get_device_status(stream=None) -> int:
    """Read and clear the device status bits (GATTN_DEVICE_* in gattn.h)."""
    bits = ctypes.c_uint(0)
    st = _lib.load().gattn_get_device_status(ctypes.byref(bits), _stream_handle(stream, None))
    if st not in (0, 5, 6):
        check(st, "gattn_get_device_status")
    return bits.value


def gattn_selftest_wait_timeout(limit_ns, waited_ns=None, stream=None):
    """Launch the bounded-wait self-test: a wait on an mbarrier nothing arrives on,
    given up after limit_ns (1e6 .. 1e8).  waited_ns: optional int64 CUDA tensor of
    one element that receives the wait's duration.  The timeout is read back with
    gattn_get_device_status()."""
    st = _lib.load().gattn_selftest_wait_timeout(int(limit_ns), _ptr(waited_ns), _stream_handle(stream, None))
    check(st, "gattn_selftest_wait_timeout")


def gattn_o_proj(x, w_o, out=None, stream=None):
    """Output projection of the attention output: out = x w_o^T.

    x [..., K] bf16 CUDA (the [B,S,H*d] or [T,H*d] output of gattn_prefill /
    gattn_prefill_varlen), contiguous; w_o [N, K] bf16 CUDA, contiguous (a linear
    layer's weight); out [..., N] bf16 (allocated if None).  K and N multiples of 64."""
    if x.dtype != torch.bfloat16 or w_o.dtype != torch.bfloat16:
        raise ValueError("x and w_o must be bfloat16")
    if not x.is_contiguous() or not w_o.is_contiguous() or w_o.dim() != 2:
        raise ValueError("x and w_o must be contiguous; w_o is [N, K]")
    K = x.shape[-1]
    N = w_o.shape[0]
    if w_o.shape[1] != K:
        raise ValueError(f"w_o is [{N}, {w_o.shape[1]}], x has K = {K}")
    T = x.numel() // K if K else 0
    if out is None:
        out = torch.empty(*x.shape[:-1], N, dtype=torch.bfloat16, device=x.device)
    elif out.dtype != torch.bfloat16 or not out.is_contiguous() or out.numel() != T * N:
        raise ValueError("out must be a contiguous bf16 tensor of T x N elements")
    st = _lib.load().gattn_o_proj(_ptr(x), _ptr(w_o), T, K, N, _ptr(out), _stream_handle(stream, x.device))
    check(st, "gattn_o_proj")
    return out


def _head_strides(t, name):
    """(token stride, head stride) in elements of a [B,S,H,*] or [B,S,H] view whose
    element (b,t,h,...) sits at (b*S + t)*token_stride + h*head_stride + ...."""
    if t.dim() not in (3, 4):
        raise ValueError(f"{name}: expected 3 or 4 dimensions")
    if t.dim() == 4 and t.stride(-1) != 1:
        raise ValueError(f"{name}: the last dimension must be contiguous")
    B, S = t.shape[0], t.shape[1]
    tok = t.stride(1) if S > 1 else t.stride(0)
    if B > 1 and S > 1 and t.stride(0) != S * t.stride(1):
        raise ValueError(f"{name}: batches must be evenly spaced tokens (stride(0) == S * stride(1))")
    return tok, t.stride(2)


def gattn_prefill(q, k, v, gate, qnorm_w, knorm_w, pos=None, *, rotary_dim, rope_base, eps=1e-6,
                  gate_mode="elementwise", gate_act="sigmoid", gate_additive=False, out=None, workspace=None,
                  stream=None):
    """Causal gated GQA attention over whole sequences.

    q [B,S,H,d] (may be a strided view, e.g. the query half of the packed q_proj
    output [B,S,H,2d]); k, v [B,S,G,d] contiguous; gate [B,S,H,d] (elementwise),
    [B,S,H] (headwise), [B,S,d] (head_shared: one vector for every head) or None;
    gate_act "sigmoid" | "ns_sigmoid" | "silu"; gate_additive: out = o + act(z)
    instead of o * act(z); qnorm_w, knorm_w [d]; pos [B,S] int32 or None.
    All on one CUDA device, bf16 or fp32 (all the same).  Returns out [B,S,H*d]."""
    mode = _mode(gate_mode, gate_act, gate_additive)
    B, S, H, d = q.shape
    G = k.shape[2]
    dt = DTYPES[q.dtype]
    qts, qhs = _head_strides(q, "q")
    if (mode & 0x0F) == GATE_MODES["head_shared"]:
        if gate.dim() != 3 or gate.stride(-1) != 1:
            raise ValueError("gate: a head-shared gate is [B,S,d] with a contiguous last dimension")
        if B > 1 and S > 1 and gate.stride(0) != S * gate.stride(1):
            raise ValueError("gate: batches must be evenly spaced tokens (stride(0) == S * stride(1))")
        gts, ghs = (gate.stride(1) if S > 1 else gate.stride(0)), 0
    elif mode & 0x0F:
        gts, ghs = _head_strides(gate, "gate")
    else:
        gate, gts, ghs = None, 0, 0
    if not (k.is_contiguous() and v.is_contiguous()):
        raise ValueError("k and v must be contiguous [B,S,G,d]")
    if pos is not None and (pos.dtype != torch.int32 or not pos.is_contiguous()):
        raise ValueError("pos must be a contiguous int32 [B,S] tensor")
    if out is None:
        out = torch.empty((B, S, H * d), dtype=q.dtype, device=q.device)
    need = gattn_prefill_workspace_size(B, S, H, G, d, q.dtype)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = _lib.load().gattn_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(qnorm_w), _ptr(knorm_w), _ptr(pos), B, S, H, G, d,
        int(rotary_dim), float(rope_base), float(eps), mode, qts, qhs, gts, ghs, dt, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _stream_handle(stream, q.device))
    check(st, "gattn_prefill")
    return out


def gattn_prefill_varlen(q, k, v, gate, qnorm_w, knorm_w, cu_seqlens, pos=None, *, rotary_dim, rope_base,
                         eps=1e-6, gate_mode="elementwise", gate_act="sigmoid", gate_additive=False, out=None,
                         workspace=None, stream=None):
    """Causal gated GQA attention over packed variable-length sequences: sequence i
    is tokens [cu_seqlens[i], cu_seqlens[i+1]) of q [T,H,d] (last dimension
    contiguous), k, v [T,G,d] contiguous and gate [T,H,d] / [T,H] / [T,d]; it sees
    only its own keys and its positions restart at 0 unless pos [T] int32 is given.
    cu_seqlens: host int32 sequence (list, numpy array or CPU tensor).  Returns
    out [T,H*d]."""
    mode = _mode(gate_mode, gate_act, gate_additive)
    T, H, d = q.shape
    G = k.shape[1]
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int32, device="cpu").contiguous()
    nseq = cu.numel() - 1
    if nseq < 1 or int(cu[-1]) != T:
        raise ValueError("cu_seqlens must have nseq+1 entries ending at T")
    if q.stride(-1) != 1:
        raise ValueError("q: the last dimension must be contiguous")
    if not (k.is_contiguous() and v.is_contiguous()):
        raise ValueError("k and v must be contiguous [T,G,d]")
    layout = mode & 0x0F
    if layout == 0:
        gate, gts, ghs = None, 0, 0
    elif layout == GATE_MODES["head_shared"]:
        gts, ghs = gate.stride(0), 0
    else:
        gts, ghs = gate.stride(0), gate.stride(1)
    if pos is not None and (pos.dtype != torch.int32 or not pos.is_contiguous()):
        raise ValueError("pos must be a contiguous int32 [T] tensor")
    if out is None:
        out = torch.empty((T, H * d), dtype=q.dtype, device=q.device)
    dt = DTYPES[q.dtype]
    need = _lib.load().gattn_prefill_varlen_workspace_size(T, nseq, H, G, d, dt)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = _lib.load().gattn_prefill_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(qnorm_w), _ptr(knorm_w), _ptr(pos), ctypes.c_void_p(cu.data_ptr()),
        nseq, H, G, d, int(rotary_dim), float(rope_base), float(eps), mode, q.stride(0), q.stride(1), gts, ghs, dt,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _stream_handle(stream, q.device))
    check(st, "gattn_prefill_varlen")
    return out


def _check_decode_inputs(q_new, kv_cache, seqlens, gate, qnorm_w, mode, out):
    """The layout checks every contiguous-cache decode entry point makes before it
    hands pointers to the library: the kernels index these tensors as dense arrays."""
    for name, t in (("q_new", q_new), ("kv_cache", kv_cache), ("seqlens", seqlens), ("qnorm_w", qnorm_w)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if mode & 0x0F and not gate.is_contiguous():
        raise ValueError("gate must be contiguous")
    if seqlens.dtype != torch.int32:
        raise ValueError("seqlens must be int32")
    if q_new.dim() != 3 or kv_cache.dim() != 5 or kv_cache.shape[0] != 2 or kv_cache.shape[1] != q_new.shape[0]:
        raise ValueError("q_new must be [B,H,d] and kv_cache [2,B,G,Lmax,d]")
    if out is not None and (not out.is_contiguous() or out.numel() != q_new.numel()):
        raise ValueError("out must be a contiguous [B,H*d] tensor")


def gattn_decode(q_new, kv_cache, seqlens, gate, qnorm_w, *, rotary_dim, rope_base, eps=1e-6,
                 gate_mode="elementwise", gate_act="sigmoid", gate_additive=False, out=None, workspace=None,
                 stream=None):
    """One decode step.  q_new [B,H,d] raw; kv_cache [2,B,G,Lmax,d] (K normed and
    rotated, V raw); seqlens [B] int32 including the new token; gate [B,H,d]
    (elementwise), [B,H] (headwise), [B,d] (head_shared) or None; gate_act and
    gate_additive as for gattn_prefill; qnorm_w [d].  bf16.  Returns out [B,H*d]."""
    mode = _mode(gate_mode, gate_act, gate_additive)
    B, H, d = q_new.shape
    G, Lmax = kv_cache.shape[2], kv_cache.shape[3]
    _check_decode_inputs(q_new, kv_cache, seqlens, gate, qnorm_w, mode, out)
    if out is None:
        out = torch.empty((B, H * d), dtype=q_new.dtype, device=q_new.device)
    need = gattn_decode_workspace_size(B, H, G, d, Lmax)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q_new.device)
    st = _lib.load().gattn_decode(
        _ptr(q_new), _ptr(kv_cache), _ptr(seqlens), _ptr(gate if mode & 0x0F else None), _ptr(qnorm_w), B, H, G, d,
        Lmax, int(rotary_dim), float(rope_base), float(eps), mode, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _stream_handle(stream, q_new.device))
    check(st, "gattn_decode")
    return out


def gattn_decode_append(q_new, k_new, v_new, kv_cache, seqlens, gate, qnorm_w, knorm_w, *, rotary_dim, rope_base,
                        eps=1e-6, gate_mode="elementwise", gate_act="sigmoid", gate_additive=False, out=None,
                        workspace=None, stream=None):
    """One decode step that first writes the new token into the cache: k_new,
    v_new [B,G,d] raw (K is normed with knorm_w and rotated at position
    seqlens[b]-1); kv_cache [2,B,G,Lmax,d] is updated in place at row
    seqlens[b]-1; the rest as gattn_decode.  Returns out [B,H*d]."""
    mode = _mode(gate_mode, gate_act, gate_additive)
    B, H, d = q_new.shape
    G, Lmax = kv_cache.shape[2], kv_cache.shape[3]
    for name, t in (("q_new", q_new), ("k_new", k_new), ("v_new", v_new), ("kv_cache", kv_cache),
                    ("seqlens", seqlens), ("qnorm_w", qnorm_w), ("knorm_w", knorm_w)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if tuple(k_new.shape) != (B, G, d) or tuple(v_new.shape) != (B, G, d):
        raise ValueError("k_new and v_new must be [B,G,d]")
    if mode & 0x0F and not gate.is_contiguous():
        raise ValueError("gate must be contiguous")
    if seqlens.dtype != torch.int32:
        raise ValueError("seqlens must be int32")
    if out is None:
        out = torch.empty((B, H * d), dtype=q_new.dtype, device=q_new.device)
    need = gattn_decode_workspace_size(B, H, G, d, Lmax)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q_new.device)
    st = _lib.load().gattn_decode_append(
        _ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(kv_cache), _ptr(seqlens), _ptr(gate if mode & 0x0F else None),
        _ptr(qnorm_w), _ptr(knorm_w), B, H, G, d, Lmax, int(rotary_dim), float(rope_base), float(eps), mode,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        _stream_handle(stream, q_new.device))
    check(st, "gattn_decode_append")
    return out


def gattn_decode_paged(q_new, kv_pages, block_table, seqlens, gate, qnorm_w, *, rotary_dim, rope_base, eps=1e-6,
                       k_new=None, v_new=None, knorm_w=None, gate_mode="elementwise", gate_act="sigmoid",
                       gate_additive=False, out=None, workspace=None, stream=None):
    """One decode step against a paged cache: kv_pages [2,num_pages,G,page_size,d]
    bf16, block_table [B,max_pages] int32 (page of each page_size-token block of
    each sequence).  With k_new, v_new [B,G,d] and knorm_w the new token is first
    written into its page.  The rest as gattn_decode.  Returns out [B,H*d]."""
    mode = _mode(gate_mode, gate_act, gate_additive)
    B, H, d = q_new.shape
    num_pages, G, page_size = kv_pages.shape[1], kv_pages.shape[2], kv_pages.shape[3]
    max_pages = block_table.shape[1]
    for name, t in (("q_new", q_new), ("kv_pages", kv_pages), ("block_table", block_table), ("seqlens", seqlens),
                    ("qnorm_w", qnorm_w)) + ((("k_new", k_new), ("v_new", v_new), ("knorm_w", knorm_w))
                                             if k_new is not None else ()):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if block_table.dtype != torch.int32 or seqlens.dtype != torch.int32:
        raise ValueError("block_table and seqlens must be int32")
    if mode & 0x0F and not gate.is_contiguous():
        raise ValueError("gate must be contiguous")
    if out is None:
        out = torch.empty((B, H * d), dtype=q_new.dtype, device=q_new.device)
    need = gattn_decode_workspace_size(B, H, G, d, max_pages * page_size)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q_new.device)
    st = _lib.load().gattn_decode_paged(
        _ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(kv_pages), _ptr(block_table), num_pages, page_size, max_pages,
        _ptr(seqlens), _ptr(gate if mode & 0x0F else None), _ptr(qnorm_w), _ptr(knorm_w), B, H, G, d,
        int(rotary_dim), float(rope_base), float(eps), mode, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _stream_handle(stream, q_new.device))
    check(st, "gattn_decode_paged")
    return out


def gattn_decode_noalloc(q_new, kv_cache, seqlens, gate, qnorm_w, *, rotary_dim, rope_base, eps=1e-6,
                         gate_mode="elementwise", gate_act="sigmoid", gate_additive=False, out=None, stream=None):
    """gattn_decode without a workspace: the partial states live in the library's
    own fixed device array (GATTN_DECODE_NOALLOC_SCRATCH_BYTES).  For callers that
    must not allocate device memory while decoding; pass `out` to allocate nothing
    here either.  Calls that overlap on the GPU race on that array."""
    mode = _mode(gate_mode, gate_act, gate_additive)
    B, H, d = q_new.shape
    G, Lmax = kv_cache.shape[2], kv_cache.shape[3]
    _check_decode_inputs(q_new, kv_cache, seqlens, gate, qnorm_w, mode, out)
    if out is None:
        out = torch.empty((B, H * d), dtype=q_new.dtype, device=q_new.device)
    st = _lib.load().gattn_decode_noalloc(
        _ptr(q_new), _ptr(kv_cache), _ptr(seqlens), _ptr(gate if mode & 0x0F else None), _ptr(qnorm_w), B, H, G, d,
        Lmax, int(rotary_dim), float(rope_base), float(eps), mode, _ptr(out), _stream_handle(stream, q_new.device))
    check(st, "gattn_decode_noalloc")
    return out
