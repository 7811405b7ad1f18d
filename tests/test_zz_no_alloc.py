"""gattn_decode_noalloc: decode for callers that cannot allocate device memory
while they decode (its partial states live in the library's own fixed device
array instead of a caller workspace).

The test drives the entry point through the C ABI with ctypes and checks two
calls in a row against gattn_decode with a workspace, within the bf16 parity
tolerance the other decode tests use; the second call uses different lengths, so
it also shows that whatever the first call left in the shared array does not
leak into the next result.  It lives in a file of its own, collected last.
"""
import ctypes

import pytest
import torch

from gated_softmax_attention_gqa_gb300 import _lib, gattn_decode, gattn_get_device_status
from gated_softmax_attention_gqa_gb300.workloads import Workload, make_decode_inputs
from tests.parity import BF16_MAX_ABS, BF16_MEAN_ABS

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GATE = {"none": 0, "elementwise": 1, "headwise": 2}
WORKSPACE_ERR = 4
SCRATCH_BYTES = 8 << 20  # GATTN_DECODE_NOALLOC_SCRATCH_BYTES


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(lib, d, w, out):
    B, H, dd = d["q_new"].shape
    G, Lmax = d["kv_cache"].shape[2], d["kv_cache"].shape[3]
    return lib.gattn_decode_noalloc(_ptr(d["q_new"]), _ptr(d["kv_cache"]), _ptr(d["seqlens"]), _ptr(d["gate"]),
                                    _ptr(d["qnorm_w"]), B, H, G, dd, Lmax, w.rotary_dim, w.rope_base, w.eps,
                                    GATE[w.gate_mode], _ptr(out),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _close(a, b):
    diff = (a.double() - b.double()).abs()
    assert torch.isfinite(a).all()
    assert diff.max().item() <= BF16_MAX_ABS and diff.mean().item() <= BF16_MEAN_ABS, diff.max().item()


def test_noalloc_decode_matches_workspace_decode_twice():
    lib = _lib.load()
    cases = [
        Workload("na1", "decode", B=6, H=8, G=2, d=256, rotary_dim=64, rope_base=1e7, gate_mode="elementwise",
                 dtype="bf16", seed=71, Lmax=3000, seqlen_range=(1, 3000)),
        Workload("na2", "decode", B=5, H=16, G=8, d=128, rotary_dim=128, rope_base=1e6, gate_mode="headwise",
                 dtype="bf16", seed=72, Lmax=1500, seqlen_range=(200, 1500)),
    ]
    for w in cases:
        d = {k: v.to(DEV) for k, v in make_decode_inputs(w).items()}
        ref = gattn_decode(d["q_new"], d["kv_cache"], d["seqlens"], d["gate"], d["qnorm_w"], rotary_dim=w.rotary_dim,
                           rope_base=w.rope_base, eps=w.eps, gate_mode=w.gate_mode)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(lib, d, w, out) == 0
        torch.cuda.synchronize()
        _close(out, ref)
        assert gattn_get_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    B, H, G, dd, Lmax = 2048, 8, 8, 256, 1  # partial states far above 8 MiB, tiny cache
    assert lib.gattn_decode_workspace_size(B, H, G, dd, Lmax) > SCRATCH_BYTES
    w = Workload("big", "decode", B=B, H=H, G=G, d=dd, rotary_dim=64, rope_base=1e7, gate_mode="none",
                 dtype="bf16", seed=73, Lmax=Lmax, seqlen_range=(1, Lmax))
    d = {k: v.to(DEV) for k, v in make_decode_inputs(w).items()}
    d["gate"] = None
    out = torch.zeros((B, H * dd), dtype=torch.bfloat16, device=DEV)
    assert _noalloc(lib, d, w, out) == WORKSPACE_ERR
    torch.cuda.synchronize()
    assert (out == 0).all()  # nothing was launched
