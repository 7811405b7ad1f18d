"""gattn_decode_noalloc: decode for callers that cannot allocate device memory
while they decode (its partial states live in the library's own fixed device
array instead of a caller workspace).

The first test drives the entry point through the C ABI with ctypes, two calls in
a row, and checks each result against the fp64 oracle and against gattn_decode
with a workspace, within the bf16 parity tolerance the other decode tests use;
the second call uses other lengths and shapes, so it also shows that whatever the
first call left in the shared array does not leak into the next result.  The
file is collected last.
"""
import ctypes

import pytest
import torch

import oracle
from gated_softmax_attention_gqa_gb300 import _lib, gattn_decode, gattn_decode_noalloc, gattn_get_device_status
from gated_softmax_attention_gqa_gb300.workloads import Workload, make_decode_inputs
from tests.parity import BF16_MAX_ABS, BF16_MEAN_ABS, assert_close_to_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GATE = {"none": 0, "elementwise": 1, "headwise": 2}
INVALID, UNSUPPORTED, WORKSPACE_ERR = 1, 2, 4
SCRATCH_BYTES = 8 << 20  # GATTN_DECODE_NOALLOC_SCRATCH_BYTES


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(lib, d, w, out, **over):
    B, H, dd = d["q_new"].shape
    G, Lmax = d["kv_cache"].shape[2], d["kv_cache"].shape[3]
    a = dict(q=_ptr(d["q_new"]), B=B)
    a.update(over)
    return lib.gattn_decode_noalloc(a["q"], _ptr(d["kv_cache"]), _ptr(d["seqlens"]), _ptr(d["gate"]),
                                    _ptr(d["qnorm_w"]), a["B"], H, G, dd, Lmax, w.rotary_dim, w.rope_base, w.eps,
                                    GATE[w.gate_mode], _ptr(out),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _oracle(inp, w):
    return oracle.decode(inp["q_new"], inp["kv_cache"][0], inp["kv_cache"][1], inp["seqlens"], inp["gate"],
                         inp["qnorm_w"], w.rotary_dim, w.rope_base, w.eps, w.gate_mode)


def _close(a, b):
    diff = (a.double() - b.double()).abs()
    assert torch.isfinite(a).all()
    assert diff.max().item() <= BF16_MAX_ABS and diff.mean().item() <= BF16_MEAN_ABS, diff.max().item()


CASES = [
    Workload("na1", "decode", B=6, H=8, G=2, d=256, rotary_dim=64, rope_base=1e7, gate_mode="elementwise",
             dtype="bf16", seed=71, Lmax=3000, seqlen_range=(1, 3000)),
    Workload("na2", "decode", B=5, H=16, G=8, d=128, rotary_dim=128, rope_base=1e6, gate_mode="headwise",
             dtype="bf16", seed=72, Lmax=1500, seqlen_range=(200, 1500)),
]


def test_noalloc_decode_matches_the_oracle_and_workspace_decode_twice():
    lib = _lib.load()
    for w in CASES:
        inp = make_decode_inputs(w)
        d = {k: v.to(DEV) for k, v in inp.items()}
        out = torch.full((w.B, w.H * w.d), float("nan"), dtype=torch.bfloat16, device=DEV)
        assert _noalloc(lib, d, w, out) == 0
        torch.cuda.synchronize()
        assert_close_to_oracle(out, _oracle(inp, w), torch.bfloat16, f"{w.name} no-alloc vs oracle")
        ref = gattn_decode(d["q_new"], d["kv_cache"], d["seqlens"], d["gate"], d["qnorm_w"], rotary_dim=w.rotary_dim,
                           rope_base=w.rope_base, eps=w.eps, gate_mode=w.gate_mode)
        torch.cuda.synchronize()
        _close(out, ref)
        assert gattn_get_device_status() == 0


def test_noalloc_python_wrapper_checks_and_matches_the_oracle():
    w = CASES[1]
    inp = make_decode_inputs(w)
    d = {k: v.to(DEV) for k, v in inp.items()}
    out = gattn_decode_noalloc(d["q_new"], d["kv_cache"], d["seqlens"], d["gate"], d["qnorm_w"],
                               rotary_dim=w.rotary_dim, rope_base=w.rope_base, eps=w.eps, gate_mode=w.gate_mode)
    torch.cuda.synchronize()
    assert_close_to_oracle(out, _oracle(inp, w), torch.bfloat16, "no-alloc wrapper vs oracle")
    kw = dict(rotary_dim=w.rotary_dim, rope_base=w.rope_base, eps=w.eps, gate_mode=w.gate_mode)
    with pytest.raises(ValueError):  # a strided view of the cache
        gattn_decode_noalloc(d["q_new"], d["kv_cache"][:, :, :, ::2], d["seqlens"], d["gate"], d["qnorm_w"], **kw)
    with pytest.raises(ValueError):  # int64 lengths
        gattn_decode_noalloc(d["q_new"], d["kv_cache"], d["seqlens"].long(), d["gate"], d["qnorm_w"], **kw)
    assert gattn_get_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    B, H, G, dd, Lmax = 2048, 8, 8, 256, 1  # partial states far above 8 MiB, tiny cache
    assert lib.gattn_decode_workspace_size(B, H, G, dd, Lmax) > SCRATCH_BYTES
    w = Workload("big", "decode", B=B, H=H, G=G, d=dd, rotary_dim=64, rope_base=1e7, gate_mode="none",
                 dtype="bf16", seed=73, Lmax=Lmax, seqlen_range=(1, Lmax))
    d = {k: v.to(DEV) for k, v in make_decode_inputs(w).items()}
    d["gate"] = None
    out = torch.full((B, H * dd), 7.0, dtype=torch.bfloat16, device=DEV)
    assert _noalloc(lib, d, w, out) == WORKSPACE_ERR
    # argument errors on a shape beyond the scratch get gattn_decode's status, not the scratch's
    assert _noalloc(lib, d, w, out, q=None) == INVALID
    assert _noalloc(lib, d, w, out, B=B + 1) == UNSUPPORTED  # more sequences than a call takes
    torch.cuda.synchronize()
    assert (out == 7.0).all()  # no launch wrote the output
    assert gattn_get_device_status() == 0
