"""C ABI checks that need no GPU: the library loads, exports every entry point
include/gattn.h declares, and rejects bad arguments on the host before any
CUDA call (so fake, never-dereferenced pointer values are safe here)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from gated_softmax_attention_gqa_gb300 import _lib
from gated_softmax_attention_gqa_gb300.workloads import prefill_flops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, CUDA, WORKSPACE, DEVICE, DEVICE_TIMEOUT = range(7)
FAKE = 0x7F0000000000  # 256-byte aligned, never dereferenced by argument checks


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build_library()
    return _lib.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "gattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gattn_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert set(names) == set(_lib.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_covers_every_status(lib):
    for s in range(7):
        assert lib.gattn_strerror(s).decode().startswith("GATTN_")
    assert b"unknown" in lib.gattn_strerror(99)


def P(off=0):
    return ctypes.c_void_p(FAKE + off)


def prefill(lib, **kw):
    a = dict(q=P(), k=P(), v=P(), gate=P(), qw=P(), kw=P(), pos=None, B=1, S=16, H=8, G=2, d=128, rd=64,
             base=1e6, eps=1e-6, gm=1, qts=0, qhs=0, gts=0, ghs=0, dt=0, ws=P(), wsb=1 << 40, out=P(1 << 20))
    a.update(kw)
    return lib.gattn_prefill(a["q"], a["k"], a["v"], a["gate"], a["qw"], a["kw"], a["pos"], a["B"], a["S"], a["H"],
                             a["G"], a["d"], a["rd"], a["base"], a["eps"], a["gm"], a["qts"], a["qhs"], a["gts"],
                             a["ghs"], a["dt"], a["ws"], a["wsb"], a["out"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), INVALID),
    (dict(out=None), INVALID),
    (dict(gate=None), INVALID),
    (dict(H=6, G=4), INVALID),           # H % G != 0
    (dict(S=0), INVALID),
    (dict(B=0), INVALID),
    (dict(rd=63), INVALID),              # odd rotary_dim
    (dict(rd=130), INVALID),             # rotary_dim > d
    (dict(base=-1.0), INVALID),
    (dict(eps=float("nan")), INVALID),
    (dict(gm=4), INVALID),               # no such gate layout
    (dict(gm=0x31), INVALID),            # no such gate activation
    (dict(gm=0x201), INVALID),           # unknown gate bit
    (dict(gm=0x10), INVALID),            # an activation without a gate
    (dict(gm=0x100), INVALID),           # additive without a gate
    (dict(gm=0x103, gate=None), INVALID),  # head-shared additive gate needs its logits
    (dict(gm=3, gate=P(2)), INVALID),    # head-shared logits are loaded by TMA: 16-byte aligned
    (dict(gm=0x23, gts=100), INVALID),   # head-shared token stride not a multiple of 8 elements
    (dict(dt=7), INVALID),
    (dict(d=96), UNSUPPORTED),           # no bf16 kernel for head_dim 96
    (dict(d=32, rd=16), UNSUPPORTED),    # bf16 needs d >= 64
    (dict(rd=24), UNSUPPORTED),          # bf16 needs rotary_dim % 16 == 0
    (dict(q=P(2)), INVALID),             # misaligned q
    (dict(qts=1028), INVALID),           # token stride not a multiple of 8 elements
    (dict(ws=None), WORKSPACE),
    (dict(ws=P(16)), WORKSPACE),         # workspace not 256-byte aligned
    (dict(wsb=1024), WORKSPACE),         # workspace too small
])
def test_prefill_rejects_bad_arguments(lib, kw, expect):
    assert prefill(lib, **kw) == expect


def test_fp32_accepts_other_shapes_only_where_supported(lib):
    assert prefill(lib, dt=1, d=96) == UNSUPPORTED
    assert prefill(lib, dt=1, d=32, rd=8, wsb=16) == WORKSPACE  # d=32 and rd=8 are fine in fp32


def decode(lib, **kw):
    a = dict(q=P(), kv=P(), sl=P(), gate=P(), qw=P(), B=4, H=8, G=2, d=256, L=1024, rd=64, base=1e7, eps=1e-6, gm=1,
             ws=P(), wsb=1 << 40, out=P(1 << 20))
    a.update(kw)
    return lib.gattn_decode(a["q"], a["kv"], a["sl"], a["gate"], a["qw"], a["B"], a["H"], a["G"], a["d"], a["L"],
                            a["rd"], a["base"], a["eps"], a["gm"], a["ws"], a["wsb"], a["out"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(kv=None), INVALID),
    (dict(sl=None), INVALID),
    (dict(H=8, G=3), INVALID),
    (dict(L=0), INVALID),
    (dict(rd=7), INVALID),
    (dict(d=96), UNSUPPORTED),
    (dict(H=32, G=2), UNSUPPORTED),      # more than 8 query heads per group
    (dict(B=100000), UNSUPPORTED),
    (dict(rd=40), UNSUPPORTED),
    (dict(kv=P(8)), INVALID),            # cache must be 16-byte aligned for TMA
    (dict(gm=0x12, gate=None), INVALID),  # headwise NS-sigmoid gate without logits
    (dict(gm=0x40), INVALID),            # an activation without a gate
])
def test_decode_rejects_bad_arguments(lib, kw, expect):
    assert decode(lib, **kw) == expect


def decode_noalloc(lib, **kw):
    a = dict(q=P(), kv=P(), sl=P(), gate=P(), qw=P(), B=4, H=8, G=2, d=256, L=1024, rd=64, base=1e7, eps=1e-6, gm=1,
             out=P(1 << 20))
    a.update(kw)
    return lib.gattn_decode_noalloc(a["q"], a["kv"], a["sl"], a["gate"], a["qw"], a["B"], a["H"], a["G"], a["d"],
                                    a["L"], a["rd"], a["base"], a["eps"], a["gm"], a["out"], None)


# The no-allocation decode reports every argument error exactly as gattn_decode
# does, before looking at its scratch limit -- also on shapes far beyond it.
@pytest.mark.parametrize("kw", [
    dict(kv=None), dict(sl=None), dict(q=None), dict(H=8, G=3), dict(L=0), dict(rd=7), dict(d=96),
    dict(H=32, G=2), dict(B=100000), dict(rd=40), dict(kv=P(8)), dict(gm=0x12, gate=None), dict(gm=0x40),
    dict(B=2048, G=8, q=None), dict(B=2048, G=8, rd=7), dict(B=2049, G=8),
])
def test_decode_noalloc_rejects_bad_arguments_like_decode(lib, kw):
    expect = decode(lib, **kw)
    assert expect in (INVALID, UNSUPPORTED)
    assert decode_noalloc(lib, **kw) == expect


def test_selftest_wait_timeout_rejects_bad_limits(lib):
    assert lib.gattn_selftest_wait_timeout(0, None, None) == INVALID
    assert lib.gattn_selftest_wait_timeout(999_999, None, None) == INVALID
    assert lib.gattn_selftest_wait_timeout(100_000_001, None, None) == INVALID


def decode_append(lib, **kw):
    a = dict(q=P(), kn=P(), vn=P(), kv=P(), sl=P(), gate=P(), qw=P(), kw=P(), B=4, H=8, G=2, d=256, L=1024, rd=64,
             base=1e7, eps=1e-6, gm=1, ws=P(), wsb=1 << 40, out=P(1 << 20))
    a.update(kw)
    return lib.gattn_decode_append(a["q"], a["kn"], a["vn"], a["kv"], a["sl"], a["gate"], a["qw"], a["kw"], a["B"],
                                   a["H"], a["G"], a["d"], a["L"], a["rd"], a["base"], a["eps"], a["gm"], a["ws"],
                                   a["wsb"], a["out"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(kn=None), INVALID),
    (dict(vn=None), INVALID),
    (dict(kw=None), INVALID),
    (dict(kn=P(8)), INVALID),            # k_new rows are read 16 bytes at a time
    (dict(kw=P(4)), INVALID),
    (dict(kv=None), INVALID),
    (dict(d=96), UNSUPPORTED),
    (dict(gm=0x40), INVALID),
])
def test_decode_append_rejects_bad_arguments(lib, kw, expect):
    assert decode_append(lib, **kw) == expect


def decode_paged(lib, **kw):
    a = dict(q=P(), kn=None, vn=None, kv=P(), bt=P(), np_=64, ps=256, mp=16, sl=P(), gate=P(), qw=P(), kw=None,
             B=4, H=8, G=2, d=256, rd=64, base=1e7, eps=1e-6, gm=1, ws=P(), wsb=1 << 40, out=P(1 << 20))
    a.update(kw)
    return lib.gattn_decode_paged(a["q"], a["kn"], a["vn"], a["kv"], a["bt"], a["np_"], a["ps"], a["mp"], a["sl"],
                                  a["gate"], a["qw"], a["kw"], a["B"], a["H"], a["G"], a["d"], a["rd"], a["base"],
                                  a["eps"], a["gm"], a["ws"], a["wsb"], a["out"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(bt=None), INVALID),
    (dict(np_=0), INVALID),
    (dict(mp=0), INVALID),
    (dict(ps=96), UNSUPPORTED),          # a key tile would straddle two pages
    (dict(kn=P()), INVALID),             # an append needs v_new and knorm_w too
    (dict(kn=P(), vn=P(), kw=P(8)), INVALID),
    (dict(kv=P(8)), INVALID),
    (dict(d=96), UNSUPPORTED),
    (dict(gm=0x40), INVALID),
])
def test_decode_paged_rejects_bad_arguments(lib, kw, expect):
    assert decode_paged(lib, **kw) == expect


def prefill_varlen(lib, cu, **kw):
    arr = (ctypes.c_int32 * len(cu))(*cu) if cu is not None else None
    a = dict(q=P(), k=P(), v=P(), gate=P(), qw=P(), kw=P(), pos=None, H=8, G=2, d=128, rd=64, base=1e6, eps=1e-6,
             gm=1, qts=0, qhs=0, gts=0, ghs=0, dt=0, ws=P(), wsb=1 << 40, out=P(1 << 20))
    a.update(kw)
    return lib.gattn_prefill_varlen(a["q"], a["k"], a["v"], a["gate"], a["qw"], a["kw"], a["pos"],
                                    ctypes.cast(arr, ctypes.c_void_p) if arr is not None else None,
                                    max(len(cu) - 1, 0) if cu is not None else 1, a["H"], a["G"], a["d"], a["rd"],
                                    a["base"], a["eps"], a["gm"], a["qts"], a["qhs"], a["gts"], a["ghs"], a["dt"],
                                    a["ws"], a["wsb"], a["out"], None)


@pytest.mark.parametrize("cu,kw,expect", [
    (None, {}, INVALID),                  # no cumulative lengths
    ([1, 5], {}, INVALID),                # must start at 0
    ([0, 5, 3], {}, INVALID),             # decreasing
    ([0], {}, INVALID),                   # no sequence
    ([0, 0, 0], {}, OK),                  # only empty sequences: nothing to launch
    ([0, 5, 9], dict(H=6, G=4), INVALID),
    ([0, 5, 9], dict(d=96), UNSUPPORTED),
    ([0, 5, 9], dict(gm=0x40), INVALID),
    ([0, 5, 9], dict(wsb=1024), WORKSPACE),
])
def test_prefill_varlen_rejects_bad_arguments(lib, cu, kw, expect):
    assert prefill_varlen(lib, cu, **kw) == expect


def test_prefill_varlen_workspace_size(lib):
    base = lib.gattn_prefill_workspace_size(1, 1000, 8, 2, 128, 0)
    got = lib.gattn_prefill_varlen_workspace_size(1000, 3, 8, 2, 128, 0)
    tiles = (1000 + 127) // 128 + 3
    rnd = lambda x: (x + 255) // 256 * 256
    assert got == base + rnd(tiles * 16) + 2 * rnd(1000 * 4)
    assert lib.gattn_prefill_varlen_workspace_size(0, 3, 8, 2, 128, 0) == 0


def test_prefill_workspace_sizes(lib):
    assert lib.gattn_prefill_workspace_size(1, 4096, 8, 2, 256, 0) == 4096 * 2 * 256 * 2
    assert lib.gattn_prefill_workspace_size(1, 64, 2, 1, 32, 1) == (64 * 2 * 32 + 64 * 32) * 4
    assert lib.gattn_prefill_workspace_size(0, 64, 2, 1, 32, 1) == 0


def test_flop_accounting_matches_the_causal_triangle():
    # c2, c3, c4 algorithmic FLOPs (QK^T and PV over the causal triangle incl. the diagonal)
    assert prefill_flops(1, 4096, 8, 256) == 68_736_253_952
    assert prefill_flops(8, 2048, 16, 128) == 137_506_062_336
    assert prefill_flops(2, 8192, 32, 128) == 1_099_645_845_504
    # brute force on a tiny case: count multiply-adds of both contractions
    B, S, H, d = 2, 5, 3, 4
    madds = sum(2 * d for b in range(B) for h in range(H) for t in range(S) for j in range(t + 1))
    assert prefill_flops(B, S, H, d) == 2 * madds


@pytest.mark.parametrize("kw", [
    dict(x=None), dict(w=None), dict(y=None), dict(T=0), dict(K=32), dict(K=96), dict(N=0), dict(N=200),
    dict(x=FAKE + 2), dict(w=FAKE + 8), dict(y=FAKE + 4),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_o_proj_rejects_bad_arguments(lib, kw):
    a = dict(x=FAKE, w=FAKE + (1 << 30), T=4096, K=2048, N=1024, y=FAKE + (1 << 31))
    a.update(kw)
    vp = lambda v: None if v is None else ctypes.c_void_p(v)
    assert lib.gattn_o_proj(vp(a["x"]), vp(a["w"]), a["T"], a["K"], a["N"], vp(a["y"]), None) == INVALID
