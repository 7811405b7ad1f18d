"""GPU decode parity: split-KV decode (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_softmax_attention_gqa_gb300 import (gattn_decode, gattn_decode_append, gattn_decode_paged,
                                              gattn_get_device_status, gattn_prefill)
from gated_softmax_attention_gqa_gb300.workloads import WORKLOADS, Workload, make_decode_inputs, make_prefill_inputs
from tests.parity import assert_close_to_oracle, gate_scale

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BAD_SEQLEN = 0x1


def dec_workload(B, H, G, d, rd, base, gate_mode, Lmax, lo, hi, seed):
    return Workload("dec", "decode", B=B, H=H, G=G, d=d, rotary_dim=rd, rope_base=base, gate_mode=gate_mode,
                    dtype="bf16", seed=seed, Lmax=Lmax, seqlen_range=(lo, hi))


def run_gpu(inp, w, out=None):
    dev = {k: v.to(DEV) for k, v in inp.items()}
    return gattn_decode(dev["q_new"], dev["kv_cache"], dev["seqlens"],
                        dev["gate"] if w.gate_mode != "none" else None, dev["qnorm_w"], rotary_dim=w.rotary_dim,
                        rope_base=w.rope_base, eps=w.eps, gate_mode=w.gate_mode, out=out)


def run_oracle(inp, w, rows=None):
    idx = slice(None) if rows is None else rows
    cache = inp["kv_cache"]
    sl = inp["seqlens"][idx]
    lmax = int(sl.max())
    return oracle.decode(inp["q_new"][idx], cache[0][idx][:, :, :lmax], cache[1][idx][:, :, :lmax], sl,
                         inp["gate"][idx], inp["qnorm_w"], w.rotary_dim, w.rope_base, w.eps, w.gate_mode)


SHAPES = [
    # B, H, G, d, rd, base, gate, Lmax, lo, hi
    (3, 8, 2, 256, 64, 1e7, "elementwise", 300, 1, 300),
    (5, 16, 8, 128, 128, 1e6, "headwise", 700, 1, 700),
    (4, 32, 4, 128, 64, 1e6, "elementwise", 1000, 500, 1000),
    (2, 4, 4, 64, 32, 1e4, "none", 129, 63, 129),
    (7, 8, 1, 128, 16, 1e4, "elementwise", 2048, 1, 2048),
    # one long sequence spread over most of the grid: its merge takes some 300 partial
    # states, eight at a time, each group with its own maximum
    (1, 8, 2, 256, 64, 1e7, "elementwise", 8192, 8192, 8192),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_decode_parity_small(shape):
    B, H, G, d, rd, base, gm, Lmax, lo, hi = shape
    w = dec_workload(B, H, G, d, rd, base, gm, Lmax, lo, hi, seed=B * 100 + d)
    inp = make_decode_inputs(w)
    out = run_gpu(inp, w)
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    assert_close_to_oracle(out, run_oracle(inp, w), torch.bfloat16, str(shape))


@pytest.mark.parametrize("shape", [(3, 8, 2, 256, 64, 1e7, 300, 1, 300), (4, 16, 8, 128, 128, 1e6, 500, 100, 500)],
                         ids=["d256", "d128"])
def test_decode_gate_variants(shape):
    """Head-shared logits, NS-sigmoid, SiLU and the additive gate ("Gated Attention"
    deep-dive, sections "门放在哪里？" and "第二条机制线索") in the decode combine."""
    B, H, G, d, rd, base, Lmax, lo, hi = shape
    for layout in ("elementwise", "headwise", "head_shared"):
        w = dec_workload(B, H, G, d, rd, base, layout, Lmax, lo, hi, seed=B * 10 + d)
        inp = make_decode_inputs(w)
        dev = {k: v.to(DEV) for k, v in inp.items()}
        lmax = int(inp["seqlens"].max())
        for act in ("sigmoid", "ns_sigmoid", "silu"):
            for additive in (False, True):
                out = gattn_decode(dev["q_new"], dev["kv_cache"], dev["seqlens"], dev["gate"], dev["qnorm_w"],
                                   rotary_dim=rd, rope_base=base, eps=w.eps, gate_mode=layout, gate_act=act,
                                   gate_additive=additive)
                torch.cuda.synchronize()
                ref = oracle.decode(inp["q_new"], inp["kv_cache"][0][:, :, :lmax], inp["kv_cache"][1][:, :, :lmax],
                                    inp["seqlens"], inp["gate"], inp["qnorm_w"], rd, base, w.eps,
                                    oracle.gate_code(layout, act, additive))
                assert_close_to_oracle(out, ref, torch.bfloat16, f"{shape} {layout} {act} additive={additive}",
                                      scale=gate_scale(inp["gate"].double().numpy(), layout, act, ref.shape))
    assert gattn_get_device_status() == 0


@pytest.mark.parametrize("shape", [(3, 8, 2, 256, 64, 1e7, 300, 1, 300), (5, 16, 8, 128, 128, 1e6, 700, 1, 700),
                                   (4, 4, 4, 64, 32, 1e4, 129, 63, 129)], ids=["d256", "d128", "d64"])
def test_decode_append_parity(shape):
    """The new token's K (normed, rotated at seqlens-1) and V written into the cache
    inside the call, then the step: output and cache against the oracle."""
    B, H, G, d, rd, base, Lmax, lo, hi = shape
    w = dec_workload(B, H, G, d, rd, base, "elementwise", Lmax, lo, hi, seed=B * 7 + d)
    inp = make_decode_inputs(w)
    g = torch.Generator().manual_seed(B + d)
    k_new = torch.randn((B, G, d), generator=g).to(torch.bfloat16)
    v_new = torch.randn((B, G, d), generator=g).to(torch.bfloat16)
    knorm_w = (1 + 0.1 * torch.randn((d,), generator=g)).to(torch.bfloat16)
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = gattn_decode_append(dev["q_new"], k_new.to(DEV), v_new.to(DEV), dev["kv_cache"], dev["seqlens"],
                              dev["gate"], dev["qnorm_w"], knorm_w.to(DEV), rotary_dim=rd, rope_base=base, eps=w.eps)
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    ref, kc, vc = oracle.decode_append(inp["q_new"], k_new, v_new, inp["kv_cache"][0], inp["kv_cache"][1],
                                       inp["seqlens"], inp["gate"], inp["qnorm_w"], knorm_w, rd, base, w.eps,
                                       "elementwise")
    assert_close_to_oracle(out, ref, torch.bfloat16, f"{shape} out")
    cache = dev["kv_cache"].cpu()
    for b in range(B):
        L = int(inp["seqlens"][b])
        assert_close_to_oracle(cache[0, b, :, L - 1], kc[b, :, L - 1], torch.bfloat16, f"{shape} K row of {b}")
        assert torch.equal(cache[1, b, :, L - 1], v_new[b]), f"V row of sequence {b}"
        assert torch.equal(cache[:, b, :, :L - 1], inp["kv_cache"][:, b, :, :L - 1]), f"earlier rows of {b}"


@pytest.mark.parametrize("shape", [(3, 8, 2, 256, 64, 1e7, 128, 4), (5, 16, 8, 128, 128, 1e6, 64, 12),
                                   (2, 4, 1, 64, 32, 1e4, 192, 3)], ids=["d256p128", "d128p64", "d64p192"])
def test_decode_paged_parity(shape):
    """The cache scattered over a shuffled page pool (with spare pages holding
    NaN): the paged step must match the oracle on the contiguous cache, with and
    without appending the new token."""
    B, H, G, d, rd, base, ps, mp = shape
    Lmax = ps * mp
    w = dec_workload(B, H, G, d, rd, base, "elementwise", Lmax, 1, Lmax, seed=B * 13 + d)
    inp = make_decode_inputs(w)
    g = torch.Generator().manual_seed(d + ps)
    num_pages = B * mp + 3
    table = torch.randperm(num_pages, generator=g)[:B * mp].view(B, mp).to(torch.int32)
    pool = torch.full((2, num_pages, G, ps, d), float("nan"), dtype=torch.bfloat16)
    for b in range(B):
        for j in range(mp):
            pool[:, table[b, j]] = inp["kv_cache"][:, b, :, j * ps:(j + 1) * ps]
    dev = {k: v.to(DEV) for k, v in inp.items()}
    pool_d, table_d = pool.to(DEV), table.to(DEV)
    out = gattn_decode_paged(dev["q_new"], pool_d, table_d, dev["seqlens"], dev["gate"], dev["qnorm_w"],
                             rotary_dim=rd, rope_base=base, eps=w.eps)
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    assert_close_to_oracle(out, run_oracle(inp, w), torch.bfloat16, f"{shape} paged")
    # with the new token appended into its page
    k_new = torch.randn((B, G, d), generator=g).to(torch.bfloat16)
    v_new = torch.randn((B, G, d), generator=g).to(torch.bfloat16)
    knorm_w = (1 + 0.1 * torch.randn((d,), generator=g)).to(torch.bfloat16)
    out = gattn_decode_paged(dev["q_new"], pool_d, table_d, dev["seqlens"], dev["gate"], dev["qnorm_w"],
                             rotary_dim=rd, rope_base=base, eps=w.eps, k_new=k_new.to(DEV), v_new=v_new.to(DEV),
                             knorm_w=knorm_w.to(DEV))
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    ref, kc, _ = oracle.decode_append(inp["q_new"], k_new, v_new, inp["kv_cache"][0], inp["kv_cache"][1],
                                      inp["seqlens"], inp["gate"], inp["qnorm_w"], knorm_w, rd, base, w.eps,
                                      "elementwise")
    assert_close_to_oracle(out, ref, torch.bfloat16, f"{shape} paged + append")
    pool_after = pool_d.cpu()
    for b in range(B):
        L = int(inp["seqlens"][b])
        page, row = int(table[b, (L - 1) // ps]), (L - 1) % ps
        assert_close_to_oracle(pool_after[0, page, :, row], kc[b, :, L - 1], torch.bfloat16, f"K row of {b}")
        assert torch.equal(pool_after[1, page, :, row], v_new[b])


def test_decode_ignores_cache_entries_past_each_sequence():
    """Tokens at or after seqlens[b] may hold anything, NaN included."""
    w = dec_workload(4, 8, 2, 256, 64, 1e7, "elementwise", 512, 1, 500, seed=21)
    inp = make_decode_inputs(w)
    poisoned = inp["kv_cache"].clone()
    for b, L in enumerate(inp["seqlens"].tolist()):
        poisoned[:, b, :, L:] = float("nan")
    out = run_gpu(dict(inp, kv_cache=poisoned), w)
    torch.cuda.synchronize()
    assert_close_to_oracle(out, run_oracle(inp, w), torch.bfloat16, "poisoned tail")


def test_decode_full_size_every_sequence():
    """The benchmark's decode workload at full size (64 sequences, 16k-32k cached
    tokens), every sequence and head against the oracle: the split kernel cuts the
    global tile list at arbitrary points, so each sequence is split differently."""
    w = WORKLOADS["qwen35_08b_decode"]
    inp = make_decode_inputs(w)
    out = run_gpu(inp, w)
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    for b0 in range(0, w.B, 8):  # eight sequences at a time keeps the fp64 copies near 1 GB
        rows = torch.arange(b0, min(b0 + 8, w.B))
        ref = run_oracle(inp, w, rows=rows)
        assert_close_to_oracle(out[rows], ref, torch.bfloat16, f"decode full size, sequences {b0}..{b0 + 7}")


def test_decode_equals_last_prefill_row():
    """Decode with a cache holding the normed, rotated keys of a prefix equals row
    L-1 of prefill over that prefix (both computed on the GPU)."""
    H, G, d, rd, base, eps = 8, 2, 256, 64, 1e7, 1e-6
    wp = Workload("p", "prefill", B=1, S=700, H=H, G=G, d=d, rotary_dim=rd, rope_base=base,
                  gate_mode="elementwise", dtype="bf16", seed=31)
    inp = make_prefill_inputs(wp)
    dev = {k: v.to(DEV) for k, v in inp.items()}
    full = gattn_prefill(dev["q"], dev["k"], dev["v"], dev["gate"], dev["qnorm_w"], dev["knorm_w"], rotary_dim=rd,
                         rope_base=base, eps=eps, gate_mode="elementwise").view(1, wp.S, H * d)
    lens = [1, 128, 129, 700]
    Lmax = 704
    kn = oracle.rmsnorm(inp["k"][0], inp["knorm_w"], eps)
    kr = oracle.rope(kn, np.arange(wp.S)[:, None], rd, base)  # [S,G,d]
    cache = torch.zeros((2, len(lens), G, Lmax, d), dtype=torch.bfloat16)
    for i, L in enumerate(lens):
        cache[0, i, :, :L] = torch.from_numpy(kr[:L]).permute(1, 0, 2).to(torch.bfloat16)
        cache[1, i, :, :L] = inp["v"][0, :L].permute(1, 0, 2)
    q_new = torch.stack([inp["q"][0, L - 1] for L in lens])
    gate = torch.stack([inp["gate"][0, L - 1] for L in lens])
    out = gattn_decode(q_new.to(DEV), cache.to(DEV), torch.tensor(lens, dtype=torch.int32, device=DEV),
                       gate.to(DEV), dev["qnorm_w"], rotary_dim=rd, rope_base=base, eps=eps)
    torch.cuda.synchronize()
    for i, L in enumerate(lens):
        diff = (out[i].double() - full[0, L - 1].double()).abs()
        assert diff.max().item() <= 2e-2 and diff.mean().item() <= 2e-3, (L, diff.max().item())


def test_bad_seqlen_is_reported_and_skipped():
    w = dec_workload(4, 8, 2, 128, 64, 1e6, "elementwise", 256, 10, 256, seed=41)
    inp = make_decode_inputs(w)
    sl = inp["seqlens"].clone()
    sl[1] = 0
    sl[2] = 257  # beyond Lmax
    bad = dict(inp, seqlens=sl)
    out = torch.full((4, 8 * 128), 3.0, dtype=torch.bfloat16, device=DEV)
    gattn_get_device_status()
    run_gpu(bad, w, out=out)
    torch.cuda.synchronize()
    assert gattn_get_device_status() & BAD_SEQLEN
    assert (out[1] == 3.0).all() and (out[2] == 3.0).all()
    good = torch.tensor([0, 3])
    ref = run_oracle(inp, w, rows=good)
    assert_close_to_oracle(out[good], ref, torch.bfloat16, "good rows next to bad ones")
    assert gattn_get_device_status() == 0
