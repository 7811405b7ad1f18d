"""GPU prefill parity: the CUDA path (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_softmax_attention_gqa_gb300 import (gattn_get_device_status, gattn_o_proj, gattn_prefill, gattn_prefill_varlen,
                                               workloads)
from gated_softmax_attention_gqa_gb300.workloads import WORKLOADS, Workload, make_prefill_inputs
from tests.parity import assert_close_to_oracle, gate_scale, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def run_gpu(inp, w, pos=None, out=None):
    dev = {k: v.to(DEV) for k, v in inp.items()}
    return gattn_prefill(dev["q"], dev["k"], dev["v"], dev["gate"] if w.gate_mode != "none" else None,
                         dev["qnorm_w"], dev["knorm_w"], None if pos is None else pos.to(DEV),
                         rotary_dim=w.rotary_dim, rope_base=w.rope_base, eps=w.eps, gate_mode=w.gate_mode, out=out)


def run_oracle(inp, w, pos=None):
    return oracle.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], inp["qnorm_w"], inp["knorm_w"],
                          None if pos is None else pos.double(), w.rotary_dim, w.rope_base, w.eps, w.gate_mode)


def small(name, B, S, H, G, d, rd, base, gate_mode, dtype="bf16", seed=11, gate_std=1.0):
    return Workload(name, "prefill", B=B, S=S, H=H, G=G, d=d, rotary_dim=rd, rope_base=base, gate_mode=gate_mode,
                    dtype=dtype, seed=seed, gate_std=gate_std)


def test_tiny_fp32_workload_full():
    w = WORKLOADS["tiny_fp32"]
    inp = make_prefill_inputs(w)
    out = run_gpu(inp, w)
    torch.cuda.synchronize()
    ref = run_oracle(inp, w)
    assert_close_to_oracle(out, ref, torch.float32, "tiny fp32")
    assert gattn_get_device_status() == 0


@pytest.mark.parametrize("shape", [
    (1, 1, 2, 1, 32, 8, 1e4, "elementwise"),
    (2, 37, 4, 2, 64, 6, 1e4, "headwise"),
    (1, 130, 2, 2, 128, 128, 1e6, "none"),
    (1, 77, 4, 1, 256, 64, 1e7, "elementwise"),
])
def test_fp32_variants(shape):
    B, S, H, G, d, rd, base, gm = shape
    w = small("f32", B, S, H, G, d, rd, base, gm, dtype="fp32", seed=S)
    inp = make_prefill_inputs(w)
    out = run_gpu(inp, w)
    torch.cuda.synchronize()
    assert_close_to_oracle(out, run_oracle(inp, w), torch.float32, str(shape))


BF16_SHAPES = [
    # B, S, H, G, d, rd, base, gate
    (1, 1, 2, 1, 128, 64, 1e4, "elementwise"),      # single token
    (1, 17, 4, 2, 64, 32, 1e4, "headwise"),         # shorter than one tile
    (2, 129, 8, 2, 256, 64, 1e7, "elementwise"),    # ragged tail, two query tiles, d=256
    (1, 300, 4, 4, 128, 128, 1e6, "headwise"),      # G = H (MHA), full rotary
    (1, 384, 8, 1, 128, 64, 1e6, "none"),           # MQA, no gate, exact tile multiple
    (2, 255, 16, 8, 128, 128, 1e6, "headwise"),     # Qwen3-0.6B head layout
    (1, 513, 4, 1, 256, 64, 1e7, "elementwise"),    # d=256 with 64-key tiles, ragged
    (1, 640, 32, 4, 128, 64, 1e6, "elementwise"),   # paper MoE head layout
    (1, 200, 2, 1, 64, 0, 1e4, "elementwise"),      # no rotary features
    (1, 256, 2, 1, 128, 16, 1e4, "elementwise"),    # small rotary block
]


@pytest.mark.parametrize("shape", BF16_SHAPES, ids=[str(s) for s in BF16_SHAPES])
def test_bf16_parity_small(shape):
    B, S, H, G, d, rd, base, gm = shape
    w = small("bf16", B, S, H, G, d, rd, base, gm, seed=S + d)
    inp = make_prefill_inputs(w)
    out = run_gpu(inp, w)
    torch.cuda.synchronize()
    assert_close_to_oracle(out, run_oracle(inp, w), torch.bfloat16, str(shape))
    assert gattn_get_device_status() == 0


# gate variants ("Gated Attention" deep-dive, section "门放在哪里？" and the NS-sigmoid
# control of section "第二条机制线索") through every prefill kernel: the CTA-pair
# kernel (d 256, H/G even), the one-head kernel at d 128 and at d 256 with H/G odd,
# and the fp32 kernel
GATE_VARIANT_SHAPES = [
    # B, S, H, G, d, rd, base, dtype
    (1, 200, 4, 2, 256, 64, 1e7, "bf16"),
    (2, 150, 4, 2, 128, 64, 1e6, "bf16"),
    (1, 130, 3, 1, 256, 64, 1e7, "bf16"),
    (1, 70, 4, 2, 64, 16, 1e4, "fp32"),
]


@pytest.mark.parametrize("shape", GATE_VARIANT_SHAPES, ids=[str(s) for s in GATE_VARIANT_SHAPES])
def test_gate_variants(shape):
    B, S, H, G, d, rd, base, dt = shape
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    for layout in ("elementwise", "headwise", "head_shared"):
        w = small("gates", B, S, H, G, d, rd, base, layout, dtype=dt, seed=S + d, gate_std=2.0)
        inp = make_prefill_inputs(w)
        dev = {k: v.to(DEV) for k, v in inp.items()}
        for act in ("sigmoid", "ns_sigmoid", "silu"):
            for additive in (False, True):
                out = gattn_prefill(dev["q"], dev["k"], dev["v"], dev["gate"], dev["qnorm_w"], dev["knorm_w"],
                                    rotary_dim=rd, rope_base=base, eps=w.eps, gate_mode=layout, gate_act=act,
                                    gate_additive=additive)
                torch.cuda.synchronize()
                ref = oracle.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], inp["qnorm_w"], inp["knorm_w"],
                                     None, rd, base, w.eps, oracle.gate_code(layout, act, additive))
                assert_close_to_oracle(out, ref, tdt, f"{shape} {layout} {act} additive={additive}",
                                      scale=gate_scale(inp["gate"].double().numpy(), layout, act, ref.shape))
    assert gattn_get_device_status() == 0


# packed variable-length sequences through every prefill kernel: ragged lengths
# (1 token, one short of a tile, exactly a tile, one over, several tiles, empty)
VARLEN_CASES = [
    # H, G, d, rd, base, dtype, gate layout, lengths
    (4, 2, 256, 64, 1e7, "bf16", "elementwise", [1, 127, 128, 129, 300, 0, 77]),   # CTA-pair kernel
    (4, 2, 128, 64, 1e6, "bf16", "headwise", [200, 5, 0, 128, 257]),              # one-head kernel, d 128
    (3, 1, 256, 64, 1e7, "bf16", "head_shared", [130, 64, 1]),                    # one-head kernel, d 256
    (4, 2, 64, 16, 1e4, "fp32", "elementwise", [33, 1, 70, 0, 64]),               # fp32 kernel
]


@pytest.mark.parametrize("case", VARLEN_CASES, ids=[f"{c[5]}-d{c[2]}-{c[6]}" for c in VARLEN_CASES])
def test_varlen_parity(case):
    H, G, d, rd, base, dt, layout, lens = case
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = small("varlen", 1, T, H, G, d, rd, base, layout, dtype=dt, seed=T + d)
    inp = make_prefill_inputs(w)
    flat = {k: (v[0] if k in ("q", "k", "v", "gate") else v) for k, v in inp.items()}
    dev = {k: v.to(DEV) for k, v in flat.items()}
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    out = gattn_prefill_varlen(dev["q"], dev["k"], dev["v"], dev["gate"], dev["qnorm_w"], dev["knorm_w"], cu,
                               rotary_dim=rd, rope_base=base, eps=w.eps, gate_mode=layout)
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    ref = oracle.prefill_varlen(flat["q"], flat["k"], flat["v"], flat["gate"], flat["qnorm_w"], flat["knorm_w"],
                                None, cu, rd, base, w.eps, layout)
    assert_close_to_oracle(out, ref, tdt, str(case))
    # explicit positions: an offset per sequence
    pos = torch.cat([torch.arange(n, dtype=torch.int32) + 1000 * i for i, n in enumerate(lens)])
    out = gattn_prefill_varlen(dev["q"], dev["k"], dev["v"], dev["gate"], dev["qnorm_w"], dev["knorm_w"], cu,
                               pos.to(DEV), rotary_dim=rd, rope_base=base, eps=w.eps, gate_mode=layout)
    torch.cuda.synchronize()
    ref = oracle.prefill_varlen(flat["q"], flat["k"], flat["v"], flat["gate"], flat["qnorm_w"], flat["knorm_w"],
                                pos.double(), cu, rd, base, w.eps, layout)
    assert_close_to_oracle(out, ref, tdt, str(case) + " with positions")


@pytest.mark.parametrize("d,H,G", [(256, 8, 2), (128, 4, 2)])
def test_varlen_equal_lengths_match_the_batched_call(d, H, G):
    """Equal-length packed sequences give exactly the batched result: every query
    tile is computed the same way, only the schedule differs."""
    B, S = 3, 300
    w = small("eq", B, S, H, G, d, 64, 1e6, "elementwise", seed=d)
    inp = make_prefill_inputs(w)
    dev = {k: v.to(DEV) for k, v in inp.items()}
    batched = gattn_prefill(dev["q"], dev["k"], dev["v"], dev["gate"], dev["qnorm_w"], dev["knorm_w"], rotary_dim=64,
                            rope_base=1e6, eps=w.eps, gate_mode="elementwise")
    packed = gattn_prefill_varlen(dev["q"].reshape(B * S, H, d), dev["k"].reshape(B * S, G, d),
                                  dev["v"].reshape(B * S, G, d), dev["gate"].reshape(B * S, H, d), dev["qnorm_w"],
                                  dev["knorm_w"], [0, S, 2 * S, 3 * S], rotary_dim=64, rope_base=1e6, eps=w.eps,
                                  gate_mode="elementwise")
    torch.cuda.synchronize()
    assert torch.equal(packed.view(B, S, H * d), batched)


def test_bf16_packed_qproj_layout_and_positions():
    """q and the gate as the two halves of the packed q_proj output [B,S,H,2d]
    (the handbook's interleaved layout), with explicit RoPE positions."""
    B, S, H, G, d = 2, 200, 8, 2, 128
    w = small("packed", B, S, H, G, d, 64, 1e6, "elementwise", seed=5)
    inp = make_prefill_inputs(w)
    packed = torch.cat([inp["q"], inp["gate"]], dim=-1)  # [B,S,H,2d]
    pos = (torch.arange(S, dtype=torch.int32)[None] * 3 + torch.tensor([[0], [1000]], dtype=torch.int32))
    dev = packed.to(DEV)
    out = gattn_prefill(dev[..., :d], inp["k"].to(DEV), inp["v"].to(DEV), dev[..., d:], inp["qnorm_w"].to(DEV),
                        inp["knorm_w"].to(DEV), pos.to(DEV), rotary_dim=64, rope_base=1e6, gate_mode="elementwise")
    torch.cuda.synchronize()
    ref = run_oracle(inp, w, pos)
    assert_close_to_oracle(out, ref, torch.bfloat16, "packed q_proj")


@pytest.mark.parametrize("name", ["qwen35_08b_prefill", "qwen3_06b_prefill", "paper_moe_prefill"])
def test_bf16_full_size_sampled_rows(name):
    """The benchmark's workloads at full size; the oracle checks a seeded sample of
    query rows (first/last 64, both sides of every tile boundary, 256 random) for
    every batch and head."""
    w = WORKLOADS[name]
    inp = make_prefill_inputs(w)
    out = run_gpu(inp, w)
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    rb, rt = sample_rows(w.S, w.B, seed=w.seed)
    ref = oracle.prefill_rows(inp["q"], inp["k"], inp["v"], inp["gate"], inp["qnorm_w"], inp["knorm_w"], None,
                              w.rotary_dim, w.rope_base, w.eps, w.gate_mode, rb, rt)
    got = out.view(w.B, w.S, -1)[torch.from_numpy(rb).long(), torch.from_numpy(rt).long()]
    assert_close_to_oracle(got, ref, torch.bfloat16, name)
    assert torch.isfinite(out).all()
    # every query row of one whole (batch, head): the last batch, the last head (the
    # last head of the last KV group), computed by the oracle on that head alone
    b, h = w.B - 1, w.H - 1
    g = h // (w.H // w.G)
    one = {"q": inp["q"][b:b + 1, :, h:h + 1], "k": inp["k"][b:b + 1, :, g:g + 1], "v": inp["v"][b:b + 1, :, g:g + 1],
           "gate": inp["gate"][b:b + 1, :, h:h + 1], "qnorm_w": inp["qnorm_w"], "knorm_w": inp["knorm_w"]}
    all_t = np.arange(w.S, dtype=np.int32)
    ref_bh = oracle.prefill_rows(one["q"], one["k"], one["v"], one["gate"], one["qnorm_w"], one["knorm_w"], None,
                                 w.rotary_dim, w.rope_base, w.eps, w.gate_mode, np.zeros_like(all_t), all_t)
    got_bh = out.view(w.B, w.S, w.H, w.d)[b, :, h]
    assert_close_to_oracle(got_bh, ref_bh, torch.bfloat16, f"{name}: every row of batch {b}, head {h}")


def test_every_output_written_and_guard_band_untouched():
    B, S, H, G, d = 1, 333, 4, 2, 128
    w = small("guard", B, S, H, G, d, 64, 1e6, "elementwise", seed=9)
    inp = make_prefill_inputs(w)
    n = B * S * H * d
    buf = torch.full((n + 4096,), float("nan"), dtype=torch.bfloat16, device=DEV)
    buf[n:] = 7.0
    out = buf[:n].view(B, S, H * d)
    run_gpu(inp, w, out=out)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all(), "some output element was never written"
    assert (buf[n:] == 7.0).all(), "kernel wrote past the end of the output"


def test_headwise_gate_equals_broadcast_elementwise():
    B, S, H, G, d = 1, 260, 8, 2, 128
    w = small("hw", B, S, H, G, d, 64, 1e6, "headwise", seed=4)
    inp = make_prefill_inputs(w)
    a = run_gpu(inp, w)
    we = small("ew", B, S, H, G, d, 64, 1e6, "elementwise", seed=4)
    inp_e = dict(inp, gate=inp["gate"][..., None].expand(B, S, H, d).contiguous())
    b = run_gpu(inp_e, we)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_zero_gate_logits_halve_the_ungated_output():
    """sigmoid(0) = 1/2 exactly, and halving commutes with bf16 rounding."""
    B, S, H, G, d = 1, 190, 4, 1, 256
    w = small("z", B, S, H, G, d, 64, 1e7, "elementwise", seed=3)
    inp = make_prefill_inputs(w)
    plain = run_gpu(inp, small("n", B, S, H, G, d, 64, 1e7, "none"))
    half = run_gpu(dict(inp, gate=torch.zeros_like(inp["gate"])), w)
    torch.cuda.synchronize()
    assert torch.equal(half, plain * 0.5)


@pytest.mark.parametrize("d", [128, 256])
def test_gqa_equals_mha_with_replicated_kv(d):
    """Head h reads group floor(h/(H/G)): replicating each group's K and V to its
    H/G heads gives the same output.  G = 2 against G = 4 (both even group sizes,
    so the same kernel computes both) must agree bit for bit; G = H (plain MHA, the
    one-head kernel) is checked against the oracle of the G = 2 problem."""
    B, S, H, G = 1, 150, 8, 2
    w = small("gqa", B, S, H, G, d, 64, 1e6, "elementwise", seed=8)
    inp = make_prefill_inputs(w)
    a = run_gpu(inp, w)

    def replicated(g2):
        rep = g2 // G
        return dict(inp, k=inp["k"].repeat_interleave(rep, dim=2).contiguous(),
                    v=inp["v"].repeat_interleave(rep, dim=2).contiguous())

    b = run_gpu(replicated(4), small("gqa4", B, S, H, 4, d, 64, 1e6, "elementwise"))
    c = run_gpu(replicated(H), small("mha", B, S, H, H, d, 64, 1e6, "elementwise"))
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    ref = run_oracle(inp, w)
    assert_close_to_oracle(a, ref, torch.bfloat16, "G = 2")
    assert_close_to_oracle(c, ref, torch.bfloat16, "G = H with replicated K/V")


def test_rope_rotation_error_bound_at_long_positions():
    """The rotated keys the pre-pass leaves in the workspace (fp32 path) against a
    fp64 rotation by the same fp32 angle pos * inv_freq: checks the kernels' own
    sine/cosine range reduction to ~1e-5 for angles up to 32k rad."""
    B, S, H, G, d, rd, base = 1, 96, 2, 2, 128, 128, 1e4
    w = small("rope", B, S, H, G, d, rd, base, "none", dtype="fp32", seed=12)
    inp = make_prefill_inputs(w)
    pos = torch.randint(0, 32768, (B, S), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    pos[0, :4] = torch.tensor([0, 1, 32767, 31416], dtype=torch.int32)
    from gated_softmax_attention_gqa_gb300 import gattn_prefill_workspace_size

    ws = torch.zeros(gattn_prefill_workspace_size(B, S, H, G, d, torch.float32), dtype=torch.uint8, device=DEV)
    dev = {k: v.to(DEV) for k, v in inp.items()}
    gattn_prefill(dev["q"], dev["k"], dev["v"], None, dev["qnorm_w"], dev["knorm_w"], pos.to(DEV), rotary_dim=rd,
                  rope_base=base, eps=w.eps, gate_mode="none", workspace=ws)
    torch.cuda.synchronize()
    q_bytes = ((B * H * S * d * 4 + 255) // 256) * 256
    kr = ws[q_bytes:q_bytes + B * G * S * d * 4].view(torch.float32).view(B, G, S, d).double().cpu().numpy()
    kn = oracle.rmsnorm(inp["k"], inp["knorm_w"], w.eps)  # [B,S,G,d] fp64
    half = rd // 2
    inv = (base ** (-2.0 * np.arange(half) / rd)).astype(np.float32)
    ang = (pos.numpy().astype(np.float32)[..., None] * inv[None, None, :]).astype(np.float64)  # fp32 product
    c, s = np.cos(ang)[:, :, None, :], np.sin(ang)[:, :, None, :]
    a, b_ = kn[..., :half], kn[..., half:rd]
    ref = np.concatenate([a * c - b_ * s, b_ * c + a * s, kn[..., rd:]], axis=-1).transpose(0, 2, 1, 3)
    err = np.abs(kr - ref)
    assert err.max() < 2e-5, err.max()


@pytest.mark.parametrize("d, H, G", [(256, 8, 2), (128, 4, 2)])
def test_output_feeds_the_o_projection(d, H, G):
    """The gated attention output is handed to the output projection as written: a
    [B*S, H*d] row-major bf16 matrix with the gate already applied, which is where
    the gate sits (between SDPA and W_O: "Gated attention" handbook chapter, "The
    code: qwen/attention.py"; "Gated Attention" deep-dive, "门放在哪里？").  A bf16
    GEMM reads it in place (same storage, no re-layout) and gives the oracle's output
    times W_O^T -- through the library's own tcgen05 projection (gattn_o_proj) and,
    as a cross-check of the handoff alone, through torch's GEMM.  W_O rows have unit
    norm, so an output error e moves each projected value by at most |e|_2 and
    typically by its RMS: the bf16 bounds still apply."""
    B, S, hidden = 2, 200, 512
    w = small("oproj", B, S, H, G, d, 64, 1e6, "elementwise", seed=21)
    inp = make_prefill_inputs(w)
    out = run_gpu(inp, w)
    a = out.view(B * S, H * d)
    assert a.data_ptr() == out.data_ptr() and a.is_contiguous() and a.dtype == torch.bfloat16
    g = torch.Generator().manual_seed(22)
    w_o = torch.randn(hidden, H * d, generator=g, dtype=torch.float64)
    w_o = (w_o / w_o.norm(dim=1, keepdim=True)).to(torch.bfloat16)
    y = gattn_o_proj(a, w_o.to(DEV))
    y_torch = a @ w_o.to(DEV).t()
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    ref = oracle.o_proj(np.asarray(run_oracle(inp, w), dtype=np.float64).reshape(B * S, H * d), w_o)
    assert_close_to_oracle(y, ref, torch.bfloat16, f"o_proj d{d}")
    assert_close_to_oracle(y_torch, ref, torch.bfloat16, f"o_proj d{d} (torch GEMM)")


# More work items than the persistent grids have CTAs (152) or CTA pairs (76), so
# that every CTA walks several items: the next item's Q tile, gate tile and output
# buffer, the tile counters and barrier phases all cross item boundaries, in the
# kernels' second instance (packed sequences and gate variants), with partial tiles
# of packed sequences (stored row by row) between TMA-stored ones.
MULTI_ITEM_VARLEN = [
    # H, G, d, gate layout, act, additive
    (16, 8, 128, "elementwise", "sigmoid", False),  # one-CTA kernel: 28 tiles x 16 heads = 448 items
    (8, 2, 256, "headwise", "ns_sigmoid", False),    # CTA pairs: 28 tiles x 4 head pairs = 112 items
]


@pytest.mark.parametrize("case", MULTI_ITEM_VARLEN, ids=[f"d{c[2]}-{c[3]}" for c in MULTI_ITEM_VARLEN])
def test_varlen_many_items_per_cta(case):
    H, G, d, layout, act, additive = case
    lens = [700, 129, 1, 300, 513, 256, 90, 1024]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = small("varlen_multi", 1, T, H, G, d, 64, 1e6, layout, seed=31 + d)
    inp = make_prefill_inputs(w)
    flat = {k: (v[0] if k in ("q", "k", "v", "gate") else v) for k, v in inp.items()}
    dev = {k: v.to(DEV) for k, v in flat.items()}
    out = gattn_prefill_varlen(dev["q"], dev["k"], dev["v"], dev["gate"], dev["qnorm_w"], dev["knorm_w"], cu,
                               rotary_dim=64, rope_base=1e6, eps=w.eps, gate_mode=layout, gate_act=act,
                               gate_additive=additive)
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    ref = oracle.prefill_varlen(flat["q"], flat["k"], flat["v"], flat["gate"], flat["qnorm_w"], flat["knorm_w"],
                                None, cu, 64, 1e6, w.eps, oracle.gate_code(layout, act, additive))
    assert_close_to_oracle(out, ref, torch.bfloat16, str(case))


@pytest.mark.parametrize("d,H,G,S,layout", [(128, 16, 8, 1280, "head_shared"), (256, 8, 2, 2560, "elementwise")])
def test_gate_variant_many_items_per_cta(d, H, G, S, layout):
    """SiLU, additive: the gate-variant instance with several items per CTA (320 items
    over 152 CTAs at d = 128, 80 over 76 CTA pairs at d = 256); sampled rows."""
    B = 2 if d == 128 else 1
    w = small("gv_multi", B, S, H, G, d, 64, 1e6, layout, seed=41 + d, gate_std=2.0)
    inp = make_prefill_inputs(w)
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = gattn_prefill(dev["q"], dev["k"], dev["v"], dev["gate"], dev["qnorm_w"], dev["knorm_w"], rotary_dim=64,
                        rope_base=1e6, eps=w.eps, gate_mode=layout, gate_act="silu", gate_additive=True)
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    rb, rt = sample_rows(S, B, seed=d, n_random=64, edge=16)
    code = oracle.gate_code(layout, "silu", True)
    ref = oracle.prefill_rows(inp["q"], inp["k"], inp["v"], inp["gate"], inp["qnorm_w"], inp["knorm_w"], None, 64,
                              1e6, w.eps, code, rb, rt)
    got = out.view(B, S, -1)[torch.from_numpy(rb).long(), torch.from_numpy(rt).long()]
    z = inp["gate"].double().numpy()
    zr = z[rb, rt]  # the sampled tokens' logits: [n, H, d] / [n, H] / [n, d]
    assert_close_to_oracle(got, ref, torch.bfloat16, f"d{d} {layout}", scale=gate_scale(zr, layout, "silu", ref.shape))


# The softmax's reference for the exponent: while the logits' bound from the norm
# weights (d max|w_q| max|w_k| log2(e)/sqrt(d), with a 2^-6 margin) is at most 40,
# the one-head kernel subtracts that bound; above it, the running row maximum with
# lazy rescale.  Weights 2.5x the benchmark's put every shape on the running
# maximum, and the larger logits make its rescale run often.
RUNNING_MAX_SHAPES = [
    # B, S, H, G, d, rd, base, gate
    (1, 700, 4, 2, 128, 64, 1e6, "headwise"),      # several items per CTA, ragged
    (2, 300, 2, 1, 64, 32, 1e4, "elementwise"),
    (1, 520, 8, 2, 256, 64, 1e7, "elementwise"),   # CTA-pair kernel
    (1, 260, 3, 1, 256, 64, 1e7, "headwise"),      # one-head kernel at d = 256 (odd H/G)
]


def bf16_operand_reference(inp, w):
    """The oracle's attention on q' = rope(rmsnorm(q)) and k' likewise, each rounded to
    bf16 as the tensor-core contraction takes them: the reference for the kernel's
    own arithmetic once the logits are large enough for the operands' rounding to
    show (an error of a few 2^-9 of |q'||k'| in every logit)."""
    B, S = inp["q"].shape[:2]
    pos = np.broadcast_to(np.arange(S, dtype=np.float64)[None, :, None], (B, S, 1))
    def op(x, wt):
        y = oracle.rope(oracle.rmsnorm(x, wt, w.eps), pos, w.rotary_dim, w.rope_base)
        return torch.from_numpy(y).to(torch.bfloat16).double().numpy()
    return oracle.sdpa_gate(op(inp["q"], inp["qnorm_w"]), op(inp["k"], inp["knorm_w"]), inp["v"], inp["gate"],
                            w.gate_mode)


@pytest.mark.parametrize("shape", RUNNING_MAX_SHAPES, ids=[str(s) for s in RUNNING_MAX_SHAPES])
def test_running_max_path_with_large_norm_weights(shape):
    B, S, H, G, d, rd, base, gm = shape
    w = small("rm", B, S, H, G, d, rd, base, gm, seed=S + 5)
    inp = make_prefill_inputs(w)
    inp["qnorm_w"] = (inp["qnorm_w"].float() * 2.5).to(inp["qnorm_w"].dtype)
    inp["knorm_w"] = (inp["knorm_w"].float() * 2.5).to(inp["knorm_w"].dtype)
    out = run_gpu(inp, w)
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    ref_op = bf16_operand_reference(inp, w)
    assert_close_to_oracle(out, ref_op, torch.bfloat16, f"{shape} against bf16 q', k'")
    # against the exact oracle: no further than the operands' rounding moves it
    exact = run_oracle(inp, w)
    got = out.double().cpu().numpy().reshape(exact.shape)
    assert (np.abs(got - exact) <= np.abs(ref_op - exact) + 2e-2).all(), str(shape)


@pytest.mark.parametrize("d,wn,sign", [(128, 1.55, -1.0), (128, 1.55, 1.0), (64, 1.8, -1.0), (256, 1.3, -1.0)])
def test_logits_at_the_fixed_bound(d, wn, sign):
    """Constant q and k = sign * q with constant norm weights wn, no rotary part: every
    logit equals sign * d wn^2 / sqrt(d), within 2% of the bound (just under 40 in
    log2 units for d <= 128), so with sign = -1 every P of a row is about 2^-79.  The
    softmax is uniform either way: out_t = the mean of v_0..v_t (no gate)."""
    B, S, H, G = 1, 300, 2, 1
    w = small("bound", B, S, H, G, d, 0, 1e4, "none", seed=d)
    inp = make_prefill_inputs(w)
    inp["q"] = torch.full_like(inp["q"], 0.75)
    inp["k"] = torch.full_like(inp["k"], 0.75 * sign)
    inp["qnorm_w"] = torch.full_like(inp["qnorm_w"], wn)
    inp["knorm_w"] = torch.full_like(inp["knorm_w"], wn)
    out = run_gpu(inp, w)
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    v = inp["v"][0, :, 0].double()                                   # [S, d]
    mean = torch.cumsum(v, 0) / torch.arange(1, S + 1, dtype=torch.float64)[:, None]
    want = mean[:, None, :].expand(S, H, d).reshape(1, S, H * d)
    assert_close_to_oracle(out, want.numpy(), torch.bfloat16, f"d={d} sign={sign}")
    assert_close_to_oracle(out, run_oracle(inp, w), torch.bfloat16, f"d={d} sign={sign} oracle")
