"""Seeded synthetic workloads and work accounting.

This module holds no step of the attention computation: only input generators
(seeded CPU random numbers in the library's layouts) and the counting of
algorithmic FLOPs and bytes used by the benchmark.  Tests, the smoke check and
the benchmark draw their inputs from here, so the GPU path and the fp64 oracle
always see the same bf16-rounded (or fp32) values.

Shapes follow the models on the source pages: the Qwen3.5-0.8B full-attention
layer (8 query heads, 2 KV groups, head_dim 256, 64 rotary features), the
Qwen3-0.6B layer (16/8 heads, head_dim 128) and the gated-attention paper's MoE
attention (32 query / 4 KV heads, head_dim 128).  No public dataset is used.
"""
from dataclasses import dataclass, field
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "prefill" | "decode"
    B: int
    H: int
    G: int
    d: int
    rotary_dim: int
    rope_base: float
    gate_mode: str  # "elementwise" | "headwise" | "head_shared" | "none"
    dtype: str  # "bf16" | "fp32"
    seed: int
    S: int = 0  # prefill tokens per sequence
    Lmax: int = 0  # decode cache capacity
    seqlen_range: Tuple[int, int] = (0, 0)  # decode: inclusive uniform range
    gate_std: float = 1.0
    eps: float = 1e-6
    description: str = field(default="", compare=False)


WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", "prefill", B=1, S=64, H=2, G=1, d=32, rotary_dim=8, rope_base=1e4,
        gate_mode="elementwise", dtype="fp32", seed=0,
        description="tiny fp32 check: B1 S64 H2 G1 d32 rd8 base 1e4"),
    "qwen35_08b_prefill": Workload(
        "qwen35_08b_prefill", "prefill", B=1, S=4096, H=8, G=2, d=256, rotary_dim=64, rope_base=1e7,
        gate_mode="elementwise", dtype="bf16", seed=1,
        description="Qwen3.5-0.8B-shaped full-attention prefill: B1 S4096 H8 G2 d256 rd64 base 1e7"),
    "qwen3_06b_prefill": Workload(
        "qwen3_06b_prefill", "prefill", B=8, S=2048, H=16, G=8, d=128, rotary_dim=128, rope_base=1e6,
        gate_mode="headwise", dtype="bf16", seed=2,
        description="Qwen3-0.6B-shaped prefill, headwise gate: B8 S2048 H16 G8 d128 rd128 base 1e6"),
    "paper_moe_prefill": Workload(
        "paper_moe_prefill", "prefill", B=2, S=8192, H=32, G=4, d=128, rotary_dim=64, rope_base=1e6,
        gate_mode="elementwise", dtype="bf16", seed=3, gate_std=2.0,
        description="gated-attention paper MoE-shaped long prefill: B2 S8192 H32 G4 d128 rd64 base 1e6"),
    "qwen35_08b_decode": Workload(
        "qwen35_08b_decode", "decode", B=64, H=8, G=2, d=256, rotary_dim=64, rope_base=1e7,
        gate_mode="elementwise", dtype="bf16", seed=5, Lmax=32768, seqlen_range=(16384, 32768),
        description="decode against a bf16 KV cache: B64 H8 G2 d256 rd64, lengths U[16384,32768]"),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def _randn(gen, shape, dtype, std=1.0, chunk=1 << 26):
    """fp32 N(0, std^2) draws rounded once to `dtype`, generated in chunks so that
    multi-GB bf16 tensors never need a full fp32 copy."""
    out = torch.empty(shape, dtype=dtype)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        x = torch.randn(n, generator=gen, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[s:s + n] = x.to(dtype)
    return out


def make_prefill_inputs(w: Workload, S: Optional[int] = None, B: Optional[int] = None, seed: Optional[int] = None):
    """Tensors (CPU) in the library layout, drawn in the fixed order
    q, k, v, gate, qnorm_w, knorm_w:
      q [B,S,H,d]  k,v [B,S,G,d]  gate [B,S,H,d], [B,S,H] or [B,S,d] (head-shared)
      norm weights [d] = 1 + 0.1 N(0,1)."""
    S = w.S if S is None else S
    B = w.B if B is None else B
    g = torch.Generator("cpu").manual_seed(w.seed if seed is None else seed)
    dt = torch_dtype(w.dtype)
    q = _randn(g, (B, S, w.H, w.d), dt)
    k = _randn(g, (B, S, w.G, w.d), dt)
    v = _randn(g, (B, S, w.G, w.d), dt)
    gshape = {"elementwise": (B, S, w.H, w.d), "head_shared": (B, S, w.d)}.get(w.gate_mode, (B, S, w.H))
    gate = _randn(g, gshape, dt, std=w.gate_std)
    qw = (1.0 + 0.1 * torch.randn(w.d, generator=g)).to(dt)
    kw = (1.0 + 0.1 * torch.randn(w.d, generator=g)).to(dt)
    return {"q": q, "k": k, "v": v, "gate": gate, "qnorm_w": qw, "knorm_w": kw}


def make_decode_inputs(w: Workload, B: Optional[int] = None, Lmax: Optional[int] = None,
                       seqlen_range: Optional[Tuple[int, int]] = None, seed: Optional[int] = None):
    """Tensors (CPU) drawn in the order seqlens, kv_cache, q_new, gate, qnorm_w:
      seqlens [B] int32 uniform in the inclusive range; kv_cache [2,B,G,Lmax,d]
      (plane 0 = K, already normed and rotated; plane 1 = V); q_new [B,H,d];
      gate [B,H,d], [B,H] or [B,d] (head-shared); qnorm_w [d]."""
    B = w.B if B is None else B
    Lmax = w.Lmax if Lmax is None else Lmax
    lo, hi = w.seqlen_range if seqlen_range is None else seqlen_range
    g = torch.Generator("cpu").manual_seed(w.seed if seed is None else seed)
    dt = torch_dtype(w.dtype)
    seqlens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    cache = _randn(g, (2, B, w.G, Lmax, w.d), dt)
    q = _randn(g, (B, w.H, w.d), dt)
    gshape = {"elementwise": (B, w.H, w.d), "head_shared": (B, w.d)}.get(w.gate_mode, (B, w.H))
    gate = _randn(g, gshape, dt, std=w.gate_std)
    qw = (1.0 + 0.1 * torch.randn(w.d, generator=g)).to(dt)
    return {"seqlens": seqlens, "kv_cache": cache, "q_new": q, "gate": gate, "qnorm_w": qw}


# ---------------------------------------------------------------- work accounting

def prefill_flops(B: int, S: int, H: int, d: int) -> int:
    """Algorithmic FLOPs of causal prefill: QK^T and PV over the causal triangle
    including the diagonal (2 FLOPs per multiply-add, two contractions)."""
    return 4 * B * H * d * S * (S + 1) // 2


def prefill_io_bytes(B: int, S: int, H: int, G: int, d: int, gate_mode: str, elt: int = 2) -> int:
    """Compulsory HBM bytes of prefill: q, k, v, gate read once; output written once."""
    gate = B * S * H * (d if gate_mode == "elementwise" else 1 if gate_mode == "headwise" else 0)
    return elt * (B * S * H * d + 2 * B * S * G * d + gate + B * S * H * d)


def kv_numbers_per_token(kv_heads: int, d: int) -> int:
    """Numbers one token adds to one layer's KV cache: a key and a value per KV head."""
    return 2 * kv_heads * d


def decode_kv_bytes(seqlens, kv_heads: int, d: int, bytes_per_number: int = 2) -> int:
    """Bytes of K and V one decode step must read: every cached token of every sequence."""
    return int(sum(int(L) for L in seqlens)) * kv_numbers_per_token(kv_heads, d) * bytes_per_number


def decode_io_bytes(seqlens, H: int, G: int, d: int, gate_mode: str, elt: int = 2) -> int:
    """Algorithmic bytes of a decode step: the K/V cache read plus q, gate in and out."""
    B = len(seqlens)
    gate = B * H * (d if gate_mode == "elementwise" else 1 if gate_mode == "headwise" else 0)
    return decode_kv_bytes(seqlens, G, d, elt) + elt * (2 * B * H * d + gate)


def decode_flops(seqlens, H: int, d: int) -> int:
    return 4 * H * d * int(sum(int(L) for L in seqlens))
