"""Shared helpers for the GPU parity tests: tolerances and comparisons."""
import numpy as np
import torch

# Tolerances against the fp64 oracle on the same bf16-rounded (or fp32) inputs.
BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3
FP32_MAX_ABS = 1e-4


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close_to_oracle(gpu, ref, dtype, what="", scale=None):
    """Max- and mean-abs error bounds against the oracle.  The bounds are set for
    a gate of at most 1 in magnitude (sigmoid); a gate that can exceed it (SiLU
    reaches |z|) multiplies the error of the attention output it scales, and the
    output's own bf16 rounding grows with it.  `scale` (broadcastable to the
    output, >= 1) then divides the error: max(1, |gate activation|, |ref|)."""
    g = to_np(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    diff = np.abs(g - ref)
    if scale is not None:
        diff = diff / np.maximum(np.maximum(1.0, np.abs(ref)), np.asarray(scale, dtype=np.float64))
    if dtype == torch.float32:
        assert diff.max() <= FP32_MAX_ABS, f"{what}: max abs {diff.max():.3e} > {FP32_MAX_ABS}"
    else:
        assert diff.max() <= BF16_MAX_ABS, f"{what}: max abs {diff.max():.3e} > {BF16_MAX_ABS}"
        assert diff.mean() <= BF16_MEAN_ABS, f"{what}: mean abs {diff.mean():.3e} > {BF16_MEAN_ABS}"
    return float(diff.max()), float(diff.mean())


def gate_scale(z, layout, act, shape):
    """|act(z)| of every output element of a [B,S,H*d] (or [B,H*d]) output, from the
    oracle's activation, for assert_close_to_oracle's `scale`."""
    import oracle
    z = np.asarray(z, dtype=np.float64)
    a = np.abs(np.vectorize(lambda x: oracle.gate_act(x, act))(z))
    *lead, hd = shape
    if layout == "elementwise":
        return a.reshape(*lead, hd)
    if layout == "headwise":  # [.., H] -> every dimension of head h
        return np.repeat(a, hd // a.shape[-1], axis=-1).reshape(*lead, hd)
    return np.tile(a, hd // a.shape[-1]).reshape(*lead, hd)  # head-shared [.., d] -> every head


def sample_rows(S, B, seed, n_random=256, edge=64, tile=128):
    """Query rows to check at full size: the first and last `edge` rows, every
    row on either side of a tile boundary, and `n_random` seeded random rows,
    for every batch."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(edge, S))) | set(range(max(0, S - edge), S))
    for t0 in range(tile, S, tile):
        rows |= {t0 - 1, t0}
    rows |= set(rng.integers(0, S, size=n_random).tolist())
    ts = sorted(rows)
    rb = [b for b in range(B) for _ in ts]
    rt = [t for _ in range(B) for t in ts]
    return np.array(rb, dtype=np.int32), np.array(rt, dtype=np.int32)
