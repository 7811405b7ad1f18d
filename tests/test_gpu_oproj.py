"""GPU parity of the output projection y = x W_O^T (gattn_o_proj, tcgen05) against
the fp64 oracle: every tile width (256, 128 and 64 output columns per tile), ragged
row counts, a single row, more tiles than CTAs (both TMEM accumulators in turn),
and the Qwen3.5-0.8B-shaped projection of the benchmark's prefill output."""
import numpy as np
import pytest
import torch

import oracle
from gated_softmax_attention_gqa_gb300 import gattn_get_device_status, gattn_o_proj
from tests.parity import assert_close_to_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

SHAPES = [
    # T, K, N
    (1, 64, 64),          # one row, one slice, 64-column tiles
    (300, 512, 192),      # ragged rows, 64-column tiles
    (129, 1024, 384),     # one row into a second tile row, 128-column tiles
    (4096, 2048, 1024),   # Qwen3.5-0.8B: [T, H*d] = [4096, 2048] -> hidden 1024
    (10000, 256, 2048),   # 632 tiles: several per CTA, both accumulators reused
    (200, 4096, 2048),    # paper-MoE head layout: H*d = 4096
]


def inputs(T, K, N, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16)  # outputs ~ N(0, 1)
    return x, w


@pytest.mark.parametrize("shape", SHAPES, ids=[f"T{s[0]}-K{s[1]}-N{s[2]}" for s in SHAPES])
def test_o_proj_matches_the_oracle(shape):
    T, K, N = shape
    x, w = inputs(T, K, N, seed=T + K + N)
    y = gattn_o_proj(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    assert gattn_get_device_status() == 0
    assert y.shape == (T, N) and y.dtype == torch.bfloat16
    assert_close_to_oracle(y, oracle.o_proj(x, w), torch.bfloat16, str(shape))


def test_o_proj_keeps_leading_dimensions_and_writes_only_its_output():
    B, S, K, N = 2, 77, 512, 256
    x, w = inputs(B * S, K, N, seed=5)
    buf = torch.full((B * S * N + 4096,), 7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[:B * S * N].view(B, S, N)
    y = gattn_o_proj(x.view(B, S, K).to(DEV), w.to(DEV), out=out)
    torch.cuda.synchronize()
    assert y.data_ptr() == out.data_ptr()
    assert (buf[B * S * N:] == 7.0).all(), "wrote past the output"
    assert_close_to_oracle(y.view(B * S, N), oracle.o_proj(x, w), torch.bfloat16, "[B,S,K]")


def test_o_proj_rejects_sizes_it_does_not_tile():
    x = torch.zeros(4, 100, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(Exception):
        gattn_o_proj(x, torch.zeros(64, 100, dtype=torch.bfloat16, device=DEV))
