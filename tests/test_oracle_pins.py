"""Pins for the fp64 oracle: the pages' worked examples, closed forms of the
mathematics, and special cases that reduce to library routines.

None of these compares the oracle with a retyped copy of itself: every expected
value is either printed on a source page (tests/golden/, with its citation), a
closed form, or the output of an independent library routine (torch).
"""
import math

import numpy as np
import pytest
import torch

import oracle


def r(x, n):
    return np.round(np.asarray(x, dtype=np.float64), n)


# ---------------------------------------------------------------- worked examples

def _three_token_inputs(g, queries):
    """Lay the page's 2-d toy out as B=1, S=3, H=G=1, d=2 (already "normed")."""
    q = np.array(queries, dtype=np.float64).reshape(1, 3, 1, 2)
    k = np.array(g["keys"]).reshape(1, 3, 1, 2)
    v = np.array(g["values"]).reshape(1, 3, 1, 2)
    return q, k, v


def test_three_token_example_weights_and_output(golden):
    g = golden("handbook_three_tokens.json")
    queries = [[0.0, 0.0], [0.0, 0.0], g["query_last_token"]]
    q, k, v = _three_token_inputs(g, queries)
    out, attn = oracle.sdpa_gate(q, k, v, None, "none", want_attn=True)
    w = attn[0, 0, 2]
    np.testing.assert_array_equal(r(w, 3), g["expected_weights_3dp"])
    assert r(w.sum(), 3) == 1.0
    np.testing.assert_array_equal(r(out[0, 2], 3), g["expected_out_3dp"])
    # the printed scores are the logits: log of the weight ratios recovers them
    scores = np.log(w / w[0]) + 0.0
    np.testing.assert_array_equal(r(scores, 2), g["expected_scores_2dp"])


def test_three_token_causal_matrix(golden):
    g = golden("handbook_three_tokens.json")
    q, k, v = _three_token_inputs(g, g["causal_queries"])
    _, attn = oracle.sdpa_gate(q, k, v, None, "none", want_attn=True)
    np.testing.assert_array_equal(r(attn[0, 0], 3), g["expected_causal_rows_3dp"])
    # entries above the diagonal are exactly zero (masked -inf -> weight 0)
    assert attn[0, 0, 0, 1] == 0.0 and attn[0, 0, 0, 2] == 0.0 and attn[0, 0, 1, 2] == 0.0


def test_zero_query_uniform_row_and_closing_gate(golden):
    g = golden("handbook_three_tokens.json")
    q, k, v = _three_token_inputs(g, [[0.0, 0.0], [0.0, 0.0], [0.0, 0.0]])
    out, attn = oracle.sdpa_gate(q, k, v, None, "none", want_attn=True)
    np.testing.assert_array_equal(r(attn[0, 0, 2], 3), g["zero_query_expected_weights_3dp"])
    np.testing.assert_array_equal(r(out[0, 2], 3), g["zero_query_expected_out_3dp"])
    z = np.full((1, 3, 1, 2), g["gate_logit"])
    gated = oracle.sdpa_gate(q, k, v, z, "elementwise")
    assert round(oracle.sigmoid(g["gate_logit"]), 4) == g["expected_gate_4dp"]
    np.testing.assert_array_equal(r(gated[0, 2], 4), g["expected_gated_out_4dp"])


def test_two_by_two_known_answer(golden):
    g = golden("worked_2x2_causal.json")
    q = np.array(g["Q"]).reshape(1, 2, 1, 2)
    k = np.array(g["K"]).reshape(1, 2, 1, 2)
    v = np.array(g["V"]).reshape(1, 2, 1, 2)
    out, attn = oracle.sdpa_gate(q, k, v, None, "none", want_attn=True)
    np.testing.assert_allclose(attn[0, 0], g["expected_A_8sig"], rtol=5e-8, atol=0)
    np.testing.assert_allclose(out[0], g["expected_O_8sig"], rtol=5e-8, atol=0)
    assert attn[0, 0, 0, 1] == 0.0 and out[0, 0, 1] == 0.0  # t=0 reads v0 only


def test_sigmoid_table(golden):
    g = golden("handbook_gate_toy.json")
    for z, expect in g["sigmoid_table_4dp"].items():
        assert round(oracle.sigmoid(float(z)), 4) == expect
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.sigmoid(-800.0) == 0.0 and oracle.sigmoid(800.0) == 1.0  # no overflow on either side
    for z in (-7.3, -0.2, 0.9, 12.0):
        assert math.isclose(oracle.sigmoid(z) + oracle.sigmoid(-z), 1.0, rel_tol=1e-15)


def test_gate_toy(golden):
    g = golden("handbook_gate_toy.json")
    W = np.array(g["W_gate"])
    for word in ("book", "she"):
        z = np.array(g["x"][word]) @ W
        np.testing.assert_array_equal(r(z, 1), g["expected_z_1dp"][word])
        y = np.array(g["heads"][word])
        out = oracle.gate(y, z.reshape(2, 2), "elementwise")
        gates = np.array([[oracle.sigmoid(v) for v in row] for row in z.reshape(2, 2)])
        np.testing.assert_array_equal(r(gates, 3), g["expected_gate_3dp"][word])
        np.testing.assert_array_equal(r(out, 3), g["expected_out_3dp"][word])


def test_deepdive_gated_heads(golden):
    g = golden("deepdive_gated_heads.json")
    y = np.array(g["head_outputs"])
    z = np.array([math.log(1 / 9), 0.0])
    out = oracle.gate(y, z, "headwise")
    for c in g["expected_isclose"]:
        assert math.isclose(out[c["head"], c["dim"]], c["value"], rel_tol=1e-9)
    zc = g["zero_logit_case"]
    out0 = oracle.gate(np.array(zc["head_outputs"]), np.array(zc["gate_logits"]), "headwise")
    assert out0.tolist() == zc["expected_exact"]  # a zero logit is exactly 0.5x


def test_paper_notes_elementwise_example(golden):
    g = golden("paper_notes_gate_example.json")
    gates = np.array(g["gates"])
    logits = np.log(gates / (1.0 - gates))
    out = oracle.gate(np.array(g["Y"]), logits, "elementwise")
    np.testing.assert_allclose(out.reshape(-1), g["expected_concat"], rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_matches_torch_rms_norm():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 64)) * 3.0
    w = 1.0 + 0.1 * rng.standard_normal(64)
    got = oracle.rmsnorm(x, w, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_rmsnorm_closed_forms():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 32))
    ones = np.ones(32)
    eps = 1e-3
    y = oracle.rmsnorm(x, ones, eps)
    ms = (x * x).mean(axis=1)
    np.testing.assert_allclose(np.sqrt((y * y).mean(axis=1)), 1.0 / np.sqrt(1.0 + eps / ms), rtol=1e-13)
    # scale invariance without eps; the weight multiplies feature by feature
    np.testing.assert_allclose(oracle.rmsnorm(7.5 * x, ones, 0.0), oracle.rmsnorm(x, ones, 0.0), rtol=1e-13)
    w = rng.uniform(0.5, 1.5, 32)
    np.testing.assert_allclose(oracle.rmsnorm(x, w, eps), y * w, rtol=1e-14)


# ---------------------------------------------------------------- RoPE (reading: rotate-half, exponent over rotary_dim)

def test_rope_two_features_is_a_plane_rotation():
    x = np.array([[0.3, -1.7]])
    for p in (0.0, 1.0, 5.0, 1234.0):
        y = oracle.rope(x, [p], 2, 10000.0)
        c, s = math.cos(p), math.sin(p)  # i = 0 has frequency base^0 = 1 for any base
        np.testing.assert_allclose(y[0], [0.3 * c + 1.7 * s, -1.7 * c + 0.3 * s], rtol=1e-13, atol=1e-15)


def test_rope_pairs_i_with_i_plus_half_and_frequency_over_rotary_dim():
    base, p = 10000.0, 3.0
    x = np.zeros((1, 8))
    x[0, 1] = 1.0  # feature 1 pairs with feature 1 + 4/2 = 3 when rotary_dim = 4
    y = oracle.rope(x, [p], 4, base)
    theta = p * base ** (-2.0 * 1 / 4)
    expect = np.zeros(8)
    expect[1], expect[3] = math.cos(theta), math.sin(theta)
    np.testing.assert_allclose(y[0], expect, rtol=1e-13, atol=1e-15)


def test_rope_identities():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 32))
    np.testing.assert_array_equal(oracle.rope(x, [0, 0, 0, 0], 8, 1e4), x)  # position 0
    np.testing.assert_array_equal(oracle.rope(x, [5, 9, 11, 100], 0, 1e4), x)  # nothing rotates
    y = oracle.rope(x, [5, 9, 11, 100], 8, 1e4)
    np.testing.assert_array_equal(y[:, 8:], x[:, 8:])  # features >= rotary_dim untouched
    for i in range(4):  # each rotated pair keeps its length
        np.testing.assert_allclose(y[:, i] ** 2 + y[:, i + 4] ** 2, x[:, i] ** 2 + x[:, i + 4] ** 2, rtol=1e-13)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(4)
    qv, kv = rng.standard_normal(64), rng.standard_normal(64)
    for base in (1e4, 1e6, 1e7):
        s1 = oracle.rope(qv[None], [37], 64, base)[0] @ oracle.rope(kv[None], [12], 64, base)[0]
        s2 = oracle.rope(qv[None], [37 + 500], 64, base)[0] @ oracle.rope(kv[None], [12 + 500], 64, base)[0]
        assert abs(s1 - s2) < 1e-11


# ---------------------------------------------------------------- attention invariants

def _rand(shape, rng):
    return rng.standard_normal(shape)


def test_rows_sum_to_one_and_future_is_invisible():
    rng = np.random.default_rng(5)
    B, S, H, G, d = 2, 9, 4, 2, 8
    q, k, v = _rand((B, S, H, d), rng), _rand((B, S, G, d), rng), _rand((B, S, G, d), rng)
    out, attn = oracle.sdpa_gate(q, k, v, None, "none", want_attn=True)
    np.testing.assert_allclose(attn.sum(-1), 1.0, rtol=1e-14)
    assert np.all(np.triu(attn, 1) == 0.0)
    t = 4
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:, t + 1:] += 3.0
    k2[:, t + 1:] -= 2.0
    v2[:, t + 1:] *= 5.0
    out2 = oracle.sdpa_gate(q2, k2, v2, None, "none")
    np.testing.assert_array_equal(out2[:, : t + 1], out[:, : t + 1])


def test_gqa_equals_mha_with_replicated_kv():
    rng = np.random.default_rng(6)
    B, S, H, G, d = 1, 7, 6, 2, 4
    q, k, v = _rand((B, S, H, d), rng), _rand((B, S, G, d), rng), _rand((B, S, G, d), rng)
    z = _rand((B, S, H, d), rng)
    gqa = oracle.sdpa_gate(q, k, v, z, "elementwise")
    rep = H // G  # head h reads group floor(h / rep): groups are contiguous
    mha = oracle.sdpa_gate(q, np.repeat(k, rep, axis=2), np.repeat(v, rep, axis=2), z, "elementwise")
    np.testing.assert_array_equal(gqa, mha)
    # a strided mapping (h % G) would differ
    strided = oracle.sdpa_gate(q, np.tile(k, (1, 1, rep, 1)), np.tile(v, (1, 1, rep, 1)), z, "elementwise")
    assert np.abs(strided - gqa).max() > 1e-3


def test_sdpa_matches_torch_with_gqa():
    rng = np.random.default_rng(7)
    B, S, H, G, d = 2, 13, 8, 2, 16
    q, k, v = _rand((B, S, H, d), rng), _rand((B, S, G, d), rng), _rand((B, S, G, d), rng)
    got = oracle.sdpa_gate(q, k, v, None, "none")
    tq, tk, tv = (torch.from_numpy(a).transpose(1, 2) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, enable_gqa=True)
    ref = ref.transpose(1, 2).reshape(B, S, H * d).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_gate_special_cases():
    rng = np.random.default_rng(8)
    B, S, H, G, d = 1, 6, 4, 1, 8
    q, k, v = _rand((B, S, H, d), rng), _rand((B, S, G, d), rng), _rand((B, S, G, d), rng)
    plain = oracle.sdpa_gate(q, k, v, None, "none")
    zero = oracle.sdpa_gate(q, k, v, np.zeros((B, S, H, d)), "elementwise")
    np.testing.assert_array_equal(zero, 0.5 * plain)  # a zero logit is exactly one half
    opened = oracle.sdpa_gate(q, k, v, np.full((B, S, H, d), 60.0), "elementwise")
    np.testing.assert_array_equal(opened, plain)  # gate forced to 1 reproduces plain SDPA
    shut = oracle.sdpa_gate(q, k, v, np.full((B, S, H), -800.0), "headwise")
    assert np.all(shut == 0.0)  # gate forced to 0 switches only the branch off
    zh = _rand((B, S, H), rng)
    head = oracle.sdpa_gate(q, k, v, zh, "headwise")
    elem = oracle.sdpa_gate(q, k, v, np.repeat(zh[..., None], d, axis=-1), "elementwise")
    np.testing.assert_array_equal(head, elem)
    # the gate multiplies the head that owns it: head 1's logits move head 1 only
    z = np.zeros((B, S, H, d))
    z[:, :, 1] = 2.0
    moved = oracle.sdpa_gate(q, k, v, z, "elementwise").reshape(B, S, H, d)
    base = zero.reshape(B, S, H, d)
    np.testing.assert_array_equal(np.delete(moved, 1, axis=2), np.delete(base, 1, axis=2))
    np.testing.assert_allclose(moved[:, :, 1], base[:, :, 1] * 2 * oracle.sigmoid(2.0), rtol=1e-14)


# ---------------------------------------------------------------- composition

def _full_inputs(rng, B, S, H, G, d):
    return (_rand((B, S, H, d), rng), _rand((B, S, G, d), rng), _rand((B, S, G, d), rng),
            _rand((B, S, H, d), rng), 1 + 0.1 * rng.standard_normal(d), 1 + 0.1 * rng.standard_normal(d))


@pytest.mark.parametrize("rd,gate_mode", [(8, "elementwise"), (32, "headwise"), (0, "none"), (16, "elementwise")])
def test_prefill_is_norm_rope_then_torch_sdpa_then_gate(rd, gate_mode):
    rng = np.random.default_rng(10 + rd)
    B, S, H, G, d = 2, 11, 4, 2, 32
    q, k, v, z, qw, kw = _full_inputs(rng, B, S, H, G, d)
    if gate_mode == "headwise":
        z = z[..., 0]
    pos = rng.integers(0, 3000, size=(B, S)).astype(np.float64)
    eps, base = 1e-6, 1e6
    got = oracle.prefill(q, k, v, z, qw, kw, pos, rd, base, eps, gate_mode)
    # norm: torch's rms_norm; rope: the pinned oracle rope; attention: torch SDPA
    qn = torch.nn.functional.rms_norm(torch.from_numpy(q), (d,), torch.from_numpy(qw), eps=eps).numpy()
    kn = torch.nn.functional.rms_norm(torch.from_numpy(k), (d,), torch.from_numpy(kw), eps=eps).numpy()
    qr = oracle.rope(qn, pos[:, :, None], rd, base)
    kr = oracle.rope(kn, pos[:, :, None], rd, base)
    tq, tk, tv = (torch.from_numpy(a).transpose(1, 2) for a in (qr, kr, v))
    y = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, enable_gqa=True)
    y = y.transpose(1, 2).numpy()  # [B,S,H,d]
    if gate_mode == "elementwise":
        y = y * torch.sigmoid(torch.from_numpy(z)).numpy()
    elif gate_mode == "headwise":
        y = y * torch.sigmoid(torch.from_numpy(z)).numpy()[..., None]
    np.testing.assert_allclose(got, y.reshape(B, S, H * d), rtol=1e-11, atol=1e-12)


def test_prefill_rows_agree_with_full_prefill():
    rng = np.random.default_rng(20)
    B, S, H, G, d = 2, 17, 4, 1, 16
    q, k, v, z, qw, kw = _full_inputs(rng, B, S, H, G, d)
    full = oracle.prefill(q, k, v, z, qw, kw, None, 8, 1e4, 1e-6, "elementwise")
    rb, rt = [0, 1, 1, 0], [0, 16, 7, 3]
    rows = oracle.prefill_rows(q, k, v, z, qw, kw, None, 8, 1e4, 1e-6, "elementwise", rb, rt)
    np.testing.assert_allclose(rows, full[rb, rt], rtol=1e-13, atol=1e-14)


def test_default_positions_are_token_indices():
    rng = np.random.default_rng(21)
    B, S, H, G, d = 1, 9, 2, 1, 16
    q, k, v, z, qw, kw = _full_inputs(rng, B, S, H, G, d)
    a = oracle.prefill(q, k, v, z, qw, kw, None, 16, 1e4, 1e-6, "elementwise")
    b = oracle.prefill(q, k, v, z, qw, kw, np.arange(S, dtype=np.float64)[None], 16, 1e4, 1e-6, "elementwise")
    np.testing.assert_array_equal(a, b)


def test_decode_equals_last_prefill_row():
    rng = np.random.default_rng(22)
    B, S, H, G, d, rd, base, eps = 2, 12, 4, 2, 32, 8, 1e7, 1e-6
    q, k, v, z, qw, kw = _full_inputs(rng, B, S, H, G, d)
    full = oracle.prefill(q, k, v, z, qw, kw, None, rd, base, eps, "elementwise")
    Lmax = 16
    kc = np.zeros((B, G, Lmax, d))
    vc = np.zeros((B, G, Lmax, d))
    seqlens = [S, S - 5]
    for b in range(B):
        L = seqlens[b]
        kn = oracle.rmsnorm(k[b, :L], kw, eps)
        kr = oracle.rope(kn, np.arange(L)[:, None], rd, base)
        kc[b, :, :L] = kr.transpose(1, 0, 2)
        vc[b, :, :L] = v[b, :L].transpose(1, 0, 2)
    qn = np.stack([q[b, seqlens[b] - 1] for b in range(B)])
    zn = np.stack([z[b, seqlens[b] - 1] for b in range(B)])
    dec = oracle.decode(qn, kc, vc, seqlens, zn, qw, rd, base, eps, "elementwise")
    # prefill row L-1 of a sequence truncated to L tokens is row L-1 of the full one (causality)
    for b in range(B):
        np.testing.assert_allclose(dec[b], full[b, seqlens[b] - 1], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- gate variants
# ("Gated Attention" deep-dive, section "门放在哪里？": head-shared scores, an additive
# gate Y + sigmoid(XW), SiLU instead of sigmoid; section "第二条机制线索": the
# non-sparse control NS-sigmoid(x) = 0.5 + 0.5 sigmoid(x).)

def test_gate_activation_closed_forms():
    # NS-sigmoid: 3/4 at 0, inside [1/2, 1], symmetric about 3/4, limits 1/2 and 1
    assert oracle.gate_act(0.0, "ns_sigmoid") == 0.75
    for x in (-30.0, -2.5, -0.3, 0.7, 4.0, 30.0):
        ns = oracle.gate_act(x, "ns_sigmoid")
        assert 0.5 <= ns <= 1.0
        assert abs(ns + oracle.gate_act(-x, "ns_sigmoid") - 1.5) < 1e-15
    assert abs(oracle.gate_act(40.0, "ns_sigmoid") - 1.0) < 1e-15
    assert abs(oracle.gate_act(-40.0, "ns_sigmoid") - 0.5) < 1e-15
    # SiLU: 0 at 0; silu(x) - silu(-x) = x; silu(ln 3) = (3/4) ln 3
    assert oracle.gate_act(0.0, "silu") == 0.0
    for x in (-7.0, -1.2, 0.4, 3.3):
        assert abs(oracle.gate_act(x, "silu") - oracle.gate_act(-x, "silu") - x) < 1e-13
    assert abs(oracle.gate_act(math.log(3.0), "silu") - 0.75 * math.log(3.0)) < 1e-15
    assert abs(oracle.gate_act(math.log(3.0), "sigmoid") - 0.75) < 1e-15


def test_silu_gate_matches_torch_silu():
    z = torch.linspace(-12, 12, 97, dtype=torch.float64)
    got = oracle.gate(np.ones((1, z.numel())), z.numpy().reshape(1, -1), oracle.gate_code("elementwise", "silu"))
    np.testing.assert_allclose(got[0], torch.nn.functional.silu(z).numpy(), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("layout,act", [(lay, act) for lay in ("elementwise", "headwise", "head_shared")
                                        for act in ("sigmoid", "ns_sigmoid", "silu")])
def test_gate_layouts_and_combine_on_constant_values(layout, act):
    # every row of v equal to c: attention returns c exactly, so the output is c*act(z)
    # (multiplicative) or c + act(z) (additive), with z read per head, per head and
    # dimension, or per dimension shared by all heads
    rng = np.random.default_rng(7)
    B, S, H, G, d = 2, 5, 4, 2, 8
    q, k = rng.standard_normal((B, S, H, d)), rng.standard_normal((B, S, G, d))
    c = rng.standard_normal((G, d))
    v = np.broadcast_to(c[None, None], (B, S, G, d)).copy()
    z = 2.0 * rng.standard_normal({"elementwise": (B, S, H, d), "headwise": (B, S, H),
                                   "head_shared": (B, S, d)}[layout])
    if layout == "elementwise":
        zfull = z
    elif layout == "headwise":
        zfull = np.broadcast_to(z[..., None], (B, S, H, d))
    else:
        zfull = np.broadcast_to(z[:, :, None, :], (B, S, H, d))
    g = np.vectorize(lambda x: oracle.gate_act(x, act))(zfull)
    cv = np.repeat(c, H // G, axis=0)  # head h reads group h // (H/G)
    for additive in (False, True):
        out = oracle.sdpa_gate(q, k, v, z, oracle.gate_code(layout, act, additive)).reshape(B, S, H, d)
        np.testing.assert_allclose(out, cv + g if additive else cv * g, rtol=1e-12, atol=1e-12)


def test_decode_head_shared_additive_equals_last_prefill_row():
    rng = np.random.default_rng(23)
    B, S, H, G, d, rd, base, eps = 2, 10, 4, 2, 16, 8, 1e6, 1e-6
    q, k, v, _, qw, kw = _full_inputs(rng, B, S, H, G, d)
    z = rng.standard_normal((B, S, d))
    mode = oracle.gate_code("head_shared", "ns_sigmoid", True)
    full = oracle.prefill(q, k, v, z, qw, kw, None, rd, base, eps, mode)
    kc, vc = np.zeros((B, G, S, d)), np.zeros((B, G, S, d))
    for b in range(B):
        kc[b] = oracle.rope(oracle.rmsnorm(k[b], kw, eps), np.arange(S)[:, None], rd, base).transpose(1, 0, 2)
        vc[b] = v[b].transpose(1, 0, 2)
    seqlens = [S, S - 3]
    qn = np.stack([q[b, seqlens[b] - 1] for b in range(B)])
    zn = np.stack([z[b, seqlens[b] - 1] for b in range(B)])
    dec = oracle.decode(qn, kc, vc, seqlens, zn, qw, rd, base, eps, mode)
    for b in range(B):
        np.testing.assert_allclose(dec[b], full[b, seqlens[b] - 1], rtol=1e-12, atol=1e-13)


def test_decode_append_equals_last_prefill_row():
    """Appending token L-1 to a cache of L-1 tokens and decoding gives row L-1 of
    the prefill; the appended K row is that token's normed, rotated key and the
    appended V row its raw value."""
    rng = np.random.default_rng(24)
    B, S, H, G, d, rd, base, eps = 2, 11, 4, 2, 16, 8, 1e6, 1e-6
    q, k, v, z, qw, kw = _full_inputs(rng, B, S, H, G, d)
    full = oracle.prefill(q, k, v, z, qw, kw, None, rd, base, eps, "elementwise")
    Lmax = 14
    seqlens = [S, S - 4]
    kc, vc = np.zeros((B, G, Lmax, d)), np.zeros((B, G, Lmax, d))
    for b in range(B):
        L = seqlens[b] - 1  # the cache holds the tokens before the new one
        kr = oracle.rope(oracle.rmsnorm(k[b, :L], kw, eps), np.arange(L)[:, None], rd, base)
        kc[b, :, :L] = kr.transpose(1, 0, 2)
        vc[b, :, :L] = v[b, :L].transpose(1, 0, 2)
    last = [seqlens[b] - 1 for b in range(B)]
    qn = np.stack([q[b, last[b]] for b in range(B)])
    kn = np.stack([k[b, last[b]] for b in range(B)])
    vn = np.stack([v[b, last[b]] for b in range(B)])
    zn = np.stack([z[b, last[b]] for b in range(B)])
    out, kc2, vc2 = oracle.decode_append(qn, kn, vn, kc, vc, seqlens, zn, qw, kw, rd, base, eps, "elementwise")
    for b in range(B):
        np.testing.assert_allclose(out[b], full[b, last[b]], rtol=1e-12, atol=1e-13)
        want_k = oracle.rope(oracle.rmsnorm(k[b, last[b]], kw, eps), [last[b]], rd, base)
        np.testing.assert_allclose(kc2[b, :, last[b]], want_k, rtol=1e-13, atol=1e-14)
        np.testing.assert_array_equal(vc2[b, :, last[b]], v[b, last[b]])
        np.testing.assert_array_equal(kc2[b, :, :last[b]], kc[b, :, :last[b]])  # earlier rows untouched


def test_varlen_sequences_are_independent_batches():
    """Packed sequences: each one equals a batch of one on its own (positions
    restarting at 0, keys of its own only); equal lengths equal the batched
    prefill; changing a neighbour changes nothing."""
    rng = np.random.default_rng(25)
    H, G, d, rd, base, eps = 4, 2, 16, 8, 1e6, 1e-6
    lens = [5, 1, 0, 9, 3]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v, z, qw, kw = _full_inputs(rng, 1, T, H, G, d)
    q, k, v, z = q[0], k[0], v[0], z[0]
    out = oracle.prefill_varlen(q, k, v, z, qw, kw, None, cu, rd, base, eps, "elementwise")
    for i, n in enumerate(lens):
        s = int(cu[i])
        if n == 0:
            continue
        alone = oracle.prefill(q[None, s:s + n], k[None, s:s + n], v[None, s:s + n], z[None, s:s + n], qw, kw, None,
                               rd, base, eps, "elementwise")[0]
        np.testing.assert_array_equal(out[s:s + n], alone)
    # a perturbed neighbour leaves sequence 3 as it was
    k2 = k.copy()
    k2[:int(cu[3])] += 1.0
    k2[int(cu[4]):] -= 1.0
    out2 = oracle.prefill_varlen(q, k2, v, z, qw, kw, None, cu, rd, base, eps, "elementwise")
    np.testing.assert_array_equal(out2[int(cu[3]):int(cu[4])], out[int(cu[3]):int(cu[4])])
    # equal lengths: the batched prefill
    B, S = 3, 6
    qb, kb, vb, zb, _, _ = _full_inputs(rng, B, S, H, G, d)
    batched = oracle.prefill(qb, kb, vb, zb, qw, kw, None, rd, base, eps, "elementwise").reshape(B * S, H * d)
    packed = oracle.prefill_varlen(qb.reshape(B * S, H, d), kb.reshape(B * S, G, d), vb.reshape(B * S, G, d),
                                   zb.reshape(B * S, H, d), qw, kw, None, np.arange(0, B * S + 1, S), rd, base, eps,
                                   "elementwise")
    np.testing.assert_array_equal(packed, batched)


def test_kv_cache_byte_accounting(golden):
    from gated_softmax_attention_gqa_gb300 import workloads

    g = golden("kv_cache_sizes.json")
    assert workloads.kv_numbers_per_token(g["G"], g["d"]) == g["expected_numbers_per_token_gqa"]
    assert workloads.kv_numbers_per_token(g["H"], g["d"]) == g["expected_numbers_per_token_mha"]
    for kv_heads, key in ((g["G"], "expected_total_MB_gqa"), (g["H"], "expected_total_MB_mha")):
        total = g["layers"] * workloads.decode_kv_bytes([g["seq_len"]], kv_heads, g["d"], g["bytes_per_number"])
        assert round(total / 2**20, 1) == g[key]


# ---- o_proj: y = x W_O^T (the step after the path)

def test_o_proj_identity_and_permutation():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 8))
    np.testing.assert_array_equal(oracle.o_proj(x, np.eye(8)), x)
    perm = np.array([3, 0, 7, 1])
    w = np.eye(8)[perm]  # row n of W_O selects feature perm[n]
    np.testing.assert_array_equal(oracle.o_proj(x, w), x[:, perm])


def test_o_proj_brute_force_and_linearity():
    rng = np.random.default_rng(4)
    x1, x2 = rng.standard_normal((3, 6)), rng.standard_normal((3, 6))
    w = rng.standard_normal((2, 6))
    want = np.array([[sum(x1[t, k] * w[n, k] for k in range(6)) for n in range(2)] for t in range(3)])
    assert np.abs(oracle.o_proj(x1, w) - want).max() < 1e-12
    lhs = oracle.o_proj(2.0 * x1 - 3.0 * x2, w)
    rhs = 2.0 * oracle.o_proj(x1, w) - 3.0 * oracle.o_proj(x2, w)
    assert np.abs(lhs - rhs).max() < 1e-12
    assert oracle.o_proj(x1[None], w).shape == (1, 3, 2)  # leading dimensions pass through
