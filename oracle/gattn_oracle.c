/*
 * gattn_oracle.c -- plain fp64 CPU oracle for the gated softmax attention core.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The GPU library
 * never links, calls or includes it, and it shares no code with the CUDA path.
 *
 * What it computes, step by step, in the order and notation of the source pages:
 *
 *   "Gated attention" handbook chapter (anrans.github.io, section "The code:
 *   qwen/attention.py" and its shape table): per head, q and k each pass through
 *   an RMSNorm over head_dim with a learned weight, then RoPE; query head h reads
 *   KV group floor(h / (H/G)); scores q.k/sqrt(d); causal mask (-inf above the
 *   diagonal); row softmax; weighted sum of V; heads concatenated to [T, H*d];
 *   multiplied by sigmoid(gate logits) before o_proj.
 *   "Gated Attention" deep-dive (cooking-agi, section "门放在哪里？"): the gate
 *   is G_h = sigmoid(X W_g,h) applied to O_h after SDPA and before W_O; headwise
 *   = one logit per token per head, elementwise = one per dimension.  The same
 *   section lists the variants the paper compares: head-shared scores (one
 *   vector for all heads), an additive gate Y' = Y + sigmoid(X W), and SiLU in
 *   place of sigmoid; section "第二条机制线索" defines the non-sparse control
 *   NS-sigmoid(x) = 0.5 + 0.5 sigmoid(x).
 *   "Attention, worked all the way through" (curtisalexander.github.io, section
 *   "Why scaling and stable softmax matter"): softmax subtracts the row max
 *   before exp; a masked -inf becomes weight 0.  Section "Qwen3's exact order":
 *   RMSNorm q and k (not V), RoPE q and k (not V), then causal GQA attention.
 *   "Multi-head attention and GQA" chapter (mlx.void.app, section "分组查询注意力"):
 *   query head h dots the K of group floor(h / group_size).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - RMSNorm body is not printed: y = x * (mean(x^2) + eps)^(-1/2) * w, with
 *     the weight multiplying directly.
 *   - RoPE body is not printed: rotate-half over the first rotary_dim features,
 *     feature i paired with i + rotary_dim/2, angle pos * base^(-2i/rotary_dim);
 *     features >= rotary_dim pass through.  The exact convention is a reading,
 *     pinned by closed forms of that reading (plane rotations), not by the pages.
 *   - The mask index is the sequence index (key j visible to query t iff j <= t);
 *     positions only feed RoPE.
 *   - Decode: the cache holds already-normed, already-rotated K and raw V; the
 *     new query sits at position seqlen-1 and sees keys 0..seqlen-1.
 *   - SiLU is not printed: silu(z) = z * sigmoid(z).  An additive gate with
 *     SiLU adds silu(z).  A head-shared gate is elementwise over head_dim.
 *
 * Everything is double precision.  Layouts (all contiguous, row-major):
 *   q [B,S,H,d]   k,v [B,S,G,d]   gate [B,S,H,d] (elementwise), [B,S,H] (headwise)
 *   or [B,S,d] (head-shared)   out [B,S,H*d]   pos [B,S] (NULL means 0..S-1)
 *
 * gate_mode = layout | activation << 4 | (256 if additive): layout 0 none,
 * 1 elementwise, 2 headwise, 3 head-shared; activation 0 sigmoid, 1 NS-sigmoid,
 * 2 SiLU.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_GATE_NONE 0
#define ORACLE_GATE_ELEMENTWISE 1
#define ORACLE_GATE_HEADWISE 2
#define ORACLE_GATE_HEAD_SHARED 3
#define ORACLE_GATE_ACT_SIGMOID 0
#define ORACLE_GATE_ACT_NS_SIGMOID 1
#define ORACLE_GATE_ACT_SILU 2
#define ORACLE_GATE_ADDITIVE 256

/* sigmoid(z) = 1 / (1 + e^-z), evaluated so that neither branch overflows
 * (the deep-dive's `sigmoid` helper takes the same two branches). */
double oracle_sigmoid(double z) {
    if (z >= 0.0) return 1.0 / (1.0 + exp(-z));
    double e = exp(z);
    return e / (1.0 + e);
}

/* RMSNorm of n_rows rows of length d: y = x * rsqrt(mean(x^2) + eps) * w. */
void oracle_rmsnorm(const double* x, const double* w, int64_t n_rows, int d, double eps, double* y) {
    for (int64_t r = 0; r < n_rows; ++r) {
        const double* xr = x + r * d;
        double ss = 0.0;
        for (int e = 0; e < d; ++e) ss += xr[e] * xr[e];
        double inv = 1.0 / sqrt(ss / (double)d + eps);
        for (int e = 0; e < d; ++e) y[r * d + e] = xr[e] * inv * w[e];
    }
}

/* Partial rotate-half RoPE on one row at integer position p. */
static void rope_row(const double* x, double p, int d, int rd, double base, double* y) {
    int half = rd / 2;
    for (int e = 0; e < d; ++e) y[e] = x[e];
    for (int i = 0; i < half; ++i) {
        double theta = p * pow(base, -2.0 * (double)i / (double)rd);
        double c = cos(theta), s = sin(theta);
        double a = x[i], b = x[i + half];
        y[i] = a * c - b * s;
        y[i + half] = b * c + a * s;
    }
}

/* RoPE on n_rows rows; row r is at position pos[r]. */
void oracle_rope(const double* x, const double* pos, int64_t n_rows, int d, int rd, double base, double* y) {
    for (int64_t r = 0; r < n_rows; ++r) rope_row(x + r * d, pos[r], d, rd, base, y + r * d);
}

/* One query row against keys 0..n_keys-1 of one KV group:
 *   s_j = q.k_j / sqrt(d); m = max s; w_j = exp(s_j - m) / sum exp(s_i - m);
 *   o = sum_j w_j v_j.  key_stride/val_stride are in elements between keys.
 * If attn != NULL the n_keys weights are written there. */
static void attend_row(const double* q, const double* kr, int64_t key_stride, const double* v,
                       int64_t val_stride, int64_t n_keys, int d, double* o, double* attn, double* scratch) {
    double scale = 1.0 / sqrt((double)d);
    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j) {
        double s = 0.0;
        for (int e = 0; e < d; ++e) s += q[e] * kr[j * key_stride + e];
        s *= scale;
        scratch[j] = s;
        if (s > m) m = s;
    }
    double z = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        scratch[j] = exp(scratch[j] - m);
        z += scratch[j];
    }
    for (int e = 0; e < d; ++e) o[e] = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        double wj = scratch[j] / z;
        if (attn) attn[j] = wj;
        for (int e = 0; e < d; ++e) o[e] += wj * v[j * val_stride + e];
    }
}

/* The gate's activation of one logit: sigmoid, NS-sigmoid = 0.5 + 0.5 sigmoid,
 * or SiLU = z sigmoid(z). */
double oracle_gate_act(double z, int act) {
    double s = oracle_sigmoid(z);
    if (act == ORACLE_GATE_ACT_NS_SIGMOID) return 0.5 + 0.5 * s;
    if (act == ORACLE_GATE_ACT_SILU) return z * s;
    return s;
}

/* Gate a head's attention output: o * act(z) (multiplicative, the default) or
 * o + act(z) (additive).  z holds d logits, or one for a headwise gate. */
static void apply_gate(double* o, const double* z, int d, int gate_mode) {
    int layout = gate_mode & 15, act = (gate_mode >> 4) & 15;
    int additive = (gate_mode & ORACLE_GATE_ADDITIVE) != 0;
    if (layout == ORACLE_GATE_NONE) return;
    for (int e = 0; e < d; ++e) {
        double g = oracle_gate_act(layout == ORACLE_GATE_HEADWISE ? z[0] : z[e], act);
        o[e] = additive ? o[e] + g : o[e] * g;
    }
}

/* The gate logits of token row `bt` (b*S + t in prefill, b in decode) for head h:
 * elementwise [.., H, d], headwise [.., H], head-shared [.., d]. */
static const double* gate_at(const double* gate, int gate_mode, int64_t bt, int H, int h, int d) {
    switch (gate_mode & 15) {
        case ORACLE_GATE_ELEMENTWISE: return gate + (bt * H + h) * d;
        case ORACLE_GATE_HEADWISE: return gate + bt * H + h;
        case ORACLE_GATE_HEAD_SHARED: return gate + bt * d;
        default: return NULL;
    }
}

/* Gate one [n_heads, d] block y with the logits z of one token (layout as
 * gate_mode says: [n_heads, d], [n_heads] or [d]). */
void oracle_gate(const double* y, const double* z, int n_heads, int d, int gate_mode, double* out) {
    for (int h = 0; h < n_heads; ++h) {
        for (int e = 0; e < d; ++e) out[h * d + e] = y[h * d + e];
        apply_gate(out + (int64_t)h * d, gate_at(z, gate_mode, 0, n_heads, h, d), d, gate_mode);
    }
}

/* Causal GQA SDPA + gate on q, k that are already normed and rotated.
 * attn (optional) receives the [B,H,S,S] weight matrix, zero above the diagonal. */
void oracle_sdpa_gate(const double* q, const double* k, const double* v, const double* gate, int B, int S,
                      int H, int G, int d, int gate_mode, double* out, double* attn) {
    int r = H / G;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            int g = h / r;
            double* scratch = (double*)malloc(sizeof(double) * (size_t)S);
            double* o = (double*)malloc(sizeof(double) * (size_t)d);
            const double* kb = k + ((int64_t)b * S * G + g) * d;
            const double* vb = v + ((int64_t)b * S * G + g) * d;
            for (int t = 0; t < S; ++t) {
                const double* qt = q + (((int64_t)b * S + t) * H + h) * d;
                double* arow = attn ? attn + (((int64_t)b * H + h) * S + t) * S : NULL;
                attend_row(qt, kb, (int64_t)G * d, vb, (int64_t)G * d, t + 1, d, o, arow, scratch);
                if (arow) for (int j = t + 1; j < S; ++j) arow[j] = 0.0;
                apply_gate(o, gate_at(gate, gate_mode, (int64_t)b * S + t, H, h, d), d, gate_mode);
                memcpy(out + ((int64_t)b * S + t) * H * d + (int64_t)h * d, o, sizeof(double) * (size_t)d);
            }
            free(scratch);
            free(o);
        }
    }
}

/* norm + rope of one [S, n_heads, d] block of batch b for head `hd`, into dst [S, d]. */
static void prologue_head(const double* x, const double* w, const double* posb, int S, int n_heads, int hd,
                          int d, int rd, double base, double eps, double* dst, double* tmp) {
    for (int t = 0; t < S; ++t) {
        const double* xr = x + ((int64_t)t * n_heads + hd) * d;
        oracle_rmsnorm(xr, w, 1, d, eps, tmp);
        rope_row(tmp, posb ? posb[t] : (double)t, d, rd, base, dst + (int64_t)t * d);
    }
}

/* Full prefill: QK-RMSNorm, partial RoPE, causal GQA SDPA, gate. */
void oracle_prefill(const double* q, const double* k, const double* v, const double* gate, const double* qnorm_w,
                    const double* knorm_w, const double* pos, int B, int S, int H, int G, int d, int rd,
                    double base, double eps, int gate_mode, double* out) {
    int r = H / G;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            int g = h / r;
            const double* posb = pos ? pos + (int64_t)b * S : NULL;
            double* qr = (double*)malloc(sizeof(double) * (size_t)S * d);
            double* kr = (double*)malloc(sizeof(double) * (size_t)S * d);
            double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
            double* o = (double*)malloc(sizeof(double) * (size_t)d);
            double* scratch = (double*)malloc(sizeof(double) * (size_t)S);
            prologue_head(q + (int64_t)b * S * H * d, qnorm_w, posb, S, H, h, d, rd, base, eps, qr, tmp);
            prologue_head(k + (int64_t)b * S * G * d, knorm_w, posb, S, G, g, d, rd, base, eps, kr, tmp);
            const double* vb = v + ((int64_t)b * S * G + g) * d;
            for (int t = 0; t < S; ++t) {
                attend_row(qr + (int64_t)t * d, kr, d, vb, (int64_t)G * d, t + 1, d, o, NULL, scratch);
                apply_gate(o, gate_at(gate, gate_mode, (int64_t)b * S + t, H, h, d), d, gate_mode);
                memcpy(out + ((int64_t)b * S + t) * H * d + (int64_t)h * d, o, sizeof(double) * (size_t)d);
            }
            free(qr); free(kr); free(tmp); free(o); free(scratch);
        }
    }
}

/* Prefill restricted to selected query rows: row i is (row_b[i], row_t[i]); all
 * heads of that token are computed and written to out[i, H*d].  The keys of each
 * (batch, group) are normed and rotated once, exactly as in oracle_prefill. */
void oracle_prefill_rows(const double* q, const double* k, const double* v, const double* gate,
                         const double* qnorm_w, const double* knorm_w, const double* pos, int B, int S, int H,
                         int G, int d, int rd, double base, double eps, int gate_mode, const int32_t* row_b,
                         const int32_t* row_t, int n_rows, double* out) {
    int r = H / G;
    double* kr_all = (double*)malloc(sizeof(double) * (size_t)B * G * S * d);
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int g = 0; g < G; ++g) {
            double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
            const double* posb = pos ? pos + (int64_t)b * S : NULL;
            prologue_head(k + (int64_t)b * S * G * d, knorm_w, posb, S, G, g, d, rd, base, eps,
                          kr_all + ((int64_t)b * G + g) * S * d, tmp);
            free(tmp);
        }
    }
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int i = 0; i < n_rows; ++i) {
        for (int h = 0; h < H; ++h) {
            int b = row_b[i], t = row_t[i], g = h / r;
            const double* posb = pos ? pos + (int64_t)b * S : NULL;
            const double* kr = kr_all + ((int64_t)b * G + g) * S * d;
            double* qr = (double*)malloc(sizeof(double) * (size_t)d);
            double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
            double* o = (double*)malloc(sizeof(double) * (size_t)d);
            double* scratch = (double*)malloc(sizeof(double) * (size_t)(t + 1));
            oracle_rmsnorm(q + (((int64_t)b * S + t) * H + h) * d, qnorm_w, 1, d, eps, tmp);
            rope_row(tmp, posb ? posb[t] : (double)t, d, rd, base, qr);
            const double* vb = v + ((int64_t)b * S * G + g) * d;
            attend_row(qr, kr, d, vb, (int64_t)G * d, t + 1, d, o, NULL, scratch);
            apply_gate(o, gate_at(gate, gate_mode, (int64_t)b * S + t, H, h, d), d, gate_mode);
            memcpy(out + (int64_t)i * H * d + (int64_t)h * d, o, sizeof(double) * (size_t)d);
            free(qr); free(tmp); free(o); free(scratch);
        }
    }
    free(kr_all);
}

/* Decode step against a KV cache.
 *   q_new [B,H,d] raw; kcache, vcache [B,G,Lmax,d] (K already normed and rotated);
 *   seqlens [B] includes the new token; its query sits at position seqlens[b]-1.
 *   gate [B,H,d], [B,H] or [B,d]; out [B,H*d]. */
void oracle_decode(const double* q_new, const double* kcache, const double* vcache, const int32_t* seqlens,
                   const double* gate, const double* qnorm_w, int B, int H, int G, int d, int Lmax, int rd,
                   double base, double eps, int gate_mode, double* out) {
    int r = H / G;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            int g = h / r;
            int L = seqlens[b];
            double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
            double* qr = (double*)malloc(sizeof(double) * (size_t)d);
            double* o = (double*)malloc(sizeof(double) * (size_t)d);
            double* scratch = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
            oracle_rmsnorm(q_new + ((int64_t)b * H + h) * d, qnorm_w, 1, d, eps, tmp);
            rope_row(tmp, (double)(L - 1), d, rd, base, qr);
            const double* kb = kcache + ((int64_t)b * G + g) * Lmax * d;
            const double* vb = vcache + ((int64_t)b * G + g) * Lmax * d;
            attend_row(qr, kb, d, vb, d, L, d, o, NULL, scratch);
            apply_gate(o, gate_at(gate, gate_mode, b, H, h, d), d, gate_mode);
            memcpy(out + (int64_t)b * H * d + (int64_t)h * d, o, sizeof(double) * (size_t)d);
            free(tmp); free(qr); free(o); free(scratch);
        }
    }
}

/* Decode step that first appends the new token to the cache, then attends
 * ("Multi-head attention and GQA" chapter, section "拼接各头 → 用 W_O 投影": K and V
 * are cached per token).  For every sequence b with 1 <= seqlens[b] <= Lmax and
 * group g, the new token's key k_new[b,g] is normed with knorm_w and rotated at
 * position seqlens[b]-1 and written to kcache[b,g,seqlens[b]-1]; its raw value
 * v_new[b,g] goes to vcache[b,g,seqlens[b]-1].  Then oracle_decode.
 *   k_new, v_new [B,G,d]; kcache, vcache [B,G,Lmax,d] (updated in place). */
void oracle_decode_append(const double* q_new, const double* k_new, const double* v_new, double* kcache,
                          double* vcache, const int32_t* seqlens, const double* gate, const double* qnorm_w,
                          const double* knorm_w, int B, int H, int G, int d, int Lmax, int rd, double base,
                          double eps, int gate_mode, double* out) {
    double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
    for (int b = 0; b < B; ++b) {
        int L = seqlens[b];
        if (L < 1 || L > Lmax) continue;
        for (int g = 0; g < G; ++g) {
            const double* kn = k_new + ((int64_t)b * G + g) * d;
            double* kdst = kcache + (((int64_t)b * G + g) * Lmax + (L - 1)) * d;
            double* vdst = vcache + (((int64_t)b * G + g) * Lmax + (L - 1)) * d;
            oracle_rmsnorm(kn, knorm_w, 1, d, eps, tmp);
            rope_row(tmp, (double)(L - 1), d, rd, base, kdst);
            memcpy(vdst, v_new + ((int64_t)b * G + g) * d, sizeof(double) * (size_t)d);
        }
    }
    free(tmp);
    oracle_decode(q_new, kcache, vcache, seqlens, gate, qnorm_w, B, H, G, d, Lmax, rd, base, eps, gate_mode, out);
}
