// prefill_fp32.cu -- fp32 causal gated GQA attention on CUDA cores.
//
// The fp32 path exists for inputs that must be matched to 1e-4: neither bf16
// nor tf32 tensor-core arithmetic can reach that, so this kernel uses plain
// fp32 FMAs and accurate expf.  It is a correctness path, not a throughput path.
//
// Per query row t of head h (group g = h / (H/G)): online softmax over keys
// j <= t of s_j = q'_t . k'_j / sqrt(d), o = sum_j softmax_j v_j, then
// o * sigmoid(gate) written to out[b, t, h*d : h*d+d].  q' and k' come from the
// norm + RoPE pre-pass.  ("Gated attention" handbook chapter, sections "The
// formula" and "The code: qwen/attention.py"; "Gated Attention" deep-dive,
// section "门放在哪里？".)
#include "common.cuh"
#include "internal.h"

namespace gattn {
namespace {

constexpr int kRowsPerBlock = 8;  // one warp per query row

__global__ void __launch_bounds__(kRowsPerBlock * 32) prefill_f32_kernel(const __grid_constant__ PrefillF32Params p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H, g = h / (p.H / p.G);
    const int t = blockIdx.x * kRowsPerBlock + warp;
    if (t >= p.S) return;
    const int d = p.d, ne = d >> 5;  // d is a multiple of 32, at most 256
    const float* q = p.qr + ((int64_t)bh * p.S + t) * d;
    const float* kb = p.kr + (int64_t)(b * p.G + g) * p.S * d;
    const float* vb = p.v + ((int64_t)b * p.S * p.G + g) * d;
    const int64_t vstride = (int64_t)p.G * d;

    float qv[8], o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        qv[i] = i < ne ? q[lane + 32 * i] : 0.f;
        o[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    // packed sequences: keys from the first token of this token's sequence
    for (int j = p.tok_start ? p.tok_start[t] : 0; j <= t; ++j) {
        const float* kj = kb + (int64_t)j * d;
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < ne) s = fmaf(qv[i], kj[lane + 32 * i], s);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        s *= p.scale;
        const float m_new = fmaxf(m, s);
        const float alpha = expf(m - m_new);
        const float pj = expf(s - m_new);
        l = l * alpha + pj;
        const float* vj = vb + (int64_t)j * vstride;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < ne) o[i] = fmaf(pj, vj[lane + 32 * i], o[i] * alpha);
        m = m_new;
    }
    const float inv_l = 1.f / l;
    const int64_t tok = (int64_t)b * p.S + t;
    float* out = p.out + (tok * p.H + h) * d;
    // the gate's activation: one per head (headwise), else per dimension
    // (elementwise, or head-shared with a head stride of 0); none: 1
    float gh = 1.f;
    if (gate_layout(p.gate_mode) == GATTN_GATE_HEADWISE) {
        const float z = p.gate[tok * p.gate_tok_stride + (int64_t)h * p.gate_head_stride];
        gh = gate_act(z, 1.f / (1.f + expf(-z)), p.gate_mode);
    }
    const bool additive = gate_additive(p.gate_mode);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i >= ne) continue;
        const int e = lane + 32 * i;
        float gv = gh;
        if (gate_per_dim(p.gate_mode)) {
            const float z = p.gate[tok * p.gate_tok_stride + (int64_t)h * p.gate_head_stride + e];
            gv = gate_act(z, 1.f / (1.f + expf(-z)), p.gate_mode);
        }
        out[e] = additive ? o[i] * inv_l + gv : o[i] * inv_l * gv;
    }
}

}  // namespace

cudaError_t launch_prefill_f32(const PrefillF32Params& p, cudaStream_t stream, cudaEvent_t ev_start,
                               cudaEvent_t ev_stop) {
    dim3 grid((p.S + kRowsPerBlock - 1) / kRowsPerBlock, p.B * p.H);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    if (ev_start) cudaEventRecord(ev_start, stream);
    prefill_f32_kernel<<<grid, kRowsPerBlock * 32, 0, stream>>>(p);
    cudaError_t err = cudaGetLastError();
    if (ev_stop) cudaEventRecord(ev_stop, stream);
    return err;
}

}  // namespace gattn
