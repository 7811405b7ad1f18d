// prologue.cu -- QK-RMSNorm + partial RoPE pre-pass.
//
// Writes rope(rmsnorm(x) * w) for every (token, head) row of a [B,S,n_heads,d]
// tensor into a contiguous [B,n_heads,S,d] tensor, the layout the attention
// kernels stream by TMA.  Used for K on the bf16 path (keys are re-read by
// every query tile of every head in their group, so they are normalised once
// here rather than in each CTA) and for both Q and K on the fp32 path.
//
// RMSNorm: y = x * rsqrt(mean(x^2) + eps) * w over head_dim, applied before RoPE
// ("Gated attention" handbook chapter, section "Four things Qwen3.5 adds to the
// textbook").  RoPE (reading: rotate-half over the first rotary_dim features,
// angle pos * base^(-2i/rotary_dim); features >= rotary_dim untouched).
#include "common.cuh"
#include "internal.h"

namespace gattn {
namespace {

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

constexpr int kWarpsPerBlock = 8;

// One warp per row; lanes own features lane, lane+32, ...  The normalised row is
// staged in shared memory so each lane can read its rotation partner.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) qk_prologue_kernel(const __grid_constant__ ProloguePlan p) {
    extern __shared__ float rows[];
    pdl_launch_dependents();  // the attention kernel may start its own prologue now
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kWarpsPerBlock + warp;
    const int64_t n_rows = (int64_t)p.B * p.S * p.n_heads;
    if (r >= n_rows) return;
    const int hd = (int)(r % p.n_heads);
    const int64_t bt = r / p.n_heads;  // b*S + t
    const int t = (int)(bt % p.S);
    const int b = (int)(bt / p.S);
    const int d = p.d;
    const Tin* x = static_cast<const Tin*>(p.x) + bt * p.tok_stride + (int64_t)hd * p.head_stride;
    const Tin* w = static_cast<const Tin*>(p.w);
    float* row = rows + warp * d;

    float ss = 0.f;
    for (int e = lane; e < d; e += 32) {
        const float v = to_f<Tin>(x[e]);
        row[e] = v;
        ss += v * v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rinv = rsqrtf(ss / (float)d + p.eps);
    for (int e = lane; e < d; e += 32) row[e] = row[e] * rinv * to_f<Tin>(w[e]);
    __syncwarp();

    const float posf = p.pos ? (float)p.pos[bt] : (float)t;
    const int half = p.rd >> 1;
    Tout* dst = static_cast<Tout*>(p.dst) + (((int64_t)b * p.n_heads + hd) * p.S + t) * d;
    for (int e = lane; e < d; e += 32) {
        float y = row[e];
        if (e < half) {
            float s, c;
            rope_sincos(posf * p.inv_freq[e], &s, &c);
            y = row[e] * c - row[e + half] * s;
        } else if (e < p.rd) {
            const int i = e - half;
            float s, c;
            rope_sincos(posf * p.inv_freq[i], &s, &c);
            y = row[e] * c + row[i] * s;
        }
        dst[e] = from_f<Tout>(y);
    }
}

// bf16 -> bf16 with rotary_dim % 16 == 0 (the tensor-core path): a row of d
// elements is spread over d/8 lanes, one 16-byte load and one 16-byte store each,
// so a warp holds 32*8/d whole rows.  The RMS is a shuffle reduction inside the
// row's lanes, and the rotation partner of a lane's 8 elements (e +- rd/2) sits in
// the lane rd/16 away within the same row.
template <int D>
__global__ void __launch_bounds__(256) qk_prologue_bf16_kernel(const __grid_constant__ ProloguePlan p) {
    pdl_launch_dependents();  // the attention kernel may start its own prologue now
    // lanes read different frequencies: from shared memory, not the (serialising) parameter bank
    __shared__ float inv_freq[kMaxRotaryHalf];
    if (threadIdx.x < kMaxRotaryHalf) inv_freq[threadIdx.x] = p.inv_freq[threadIdx.x];
    __syncthreads();
    constexpr int LPR = D / 8;        // lanes per row
    constexpr int RPW = 32 / LPR;     // rows per warp
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR;       // this lane's 8-element block within the row
    const int64_t r = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW + lane / LPR;
    const int64_t n_rows = (int64_t)p.B * p.S * p.n_heads;
    const bool live = r < n_rows;
    const int64_t rr = live ? r : 0;
    const int hd = (int)(rr % p.n_heads);
    const int64_t bt = rr / p.n_heads;  // b*S + t
    const int t = (int)(bt % p.S);
    const int b = (int)(bt / p.S);
    const bf16* x = static_cast<const bf16*>(p.x) + bt * p.tok_stride + (int64_t)hd * p.head_stride + 8 * sub;
    const uint4 xv = live ? *reinterpret_cast<const uint4*>(x) : make_uint4(0, 0, 0, 0);
    const uint4 wv = *reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.w) + 8 * sub);
    const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, ws[4] = {wv.x, wv.y, wv.z, wv.w};
    float y[8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = bf16_lo(xs[i]), c = bf16_hi(xs[i]);
        ss = fmaf(a, a, fmaf(c, c, ss));
        y[2 * i] = a * bf16_lo(ws[i]);
        y[2 * i + 1] = c * bf16_hi(ws[i]);
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rinv = rsqrtf(ss / (float)D + p.eps);
    // rotation: block e0 = 8*sub pairs with e0 + half (first half) or e0 - half (second half)
    const int half = p.rd >> 1, dl = half >> 3;  // partner distance in lanes
    const int e0 = 8 * sub;
    const bool first = e0 < half, rot = e0 < p.rd;
    const int src = lane + (first ? dl : -dl);
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __shfl_sync(0xffffffffu, y[i], rot ? src : lane);
    const float posf = live ? (p.pos ? (float)p.pos[bt] : (float)t) : 0.f;
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        float v0 = y[i], v1 = y[i + 1];
        if (rot) {
            const int f = (first ? e0 : e0 - half) + i;
            float s0, c0, s1, c1;
            rope_sincos(posf * inv_freq[f], &s0, &c0);
            rope_sincos(posf * inv_freq[f + 1], &s1, &c1);
            v0 = first ? y[i] * c0 - q[i] * s0 : y[i] * c0 + q[i] * s0;
            v1 = first ? y[i + 1] * c1 - q[i + 1] * s1 : y[i + 1] * c1 + q[i + 1] * s1;
        }
        o[i >> 1] = pack_bf16x2(v0 * rinv, v1 * rinv);
    }
    if (live) {
        bf16* dst = static_cast<bf16*>(p.dst) + (((int64_t)b * p.n_heads + hd) * p.S + t) * D + 8 * sub;
        *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_prologue(const ProloguePlan& p, bool bf16_in, bool bf16_out, cudaStream_t stream) {
    const int64_t n_rows = (int64_t)p.B * p.S * p.n_heads;
    if (bf16_in && bf16_out && p.rd % 16 == 0 && (p.d == 64 || p.d == 128 || p.d == 256)) {
        const int64_t rows_per_block = 8 * (256 / p.d);  // 8 warps, 32*8/d rows each
        const int64_t nb = (n_rows + rows_per_block - 1) / rows_per_block;
        if (nb > 0x7fffffff) return cudaErrorInvalidValue;
        if (p.d == 64) qk_prologue_bf16_kernel<64><<<(unsigned)nb, 256, 0, stream>>>(p);
        else if (p.d == 128) qk_prologue_bf16_kernel<128><<<(unsigned)nb, 256, 0, stream>>>(p);
        else qk_prologue_bf16_kernel<256><<<(unsigned)nb, 256, 0, stream>>>(p);
        return cudaGetLastError();
    }
    const int64_t blocks = (n_rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    const size_t smem = (size_t)kWarpsPerBlock * p.d * sizeof(float);
    if (bf16_in && bf16_out)
        qk_prologue_kernel<bf16, bf16><<<(unsigned)blocks, kWarpsPerBlock * 32, smem, stream>>>(p);
    else if (!bf16_in && !bf16_out)
        qk_prologue_kernel<float, float><<<(unsigned)blocks, kWarpsPerBlock * 32, smem, stream>>>(p);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace gattn
