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

}  // namespace

cudaError_t launch_prologue(const ProloguePlan& p, bool bf16_in, bool bf16_out, cudaStream_t stream) {
    const int64_t n_rows = (int64_t)p.B * p.S * p.n_heads;
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
