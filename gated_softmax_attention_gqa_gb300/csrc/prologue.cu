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
#include <algorithm>

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
    // this block's rows are written: the attention kernel may be scheduled once every
    // block has got this far (it still waits for the whole grid before reading them)
    pdl_launch_dependents();
}

// bf16 -> bf16 with rotary_dim % 16 == 0 (the tensor-core path).
//
// A row of D elements is spread over D/8 lanes, one 16-byte load and one 16-byte
// store each, so a warp holds RPW = 32*8/D whole rows at a time.  The RMS is a
// shuffle reduction inside the row's lanes, and the rotation partner of a lane's
// 8 elements (e +- rd/2) sits in the lane rd/16 away within the same row.
//
// A work item is one RoPE position and up to U*RPW of the rows rotated by it: with
// default positions (pos == NULL) that is token t of every batch and head,
// otherwise token t of one batch, every head.  The lane's 8 (cos, sin) pairs are
// computed once and reused for all of those rows, so the sine/cosine work is per
// position rather than per row; the U row loads are issued together before any
// arithmetic.
//
// The grid is one resident wave (the launch sizes it to the blocks the SMs hold at
// once) and each warp walks the items with a stride.  The attention kernel launched
// behind it (programmatic dependent launch) may then be scheduled from the start:
// its CTAs take an SM only as this pass's blocks leave it, never ahead of blocks of
// this pass still waiting to run.
template <int D>
__global__ void __launch_bounds__(256) qk_prologue_bf16_kernel(const __grid_constant__ ProloguePlan p,
                                                               uint32_t n_items, uint32_t n_tau, int nb) {
    constexpr int LPR = D / 8;        // lanes per row
    constexpr int RPW = 32 / LPR;     // rows per warp step
    constexpr int U = 4;              // warp steps per item
    pdl_launch_dependents();  // the attention kernel may start its own prologue now
    // lanes read different frequencies: from shared memory, not the (serialising) parameter bank
    __shared__ float inv_freq[kMaxRotaryHalf];
    if (threadIdx.x < kMaxRotaryHalf) inv_freq[threadIdx.x] = p.inv_freq[threadIdx.x];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR;       // this lane's 8-element block within the row
    const int e0 = 8 * sub;
    const uint4 wv = *reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.w) + e0);
    const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
    const uint32_t n_rows = (uint32_t)nb * (uint32_t)p.n_heads;  // rows sharing a position
    const uint32_t stride = gridDim.x * (blockDim.x >> 5);
    for (uint32_t item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < n_items; item += stride) {
        // the position this warp rotates by: tau = t (default positions) or b*S + t.
        // Consecutive warps take consecutive positions of the same chunk of rows, so a
        // CTA reads and writes contiguous runs of every (batch, head) plane.
        const uint32_t chunk = item / n_tau;
        const uint32_t tau = item - chunk * n_tau;
        const int t = p.pos ? (int)(tau % (uint32_t)p.S) : (int)tau;
        const int b_fixed = p.pos ? (int)(tau / (uint32_t)p.S) : 0;
        const float posf = p.pos ? (float)p.pos[tau] : (float)tau;
        const int half = p.rd >> 1, dl = half >> 3;  // rotation partner distance in lanes
        const bool first = e0 < half, rot = e0 < p.rd;
        const int src = lane + (first ? dl : -dl);
        float cs[8], sn[8];
    #pragma unroll
        for (int i = 0; i < 8; ++i) {
            cs[i] = 1.f;
            sn[i] = 0.f;
            if (rot) rope_sincos(posf * inv_freq[(first ? e0 : e0 - half) + i], &sn[i], &cs[i]);
        }
        uint4 xv[U];
        int rb[U], rh[U];
        bool live[U];
    #pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t r = (chunk * U + u) * RPW + (uint32_t)(lane / LPR);
            live[u] = r < n_rows;
            const uint32_t rr = live[u] ? r : 0u;
            rh[u] = (int)(rr % (uint32_t)p.n_heads);
            rb[u] = p.pos ? b_fixed : (int)(rr / (uint32_t)p.n_heads);
            const bf16* x = static_cast<const bf16*>(p.x) + ((int64_t)rb[u] * p.S + t) * p.tok_stride +
                            (int64_t)rh[u] * p.head_stride + e0;
            xv[u] = live[u] ? __ldcs(reinterpret_cast<const uint4*>(x)) : make_uint4(0, 0, 0, 0);
        }
    #pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t xs[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
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
            float q[8];
    #pragma unroll
            for (int i = 0; i < 8; ++i) q[i] = __shfl_sync(0xffffffffu, y[i], rot ? src : lane);
            uint32_t o[4];
    #pragma unroll
            for (int i = 0; i < 8; i += 2) {
                // first half: x*cos - partner*sin; second half: x*cos + partner*sin (cs=1, sn=0 past rd)
                const float s0 = first ? -sn[i] : sn[i], s1 = first ? -sn[i + 1] : sn[i + 1];
                const float v0 = fmaf(y[i], cs[i], q[i] * s0);
                const float v1 = fmaf(y[i + 1], cs[i + 1], q[i + 1] * s1);
                o[i >> 1] = pack_bf16x2(v0 * rinv, v1 * rinv);
            }
            if (live[u]) {
                bf16* dst = static_cast<bf16*>(p.dst) + (((int64_t)rb[u] * p.n_heads + rh[u]) * p.S + t) * D + e0;
                *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

template <int D>
cudaError_t launch_bf16(const ProloguePlan& p, cudaStream_t stream) {
    constexpr int RPW = 32 / (D / 8);
    constexpr int U = 4;
    const int64_t n_tau = p.pos ? (int64_t)p.B * p.S : (int64_t)p.S;
    const int64_t rows_per_tau = p.pos ? (int64_t)p.n_heads : (int64_t)p.B * p.n_heads;
    const int64_t n_chunks = (rows_per_tau + U * RPW - 1) / (U * RPW);
    const int64_t n_items = n_tau * n_chunks;
    if (rows_per_tau >= 0x7fffffffLL || n_items + 8 >= 0x7fffffffLL) return cudaErrorInvalidValue;
    // one resident wave at most (see the kernel)
    static int per_sm[3] = {0, 0, 0};
    int& occ = per_sm[D == 64 ? 0 : D == 128 ? 1 : 2];
    if (occ == 0) {
        int dev = 0, n_sm = 0, b = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, qk_prologue_bf16_kernel<D>, 256, 0) != cudaSuccess)
            return cudaErrorInvalidValue;
        occ = (b > 0 ? b : 1) * n_sm;
    }
    const int64_t blocks = std::min<int64_t>((n_items + 7) / 8, occ);
    qk_prologue_bf16_kernel<D><<<(unsigned)blocks, 256, 0, stream>>>(p, (uint32_t)n_items, (uint32_t)n_tau,
                                                                        p.pos ? 1 : p.B);
    return cudaGetLastError();
}

// One CTA per query tile of the table: the tile's 128 tokens get their position
// within the sequence and the sequence's first token.
__global__ void __launch_bounds__(128) varlen_positions_kernel(const int4* tiles, int32_t* pos, int32_t* tok_start) {
    const int4 e = tiles[blockIdx.x];  // start, length, tile, sequence
    const int t = e.z * 128 + (int)threadIdx.x;
    if (t < e.y) {
        pos[e.x + t] = t;
        tok_start[e.x + t] = e.x;
    }
}

}  // namespace

cudaError_t launch_varlen_positions(const int4* tiles, int n_tiles, int32_t* pos, int32_t* tok_start,
                                    cudaStream_t stream) {
    if (n_tiles <= 0) return cudaSuccess;
    varlen_positions_kernel<<<(unsigned)n_tiles, 128, 0, stream>>>(tiles, pos, tok_start);
    return cudaGetLastError();
}

cudaError_t launch_prologue(const ProloguePlan& p, bool bf16_in, bool bf16_out, cudaStream_t stream) {
    const int64_t n_rows = (int64_t)p.B * p.S * p.n_heads;
    if (n_rows == 0) return cudaSuccess;
    if (bf16_in && bf16_out && p.rd % 16 == 0 && n_rows < 0x40000000LL) {
        if (p.d == 64) return launch_bf16<64>(p, stream);
        if (p.d == 128) return launch_bf16<128>(p, stream);
        if (p.d == 256) return launch_bf16<256>(p, stream);
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
