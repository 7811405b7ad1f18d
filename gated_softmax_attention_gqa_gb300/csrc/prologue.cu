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
// A row of D elements is spread over D/16 lanes: the first rd/16 lanes of a row
// each own 8 rotation pairs (x_i and x_{i+rd/2}, i in [8k, 8k+8)), the others 16
// consecutive unrotated features, as two 16-byte loads and stores each -- so a lane
// has both members of every pair it rotates, and a warp step covers RPW = 512/D
// rows.  The RMS is a shuffle reduction inside the row's lanes.
//
// A work item is RPW consecutive tokens of one batch and every head (plane) of the
// tensor: the RPW rows of a warp step are those tokens of one head, and the warp
// walks the heads, PF of them loaded ahead.  A lane's token is fixed for the item,
// so its 8 (cos, sin) pairs -- folded with its norm weights into the four factors
// of the rotation -- are computed once and serve every head, and the item reads
// whole token rows (all heads) and writes RPW consecutive rows of each head's
// plane.
//
// The grid is one resident wave (the launch sizes it to the blocks the SMs hold at
// once) and each warp walks the items with a stride.  The attention kernel launched
// behind it (programmatic dependent launch) may then be scheduled from the start:
// its CTAs take an SM only as this pass's blocks leave it, never ahead of blocks of
// this pass still waiting to run.
template <int D>
__global__ void __launch_bounds__(256) qk_prologue_bf16_kernel(const __grid_constant__ ProloguePlan p,
                                                                  uint32_t n_items, uint32_t n_tblocks) {
    constexpr int LPR = D / 16;       // lanes per row
    constexpr int RPW = 32 / LPR;     // rows (tokens) per warp step
    constexpr int PF = 4;             // heads loaded ahead
    pdl_launch_dependents();  // the attention kernel may start its own prologue now
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR;                    // this lane's place within the row
    const int rsub = lane / LPR;                   // this lane's token within the item
    const int npl = p.rd >> 4;                     // pair lanes per row
    const bool rot = sub < npl;
    // this lane's two 8-element blocks: x_i and x_{i+rd/2}, or 16 unrotated features
    const int o1 = rot ? 8 * sub : p.rd + 16 * (sub - npl);
    const int o2 = rot ? o1 + (p.rd >> 1) : o1 + 8;
    const int nh = p.n_heads;
    const uint32_t stride = gridDim.x * (blockDim.x >> 5);
    for (uint32_t item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < n_items; item += stride) {
        const int b = (int)(item / n_tblocks);
        const int t = (int)(item - (uint32_t)b * n_tblocks) * RPW + rsub;
        const bool live = t < p.S;
        const int tc = live ? t : 0;
        const bf16* x0 = static_cast<const bf16*>(p.x) + ((int64_t)b * p.S + tc) * p.tok_stride;
        bf16* d0 = static_cast<bf16*>(p.dst) + ((int64_t)b * nh * p.S + tc) * D;
        const int64_t dplane = (int64_t)p.S * D;  // from one head's plane to the next
        uint4 xa[PF], xb[PF];
        auto load = [&](int j, int hh) {
            const bf16* x = x0 + (int64_t)hh * p.head_stride;
            const bool ok = live && hh < nh;
            xa[j] = ok ? __ldcs(reinterpret_cast<const uint4*>(x + o1)) : make_uint4(0, 0, 0, 0);
            xb[j] = ok ? __ldcs(reinterpret_cast<const uint4*>(x + o2)) : make_uint4(0, 0, 0, 0);
        };
#pragma unroll
        for (int j = 0; j < PF; ++j) load(j, j);
        // this lane's rotation at its token's position, with the norm weights w (of x_i)
        // and w' (of x_{i+rd/2}): lo = (x_i ka + x_{i+rd/2} kb) rinv, hi = (x_{i+rd/2} kc +
        // x_i kd) rinv with ka = w cos, kb = -w' sin, kc = w' cos, kd = w sin (cos = 1,
        // sin = 0 for unrotated features)
        float2 ka[4], kb[4], kc[4], kd[4];
        {
            float wa[8], wb[8];
            unpack8(*reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.w) + o1), wa);
            unpack8(*reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.w) + o2), wb);
            const float posf = p.pos ? (float)p.pos[(int64_t)b * p.S + tc] : (float)tc;
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                float2 s2 = make_float2(0.f, 0.f), c2 = make_float2(1.f, 1.f);
                if (rot)
                    rope_sincos2(mul2(make_float2(posf, posf),
                                      make_float2(p.inv_freq[8 * sub + i], p.inv_freq[8 * sub + i + 1])),
                                 &s2, &c2);
                const float2 w1 = make_float2(wa[i], wa[i + 1]), w2 = make_float2(wb[i], wb[i + 1]);
                ka[i >> 1] = mul2(w1, c2);
                kb[i >> 1] = mul2(w2, make_float2(-s2.x, -s2.y));
                kc[i >> 1] = mul2(w2, c2);
                kd[i >> 1] = mul2(w1, s2);
            }
        }
        for (int h0 = 0; h0 < nh; h0 += PF) {
#pragma unroll
            for (int j = 0; j < PF; ++j) {
                const int h = h0 + j;  // warp-uniform
                if (h >= nh) break;
                float a[8], bv[8];
                unpack8(xa[j], a);
                unpack8(xb[j], bv);
                load(j, h + PF);  // the head PF further on, into the registers just read
                float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    ss2 = fma2(make_float2(a[i], a[i + 1]), make_float2(a[i], a[i + 1]), ss2);
                    ss2 = fma2(make_float2(bv[i], bv[i + 1]), make_float2(bv[i], bv[i + 1]), ss2);
                }
                float ss = ss2.x + ss2.y;
#pragma unroll
                for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float rinv = rsqrtf(ss / (float)D + p.eps);
                const float2 r2 = make_float2(rinv, rinv);
                uint32_t lo[4], hi[4];
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const float2 av = make_float2(a[i], a[i + 1]), bw = make_float2(bv[i], bv[i + 1]);
                    const float2 l = mul2(fma2(av, ka[i >> 1], mul2(bw, kb[i >> 1])), r2);
                    const float2 r = mul2(fma2(bw, kc[i >> 1], mul2(av, kd[i >> 1])), r2);
                    lo[i >> 1] = pack_bf16x2(l.x, l.y);
                    hi[i >> 1] = pack_bf16x2(r.x, r.y);
                }
                if (live) {
                    bf16* d = d0 + (int64_t)h * dplane;
                    *reinterpret_cast<uint4*>(d + o1) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    *reinterpret_cast<uint4*>(d + o2) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                }
            }
        }
    }
}

template <int D>
cudaError_t launch_bf16(const ProloguePlan& p, cudaStream_t stream) {
    constexpr int RPW = 32 / (D / 16);
    const int64_t n_tblocks = (p.S + RPW - 1) / RPW;
    const int64_t n_items = (int64_t)p.B * n_tblocks;
    if (n_items + 2048 >= 0x7fffffffLL) return cudaErrorInvalidValue;
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
    qk_prologue_bf16_kernel<D><<<(unsigned)blocks, 256, 0, stream>>>(p, (uint32_t)n_items, (uint32_t)n_tblocks);
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
