// decode.cu -- one decode step of gated GQA attention against a bf16 KV cache.
//
// Each sequence's newest query (at position seqlens[b]-1) attends to every
// cached key of its KV group; the cache holds K already normed and rotated and
// raw V ("Multi-head attention and GQA" chapter, section "拼接各头 → 用 W_O
// 投影": K and V are cached per token, Q is not; the new query dots every
// cached key).  The step is bound by reading the cache from HBM, so the design
// goal is to keep every SM streaming:
//
//   decode_split_kernel  persistent, one CTA per SM.  The cache of all
//       (sequence, group) pairs is cut into 64-key tiles and the global tile
//       list is divided into equal contiguous ranges, one per CTA, so every SM
//       streams the same number of bytes whatever the length mix.  A producer
//       warp feeds K and V tiles through a TMA ring (128 B swizzle); four
//       consumer warps each take 16 keys of every tile.  The H/G query heads of
//       a group are packed as the rows of one m16n8k16 tile (S = Q K^T), and
//       O^T += V^T P^T reuses the S accumulator registers directly as the B
//       operand.  Warp-level mma keeps the arithmetic far off the critical path
//       of this memory-bound loop.  At the end of each (sequence, group) piece a
//       warp writes its partial softmax state (max, sum, unnormalised O).
//   decode_combine_kernel  one CTA per (sequence, group), one warp per query
//       head: merges the partial states of the CTAs that covered it (all the
//       loads of eight slots in flight together, no barrier), divides by the sum
//       and applies sigmoid(gate), writing bf16 [B, H*d].
#include "common.cuh"
#include "internal.h"

namespace gattn {
namespace {

constexpr int BT = kDecodeTileKeys;  // keys per tile
constexpr int NCW = kDecodeConsumerWarps;
constexpr int MAXB = 2048;           // sequences per call

template <int D>
struct DecCfg {
    static constexpr int KCH = D / 64;
    static constexpr int CHUNK_BYTES = BT * 128;
    static constexpr int TILE_BYTES = BT * D * 2;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile then V tile
    static constexpr int NS = (196608 / STAGE_BYTES) > 8 ? 8 : (196608 / STAGE_BYTES);
    static constexpr int THREADS = 32 * (NCW + 1);
    static constexpr int OFF_PB = NS * STAGE_BYTES;            // int [MAXB + 1] tile prefix
    static constexpr int OFF_RED = OFF_PB + (MAXB + 1) * 4;    // int [8] scan scratch
    static constexpr int OFF_BAR = (OFF_RED + 8 * 4 + 7) & ~7;
    static constexpr int OFF_MISC = OFF_BAR + 2 * NS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
};

__device__ __forceinline__ int seq_tiles(int L, int Lmax) { return (L >= 1 && L <= Lmax) ? (L + BT - 1) / BT : 0; }

// Exclusive prefix of per-sequence tile counts into pb[0..B]; all threads.
__device__ void tile_prefix(const int32_t* seqlens, int B, int Lmax, int* pb, int* red) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5, nwarp = nthr >> 5;
    int carry = 0;
    for (int base = 0; base < B; base += nthr) {
        const int i = base + tid;
        int v = i < B ? seq_tiles(seqlens[i], Lmax) : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        if (lane == 31) red[warp] = v;
        __syncthreads();
        int before = carry;
        for (int w = 0; w < warp; ++w) before += red[w];
        if (i < B) pb[i + 1] = before + v;
        int total = 0;
        for (int w = 0; w < nwarp; ++w) total += red[w];
        __syncthreads();
        carry += total;
    }
    if (tid == 0) pb[0] = 0;
    __syncthreads();
}

// Walks the global tile list: tile u belongs to sequence b, group g, local tile i.
struct TileWalker {
    int b, g, i, nt;
    __device__ void seek(int64_t u, const int* pb, int B, int G) {
        int lo = 0, hi = B - 1;  // largest b with G*pb[b] <= u
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)G * pb[mid] <= u) lo = mid; else hi = mid - 1;
        }
        b = lo;
        nt = pb[b + 1] - pb[b];
        const int64_t rel = u - (int64_t)G * pb[b];
        g = (int)(rel / nt);
        i = (int)(rel % nt);
    }
    __device__ void next(const int* pb, int B, int G) {
        if (++i < nt) return;
        i = 0;
        if (++g < G) return;
        g = 0;
        do { ++b; } while (b < B && pb[b + 1] == pb[b]);
        if (b < B) nt = pb[b + 1] - pb[b];
    }
};

template <int D>
__global__ void __launch_bounds__(DecCfg<D>::THREADS, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ DecodeParams p) {
    using C = DecCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int* pb = reinterpret_cast<int*>(smem + C::OFF_PB);
    const uint32_t bar_full = sbase + C::OFF_BAR, bar_empty = bar_full + 8 * C::NS;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
    pdl_launch_dependents();  // the combine kernel may become resident; it waits for this grid to finish

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, NCW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == NCW && lane == 0) tma_prefetch_desc(&tm);
    tile_prefix(p.seqlens, p.B, p.Lmax, pb, reinterpret_cast<int*>(smem + C::OFF_RED));  // ends with a block barrier

    const int64_t T = (int64_t)p.G * pb[p.B];
    const int64_t u_begin = (int64_t)blockIdx.x * T / p.n_ctas;
    const int64_t u_end = (int64_t)(blockIdx.x + 1) * T / p.n_ctas;
    const int r = p.H / p.G;

    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && u_begin < u_end) {
            TileWalker wk;
            wk.seek(u_begin, pb, p.B, p.G);
            const bool paged = p.block_table != nullptr;
            const int64_t plane = paged ? (int64_t)p.num_pages * p.G * p.page_size : (int64_t)p.B * p.G * p.Lmax;
            int cached_b = -1, cached_slot = -1, page = 0;  // the last block table entry read
            int n = 0;
            for (int64_t u = u_begin; u < u_end; ++u, ++n, wk.next(pb, p.B, p.G)) {
                const int st = n % C::NS;
                if (n >= C::NS &&
                    !mbar_wait(bar_empty + 8 * st, ((uint32_t)(n / C::NS) & 1u) ^ 1u, abort_flag, p.status))
                    break;
                mbar_arrive_expect_tx(bar_full + 8 * st, C::STAGE_BYTES);
                int rowk;
                if (paged) {
                    const int key0 = wk.i * BT, slot = key0 / p.page_size;
                    if (wk.b != cached_b || slot != cached_slot) {
                        page = p.block_table[(int64_t)wk.b * p.max_pages + slot];
                        if (page < 0 || page >= p.num_pages) {
                            atomicOr(p.status, GATTN_DEVICE_BAD_PAGE);
                            page = 0;
                        }
                        cached_b = wk.b;
                        cached_slot = slot;
                    }
                    rowk = (int)(((int64_t)page * p.G + wk.g) * p.page_size + key0 % p.page_size);
                } else {
                    rowk = (int)(((int64_t)wk.b * p.G + wk.g) * p.Lmax + (int64_t)wk.i * BT);
                }
                const int rowv = (int)(rowk + plane);
                const uint32_t dst = sbase + st * C::STAGE_BYTES;
#pragma unroll
                for (int c = 0; c < C::KCH; ++c) tma_load_2d(dst + c * C::CHUNK_BYTES, &tm, bar_full + 8 * st, c * 64, rowk);
#pragma unroll
                for (int c = 0; c < C::KCH; ++c)
                    tma_load_2d(dst + C::TILE_BYTES + c * C::CHUNK_BYTES, &tm, bar_full + 8 * st, c * 64, rowv);
            }
            for (int j = n > C::NS ? n - C::NS : 0; j < n; ++j)
                mbar_wait_drain(bar_full + 8 * (j % C::NS), (uint32_t)(j / C::NS) & 1u, p.status);
        }
        __syncwarp();
    } else if (u_begin < u_end) {
        // ------------------------------------------------------------ consumers
        const int hrow = lane >> 2;  // head row of the S accumulator
        const int quad = lane & 3;
        const float sl2 = p.scale_log2;
        const int half = p.rd >> 1;
        uint32_t qa0[D / 16], qa2[D / 16];
        float oacc[D / 16][4];
        float m_run = -INFINITY, l_part = 0.f;
        int L = 0;
        TileWalker wk;
        wk.seek(u_begin, pb, p.B, p.G);
        int n = 0;
        for (int64_t u = u_begin; u < u_end; ++u, ++n, wk.next(pb, p.B, p.G)) {
            if (u == u_begin || wk.i == 0) {
                // -------- start of a (sequence, group) piece: this lane's share of the rotated queries.
                // Lane (hrow, quad) holds, for head hrow of the group, the element pairs
                // e0 = 8f + 2*quad (f = 0..D/8-1), exactly the A-fragment elements it feeds
                // to S = Q K^T.  With rotary_dim a multiple of 16 the rotation partner of
                // e0 (e0 +- rotary_dim/2) is another pair of the same lane.
                L = p.seqlens[wk.b];
                const float posf = (float)(L - 1);
                float y[D / 8][2];
                float ss = 0.f;
                const bool live = hrow < r;
                const bf16* qrow = static_cast<const bf16*>(p.q) + ((int64_t)wk.b * p.H + wk.g * r + (live ? hrow : 0)) * D;
                const bf16* wq = static_cast<const bf16*>(p.qnorm_w);
#pragma unroll
                for (int f = 0; f < D / 8; ++f) {
                    const int e0 = 8 * f + 2 * quad;
                    const uint32_t xv = live ? *reinterpret_cast<const uint32_t*>(qrow + e0) : 0u;
                    const uint32_t wv = *reinterpret_cast<const uint32_t*>(wq + e0);
                    const float x0 = bf16_lo(xv), x1 = bf16_hi(xv);
                    ss = fmaf(x0, x0, fmaf(x1, x1, ss));
                    y[f][0] = x0 * bf16_lo(wv);
                    y[f][1] = x1 * bf16_hi(wv);
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                const float rinv = rsqrtf(ss / (float)D + p.eps);
                const int hf = half >> 3;  // rotation partner distance in pairs
#pragma unroll
                for (int f = 0; f < D / 8; ++f) {
                    const int e0 = 8 * f + 2 * quad;
                    float o0 = y[f][0], o1 = y[f][1];
                    if (e0 < p.rd) {
                        const bool first = e0 < half;
                        const int fp = first ? f + hf : f - hf;
                        const int i0 = first ? e0 : e0 - half;
                        float s0, c0, s1, c1;
                        rope_sincos(posf * p.inv_freq[i0], &s0, &c0);
                        rope_sincos(posf * p.inv_freq[i0 + 1], &s1, &c1);
                        float q0 = 0.f, q1 = 0.f;
#pragma unroll
                        for (int ff = 0; ff < D / 8; ++ff)
                            if (ff == fp) { q0 = y[ff][0]; q1 = y[ff][1]; }
                        o0 = first ? y[f][0] * c0 - q0 * s0 : y[f][0] * c0 + q0 * s0;
                        o1 = first ? y[f][1] * c1 - q1 * s1 : y[f][1] * c1 + q1 * s1;
                    }
                    const uint32_t pk = pack_bf16x2(o0 * rinv, o1 * rinv);
                    if (f & 1) qa2[f >> 1] = pk; else qa0[f >> 1] = pk;
                }
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt)
                    oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
                m_run = -INFINITY;
                l_part = 0.f;
            }

            const int st = n % C::NS;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(bar_full + 8 * st, (uint32_t)(n / C::NS) & 1u, abort_flag, p.status)))
                break;
            const uint32_t kt = sbase + st * C::STAGE_BYTES;
            const uint32_t vt = kt + C::TILE_BYTES;
            const int key0 = wk.i * BT + 16 * warp;  // first key of this warp's slice
            const uint32_t lrow = 16 * warp + (lane & 7) + ((lane >> 4) << 3);
            const uint32_t lsel = (lane >> 3) & 1;

            // ---- S = Q K^T over this warp's 16 keys
            float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t c8 = 2 * kk + lsel;
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(kt + (c8 >> 3) * C::CHUNK_BYTES + sw128_offset(lrow, c8 & 7), b0, b1, b2, b3);
                mma_bf16_16816(sacc[0], qa0[kk], 0u, qa2[kk], 0u, b0, b1);
                mma_bf16_16816(sacc[1], qa0[kk], 0u, qa2[kk], 0u, b2, b3);
            }
            // ---- online softmax (per head row); keys >= L are masked
            float x[2][2];
            float tmax = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = key0 + nt * 8 + 2 * quad + e;
                    x[nt][e] = key < L ? sacc[nt][e] * sl2 : -INFINITY;
                    tmax = fmaxf(tmax, x[nt][e]);
                }
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
            const float m_new = fmaxf(m_run, tmax);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = ex2_approx(m_run - m_use);
            float pr[2][2];
            float psum = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    pr[nt][e] = ex2_approx(x[nt][e] - m_use);
                    psum += pr[nt][e];
                }
            l_part = l_part * alpha + psum;
            m_run = m_new;
            const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * quad);
            const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * quad + 4);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                oacc[mt][0] *= a_lo;
                oacc[mt][1] *= a_hi;
                oacc[mt][2] *= a_lo;
                oacc[mt][3] *= a_hi;
            }
            const uint32_t pb0 = pack_bf16x2(pr[0][0], pr[0][1]);
            const uint32_t pb1 = pack_bf16x2(pr[1][0], pr[1][1]);

            // ---- cached rows past the sequence end may hold anything: zero this warp's V rows there
            if (key0 + 16 > L) {
                const int first = L - key0 > 0 ? L - key0 : 0;
                uint8_t* vrow_base = smem + st * C::STAGE_BYTES + C::TILE_BYTES;
                for (int idx = lane; idx < (16 - first) * C::KCH * 8; idx += 32) {
                    const int rr = first + idx / (C::KCH * 8);
                    const int cc = idx % (C::KCH * 8);
                    const uint32_t row = 16 * warp + rr;
                    *reinterpret_cast<uint4*>(vrow_base + (cc >> 3) * C::CHUNK_BYTES + sw128_offset(row, cc & 7)) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- O^T += V^T P^T
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const uint32_t c8 = 2 * mt + lsel;
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4_trans(vt + (c8 >> 3) * C::CHUNK_BYTES + sw128_offset(lrow, c8 & 7), a0, a1, a2, a3);
                mma_bf16_16816(oacc[mt], a0, a1, a2, a3, pb0, pb1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * st);

            // ---- end of this CTA's piece of the (sequence, group): write the partial state
            if (wk.i == wk.nt - 1 || u == u_end - 1) {
                float l_tot = l_part;
                l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 1);
                l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 2);
                const int64_t seg = (int64_t)wk.b * p.G + wk.g;
                const int64_t slot = ((int64_t)blockIdx.x + seg) * NCW + warp;
                float* ps = p.part + slot * (int64_t)(2 * r + r * D);
                if (quad == 0 && hrow < r) {
                    ps[hrow] = m_run;
                    ps[r + hrow] = l_tot;
                }
                const int hA = 2 * quad, hB = 2 * quad + 1;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    const int d0 = mt * 16 + hrow;
                    if (hA < r) {
                        ps[2 * r + hA * D + d0] = oacc[mt][0];
                        ps[2 * r + hA * D + d0 + 8] = oacc[mt][2];
                    }
                    if (hB < r) {
                        ps[2 * r + hB * D + d0] = oacc[mt][1];
                        ps[2 * r + hB * D + d0 + 8] = oacc[mt][3];
                    }
                }
            }
        }
    }
    __syncthreads();
}

// Merge the partial states of one (sequence, group) and apply the gate.  The
// CTAs whose tile ranges overlap this (sequence, group) each left one partial
// state per consumer warp; their (max, sum) pairs are first turned into merge
// weights w_s = 2^(m_s - max_s m_s) in shared memory, then every output element is
// sum_s w_s O_s / sum_s w_s l_s -- independent, coalesced loads across the slots.
template <int D>
__global__ void __launch_bounds__(256, 1) decode_combine_kernel(const __grid_constant__ DecodeParams p) {
    // one CTA per (sequence, group), one warp per query head of the group; lane l
    // owns columns [l DPL, l DPL + DPL) of the head's output
    constexpr int DPL = D / 32;
    constexpr int CH = 8;  // slots whose loads are in flight together
    const int b = blockIdx.x / p.G, g = blockIdx.x % p.G;
    const int r = p.H / p.G;
    const int lane = threadIdx.x & 31, hl = threadIdx.x >> 5;
    const int h = g * r + hl;
    // tiles before this sequence, and in total
    int before = 0, total = 0;
    for (int i = lane; i < p.B; i += 32) {
        const int nt = seq_tiles(p.seqlens[i], p.Lmax);
        total += nt;
        if (i < b) before += nt;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, o);
        total += __shfl_xor_sync(0xffffffffu, total, o);
    }
    const int L = p.seqlens[b];
    const int nt = seq_tiles(L, p.Lmax);
    if (nt == 0) {
        if (lane == 0 && hl == 0 && g == 0) atomicOr(p.status, GATTN_DEVICE_BAD_SEQLEN);
        return;
    }
    const int64_t T = (int64_t)p.G * total, N = p.n_ctas;
    const int64_t u0 = (int64_t)p.G * before + (int64_t)g * nt, u1 = u0 + nt - 1;
    auto cmax = [&](int64_t x) -> int64_t {  // last CTA whose range starts at or before tile x
        const int64_t c = ((x + 1) * N - 1) / T;
        return c < N - 1 ? c : N - 1;
    };
    const int64_t c_first = cmax(u0);
    const int n_slots = (int)(cmax(u1) - c_first + 1) * NCW;
    const int64_t seg = (int64_t)b * p.G + g;
    const int slot_floats = 2 * r + r * D;
    const float* part0 = p.part + (c_first + seg) * NCW * (int64_t)slot_floats;  // slot s at part0 + s*slot_floats
    // whether slot s holds a state of this (sequence, group): its CTA's tile range
    // meets the piece (a slot of a CTA that covered none of it may hold stale data)
    auto covers = [&](int sl) -> bool {
        const int64_t c = c_first + sl / NCW;
        const int64_t s0 = c * T / N, s1 = (c + 1) * T / N;
        return s0 < s1 && s0 <= u1 && s1 > u0;
    };
    // gate logits of this lane's columns: [B,H,d] elementwise, [B,H] headwise, [B,d] head-shared
    const int layout = gate_layout(p.gate_mode);
    float gl[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
        const int e = lane * DPL + k;
        gl[k] = 0.f;
        if (layout == GATTN_GATE_ELEMENTWISE)
            gl[k] = __bfloat162float(static_cast<const bf16*>(p.gate)[((int64_t)b * p.H + h) * D + e]);
        else if (layout == GATTN_GATE_HEADWISE)
            gl[k] = __bfloat162float(static_cast<const bf16*>(p.gate)[(int64_t)b * p.H + h]);
        else if (layout == GATTN_GATE_HEAD_SHARED)
            gl[k] = __bfloat162float(static_cast<const bf16*>(p.gate)[(int64_t)b * D + e]);
    }

    // everything above reads only the inputs; the partial states come from the split kernel
    pdl_wait_prerequisites();
    // o = sum_s w_s O_s / sum_s w_s l_s with w_s = 2^(m_s - max_s m_s), the slots taken
    // CH at a time with every load of a group in flight together; a later group with a
    // larger maximum rescales what is summed so far (never the case for pieces
    // covered by at most CH / NCW CTAs, where this is one pass with the common max)
    float m_run = -INFINITY, den = 0.f, num[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) num[k] = 0.f;
    for (int sl0 = 0; sl0 < n_slots; sl0 += CH) {
        float ms[CH], ls[CH], os[CH][DPL];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const int sl = sl0 + j;
            const bool live = sl < n_slots && covers(sl);
            const float* ps = part0 + (int64_t)(live ? sl : 0) * slot_floats;
            ms[j] = live ? ps[hl] : -INFINITY;
            ls[j] = live ? ps[r + hl] : 0.f;
            const float* po = ps + 2 * r + hl * D + lane * DPL;
            if constexpr (DPL % 2 == 0) {
#pragma unroll
                for (int k = 0; k < DPL; k += 2) {
                    const float2 v = live ? *reinterpret_cast<const float2*>(po + k) : make_float2(0.f, 0.f);
                    os[j][k] = v.x;
                    os[j][k + 1] = v.y;
                }
            } else {
#pragma unroll
                for (int k = 0; k < DPL; ++k) os[j][k] = live ? po[k] : 0.f;
            }
        }
        float mx = m_run;
#pragma unroll
        for (int j = 0; j < CH; ++j) mx = fmaxf(mx, ms[j]);
        if (mx == -INFINITY) continue;  // no state in this group yet
        const float keep = m_run == -INFINITY ? 0.f : ex2_approx(m_run - mx);
        den *= keep;
#pragma unroll
        for (int k = 0; k < DPL; ++k) num[k] *= keep;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const float wgt = ms[j] == -INFINITY ? 0.f : ex2_approx(ms[j] - mx);
            den += wgt != 0.f ? wgt * ls[j] : 0.f;
#pragma unroll
            for (int k = 0; k < DPL; ++k) num[k] += wgt != 0.f ? wgt * os[j][k] : 0.f;
        }
        m_run = mx;
    }
    bf16 ob[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
        const float gv = layout == GATTN_GATE_NONE ? 1.f : gate_act(gl[k], sigmoidf_dev(gl[k]), p.gate_mode);
        const float o = num[k] / den;
        ob[k] = __float2bfloat16_rn(gate_additive(p.gate_mode) ? o + gv : o * gv);
    }
    bf16* orow = static_cast<bf16*>(p.out) + ((int64_t)b * p.H + h) * D + lane * DPL;
#pragma unroll
    for (int k = 0; k < DPL; ++k) orow[k] = ob[k];
}

template <int D>
cudaError_t launch_dec(const DecodeParams& p, const CUtensorMap& tm, cudaStream_t stream, cudaEvent_t ev_start,
                       cudaEvent_t ev_stop) {
    using C = DecCfg<D>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(decode_split_kernel<D>), C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    if (ev_start) cudaEventRecord(ev_start, stream);
    decode_split_kernel<D><<<p.n_ctas, C::THREADS, C::SMEM_ALLOC, stream>>>(tm, p);
    e = cudaGetLastError();
    if (ev_stop) cudaEventRecord(ev_stop, stream);
    if (e != cudaSuccess) return e;
    // programmatic serialisation: the combine CTAs become resident while the split
    // kernel drains and wait on its completion inside the kernel
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * p.G));
    cfg.blockDim = dim3(32 * (p.H / p.G));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, p);
}

// The new token's K and V into the cache before the step reads it: one row of D
// elements per (sequence, group), spread over D/8 lanes (16-byte loads and
// stores); the RMS is a shuffle reduction over the row's lanes, and the rotation
// partner of a lane's 8 features (e +- rd/2) sits rd/16 lanes away.  Sequences
// whose length is outside [1, Lmax] are left alone (the step reports them).
template <int D>
__global__ void __launch_bounds__(256) decode_append_kernel(const __grid_constant__ AppendParams p) {
    constexpr int LPR = D / 8, RPW = 32 / LPR;
    const int lane = threadIdx.x & 31;
    const int64_t row = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * RPW + lane / LPR;  // b * G + g
    const bool in_range = row < (int64_t)p.B * p.G;
    const int b = in_range ? (int)(row / p.G) : 0;
    const int L = in_range ? p.seqlens[b] : 0;
    const bool live = in_range && L >= 1 && L <= p.Lmax;
    const int e0 = 8 * (lane % LPR);
    const int half = p.rd >> 1, dl = half >> 3;
    const bool first = e0 < half, rot = e0 < p.rd;
    const int src = lane + (first ? dl : -dl);
    const int64_t r = in_range ? row : 0;
    const uint4 kv = *reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.k_new) + r * D + e0);
    const uint4 vv = *reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.v_new) + r * D + e0);
    const uint4 wv = *reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.knorm_w) + e0);
    const uint32_t xs[4] = {kv.x, kv.y, kv.z, kv.w}, ws[4] = {wv.x, wv.y, wv.z, wv.w};
    float y[8], ss = 0.f;
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
    const float posf = live ? (float)(L - 1) : 0.f;
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        float s0 = 0.f, c0 = 1.f, s1 = 0.f, c1 = 1.f;
        if (rot) {
            const int f = first ? e0 : e0 - half;
            rope_sincos(posf * p.inv_freq[f + i], &s0, &c0);
            rope_sincos(posf * p.inv_freq[f + i + 1], &s1, &c1);
        }
        // first half: x*cos - partner*sin; second half: x*cos + partner*sin
        const float v0 = fmaf(y[i], c0, q[i] * (first ? -s0 : s0));
        const float v1 = fmaf(y[i + 1], c1, q[i + 1] * (first ? -s1 : s1));
        o[i >> 1] = pack_bf16x2(v0 * rinv, v1 * rinv);
    }
    if (live) {
        // the row of token L-1: contiguous [2,B,G,Lmax,d], or paged [2,pages,G,page_size,d]
        int64_t plane, off;
        if (p.block_table) {
            const int g = (int)(r % p.G);
            const int page = p.block_table[(int64_t)b * p.max_pages + (L - 1) / p.page_size];
            if (page < 0 || page >= p.num_pages) {
                if (lane % LPR == 0) atomicOr(p.status, GATTN_DEVICE_BAD_PAGE);
                return;
            }
            plane = (int64_t)p.num_pages * p.G * p.page_size * D;
            off = (((int64_t)page * p.G + g) * p.page_size + (L - 1) % p.page_size) * D + e0;
        } else {
            plane = (int64_t)p.B * p.G * p.Lmax * D;  // K half, then V half of the cache
            off = (r * p.Lmax + (L - 1)) * D + e0;
        }
        bf16* cache = static_cast<bf16*>(p.cache);
        *reinterpret_cast<uint4*>(cache + off) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(cache + plane + off) = vv;
    }
}

template <int D>
cudaError_t launch_append_d(const AppendParams& p, cudaStream_t stream) {
    constexpr int RPW = 32 / (D / 8);
    const int64_t rows = (int64_t)p.B * p.G;
    const int64_t blocks = (rows + 8 * RPW - 1) / (8 * RPW);
    decode_append_kernel<D><<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_append(const AppendParams& p, cudaStream_t stream) {
    switch (p.d) {
        case 64: return launch_append_d<64>(p, stream);
        case 128: return launch_append_d<128>(p, stream);
        case 256: return launch_append_d<256>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

int decode_slot_floats(int r, int d) { return 2 * r + r * d; }
int64_t decode_num_slots(int n_ctas, int B, int G) { return ((int64_t)n_ctas + (int64_t)B * G) * NCW; }
int decode_max_batch() { return MAXB; }

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& tm, cudaStream_t stream, cudaEvent_t ev_start,
                          cudaEvent_t ev_stop) {
    switch (p.d) {
        case 64: return launch_dec<64>(p, tm, stream, ev_start, ev_stop);
        case 128: return launch_dec<128>(p, tm, stream, ev_start, ev_stop);
        case 256: return launch_dec<256>(p, tm, stream, ev_start, ev_stop);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gattn
