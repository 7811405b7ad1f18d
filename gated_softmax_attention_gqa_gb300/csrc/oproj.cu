// oproj.cu -- the output projection that follows the gated attention,
// y = x W_O^T, on 5th-generation tensor cores.
//
// x is the gated attention output [T, K] (K = H*d, row-major: the layout the
// prefill kernels write, heads side by side), W_O the projection's weight [N, K]
// (a linear layer, y = x W^T), y [T, N]; bf16 in and out, fp32 accumulation in
// TMEM, one rounding.  ("Transformer by Hand, ch. 6", section "The code:
// qwen/attention.py": the heads are concatenated, multiplied by the gate's sigmoid
// and projected by o_proj; "Gated Attention for LLMs 论文阅读": the gate acts on the
// SDPA output before the output projection.)
//
// Persistent clusters of two CTAs walk 256 x BN output tiles, rows of x fastest so
// that the clusters working at the same time share the same slices of W_O in L2.
// The pair's tensor cores run one M = 256 MMA (cta_group::2): each CTA holds its
// 128 rows of x and half of the W_O slice (BN/2 rows), and the MMA reads both
// halves, so an SM takes in 32 KB per 64-wide slice of K for the work that needs 48
// KB on one SM alone (the one-SM form was bound by that intake).  K streams through
// a 6-stage TMA ring (128-byte swizzle, both operands K-major), four MMAs of K = 16
// per slice.  Two TMEM accumulators: the epilogue of one tile (four warps per CTA,
// one thread per output row: TMEM -> bf16 -> global) runs under the MMAs of the
// next.  Every wait is bounded (the kernels' common limit), after which the CTA
// raises its abort flag, records GATTN_DEVICE_TIMEOUT and winds down.
//
// Warps: 0 TMA producer; 1 in the even CTA the MMA issuer, in the odd one the
// forwarder of its slices' landing to the even CTA; 1 also owns TMEM; 2..5 epilogue.
#include "common.cuh"
#include "internal.h"

namespace gattn {
namespace {

template <int BN>
struct OpCfg {
    static constexpr int BM = 128, BK = 64, NST = 6;  // rows per CTA (256 per pair); ring stages
    static constexpr int A_BYTES = BM * BK * 2;       // one slice of this CTA's rows of x: 128 x 128 B
    static constexpr int B_BYTES = (BN / 2) * BK * 2;  // this CTA's half of a W_O slice: BN/2 rows x 128 B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int OFF_BAR = NST * STAGE_BYTES;
    static constexpr int NBAR = 2 * NST + 5;  // full[s], empty[s], acc_full[2], acc_empty[2], drain
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;  // + slack for the 1024-byte alignment
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static constexpr int TM_COLS = 2 * BN;  // two fp32 accumulators of BN columns per CTA
    static_assert(TM_COLS >= 32 && TM_COLS <= 512 && (TM_COLS & (TM_COLS - 1)) == 0, "TMEM allocation");
    static constexpr int THREADS = 192;
    static constexpr uint32_t IDESC = make_idesc_bf16(256, BN, false);
};

struct OpBars {
    uint32_t base;
    static constexpr int NST = OpCfg<64>::NST;  // ring depth, the same for every BN
    // full: in the even CTA two arrivals (its producer's, carrying the bytes, and the
    // odd CTA's forward), in the odd CTA one; empty, acc_full: the issuer's commits,
    // multicast to both CTAs; acc_empty (even CTA): every epilogue warp of both CTAs
    __device__ uint32_t full(int s) const { return base + 8u * (uint32_t)s; }
    __device__ uint32_t empty(int s) const { return base + 8u * (uint32_t)(NST + s); }
    __device__ uint32_t acc_full(int a) const { return base + 8u * (uint32_t)(2 * NST + a); }
    __device__ uint32_t acc_empty(int a) const { return base + 8u * (uint32_t)(2 * NST + 2 + a); }
    __device__ uint32_t drain() const { return base + 8u * (uint32_t)(2 * NST + 4); }
};

// Arrive on the even CTA's copy of barrier `bar`: locally in the even CTA, at CTA
// scope from the odd one (what is announced has already completed).
__device__ __forceinline__ void op_arrive_even(uint32_t bar, uint32_t cr) {
    if (cr == 0) mbar_arrive(bar);
    else mbar_arrive_remote_cta(mapa_shared(bar, 0));
}

// The four K = 16 steps of one 64-wide slice: +32 bytes along the swizzled rows of
// both operands (descriptor address units of 16 bytes).
template <int BN, int KK>
__device__ __forceinline__ void op_slice(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t acc0) {
    if constexpr (KK < 4) {
        mma2_ss_lo<KK * 2, KK * 2>(d_tmem, a_lo, b_lo, sdesc_sw128_hi(), OpCfg<BN>::IDESC, KK > 0 ? 1u : acc0);
        op_slice<BN, KK + 1>(d_tmem, a_lo, b_lo, acc0);
    }
}

template <int BN>
__global__ void __launch_bounds__(OpCfg<BN>::THREADS, 1)
    oproj_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ OprojParams p) {
    using C = OpCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const OpBars bars{sbase + C::OFF_BAR};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    const uint32_t cr = cluster_ctarank();
    const int cl = (int)(blockIdx.x >> 1), n_cl = (int)(gridDim.x >> 1);
    const int n_m = (p.T + C::BM - 1) / C::BM, n_k = p.K / C::BK;
    // work unit u of the cluster: column block n = u / n_pairs, this CTA's rows in row
    // tile 2 (u % n_pairs) + cr (past the last one when their count is odd: zero-filled
    // by TMA and never stored, the CTA still loads its half of W_O for the pair)
    const int n_pairs = (n_m + 1) / 2;
    const int n_units = n_pairs * (p.N / BN);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(bars.full(s), cr == 0 ? 2u : 1u);
            mbar_init(bars.empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bars.acc_full(a), 1);
            mbar_init(bars.acc_empty(a), 8);
        }
        mbar_init(bars.drain(), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc2(smem_u32(tmem_slot), C::TM_COLS);
        tmem_relinquish2();
    }
    // both CTAs' barriers are initialised and the pair's TMEM allocated before any
    // cross-CTA arrival or MMA
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {  // producer: this CTA's rows of x and its half of W_O, slice by slice
            int it = 0;
            bool ok = true;
            for (int u = cl; ok && u < n_units; u += n_cl) {
                const int m = 2 * (u % n_pairs) + (int)cr, n = u / n_pairs;
                for (int k = 0; k < n_k; ++k, ++it) {
                    const int s = it % C::NST;
                    if (it >= C::NST &&
                        !(ok = mbar_wait(bars.empty(s), (uint32_t)((it / C::NST) & 1) ^ 1u, abort_flag, p.status)))
                        break;
                    const uint32_t dst = sbase + s * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(bars.full(s), C::STAGE_BYTES);
                    tma_load_2d(dst, &tmA, bars.full(s), k * C::BK, m * C::BM);
                    tma_load_2d(dst + C::A_BYTES, &tmB, bars.full(s), k * C::BK, n * BN + (int)cr * (BN / 2));
                }
            }
            // every copy this thread started must land before the CTA can exit
            for (int j = it > C::NST ? it - C::NST : 0; j < it; ++j)
                mbar_wait_drain(bars.full(j % C::NST), (uint32_t)(j / C::NST) & 1u, p.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && cr == 1) {  // forwarder: each slice landed here -> the even CTA's full barrier
            int it = 0;
            const int n_it = ((n_units - cl + n_cl - 1) / n_cl) * n_k;
            for (; it < (cl < n_units ? n_it : 0); ++it) {
                const int s = it % C::NST;
                if (!mbar_wait(bars.full(s), (uint32_t)(it / C::NST) & 1u, abort_flag, p.status)) break;
                op_arrive_even(bars.full(s), 1);
            }
        } else if (lane == 0) {  // MMA issuer (even CTA)
            int it = 0, tc = 0;
            bool ok = true;
            for (int u = cl; ok && u < n_units; u += n_cl, ++tc) {
                const int a = tc & 1;
                // accumulator a was last read by the epilogues of tile tc - 2
                if (tc >= 2 &&
                    !(ok = mbar_wait(bars.acc_empty(a), (uint32_t)((tc >> 1) - 1) & 1u, abort_flag, p.status)))
                    break;
                tc_fence_after();
                for (int k = 0; k < n_k; ++k, ++it) {
                    const int s = it % C::NST;
                    if (!(ok = mbar_wait(bars.full(s), (uint32_t)(it / C::NST) & 1u, abort_flag, p.status))) break;
                    tc_fence_after();
                    const uint32_t a_lo = sdesc_sw128_lo(sbase + s * C::STAGE_BYTES, 16);
                    const uint32_t b_lo = sdesc_sw128_lo(sbase + s * C::STAGE_BYTES + C::A_BYTES, 16);
                    op_slice<BN, 0>(tm + a * BN, a_lo, b_lo, k > 0 ? 1u : 0u);
                    tc_commit2(bars.empty(s), (uint16_t)0x3);  // the slot is free in both CTAs
                }
                if (ok) tc_commit2(bars.acc_full(a), (uint16_t)0x3);
            }
            // whatever happened, no MMA may still be in flight when TMEM is released
            tc_commit2(bars.drain(), (uint16_t)0x1);
            mbar_wait_drain(bars.drain(), 0, p.status);
        }
        __syncwarp();
    } else {  // epilogue: warp w reads this CTA's TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31
        const int q = warp & 3, row = q * 32 + lane;
        const uint32_t tl = tm + ((uint32_t)(q * 32) << 16);
        int tc = 0;
        for (int u = cl; u < n_units; u += n_cl, ++tc) {
            const int a = tc & 1, m = 2 * (u % n_pairs) + (int)cr, n = u / n_pairs;
            if (!__all_sync(0xffffffffu, mbar_wait(bars.acc_full(a), (uint32_t)(tc >> 1) & 1u, abort_flag, p.status)))
                break;
            tc_fence_after();
            const int trow = m * C::BM + row;
            bf16* yrow = static_cast<bf16*>(p.y) + (int64_t)trow * p.N + n * BN;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tl + a * BN + c0, r);
                if (c0 + 32 == BN) {  // the accumulator is read: the tile after next may use it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) op_arrive_even(bars.acc_empty(a), cr);
                }
                if (trow < p.T) {
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(r[j + 0]), __uint_as_float(r[j + 1]));
                        v.y = pack_bf16x2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                        v.z = pack_bf16x2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
                        v.w = pack_bf16x2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
                        *reinterpret_cast<uint4*>(yrow + c0 + j) = v;
                    }
                }
            }
        }
    }
    // both CTAs are done with the pair's TMEM (the issuer drained every MMA) and no
    // cross-CTA arrival is still on its way before it is released
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc2(tm, C::TM_COLS);
    }
}

template <int BN>
cudaError_t launch_bn(const OprojParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, cudaStream_t stream,
                      cudaEvent_t ev_start, cudaEvent_t ev_stop) {
    using C = OpCfg<BN>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(oproj_kernel<BN>), C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    const int64_t n_units = (int64_t)(((p.T + C::BM - 1) / C::BM + 1) / 2) * (p.N / BN);
    const int64_t max_cl = p.n_sms >= 2 ? p.n_sms / 2 : 1;
    const int64_t n_cl = n_units < max_cl ? n_units : max_cl;
    if (ev_start) cudaEventRecord(ev_start, stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * n_cl));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, oproj_kernel<BN>, tmA, tmB, p);
    if (ev_stop) cudaEventRecord(ev_stop, stream);
    return e;
}

}  // namespace

int oproj_block_n(int N) { return N % 256 == 0 ? 256 : N % 128 == 0 ? 128 : 64; }
int oproj_box_rows(int N) { return oproj_block_n(N) / 2; }  // each CTA of a pair holds half a W_O slice

cudaError_t launch_oproj(const OprojParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, cudaStream_t stream,
                         cudaEvent_t ev_start, cudaEvent_t ev_stop) {
    switch (oproj_block_n(p.N)) {
        case 256: return launch_bn<256>(p, tmA, tmB, stream, ev_start, ev_stop);
        case 128: return launch_bn<128>(p, tmA, tmB, stream, ev_start, ev_stop);
        default: return launch_bn<64>(p, tmA, tmB, stream, ev_start, ev_stop);
    }
}

}  // namespace gattn
