// prefill_pair.cu -- bf16 causal gated GQA attention on CTA pairs (cta_group::2).
//
// Computes, like prefill_tc.cu,
//   out[b, t, h*d:(h+1)*d] = sigmoid(z) * sum_{j<=t} softmax_j(q'_t . k'_j / sqrt(d)) v_j
// with q' = rope(rmsnorm(q)), k' = rope(rmsnorm(k)) and head h reading KV group
// g = floor(h / (H/G)).  ("Gated attention" handbook chapter, sections "The
// formula" and "Four things Qwen3.5 adds to the textbook"; "Attention, worked all
// the way through", section "Why scaling and stable softmax matter"; "Gated
// Attention" deep-dive, section "门放在哪里？".)
//
// A cluster of two CTAs takes one 128-row query tile of two heads 2p and 2p+1,
// which share their KV group whenever H/G is even; CTA rank c owns head 2p + c.
// The two heads' query rows stack into one M = 256 tensor-core operand, so each
// MMA (issued once, by the even CTA) serves both heads, while each CTA keeps only
// half of every K/V tile in its shared memory: keys [64c, 64c+64) of a 128-key K'
// tile (the B operand of S = Q'K'^T is split along N) and value columns
// [c d/2, (c+1) d/2) of the V tile (the B operand of O += P V, split along N = d).
// That halved footprint is what buys 128-key tiles at d = 256.
//
// Roles per CTA (10 warps):
//   warp 0      TMA producer of this CTA's halves: per work item the raw Q tile of its
//               own head, K' and V halves into rings, at the end its gate tile into
//               the idle V ring, and finally the staged output tile back to global
//               memory with TMA stores.
//   warp 1      allocates TMEM for the pair.  Even CTA: issues every MMA.  Odd CTA:
//               forwards the landing of its K'/V halves to the even CTA's barriers.
//   warps 2..9  two threads per query row of this CTA's head, each owning half of
//               the row's keys in every tile (and half of its O columns): the fused
//               Q prologue (Q' = rope(rmsnorm(q)) written over the raw Q tile in
//               shared memory), the online softmax and the gate epilogue.  The two
//               halves of a row swap tile maxima through shared memory; their row
//               sums are added once, in the epilogue.
//
// TMEM (per CTA, lane = query row): O [0, d) | S0 [d, d+128) | S1 [d+128, d+256).
// Key tile j's scores go to S_{j%2}, and its probabilities P_j overwrite them in
// place as bf16 pairs, which the PV MMA reads straight from TMEM.
// Shared memory (per CTA): Q' tile | K' ring | V ring | barriers | q norm weights |
// row-half exchange.  Once an item's last PV is done, the V ring holds its gate
// tile, which the epilogue overwrites with the output tile.
//
// Work items follow one another without a gap in the tensor pipe's inputs: the
// next item's Q tile lands as soon as the last QK has read the Q buffer, its K'
// tiles as soon as the ring frees up, and the softmax warps normalise it before
// running the current item's epilogue, so that the next item's first QK MMAs run
// meanwhile; its V tiles follow the output tile out of the V ring.
//
// Issue order (one issuer, the tensor pipe runs in order): QK(0), QK(1), then per
// tile PV(j), QK(j+2).  QK(j+2) reuses S_{j%2} right behind the PV that reads P_j
// from it, so while the softmax turns S_j into P_j the tensor core runs PV(j-1)
// and QK(j+1): the softmax has a whole tile period.  The running max is refreshed
// (and O rescaled in TMEM) only when it grows by more than 2^8, so O and l always
// share one reference max.
//
// Cross-CTA signalling: tensor-core completions are multicast to both CTAs by
// tcgen05.commit.  The odd CTA's threads arrive on the even CTA's barriers; every
// such arrival announces work that has already completed (a TMA copy whose
// barrier was observed, tcgen05 stores waited on, tcgen05 loads in registers), so
// CTA-scope arrivals suffice, except for Q', which is written by ordinary stores
// and announced once with a cluster-scope release.
#include "common.cuh"
#include "internal.h"

namespace gattn {
namespace {

struct PairBars {
    uint32_t base;
    __device__ uint32_t at(int i) const { return base + 8u * (uint32_t)i; }
    // k_full / v_full: in the even CTA they expect two arrivals (its own producer's,
    // carrying the bytes, and the odd CTA's forward); in the odd CTA one.
    __device__ uint32_t k_full(int s) const { return at(s); }
    __device__ uint32_t v_full(int s) const { return at(2 + s); }
    // QK(j) complete, j % 2 == i (both CTAs): S_j is in score buffer i and K' stage i is free
    __device__ uint32_t s_full(int i) const { return at(4 + i); }
    __device__ uint32_t p_full(int i) const { return at(6 + i); }   // P_j of both CTAs in buffer i (even CTA)
    // PV(j) complete, j % 2 == i (both CTAs): V stage i is free, O holds the tiles up to j
    __device__ uint32_t pv_done(int i) const { return at(8 + i); }
    __device__ uint32_t o_final() const { return at(10); }          // every PV complete (both CTAs)
    __device__ uint32_t q_ready() const { return at(11); }          // Q' of both CTAs written (even CTA)
    __device__ uint32_t q_full() const { return at(12); }           // raw Q tile + weights landed
    __device__ uint32_t g_full() const { return at(13); }           // gate tile landed (in the V ring)
    __device__ uint32_t drain() const { return at(14); }            // the issuer's MMAs all complete
    __device__ uint32_t xchg(int q) const { return at(15 + q); }    // both halves of row quarter q posted
    __device__ uint32_t o_free() const { return at(19); }   // an item's epilogue has read O (even CTA, both CTAs arrive)
    __device__ uint32_t o_staged() const { return at(20); } // every softmax warp staged its output rows (this CTA)
    static constexpr int COUNT = 21;
};

template <int D>
struct PairCfg {
    static constexpr int BM = 128;        // query rows per CTA
    static constexpr int BN = 128;        // keys per tile
    static constexpr int KH = BN / 2;     // keys of a K' tile held by one CTA
    static constexpr int DH = D / 2;      // value columns held by one CTA
    // two stages each: stage j % 2 is released by the completion of QK(j) / PV(j),
    // the same commits that hand S_j to the softmax and close O's tile j
    static constexpr int NSK = 2;  // K' ring stages
    static constexpr int NSV = 2;  // V ring stages
    static constexpr int KCH = D / 64;    // 128-byte chunks of a K' row
    static constexpr int K_CHUNK = KH * 128;
    static constexpr int K_TILE = KCH * K_CHUNK;
    static constexpr int VCH = DH / 64;   // 128-byte chunks of a V half-row
    static constexpr int V_CHUNK = BN * 128;
    static constexpr int V_TILE = VCH * V_CHUNK;
    static constexpr int ROWBOX_BYTES = BM * 128;  // one Q/gate TMA box: 128 rows x 64 bf16
    static constexpr int QTILE_BYTES = BM * D * 2;
    static_assert(QTILE_BYTES == NSV * V_TILE, "the gate / output tile fills the V ring");
    static constexpr int TM_O = 0;
    static constexpr int TM_S = D;                // score buffer b at TM_S + b * BN
    static constexpr int TM_COLS = 512;
    static_assert(TM_S + 2 * BN <= TM_COLS, "TMEM budget");
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = QTILE_BYTES;
    static constexpr int OFF_V = OFF_K + NSK * K_TILE;
    static constexpr int OFF_BAR = OFF_V + NSV * V_TILE;
    static constexpr int NBAR = PairBars::COUNT;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int OFF_W = (OFF_MISC + 16 + 127) & ~127;
    // row-half exchange: tile maxima [2 buffers][2 halves][BM], row sums and sums of
    // squares of q [2 halves][BM] each
    static constexpr int OFF_X = OFF_W + D * 2;
    static constexpr int SMEM_BYTES = OFF_X + (2 * 2 * BM + 2 * 2 * BM) * 4;
    // never less than 120 KB, so that no second CTA (and TMEM allocation) shares the SM
    static constexpr int SMEM_ALLOC = (SMEM_BYTES + 1024) > 122880 ? (SMEM_BYTES + 1024) : 122880;
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static constexpr int SOFTMAX_WARPS = 8;  // two per row quarter: each thread takes half a row
    static constexpr int THREADS = 64 + 32 * SOFTMAX_WARPS;
    static constexpr int P_ARRIVALS = 2 * SOFTMAX_WARPS;   // P_j: every softmax warp of both CTAs
    static constexpr int Q_ARRIVALS = 2 * SOFTMAX_WARPS;   // Q': every softmax warp of both CTAs
    static constexpr uint32_t IDESC_QK = make_idesc_bf16(256, BN, false);
    static constexpr uint32_t IDESC_PV = make_idesc_bf16(256, D, true);
    static constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 domain
};

// Arrive on the even CTA's copy of barrier `bar`: locally from the even CTA, at
// CTA scope from the odd one (what is announced has already completed).
__device__ __forceinline__ void arrive_even(uint32_t bar, uint32_t cr) {
    if (cr == 0) mbar_arrive(bar);
    else mbar_arrive_remote_cta(mapa_shared(bar, 0));
}

// ----------------------------------------------------------------- work items

// The grid is persistent: one cluster per pair of SMs at most.  Work item u is
// query tile n_qtiles - 1 - u / (B*H/2) (heaviest first) of batch and head pair
// u % (B*H/2); cluster cl of ncl takes items cl, 2 ncl - 1 - cl, 2 ncl + cl, ...
// (a snake over rounds, so that heavy and light tiles share a cluster).  Every
// role walks the same list; ring stages, score buffers and barrier phases run on
// a tile counter that continues across items.
struct PairItem {
    int qt, b, hp, n_kv;
    int t0, len;  // the sequence's first token on the S axis of batch b, and its length
    bool direct;  // a partial tile of packed sequences: rows are stored one by one
};

template <bool GV>
__device__ __forceinline__ bool pair_item(const PrefillParams& p, int cl, int ncl, int r, PairItem& it) {
    const int n_hp = p.H / 2;
    const long long u = (long long)r * ncl + ((r & 1) ? ncl - 1 - cl : cl);
    if (GV && p.vtiles) {
        // packed sequences: query tile u / n_hp of the table (heaviest first), head pair u % n_hp
        if (u >= (long long)p.n_vtiles * n_hp) return false;
        const int4 e = p.vtiles[u / n_hp];
        it.qt = e.z;
        it.t0 = e.x;
        it.len = e.y;
        it.b = 0;
        it.hp = (int)(u % n_hp);
        it.direct = (it.qt + 1) * 128 > it.len;  // a TMA store of 128 rows would reach the next sequence
    } else {
        const int pairs = p.B * n_hp;
        if (u >= (long long)p.n_qtiles * pairs) return false;
        it.qt = p.n_qtiles - 1 - (int)(u / pairs);
        const int bp = (int)(u % pairs);
        it.b = bp / n_hp;
        it.hp = bp % n_hp;
        it.t0 = 0;
        it.len = p.S;
        it.direct = false;
    }
    it.n_kv = (min(it.len, (it.qt + 1) * 128) + 127) / 128;
    return true;
}

// ----------------------------------------------------------------- producer

template <int D, bool GV>
__device__ void pair_producer(const CUtensorMap* tmK, const CUtensorMap* tmV, const CUtensorMap* tmQ,
                              const CUtensorMap* tmG, const CUtensorMap* tmO, const PrefillParams& p,
                              const PairBars& bars, uint32_t sbase, int cl, int ncl, uint32_t cr, volatile int* abort_flag,
                              unsigned int* status) {
    using C = PairCfg<D>;
    // a gate tile per item when the logits vary over head_dim (elementwise, or one
    // head-shared vector per token: the gate map then has a single head)
    const bool gate_tile = GV ? gate_per_dim(p.gate_mode) : p.gate_mode == GATTN_GATE_ELEMENTWISE;
    const bool shared = GV && gate_layout(p.gate_mode) == GATTN_GATE_HEAD_SHARED;
    int nk = 0, nv = 0;  // K' / V tiles issued, over all items
    int jb = 0;          // tiles of the items before the current one
    int n_it = 0, n_g = 0;
    bool ok = true;
    PairItem it;
    // the previous item, whose output still occupies the V ring
    int prev_h = 0, prev_row = 0, prev_b = 0;  // prev_row: first query row on the S axis
    bool prev_direct = false;
    // the V ring is free once every PV of the previous item has completed
    auto v_ring_idle = [&]() -> bool {
        for (int j = jb - C::NSV > 0 ? jb - C::NSV : 0; j < jb; ++j)
            if (!mbar_test_wait(bars.pv_done(j % C::NSV), (uint32_t)(j / C::NSV) & 1u)) return false;
        return true;
    };
    // the previous item's gate tile, read by its epilogue, goes into the idle V ring
    auto load_gate = [&]() {
        mbar_arrive_expect_tx(bars.g_full(), C::QTILE_BYTES);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
            tma_load_4d(sbase + C::OFF_V + c * C::ROWBOX_BYTES, tmG, bars.g_full(), c * 64, shared ? 0 : prev_h,
                        prev_row, prev_b);
        ++n_g;
    };
    // the softmax warps staged the previous item's output rows in the V ring (over
    // the gate tile): write them out (TMA stores, rows past the end clipped) and wait
    // until the copies have read shared memory, after which the ring may be refilled
    // (a partial tile of packed sequences was written row by row by the softmax warps)
    auto store_output = [&]() {
        if (prev_direct) return;
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
            tma_store_4d(tmO, sbase + C::OFF_V + c * C::ROWBOX_BYTES, c * 64, prev_h, prev_row, prev_b);
        bulk_commit_group();
        bulk_wait_group_read0();
    };
    for (int r = 0; ok && pair_item<GV>(p, cl, ncl, r, it); ++r) {
        const int h = 2 * it.hp + (int)cr, g = h / (p.H / p.G);
        // raw Q tile of this CTA's head (normalised in place later): the Q buffer is
        // free once every QK of the previous item has completed
        if (n_it > 0 && !(ok = mbar_wait(bars.s_full((jb - 1) & 1), (uint32_t)((jb - 1) >> 1) & 1u, abort_flag, status)))
            break;
        mbar_arrive_expect_tx(bars.q_full(), C::QTILE_BYTES + (n_it == 0 ? D * 2 : 0));
        if (n_it == 0) bulk_load(sbase + C::OFF_W, p.qnorm_w, D * 2, bars.q_full());
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
            tma_load_4d(sbase + C::OFF_Q + c * C::ROWBOX_BYTES, tmQ, bars.q_full(), c * 64, h,
                        it.t0 + it.qt * C::BM, it.b);
        ++n_it;
        // the gate tile is read at the very end of the item: start it on its way to L2 now
        if (gate_tile) {
#pragma unroll
            for (int c = 0; c < C::KCH; ++c)
                tma_prefetch_l2_4d(tmG, c * 64, shared ? 0 : h, it.t0 + it.qt * C::BM, it.b);
        }
        // K' comes from the pre-pass kernel launched just before this one
        if (n_it == 1) pdl_wait_prerequisites();

        // K' and V tiles, each stream as soon as its own stage frees up.  Meanwhile the
        // previous item finishes in the V ring: its gate tile once the ring is idle,
        // then its output once staged; this item's V tiles follow.
        bool g_sent = n_it == 1 || !gate_tile, v_open = n_it == 1;
        const int ke = nk + it.n_kv, ve = nv + it.n_kv;
        const unsigned long long t0 = global_timer_ns();
        uint32_t spins = 0;
        while (nk < ke || nv < ve) {
            bool progressed = false;
            if (!g_sent && v_ring_idle()) {
                load_gate();
                g_sent = progressed = true;
            }
            if (g_sent && !v_open && mbar_test_wait(bars.o_staged(), (uint32_t)(n_it - 2) & 1u)) {
                store_output();
                v_open = progressed = true;
            }
            if (nk < ke && (nk < C::NSK || mbar_test_wait(bars.s_full(nk % C::NSK), ((uint32_t)(nk / C::NSK) & 1u) ^ 1u))) {
                const int st = nk % C::NSK;
                mbar_arrive_expect_tx(bars.k_full(st), C::K_TILE);
                const uint32_t kdst = sbase + C::OFF_K + st * C::K_TILE;
#pragma unroll
                for (int c = 0; c < C::KCH; ++c)
                    tma_load_3d(kdst + c * C::K_CHUNK, tmK, bars.k_full(st), c * 64,
                                it.t0 + (nk - jb) * C::BN + (int)cr * C::KH, it.b * p.G + g);
                ++nk;
                progressed = true;
            }
            if (v_open && nv < ve &&
                (nv < C::NSV || mbar_test_wait(bars.pv_done(nv % C::NSV), ((uint32_t)(nv / C::NSV) & 1u) ^ 1u))) {
                const int st = nv % C::NSV;
                mbar_arrive_expect_tx(bars.v_full(st), C::V_TILE);
                const uint32_t vdst = sbase + C::OFF_V + st * C::V_TILE;
#pragma unroll
                for (int c = 0; c < C::VCH; ++c)
                    tma_load_4d(vdst + c * C::V_CHUNK, tmV, bars.v_full(st), (int)cr * C::DH + c * 64, g,
                                it.t0 + (nv - jb) * C::BN, it.b);
                ++nv;
                progressed = true;
            }
            if (progressed) {
                spins = 0;
                continue;
            }
            if ((++spins & 63u) == 0) {
                if (*abort_flag) break;
                if (global_timer_ns() - t0 > 4 * kWaitLimitNs) {
                    *abort_flag = 1;
                    atomicOr(status, GATTN_DEVICE_TIMEOUT);
                    break;
                }
            }
        }
        if (nk != ke || nv != ve) { ok = false; break; }
        jb += it.n_kv;
        prev_h = h;
        prev_row = it.t0 + it.qt * C::BM;
        prev_b = it.b;
        prev_direct = it.direct;
    }
    // the last item's gate and output
    if (ok && n_it > 0) {
        if (gate_tile) {
            for (int j = jb - C::NSV > 0 ? jb - C::NSV : 0; ok && j < jb; ++j)
                ok = mbar_wait(bars.pv_done(j % C::NSV), (uint32_t)(j / C::NSV) & 1u, abort_flag, status);
            if (ok) load_gate();
        }
        if (ok && mbar_wait(bars.o_staged(), (uint32_t)(n_it - 1) & 1u, abort_flag, status)) store_output();
        bulk_wait_group0();
    }
    // every copy this thread started lands before the CTA can exit
    if (n_it > 0) mbar_wait_drain(bars.q_full(), (uint32_t)(n_it - 1) & 1u, status);
    for (int j = nk > C::NSK ? nk - C::NSK : 0; j < nk; ++j)
        mbar_wait_drain(bars.k_full(j % C::NSK), (uint32_t)(j / C::NSK) & 1u, status);
    for (int j = nv > C::NSV ? nv - C::NSV : 0; j < nv; ++j)
        mbar_wait_drain(bars.v_full(j % C::NSV), (uint32_t)(j / C::NSV) & 1u, status);
    if (n_g > 0) mbar_wait_drain(bars.g_full(), (uint32_t)(n_g - 1) & 1u, status);
}

// Odd CTA: tell the even CTA's issuer, in order, that each K'/V half has landed here.
template <int D, bool GV>
__device__ void pair_forwarder(const PrefillParams& p, const PairBars& bars, int cl, int ncl, volatile int* abort_flag,
                               unsigned int* status) {
    using C = PairCfg<D>;
    int n_kv = 0;  // tiles over all of this cluster's items
    PairItem it;
    for (int r = 0; pair_item<GV>(p, cl, ncl, r, it); ++r) n_kv += it.n_kv;
    int fk = 0, fv = 0;
    const unsigned long long t0 = global_timer_ns();
    uint32_t spins = 0;
    while (fk < n_kv || fv < n_kv) {
        bool progressed = false;
        if (fk < n_kv && mbar_test_wait(bars.k_full(fk % C::NSK), (uint32_t)(fk / C::NSK) & 1u)) {
            arrive_even(bars.k_full(fk % C::NSK), 1);
            ++fk;
            progressed = true;
        }
        if (fv < n_kv && mbar_test_wait(bars.v_full(fv % C::NSV), (uint32_t)(fv / C::NSV) & 1u)) {
            arrive_even(bars.v_full(fv % C::NSV), 1);
            ++fv;
            progressed = true;
        }
        if (progressed) {
            spins = 0;
            continue;
        }
        if ((++spins & 63u) == 0) {
            if (*abort_flag) break;
            if (global_timer_ns() - t0 > 4 * kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(status, GATTN_DEVICE_TIMEOUT);
                break;
            }
        }
    }
}

// ----------------------------------------------------------------- MMA issuer (even CTA)

// The K-steps [k0, k1) of S = Q'K'^T (A = Q' and B = K' K-major in shared memory)
// and of O += P V (A = P in TMEM, B = V MN-major in shared memory), unrolled at
// compile time with immediate descriptor offsets (mma2_ss_lo): a few instructions
// per MMA, so that the tensor pipe is fed at its own rate even while softmax warps
// of the same sub-partition are busy.
template <int D, int KK>
__device__ __forceinline__ void pair_qk_steps(uint32_t d_tmem, uint32_t q_lo, uint32_t k_lo, int k0, int k1) {
    using C = PairCfg<D>;
    if constexpr (KK < D / 16) {
        if (KK >= k0 && KK < k1)
            mma2_ss_lo<((KK >> 2) * C::ROWBOX_BYTES + (KK & 3) * 32) / 16, ((KK >> 2) * C::K_CHUNK + (KK & 3) * 32) / 16>(
                d_tmem, q_lo, k_lo, sdesc_sw128_hi(), C::IDESC_QK, KK > 0 ? 1u : 0u);
        pair_qk_steps<D, KK + 1>(d_tmem, q_lo, k_lo, k0, k1);
    }
}
template <int D, int KK>
__device__ __forceinline__ void pair_pv_steps(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_lo, uint32_t acc0, int k0,
                                              int k1) {
    using C = PairCfg<D>;
    if constexpr (KK < C::BN / 16) {
        if (KK >= k0 && KK < k1)
            mma2_ts_lo<KK * 8, KK * 16 * 128 / 16>(d_tmem, p_tmem, v_lo, sdesc_sw128_hi(), C::IDESC_PV,
                                                   KK > 0 ? 1u : acc0);
        pair_pv_steps<D, KK + 1>(d_tmem, p_tmem, v_lo, acc0, k0, k1);
    }
}

// Issue order QK(0), QK(1), then per tile PV(j), QK(j+2).  One thread can put an
// MMA into the tensor queue only every ~47 cycles, and the queue is mostly full,
// so the issuer runs almost in step with the pipe: the inputs of the next MMA
// group are polled while the tail of the current one is still queued, so that
// the commits and waits between groups do not leave the pipe idle.
template <int D, bool GV>
__device__ void pair_mma(const PrefillParams& p, const PairBars& bars, uint32_t sbase, uint32_t tm, int cl, int ncl,
                         volatile int* abort_flag, unsigned int* status) {
    using C = PairCfg<D>;
    constexpr int QK_MMAS = D / 16, PV_MMAS = C::BN / 16;
    constexpr int QK_HEAD = QK_MMAS - 4, PV_HEAD = PV_MMAS - 2;  // issued before polling the next group's inputs
    const uint32_t q_lo = sdesc_sw128_lo(sbase + C::OFF_Q, 16);
    const uint32_t k_lo = sdesc_sw128_lo(sbase + C::OFF_K, 16);
    const uint32_t v_lo = sdesc_sw128_lo(sbase + C::OFF_V, C::V_CHUNK);
    // S_j = Q' K'_j^T into score buffer j % 2, MMAs [k0, k1) of the group (j counts tiles over all items)
    auto qk = [&](int j, int k0, int k1) {
        pair_qk_steps<D, 0>(tm + C::TM_S + (uint32_t)(j & 1) * C::BN, q_lo,
                            k_lo + (uint32_t)(((j % C::NSK) * C::K_TILE) >> 4), k0, k1);
    };
    // O += P_j V_j, P_j read from TMEM where it overwrote S_j; the first tile of an item overwrites O
    auto pv = [&](int j, bool first, int k0, int k1) {
        pair_pv_steps<D, 0>(tm + C::TM_O, tm + C::TM_S + (uint32_t)(j & 1) * C::BN,
                            v_lo + (uint32_t)(((j % C::NSV) * C::V_TILE) >> 4), first ? 0u : 1u, k0, k1);
    };
    auto k_ready = [&](int j) { return mbar_test_wait(bars.k_full(j % C::NSK), (uint32_t)(j / C::NSK) & 1u); };
    auto k_wait = [&](int j) { return mbar_wait(bars.k_full(j % C::NSK), (uint32_t)(j / C::NSK) & 1u, abort_flag, status); };
    auto pv_ready = [&](int j) {
        return mbar_test_wait(bars.p_full(j & 1), (uint32_t)(j >> 1) & 1u) &&
               mbar_test_wait(bars.v_full(j % C::NSV), (uint32_t)(j / C::NSV) & 1u);
    };
    auto pv_wait = [&](int j) {
        return mbar_wait(bars.p_full(j & 1), (uint32_t)(j >> 1) & 1u, abort_flag, status) &&
               mbar_wait(bars.v_full(j % C::NSV), (uint32_t)(j / C::NSV) & 1u, abort_flag, status);
    };

    bool ok = true;
    int jb = 0, n_it = 0;
    PairItem it;
    for (int r = 0; ok && pair_item<GV>(p, cl, ncl, r, it); ++r, ++n_it) {
        const int n = it.n_kv;
        ok = mbar_wait(bars.q_ready(), (uint32_t)n_it & 1u, abort_flag, status);  // Q' of both heads ready
        for (int j = 0; ok && j < 2 && j < n; ++j) {
            ok = k_wait(jb + j);
            if (!ok) break;
            tc_fence_after();
            qk(jb + j, 0, QK_MMAS);
            tc_commit2(bars.s_full((jb + j) & 1), 3);
        }
        // PV(0) overwrites O: the previous item's epilogue (both CTAs) must have read it
        if (ok && n_it > 0) ok = mbar_wait(bars.o_free(), (uint32_t)(n_it - 1) & 1u, abort_flag, status);
        if (ok && n > 0) ok = pv_wait(jb);
        for (int j = 0; ok && j < n; ++j) {
            const int jg = jb + j;
            // ---- PV(j): its inputs were checked before
            tc_fence_after();
            pv(jg, j == 0, 0, PV_HEAD);
            const bool more = j + 2 < n;
            const bool kr = more && k_ready(jg + 2);
            pv(jg, j == 0, PV_HEAD, PV_MMAS);
            tc_commit2(bars.pv_done(jg & 1), 3);
            // ---- QK(j+2) into the buffer PV(j) has just been queued to read
            if (more) {
                if (!kr && !k_wait(jg + 2)) { ok = false; break; }
                tc_fence_after();
                qk(jg + 2, 0, QK_HEAD);
            }
            const bool next = j + 1 < n;
            const bool pr = next && pv_ready(jg + 1);
            if (more) {
                qk(jg + 2, QK_HEAD, QK_MMAS);
                tc_commit2(bars.s_full(jg & 1), 3);
            }
            if (next && !pr && !pv_wait(jg + 1)) { ok = false; break; }
        }
        if (ok) tc_commit2(bars.o_final(), 3);
        jb += n;
    }
    tc_commit2(bars.drain(), 1);
    // no MMA of the pair may still be running when the CTAs tear down
    mbar_wait_drain(bars.drain(), 0, status);
}

// ----------------------------------------------------------------- softmax / prologue / epilogue

// GV: the gate variants (head-shared logits, NS-sigmoid, SiLU, additive) and
// packed variable-length sequences -- a second instance of the kernel, so that
// the default (batched, elementwise / headwise multiplicative sigmoid gate)
// compiles exactly as it would alone.
template <int D, bool GV>
__device__ void pair_softmax(const PrefillParams& p, const PairBars& bars, uint32_t sbase, uint8_t* smem_x, uint32_t tm,
                             uint32_t cr, int quarter, int hf, int lane, int cl, int ncl, volatile int* abort_flag) {
    using C = PairCfg<D>;
    constexpr int HB = C::BN / 2;  // keys of a tile owned by this thread
    const int row = quarter * 32 + lane;
    const uint32_t tl = tm + ((uint32_t)(quarter * 32) << 16);
    // the two threads of a row swap values through shared memory and then meet on
    // an mbarrier (one phase per use: every tile, and twice per item)
    float* xmax = reinterpret_cast<float*>(smem_x);          // [2][2][BM] tile maxima
    float* xsum = xmax + 2 * 2 * C::BM;                      // [2][BM] row sums
    float* xss = xsum + 2 * C::BM;                           // [2][BM] sums of squares of q
    const uint32_t xbar = bars.xchg(quarter);
    int xphase = 0;
    auto meet = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(xbar);
        return __all_sync(0xffffffffu, mbar_wait(xbar, (uint32_t)(xphase++) & 1u, abort_flag, p.status));
    };

    // ---- fused Q prologue of item k: rmsnorm then partial rotate-half RoPE, written
    // as bf16 over the raw row in the Q tile (the A operand of S = Q'K'^T).  The two
    // threads of a row each sum the squares of their half of it; the 8-column chunks
    // are then shared out alternately, a rotated pair (i, i + rd/2) going with the
    // chunk of i.  Rows past the sequence end were zero-filled by TMA.
    auto q_prologue = [&](const PairItem& it, int k) -> bool {
        const int t = it.qt * C::BM + row;  // from the start of the sequence
        const bool valid = t < it.len;
        if (!__all_sync(0xffffffffu, mbar_wait(bars.q_full(), (uint32_t)k & 1u, abort_flag, p.status))) return false;
        const uint32_t qbase = sbase + C::OFF_Q;
        const uint32_t wbase = sbase + C::OFF_W;
        float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
            float f[8];
            unpack8(lds_v4(rowtile_addr(qbase, row, hf * (D / 2) + 8 * c)), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss[e & 3] = fmaf(f[e], f[e], ss[e & 3]);
        }
        xss[hf * C::BM + row] = (ss[0] + ss[1]) + (ss[2] + ss[3]);
        // past the meet both halves have read the raw row: the writes below may begin
        if (!meet()) return false;
        const float rinv = rsqrtf((xss[row] + xss[C::BM + row]) / (float)D + p.eps);
        const float posf = valid ? (p.pos ? (float)p.pos[(int64_t)it.b * p.S + it.t0 + t] : (float)t) : 0.f;
        const int half = p.rd >> 1;
        for (int i0 = 8 * hf; i0 < half; i0 += 16) {
            float xa[8], xb[8], wa[8], wb[8];
            unpack8(lds_v4(rowtile_addr(qbase, row, i0)), xa);
            unpack8(lds_v4(rowtile_addr(qbase, row, i0 + half)), xb);
            unpack8(lds_v4(wbase + 2 * i0), wa);
            unpack8(lds_v4(wbase + 2 * (i0 + half)), wb);
            uint32_t lo[4], hi[4];
            rope_rotate8(xa, xb, wa, wb, p.inv_freq + i0, posf, rinv, lo, hi);
            sts_v4(rowtile_addr(qbase, row, i0), lo[0], lo[1], lo[2], lo[3]);
            sts_v4(rowtile_addr(qbase, row, i0 + half), hi[0], hi[1], hi[2], hi[3]);
        }
        for (int e0 = p.rd + 8 * hf; e0 < D; e0 += 16) {
            float x[8], w[8];
            unpack8(lds_v4(rowtile_addr(qbase, row, e0)), x);
            unpack8(lds_v4(wbase + 2 * e0), w);
            uint32_t o[4];
            scale8_bf16(x, w, rinv, o);
            sts_v4(rowtile_addr(qbase, row, e0), o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();  // the tensor core reads Q' through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(bars.q_ready(), 0));  // ordinary stores: cluster release
        return true;
    };

    int jb = 0, n_it = 0;
    PairItem item, next;
    bool have = pair_item<GV>(p, cl, ncl, 0, item);
    if (have && !q_prologue(item, 0)) return;
    for (int r = 0; have; ++r, ++n_it) {
        const int qt = item.qt, b = item.b, h = 2 * item.hp + (int)cr, n_kv = item.n_kv;
        const int t = qt * C::BM + row;  // from the start of the sequence
        const bool valid = t < item.len;
        float gate_head = 1.f;  // the activation of a headwise logit
        if ((GV ? gate_layout(p.gate_mode) : p.gate_mode) == GATTN_GATE_HEADWISE && valid) {
            const int64_t tok = (int64_t)b * p.S + item.t0 + t;
            const bf16* grow = static_cast<const bf16*>(p.gate) + tok * p.gate_tok_stride + (int64_t)h * p.gate_head_stride;
            const float z = __bfloat162float(grow[0]);
            gate_head = GV ? gate_act(z, sigmoid_tanh(z), p.gate_mode) : sigmoid_tanh(z);
        }

        // ---- main loop: online softmax over the KV tiles this query tile can see.
        // This thread owns keys [64 hf, 64 hf + 64) of every tile and O columns
        // [hf D/2, (hf+1) D/2); its partner (same row, other half) runs in warp +- 4.
        const float sl2 = p.scale_log2;
        const int row_min = qt * C::BM;
        float m_ref = -INFINITY;  // reference max (log2 domain) shared by O and l
        float l = 0.f;            // this half's share of the row sum
        for (int j = 0; j < n_kv; ++j) {
            const int jg = jb + j;  // tile counter over all items: buffers and phases
            const uint32_t s_col = C::TM_S + (uint32_t)(jg & 1) * C::BN;
            if (!__all_sync(0xffffffffu, mbar_wait(bars.s_full(jg & 1), (uint32_t)(jg >> 1) & 1u, abort_flag, p.status)))
                return;
            tc_fence_after();
            float s[HB];
            {
                uint32_t r[64];
                tmem_ld64(tl + s_col + hf * HB, r);
#pragma unroll
                for (int e = 0; e < 64; ++e) s[e] = __uint_as_float(r[e]);
            }
            const int key0 = j * C::BN + hf * HB;
            if (key0 + HB - 1 > row_min) {
#pragma unroll
                for (int c = 0; c < HB; ++c)
                    if (key0 + c > t) s[c] = -INFINITY;
            }
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
            for (int c = 8; c < HB; c += 2) mx[(c >> 1) & 7] = max3(mx[(c >> 1) & 7], s[c], s[c + 1]);
            float mt = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            // the row's maximum over the whole tile: swap halves (buffer j%2, so a slow
            // partner still reading tile j-1 is never overwritten).  Passing the meet also
            // means the partner has read its S columns, which P overwrites below.
            xmax[((jg & 1) * 2 + hf) * C::BM + row] = mt;
            if (!meet()) return;
            mt = fmaxf(mt, xmax[((jg & 1) * 2 + (hf ^ 1)) * C::BM + row]);
            const float m_new = fmaxf(m_ref, mt * sl2);
            const bool need = (m_new - m_ref) > C::RESCALE_THRESHOLD;
            if (j == 0) {
                m_ref = m_new;
            } else if (__any_sync(0xffffffffu, need)) {
                const float alpha = need ? ex2_approx(m_ref - m_new) : 1.f;
                if (need) {
                    l *= alpha;
                    m_ref = m_new;
                }
                __syncwarp();
                // O is touched only once PV(j-1) has landed (PV(j-2) already had: QK(j)
                // was issued behind it)
                if (!__all_sync(0xffffffffu, mbar_wait(bars.pv_done((jg - 1) & 1), (uint32_t)((jg - 1) >> 1) & 1u,
                                                       abort_flag, p.status)))
                    return;
                tc_fence_after();
#pragma unroll 1
                for (int c = hf * (D / 2); c < (hf + 1) * (D / 2); c += 32) {
                    uint32_t r[32];
                    tmem_ld32(tl + C::TM_O + c, r);
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                    tmem_st32(tl + C::TM_O + c, r);
                }
            }
            // P = exp2(s * scale * log2e - m_ref) as bf16 pairs over this thread's keys:
            // columns [32 hf, 32 hf + 32) of the score buffer
            const float mref = m_ref;
            uint32_t pk[32];
            float2 rs2[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
            const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(-mref, -mref);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float2 x = fma2(make_float2(s[2 * e], s[2 * e + 1]), sl2x2, negm);
                const float2 pe = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                rs2[e & 3] = add2(rs2[e & 3], pe);
                pk[e] = pack_bf16x2(pe.x, pe.y);
            }
            tmem_st32(tl + s_col + hf * (HB / 2), pk);
            l += ((rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y)) + ((rs2[2].x + rs2[2].y) + (rs2[3].x + rs2[3].y));
            tmem_wait_st();  // P (and an O rescale above, if any) has landed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_even(bars.p_full(jg & 1), cr);
        }

        // ---- the next item's Q prologue: its QK MMAs then run during this epilogue
        const bool more = pair_item<GV>(p, cl, ncl, r + 1, next);
        if (more && !q_prologue(next, n_it + 1)) return;

        // ---- epilogue: O / l * act(gate) (or O / l + act(gate) for an additive gate),
        // this thread's half of the columns, as bf16
        // into the staging tile in the V ring (the gate tile's own slots when there is
        // one: each thread overwrites only what it has just read); the producer then
        // writes the tile to [B,S,H*d] with TMA stores (rows past the end clipped)
        xsum[hf * C::BM + row] = l;
        if (!meet()) return;
        const float l_row = xsum[row] + xsum[C::BM + row];
        if (!__all_sync(0xffffffffu, mbar_wait(bars.o_final(), (uint32_t)n_it & 1u, abort_flag, p.status))) return;
        const bool elementwise = GV ? gate_per_dim(p.gate_mode) : p.gate_mode == GATTN_GATE_ELEMENTWISE;
        constexpr bool plain = !GV;
        const bool additive = GV && gate_additive(p.gate_mode);
        if (elementwise && !__all_sync(0xffffffffu, mbar_wait(bars.g_full(), (uint32_t)n_it & 1u, abort_flag, p.status)))
            return;
        tc_fence_after();
        const float inv_l = 1.f / l_row;
        // out = o * gm + ga
        const float gh = additive ? inv_l : inv_l * gate_head, gha = additive ? gate_head : 0.f;
        const uint32_t gbase = sbase + C::OFF_V;
        // staged for the producer's TMA store, or (a partial tile of packed
        // sequences) stored straight to this row of out, valid rows only
        const bool direct = item.direct;
        bf16* orow = static_cast<bf16*>(p.out) + (((int64_t)b * p.S + item.t0 + t) * p.H + h) * D;
        auto put = [&](uint32_t addr, int col, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
            if (!direct) sts_v4(addr, w0, w1, w2, w3);
            else if (valid) *reinterpret_cast<uint4*>(orow + col) = make_uint4(w0, w1, w2, w3);
        };
#pragma unroll 1
        for (int c = hf * (D / 2); c < (hf + 1) * (D / 2); c += 32) {
            uint32_t r[32];
            __syncwarp();
            tmem_ld32(tl + C::TM_O + c, r);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const uint32_t addr = rowtile_addr(gbase, row, c + 8 * q4);
                const float* o = reinterpret_cast<const float*>(r + 8 * q4);
                if constexpr (plain) {  // the default multiplicative sigmoid gate
                    float gv[8];
                    if (elementwise) {
                        float f[8];
                        unpack8(lds_v4(addr), f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) gv[e] = inv_l * sigmoid_tanh(f[e]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) gv[e] = gh;
                    }
                    put(addr, c + 8 * q4, pack_bf16x2(o[0] * gv[0], o[1] * gv[1]), pack_bf16x2(o[2] * gv[2], o[3] * gv[3]),
                        pack_bf16x2(o[4] * gv[4], o[5] * gv[5]), pack_bf16x2(o[6] * gv[6], o[7] * gv[7]));
                } else {
                float gv[8], ga[8];  // out = o * gv + ga
                if (elementwise) {
                    float f[8];
                    unpack8(lds_v4(addr), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float a = gate_act(f[e], sigmoid_tanh(f[e]), p.gate_mode);
                        gv[e] = additive ? inv_l : inv_l * a;
                        ga[e] = additive ? a : 0.f;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        gv[e] = gh;
                        ga[e] = gha;
                    }
                }
                put(addr, c + 8 * q4, pack_bf16x2(fmaf(o[0], gv[0], ga[0]), fmaf(o[1], gv[1], ga[1])),
                       pack_bf16x2(fmaf(o[2], gv[2], ga[2]), fmaf(o[3], gv[3], ga[3])),
                       pack_bf16x2(fmaf(o[4], gv[4], ga[4]), fmaf(o[5], gv[5], ga[5])),
                       pack_bf16x2(fmaf(o[6], gv[6], ga[6]), fmaf(o[7], gv[7], ga[7])));
                }
            }
        }
        // O has been read: the next item's first PV may overwrite it
        tc_fence_before();
        fence_proxy_async_smem();  // the TMA store reads the staged rows through the async proxy
        __syncwarp();
        if (lane == 0) {
            arrive_even(bars.o_free(), cr);
            mbar_arrive(bars.o_staged());
        }
        jb += n_kv;
        item = next;
        have = more;
    }
}

// ----------------------------------------------------------------- kernel

template <int D, bool GV>
__global__ void __launch_bounds__(PairCfg<D>::THREADS, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmG,
                        const __grid_constant__ CUtensorMap tmO, const __grid_constant__ PrefillParams p) {
    using C = PairCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const PairBars bars{sbase + C::OFF_BAR};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    const uint32_t cr = cluster_ctarank();

    // cluster cl of ncl walks its list of work items (see pair_item)
    const int cl = (int)(blockIdx.x >> 1), ncl = (int)(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        const uint32_t full_count = cr == 0 ? 2u : 1u;
        for (int i = 0; i < 2; ++i) {
            mbar_init(bars.k_full(i), full_count);
            mbar_init(bars.v_full(i), full_count);
            mbar_init(bars.s_full(i), 1);
            mbar_init(bars.p_full(i), C::P_ARRIVALS);
            mbar_init(bars.pv_done(i), 1);
        }
        mbar_init(bars.o_final(), 1);
        mbar_init(bars.q_ready(), C::Q_ARRIVALS);
        mbar_init(bars.q_full(), 1);
        mbar_init(bars.g_full(), 1);
        mbar_init(bars.drain(), 1);
        for (int q = 0; q < 4; ++q) mbar_init(bars.xchg(q), 2);
        mbar_init(bars.o_free(), C::P_ARRIVALS);
        mbar_init(bars.o_staged(), C::SOFTMAX_WARPS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
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
        if (lane == 0)
            pair_producer<D, GV>(&tmK, &tmV, &tmQ, &tmG, &tmO, p, bars, sbase, cl, ncl, cr, abort_flag, p.status);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            if (cr == 0) pair_mma<D, GV>(p, bars, sbase, tm, cl, ncl, abort_flag, p.status);
            else pair_forwarder<D, GV>(p, bars, cl, ncl, abort_flag, p.status);
        }
        __syncwarp();
    } else {
        pair_softmax<D, GV>(p, bars, sbase, smem + C::OFF_X, tm, cr, warp & 3, (warp - 2) >> 2, lane, cl, ncl, abort_flag);
    }
    // both CTAs are done with the pair's TMEM (the issuer drained every MMA) before it is released
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc2(tm, C::TM_COLS);
    }
}

template <int D>
cudaError_t launch_pair_d(const PrefillParams& p, const PrefillMaps& maps, cudaStream_t stream, cudaEvent_t ev_start,
                          cudaEvent_t ev_stop) {
    using C = PairCfg<D>;
    const bool gv = !gate_plain(p.gate_mode) || gate_layout(p.gate_mode) == GATTN_GATE_HEAD_SHARED || p.vtiles;
    auto kernel = gv ? prefill_pair_kernel<D, true> : prefill_pair_kernel<D, false>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kernel), C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    const long long n_items = p.vtiles ? (long long)p.n_vtiles * (p.H / 2) : (long long)p.n_qtiles * p.B * (p.H / 2);
    const long long max_clusters = p.n_sms >= 2 ? p.n_sms / 2 : 1;
    const long long blocks = 2 * (n_items < max_clusters ? n_items : max_clusters);
    if (n_items * 2 > 0x7fffffffLL || blocks < 2) return cudaErrorInvalidValue;
    if (ev_start) cudaEventRecord(ev_start, stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, maps.k, maps.v, maps.q, maps.gate, maps.out, p);
    if (ev_stop) cudaEventRecord(ev_stop, stream);
    return err;
}

}  // namespace

// d = 256 only: at d = 128 the one-head kernel (64-column P and S in TMEM, two
// score buffers) is faster, the softmax rather than K/V traffic being its bound.
bool prefill_pair_supported(int d, int H, int G) { return d == 256 && ((H / G) % 2 == 0); }
int prefill_pair_key_rows() { return PairCfg<256>::KH; }
int prefill_pair_value_rows() { return PairCfg<256>::BN; }

cudaError_t launch_prefill_pair(const PrefillParams& p, const PrefillMaps& maps, cudaStream_t stream,
                                cudaEvent_t ev_start, cudaEvent_t ev_stop) {
    if (p.d == 256) return launch_pair_d<256>(p, maps, stream, ev_start, ev_stop);
    if (p.d == 128) return launch_pair_d<128>(p, maps, stream, ev_start, ev_stop);
    return cudaErrorInvalidValue;
}

}  // namespace gattn
