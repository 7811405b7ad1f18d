// prefill_tc.cu -- bf16 causal gated GQA attention on 5th-generation tensor cores.
//
// A CTA computes 128-row query tiles of one head at a time:
//   out[b, t, h*d:(h+1)*d] = sigmoid(z) * sum_{j<=t} softmax_j(q'_t . k'_j / sqrt(d)) v_j
// where q' = rope(rmsnorm(q)), k' = rope(rmsnorm(k)) and head h reads KV group
// g = floor(h / (H/G)).  ("Gated attention" handbook chapter, sections "The
// formula", "Four things Qwen3.5 adds to the textbook" and "The code:
// qwen/attention.py"; "Attention, worked all the way through", section "Why
// scaling and stable softmax matter"; "Gated Attention" deep-dive, section
// "门放在哪里？".)
//
// d <= 128: the grid is persistent (one CTA per SM at most) and walks a list of
// work items (query tile, head, batch), heaviest tile first, in a snake over
// rounds; ring stages, score buffers and barrier phases run on tile and item
// counters that continue across items.  While one item finishes (last softmax,
// PV, epilogue, output store) the next one's Q' is in TMEM already (computed by a
// warpgroup of its own during the previous item), its first K' tiles have landed
// and its first QK MMAs are in the tensor pipe.  d = 256 (odd H/G only): one item
// per CTA.
//
// Roles (16 warps at d <= 128, 7 at d = 256):
//   warp 0      TMA producer: per item the raw Q tile, K' tiles (keys normed and
//               rotated by the pre-pass) and raw V tiles into 2-stage rings (128 B
//               swizzle), the gate tile, and the TMA stores of the staged output.
//   warps 1, 2  MMA issuers (warp 1 also owns TMEM): warp 1 + i issues S = Q'K'^T
//               (tcgen05.mma, A read from TMEM) and O += P V of the KV tiles j
//               with j % 2 == i (j counting tiles over all items).
//   softmax     the online softmax.  d <= 128: warps 4..11, two threads per query
//               row (warps w and w + 4 share the row's TMEM lanes), each owning half
//               of the keys of every tile and half of O's columns (the halves swap
//               tile maxima through shared memory); d = 256: warps 3..6, one thread
//               per row, which also run the Q prologue and the gate epilogue.
//   prologue /  d <= 128: warps 12..15, one thread per query row: the fused Q
//   epilogue    prologue (RMSNorm + RoPE of the raw query row, read from shared
//               memory, written as bf16 straight into TMEM) of the item after next,
//               and the gate epilogue of the item the softmax has just finished.
//   (warp 3 is idle at d <= 128: setmaxnreg acts on whole warpgroups.)
//
// Shared memory, d <= 128: raw Q tile | K ring | V ring | gate tile, which the
// epilogue overwrites with the output tile staged for the TMA stores.  d = 256:
// K ring | V ring | two P buffers; the raw Q tile sits in the V ring before any V
// tile is loaded, the gate tile in the K ring once every K' tile is consumed, the
// staged output in the V ring once every PV is done.  Every reuse is ordered by
// mbarriers.
//
// TMEM (512 columns x 128 lanes, lane = query row):
//   [0, d)             O accumulator, fp32 (the first PV of an item overwrites it)
//   [d, d+BN)          S buffer 0 (fp32 scores)
//   [d+BN, d+2BN)      S buffer 1
//   [d+2BN, d+2BN+d/2) Q' as packed bf16 pairs (A operand of S = Q'K'^T); d <= 128:
//                      two such buffers, item n in buffer n % 2
//   P (bf16 pairs, the A operand of O += PV) is written over its own scores (d <=
//   128), or goes to shared memory (d = 256)
//
// Pipeline, d <= 128: the issuer of tile j issues S_{j+2} = Q'K'_{j+2}^T into
// tile j's score buffer right behind PV_j, which reads P_j from there (one
// thread's MMAs run in issue order), so S_{j+1} is waiting while the softmax works
// on tile j.  d = 256: a score buffer is handed back as soon as the softmax has
// loaded S_j, and P_j goes to shared-memory buffer j % 2 once PV_{j-2} has read it.
// P_j V_j follows as soon as P_j lands.
// The exponent's reference is the logits' bound from the QK-norm weights when that
// is small enough (no row maximum at all); otherwise a running max, refreshed (and
// O rescaled in TMEM) only when it grows by more than 2^8, so the rescale is rare
// and exact: O and l always share one reference.  The causal mask is applied by
// skipping every KV tile past the query tile and masking only the tiles that
// straddle the diagonal.
#include "common.cuh"
#include "internal.h"

namespace gattn {
namespace {

template <int D>
struct PfCfg {
    static constexpr int BM = 128;
    // d = 256: 64-key tiles (TMEM: O 256 + two S 64 + Q' 128 columns) and P goes to
    // shared memory.  d <= 128: 128-key tiles, P in a TMEM buffer of its own.
    static constexpr int BN = (D == 256) ? 64 : 128;
    static constexpr bool PSMEM = (D == 256);
    // d <= 128: persistent CTAs with their own raw-Q and gate/output buffers, and two
    // threads per query row (8 softmax warps), each owning half of the row's keys in
    // every tile and half of O's columns (four per row, 16 warps, measured slower)
    static constexpr bool PERSIST = !PSMEM;
    static constexpr int NH = PSMEM ? 1 : 2;
    static constexpr bool SPLIT = NH > 1;
    static constexpr int SOFTMAX_WARPS = 4 * NH;
    // d <= 128: a warpgroup of its own runs each item's epilogue and the Q prologue
    // two items ahead, into the other of two Q' buffers in TMEM, so that the softmax
    // warps go from an item's last tile straight to the next item's first.  d = 256:
    // the softmax warps run both (no TMEM left for a second Q').
    static constexpr bool QPW = PERSIST;
    static constexpr int NQB = QPW ? 2 : 1;            // Q' buffers in TMEM: item n uses n % NQB
    static constexpr int SM_WARP0 = QPW ? 4 : 3;       // first softmax warp
    static constexpr int PRO_WARPS = QPW ? 4 : 0;      // prologue warps (the last warpgroup)
    static constexpr int NSB = 2;  // score buffers in TMEM: tile j uses buffer j % 2
    static constexpr int NPB = PSMEM ? 2 : 0;  // P buffers in shared memory
    static constexpr int NSK = PERSIST ? 2 : 3;  // K ring stages
    static constexpr int NSV = PERSIST ? 2 : 3;  // V ring stages
    static constexpr int KCH = D / 64;               // 128-byte chunks along head_dim
    static constexpr int CHUNK_BYTES = BN * 128;     // one K/V TMA box: BN rows x 64 bf16
    static constexpr int TILE_BYTES = BN * D * 2;
    static constexpr int ROWBOX_BYTES = BM * 128;    // one Q/gate/output TMA box: 128 rows x 64 bf16
    static constexpr int QTILE_BYTES = BM * D * 2;
    static constexpr int P_BUF_BYTES = PSMEM ? BM * BN * 2 : 0;  // [BN/64 chunks][128 rows][128 B]
    static constexpr int TM_O = 0;
    static constexpr int TM_S = D;                   // score buffer b at TM_S + b * BN
    static constexpr int TM_Q = D + NSB * BN;
    static constexpr int TM_COLS = 512;
    static_assert(TM_Q + NQB * (D / 2) <= TM_COLS, "TMEM budget");
    // d <= 128: P_j (bf16 pairs) is written over S_j in TMEM, and the issuer of tile j
    // issues S_{j+2} = Q'K'_{j+2}^T right behind PV_j (the tensor pipe runs one
    // thread's MMAs in issue order).  d = 256: P_j in shared memory, S_{j+2} as soon
    // as the softmax has read S_j.
    static constexpr bool P_OVER_S = !PSMEM;
    static constexpr int OFF_QB = 0;                                  // raw Q tile (PERSIST)
    static constexpr int OFF_K = PERSIST ? QTILE_BYTES : 0;
    static constexpr int OFF_V = OFF_K + NSK * TILE_BYTES;
    static constexpr int OFF_GB = OFF_V + NSV * TILE_BYTES;           // gate / output tile (PERSIST)
    static constexpr int OFF_P = OFF_GB + (PERSIST ? QTILE_BYTES : 0);
    static constexpr int OFF_BAR = OFF_P + NPB * P_BUF_BYTES;
    // where the raw Q tile, the gate tile and the staged output live
    static constexpr int OFF_Q = PERSIST ? OFF_QB : OFF_V;
    static constexpr int OFF_G = PERSIST ? OFF_GB : OFF_K;
    static constexpr int OFF_OUT = PERSIST ? OFF_GB : OFF_V;
    static_assert(PERSIST || (QTILE_BYTES <= NSV * TILE_BYTES && QTILE_BYTES <= NSK * TILE_BYTES),
                  "raw Q, gate and output tiles must fit the rings they borrow");
    static constexpr int NBAR = 2 * NSK + 2 * NSV + 21;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int OFF_W = (OFF_MISC + 16 + 127) & ~127;  // qnorm weights, D bf16
    static constexpr int OFF_X = OFF_W + D * 2;                  // exchange between a row's threads (SPLIT)
    static constexpr int SMEM_BYTES = OFF_X + (SPLIT ? 4 * NH * BM * 4 : 0);
    // + slack for 1024-byte alignment; never less than 120 KB, so that a second CTA
    // can never share the SM (each CTA allocates all 512 TMEM columns).
    static constexpr int SMEM_ALLOC = (SMEM_BYTES + 1024) > 122880 ? (SMEM_BYTES + 1024) : 122880;
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    // QPW: warpgroup 0 = producer, two issuers and an idle warp; warpgroups 1-2 the
    // softmax; warpgroup 3 the Q prologues and the epilogues.  The registers of the
    // launch (128 a thread) are split by setmaxnreg: 72 | 168 | 104, summing exactly
    // to the 64 K the block was launched with.
    static constexpr int THREADS = QPW ? 128 * 4 : 96 + 32 * SOFTMAX_WARPS;
    static constexpr int REG_LAUNCH = 128, REG_CTRL = 72, REG_SOFTMAX = 168, REG_PRO = 104;
    static_assert(!QPW || (SM_WARP0 == 4 && SOFTMAX_WARPS == 8 && PRO_WARPS == 4), "one role per warpgroup");
    static_assert(!QPW || 128 * REG_CTRL + 32 * SOFTMAX_WARPS * REG_SOFTMAX + 32 * PRO_WARPS * REG_PRO <=
                              THREADS * REG_LAUNCH,
                  "register split within the launch allocation");
    static constexpr uint32_t IDESC_QK = make_idesc_bf16(128, BN, false);
    static constexpr uint32_t IDESC_PV = make_idesc_bf16(128, D, true);
    static constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 domain: rescale when the max grows by > 2^8
};

struct Bars {
    uint32_t base;
    int nsk, nsv;
    __device__ uint32_t at(int i) const { return base + 8u * (uint32_t)i; }
    __device__ uint32_t k_full(int s) const { return at(s); }
    __device__ uint32_t k_empty(int s) const { return at(nsk + s); }
    __device__ uint32_t v_full(int s) const { return at(2 * nsk + s); }
    __device__ uint32_t v_empty(int s) const { return at(2 * nsk + nsv + s); }
    __device__ int r() const { return 2 * nsk + 2 * nsv; }
    __device__ uint32_t s_full(int i) const { return at(r() + i); }        // S of a tile in buffer i
    __device__ uint32_t s_free(int i) const { return at(r() + 2 + i); }    // S of a tile read out of buffer i
    __device__ uint32_t p_full(int i) const { return at(r() + 4 + i); }    // P_j ready, j % 2 == i
    __device__ uint32_t pv_done(int i) const { return at(r() + 6 + i); }   // PV_j complete, j % 2 == i
    __device__ uint32_t o_final() const { return at(r() + 8); }   // every PV of an item complete
    __device__ uint32_t q_ready() const { return at(r() + 9); }   // an item's Q' in TMEM, its raw Q no longer read
    __device__ uint32_t drain() const { return at(r() + 10); }
    __device__ uint32_t q_full() const { return at(r() + 11); }   // an item's raw Q tile landed
    __device__ uint32_t g_full() const { return at(r() + 12); }   // an item's gate tile landed / output buffer free
    __device__ uint32_t xchg(int q) const { return at(r() + 13 + q); }  // both halves of row quarter q posted
    __device__ uint32_t o_staged() const { return at(r() + 17); }  // every epilogue warp staged an item's output
    __device__ uint32_t o_free() const { return at(r() + 18); }    // an item's epilogue has read O
    // QPW: the softmax posted the row sums of item n, n % 2 == i
    __device__ uint32_t l_full(int i) const { return at(r() + 19 + i); }
};

// ----------------------------------------------------------------- TMA with L2 priorities

// L2 eviction priorities for TMA copies (an access-policy operand; it changes only
// which lines L2 gives up first, never what is read or written): evict_first for
// data touched once, evict_last for tiles that other CTAs or later items read again.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                                 int c2, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                                 int c2, int c3, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tma_store_4d_hint(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2,
                                                  int c3, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%2, %3, %4, %5}], [%1], "
        "%6;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(pol)
        : "memory");
}

// ----------------------------------------------------------------- work items

// Work item u: query tile n_qtiles - 1 - u / (B*H) (heaviest first) of batch and
// head u % (B*H), heads of one KV group adjacent (their CTAs share K/V tiles in
// L2); packed sequences: tile u / H of the table (also heaviest first), head u % H.
// CTA c of n takes items c, 2n - 1 - c, 2n + c, ... (a snake over rounds, so that
// heavy and light tiles share a CTA).
struct TcItem {
    int qt, b, h, n_kv;
    int t0, len;  // the sequence's first token on the S axis of batch b, and its length
    bool direct;  // a partial tile of packed sequences: rows are stored one by one
};

// The launch keeps the item count below 2^31, so u (at most the count plus the
// grid size) and every product here fit 32-bit unsigned arithmetic, whose
// division is a few instructions (the 64-bit one is a long software sequence, run
// by every role at every item boundary).
template <int D, bool GV>
__device__ __forceinline__ bool tc_item(const PrefillParams& p, int c, int n, int r, TcItem& it) {
    using C = PfCfg<D>;
    const unsigned u = (unsigned)r * (unsigned)n + (unsigned)((r & 1) ? n - 1 - c : c);
    const unsigned nh = (unsigned)p.H;
    if (GV && p.vtiles) {
        if (u >= (unsigned)p.n_vtiles * nh) return false;
        const unsigned tile = u / nh;
        const int4 e = p.vtiles[tile];
        it.qt = e.z;
        it.t0 = e.x;
        it.len = e.y;
        it.b = 0;
        it.h = (int)(u - tile * nh);
        it.direct = (it.qt + 1) * C::BM > it.len;  // a TMA store of 128 rows would reach the next sequence
    } else {
        const unsigned bh_count = (unsigned)p.B * nh;
        if (u >= (unsigned)p.n_qtiles * bh_count) return false;
        const unsigned q = u / bh_count;
        it.qt = p.n_qtiles - 1 - (int)q;
        const unsigned bh = u - q * bh_count, b = bh / nh;
        it.b = (int)b;
        it.h = (int)(bh - b * nh);
        it.t0 = 0;
        it.len = p.S;
        it.direct = false;
    }
    it.n_kv = (min(it.len, (it.qt + 1) * C::BM) + C::BN - 1) / C::BN;
    return true;
}

// ----------------------------------------------------------------- producer

template <int D, bool GV>
__device__ void run_producer(const CUtensorMap* tmK, const CUtensorMap* tmV, const CUtensorMap* tmQ,
                             const CUtensorMap* tmG, const CUtensorMap* tmO, const PrefillParams& p, const Bars& bars,
                             uint32_t sbase, int cta, int ncta, volatile int* abort_flag, unsigned int* status) {
    using C = PfCfg<D>;
    // a gate tile per item when the logits vary over head_dim (elementwise, or one
    // head-shared vector per token: the gate map then has a single head)
    const bool gate_tile = GV ? gate_per_dim(p.gate_mode) : p.gate_mode == GATTN_GATE_ELEMENTWISE;
    const bool shared = GV && gate_layout(p.gate_mode) == GATTN_GATE_HEAD_SHARED;
    // raw Q, gate and output tiles pass through L2 once; K'/V tiles are read again by
    // the group's other heads and by later query tiles, so they are the ones L2 keeps
    const uint64_t pol_once = l2_policy_evict_first(), pol_kv = l2_policy_evict_last();
    int nk = 0, nv = 0;  // K' / V tiles issued, over all items
    int jb = 0;          // tiles of the items before the current one
    int n_it = 0;
    int q_last = -1, g_last = -1;  // the items whose raw Q / gate tile copies were issued last
    bool ok = true;
    TcItem it, prev;
    auto row0_of = [&](const TcItem& x) { return x.t0 + x.qt * C::BM; };
    // an item's gate tile into the gate/output buffer, or (no gate tile) just the
    // news that the buffer is free for the item's staged output
    auto gate_in = [&](const TcItem& x) {
        if (gate_tile) {
            mbar_arrive_expect_tx(bars.g_full(), C::QTILE_BYTES);
#pragma unroll
            for (int c = 0; c < C::KCH; ++c)
                tma_load_4d_hint(sbase + C::OFF_G + c * C::ROWBOX_BYTES, tmG, bars.g_full(), c * 64, shared ? 0 : x.h,
                                 row0_of(x), x.b, pol_once);
            g_last = n_it;
        } else {
            mbar_arrive(bars.g_full());
        }
    };
    // an item's output, staged by the softmax warps: TMA stores (rows past S clipped),
    // then wait until the copies have read shared memory (a partial tile of packed
    // sequences was stored row by row instead)
    auto store_out = [&](const TcItem& x) {
        if (x.direct) return;
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
            tma_store_4d_hint(tmO, sbase + C::OFF_OUT + c * C::ROWBOX_BYTES, c * 64, x.h, row0_of(x), x.b, pol_once);
        bulk_commit_group();
        bulk_wait_group_read0();
    };

    // item k's raw Q tile (and with the first item the q norm weights)
    auto load_q = [&](const TcItem& x, int k) {
        mbar_arrive_expect_tx(bars.q_full(), C::QTILE_BYTES + (k == 0 ? D * 2 : 0));
        if (k == 0) bulk_load(sbase + C::OFF_W, p.qnorm_w, D * 2, bars.q_full());
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
            tma_load_4d_hint(sbase + C::OFF_Q + c * C::ROWBOX_BYTES, tmQ, bars.q_full(), c * 64, x.h, row0_of(x), x.b,
                             pol_once);
        q_last = k;
    };
    TcItem nxt;
    bool have = tc_item<D, GV>(p, cta, ncta, 0, it);
    bool q_sent = false;  // the current item's raw Q tile is already on its way
    for (int r = 0; ok && have; ++r, ++n_it) {
        const int g = it.h / (p.H / p.G);
        const bool more = tc_item<D, GV>(p, cta, ncta, r + 1, nxt);
        // raw Q tile: its buffer is free once the previous item's prologue has read it
        // (persistent: normally sent during the previous item already, see below)
        if (!q_sent) {
            if (C::PERSIST && n_it > 0 &&
                !(ok = mbar_wait(bars.q_ready(), (uint32_t)(n_it - 1) & 1u, abort_flag, status)))
                break;
            load_q(it, n_it);
        }
        bool nq_sent = false;  // the next item's raw Q tile is on its way
        // the gate tile is read at the very end of the item: start it on its way to L2 now
        if (gate_tile) {
#pragma unroll
            for (int c = 0; c < C::KCH; ++c)
                tma_prefetch_l2_4d(tmG, c * 64, shared ? 0 : it.h, row0_of(it), it.b);
        }
        // K' is written by the pre-pass kernel just before this one (programmatic
        // dependent launch): wait for it to finish before the first K' load.
        if (n_it == 0) pdl_wait_prerequisites();
        // Persistent: the first item's gate goes straight in; later ones once the
        // previous item's output has been stored.  One item per CTA: the gate tile
        // borrows the K ring after the last K' tile (below), and the V tiles wait
        // until the prologue has read the raw Q tile out of the V ring.
        bool g_done = !C::PERSIST;
        if (C::PERSIST && n_it == 0) {
            gate_in(it);
            g_done = true;
        }
        bool v_open = C::PERSIST;
        // tiles [jb, ke) of K' and V belong to this item.  Persistent: once its K' tiles
        // are all on their way, the next item's first ones (up to the ring's depth) go
        // out from this loop too, while it still waits for ring stages of V.
        const int ke = jb + it.n_kv, ve = jb + it.n_kv;
        const int kx = ke + (C::PERSIST && more ? min(nxt.n_kv, C::NSK) : 0);
        const unsigned long long t0 = global_timer_ns();
        uint32_t spins = 0;
        while (nk < ke || nv < ve) {
            bool progressed = false;
            // persistent: the next item's raw Q tile as soon as this item's prologue has
            // read the buffer, so that it has landed by the time this item ends
            if (C::PERSIST && more && !nq_sent && mbar_test_wait(bars.q_ready(), (uint32_t)n_it & 1u)) {
                load_q(nxt, n_it + 1);
                nq_sent = progressed = true;
            }
            if (!g_done && mbar_test_wait(bars.o_staged(), (uint32_t)(n_it - 1) & 1u)) {
                store_out(prev);
                gate_in(it);
                g_done = progressed = true;
            }
            if (nk < kx &&
                (nk < C::NSK || mbar_test_wait(bars.k_empty(nk % C::NSK), ((uint32_t)(nk / C::NSK) & 1u) ^ 1u))) {
                const int st = nk % C::NSK;
                mbar_arrive_expect_tx(bars.k_full(st), C::TILE_BYTES);
                const uint32_t kdst = sbase + C::OFF_K + st * C::TILE_BYTES;
                const bool cur = nk < ke;
                const int krow = cur ? it.t0 + (nk - jb) * C::BN : nxt.t0 + (nk - ke) * C::BN;
                const int kgrp = cur ? it.b * p.G + g : nxt.b * p.G + nxt.h / (p.H / p.G);
#pragma unroll
                for (int c = 0; c < C::KCH; ++c)
                    tma_load_3d_hint(kdst + c * C::CHUNK_BYTES, tmK, bars.k_full(st), c * 64, krow, kgrp, pol_kv);
                ++nk;
                progressed = true;
            }
            if (!v_open) v_open = mbar_test_wait(bars.q_ready(), 0);
            if (v_open && nv < ve &&
                (nv < C::NSV || mbar_test_wait(bars.v_empty(nv % C::NSV), ((uint32_t)(nv / C::NSV) & 1u) ^ 1u))) {
                const int st = nv % C::NSV;
                mbar_arrive_expect_tx(bars.v_full(st), C::TILE_BYTES);
                const uint32_t vdst = sbase + C::OFF_V + st * C::TILE_BYTES;
#pragma unroll
                for (int c = 0; c < C::KCH; ++c)
                    tma_load_4d_hint(vdst + c * C::CHUNK_BYTES, tmV, bars.v_full(st), c * 64, g,
                                     it.t0 + (nv - jb) * C::BN, it.b, pol_kv);
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
        if (nk < ke || nv != ve) {
            ok = false;
            break;
        }
        if (!g_done) {  // persistent: the previous output has not been staged yet
            if (!(ok = mbar_wait(bars.o_staged(), (uint32_t)(n_it - 1) & 1u, abort_flag, status))) break;
            store_out(prev);
            gate_in(it);
        }
        if (!C::PERSIST && gate_tile) {
            // one item per CTA: the gate tile goes into the K ring once every K' stage
            // has been consumed for the last time
            for (int j = ke > C::NSK ? ke - C::NSK : 0; ok && j < ke; ++j)
                ok = mbar_wait(bars.k_empty(j % C::NSK), (uint32_t)(j / C::NSK) & 1u, abort_flag, status);
            if (!ok) break;
            gate_in(it);
        }
        jb = ke;
        prev = it;
        it = nxt;
        have = more;
        q_sent = nq_sent;
    }
    // the last item's output
    if (ok && n_it > 0 && mbar_wait(bars.o_staged(), (uint32_t)(n_it - 1) & 1u, abort_flag, status)) store_out(prev);
    bulk_wait_group0();
    // Drain: every copy this thread started must land before the CTA can exit.
    if (q_last >= 0) mbar_wait_drain(bars.q_full(), (uint32_t)q_last & 1u, status);
    for (int j = nk > C::NSK ? nk - C::NSK : 0; j < nk; ++j)
        mbar_wait_drain(bars.k_full(j % C::NSK), (uint32_t)(j / C::NSK) & 1u, status);
    for (int j = nv > C::NSV ? nv - C::NSV : 0; j < nv; ++j)
        mbar_wait_drain(bars.v_full(j % C::NSV), (uint32_t)(j / C::NSV) & 1u, status);
    if (g_last >= 0) mbar_wait_drain(bars.g_full(), (uint32_t)g_last & 1u, status);
}

// ----------------------------------------------------------------- MMA issuer

// Two threads issue MMAs: a single thread can issue one tcgen05.mma only every
// ~54 cycles whatever its size (measured on GB300), which at d = 256 (D/16 narrow
// QK^T MMAs per 64-key tile) is slower than the tensor pipe executes them.  So
// there is one issuer per tile parity: issuer i issues QK^T and PV of the tiles j
// with j % 2 == i (j counting tiles over all items), each issuing half the MMAs;
// their MMAs interleave freely in the pipe.  PV_j waits for PV_{j-1} to complete,
// so O sums the tiles in the same order on every run (the result is deterministic).
// The K-steps of S = Q'K'^T (A = Q' in TMEM, B = K' K-major in shared memory) and of
// O += P V (A = P in TMEM, or at d = 256 in shared memory; B = V MN-major in shared
// memory), unrolled at compile time with immediate descriptor offsets (mma_ts_lo):
// a few instructions per MMA, so that the tensor pipe is fed at its own rate even
// while softmax warps of the same sub-partition are busy.
template <int D, int KK>
__device__ __forceinline__ void tc_qk_steps(uint32_t d_tmem, uint32_t q_tmem, uint32_t k_lo) {
    using C = PfCfg<D>;
    if constexpr (KK < D / 16) {
        mma_ts_lo<KK * 8, ((KK >> 2) * C::CHUNK_BYTES + (KK & 3) * 32) / 16>(d_tmem, q_tmem, k_lo, sdesc_sw128_hi(),
                                                                           C::IDESC_QK, KK > 0 ? 1u : 0u);
        tc_qk_steps<D, KK + 1>(d_tmem, q_tmem, k_lo);
    }
}
template <int D, int KK>
__device__ __forceinline__ void tc_pv_steps(uint32_t d_tmem, uint32_t p_tmem, uint32_t p_lo, uint32_t v_lo,
                                            uint32_t acc0) {
    using C = PfCfg<D>;
    if constexpr (KK < C::BN / 16) {
        if constexpr (C::PSMEM)
            mma_ss_lo<((KK >> 2) * (C::BM * 128) + (KK & 3) * 32) / 16, KK * 16 * 128 / 16>(
                d_tmem, p_lo, v_lo, sdesc_sw128_hi(), C::IDESC_PV, KK > 0 ? 1u : acc0);
        else  // keys [16 KK, 16 KK + 16) of half h = KK / 4: P columns 32 h + 8 KK of the score buffer
            mma_ts_lo<KK * 8 + 32 * (KK / 4), KK * 16 * 128 / 16>(d_tmem, p_tmem, v_lo, sdesc_sw128_hi(), C::IDESC_PV,
                                                                 KK > 0 ? 1u : acc0);
        tc_pv_steps<D, KK + 1>(d_tmem, p_tmem, p_lo, v_lo, acc0);
    }
}

template <int D>
__device__ __forceinline__ bool issue_qk(int j, const Bars& bars, uint32_t tm, uint32_t q_col, uint32_t k_lo0,
                                         volatile int* abort_flag, unsigned int* status) {
    using C = PfCfg<D>;
    const int sb = j & 1;
    // score buffer sb was last used by tile j-2.  P over S: P_{j-2} there is read by
    // PV_{j-2}, which this thread issued before.  Else the buffer is free once the
    // softmax has read S_{j-2}.
    if (!C::P_OVER_S && j >= 2 && !mbar_wait(bars.s_free(sb), (uint32_t)((j >> 1) - 1) & 1u, abort_flag, status))
        return false;
    const int st = j % C::NSK;
    if (!mbar_wait(bars.k_full(st), (uint32_t)(j / C::NSK) & 1u, abort_flag, status)) return false;
    tc_fence_after();
    tc_qk_steps<D, 0>(tm + C::TM_S + sb * C::BN, tm + q_col, k_lo0 + (uint32_t)((st * C::TILE_BYTES) >> 4));
    tc_commit(bars.k_empty(st));
    tc_commit(bars.s_full(sb));
    return true;
}

// PV_j; the first tile of an item (first) overwrites O, once the previous item's
// epilogue (item n_it - 1) has read it
template <int D>
__device__ __forceinline__ bool issue_pv(int j, bool first, int n_it, const Bars& bars, uint32_t tm, uint32_t v_lo0,
                                         uint32_t p_lo0, volatile int* abort_flag, unsigned int* status) {
    using C = PfCfg<D>;
    // The waits that are normally over already come first, so that the MMAs follow
    // the wait for P_j directly.  O accumulates the PVs in tile order, run after run:
    // PV_j starts once the other issuer's PV_{j-1} has completed (its QKs keep the
    // pipe busy meanwhile).
    if (j >= 1 && !mbar_wait(bars.pv_done((j - 1) & 1), (uint32_t)((j - 1) >> 1) & 1u, abort_flag, status))
        return false;
    if (first && n_it > 0 && !mbar_wait(bars.o_free(), (uint32_t)(n_it - 1) & 1u, abort_flag, status)) return false;
    const int st = j % C::NSV;
    if (!mbar_wait(bars.v_full(st), (uint32_t)(j / C::NSV) & 1u, abort_flag, status)) return false;
    if (!mbar_wait(bars.p_full(j & 1), (uint32_t)(j >> 1) & 1u, abort_flag, status)) return false;
    tc_fence_after();
    tc_pv_steps<D, 0>(tm + C::TM_O, tm + C::TM_S + (j & 1) * C::BN, p_lo0 + (uint32_t)(((j & 1) * C::P_BUF_BYTES) >> 4),
                      v_lo0 + (uint32_t)((st * C::TILE_BYTES) >> 4), first ? 0u : 1u);
    tc_commit(bars.v_empty(st));
    tc_commit(bars.pv_done(j & 1));
    return true;
}

template <int D, bool GV>
__device__ void run_mma(int parity, const PrefillParams& p, const Bars& bars, uint32_t sbase, uint32_t tm, int cta,
                        int ncta, volatile int* abort_flag, unsigned int* status) {
    using C = PfCfg<D>;
    const uint32_t kdesc0 = sdesc_sw128_lo(sbase + C::OFF_K, 16);
    const uint32_t vdesc0 = sdesc_sw128_lo(sbase + C::OFF_V, C::CHUNK_BYTES);
    const uint32_t pdesc0 = sdesc_sw128_lo(sbase + C::OFF_P, 16);
    bool ok = true;
    int jb = 0, n_it = 0;
    TcItem it;
    for (int r = 0; ok && tc_item<D, GV>(p, cta, ncta, r, it); ++r, ++n_it) {
        const int je = jb + it.n_kv;
        // the item's Q' is in TMEM
        if (!(ok = mbar_wait(bars.q_ready(), (uint32_t)n_it & 1u, abort_flag, status))) break;
        tc_fence_after();
        const uint32_t q_col = (uint32_t)(C::TM_Q + (n_it % C::NQB) * (D / 2));  // the item's Q' buffer
        const int j0 = jb + ((jb & 1) != parity ? 1 : 0);
        if (j0 < je) ok = issue_qk<D>(j0, bars, tm, q_col, kdesc0, abort_flag, status);
        for (int j = j0; ok && j < je; j += 2) {
            if constexpr (C::P_OVER_S) {
                // S_{j+2} is written over P_j, right behind the PV_j that reads it
                if (!issue_pv<D>(j, j == jb, n_it, bars, tm, vdesc0, pdesc0, abort_flag, status)) { ok = false; break; }
                if (j + 2 < je && !issue_qk<D>(j + 2, bars, tm, q_col, kdesc0, abort_flag, status)) { ok = false; break; }
            } else {
                // QK of this issuer's next tile goes out as soon as its score buffer is
                // free, ahead of the PV that is still waiting for its P
                if (j + 2 < je && !issue_qk<D>(j + 2, bars, tm, q_col, kdesc0, abort_flag, status)) { ok = false; break; }
                if (!issue_pv<D>(j, j == jb, n_it, bars, tm, vdesc0, pdesc0, abort_flag, status)) { ok = false; break; }
            }
        }
        if (ok) tc_commit(bars.o_final());  // count 2: both issuers' PVs of the item complete
        jb = je;
    }
    tc_commit(bars.drain());
}

// ----------------------------------------------------------------- gated output

// Columns [c, c + 32) of one query row of the output: o (the unnormalised O row from
// TMEM, fp32 bits) / l times act(gate), or plus act(gate) for an additive gate, as
// bf16 pairs handed to put(col, w0, w1, w2, w3), 8 columns at a time.  Logits that
// vary over head_dim are read from the row-major gate tile at gbase; otherwise the
// factors are the headwise (or unit) ones: out = o gh + gha.
template <bool GV, typename Put>
__device__ __forceinline__ void gate_out32(const PrefillParams& p, const uint32_t* ov, int c, int row, uint32_t gbase,
                                           bool elementwise, bool additive, float inv_l, float gh, float gha,
                                           Put&& put) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        float gv[8], ga[8];  // out = o * gv + ga
        if (elementwise) {
            float f[8];
            unpack8(lds_v4(rowtile_addr(gbase, row, c + 8 * q4)), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if constexpr (GV) {
                    const float a = gate_act(f[e], sigmoid_tanh(f[e]), p.gate_mode);
                    gv[e] = additive ? inv_l : inv_l * a;
                    ga[e] = additive ? a : 0.f;
                } else {
                    gv[e] = inv_l * sigmoid_tanh(f[e]);
                    ga[e] = 0.f;
                }
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                gv[e] = gh;
                ga[e] = gha;
            }
        }
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = 2 * i;
            const float o0 = __uint_as_float(ov[8 * q4 + e]), o1 = __uint_as_float(ov[8 * q4 + e + 1]);
            if constexpr (GV)
                w[i] = pack_bf16x2(fmaf(o0, gv[e], ga[e]), fmaf(o1, gv[e + 1], ga[e + 1]));
            else
                w[i] = pack_bf16x2(o0 * gv[e], o1 * gv[e + 1]);
        }
        put(c + 8 * q4, w[0], w[1], w[2], w[3]);
    }
}

// ----------------------------------------------------------------- Q prologue / epilogue warpgroup (QPW)

// The warpgroup runs, one thread per query row (warp w reaches TMEM lanes
// 32 (w % 4) + [0, 32)), the Q prologues of items 0 and 1 and then, per item n, the
// epilogue of item n followed by the prologue of item n + 2, so that the softmax
// warps go from an item's last tile straight to the next one.
//
// Prologue of item n: Q' = rope(rmsnorm(q)) as bf16 pairs into TMEM buffer n % 2,
// which item n - 2's QK MMAs last read (this warpgroup saw them complete in that
// item's epilogue); the raw Q tile has landed (q_full).  The arithmetic is the
// split-row prologue of the softmax warps (d = 256) in the same order (the two
// halves' sums of squares, each over four interleaved partial sums, then added;
// every rotated pair on its own), so Q' is bit for bit the same either way.
//
// Epilogue of item n: the row sum (the softmax's two halves, posted in shared memory
// buffer n % 2), every PV of the item complete (o_final), the gate tile landed, then
// O / l * act(gate) (additive gate: O / l + act(gate)) as bf16 into the staged output
// tile (over the gate tile, each thread overwriting only gate values it has read),
// which the producer writes to [B,S,H*d] with TMA stores (rows past S clipped); a
// partial tile of packed sequences is stored row by row instead.  O is released
// (o_free) once read, so that the next item's first PV may overwrite it.
template <int D, bool GV>
__device__ void run_qwg(const PrefillParams& p, const Bars& bars, uint32_t sbase, const float* xsum, uint32_t tm,
                        int quarter, int lane, int cta, int ncta, volatile int* abort_flag) {
    using C = PfCfg<D>;
    constexpr int OC = D / C::NH;
    const int row = quarter * 32 + lane;
    const uint32_t tl = tm + ((uint32_t)(quarter * 32) << 16);
    const uint32_t qbase = sbase + C::OFF_Q;
    const uint32_t wbase = sbase + C::OFF_W;

    auto prologue = [&](const TcItem& it, int n) -> bool {
        if (!__all_sync(0xffffffffu, mbar_wait(bars.q_full(), (uint32_t)n & 1u, abort_flag, p.status))) return false;
        tc_fence_after();
        const int t = it.qt * C::BM + row;  // from the start of the sequence
        const bool valid = t < it.len;
        const int64_t tok = (int64_t)it.b * p.S + it.t0 + (valid ? t : 0);
        float sq = 0.f;
#pragma unroll
        for (int hf = 0; hf < C::NH; ++hf) {
            float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < OC / 8; ++c) {
                float f[8];
                unpack8(lds_v4(rowtile_addr(qbase, row, hf * OC + 8 * c)), f);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss[e & 3] = fmaf(f[e], f[e], ss[e & 3]);
            }
            const float part = (ss[0] + ss[1]) + (ss[2] + ss[3]);
            sq = hf == 0 ? part : sq + part;
        }
        const float rinv = rsqrtf(sq / (float)D + p.eps);
        const float posf = valid ? (p.pos ? (float)p.pos[tok] : (float)t) : 0.f;
        const int half = p.rd >> 1;
        const uint32_t qcol = tl + (uint32_t)(C::TM_Q + (n & 1) * (D / 2));
#pragma unroll 1
        for (int i0 = 0; i0 < half; i0 += 8) {
            float xa[8], xb[8], wa[8], wb[8];
            unpack8(lds_v4(rowtile_addr(qbase, row, i0)), xa);
            unpack8(lds_v4(rowtile_addr(qbase, row, i0 + half)), xb);
            unpack8(lds_v4(wbase + 2 * i0), wa);
            unpack8(lds_v4(wbase + 2 * (i0 + half)), wb);
            uint32_t lo[4], hi[4];
            rope_rotate8(xa, xb, wa, wb, p.inv_freq + i0, posf, rinv, lo, hi);
            __syncwarp();
            tmem_st4(qcol + (i0 >> 1), lo[0], lo[1], lo[2], lo[3]);
            tmem_st4(qcol + ((i0 + half) >> 1), hi[0], hi[1], hi[2], hi[3]);
        }
#pragma unroll 1
        for (int e0 = p.rd; e0 < D; e0 += 8) {
            float x[8], w[8];
            unpack8(lds_v4(rowtile_addr(qbase, row, e0)), x);
            unpack8(lds_v4(wbase + 2 * e0), w);
            uint32_t o[4];
            scale8_bf16(x, w, rinv, o);
            __syncwarp();
            tmem_st4(qcol + (e0 >> 1), o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();  // our reads of the raw Q tile happen before the next copy overwrites it
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.q_ready());
        return true;
    };

    auto epilogue = [&](const TcItem& it, int n) -> bool {
        const int t = it.qt * C::BM + row;
        const bool valid = t < it.len;
        const int64_t tok = (int64_t)it.b * p.S + it.t0 + (valid ? t : 0);
        const bool headwise = (GV ? gate_layout(p.gate_mode) : p.gate_mode) == GATTN_GATE_HEADWISE && valid;
        bf16 z_head = __float2bfloat16(0.f);
        if (headwise)
            z_head = static_cast<const bf16*>(p.gate)[tok * p.gate_tok_stride + (int64_t)it.h * p.gate_head_stride];
        if (!__all_sync(0xffffffffu, mbar_wait(bars.l_full(n & 1), (uint32_t)(n >> 1) & 1u, abort_flag, p.status)))
            return false;
        const float* xs = xsum + (n & 1) * C::NH * C::BM;
        float l_row = xs[row];
#pragma unroll
        for (int i = 1; i < C::NH; ++i) l_row += xs[i * C::BM + row];
        if (!__all_sync(0xffffffffu, mbar_wait(bars.o_final(), (uint32_t)n & 1u, abort_flag, p.status))) return false;
        // the gate/output buffer holds this item's gate tile (or is free)
        if (!__all_sync(0xffffffffu, mbar_wait(bars.g_full(), (uint32_t)n & 1u, abort_flag, p.status))) return false;
        tc_fence_after();
        const bool elementwise = GV ? gate_per_dim(p.gate_mode) : p.gate_mode == GATTN_GATE_ELEMENTWISE;
        const bool additive = GV && gate_additive(p.gate_mode);
        const float inv_l = 1.f / l_row;
        float gate_head = 1.f;  // the activation of the headwise logit
        if (headwise) {
            const float z = __bfloat162float(z_head);
            gate_head = GV ? gate_act(z, sigmoid_tanh(z), p.gate_mode) : sigmoid_tanh(z);
        }
        const float gh = additive ? inv_l : inv_l * gate_head, gha = additive ? gate_head : 0.f;
        bf16* orow = static_cast<bf16*>(p.out) + (tok * p.H + it.h) * D;
        const uint32_t gbase = sbase + C::OFF_G;
        const uint32_t obase = sbase + C::OFF_OUT;
        const bool direct = it.direct;
        auto put = [&](int col, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
            if (!direct) sts_v4(rowtile_addr(obase, row, col), w0, w1, w2, w3);
            else if (valid) *reinterpret_cast<uint4*>(orow + col) = make_uint4(w0, w1, w2, w3);
        };
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t ro[32];
            __syncwarp();
            tmem_ld32(tl + C::TM_O + c0, ro);
            if (c0 + 32 == D) {  // all of O read: the next item's first PV may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.o_free());
            }
            gate_out32<GV>(p, ro, c0, row, gbase, elementwise, additive, inv_l, gh, gha, put);
        }
        // the output buffer may be written out (a directly stored tile only frees it)
        fence_proxy_async_smem();  // the TMA stores read the staged tile through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.o_staged());
        return true;
    };

    TcItem it[3];  // items n, n + 1, n + 2
    bool have[3];
    have[0] = tc_item<D, GV>(p, cta, ncta, 0, it[0]);
    have[1] = tc_item<D, GV>(p, cta, ncta, 1, it[1]);
    if (have[0] && !prologue(it[0], 0)) return;
    if (have[1] && !prologue(it[1], 1)) return;
    for (int n = 0; have[0]; ++n) {
        if (!epilogue(it[0], n)) return;
        have[2] = tc_item<D, GV>(p, cta, ncta, n + 2, it[2]);
        if (have[2] && !prologue(it[2], n + 2)) return;
        it[0] = it[1];
        have[0] = have[1];
        it[1] = it[2];
        have[1] = have[2];
    }
}

// ----------------------------------------------------------------- softmax / prologue / epilogue

// GV: the gate variants (head-shared logits, NS-sigmoid, SiLU, additive) and
// packed variable-length sequences -- a second instance of the kernel, so that
// the default (batched, elementwise / headwise multiplicative sigmoid gate)
// compiles exactly as it would alone.
template <int D, bool GV>
__device__ void run_softmax(const PrefillParams& p, const Bars& bars, uint32_t sbase, uint8_t* smem_x, uint32_t tm,
                            int quarter, int hf, int lane, int cta, int ncta, volatile int* abort_flag) {
    using C = PfCfg<D>;
    constexpr int NH = C::NH;             // threads per query row
    constexpr int KB = C::BN / NH;        // keys of every tile owned by this thread: [hf KB, hf KB + KB)
    static_assert(KB == 64, "one 64-column TMEM load of S and one 32-column store of P per thread and tile");
    constexpr int OC = D / NH;            // O columns owned by this thread: [hf OC, hf OC + OC)
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tl = tm + lane_off;
    // With several threads per row (warps w, w + 4, ... share the row's TMEM lanes)
    // the parts swap values through shared memory and then meet on an mbarrier (one
    // phase per use: every prologue, tile and epilogue).
    float* xmax = reinterpret_cast<float*>(smem_x);  // [2][NH][BM] tile maxima
    float* xsum = xmax + 2 * NH * C::BM;             // [NH][BM] row sums (QPW: [2][NH][BM], by item parity)
    float* xss = xsum + NH * C::BM;                  // [NH][BM] sums of squares of q (not QPW)
    const uint32_t xbar = bars.xchg(quarter);
    int xphase = 0;
    auto meet = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(xbar);
        return __all_sync(0xffffffffu, mbar_wait(xbar, (uint32_t)(xphase++) & 1u, abort_flag, p.status));
    };

    // ---- fused Q prologue of item k: rmsnorm then partial rotate-half RoPE, bf16
    // into TMEM.  The raw row is read from the item's Q tile (rows past the sequence
    // end were zero-filled by TMA).  Split rows: each half sums the squares of its
    // columns, and the 8-column chunks (a rotated pair (i, i + rd/2) going with the
    // chunk of i) are shared out alternately.  Q' of the previous item is no longer
    // read: the softmax has seen the scores of its last tile.
    auto prologue = [&](const TcItem& it, int k) -> bool {
        const int t = it.qt * C::BM + row;  // from the start of the sequence
        const bool valid = t < it.len;
        const int64_t tok = (int64_t)it.b * p.S + it.t0 + (valid ? t : 0);
        if (!__all_sync(0xffffffffu, mbar_wait(bars.q_full(), (uint32_t)k & 1u, abort_flag, p.status))) return false;
        const uint32_t qbase = sbase + C::OFF_Q;
        const uint32_t wbase = sbase + C::OFF_W;
        float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < OC / 8; ++c) {
            float f[8];
            unpack8(lds_v4(rowtile_addr(qbase, row, hf * OC + 8 * c)), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss[e & 3] = fmaf(f[e], f[e], ss[e & 3]);
        }
        float sq = (ss[0] + ss[1]) + (ss[2] + ss[3]);
        if constexpr (C::SPLIT) {
            xss[hf * C::BM + row] = sq;
            if (!meet()) return false;
            sq = xss[row];
#pragma unroll
            for (int i = 1; i < NH; ++i) sq += xss[i * C::BM + row];
        }
        const float rinv = rsqrtf(sq / (float)D + p.eps);
        const float posf = valid ? (p.pos ? (float)p.pos[tok] : (float)t) : 0.f;
        const int half = p.rd >> 1;
        for (int i0 = 8 * hf; i0 < half; i0 += 8 * NH) {
            float xa[8], xb[8], wa[8], wb[8];
            unpack8(lds_v4(rowtile_addr(qbase, row, i0)), xa);
            unpack8(lds_v4(rowtile_addr(qbase, row, i0 + half)), xb);
            unpack8(lds_v4(wbase + 2 * i0), wa);
            unpack8(lds_v4(wbase + 2 * (i0 + half)), wb);
            uint32_t lo[4], hi[4];
            rope_rotate8(xa, xb, wa, wb, p.inv_freq + i0, posf, rinv, lo, hi);
            __syncwarp();
            tmem_st4(tl + C::TM_Q + (i0 >> 1), lo[0], lo[1], lo[2], lo[3]);
            tmem_st4(tl + C::TM_Q + ((i0 + half) >> 1), hi[0], hi[1], hi[2], hi[3]);
        }
        for (int e0 = p.rd + 8 * hf; e0 < D; e0 += 8 * NH) {
            float x[8], w[8];
            unpack8(lds_v4(rowtile_addr(qbase, row, e0)), x);
            unpack8(lds_v4(wbase + 2 * e0), w);
            uint32_t o[4];
            scale8_bf16(x, w, rinv, o);
            __syncwarp();
            tmem_st4(tl + C::TM_Q + (e0 >> 1), o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();  // our reads of the raw Q tile happen before the next copy overwrites it
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.q_ready());
        return true;
    };

    const float sl2 = p.scale_log2;
    // the exponent's reference: the logits' bound when it is small enough (the same
    // in every thread), else the running maximum
    const float m_fix = fixed_logit_ref(static_cast<const bf16*>(p.qnorm_w), static_cast<const bf16*>(p.knorm_w), D,
                                        sl2);
    const bool fixed = m_fix != INFINITY;
    bool s_seen = false;  // the next tile's scores were seen in TMEM already
    int jb = 0, n_it = 0;
    TcItem item, next;
    bool have = tc_item<D, GV>(p, cta, ncta, 0, item);
    if (!C::QPW && have && !prologue(item, 0)) return;
    for (int r = 0; have; ++r, ++n_it) {
        const int qt = item.qt, b = item.b, h = item.h, n_kv = item.n_kv;
        const int t = qt * C::BM + row;  // from the start of the sequence
        const bool valid = t < item.len;
        const int64_t tok = (int64_t)b * p.S + item.t0 + (valid ? t : 0);
        // a headwise logit: loaded now, activated in the epilogue (so that nothing
        // waits for the load before the first scores)
        const bool headwise = (GV ? gate_layout(p.gate_mode) : p.gate_mode) == GATTN_GATE_HEADWISE && valid;
        bf16 z_head = __float2bfloat16(0.f);
        if (headwise)
            z_head = static_cast<const bf16*>(p.gate)[tok * p.gate_tok_stride + (int64_t)h * p.gate_head_stride];

        // ---- main loop: online softmax over the KV tiles this query tile can see
        const int row_min = qt * C::BM;
        float m_ref = -INFINITY;  // reference max (log2 domain) shared by O and l (and by both halves of a row)
        float l = 0.f;            // this thread's share of the row sum
        for (int j = 0; j < n_kv; ++j) {
            const int jg = jb + j;  // tile counter over all items: buffers and phases
            const int sb = jg & 1;
            const uint32_t s_col = C::TM_S + sb * C::BN;
            if (!__all_sync(0xffffffffu, s_seen) &&
                !__all_sync(0xffffffffu, mbar_wait(bars.s_full(sb), (uint32_t)(jg >> 1) & 1u, abort_flag, p.status)))
                return;
            tc_fence_after();
            float s[KB];
            {
                uint32_t rr[64];
                tmem_ld64(tl + s_col + hf * KB, rr);
#pragma unroll
                for (int e = 0; e < 64; ++e) s[e] = __uint_as_float(rr[e]);
            }
            // S_j is in registers: its buffer may now take the scores of tile j + 2 (P
            // over S: once PV_j has read P_j from it, which the issuers see to)
            if constexpr (!C::P_OVER_S) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.s_free(sb));
            }
            const int key0 = j * C::BN + hf * KB;
            if (key0 + KB - 1 > row_min) {
#pragma unroll
                for (int c = 0; c < KB; ++c)
                    if (key0 + c > t) s[c] = -INFINITY;
            }
            if (fixed) {
                m_ref = m_fix;
            } else {
                float mx[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
                for (int c = 8; c < KB; c += 2) mx[(c >> 1) & 7] = max3(mx[(c >> 1) & 7], s[c], s[c + 1]);
                float mt = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                if constexpr (C::SPLIT) {
                    // the row's maximum over the whole tile (buffer jg%2, so a slow partner
                    // still reading tile jg-1 is never overwritten)
                    xmax[((jg & 1) * NH + hf) * C::BM + row] = mt;
                    if (!meet()) return;
#pragma unroll
                    for (int i = 0; i < NH; ++i)
                        if (i != hf) mt = fmaxf(mt, xmax[((jg & 1) * NH + i) * C::BM + row]);
                }
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
                    // O is only touched once every earlier P V of the item has landed (the
                    // two issuers' PVs may complete in either order).
                    if (!__all_sync(0xffffffffu, mbar_wait(bars.pv_done((jg - 1) & 1), (uint32_t)((jg - 1) >> 1) & 1u,
                                                           abort_flag, p.status)))
                        return;
                    if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(bars.pv_done(jg & 1), (uint32_t)((jg - 2) >> 1) & 1u,
                                                                      abort_flag, p.status)))
                        return;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = hf * OC; c < (hf + 1) * OC; c += 32) {
                        uint32_t rr[32];
                        tmem_ld32(tl + C::TM_O + c, rr);
#pragma unroll
                        for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
                        tmem_st32(tl + C::TM_O + c, rr);
                    }
                }
            }
            // whether the next tile's scores are in, asked now and used after the
            // exponentials, so that the answer is not waited for
            s_seen = j + 1 < n_kv && mbar_test_wait(bars.s_full(sb ^ 1), (uint32_t)((jg + 1) >> 1) & 1u);
            // P = exp2(s * scale * log2e - m_ref), packed bf16: over this thread's own
            // scores in TMEM (this half's keys to columns [hf KB, hf KB + KB/2) of the
            // score buffer), or (PSMEM) as this thread's 128-byte-swizzled row of P
            // buffer jg%2 in shared memory.
            float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            const float mref = m_ref;
            if constexpr (C::PSMEM) {
                // P buffer jg%2 held P_{jg-2}: PV_{jg-2} must have finished reading it
                if (jg >= 2 && !__all_sync(0xffffffffu, mbar_wait(bars.pv_done(jg & 1), (uint32_t)((jg - 2) >> 1) & 1u,
                                                                   abort_flag, p.status)))
                    return;
                const uint32_t pbase = sbase + C::OFF_P + (jg & 1) * C::P_BUF_BYTES;
#pragma unroll
                for (int c8 = 0; c8 < C::BN / 8; ++c8) {
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p0 = ex2_approx(fmaf(s[8 * c8 + 2 * e], sl2, -mref));
                        const float p1 = ex2_approx(fmaf(s[8 * c8 + 2 * e + 1], sl2, -mref));
                        rs[(2 * c8 + (e >> 1)) & 7] += p0 + p1;
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                    const uint32_t addr = pbase + (uint32_t)(c8 >> 3) * (C::BM * 128) + sw128_offset(row, c8 & 7);
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(pk[0]), "r"(pk[1]),
                                 "r"(pk[2]), "r"(pk[3])
                                 : "memory");
                }
                l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
                fence_proxy_async_smem();  // the tensor core reads P through the async proxy
                tmem_wait_st();            // an O rescale above, if any, has landed
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.p_full(jg & 1));
            } else {
                uint32_t pk[KB / 2];
                float2 rs2[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
                const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(-mref, -mref);
#pragma unroll
                for (int e = 0; e < KB / 2; ++e) {
                    const float2 x = fma2(make_float2(s[2 * e], s[2 * e + 1]), sl2x2, negm);
                    const float2 pe = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    rs2[e & 3] = add2(rs2[e & 3], pe);
                    pk[e] = pack_bf16x2(pe.x, pe.y);
                }
                tmem_st32(tl + s_col + hf * KB, pk);
                l += ((rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y)) + ((rs2[2].x + rs2[2].y) + (rs2[3].x + rs2[3].y));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.p_full(jg & 1));
            }
        }

        const bool more = tc_item<D, GV>(p, cta, ncta, r + 1, next);
        if constexpr (C::QPW) {
            // this half's row sum to the epilogue warpgroup (buffer n_it % 2), which
            // finishes the item; on to the next item's first tile
            xsum[((n_it & 1) * NH + hf) * C::BM + row] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.l_full(n_it & 1));
            jb += n_kv;
            item = next;
            have = more;
            continue;
        }
        // ---- the next item's Q prologue: its first QK MMAs then run during this epilogue
        if (more && !prologue(next, n_it + 1)) return;

        // ---- epilogue: O / l * act(gate) (additive gate: O / l + act(gate)) -> bf16, this
        // thread's O columns, into the output tile (over the gate tile, each thread
        // overwriting only gate values it has read; d = 256: in the idle V ring); the
        // producer writes it to [B,S,H*d] with TMA stores (rows past S clipped).  A
        // partial tile of packed sequences is stored row by row instead (a 128-row TMA
        // store would reach into the next sequence).
        float l_row = l;
        if constexpr (C::SPLIT) {
            xsum[hf * C::BM + row] = l;
            if (!meet()) return;
            l_row = xsum[row];
#pragma unroll
            for (int i = 1; i < NH; ++i) l_row += xsum[i * C::BM + row];
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bars.o_final(), (uint32_t)n_it & 1u, abort_flag, p.status))) return;
        const bool elementwise = GV ? gate_per_dim(p.gate_mode) : p.gate_mode == GATTN_GATE_ELEMENTWISE;
        const bool additive = GV && gate_additive(p.gate_mode);
        // persistent: the gate/output buffer holds this item's gate tile (or is free)
        if ((C::PERSIST || elementwise) &&
            !__all_sync(0xffffffffu, mbar_wait(bars.g_full(), (uint32_t)n_it & 1u, abort_flag, p.status)))
            return;
        tc_fence_after();
        const float inv_l = 1.f / l_row;
        // out = o * gv + ga
        float gate_head = 1.f;  // the activation of the headwise logit
        if (headwise) {
            const float z = __bfloat162float(z_head);
            gate_head = GV ? gate_act(z, sigmoid_tanh(z), p.gate_mode) : sigmoid_tanh(z);
        }
        const float gh = additive ? inv_l : inv_l * gate_head, gha = additive ? gate_head : 0.f;
        bf16* orow = static_cast<bf16*>(p.out) + (tok * p.H + h) * D;
        const uint32_t gbase = sbase + C::OFF_G;
        const uint32_t obase = sbase + C::OFF_OUT;
        const bool direct = item.direct;
        auto put = [&](int col, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
            if (!direct) sts_v4(rowtile_addr(obase, row, col), w0, w1, w2, w3);
            else if (valid) *reinterpret_cast<uint4*>(orow + col) = make_uint4(w0, w1, w2, w3);
        };
        // persistent: all of this thread's O columns are read first, so that the next
        // item's first PV may overwrite O while the outputs are formed
        constexpr int OCH = C::PERSIST ? OC : 32;
#pragma unroll 1
        for (int c0 = hf * OC; c0 < (hf + 1) * OC; c0 += OCH) {
            uint32_t ro[OCH];
            __syncwarp();
#pragma unroll
            for (int c = 0; c < OCH; c += 32)
                tmem_ld32(tl + C::TM_O + c0 + c, *reinterpret_cast<uint32_t(*)[32]>(ro + c));
            if (C::PERSIST) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.o_free());
            }
#pragma unroll
            for (int c1 = 0; c1 < OCH; c1 += 32)
                gate_out32<GV>(p, ro + c1, c0 + c1, row, gbase, elementwise, additive, inv_l, gh, gha, put);
        }
        // the output buffer may be written out (a directly stored tile only frees it)
        fence_proxy_async_smem();  // the TMA stores read the staged tile through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.o_staged());
        jb += n_kv;
        item = next;
        have = more;
    }
}

// ----------------------------------------------------------------- kernel

template <int D, bool GV>
__global__ void __launch_bounds__(PfCfg<D>::THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmG,
                      const __grid_constant__ CUtensorMap tmO, const __grid_constant__ PrefillParams p) {
    using C = PfCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Bars bars{sbase + C::OFF_BAR, C::NSK, C::NSV};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    const int cta = (int)blockIdx.x, ncta = (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NSK; ++s) {
            mbar_init(bars.k_full(s), 1);
            mbar_init(bars.k_empty(s), 1);
        }
        for (int s = 0; s < C::NSV; ++s) {
            mbar_init(bars.v_full(s), 1);
            mbar_init(bars.v_empty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bars.s_full(i), 1);
            mbar_init(bars.s_free(i), C::SOFTMAX_WARPS);
            mbar_init(bars.p_full(i), C::SOFTMAX_WARPS);
            mbar_init(bars.pv_done(i), 1);
        }
        for (int q = 0; q < 4; ++q) mbar_init(bars.xchg(q), C::NH);
        mbar_init(bars.o_final(), 2);
        mbar_init(bars.q_ready(), C::QPW ? C::PRO_WARPS : C::SOFTMAX_WARPS);
        for (int i = 0; i < 2; ++i) mbar_init(bars.l_full(i), C::SOFTMAX_WARPS);
        mbar_init(bars.o_staged(), C::QPW ? C::PRO_WARPS : C::SOFTMAX_WARPS);
        mbar_init(bars.o_free(), C::QPW ? C::PRO_WARPS : C::SOFTMAX_WARPS);
        mbar_init(bars.drain(), 2);
        mbar_init(bars.q_full(), 1);
        mbar_init(bars.g_full(), 1);
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
        tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;

    if constexpr (C::QPW) {
        if (warp >= C::SM_WARP0 + C::SOFTMAX_WARPS) {
            regs_lower<C::REG_PRO>();
            run_qwg<D, GV>(p, bars, sbase, reinterpret_cast<const float*>(smem + C::OFF_X) + 2 * C::NH * C::BM, tm,
                           warp & 3, lane, cta, ncta, abort_flag);
        } else if (warp >= C::SM_WARP0) {
            regs_raise<C::REG_SOFTMAX>();
            run_softmax<D, GV>(p, bars, sbase, smem + C::OFF_X, tm, warp & 3, (warp - C::SM_WARP0) >> 2, lane, cta,
                               ncta, abort_flag);
        } else {
            regs_lower<C::REG_CTRL>();
            if (warp == 0) {
                if (lane == 0)
                    run_producer<D, GV>(&tmK, &tmV, &tmQ, &tmG, &tmO, p, bars, sbase, cta, ncta, abort_flag, p.status);
            } else if (warp == 1 || warp == 2) {
                if (lane == 0) {
                    run_mma<D, GV>(warp - 1, p, bars, sbase, tm, cta, ncta, abort_flag, p.status);
                    // no MMA of either issuer may still be in flight when TMEM is released
                    if (warp == 2) mbar_wait_drain(bars.drain(), 0, p.status);
                }
            }
            __syncwarp();
        }
    } else if (warp == 0) {
        if (lane == 0) run_producer<D, GV>(&tmK, &tmV, &tmQ, &tmG, &tmO, p, bars, sbase, cta, ncta, abort_flag, p.status);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) run_mma<D, GV>(0, p, bars, sbase, tm, cta, ncta, abort_flag, p.status);
        __syncwarp();
    } else if (warp == 2) {
        if (lane == 0) {
            run_mma<D, GV>(1, p, bars, sbase, tm, cta, ncta, abort_flag, p.status);
            // Whatever happened, no MMA of either issuer may still be in flight when TMEM is released.
            mbar_wait_drain(bars.drain(), 0, p.status);
        }
        __syncwarp();
    } else {
        run_softmax<D, GV>(p, bars, sbase, smem + C::OFF_X, tm, warp & 3, (warp - C::SM_WARP0) >> 2, lane, cta,
                           ncta, abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, C::TM_COLS);
    }
}

template <int D>
cudaError_t launch_d(const PrefillParams& p, const PrefillMaps& maps, cudaStream_t stream, cudaEvent_t ev_start,
                     cudaEvent_t ev_stop) {
    using C = PfCfg<D>;
    const bool gv = !gate_plain(p.gate_mode) || gate_layout(p.gate_mode) == GATTN_GATE_HEAD_SHARED || p.vtiles;
    auto kernel = gv ? prefill_tc_kernel<D, true> : prefill_tc_kernel<D, false>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kernel), C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    if (C::QPW) {
        // the setmaxnreg split draws on the launch's registers: never launch with fewer
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kernel))) != cudaSuccess) return e;
        if (fa.numRegs != C::REG_LAUNCH) return cudaErrorInvalidConfiguration;
    }
    const long long n_items = p.vtiles ? (long long)p.n_vtiles * p.H : (long long)p.n_qtiles * p.B * p.H;
    if (n_items > 0x7fffffffLL || n_items < 1) return cudaErrorInvalidValue;
    // persistent: one CTA per SM at most; one item per CTA otherwise
    const long long blocks = C::PERSIST && p.n_sms > 0 && n_items > p.n_sms ? p.n_sms : n_items;
    if (ev_start) cudaEventRecord(ev_start, stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, maps.k, maps.v, maps.q, maps.gate, maps.out, p);
    if (ev_stop) cudaEventRecord(ev_stop, stream);
    return err;
}

}  // namespace

int prefill_block_n(int d) { return d == 256 ? PfCfg<256>::BN : d == 128 ? PfCfg<128>::BN : PfCfg<64>::BN; }

cudaError_t launch_prefill_tc(const PrefillParams& p, const PrefillMaps& maps, cudaStream_t stream,
                              cudaEvent_t ev_start, cudaEvent_t ev_stop) {
    switch (p.d) {
        case 64: return launch_d<64>(p, maps, stream, ev_start, ev_stop);
        case 128: return launch_d<128>(p, maps, stream, ev_start, ev_stop);
        case 256: return launch_d<256>(p, maps, stream, ev_start, ev_stop);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gattn
