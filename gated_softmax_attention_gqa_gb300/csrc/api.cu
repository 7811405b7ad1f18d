// api.cu -- the libgattn C ABI: argument validation, workspace sizing, TMA
// tensor maps and kernel launches.  See include/gattn.h for the contract.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <vector>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

using namespace gattn;

namespace {

__device__ unsigned int g_device_status;

cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Device address of the status word on the current device.
unsigned int* status_ptr() {
    static unsigned int* ptrs[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<unsigned int*>(p);
    }
    return ptrs[dev];
}

int sm_count() {
    static int cached[64] = {};
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

void fill_inv_freq(float* dst, int rd, double base) {
    for (int i = 0; i < kMaxRotaryHalf; ++i)
        dst[i] = (i < rd / 2) ? (float)std::pow(base, -2.0 * (double)i / (double)rd) : 0.f;
}

// Recently encoded tensor maps, so that repeated calls on the same buffers skip
// the host-side encoding.  A map depends only on the arguments below.
struct MapKey {
    const void* base;
    int rank;
    uint64_t dims[5], strides[4];
    uint32_t box[5];
    bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
struct MapCache {
    static constexpr int kEntries = 16;
    MapKey key[kEntries];
    CUtensorMap map[kEntries];
    bool used[kEntries] = {};
    int next = 0;
    std::mutex mu;
};
MapCache g_maps;

bool encode_bf16_map_uncached(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                              const uint64_t* strides_bytes, const uint32_t* box);

// bf16 tensor map with a 64-element (128 B) inner box and 128 B swizzle.
bool encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                     const uint32_t* box) {
    MapKey k;
    std::memset(&k, 0, sizeof(k));
    k.base = base;
    k.rank = rank;
    for (int i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
        if (i + 1 < rank) k.strides[i] = strides_bytes[i];
    }
    std::lock_guard<std::mutex> lock(g_maps.mu);
    for (int i = 0; i < MapCache::kEntries; ++i)
        if (g_maps.used[i] && g_maps.key[i] == k) {
            *map = g_maps.map[i];
            return true;
        }
    if (!encode_bf16_map_uncached(map, base, rank, dims, strides_bytes, box)) return false;
    const int slot = g_maps.next;
    g_maps.next = (slot + 1) % MapCache::kEntries;
    g_maps.key[slot] = k;
    g_maps.map[slot] = *map;
    g_maps.used[slot] = true;
    return true;
}

bool encode_bf16_map_uncached(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                              const uint64_t* strides_bytes, const uint32_t* box) {
    auto fn = get_encode_fn();
    if (!fn) return false;
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
                    reinterpret_cast<const cuuint64_t*>(dims), reinterpret_cast<const cuuint64_t*>(strides_bytes),
                    reinterpret_cast<const cuuint32_t*>(box), elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// layout | activation | additive; no gate means no activation or combine bits either
bool valid_gate_mode(int m) {
    if (m < 0 || (m & ~0x1FF)) return false;
    const int layout = m & 0x0F, act = m & 0xF0;
    if (layout > GATTN_GATE_HEAD_SHARED) return false;
    if (act != GATTN_GATE_ACT_SIGMOID && act != GATTN_GATE_ACT_NS_SIGMOID && act != GATTN_GATE_ACT_SILU) return false;
    return layout != GATTN_GATE_NONE || m == GATTN_GATE_NONE;
}

// The bounded-wait self-test: an mbarrier that nothing arrives on.  Warp 0 waits on
// it through mbar_wait with the caller's short limit, runs out, raises the abort
// flag and the GATTN_DEVICE_TIMEOUT bit; warp 1 waits with the kernels' own 2 s
// limit and must leave on the abort flag alone, as a kernel's other roles do when
// one of them gives up.  Every wait ends; the block exits normally.
__global__ void __launch_bounds__(64) selftest_wait_kernel(unsigned long long limit_ns, unsigned int* status,
                                                           unsigned long long* waited_ns) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_word;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_word = 0;
        fence_mbar_init();
    }
    __syncthreads();
    volatile int* abort_flag = &abort_word;
    const unsigned long long t0 = global_timer_ns();
    if (threadIdx.x < 32) {
        mbar_wait(b, 0, abort_flag, status, limit_ns);
        if (threadIdx.x == 0 && waited_ns) *waited_ns = global_timer_ns() - t0;
    } else {
        mbar_wait(b, 0, abort_flag, status);
    }
    __syncthreads();
}

size_t prefill_ws(int B, int S, int H, int G, int d, int dtype) {
    if (B < 1 || S < 1 || H < 1 || G < 1 || d < 1) return 0;
    const size_t kr = (size_t)B * G * S * d, qr = (size_t)B * H * S * d;
    if (dtype == GATTN_BF16) return round_up(kr * 2, 256);
    if (dtype == GATTN_FP32) return round_up(qr * 4, 256) + round_up(kr * 4, 256);
    return 0;
}

}  // namespace

// Packed sequences: host copy of the cumulative sequence lengths.
struct Varlen {
    const int32_t* cu;  // [nseq + 1]
    int nseq;
};

// At most ceil(T/128) + nseq query tiles (each sequence adds at most one partial tile).
size_t varlen_max_tiles(int T, int nseq) { return (size_t)(T + 127) / 128 + (size_t)nseq; }

// Workspace after the K' (and q') part: the tile table, positions, sequence starts.
size_t varlen_ws(int T, int nseq) {
    return round_up(varlen_max_tiles(T, nseq) * 16, 256) + 2 * round_up((size_t)T * 4, 256);
}

gattn_status prefill_impl(const void* q, const void* k, const void* v, const void* gate, const void* qnorm_w,
                           const void* knorm_w, const int32_t* pos, int B, int S, int H, int G, int d,
                           int rotary_dim, double rope_base, float eps, int gate_mode, int64_t q_tok_stride,
                           int64_t q_head_stride, int64_t gate_tok_stride, int64_t gate_head_stride, int dtype,
                           void* workspace, size_t workspace_bytes, void* out, void* stream_,
                          const Varlen* vl) {
    // ---- arguments
    if (!q || !k || !v || !qnorm_w || !knorm_w || !out) return GATTN_ERR_INVALID_ARG;
    if (!valid_gate_mode(gate_mode) || (gate_layout(gate_mode) != GATTN_GATE_NONE && !gate))
        return GATTN_ERR_INVALID_ARG;
    if (dtype != GATTN_BF16 && dtype != GATTN_FP32) return GATTN_ERR_INVALID_ARG;
    if (B < 1 || S < 1 || H < 1 || G < 1 || d < 1 || H % G != 0) return GATTN_ERR_INVALID_ARG;
    if (rotary_dim < 0 || rotary_dim > d || (rotary_dim & 1)) return GATTN_ERR_INVALID_ARG;
    if (rotary_dim > 0 && !(rope_base > 0.0 && std::isfinite(rope_base))) return GATTN_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return GATTN_ERR_INVALID_ARG;
    if ((int64_t)B * S > INT32_MAX || (int64_t)B * G > INT32_MAX || (int64_t)B * H > INT32_MAX)
        return GATTN_ERR_INVALID_ARG;
    const bool bf = dtype == GATTN_BF16;
    const int elt = bf ? 2 : 4;
    if (bf ? !(d == 64 || d == 128 || d == 256) : !(d == 32 || d == 64 || d == 128 || d == 256))
        return GATTN_ERR_UNSUPPORTED;
    if (bf && rotary_dim % 16 != 0) return GATTN_ERR_UNSUPPORTED;
    if (q_tok_stride == 0) q_tok_stride = (int64_t)H * d;
    if (q_head_stride == 0) q_head_stride = d;
    const int glayout = gate_layout(gate_mode);
    const bool headwise = glayout == GATTN_GATE_HEADWISE, shared = glayout == GATTN_GATE_HEAD_SHARED;
    if (gate_tok_stride == 0) gate_tok_stride = headwise ? H : shared ? d : (int64_t)H * d;
    if (gate_head_stride == 0) gate_head_stride = headwise ? 1 : d;
    if (shared) gate_head_stride = 0;  // one vector of logits for every head
    if (q_tok_stride < 0 || q_head_stride < 0 || gate_tok_stride < 0 || gate_head_stride < 0)
        return GATTN_ERR_INVALID_ARG;
    const int64_t vec = 16 / elt;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return GATTN_ERR_INVALID_ARG;
    if (q_tok_stride % vec || q_head_stride % vec) return GATTN_ERR_INVALID_ARG;
    if (gate_per_dim(gate_mode) && (!aligned(gate, 16) || gate_tok_stride % vec || gate_head_stride % vec))
        return GATTN_ERR_INVALID_ARG;
    if (bf && (!aligned(qnorm_w, 16) || !aligned(knorm_w, 16))) return GATTN_ERR_INVALID_ARG;
    const size_t base_ws = prefill_ws(B, S, H, G, d, dtype);
    const size_t need = base_ws + (vl ? varlen_ws(S, vl->nseq) : 0);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return GATTN_ERR_WORKSPACE;

    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    unsigned int* status = status_ptr();
    if (!status) return GATTN_ERR_CUDA;

    // ---- packed sequences: the query-tile table (heaviest first) into the workspace,
    // then every token's position within its sequence (unless pos is given) and its
    // sequence's first token
    const int4* vtiles = nullptr;
    int n_vtiles = 0;
    int32_t* vstart = nullptr;
    if (vl) {
        std::vector<int4> tiles;
        for (int i = 0; i < vl->nseq; ++i) {
            const int len = vl->cu[i + 1] - vl->cu[i];
            for (int qt = 0; qt * 128 < len; ++qt) tiles.push_back(make_int4(vl->cu[i], len, qt, i));
        }
        std::stable_sort(tiles.begin(), tiles.end(), [](const int4& x, const int4& y) { return x.z > y.z; });
        char* extra = static_cast<char*>(workspace) + base_ws;
        int4* dtiles = reinterpret_cast<int4*>(extra);
        int32_t* vpos = reinterpret_cast<int32_t*>(extra + round_up(varlen_max_tiles(S, vl->nseq) * 16, 256));
        vstart = vpos + round_up((size_t)S * 4, 256) / 4;
        n_vtiles = (int)tiles.size();
        if (n_vtiles > 0 &&
            cudaMemcpyAsync(dtiles, tiles.data(), tiles.size() * sizeof(int4), cudaMemcpyHostToDevice, stream) !=
                cudaSuccess)
            return GATTN_ERR_CUDA;
        if (launch_varlen_positions(dtiles, n_vtiles, vpos, vstart, stream) != cudaSuccess) return GATTN_ERR_CUDA;
        vtiles = dtiles;
        if (!pos) pos = vpos;
    }

    // ---- K' = rope(rmsnorm(k)) into the workspace, [B,G,S,d]
    ProloguePlan kp;
    std::memset(&kp, 0, sizeof(kp));
    kp.x = k;
    kp.tok_stride = (int64_t)G * d;
    kp.head_stride = d;
    kp.w = knorm_w;
    kp.pos = pos;
    kp.B = B;
    kp.S = S;
    kp.n_heads = G;
    kp.d = d;
    kp.rd = rotary_dim;
    kp.eps = eps;
    kp.status = status;
    fill_inv_freq(kp.inv_freq, rotary_dim, rope_base);

    if (bf) {
        kp.dst = workspace;
        if (launch_prologue(kp, true, true, stream) != cudaSuccess) return GATTN_ERR_CUDA;
        PrefillMaps maps;
        // two heads of a KV group per CTA pair when H/G is even, else one head per CTA
        const bool pair = prefill_pair_supported(d, H, G);
        const uint32_t kbn = pair ? (uint32_t)prefill_pair_key_rows() : (uint32_t)prefill_block_n(d);
        const uint32_t vbn = pair ? (uint32_t)prefill_pair_value_rows() : (uint32_t)prefill_block_n(d);
        const uint64_t kdims[3] = {(uint64_t)d, (uint64_t)S, (uint64_t)B * G};
        const uint64_t kstr[2] = {(uint64_t)d * 2, (uint64_t)S * d * 2};
        const uint32_t kbox[3] = {64, kbn, 1};
        const uint64_t vdims[4] = {(uint64_t)d, (uint64_t)G, (uint64_t)S, (uint64_t)B};
        const uint64_t vstr[3] = {(uint64_t)d * 2, (uint64_t)G * d * 2, (uint64_t)S * G * d * 2};
        const uint32_t vbox[4] = {64, 1, vbn, 1};
        // raw q and gate: [B,S,H,d] views with token/head strides; 128-token boxes
        const uint64_t hdims[4] = {(uint64_t)d, (uint64_t)H, (uint64_t)S, (uint64_t)B};
        const uint64_t qstr[3] = {(uint64_t)q_head_stride * 2, (uint64_t)q_tok_stride * 2,
                                  (uint64_t)S * q_tok_stride * 2};
        const uint32_t rbox[4] = {64, 1, 128, 1};
        if (!encode_bf16_map(&maps.k, workspace, 3, kdims, kstr, kbox)) return GATTN_ERR_CUDA;
        if (!encode_bf16_map(&maps.v, v, 4, vdims, vstr, vbox)) return GATTN_ERR_CUDA;
        if (!encode_bf16_map(&maps.q, q, 4, hdims, qstr, rbox)) return GATTN_ERR_CUDA;
        if (gate_per_dim(gate_mode)) {
            // (d, H, S, B); a head-shared gate has a single head (its stride is unused)
            const uint64_t gdims[4] = {(uint64_t)d, shared ? 1u : (uint64_t)H, (uint64_t)S, (uint64_t)B};
            const uint64_t gstr[3] = {(uint64_t)(shared ? gate_tok_stride : gate_head_stride) * 2,
                                      (uint64_t)gate_tok_stride * 2, (uint64_t)S * gate_tok_stride * 2};
            if (!encode_bf16_map(&maps.gate, gate, 4, gdims, gstr, rbox)) return GATTN_ERR_CUDA;
        } else {
            maps.gate = maps.q;  // never read
        }
        // out [B,S,H*d] seen as (d, H, S, B)
        const uint64_t ostr[3] = {(uint64_t)d * 2, (uint64_t)H * d * 2, (uint64_t)S * H * d * 2};
        if (!encode_bf16_map(&maps.out, out, 4, hdims, ostr, rbox)) return GATTN_ERR_CUDA;
        PrefillParams pp;
        std::memset(&pp, 0, sizeof(pp));
        pp.q = q;
        pp.gate = gate;
        pp.qnorm_w = qnorm_w;
        pp.knorm_w = knorm_w;
        pp.pos = pos;
        pp.out = out;
        pp.q_tok_stride = q_tok_stride;
        pp.q_head_stride = q_head_stride;
        pp.gate_tok_stride = gate_tok_stride;
        pp.gate_head_stride = gate_head_stride;
        pp.B = B;
        pp.S = S;
        pp.H = H;
        pp.G = G;
        pp.d = d;
        pp.rd = rotary_dim;
        pp.gate_mode = gate_mode;
        pp.n_qtiles = (S + 127) / 128;
        pp.n_sms = sm_count();
        pp.eps = eps;
        pp.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
        pp.status = status;
        pp.vtiles = vtiles;
        pp.n_vtiles = n_vtiles;
        std::memcpy(pp.inv_freq, kp.inv_freq, sizeof(pp.inv_freq));
        const cudaError_t le = pair ? launch_prefill_pair(pp, maps, stream, g_prof_start, g_prof_stop)
                                    : launch_prefill_tc(pp, maps, stream, g_prof_start, g_prof_stop);
        if (le != cudaSuccess) return GATTN_ERR_CUDA;
        return GATTN_OK;
    }

    // ---- fp32: q' and k' into the workspace, then the CUDA-core kernel
    float* qr = static_cast<float*>(workspace);
    float* kr = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up((size_t)B * H * S * d * 4, 256));
    kp.dst = kr;
    if (launch_prologue(kp, false, false, stream) != cudaSuccess) return GATTN_ERR_CUDA;
    ProloguePlan qp = kp;
    qp.x = q;
    qp.tok_stride = q_tok_stride;
    qp.head_stride = q_head_stride;
    qp.w = qnorm_w;
    qp.n_heads = H;
    qp.dst = qr;
    if (launch_prologue(qp, false, false, stream) != cudaSuccess) return GATTN_ERR_CUDA;
    PrefillF32Params fp;
    std::memset(&fp, 0, sizeof(fp));
    fp.qr = qr;
    fp.kr = kr;
    fp.v = static_cast<const float*>(v);
    fp.gate = static_cast<const float*>(gate);
    fp.out = static_cast<float*>(out);
    fp.gate_tok_stride = gate_tok_stride;
    fp.gate_head_stride = gate_head_stride;
    fp.B = B;
    fp.S = S;
    fp.H = H;
    fp.G = G;
    fp.d = d;
    fp.gate_mode = gate_mode;
    fp.scale = (float)(1.0 / std::sqrt((double)d));
    fp.tok_start = vstart;
    if (launch_prefill_f32(fp, stream, g_prof_start, g_prof_stop) != cudaSuccess) return GATTN_ERR_CUDA;
    return GATTN_OK;
}


extern "C" {

const char* gattn_strerror(gattn_status s) {
    switch (s) {
        case GATTN_OK: return "GATTN_OK";
        case GATTN_ERR_INVALID_ARG: return "GATTN_ERR_INVALID_ARG: invalid argument";
        case GATTN_ERR_UNSUPPORTED: return "GATTN_ERR_UNSUPPORTED: no kernel for this configuration";
        case GATTN_ERR_CUDA: return "GATTN_ERR_CUDA: a CUDA call or kernel launch failed";
        case GATTN_ERR_WORKSPACE: return "GATTN_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case GATTN_ERR_DEVICE: return "GATTN_ERR_DEVICE: a kernel reported a device-side problem";
        case GATTN_ERR_DEVICE_TIMEOUT: return "GATTN_ERR_DEVICE_TIMEOUT: a bounded wait inside a kernel ran out";
    }
    return "unknown gattn_status";
}

void gattn_set_profile_events(void* start, void* stop) {
    g_prof_start = static_cast<cudaEvent_t>(start);
    g_prof_stop = static_cast<cudaEvent_t>(stop);
}

size_t gattn_prefill_workspace_size(int B, int S, int H, int G, int d, int dtype) {
    return prefill_ws(B, S, H, G, d, dtype);
}

gattn_status gattn_prefill(const void* q, const void* k, const void* v, const void* gate, const void* qnorm_w,
                           const void* knorm_w, const int32_t* pos, int B, int S, int H, int G, int d,
                           int rotary_dim, double rope_base, float eps, int gate_mode, int64_t q_tok_stride,
                           int64_t q_head_stride, int64_t gate_tok_stride, int64_t gate_head_stride, int dtype,
                           void* workspace, size_t workspace_bytes, void* out, void* stream) {
    return prefill_impl(q, k, v, gate, qnorm_w, knorm_w, pos, B, S, H, G, d, rotary_dim, rope_base, eps, gate_mode,
                        q_tok_stride, q_head_stride, gate_tok_stride, gate_head_stride, dtype, workspace,
                        workspace_bytes, out, stream, nullptr);
}

gattn_status gattn_o_proj(const void* x, const void* w_o, int T, int K, int N, void* y, void* stream_) {
    if (!x || !w_o || !y) return GATTN_ERR_INVALID_ARG;
    if (T < 1 || K < 64 || N < 64 || K % 64 != 0 || N % 64 != 0) return GATTN_ERR_INVALID_ARG;
    if ((int64_t)T * K >= ((int64_t)1 << 40) || (int64_t)T * N >= ((int64_t)1 << 40)) return GATTN_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w_o, 16) || !aligned(y, 16)) return GATTN_ERR_INVALID_ARG;
    unsigned int* status = status_ptr();
    if (!status) return GATTN_ERR_CUDA;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    // x [T, K] and W_O [N, K] as (K, rows): 64-element (128-byte) slices, 128 rows of x
    // and oproj_box_rows(N) rows of W_O per box
    CUtensorMap ta, tb;
    const uint64_t adims[2] = {(uint64_t)K, (uint64_t)T}, bdims[2] = {(uint64_t)K, (uint64_t)N};
    const uint64_t str[1] = {(uint64_t)K * 2};
    const uint32_t abox[2] = {64, 128}, bbox[2] = {64, (uint32_t)oproj_box_rows(N)};
    if (!encode_bf16_map(&ta, x, 2, adims, str, abox)) return GATTN_ERR_CUDA;
    if (!encode_bf16_map(&tb, w_o, 2, bdims, str, bbox)) return GATTN_ERR_CUDA;
    OprojParams op;
    std::memset(&op, 0, sizeof(op));
    op.y = y;
    op.T = T;
    op.K = K;
    op.N = N;
    op.n_sms = sm_count();
    op.status = status;
    if (launch_oproj(op, ta, tb, stream, g_prof_start, g_prof_stop) != cudaSuccess) return GATTN_ERR_CUDA;
    return GATTN_OK;
}

size_t gattn_prefill_varlen_workspace_size(int T, int nseq, int H, int G, int d, int dtype) {
    if (T < 1 || nseq < 1) return 0;
    const size_t base = prefill_ws(1, T, H, G, d, dtype);
    return base ? base + varlen_ws(T, nseq) : 0;
}

gattn_status gattn_prefill_varlen(const void* q, const void* k, const void* v, const void* gate, const void* qnorm_w,
                                  const void* knorm_w, const int32_t* pos, const int32_t* cu_seqlens, int nseq, int H,
                                  int G, int d, int rotary_dim, double rope_base, float eps, int gate_mode,
                                  int64_t q_tok_stride, int64_t q_head_stride, int64_t gate_tok_stride,
                                  int64_t gate_head_stride, int dtype, void* workspace, size_t workspace_bytes,
                                  void* out, void* stream) {
    if (!cu_seqlens || nseq < 1 || cu_seqlens[0] != 0) return GATTN_ERR_INVALID_ARG;
    for (int i = 0; i < nseq; ++i)
        if (cu_seqlens[i + 1] < cu_seqlens[i]) return GATTN_ERR_INVALID_ARG;
    const int T = cu_seqlens[nseq];
    if (T < 1) return GATTN_OK;  // nothing to compute
    const Varlen vl{cu_seqlens, nseq};
    return prefill_impl(q, k, v, gate, qnorm_w, knorm_w, pos, 1, T, H, G, d, rotary_dim, rope_base, eps, gate_mode,
                        q_tok_stride, q_head_stride, gate_tok_stride, gate_head_stride, dtype, workspace,
                        workspace_bytes, out, stream, &vl);
}

size_t gattn_decode_workspace_size(int B, int H, int G, int d, int Lmax) {
    if (B < 1 || H < 1 || G < 1 || d < 1 || Lmax < 1 || H % G != 0) return 0;
    const int n = sm_count();
    if (n <= 0) return 0;
    return round_up((size_t)decode_num_slots(n, B, G) * decode_slot_floats(H / G, d) * sizeof(float), 256);
}

}  // extern "C"

namespace {

// A paged cache: [2, num_pages, G, page_size, d] and the [B, max_pages] block table.
struct PagedCache {
    const int32_t* block_table;
    int num_pages, page_size, max_pages;
};

// The decode step; with append != NULL the new token's K and V are first written
// into the cache (k_new, v_new, knorm_w of *append); with paged != NULL the cache
// is paged (Lmax = max_pages * page_size).
}  // namespace

// Every host-side check of a decode step's arguments except the workspace (shared
// by gattn_decode and its variants, so that they report the same status).
gattn_status gattn::decode_check_args(const void* q_new, const void* kv_cache, const int32_t* seqlens,
                                      const void* gate, const void* qnorm_w, int B, int H, int G, int d, int Lmax,
                                      int rotary_dim, double rope_base, float eps, int gate_mode, const void* out,
                                      int64_t cache_rows) {
    if (!q_new || !kv_cache || !seqlens || !qnorm_w || !out) return GATTN_ERR_INVALID_ARG;
    if (!valid_gate_mode(gate_mode) || (gate_layout(gate_mode) != GATTN_GATE_NONE && !gate))
        return GATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || G < 1 || d < 1 || Lmax < 1 || H % G != 0) return GATTN_ERR_INVALID_ARG;
    if (rotary_dim < 0 || rotary_dim > d || (rotary_dim & 1)) return GATTN_ERR_INVALID_ARG;
    if (rotary_dim > 0 && !(rope_base > 0.0 && std::isfinite(rope_base))) return GATTN_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return GATTN_ERR_INVALID_ARG;
    if (!(d == 64 || d == 128 || d == 256) || H / G > 8 || rotary_dim % 16 != 0 || B > decode_max_batch())
        return GATTN_ERR_UNSUPPORTED;
    if (cache_rows < 0) cache_rows = 2 * (int64_t)B * G * Lmax;
    if (cache_rows + kDecodeTileKeys > INT32_MAX) return GATTN_ERR_UNSUPPORTED;
    if (!aligned(kv_cache, 16) || !aligned(q_new, 4) || !aligned(qnorm_w, 4) || !aligned(out, 2))
        return GATTN_ERR_INVALID_ARG;
    return GATTN_OK;
}

namespace {

gattn_status decode_impl(const void* q_new, const void* kv_cache, const int32_t* seqlens, const void* gate,
                         const void* qnorm_w, int B, int H, int G, int d, int Lmax, int rotary_dim, double rope_base,
                         float eps, int gate_mode, void* workspace, size_t workspace_bytes, void* out, void* stream_,
                         const AppendParams* append, const PagedCache* paged) {
    const int64_t cache_rows = paged ? 2 * (int64_t)paged->num_pages * G * paged->page_size : 2 * (int64_t)B * G * Lmax;
    const gattn_status arg = decode_check_args(q_new, kv_cache, seqlens, gate, qnorm_w, B, H, G, d, Lmax, rotary_dim,
                                               rope_base, eps, gate_mode, out, cache_rows);
    if (arg != GATTN_OK) return arg;
    const int n_ctas = sm_count();
    if (n_ctas <= 0) return GATTN_ERR_CUDA;
    const size_t need = gattn_decode_workspace_size(B, H, G, d, Lmax);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return GATTN_ERR_WORKSPACE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    unsigned int* status = status_ptr();
    if (!status) return GATTN_ERR_CUDA;

    CUtensorMap tm;
    const uint64_t dims[2] = {(uint64_t)d, (uint64_t)cache_rows};
    const uint64_t str[1] = {(uint64_t)d * 2};
    const uint32_t box[2] = {64, (uint32_t)kDecodeTileKeys};
    if (!encode_bf16_map(&tm, kv_cache, 2, dims, str, box)) return GATTN_ERR_CUDA;

    DecodeParams dp;
    std::memset(&dp, 0, sizeof(dp));
    dp.q = q_new;
    dp.seqlens = seqlens;
    dp.gate = gate;
    dp.qnorm_w = qnorm_w;
    dp.out = out;
    dp.part = static_cast<float*>(workspace);
    dp.B = B;
    dp.H = H;
    dp.G = G;
    dp.d = d;
    dp.Lmax = Lmax;
    dp.rd = rotary_dim;
    dp.gate_mode = gate_mode;
    dp.n_ctas = n_ctas;
    dp.eps = eps;
    dp.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
    dp.status = status;
    fill_inv_freq(dp.inv_freq, rotary_dim, rope_base);
    if (paged) {
        dp.block_table = paged->block_table;
        dp.num_pages = paged->num_pages;
        dp.page_size = paged->page_size;
        dp.max_pages = paged->max_pages;
    }
    if (append) {
        AppendParams ap = *append;
        ap.cache = const_cast<void*>(kv_cache);
        ap.seqlens = seqlens;
        ap.B = B;
        ap.G = G;
        ap.d = d;
        ap.Lmax = Lmax;
        ap.rd = rotary_dim;
        ap.eps = eps;
        ap.status = status;
        ap.block_table = dp.block_table;
        ap.num_pages = dp.num_pages;
        ap.page_size = dp.page_size;
        ap.max_pages = dp.max_pages;
        std::memcpy(ap.inv_freq, dp.inv_freq, sizeof(ap.inv_freq));
        if (launch_decode_append(ap, stream) != cudaSuccess) return GATTN_ERR_CUDA;
    }
    if (launch_decode(dp, tm, stream, g_prof_start, g_prof_stop) != cudaSuccess) return GATTN_ERR_CUDA;
    return GATTN_OK;
}

}  // namespace

extern "C" {

gattn_status gattn_decode(const void* q_new, const void* kv_cache, const int32_t* seqlens, const void* gate,
                          const void* qnorm_w, int B, int H, int G, int d, int Lmax, int rotary_dim,
                          double rope_base, float eps, int gate_mode, void* workspace, size_t workspace_bytes,
                          void* out, void* stream_) {
    return decode_impl(q_new, kv_cache, seqlens, gate, qnorm_w, B, H, G, d, Lmax, rotary_dim, rope_base, eps,
                       gate_mode, workspace, workspace_bytes, out, stream_, nullptr, nullptr);
}

gattn_status gattn_decode_append(const void* q_new, const void* k_new, const void* v_new, void* kv_cache,
                                 const int32_t* seqlens, const void* gate, const void* qnorm_w, const void* knorm_w,
                                 int B, int H, int G, int d, int Lmax, int rotary_dim, double rope_base, float eps,
                                 int gate_mode, void* workspace, size_t workspace_bytes, void* out, void* stream) {
    if (!k_new || !v_new || !knorm_w) return GATTN_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(knorm_w, 16)) return GATTN_ERR_INVALID_ARG;
    AppendParams ap;
    std::memset(&ap, 0, sizeof(ap));
    ap.k_new = k_new;
    ap.v_new = v_new;
    ap.knorm_w = knorm_w;
    return decode_impl(q_new, kv_cache, seqlens, gate, qnorm_w, B, H, G, d, Lmax, rotary_dim, rope_base, eps,
                       gate_mode, workspace, workspace_bytes, out, stream, &ap, nullptr);
}

gattn_status gattn_decode_paged(const void* q_new, const void* k_new, const void* v_new, void* kv_pages,
                                const int32_t* block_table, int num_pages, int page_size, int max_pages,
                                const int32_t* seqlens, const void* gate, const void* qnorm_w, const void* knorm_w,
                                int B, int H, int G, int d, int rotary_dim, double rope_base, float eps, int gate_mode,
                                void* workspace, size_t workspace_bytes, void* out, void* stream) {
    if (!block_table || num_pages < 1 || max_pages < 1 || page_size < 1) return GATTN_ERR_INVALID_ARG;
    if (page_size % kDecodeTileKeys != 0) return GATTN_ERR_UNSUPPORTED;  // a key tile never straddles two pages
    if ((int64_t)max_pages * page_size > INT32_MAX) return GATTN_ERR_INVALID_ARG;
    PagedCache pc{block_table, num_pages, page_size, max_pages};
    AppendParams ap;
    std::memset(&ap, 0, sizeof(ap));
    if (k_new || v_new) {
        if (!k_new || !v_new || !knorm_w) return GATTN_ERR_INVALID_ARG;
        if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(knorm_w, 16)) return GATTN_ERR_INVALID_ARG;
        ap.k_new = k_new;
        ap.v_new = v_new;
        ap.knorm_w = knorm_w;
    }
    return decode_impl(q_new, kv_pages, seqlens, gate, qnorm_w, B, H, G, d, max_pages * page_size, rotary_dim,
                       rope_base, eps, gate_mode, workspace, workspace_bytes, out, stream, k_new ? &ap : nullptr, &pc);
}



gattn_status gattn_get_device_status(unsigned int* bits, void* stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    unsigned int* status = status_ptr();
    if (!status) return GATTN_ERR_CUDA;
    unsigned int h = 0;
    if (cudaMemcpyAsync(&h, status, sizeof(h), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return GATTN_ERR_CUDA;
    if (cudaMemsetAsync(status, 0, sizeof(h), stream) != cudaSuccess) return GATTN_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GATTN_ERR_CUDA;
    if (bits) *bits = h;
    return (h & GATTN_DEVICE_TIMEOUT) ? GATTN_ERR_DEVICE_TIMEOUT : h ? GATTN_ERR_DEVICE : GATTN_OK;
}

gattn_status gattn_selftest_wait_timeout(unsigned long long limit_ns, unsigned long long* waited_ns, void* stream_) {
    if (limit_ns < 1000000ull || limit_ns > 100000000ull) return GATTN_ERR_INVALID_ARG;
    unsigned int* status = status_ptr();
    if (!status) return GATTN_ERR_CUDA;
    selftest_wait_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream_)>>>(limit_ns, status, waited_ns);
    return cudaGetLastError() == cudaSuccess ? GATTN_OK : GATTN_ERR_CUDA;
}

}  // extern "C"
