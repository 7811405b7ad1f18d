// decode_noalloc.cu -- gattn_decode_noalloc: one decode step with no caller
// workspace and no device allocation.
//
// gattn_decode needs a workspace for the partial softmax states of its
// split-KV pass, and the usual way to get one is cudaMalloc (directly or through
// a caching allocator).  Some callers cannot do that at the point where they run
// a decode step: serving loops that must never call cudaMalloc while requests are
// in flight (it can synchronise the device and stall every other stream), and
// host frameworks that hand a plugin its input and output buffers but forbid it
// to allocate device memory of its own.  For them this entry point keeps the
// partial states in a fixed array of device memory that the library defines at
// file scope, sized kScratchBytes.  Every GPU that loads the library holds that
// array until the process exits.
//
// The array's name, used from host code, is only a host-side stand-in for the
// device symbol; its device address is fetched once per device with
// cudaGetSymbolAddress (with that device current) and handed to the kernels as
// an ordinary workspace pointer.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB, see GATTN_DECODE_NOALLOC_SCRATCH_BYTES

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Device address of g_decode_scratch on the current device, looked up on the
// first call made with that device current.
void* scratch_address() {
    static void* addr[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

extern "C" gattn_status gattn_decode_noalloc(const void* q_new, const void* kv_cache, const int32_t* seqlens,
                                             const void* gate, const void* qnorm_w, int B, int H, int G, int d,
                                             int Lmax, int rotary_dim, double rope_base, float eps, int gate_mode,
                                             void* out, void* stream) {
    static_assert(GATTN_DECODE_NOALLOC_SCRATCH_BYTES == kScratchBytes, "header and library disagree on the limit");
    // Argument errors first, with the status gattn_decode gives them; only then the
    // scratch limit and the one-time address lookup.
    const gattn_status arg = gattn::decode_check_args(q_new, kv_cache, seqlens, gate, qnorm_w, B, H, G, d, Lmax,
                                                      rotary_dim, rope_base, eps, gate_mode, out, -1);
    if (arg != GATTN_OK) return arg;
    const size_t need = gattn_decode_workspace_size(B, H, G, d, Lmax);
    if (need > kScratchBytes) return GATTN_ERR_WORKSPACE;
    void* scratch = scratch_address();
    if (!scratch) return GATTN_ERR_CUDA;
    // The partial states need no clearing: every slot the combine pass reads is
    // written earlier in the same call by the split pass.
    return gattn_decode(q_new, kv_cache, seqlens, gate, qnorm_w, B, H, G, d, Lmax, rotary_dim, rope_base, eps,
                        gate_mode, scratch, kScratchBytes, out, stream);
}
