// common.cuh -- device helpers shared by the libgattn kernels (sm_103a).
//
// Thin wrappers over PTX for mbarriers, TMA bulk-tensor copies, tcgen05 (5th
// generation tensor cores with TMEM accumulators) and warp-level mma, plus the
// bounded-wait discipline every spin in this library follows: a wait gives up
// after a wall-clock limit, raises the CTA's abort flag and a device status
// bit, and the caller unwinds instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gattn.h"

namespace gattn {

typedef __nv_bfloat16 bf16;

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s wall clock per wait

// ------------------------------------------------------------------ misc

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A fixed reference for the softmax exponent, in place of the running row maximum.
// q' and k' are RMS-normalised (|x / rms(x)|_2 <= sqrt(d)), scaled by the norm
// weights and rotated (which keeps the norm), so |q'|_2 <= sqrt(d) max|w_q|, the
// same for k', and every logit obeys |q'.k'| scale_log2 <= d max|w_q| max|w_k|
// scale_log2 = bound (with a 2^-6 margin for the bf16 rounding of q' and k' and for
// the fp32 sums).  Softmax is unchanged by the constant subtracted from the
// logits; with the bound every exponent is <= 0, so no running maximum, no
// exchange of it and no rescale of O are needed.  Used only while bound <=
// kFixedRefLimit: the largest P of a row is then >= 2^(-2 bound), so P, l and O
// stay far from fp32 underflow.  Returns +INF (use the running maximum) otherwise.
// All 32 lanes of the warp call it.
constexpr float kFixedRefLimit = 40.f;
__device__ __forceinline__ float fixed_logit_ref(const __nv_bfloat16* wq, const __nv_bfloat16* wk, int d,
                                                 float scale_log2) {
    float mq = 0.f, mk = 0.f;
    for (int i = (int)(threadIdx.x & 31u); i < d; i += 32) {
        mq = fmaxf(mq, fabsf(__bfloat162float(wq[i])));
        mk = fmaxf(mk, fabsf(__bfloat162float(wk[i])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
        mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
    }
    const float b = (float)d * mq * mk * fabsf(scale_log2) * (1.f + 1.f / 64.f);
    return b <= kFixedRefLimit ? b : INFINITY;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Paired fp32 arithmetic (sm_100 and later): one instruction works on two fp32
// lanes held in a 64-bit register pair, each lane rounded exactly as the scalar
// instruction rounds it.  The softmax issues half as many FMA / add instructions.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// max of three fp32 values in one instruction (sm_100 and later)
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// sigmoid(z) = 1 / (1 + 2^(-z log2 e)) with the hardware exp2 and reciprocal
// approximations (relative error a few ulp; z -> -inf gives 0, z -> +inf gives 1).
__device__ __forceinline__ float sigmoidf_dev(float z) {
    return rcp_approx(1.0f + ex2_approx(-1.4426950408889634f * z));
}

// sigmoid(z) = (1 + tanh(z/2)) / 2 with the hardware tanh: one multi-function
// unit operation instead of two (exact at z = 0; absolute error ~3e-4, far below
// a bf16 step of the gated output), for epilogues that gate every element.
__device__ __forceinline__ float sigmoid_tanh(float z) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return fmaf(0.5f, t, 0.5f);
}

// Gate variants (gattn_gate_mode bit fields).  gate_plain: the default
// multiplicative sigmoid gate, for which the epilogues keep their fast path.
__host__ __device__ __forceinline__ int gate_layout(int mode) { return mode & 0x0F; }
__host__ __device__ __forceinline__ bool gate_additive(int mode) { return (mode & 0x100) != 0; }
__host__ __device__ __forceinline__ bool gate_plain(int mode) { return (mode & 0x1F0) == 0; }
// Logits held per (token, head, dimension) -- elementwise, or head-shared [.., d].
__host__ __device__ __forceinline__ bool gate_per_dim(int mode) {
    return gate_layout(mode) == 1 || gate_layout(mode) == 3;
}

// The gate activation of logit z given s = sigmoid(z): sigmoid, NS-sigmoid
// 0.5 + 0.5 sigmoid(z), or SiLU z sigmoid(z).
__device__ __forceinline__ float gate_act(float z, float s, int mode) {
    const int act = mode & 0xF0;
    return act == 0x10 ? fmaf(0.5f, s, 0.5f) : act == 0x20 ? z * s : s;
}

// sin and cos of a RoPE angle.  Cody-Waite reduction by 2*pi (the constant split
// into a float head and a float tail, k = round(x / 2pi)) brings x into
// [-pi, pi], where the hardware sine/cosine approximations are accurate to about
// 2^-21 absolute; the reduction adds ~1e-7 rad for |x| up to 1e5.  Angles here
// are pos * inv_freq with pos < 2^24, whose own fp32 rounding (ulp(x)/2) is the
// larger error.
__device__ __forceinline__ void rope_sincos(float x, float* s, float* c) {
    constexpr float kInv2Pi = 0.15915494309189535f;
    constexpr float k2PiHi = 6.28318548202514648f;      // 2*pi rounded to float
    constexpr float k2PiLo = -1.7484556000744487e-07f;  // 2*pi - k2PiHi
    const float k = rintf(x * kInv2Pi);
    float r = fmaf(-k, k2PiHi, x);
    r = fmaf(-k, k2PiLo, r);
    *s = __sinf(r);
    *c = __cosf(r);
}

// rope_sincos of two angles, the reduction in paired fp32 arithmetic: the same
// values as two rope_sincos calls (each lane is rounded as the scalar instruction).
__device__ __forceinline__ void rope_sincos2(float2 x, float2* s, float2* c) {
    constexpr float kInv2Pi = 0.15915494309189535f;
    constexpr float k2PiHi = 6.28318548202514648f;
    constexpr float k2PiLo = -1.7484556000744487e-07f;
    const float2 kx = mul2(x, make_float2(kInv2Pi, kInv2Pi));
    const float2 nk = make_float2(-rintf(kx.x), -rintf(kx.y));
    float2 r = fma2(nk, make_float2(k2PiHi, k2PiHi), x);
    r = fma2(nk, make_float2(k2PiLo, k2PiLo), r);
    *s = make_float2(__sinf(r.x), __sinf(r.y));
    *c = make_float2(__cosf(r.x), __cosf(r.y));
}

// One rotated pair of chunks of a RoPE row (x_i and x_{i+rd/2}, 8 values each,
// with their norm weights) scaled by rinv: lo = (a cos - b sin), hi = (b cos +
// a sin) with a = x_i w_i rinv, b = x_{i+rd/2} w_{i+rd/2} rinv, as bf16 pairs.
__device__ __forceinline__ void rope_rotate8(const float (&xa)[8], const float (&xb)[8], const float (&wa)[8],
                                             const float (&wb)[8], const float* inv_freq, float posf, float rinv,
                                             uint32_t (&lo)[4], uint32_t (&hi)[4]) {
    const float2 r2 = make_float2(rinv, rinv), p2 = make_float2(posf, posf);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        float2 sn, cs;
        rope_sincos2(mul2(p2, make_float2(inv_freq[e], inv_freq[e + 1])), &sn, &cs);
        const float2 a = mul2(make_float2(xa[e], xa[e + 1]), mul2(make_float2(wa[e], wa[e + 1]), r2));
        const float2 b = mul2(make_float2(xb[e], xb[e + 1]), mul2(make_float2(wb[e], wb[e + 1]), r2));
        const float2 bs = mul2(b, sn), as = mul2(a, sn);
        const float2 l = fma2(a, cs, make_float2(-bs.x, -bs.y));
        const float2 h = fma2(b, cs, as);
        lo[e >> 1] = pack_bf16x2(l.x, l.y);
        hi[e >> 1] = pack_bf16x2(h.x, h.y);
    }
}

// Eight values x w rinv (x times its norm weight, then rinv) as four bf16 pairs.
__device__ __forceinline__ void scale8_bf16(const float (&x)[8], const float (&w)[8], float rinv, uint32_t (&o)[4]) {
    const float2 r2 = make_float2(rinv, rinv);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const float2 v = mul2(mul2(make_float2(x[e], x[e + 1]), make_float2(w[e], w[e + 1])), r2);
        o[e >> 1] = pack_bf16x2(v.x, v.y);
    }
}

// Raise a kernel's dynamic shared-memory limit once per device (host side).
// `func` identifies the kernel; up to 16 kernels per device are remembered
// (beyond that the attribute is simply set again on every call).
inline cudaError_t set_smem_once(const void* func, int bytes) {
    static const void* seen[64][16] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64)
        for (int i = 0; i < 16; ++i)
            if (seen[dev][i] == func) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess || dev < 0 || dev >= 64) return e;
    for (int i = 0; i < 16; ++i)
        if (!seen[dev][i]) {
            seen[dev][i] = func;
            break;
        }
    return cudaSuccess;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of a phase (mbarrier.test_wait).  try_wait may suspend the
// thread for a while when the phase is not complete yet, which a thread that polls
// several barriers in turn (or looks ahead between MMA groups) cannot afford.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up when another
// thread of the CTA raised *abort, or after limit_ns of wall-clock time (2 s in
// every attention kernel; the wait self-test passes a short limit); on a timeout
// it raises *abort and the device status bit.  Returns true iff the phase completed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          unsigned int* status, unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort = 1;
                atomicOr(status, GATTN_DEVICE_TIMEOUT);
                return false;
            }
        }
    }
}

// Teardown wait: ignores the abort flag (used to drain copies already in
// flight before a CTA exits), still bounded by the wall-clock limit.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, unsigned int* status,
                                                unsigned long long limit_ns = kWaitLimitNs) {
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, GATTN_DEVICE_TIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------------------------ clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster (used only at start-up and teardown,
// where all threads are known to arrive).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier of another CTA of the cluster (release, cluster scope:
// orders this thread's earlier memory writes for the other CTA; ~300 cycles).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster at CTA scope (a few cycles).
// Enough when what the arrival announces has already completed -- a TMA copy
// whose barrier was observed, a tcgen05.st waited on with tcgen05.wait::st, a
// tcgen05.ld already in registers -- rather than being ordered by the arrival.
__device__ __forceinline__ void mbar_arrive_remote_cta(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// mbar_wait for barriers that threads of the other CTA arrive on: acquire at
// cluster scope; same bounds and abort behaviour as mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  unsigned int* status) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicOr(status, GATTN_DEVICE_TIMEOUT);
                return false;
            }
        }
    }
}

// Programmatic dependent launch: let the next kernel on the stream start its
// independent prologue early / wait until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prerequisites() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
        "%5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
        "%5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// 4-D tile store shared -> global (same box geometry and swizzle as the map's
// loads); completion is tracked per thread with bulk groups.  Rows outside the
// tensor are not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// This thread's bulk stores have finished reading shared memory (it may be reused).
__device__ __forceinline__ void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// This thread's bulk stores are complete (written to global memory).
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Pull a 4-D tile into L2 ahead of its use (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's generic-proxy global-memory writes before later async-proxy
// (TMA) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier of nthreads threads that also ANDs a predicate over them: every
// participant gets true only if all of them passed true.  Threads that must give up
// (a bounded wait ran out) still arrive, with false, so that all of them leave
// together and none is left waiting at the barrier.
__device__ __forceinline__ bool named_barrier_and(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// The same for a CTA pair (cta_group::2): one warp of EACH CTA of the pair issues
// the allocation; both receive the same column address.  A kernel uses one
// cta_group throughout.
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish2() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar));
}

// Completion of this thread's earlier pair MMAs, signalled on the mbarrier at
// offset `bar` of every CTA in `cta_mask`.
__device__ __forceinline__ void tc_commit2(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(cta_mask));
}

// Pair MMA (M = 256): rows 0..127 of A and D live in the even CTA, rows 128..255
// in the odd one; each CTA holds N/2 rows (K-major) or columns (MN-major) of B
// at the same shared-memory offset.  Issued by one thread of the even CTA.
__device__ __forceinline__ void mma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma2_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// D(tmem) (+)= A(tmem) * B(smem), kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// D(tmem) (+)= A(smem) * B(smem), kind::f16.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// The same two MMAs with every shared-memory descriptor given as its low word plus a
// compile-time offset (16-byte units) and a common high word, the additions done
// inside the asm.  An unrolled stream of these leaves the compiler nothing to hoist
// (hoisted descriptors spill in a thread with few registers), and the issuing thread
// runs only a handful of instructions per MMA: with warps of the same sub-partition
// busy on softmax work, a thread that runs more issues an M128 N128 MMA only every
// 100-140 cycles against the 64 the tensor pipe needs (measured on GB300).
template <int A_OFF, int B_OFF>
__device__ __forceinline__ void mma_ss_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t d_hi, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 la, lb;\n\t.reg .b64 da, db;\n\t"
        "add.u32 la, %1, %6;\n\tadd.u32 lb, %2, %7;\n\tmov.b64 da, {la, %3};\n\tmov.b64 db, {lb, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(d_hi), "r"(idesc), "r"(accumulate), "n"(A_OFF), "n"(B_OFF));
}
template <int A_COL, int B_OFF>
__device__ __forceinline__ void mma_ts_lo(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t d_hi, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 ta, lb;\n\t.reg .b64 db;\n\t"
        "add.u32 ta, %1, %6;\n\tadd.u32 lb, %2, %7;\n\tmov.b64 db, {lb, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(d_hi), "r"(idesc), "r"(accumulate), "n"(A_COL), "n"(B_OFF));
}

// The same for a CTA pair (cta_group::2), issued by one thread of the even CTA.
template <int A_OFF, int B_OFF>
__device__ __forceinline__ void mma2_ss_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t d_hi,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 la, lb;\n\t.reg .b64 da, db;\n\t"
        "add.u32 la, %1, %6;\n\tadd.u32 lb, %2, %7;\n\tmov.b64 da, {la, %3};\n\tmov.b64 db, {lb, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\ttcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(d_hi), "r"(idesc), "r"(accumulate), "n"(A_OFF), "n"(B_OFF));
}
template <int A_COL, int B_OFF>
__device__ __forceinline__ void mma2_ts_lo(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t d_hi,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 ta, lb;\n\t.reg .b64 db;\n\t"
        "add.u32 ta, %1, %6;\n\tadd.u32 lb, %2, %7;\n\tmov.b64 db, {lb, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\ttcgen05.mma.cta_group::2.kind::f16 [%0], [ta], db, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(d_hi), "r"(idesc), "r"(accumulate), "n"(A_COL), "n"(B_OFF));
}

// High word of every 128-byte-swizzled shared-memory descriptor used here (stride
// 1024 bytes, descriptor version, swizzle mode); descriptors differ only in their
// low word, start address >> 4 (14 bits) and leading-byte offset.
__host__ __device__ constexpr uint32_t sdesc_sw128_hi() { return (uint32_t)((1024u >> 4) | (1u << 14) | (2u << 29)); }
__device__ __forceinline__ uint32_t sdesc_sw128_lo(uint32_t saddr, uint32_t lbo_bytes) {
    return ((saddr >> 4) & 0x3FFFu) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, dense.
// b_mn_major: B stored with N contiguous (otherwise K contiguous).
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4)                              // D format: f32
           | (1u << 7)                            // A format: bf16
           | (1u << 10)                           // B format: bf16
           | ((b_mn_major ? 1u : 0u) << 16)       // B major-ness
           | ((uint32_t)(N >> 3) << 17)           // N / 8
           | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile whose
// 8-row x 128-byte swizzle atoms start on 1024-byte boundaries.
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;  // swizzle: 128 B
    return d;
}

#define GATTN_R8(p, i) "=r"(p[i + 0]), "=r"(p[i + 1]), "=r"(p[i + 2]), "=r"(p[i + 3]), \
                       "=r"(p[i + 4]), "=r"(p[i + 5]), "=r"(p[i + 6]), "=r"(p[i + 7])
#define GATTN_W8(p, i) "r"(p[i + 0]), "r"(p[i + 1]), "r"(p[i + 2]), "r"(p[i + 3]), \
                       "r"(p[i + 4]), "r"(p[i + 5]), "r"(p[i + 6]), "r"(p[i + 7])

// 32 consecutive 32-bit TMEM columns of this thread's lane, waited on.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GATTN_R8(r, 0), GATTN_R8(r, 8), GATTN_R8(r, 16), GATTN_R8(r, 24)
        : "r"(taddr)
        : "memory");
}

// 64 consecutive columns (two loads, one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GATTN_R8(r, 0), GATTN_R8(r, 8), GATTN_R8(r, 16), GATTN_R8(r, 24), GATTN_R8(r, 32), GATTN_R8(r, 40),
          GATTN_R8(r, 48), GATTN_R8(r, 56)
        : "r"(taddr), "r"(taddr + 32)
        : "memory");
}

// Two runs of 64 consecutive columns at independent addresses (four loads, one wait).
__device__ __forceinline__ void tmem_ld64x2(uint32_t taddr_a, uint32_t (&a)[64], uint32_t taddr_b, uint32_t (&b)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
        "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
        "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GATTN_R8(a, 0), GATTN_R8(a, 8), GATTN_R8(a, 16), GATTN_R8(a, 24), GATTN_R8(a, 32), GATTN_R8(a, 40),
          GATTN_R8(a, 48), GATTN_R8(a, 56), GATTN_R8(b, 0), GATTN_R8(b, 8), GATTN_R8(b, 16), GATTN_R8(b, 24),
          GATTN_R8(b, 32), GATTN_R8(b, 40), GATTN_R8(b, 48), GATTN_R8(b, 56)
        : "r"(taddr_a), "r"(taddr_a + 32), "r"(taddr_b), "r"(taddr_b + 32)
        : "memory");
}

// 128 consecutive columns (four loads, one wait).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
        "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
        "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GATTN_R8(r, 0), GATTN_R8(r, 8), GATTN_R8(r, 16), GATTN_R8(r, 24), GATTN_R8(r, 32), GATTN_R8(r, 40),
          GATTN_R8(r, 48), GATTN_R8(r, 56), GATTN_R8(r, 64), GATTN_R8(r, 72), GATTN_R8(r, 80), GATTN_R8(r, 88),
          GATTN_R8(r, 96), GATTN_R8(r, 104), GATTN_R8(r, 112), GATTN_R8(r, 120)
        : "r"(taddr), "r"(taddr + 32), "r"(taddr + 64), "r"(taddr + 96)
        : "memory");
}

// Store 32 / 16 / 4 consecutive 32-bit columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        GATTN_W8(r, 0), GATTN_W8(r, 8), GATTN_W8(r, 16), GATTN_W8(r, 24)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        GATTN_W8(r, 0), GATTN_W8(r, 8)
        : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ register split

// Hand registers between the warpgroups of a block (every warp of a warpgroup runs
// the same one).  The block's total never changes: what the .dec warpgroups give
// back is what the .inc ones take, so the sum over warpgroups of the new counts
// must equal the count the block was launched with -- an .inc beyond that waits.
template <int N>
__device__ __forceinline__ void regs_raise() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_lower() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

// ------------------------------------------------------------------ warp-level mma (decode)

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// C[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile of
// 128-byte rows written by TMA with 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
    return r;
}

__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Shared-memory address of elements e0..e0+7 of row `row` in a tile stored as
// 128-byte-swizzled TMA boxes of [128 rows x 64 bf16].
__device__ __forceinline__ uint32_t rowtile_addr(uint32_t base, int row, int e0) {
    return base + (uint32_t)(e0 >> 6) * (128u * 128u) + sw128_offset((uint32_t)row, (uint32_t)((e0 >> 3) & 7));
}

}  // namespace gattn
