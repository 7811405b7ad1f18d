/*
 * gattn.h -- C ABI of libgattn, the GB300 (sm_103a) gated softmax attention core.
 *
 * The library computes, on one GPU, the part of a gated full-attention layer
 * that sits between the Q/K/V/gate projections and the output projection W_O:
 *
 *   1. QK-RMSNorm: per token and head, q and k (not v) are scaled by
 *      rsqrt(mean(x^2) + eps) and a learned weight of length head_dim.
 *      ("Gated attention" handbook chapter, section "Four things Qwen3.5 adds to
 *      the textbook", QK-Norm; "Attention, worked all the way through",
 *      section "Qwen3's exact order".)
 *   2. Partial RoPE on the first rotary_dim features of q and k only
 *      (handbook chapter, same section: "RoPE rotates only the first 64
 *      dimensions").  Reading used: rotate-half, feature i paired with
 *      i + rotary_dim/2, angle pos * rope_base^(-2i/rotary_dim).
 *   3. Causal scaled-dot-product attention with GQA sharing: query head h reads
 *      KV head floor(h / (H/G)); scores q.k / sqrt(head_dim); key j visible to
 *      query t iff j <= t; row softmax; weighted sum of v.
 *      (handbook chapter, section "The formula" and "The code:
 *      qwen/attention.py"; "Multi-head attention and GQA" chapter, section
 *      "分组查询注意力".)
 *   4. Output gate G1: the attention output of each head is multiplied by
 *      sigmoid(gate logits) -- one logit per dimension (elementwise) or one per
 *      head (headwise) -- and the heads are concatenated to [tokens, H*d].
 *      ("Gated Attention" deep-dive, section "门放在哪里？"; paper reading notes,
 *      section "从标准注意力走到门控，计算流程有什么变化".)  The variants the
 *      deep-dive compares are epilogue switches of the same kernels (see
 *      gattn_gate_mode): head-shared logits, NS-sigmoid (section "第二条机制
 *      线索": 0.5 + 0.5 sigmoid), SiLU (z * sigmoid(z)) and the additive form
 *      Y + act(z).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or retains them, and keeps no per-call state.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream).  Argument errors are detected on the
 *     host before anything is launched, and return a status without touching
 *     the GPU.
 *   - `out` must not alias any input or the workspace.
 *   - Element types: GATTN_BF16 means q, k, v, gate, norm weights, cache and out
 *     are all bfloat16 (fp32 accumulation inside); GATTN_FP32 means all fp32.
 *   - Strides are in ELEMENTS.  A stride of 0 selects the contiguous default.
 *   - Kernels never trap.  Problems found on the device (a sequence length
 *     outside [1, Lmax], a bounded wait that ran out) set bits in a device
 *     status word readable with gattn_get_device_status().
 */
#ifndef GATTN_H
#define GATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GATTN_OK = 0,
    GATTN_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer or stride */
    GATTN_ERR_UNSUPPORTED = 2,  /* valid arguments this build has no kernel for (e.g. head_dim 96) */
    GATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed */
    GATTN_ERR_WORKSPACE = 4,    /* workspace pointer missing, misaligned or too small */
    GATTN_ERR_DEVICE = 5,       /* gattn_get_device_status found a device-side problem (not a timeout) */
    GATTN_ERR_DEVICE_TIMEOUT = 6 /* gattn_get_device_status found that a bounded wait inside a kernel ran out */
} gattn_status;

/*
 * Gate mode = layout | activation | combine (bit fields; the plain layout values
 * alone mean the default multiplicative sigmoid gate).
 *   layout (bits 0-3): NONE (no gate; activation and combine must be 0),
 *     ELEMENTWISE logits [B,S,H,d] (decode [B,H,d]), HEADWISE [B,S,H] ([B,H]),
 *     HEAD_SHARED [B,S,d] ([B,d]): one vector of logits used by every head.
 *   activation (bits 4-7): SIGMOID, NS_SIGMOID = 0.5 + 0.5 sigmoid(z),
 *     SILU = z * sigmoid(z).
 *   combine (bit 8): multiplicative out = o * act(z) (default) or
 *     GATTN_GATE_ADDITIVE out = o + act(z).
 * Any other value is GATTN_ERR_INVALID_ARG.
 */
typedef enum {
    GATTN_GATE_NONE = 0,
    GATTN_GATE_ELEMENTWISE = 1,
    GATTN_GATE_HEADWISE = 2,
    GATTN_GATE_HEAD_SHARED = 3,
    GATTN_GATE_ACT_SIGMOID = 0x00,
    GATTN_GATE_ACT_NS_SIGMOID = 0x10,
    GATTN_GATE_ACT_SILU = 0x20,
    GATTN_GATE_ADDITIVE = 0x100
} gattn_gate_mode;
#define GATTN_GATE_LAYOUT_MASK 0x0Fu
#define GATTN_GATE_ACT_MASK 0xF0u

typedef enum { GATTN_BF16 = 0, GATTN_FP32 = 1 } gattn_dtype;

/* Device status bits (gattn_get_device_status). */
#define GATTN_DEVICE_BAD_SEQLEN 0x1u  /* a decode seqlens[b] was outside [1, Lmax]; that sequence was skipped */
#define GATTN_DEVICE_TIMEOUT 0x2u     /* a bounded wait inside a kernel ran out; its output is not valid */
#define GATTN_DEVICE_BAD_PAGE 0x4u    /* a paged-cache block table entry was outside [0, num_pages); page 0 was read
                                         instead and nothing was appended there */

/* Human-readable name of a status code.  Never NULL. */
const char* gattn_strerror(gattn_status status);

/*
 * Bytes of workspace gattn_prefill needs.  The workspace holds the normed and
 * rotated keys (and, for GATTN_FP32, the normed and rotated queries), written
 * and read within one call.  Returns 0 for invalid sizes.
 */
size_t gattn_prefill_workspace_size(int B, int S, int H, int G, int d, int dtype);

/*
 * Causal gated GQA attention over whole sequences (prefill).
 *
 * q        [B,S,H,d] raw query projections.  Element (b,t,h,e) is at
 *          q[(b*S + t)*q_tok_stride + h*q_head_stride + e]; defaults
 *          q_tok_stride = H*d, q_head_stride = d.  This lets q point into the
 *          packed q_proj output [B,S,H,2d] whose first d values per head are the
 *          query (handbook chapter, section "Why the gate is packed into
 *          q_proj"): pass q_tok_stride = 2*H*d, q_head_stride = 2*d.
 * k, v     [B,S,G,d] contiguous raw key / value projections.
 * gate     gate logits; elementwise [B,S,H,d] at gate[(b*S+t)*gate_tok_stride +
 *          h*gate_head_stride + e] (defaults H*d, d), headwise [B,S,H] at
 *          gate[(b*S+t)*gate_tok_stride + h*gate_head_stride] (defaults H, 1),
 *          head-shared [B,S,d] at gate[(b*S+t)*gate_tok_stride + e] (default d;
 *          gate_head_stride ignored).  Ignored (may be NULL) for GATTN_GATE_NONE.
 * qnorm_w, knorm_w  [d] RMSNorm weights, shared by all heads.
 * pos      [B,S] int32 RoPE positions, or NULL for positions 0..S-1.  The mask
 *          always uses the token index, not pos.
 * B,S,H,G,d  batch, tokens per sequence, query heads, KV heads, head_dim.
 *          Requires H % G == 0, S >= 1.  d in {64,128,256} for GATTN_BF16 and
 *          d in {32,64,128,256} for GATTN_FP32 (others: GATTN_ERR_UNSUPPORTED).
 *          bf16 d = 32 has no kernel: the tensor-core kernels move Q, K, V, the
 *          gate and the output as 128-byte (64-element) swizzled TMA boxes along
 *          head_dim, and a 32-element bf16 row is only 64 bytes wide.
 * rotary_dim  even, 0 <= rotary_dim <= d.  rope_base > 0.  eps >= 0.
 * workspace  device buffer of at least gattn_prefill_workspace_size() bytes,
 *          256-byte aligned.
 * out      [B,S,H*d] contiguous; head h occupies columns h*d .. h*d+d-1.
 * Alignment: q, k, v, gate, out and the workspace must be 16-byte aligned, and
 *          the q/gate strides multiples of 8 elements (bf16) / 4 (fp32), except
 *          headwise gate strides which may be anything.
 */
gattn_status gattn_prefill(const void* q, const void* k, const void* v, const void* gate, const void* qnorm_w,
                           const void* knorm_w, const int32_t* pos, int B, int S, int H, int G, int d,
                           int rotary_dim, double rope_base, float eps, int gate_mode, int64_t q_tok_stride,
                           int64_t q_head_stride, int64_t gate_tok_stride, int64_t gate_head_stride, int dtype,
                           void* workspace, size_t workspace_bytes, void* out, void* stream);

/*
 * Causal gated GQA attention over PACKED variable-length sequences (varlen):
 * sequence i occupies tokens [cu_seqlens[i], cu_seqlens[i+1]) of the packed
 * tensors and attends only to its own keys, its RoPE positions restarting at 0
 * (a padding-free form of the causal / padding mask M of the "Gated Attention"
 * deep-dive's statement of the layer).
 *
 * q        [T,H,d] at q[t*q_tok_stride + h*q_head_stride + e] (defaults H*d, d).
 * k, v     [T,G,d] contiguous.
 * gate     [T,H,d], [T,H] or [T,d] per gate_mode, strides as for gattn_prefill.
 * pos      [T] int32 device positions, or NULL for 0..len-1 within each sequence.
 * cu_seqlens  [nseq+1] int32 HOST array: 0 = cu_seqlens[0] <= ... <=
 *          cu_seqlens[nseq] = T; empty sequences are allowed.  The library builds
 *          its schedule from it on the host and copies that into the workspace on
 *          `stream` before returning.
 * out      [T,H*d].  Everything else as gattn_prefill, with B = 1 and S = T.
 * workspace  >= gattn_prefill_varlen_workspace_size(T, nseq, H, G, d, dtype).
 * T = 0 returns GATTN_OK without launching anything.
 */
size_t gattn_prefill_varlen_workspace_size(int T, int nseq, int H, int G, int d, int dtype);
gattn_status gattn_prefill_varlen(const void* q, const void* k, const void* v, const void* gate, const void* qnorm_w,
                                  const void* knorm_w, const int32_t* pos, const int32_t* cu_seqlens, int nseq, int H,
                                  int G, int d, int rotary_dim, double rope_base, float eps, int gate_mode,
                                  int64_t q_tok_stride, int64_t q_head_stride, int64_t gate_tok_stride,
                                  int64_t gate_head_stride, int dtype, void* workspace, size_t workspace_bytes,
                                  void* out, void* stream);

/*
 * Output projection that follows the attention: y = x W_O^T, x the gated attention
 * output in the layout gattn_prefill / gattn_prefill_varlen write ("Transformer by
 * Hand, ch. 6", section "The code: qwen/attention.py": the concatenated heads, times
 * the gate's sigmoid, go through o_proj; "Gated Attention for LLMs 论文阅读": the
 * gate acts on the SDPA output ahead of the output projection).
 *
 * x    [T, K] bf16 device, row-major (K = H*d; row stride K elements).
 * w_o  [N, K] bf16 device, row-major: the weight of a linear layer, y = x w_o^T.
 * y    [T, N] bf16 device, row-major: sum_k x[t,k] w_o[n,k] in fp32, rounded once.
 * T >= 1; K and N multiples of 64 (>= 64); x, w_o and y 16-byte aligned.  y must
 * not overlap x or w_o.  Asynchronous on `stream`; the caller owns every buffer.
 * Returns GATTN_ERR_INVALID_ARG for bad sizes, pointers or alignment, GATTN_ERR_CUDA
 * if a launch fails; a bounded wait that runs out inside the kernel sets
 * GATTN_DEVICE_TIMEOUT (gattn_get_device_status) and leaves y incomplete.
 */
gattn_status gattn_o_proj(const void* x, const void* w_o, int T, int K, int N, void* y, void* stream);

/*
 * Bytes of workspace gattn_decode needs (per-split partial softmax states).
 * Depends on the current device's SM count.  Returns 0 for invalid sizes.
 */
size_t gattn_decode_workspace_size(int B, int H, int G, int d, int Lmax);

/*
 * One decode step: each sequence's newest query attends to its cached keys.
 * (KV cache: "Multi-head attention and GQA" chapter, section "拼接各头 → 用 W_O
 * 投影": K and V are cached per token, Q is not; the new query dots every cached
 * key and mixes every cached value.)
 *
 * q_new    [B,H,d] raw query projections of the newest token (not yet normed or
 *          rotated); it sits at position seqlens[b]-1.
 * kv_cache [2,B,G,Lmax,d] contiguous: plane 0 holds K already normed and rotated
 *          (as the prefill path computes it), plane 1 holds raw V.  Only tokens
 *          0..seqlens[b]-1 are read; entries beyond may hold anything.
 * seqlens  [B] int32 device array, cached tokens per sequence INCLUDING the new
 *          one, each in [1, Lmax].  A value outside that range sets
 *          GATTN_DEVICE_BAD_SEQLEN and leaves that sequence's output unwritten.
 * gate     [B,H,d] (elementwise), [B,H] (headwise) or [B,d] (head-shared)
 *          logits; NULL for none.
 * qnorm_w  [d].  d in {64,128,256}; H/G <= 8; only GATTN_BF16 (implied).
 * workspace  >= gattn_decode_workspace_size() bytes, 256-byte aligned.
 * out      [B,H*d] bf16.
 */
gattn_status gattn_decode(const void* q_new, const void* kv_cache, const int32_t* seqlens, const void* gate,
                          const void* qnorm_w, int B, int H, int G, int d, int Lmax, int rotary_dim,
                          double rope_base, float eps, int gate_mode, void* workspace, size_t workspace_bytes,
                          void* out, void* stream);

/*
 * One decode step that first appends the new token to the cache: for every
 * sequence b with 1 <= seqlens[b] <= Lmax and KV head g,
 *   kv_cache[0,b,g,seqlens[b]-1,:] = rope(rmsnorm(k_new[b,g,:]) * knorm_w)
 *                                    at position seqlens[b]-1,
 *   kv_cache[1,b,g,seqlens[b]-1,:] = v_new[b,g,:],
 * then exactly gattn_decode (which reads the appended row).  This is the caller
 * pass before gattn_decode folded into the call: the new token's QK-RMSNorm and
 * partial RoPE for K ("Gated attention" handbook chapter, section "Four things
 * Qwen3.5 adds to the textbook") and the per-token K/V cache ("Multi-head
 * attention and GQA" chapter, section "拼接各头 → 用 W_O 投影").
 *
 * k_new, v_new  [B,G,d] bf16 contiguous raw key / value projections of the new
 *          token, 16-byte aligned.
 * kv_cache [2,B,G,Lmax,d] as for gattn_decode, written at row seqlens[b]-1.
 * knorm_w  [d] bf16, 16-byte aligned.
 * Everything else, and the errors, as gattn_decode; sequences whose length is
 * outside [1, Lmax] are neither appended nor decoded (GATTN_DEVICE_BAD_SEQLEN).
 */
gattn_status gattn_decode_append(const void* q_new, const void* k_new, const void* v_new, void* kv_cache,
                                 const int32_t* seqlens, const void* gate, const void* qnorm_w, const void* knorm_w,
                                 int B, int H, int G, int d, int Lmax, int rotary_dim, double rope_base, float eps,
                                 int gate_mode, void* workspace, size_t workspace_bytes, void* out, void* stream);

/*
 * One decode step against a PAGED KV cache, optionally appending the new token
 * first.  The cache is a pool of pages, each holding page_size consecutive tokens
 * of one sequence for every KV head:
 *   kv_pages    [2, num_pages, G, page_size, d] bf16 contiguous, 16-byte aligned
 *               (plane 0 K normed and rotated, plane 1 raw V, as in gattn_decode);
 *   block_table [B, max_pages] int32 device array: the tokens
 *               [p*page_size, (p+1)*page_size) of sequence b are in page
 *               block_table[b*max_pages + p].  Only the entries that cover tokens
 *               0..seqlens[b]-1 are read.
 * page_size must be a multiple of 64 (a key tile of the kernel never straddles
 * two pages; others: GATTN_ERR_UNSUPPORTED); sequences hold at most
 * max_pages*page_size tokens (seqlens[b] in [1, max_pages*page_size]).  An entry
 * outside [0, num_pages) sets GATTN_DEVICE_BAD_PAGE (that step's output is not
 * valid; nothing is read or written outside the pool).
 * k_new, v_new, knorm_w: NULL for no append, else as gattn_decode_append (the new
 * token goes to row (seqlens[b]-1) % page_size of page
 * block_table[b*max_pages + (seqlens[b]-1)/page_size]).
 * Everything else as gattn_decode, with Lmax = max_pages * page_size for
 * gattn_decode_workspace_size.
 */
gattn_status gattn_decode_paged(const void* q_new, const void* k_new, const void* v_new, void* kv_pages,
                                const int32_t* block_table, int num_pages, int page_size, int max_pages,
                                const int32_t* seqlens, const void* gate, const void* qnorm_w, const void* knorm_w,
                                int B, int H, int G, int d, int rotary_dim, double rope_base, float eps, int gate_mode,
                                void* workspace, size_t workspace_bytes, void* out, void* stream);

/*
 * One decode step exactly like gattn_decode, for callers that cannot allocate
 * device memory when they run it -- for example a serving loop that must not call
 * cudaMalloc while requests are in flight (it can synchronise the whole device),
 * or a host framework that hands a plugin its buffers and forbids it to allocate
 * any of its own.  The source pages have no counterpart to this entry point: it
 * exists only to spare such callers the workspace.
 *
 * Arguments, layouts and errors are those of gattn_decode minus the workspace.
 * The partial softmax states live instead in one fixed array of device memory
 * inside the library, GATTN_DECODE_NOALLOC_SCRATCH_BYTES (8 MiB) long, that every
 * GPU which loads the library holds until the process exits.  A problem whose
 * gattn_decode_workspace_size() exceeds that limit is rejected with
 * GATTN_ERR_WORKSPACE before anything is launched.  The entry point itself calls
 * no cudaMalloc, cudaFree or other allocating routine.
 *
 * Set-up: the first call with a given device current looks up the array's device
 * address (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.  All calls share the one array and it keeps the last call's
 * contents; nothing in it needs to start at zero.  Calls whose executions overlap
 * on the GPU (on different streams, say) race on the array and give wrong
 * results: serialise them.
 */
#define GATTN_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
gattn_status gattn_decode_noalloc(const void* q_new, const void* kv_cache, const int32_t* seqlens, const void* gate,
                                  const void* qnorm_w, int B, int H, int G, int d, int Lmax, int rotary_dim,
                                  double rope_base, float eps, int gate_mode, void* out, void* stream);

/*
 * Read (synchronously on `stream`) and clear the device status word.  Writes the
 * GATTN_DEVICE_* bits seen since the last call to *bits (may be NULL) and returns
 * GATTN_ERR_DEVICE_TIMEOUT if GATTN_DEVICE_TIMEOUT is among them,
 * GATTN_ERR_DEVICE if any other bit was set, GATTN_OK otherwise.
 */
gattn_status gattn_get_device_status(unsigned int* bits, void* stream);

/*
 * Self-test of the bounded-wait machinery every kernel of this library relies on
 * (no counterpart on the source pages).  Launches one small kernel on `stream`
 * whose threads wait on an mbarrier that nothing ever arrives on, through the same
 * wait routine the attention kernels use, with a wall-clock limit of
 * `limit_ns` nanoseconds (1 .. 100 ms) instead of the kernels' 2 s.  One thread
 * runs out of time, raises the block's abort flag and sets GATTN_DEVICE_TIMEOUT in
 * the device status word; the other threads see the flag and stop waiting; the
 * block returns normally, so the CUDA context stays usable.  *waited_ns (device
 * memory, may be NULL) receives how long the timed-out wait lasted.
 * Returns GATTN_ERR_INVALID_ARG for a limit outside that range, GATTN_ERR_CUDA if
 * the launch fails, GATTN_OK otherwise; the timeout itself is read back with
 * gattn_get_device_status().
 */
gattn_status gattn_selftest_wait_timeout(unsigned long long limit_ns, unsigned long long* waited_ns, void* stream);

/*
 * Profiling hook.  When both events are non-NULL (cudaEvent_t passed as void*),
 * every later gattn_prefill / gattn_decode / gattn_o_proj records `start` on its
 * stream just before its main kernel and `stop` just after it, so a caller can
 * time that kernel alone.  Pass NULL, NULL to switch it off.  Not thread-safe.
 */
void gattn_set_profile_events(void* start, void* stop);

#ifdef __cplusplus
}
#endif

#endif /* GATTN_H */
