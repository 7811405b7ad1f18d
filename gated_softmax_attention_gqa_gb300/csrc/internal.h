// internal.h -- parameter blocks and launchers shared between the host ABI
// (api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gattn.h"

namespace gattn {

constexpr int kMaxRotaryHalf = 128;  // rotary_dim <= 256

// Normalise + rotate rows of a [B,S,n_heads,d] tensor (token/head strides in
// elements) into a contiguous [B,n_heads,S,d] tensor of the same or wider type.
struct ProloguePlan {
    const void* x;
    int64_t tok_stride, head_stride;
    const void* w;
    const int32_t* pos;
    void* dst;
    int B, S, n_heads, d, rd;
    float eps;
    unsigned int* status;  // device status word (bounded-wait expiry)
    float inv_freq[kMaxRotaryHalf];
};

// bf16 tcgen05 prefill.
struct PrefillParams {
    const void* q;
    const void* gate;
    const void* qnorm_w;
    const void* knorm_w;  // read by the attention kernels only to bound the logits
    const int32_t* pos;
    void* out;
    int64_t q_tok_stride, q_head_stride, gate_tok_stride, gate_head_stride;
    int B, S, H, G, d, rd, gate_mode, n_qtiles;
    int n_sms;  // multiprocessors of the device (persistent grids)
    float eps, scale_log2;
    unsigned int* status;
    // packed variable-length sequences (vtiles != NULL; then B = 1 and S is the
    // packed token count): the query tiles, heaviest first, each
    // {start token, sequence length, tile index within the sequence, sequence}
    const int4* vtiles;
    int n_vtiles;
    float inv_freq[kMaxRotaryHalf];
};

// fp32 SIMT prefill over pre-normed/rotated q', k' (workspace) and raw v.
struct PrefillF32Params {
    const float* qr;  // [B,H,S,d]
    const float* kr;  // [B,G,S,d]
    const float* v;   // [B,S,G,d]
    const float* gate;
    float* out;
    int64_t gate_tok_stride, gate_head_stride;
    int B, S, H, G, d, gate_mode;
    float scale;
    const int32_t* tok_start;  // packed sequences: first token of each token's sequence (else NULL)
};

// bf16 split-KV decode.
struct DecodeParams {
    const void* q;  // [B,H,d]
    const int32_t* seqlens;
    const void* gate;
    const void* qnorm_w;
    void* out;      // [B,H*d]
    float* part;    // partial softmax states
    int B, H, G, d, Lmax, rd, gate_mode, n_ctas;
    float eps, scale_log2;
    unsigned int* status;
    // paged cache (block_table != NULL): [2, num_pages, G, page_size, d]; the keys
    // [p*page_size, (p+1)*page_size) of sequence b live in page block_table[b*max_pages + p]
    const int32_t* block_table;
    int max_pages, page_size, num_pages;
    float inv_freq[kMaxRotaryHalf];
};

// Append of the new token to the decode KV cache: k' = rope(rmsnorm(k_new) * w) at
// position seqlens[b]-1 and the raw v_new, into cache[0/1, b, g, seqlens[b]-1, :].
struct AppendParams {
    const void* k_new;  // [B,G,d]
    const void* v_new;  // [B,G,d]
    const void* knorm_w;
    void* cache;        // [2,B,G,Lmax,d]
    const int32_t* seqlens;
    int B, G, d, Lmax, rd;
    float eps;
    unsigned int* status;
    const int32_t* block_table;  // paged cache, as in DecodeParams (NULL: contiguous)
    int max_pages, page_size, num_pages;
    float inv_freq[kMaxRotaryHalf];
};

// TMA descriptors of the tcgen05 prefill: normed keys (workspace), raw V, raw Q,
// (elementwise gate only) the gate logits and the output; all bf16, 64-element inner boxes.
struct PrefillMaps {
    CUtensorMap k, v, q, gate, out;  // out: [B,S,H*d] as (d, H, S, B), written by TMA stores
};

cudaError_t launch_prologue(const ProloguePlan& p, bool bf16_in, bool bf16_out, cudaStream_t stream);
// Packed sequences: from the query-tile table, every token's position within its
// sequence and the first token of its sequence.
cudaError_t launch_varlen_positions(const int4* tiles, int n_tiles, int32_t* pos, int32_t* tok_start,
                                    cudaStream_t stream);
cudaError_t launch_prefill_tc(const PrefillParams& p, const PrefillMaps& maps, cudaStream_t stream,
                              cudaEvent_t ev_start, cudaEvent_t ev_stop);
// CTA-pair (cta_group::2) tcgen05 prefill: two heads of one KV group per cluster.
bool prefill_pair_supported(int d, int H, int G);
int prefill_pair_key_rows();    // K' rows per TMA box
int prefill_pair_value_rows();  // V rows per TMA box
cudaError_t launch_prefill_pair(const PrefillParams& p, const PrefillMaps& maps, cudaStream_t stream,
                                cudaEvent_t ev_start, cudaEvent_t ev_stop);
cudaError_t launch_prefill_f32(const PrefillF32Params& p, cudaStream_t stream, cudaEvent_t ev_start,
                               cudaEvent_t ev_stop);
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& tm_kv, cudaStream_t stream,
                          cudaEvent_t ev_start, cudaEvent_t ev_stop);
cudaError_t launch_decode_append(const AppendParams& p, cudaStream_t stream);

// Output projection y = x W_O^T (bf16, tcgen05): x [T, K], W_O [N, K], y [T, N].
struct OprojParams {
    void* y;
    int T, K, N;
    int n_sms;
    unsigned int* status;
};
int oproj_block_n(int N);   // output columns per tile
int oproj_box_rows(int N);  // W_O rows per TMA box (half a tile's: each CTA of a pair holds half)
cudaError_t launch_oproj(const OprojParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, cudaStream_t stream,
                         cudaEvent_t ev_start, cudaEvent_t ev_stop);

// Prefill tile geometry for the tcgen05 kernel, per head_dim.
int prefill_block_n(int d);

int decode_max_batch();

// Host-side argument checks of a decode step, every one but the workspace's, with
// the status gattn_decode returns for them (cache_rows < 0: the contiguous cache
// [2,B,G,Lmax,d]).
gattn_status decode_check_args(const void* q_new, const void* kv_cache, const int32_t* seqlens, const void* gate,
                               const void* qnorm_w, int B, int H, int G, int d, int Lmax, int rotary_dim,
                               double rope_base, float eps, int gate_mode, const void* out, int64_t cache_rows);

// Decode work split: the size of one partial-state slot in floats and the
// number of slots the workspace must hold.
int decode_slot_floats(int r, int d);
int64_t decode_num_slots(int n_ctas, int B, int G);
constexpr int kDecodeConsumerWarps = 4;
constexpr int kDecodeTileKeys = 64;

}  // namespace gattn
