// Host-side launchers of the QSA kernels (internal to libqsa.so).
#pragma once

#include <cuda_runtime.h>
#include <cuda.h>
#include <stdint.h>

namespace qsa {

// Message for qsa_last_error_detail() on this host thread.
void set_error_detail(const char *msg);

// inv_freq[i] = theta^(-2i/64), computed on the host in double.
struct RopeFreqs {
    double inv_freq[32];
};

// Block keys of blocks t_begin/4 .. L/4-1 and RoPE'd K rows t_begin .. L-1
// (t_begin = 0: everything).
cudaError_t launch_kprep(int batch, int64_t t_begin, int64_t L, int64_t max_ctx, const uint16_t *ki,
                         const uint16_t *k, uint16_t *k_rot, uint16_t *kblk,
                         const RopeFreqs &freqs, int sms, cudaStream_t stream);

// ---- prefill indexer + selection (tcgen05) ----
int index_grid(int64_t L, int sms);
size_t index_cand_bytes(int64_t L, int sms);
// Queries are tokens q_off .. q_off+Lq-1 (qi, w, idx, score hold their Lq
// rows); the keys (map_k) cover every complete selection unit before
// q_off+Lq.  unit_tokens: 4 (micro-blocks) or 1 (a token-level indexer).
cudaError_t launch_index(const CUtensorMap &map_q, const CUtensorMap &map_k, int64_t q_off, int64_t Lq,
                         int unit_tokens, int budget, const uint16_t *w, int32_t *idx, float *score,
                         float *dense, void *cand_ws, int32_t *status, int sms, int *stop,
                         cudaStream_t stream);
// The prediction stop word of a call: the last 256 bytes of a candidate
// workspace of index_cand_bytes(L, sms) bytes (zeroed by the caller once per call).
inline int *index_stop_word(void *cand_ws, size_t cand_bytes) {
    return reinterpret_cast<int *>(static_cast<uint8_t *>(cand_ws) + cand_bytes - 256);
}
cudaError_t launch_fill_current_only(int64_t q_off, int64_t Lq, int unit_tokens, int budget, int32_t *idx,
                                     float *score, cudaStream_t stream);

// ---- block-sparse attention (prefill and decode splits) ----
struct AttnArgs {
    const uint16_t *q;       // [items, 24, 256] pre-RoPE
    const uint16_t *k;       // key rows (post-RoPE), sequence s starts at s * seq_stride rows
    const uint16_t *v;
    int64_t seq_stride;      // rows between sequences (decode: max_ctx; prefill: 0)
    const int32_t *idx;      // [items, budget]
    int budget;
    const int32_t *seq_lens; // decode: [B] device; prefill: null
    int64_t L;               // prefill: number of query rows
    int64_t q_off;           // prefill: position of the first query row (0 without a cached prefix)
    uint16_t *out;           // final output (nsplit == 1)
    float *lse;              // final lse or null
    float *part_o;           // [B, nsplit, 24, 256] (nsplit > 1)
    float *part_lse;         // [B, nsplit, 24]
    int nsplit;
    float scale_log2;        // softmax scale * log2(e)
    int32_t *status;
};
cudaError_t launch_attn_prefill(const AttnArgs &a, const RopeFreqs &f, cudaStream_t stream);
cudaError_t launch_attn_decode(const AttnArgs &a, int batch, const RopeFreqs &f,
                               cudaStream_t stream);
cudaError_t launch_attn_combine(const float *part_o, const float *part_lse, int batch,
                                int nsplit, uint16_t *out, float *lse, cudaStream_t stream);
// The same attention on the tcgen05 tensor cores (sparse_attn_tc.cu).  map_k
// and map_v are 5-D maps {64 dims, rows per sequence, 2 KV heads, 4 dim
// chunks, sequences} of K' and V with boxes {64, 4, 2, 4, 1} (one block,
// 128-byte swizzle); key_rows = rows per sequence (the coordinate of an
// unused slot, read as zeros).
cudaError_t launch_attn_prefill_tc(const AttnArgs &a, const RopeFreqs &f, const CUtensorMap &map_k,
                                   const CUtensorMap &map_v, int64_t key_rows, cudaStream_t stream);
cudaError_t launch_attn_decode_tc(const AttnArgs &a, int batch, const RopeFreqs &f, const CUtensorMap &map_k,
                                  const CUtensorMap &map_v, cudaStream_t stream);

// ---- decode indexer ----
struct DecodePlan {
    int64_t chunk;    // blocks per scan CTA
    int nchunk;       // scan CTAs per sequence
    int nsplit;       // attention splits per sequence
};
DecodePlan decode_plan(int batch, int64_t max_ctx, int sms);
size_t decode_ws_bytes(int batch, int64_t max_ctx, int budget, int sms);
size_t decode_index_ws_bytes(int batch, int64_t max_ctx);  // leading part of the decode workspace
// k_cache / v_cache (or null): the filter prefetches the K and V rows of its
// candidate blocks into L2 for the decode attention that follows.
cudaError_t launch_decode_index(int batch, int64_t max_ctx, const DecodePlan &plan,
                                const uint16_t *qi, const uint16_t *w, const uint16_t *kblk,
                                const int32_t *seq_lens, int budget, void *ws, int32_t *idx_out,
                                int32_t *status, const uint16_t *k_cache, const uint16_t *v_cache,
                                cudaStream_t stream);

}  // namespace qsa
