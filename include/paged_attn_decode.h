/*
 * paged_attn_decode.h -- C ABI of the single-query paged attention decode.
 *
 * What is computed follows atrex-bench "paged_attention_decode" (page #024,
 * reference.py, Model.forward): for sequence i with ctx_len = seq_lens[i]
 * context tokens, every query head h gets
 *
 *     out[i, h, :] = softmax(query[i, h, :] . K_i^T * head_size^-1/2) V_i
 *
 * where token t of the context sits at position t % block_size of physical
 * block block_tables[i][t / block_size], KV head g = h / (Hq / Hkv) serves
 * Hq / Hkv consecutive query heads, and
 *
 *     key[d]   = k_cache[block][g][d / 8][t % block_size][d % 8]
 *     value[d] = v_cache[block][g][d][t % block_size].
 *
 * A sequence with ctx_len <= 0 gets zero rows.  Accumulation is fp32; the
 * output is rounded to the input type (nearest even).  Return codes are the
 * ATTN_VARLEN_* codes of attn_varlen.h; device-side errors are reported by
 * attn_varlen_check on the same stream.
 */
#ifndef PAGED_ATTN_DECODE_H_
#define PAGED_ATTN_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime.h>

#include "attn_varlen.h"

#ifdef __cplusplus
extern "C" {
#endif

#define PAGED_ATTN_BF16 0
#define PAGED_ATTN_FP16 1

/*
 * paged_attn_decode -- one decode step of attention over a paged KV cache.
 *
 *   query          device [num_seqs, num_query_heads, head_size], 16-byte aligned
 *   k_cache        device [num_blocks, num_kv_heads, head_size / 8, block_size, 8]
 *   v_cache        device [num_blocks, num_kv_heads, head_size, block_size]
 *   block_tables   int32 device [num_seqs, max_blocks_per_seq]; every entry a
 *                  sequence's context reaches must lie in [0, num_blocks); an
 *                  entry outside it is not read, and attn_varlen_check then
 *                  returns ATTN_VARLEN_ERR_BAD_BLOCK_TABLE
 *   seq_lens       int32 device [num_seqs]; tokens beyond
 *                  max_blocks_per_seq * block_size are not read
 *   num_seqs       >= 0 (0: returns ATTN_VARLEN_OK, launches nothing)
 *   num_query_heads, num_kv_heads
 *                  >= 1, num_query_heads a multiple of num_kv_heads
 *   head_size      64, 128 or 256 (else ATTN_VARLEN_ERR_UNSUPPORTED_DIM)
 *   block_size     16 (the page's; others return ATTN_VARLEN_ERR_INVALID_ARG)
 *   max_blocks_per_seq, num_blocks
 *                  >= 1 when num_seqs > 0
 *   dtype          PAGED_ATTN_BF16 or PAGED_ATTN_FP16, for query, caches and out
 *   out            device [num_seqs, num_query_heads, head_size], 16-byte aligned
 *   stream         CUDA stream the work is queued on
 *
 * All buffers are caller-owned.  The call is asynchronous and uses the
 * library-owned per-device workspace for its status word only.
 */
int paged_attn_decode(const void* query, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                      int num_query_heads, int num_kv_heads, int head_size, int block_size,
                      int max_blocks_per_seq, int num_blocks, int dtype, void* out,
                      cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_DECODE_H_ */
