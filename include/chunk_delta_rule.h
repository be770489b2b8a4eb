/*
 * chunk_delta_rule.h -- C ABI of the chunked gated delta-rule output.
 *
 * What is computed follows atrex-bench "chunk_delta_rule_output" (page #004,
 * reference.py, Model.forward).  Tokens are cut into chunks of chunk_size;
 * for chunk c of batch b and value head hd, which reads query/key head
 * qh = min(hd / max(Hv / Hq, 1), Hq - 1), and rows r, j of the chunk:
 *
 *   out[r,:] = scale * ( exp(g[r]) * q[r] h[c]
 *                        + sum over j <= r with g[r] <= g[j] of
 *                          bf16(q[r] . k[j] * exp(g[r] - g[j])) * v[j] )
 *
 * bf16() rounds to bfloat16 (nearest even) as the page does before the value
 * product; accumulation is fp32 and the output is rounded to bf16.
 * scale = key_dim^-1/2 when scale <= 0.  Return codes are the ATTN_VARLEN_*
 * codes of attn_varlen.h.
 */
#ifndef CHUNK_DELTA_RULE_H_
#define CHUNK_DELTA_RULE_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime.h>

#include "attn_varlen.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * chunk_delta_rule_output -- the output stage of a chunked gated delta rule.
 *
 *   q, k        bf16 device [batch, tokens, num_q_heads, key_dim], 16-byte aligned
 *   v           bf16 device [batch, tokens, num_v_heads, value_dim]
 *   h           bf16 device [batch, ceil(tokens / chunk_size), num_v_heads,
 *               key_dim, value_dim]: the state entering each chunk
 *   g           float32 device [batch, tokens, num_v_heads]: per-token log gates
 *   batch, tokens  >= 0 (either 0: returns ATTN_VARLEN_OK, launches nothing)
 *   num_q_heads, num_v_heads  >= 1
 *   key_dim, value_dim  128 (else ATTN_VARLEN_ERR_UNSUPPORTED_DIM)
 *   chunk_size  64 (the page's; else ATTN_VARLEN_ERR_INVALID_ARG)
 *   scale       > 0, or <= 0 for key_dim^-1/2
 *   out         bf16 device [batch, tokens, num_v_heads, value_dim], 16-byte
 *               aligned, not overlapping the inputs
 *   stream      CUDA stream the work is queued on
 *
 * All buffers are caller-owned; the call is asynchronous and allocates
 * nothing.
 */
int chunk_delta_rule_output(const void* q, const void* k, const void* v, const void* h,
                            const float* g, int batch, int tokens, int num_q_heads,
                            int num_v_heads, int key_dim, int value_dim, int chunk_size,
                            float scale, void* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CHUNK_DELTA_RULE_H_ */
