/*
 * attn_varlen.h -- C ABI of the GB300 (sm_103a) packed variable-length
 * attention forward.
 *
 * The operation is atrex-bench "attention_forward" (page #001, reference.py,
 * Model.forward): for every sequence i whose query slice
 * [cu_seqlens_q[i], cu_seqlens_q[i+1]) is non-empty and every head h,
 *
 *     out[slice_q, h, :] = softmax(q[slice_q, h, :] . k[slice_k, h, :]^T * D^-1/2)
 *                          . v[slice_k, h, :]
 *
 * with slice_k = [cu_seqlens_k[i], cu_seqlens_k[i+1]), non-causal, and the
 * scale fixed at head_dim^-1/2 (the page passes no scale, so the library
 * default applies, computed with the true head_dim).  Sequences with an empty
 * query slice are skipped (the page's loop does the same); a non-empty query
 * slice with an empty key slice gets zero rows.  Output rows that no query
 * slice covers are never written (the page allocates the output with
 * empty_like).
 *
 * Layout (page #001, input.py): q, out are bf16 [total_q, num_heads,
 * head_dim] and k, v are bf16 [total_k, num_heads, head_dim], contiguous,
 * token-major; cu_seqlens_q/k are int32 [num_seqs + 1] prefix offsets in
 * DEVICE memory.  Every pointer argument below is a caller-owned CUDA device
 * pointer that the library never frees.  Calls are asynchronous on `stream`:
 * the library never copies cu_seqlens to the host and never synchronises,
 * except when it grows its own workspace (see attn_varlen_fwd).
 *
 * Preconditions the library cannot check without reading device memory:
 * every offset in cu_seqlens_q lies in [0, total_q] and every offset in
 * cu_seqlens_k in [0, total_k], where total_* is the row count of the
 * caller's buffers.  A negative slice length is read as an empty slice.
 */
#ifndef ATTN_VARLEN_H
#define ATTN_VARLEN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define ATTN_VARLEN_OK                     0
#define ATTN_VARLEN_ERR_INVALID_ARG       -1  /* null pointer, negative count, ... */
#define ATTN_VARLEN_ERR_UNSUPPORTED_DIM   -2  /* head_dim not 64, 72, 80, 96, 128  */
#define ATTN_VARLEN_ERR_MISALIGNED        -3  /* q, k, v or out not 16-byte aligned */
#define ATTN_VARLEN_ERR_UNSUPPORTED_DEVICE -4 /* current device is not sm_103       */
#define ATTN_VARLEN_ERR_CUDA              -5  /* a CUDA runtime call failed         */
#define ATTN_VARLEN_ERR_OOM               -6  /* workspace allocation failed        */
#define ATTN_VARLEN_ERR_DEVICE_TIMEOUT    -7  /* a kernel wait ran out of time      */
#define ATTN_VARLEN_ERR_WORKSPACE_SMALL   -8  /* caller workspace below the minimum */
#define ATTN_VARLEN_ERR_DRIVER            -9  /* tensor-map encoder unavailable     */
#define ATTN_VARLEN_ERR_NOALLOC_LIMIT    -10  /* num_seqs above the fixed scratch   */
#define ATTN_VARLEN_ERR_BAD_BLOCK_TABLE  -11  /* paged decode: block id out of range */

/*
 * attn_varlen_fwd -- the attention forward described above.
 *
 *   q, k, v       bf16 device buffers, layout above, 16-byte aligned
 *   cu_seqlens_q  int32 device array [num_seqs + 1]
 *   cu_seqlens_k  int32 device array [num_seqs + 1]
 *   num_seqs      >= 0; 0 returns ATTN_VARLEN_OK without launching anything
 *   num_heads     >= 1 (query, key and value heads are the same count)
 *   head_dim      64, 72, 80, 96 or 128.  The page's shapes use 72 and 128; 72
 *                 runs padded to 80 (zero columns add nothing to Q.K^T), and 64,
 *                 80 and 96 run on the same schedule, always scaled by the true
 *                 head_dim
 *   out           bf16 device buffer [total_q, num_heads, head_dim], 16-byte
 *                 aligned; must not overlap q, k or v
 *   stream        CUDA stream the work is queued on (0 = legacy default)
 *
 * Uses a workspace that the library owns, one per device, sized by num_seqs
 * plus a region of four times the SM count partial slots (about 135 KB each,
 * 82 MB on 152 SMs) in which the units at the end of the schedule may be
 * split along the key range and merged (fp32 partials, merged in a fixed
 * order, so results are deterministic).  Which units are split is planned on
 * the device from the lengths: those that a longest-first list schedule of
 * the persistent grid would finish late.  When the workspace must grow, the
 * call synchronises the device once to free the old one.  Calls that share a
 * device must be ordered (same stream, or
 * synchronised); concurrent calls on different streams must each pass their
 * own workspace to attn_varlen_fwd_ws.  Errors detected inside the kernels
 * (a wait that timed out) are recorded in the workspace and reported by
 * attn_varlen_check.  Returns an ATTN_VARLEN_* code.
 */
int attn_varlen_fwd(const void* q, const void* k, const void* v,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                    int num_seqs, int num_heads, int head_dim,
                    void* out, cudaStream_t stream);

/*
 * attn_varlen_fwd_causal -- attn_varlen_fwd with a causal mask.  The page's
 * operation is non-causal (its scaled_dot_product_attention call passes
 * is_causal=False); this is the common prefill neighbour.  Row r of sequence
 * i (0-based within its query slice) sees only the keys j <= r + L_k - L_q of
 * that sequence: the mask is aligned to the bottom-right corner, so the last
 * query row sees every key (prefill after L_k - L_q cached tokens); for
 * L_q = L_k it is the usual lower triangle.  A row that sees no key (possible
 * only when L_q > L_k) gets a zero row.  Arguments, layout, workspace and
 * errors are those of attn_varlen_fwd; key tiles wholly above a row block's
 * diagonal are skipped, and units are never split along keys.
 */
int attn_varlen_fwd_causal(const void* q, const void* k, const void* v,
                           const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                           int num_seqs, int num_heads, int head_dim,
                           void* out, cudaStream_t stream);

/*
 * attn_varlen_fwd_heads -- heads [head_begin, head_begin + head_count) only.
 *
 * The same operation as attn_varlen_fwd (causal != 0: attn_varlen_fwd_causal)
 * restricted to a contiguous range of heads of the same packed tensors: q, k,
 * v and out are the whole [total, num_heads, head_dim] buffers, read and
 * written in place; out rows of heads outside the range are not touched.
 * Heads are independent in this operation (each head's output depends on its
 * own q, k and v slices only), so G processes (one per GPU, each with a copy
 * of the inputs) can split the heads between them with no exchange, and
 * the output needs gathering only if one process wants it whole.
 *
 *   head_begin, head_count   0 <= head_begin, head_begin + head_count <=
 *                            num_heads; head_count 0 returns ATTN_VARLEN_OK
 *                            without launching anything
 *
 * Other arguments, the workspace and the errors are those of attn_varlen_fwd
 * (ATTN_VARLEN_ERR_INVALID_ARG for a range outside [0, num_heads)).
 */
int attn_varlen_fwd_heads(const void* q, const void* k, const void* v,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                          int num_seqs, int num_heads, int head_begin, int head_count,
                          int head_dim, int causal, void* out, cudaStream_t stream);

/* Bytes of workspace attn_varlen_fwd_ws needs for num_seqs sequences
 * (0 for num_seqs < 0). */
size_t attn_varlen_workspace_size(int num_seqs);

/*
 * attn_varlen_fwd_ws -- attn_varlen_fwd with a caller-owned workspace.
 *
 *   workspace        device buffer, 256-byte aligned, at least
 *                    attn_varlen_workspace_size(num_seqs) bytes, zero-filled
 *                    before its first use (the first 4 bytes are the sticky
 *                    device status word; the rest is rewritten every call)
 *   workspace_bytes  its size in bytes
 *
 * Calls that share one workspace must be ordered on the device.  Nothing is
 * allocated.  Returns an ATTN_VARLEN_* code.
 */
int attn_varlen_fwd_ws(const void* q, const void* k, const void* v,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                       int num_seqs, int num_heads, int head_dim, void* out,
                       void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/*
 * attn_varlen_check -- synchronise `stream`, then read and clear the status
 * word of the current device's library-owned workspace.  Returns
 * ATTN_VARLEN_OK, ATTN_VARLEN_ERR_DEVICE_TIMEOUT when a kernel wait ran out of
 * time since the last check, or ATTN_VARLEN_ERR_CUDA when the stream reports
 * an error.
 */
int attn_varlen_check(cudaStream_t stream);

/* attn_varlen_check for a caller-owned workspace. */
int attn_varlen_check_ws(void* workspace, cudaStream_t stream);

/*
 * attn_varlen_fwd_noalloc -- attn_varlen_fwd without any device allocation.
 *
 * The paper has no counterpart to this call; it exists for callers that
 * cannot allocate device memory when they run attention: a serving process
 * that fixes its whole memory footprint at start-up, a host framework that
 * owns every allocation a plug-in makes, or a latency-critical path where
 * cudaMalloc/cudaFree would synchronise the device.  Instead of the
 * library-owned workspace, it uses one scratch array compiled into the
 * library (about 1033 KiB, held on every GPU that loads the library until
 * the process exits), so it supports at most
 * ATTN_VARLEN_NOALLOC_MAX_SEQS sequences per call and returns
 * ATTN_VARLEN_ERR_NOALLOC_LIMIT above that.  Arguments, layout and results
 * are those of attn_varlen_fwd; the call never calls cudaMalloc, cudaFree
 * or any allocating routine.
 *
 * The first call on a device looks up the scratch array's device address
 * (once, with that device current); make that first call before any stream
 * capture.  Every call on a device shares the one array: calls that can
 * overlap on the GPU (different streams without ordering) race and give
 * wrong results, so order them.  The array's first word is this variant's
 * device status word: zero when the library loads, set by a kernel wait that
 * timed out, kept across calls, and read and cleared only by
 * attn_varlen_check_noalloc (attn_varlen_check reads the library-owned
 * workspace instead).
 */
#define ATTN_VARLEN_NOALLOC_MAX_SEQS 1024
int attn_varlen_fwd_noalloc(const void* q, const void* k, const void* v,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int num_seqs, int num_heads, int head_dim, void* out,
                            cudaStream_t stream);

/*
 * attn_varlen_check_noalloc -- attn_varlen_check for the fixed scratch of
 * attn_varlen_fwd_noalloc: synchronise `stream`, then read and clear that
 * scratch's status word on the current device.  Returns ATTN_VARLEN_OK (also
 * when attn_varlen_fwd_noalloc never ran on this device),
 * ATTN_VARLEN_ERR_DEVICE_TIMEOUT when a kernel wait of a no-alloc call ran out
 * of time since the last check, or ATTN_VARLEN_ERR_CUDA.  Allocates nothing.
 */
int attn_varlen_check_noalloc(cudaStream_t stream);

/* Static, human-readable text for an ATTN_VARLEN_* code. */
const char* attn_varlen_strerror(int code);

/* Text of the last CUDA runtime error behind an ATTN_VARLEN_ERR_CUDA return
 * on the calling thread ("no CUDA error" if none).  Static storage. */
const char* attn_varlen_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int attn_varlen_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_VARLEN_H */
