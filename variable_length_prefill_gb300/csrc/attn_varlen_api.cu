// C ABI of the packed variable-length attention forward (declared in
// include/attn_varlen.h): argument checks, the per-device workspace, the
// tensor-map templates and the two launches.  No step of the computation runs
// on the host; cu_seqlens stay on the device.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn_varlen.h"
#include "attn_varlen_internal.h"
#include "chunk_delta_rule.h"
#include "chunk_o_internal.h"
#include "paged_attn_decode.h"
#include "paged_decode_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// The tensor-map templates of the last call on a device: encoding them is
// pure host work that depends only on the buffers and the shape, so a call
// with the same q, k, v, num_heads and head_dim reuses them.
struct TemplateCache {
  const void* bases[avp::kTensors] = {nullptr, nullptr, nullptr, nullptr};
  int num_heads = 0;
  int head_dim = 0;
  CUtensorMap tmpl[2][avp::kMapsPerSeq];
};

struct DeviceState {
  TemplateCache tc;
  bool probed = false;
  bool supported = false;
  bool prepared[129] = {};  // kernel attributes set, by head_dim
  bool chunk_prepared = false;  // the chunk-output kernel's attribute set
  int sm_count = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Fixed scratch of attn_varlen_fwd_noalloc: the workspace of
// ATTN_VARLEN_NOALLOC_MAX_SEQS sequences.  In host code the name stands for
// the symbol, not a device address; each device's address comes from
// cudaGetSymbolAddress (g_noalloc_ptr).
constexpr size_t kNoAllocBytes = avp::ws_layout(ATTN_VARLEN_NOALLOC_MAX_SEQS).total;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];
void* g_noalloc_ptr[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_probed = false;

// Last CUDA runtime error this library saw on the calling thread.
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

#ifndef ATTN_VARLEN_TEST_HOOKS
#define ATTN_VARLEN_TEST_HOOKS 0
#endif
// Set only through the test build's attn_varlen_test_withhold (FwdParams).
int g_test_withhold = 0;

int fail_cuda(cudaError_t e) {
  g_last_cuda_error = e;
  cudaGetLastError();  // do not leave the error pending for the caller
  return ATTN_VARLEN_ERR_CUDA;
}

int map_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_VARLEN_OK : fail_cuda(e); }

// Called with g_mu held.
int probe_device(int dev, DeviceState& st) {
  if (st.probed) return st.supported ? ATTN_VARLEN_OK : ATTN_VARLEN_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0, sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail_cuda(e);
  st.probed = true;
  st.supported = (major == 10 && minor == 3);
  st.sm_count = sms;
  return st.supported ? ATTN_VARLEN_OK : ATTN_VARLEN_ERR_UNSUPPORTED_DEVICE;
}

// Called with g_mu held.
int get_encoder() {
  if (!g_encode_probed) {
    g_encode_probed = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode ? ATTN_VARLEN_OK : ATTN_VARLEN_ERR_DRIVER;
}

int check_args(const void* q, const void* k, const void* v, const int32_t* cu_q,
               const int32_t* cu_k, int num_seqs, int num_heads, int head_dim, const void* out) {
  if (num_seqs < 0 || num_heads < 1) return ATTN_VARLEN_ERR_INVALID_ARG;
  if (!avp::head_dim_supported(head_dim)) return ATTN_VARLEN_ERR_UNSUPPORTED_DIM;
  if (num_seqs == 0) return ATTN_VARLEN_OK;
  if (!q || !k || !v || !cu_q || !cu_k || !out) return ATTN_VARLEN_ERR_INVALID_ARG;
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) &
                        15u;
  if (mis) return ATTN_VARLEN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(cu_q) | reinterpret_cast<uintptr_t>(cu_k)) & 3u)
    return ATTN_VARLEN_ERR_MISALIGNED;
  // token stride must fit the tensor-map stride field (< 2^40 bytes)
  if ((uint64_t)num_heads * (uint64_t)head_dim * 2u >= (1ull << 40)) return ATTN_VARLEN_ERR_INVALID_ARG;
  return ATTN_VARLEN_OK;
}

}  // namespace

namespace avp {

int encode_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, int num_heads, int head_dim,
               uint64_t rows, int box_rows, int box_cols, bool swizzle_128) {
  cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_heads * head_dim * 2};
  cuuint32_t boxdim[3] = {(cuuint32_t)box_cols, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz =
      swizzle_128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  return (int)enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  boxdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Templates: a 3-D bf16 map {head_dim, num_heads, rows} with box {cols, 1,
// rows per tile} (128 query rows for q, kv_tile_rows keys for k and v,
// kStoreRows output rows for out), one for box A (columns [0, 64)) and one
// for box B (the columns past 64); the plan kernel patches the address and
// the row extent per sequence.
// Class 0 is encoded one row short of kMapLargeBytes, class 1 at it.
int encode_templates(EncodeTiledFn enc, PlanParams& pp, const void* const bases[kTensors],
                     int num_heads, int head_dim) {
  const uint64_t row_bytes = (uint64_t)num_heads * head_dim * 2;
  const uint64_t large_rows = (kMapLargeBytes + row_bytes - 1) / row_bytes;
  const uint64_t small_rows = large_rows > 1 ? large_rows - 1 : 1;
  for (int m = 0; m < kMapsPerSeq; ++m) {
    const int t = m % kTensors;
    const bool b = m >= kTensors;
    const int box_rows = t == 0 ? kBlockM : (t == kOut ? kStoreRows : kv_tile_rows(head_dim));
    const int cols = b ? box_b_cols(head_dim) : box_cols(head_dim);
    const bool swz = b ? box_b_swizzle_128(head_dim) : true;
    for (int cls = 0; cls < 2; ++cls) {
      const int r = encode_map(enc, &pp.tmpl[cls][m], bases[t], num_heads, head_dim,
                               cls ? large_rows : small_rows, box_rows, cols, swz);
      if (r) return r;
    }
  }
  return 0;
}

}  // namespace avp

namespace {

// `split_cap` > 0 (library-owned workspace only): the tail-split region for
// that many items is the last split_layout(split_cap).total bytes of the
// allocation, so it stays in one place, whatever num_seqs, until the
// workspace is reallocated (its row counters persist from call to call).  Heads [head_begin,
// head_begin + head_count) of the num_heads-head tensors are computed
// (head_count < 0: all of them).
int run(const void* q, const void* k, const void* v, const int32_t* cu_q, const int32_t* cu_k,
        int num_seqs, int num_heads, int head_dim, void* out, void* ws, int split_cap, int dev,
        DeviceState& st, cudaStream_t stream, bool causal = false, int head_begin = 0,
        int head_count = -1) {
  if (head_count < 0) head_count = num_heads;
  avp::PlanParams pp;
  std::memset(&pp, 0, sizeof(pp));
  const void* bases[avp::kTensors] = {q, k, v, out};
  TemplateCache& tc = st.tc;
  static_assert(sizeof(tc.tmpl) == sizeof(pp.tmpl), "template cache");
  if (tc.bases[0] == q && tc.bases[1] == k && tc.bases[2] == v && tc.bases[3] == out &&
      tc.num_heads == num_heads && tc.head_dim == head_dim) {
    std::memcpy(pp.tmpl, tc.tmpl, sizeof(pp.tmpl));
  } else {
    if (avp::encode_templates(reinterpret_cast<avp::EncodeTiledFn>(g_encode), pp, bases,
                              num_heads, head_dim) != 0)
      return ATTN_VARLEN_ERR_DRIVER;
    std::memcpy(tc.tmpl, pp.tmpl, sizeof(pp.tmpl));
    tc.bases[0] = q;
    tc.bases[1] = k;
    tc.bases[2] = v;
    tc.bases[3] = out;
    tc.num_heads = num_heads;
    tc.head_dim = head_dim;
  }
  for (int m = 0; m < avp::kTensors; ++m) pp.base[m] = static_cast<const uint8_t*>(bases[m]);
  pp.cu_q = cu_q;
  pp.cu_k = cu_k;
  pp.ws = static_cast<uint8_t*>(ws);
  uint8_t* split = split_cap > 0 ? static_cast<uint8_t*>(st.ws) + st.ws_bytes -
                                       avp::split_layout(split_cap).total
                                 : nullptr;
  pp.split = split;
  pp.split_cap = split_cap;
  pp.grid = st.sm_count;
  pp.kv_rows = avp::kv_tile_rows(head_dim);
  pp.causal = causal ? 1 : 0;
  pp.num_seqs = num_seqs;
  pp.num_heads = head_count;
  pp.row_bytes = num_heads * head_dim * 2;

  avp::FwdParams fp;
  fp.ws = static_cast<const uint8_t*>(ws);
  fp.split = split;
  fp.split_cap = split_cap;
  fp.status = static_cast<int*>(ws);
  fp.cu_q = cu_q;
  fp.cu_k = cu_k;
  fp.out = static_cast<uint16_t*>(out);
  fp.num_seqs = num_seqs;
  fp.num_heads = num_heads;
  fp.head_begin = head_begin;
  fp.causal = causal ? 1 : 0;
  fp.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)head_dim));
  fp.test_withhold = g_test_withhold;

  const int slot = head_dim;
  if (!st.prepared[slot]) {
    cudaError_t pe = avp::prepare_fwd(head_dim);
    if (pe != cudaSuccess) return fail_cuda(pe);
    st.prepared[slot] = true;
  }
  (void)dev;
  cudaError_t e = avp::launch_plan(pp, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  e = avp::launch_fwd(head_dim, fp, st.sm_count, stream);
  return map_cuda(e);
}

// Grow the library-owned workspace of `dev` (g_mu held).  Keeps the status
// word across the reallocation.
int ensure_workspace(DeviceState& st, size_t need) {
  if (st.ws && st.ws_bytes >= need) return ATTN_VARLEN_OK;
  size_t bytes = need < (1u << 16) ? (1u << 16) : need + need / 2;
  bytes = (bytes + 255) & ~(size_t)255;
  int status = 0;
  if (st.ws) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&status, st.ws, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(e);
    cudaFree(st.ws);
    st.ws = nullptr;
    st.ws_bytes = 0;
  }
  void* p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_VARLEN_ERR_OOM;
  }
  // header: the carried status word, and the split region's row counters
  // marked dirty (the first plan zeroes them)
  int hdr[avp::kHdrCountersDirty + 1] = {};
  hdr[0] = status;
  hdr[avp::kHdrCountersDirty] = 1;
  cudaError_t e = cudaMemset(p, 0, 256);
  if (e == cudaSuccess) e = cudaMemcpy(p, hdr, sizeof(hdr), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(p);
    return fail_cuda(e);
  }
  st.ws = p;
  st.ws_bytes = bytes;
  return ATTN_VARLEN_OK;
}

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (*dev < 0 || *dev >= kMaxDevices) return ATTN_VARLEN_ERR_UNSUPPORTED_DEVICE;
  return ATTN_VARLEN_OK;
}

int read_and_clear_status(void* ws, cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  int status = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&status, ws, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  if (status != 0) {
    const int zero = 0;
    e = cudaMemcpy(ws, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda(e);
    if (status == avp::kPagedStatusBadBlock) return ATTN_VARLEN_ERR_BAD_BLOCK_TABLE;
    return ATTN_VARLEN_ERR_DEVICE_TIMEOUT;
  }
  return ATTN_VARLEN_OK;
}

}  // namespace

extern "C" {

size_t attn_varlen_workspace_size(int num_seqs) {
  if (num_seqs < 0) return 0;
  return avp::ws_layout(num_seqs).total;
}

static int fwd_owned(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                     const int32_t* cu_seqlens_k, int num_seqs, int num_heads, int head_dim,
                     void* out, cudaStream_t stream, bool causal, int head_begin = 0,
                     int head_count = -1) {
  int rc = check_args(q, k, v, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, out);
  if (rc || num_seqs == 0 || head_count == 0) return rc;
  int dev = 0;
  if ((rc = current_device(&dev))) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if ((rc = probe_device(dev, st))) return rc;
  if ((rc = get_encoder())) return rc;
  // the library-owned workspace also holds the tail-split region
  // (kSplitWaves items per CTA of the persistent grid)
  const int cap = avp::tail_split_supported(head_dim) ? avp::kSplitWaves * st.sm_count : 0;
  if ((rc = ensure_workspace(st, avp::ws_layout(num_seqs).total + avp::split_layout(cap).total)))
    return rc;
  return run(q, k, v, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, out, st.ws, cap,
             dev, st, stream, causal, head_begin, head_count);
}

int attn_varlen_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                    const int32_t* cu_seqlens_k, int num_seqs, int num_heads, int head_dim,
                    void* out, cudaStream_t stream) {
  return fwd_owned(q, k, v, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, out, stream,
                   false);
}

int attn_varlen_fwd_causal(const void* q, const void* k, const void* v,
                           const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int num_seqs,
                           int num_heads, int head_dim, void* out, cudaStream_t stream) {
  return fwd_owned(q, k, v, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, out, stream,
                   true);
}

int attn_varlen_fwd_heads(const void* q, const void* k, const void* v,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int num_seqs,
                          int num_heads, int head_begin, int head_count, int head_dim, int causal,
                          void* out, cudaStream_t stream) {
  if (num_heads < 1 || head_begin < 0 || head_count < 0 || head_begin > num_heads ||
      head_count > num_heads - head_begin)
    return ATTN_VARLEN_ERR_INVALID_ARG;
  return fwd_owned(q, k, v, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, out, stream,
                   causal != 0, head_begin, head_count);
}

int attn_varlen_fwd_ws(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                       const int32_t* cu_seqlens_k, int num_seqs, int num_heads, int head_dim,
                       void* out, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_args(q, k, v, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, out);
  if (rc || num_seqs == 0) return rc;
  if (!workspace) return ATTN_VARLEN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_VARLEN_ERR_MISALIGNED;
  if (workspace_bytes < avp::ws_layout(num_seqs).total) return ATTN_VARLEN_ERR_WORKSPACE_SMALL;
  int dev = 0;
  if ((rc = current_device(&dev))) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if ((rc = probe_device(dev, st))) return rc;
  if ((rc = get_encoder())) return rc;
  return run(q, k, v, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, out, workspace,
             0, dev, st, stream);
}

int attn_varlen_fwd_noalloc(const void* q, const void* k, const void* v,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int num_seqs, int num_heads, int head_dim, void* out,
                            cudaStream_t stream) {
  int rc = check_args(q, k, v, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, out);
  if (rc || num_seqs == 0) return rc;
  if (num_seqs > ATTN_VARLEN_NOALLOC_MAX_SEQS) return ATTN_VARLEN_ERR_NOALLOC_LIMIT;
  int dev = 0;
  if ((rc = current_device(&dev))) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if ((rc = probe_device(dev, st))) return rc;
  if ((rc = get_encoder())) return rc;
  if (!g_noalloc_ptr[dev]) {
    // once per device, with `dev` current: the device address of the scratch
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e);
    if (!ptr) return ATTN_VARLEN_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  // The plan kernel rewrites everything the attention kernel reads.  The
  // status word (zero when the module loads) is left alone: it is sticky
  // until attn_varlen_check_noalloc reads and clears it.
  void* ws = g_noalloc_ptr[dev];
  return run(q, k, v, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, out, ws, 0, dev,
             st, stream);
}

int paged_attn_decode(const void* query, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                      int num_query_heads, int num_kv_heads, int head_size, int block_size,
                      int max_blocks_per_seq, int num_blocks, int dtype, void* out,
                      cudaStream_t stream) {
  if (num_seqs < 0 || num_query_heads < 1 || num_kv_heads < 1 ||
      num_query_heads % num_kv_heads != 0)
    return ATTN_VARLEN_ERR_INVALID_ARG;
  if (dtype != PAGED_ATTN_BF16 && dtype != PAGED_ATTN_FP16) return ATTN_VARLEN_ERR_INVALID_ARG;
  if (!avp::paged_head_size_supported(head_size)) return ATTN_VARLEN_ERR_UNSUPPORTED_DIM;
  if (block_size != 16) return ATTN_VARLEN_ERR_INVALID_ARG;
  if (num_seqs == 0) return ATTN_VARLEN_OK;
  if (max_blocks_per_seq < 1 || num_blocks < 1) return ATTN_VARLEN_ERR_INVALID_ARG;
  if (!query || !k_cache || !v_cache || !block_tables || !seq_lens || !out)
    return ATTN_VARLEN_ERR_INVALID_ARG;
  auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  auto a4 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; };
  if (!a16(query) || !a16(k_cache) || !a16(v_cache) || !a16(out) || !a4(block_tables) ||
      !a4(seq_lens))
    return ATTN_VARLEN_ERR_MISALIGNED;
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if ((rc = probe_device(dev, st))) return rc;
  if ((rc = ensure_workspace(st, 256))) return rc;  // the status word
  avp::PagedParams p;
  p.query = query;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.out = out;
  p.status = static_cast<int*>(st.ws);
  p.num_seqs = num_seqs;
  p.num_query_heads = num_query_heads;
  p.num_kv_heads = num_kv_heads;
  p.qpk = num_query_heads / num_kv_heads;
  p.head_size = head_size;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.sm_count = st.sm_count;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)head_size));
  return map_cuda(avp::launch_paged_decode(p, dtype == PAGED_ATTN_FP16, stream));
}

int chunk_delta_rule_output(const void* q, const void* k, const void* v, const void* h,
                            const float* g, int batch, int tokens, int num_q_heads,
                            int num_v_heads, int key_dim, int value_dim, int chunk_size,
                            float scale, void* out, cudaStream_t stream) {
  if (batch < 0 || tokens < 0 || num_q_heads < 1 || num_v_heads < 1)
    return ATTN_VARLEN_ERR_INVALID_ARG;
  if (key_dim != 128 || value_dim != 128) return ATTN_VARLEN_ERR_UNSUPPORTED_DIM;
  if (chunk_size != 64) return ATTN_VARLEN_ERR_INVALID_ARG;
  if (batch == 0 || tokens == 0) return ATTN_VARLEN_OK;
  if (!q || !k || !v || !h || !g || !out) return ATTN_VARLEN_ERR_INVALID_ARG;
  auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  if (!a16(q) || !a16(k) || !a16(v) || !a16(h) || !a16(out) ||
      (reinterpret_cast<uintptr_t>(g) & 3u))
    return ATTN_VARLEN_ERR_MISALIGNED;
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if ((rc = probe_device(dev, st))) return rc;
  if ((rc = get_encoder())) return rc;
  if ((rc = ensure_workspace(st, 256))) return rc;  // the status word
  avp::ChunkParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.h = h;
  p.g = g;
  p.out = out;
  p.batch = batch;
  p.tokens = tokens;
  p.num_q_heads = num_q_heads;
  p.num_v_heads = num_v_heads;
  if (!st.chunk_prepared) {
    if ((rc = map_cuda(avp::prepare_chunk_o()))) return rc;
    st.chunk_prepared = true;
  }
  p.status = static_cast<int*>(st.ws);
  p.sm_count = st.sm_count;
  p.scale = scale > 0.f ? scale : (float)(1.0 / std::sqrt((double)key_dim));
  return map_cuda(avp::launch_chunk_o(p, g_encode, stream));
}

int attn_varlen_check(cudaStream_t stream) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ws = g_dev[dev].ws;
  }
  if (!ws) return map_cuda(cudaStreamSynchronize(stream));
  return read_and_clear_status(ws, stream);
}

int attn_varlen_check_ws(void* workspace, cudaStream_t stream) {
  if (!workspace) return ATTN_VARLEN_ERR_INVALID_ARG;
  return read_and_clear_status(workspace, stream);
}

int attn_varlen_check_noalloc(cudaStream_t stream) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ws = g_noalloc_ptr[dev];
  }
  if (!ws) return map_cuda(cudaStreamSynchronize(stream));
  return read_and_clear_status(ws, stream);
}

#if ATTN_VARLEN_TEST_HOOKS
// Test builds only: make the next calls withhold one K/V tile (see
// ATTN_VARLEN_TEST_HOOKS in attn_varlen_kernels.cu) so a bounded wait runs out.
void attn_varlen_test_withhold(int on) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_test_withhold = on ? 1 : 0;
}
#endif

const char* attn_varlen_strerror(int code) {
  switch (code) {
    case ATTN_VARLEN_OK: return "ok";
    case ATTN_VARLEN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_VARLEN_ERR_UNSUPPORTED_DIM: return "head_dim must be 64, 72, 80, 96, 128 or 256";
    case ATTN_VARLEN_ERR_MISALIGNED: return "q, k, v and out must be 16-byte aligned (cu_seqlens 4-byte)";
    case ATTN_VARLEN_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103 (GB300)";
    case ATTN_VARLEN_ERR_CUDA: return "CUDA runtime error";
    case ATTN_VARLEN_ERR_OOM: return "workspace allocation failed";
    case ATTN_VARLEN_ERR_DEVICE_TIMEOUT: return "a kernel wait ran out of time";
    case ATTN_VARLEN_ERR_WORKSPACE_SMALL: return "workspace smaller than attn_varlen_workspace_size()";
    case ATTN_VARLEN_ERR_DRIVER: return "cuTensorMapEncodeTiled unavailable or failed";
    case ATTN_VARLEN_ERR_BAD_BLOCK_TABLE:
      return "paged decode: a block table entry was outside [0, num_blocks)";
    case ATTN_VARLEN_ERR_NOALLOC_LIMIT:
      return "num_seqs exceeds ATTN_VARLEN_NOALLOC_MAX_SEQS (1024), the fixed scratch of "
             "attn_varlen_fwd_noalloc";
    default: return "unknown error code";
  }
}

int attn_varlen_version(void) { return 100; }

const char* attn_varlen_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(g_last_cuda_error);
}

}  // extern "C"
