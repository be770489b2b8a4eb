// Launch parameters of the paged single-query decode kernel (paged_decode.cu),
// filled by the C ABI in attn_varlen_api.cu.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace avp {

// Status word bit (shared with the attention kernels' word): a block table
// entry outside [0, num_blocks) was met; that block was not read.
constexpr int kPagedStatusBadBlock = 16;

struct PagedParams {
  const void* query;          // [num_seqs, Hq, D]
  const void* k_cache;        // [num_blocks, Hkv, D/8, 16, 8]
  const void* v_cache;        // [num_blocks, Hkv, D, 16]
  const int32_t* block_tables;  // [num_seqs, max_blocks]
  const int32_t* seq_lens;      // [num_seqs]
  void* out;                  // [num_seqs, Hq, D]
  int* status;
  int num_seqs;
  int num_query_heads;
  int num_kv_heads;
  int qpk;                    // query heads per KV head
  int head_size;
  int max_blocks;
  int num_blocks;
  int sm_count;               // SMs of the device (sizes the head group)
  float scale_log2;           // head_size^-1/2 * log2(e)
};

bool paged_head_size_supported(int head_size);  // 64, 128, 256
cudaError_t launch_paged_decode(const PagedParams& p, bool fp16, cudaStream_t stream);

}  // namespace avp
