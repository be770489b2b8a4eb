// Launch parameters of the chunked gated delta-rule output kernel
// (chunk_o.cu), filled by the C ABI in attn_varlen_api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>

#include "attn_varlen_internal.h"

namespace avp {

struct ChunkParams {
  const void* q;    // bf16 [batch, tokens, num_q_heads, 128]
  const void* k;    // bf16 [batch, tokens, num_q_heads, 128]
  const void* v;    // bf16 [batch, tokens, num_v_heads, 128]
  const void* h;    // bf16 [batch, chunks, num_v_heads, 128, 128]
  const float* g;   // f32 [batch, tokens, num_v_heads]
  void* out;        // bf16 [batch, tokens, num_v_heads, 128]
  int* status;      // device status word: timeout bits
  int batch;
  int tokens;
  int num_q_heads;
  int num_v_heads;
  int sm_count;     // persistent grid size bound
  float scale;
};

// Status bit a chunk-output wait that gave up sets.
constexpr int kChunkStatusTimeout = 32;

size_t chunk_o_smem_bytes();
// Opts the kernel into its dynamic shared memory on the current device; once
// per device before the first launch there.
cudaError_t prepare_chunk_o();
// Encodes the kernel's tensor maps with `enc` and launches on the current
// device.  Returns a CUDA error, or cudaErrorInvalidValue when a map cannot
// be encoded.
cudaError_t launch_chunk_o(const ChunkParams& p, EncodeTiledFn enc, cudaStream_t stream);

}  // namespace avp
