// Single-query paged attention decode for sm_103a.
//
// What is computed: atrex-bench "paged_attention_decode" (page #024,
// reference.py, Model.forward).  Sequence i has one query row per query head
// and ctx_len = seq_lens[i] context tokens; token t is at position t % 16 of
// physical block block_tables[i][t / 16] of a split-x key cache
// [num_blocks, Hkv, D/8, 16, 8] and a transposed value cache
// [num_blocks, Hkv, D, 16].  Query head h reads KV head h / (Hq / Hkv).  The
// output row is softmax(q . K^T * D^-1/2) V over the context; a sequence with
// ctx_len <= 0 gets a zero row.
//
// The operation is a gather-GEMV: every context byte is read once and each
// (block, KV head) holds 4 KB of contiguous K (D = 128) and 4 KB of V, so the
// kernel is bound by HBM (or, for the page's small shapes, by latency).  It
// uses plain coalesced 16-byte loads, no tensor cores:
//   CTA  = (sequence, KV head, group of up to MQ query heads), 4 warps, MQ
//          the power of two (at most 8) that covers the query heads per KV
//          head, so registers scale with the group;
//   warp = every 4th block of the context, an exp2 online softmax per head;
//   keys:   lane = (token 0-15, half of the head dimension): 16-byte chunks
//           [c][token][8] of one half are 256 contiguous bytes per warp load,
//           the two halves' partial dot products meet by one shuffle;
//   values: lane = D/32 consecutive dimensions, each a 32-byte row of the
//           block's 16 tokens;
//   the four warps' (m, l, O) merge through shared memory at the end.
// A block's value rows are loaded together with its key chunks, and each
// warp reads its next block-table entry before working on the current block,
// so a block costs one dependent memory round trip.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "paged_decode_internal.h"

namespace avp {
namespace {

constexpr int kWarps = 4;
constexpr int kBlock = 16;   // tokens per cache block
constexpr int kMaxQ = 8;     // query heads per CTA at most

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

// 8 consecutive elements of a 16-byte chunk -> fp32
template <typename T>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = to_f32<T>(e[i]);
}

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, typename T, int MQ>
__global__ void __launch_bounds__(32 * kWarps) paged_decode_kernel(const __grid_constant__ PagedParams p) {
  constexpr int NCH = D / 8;        // 16-byte chunks of a key row
  constexpr int HCH = NCH / 2;      // chunks per lane (one half of the row)
  constexpr int DPL = D / 32;       // value dimensions per lane
  // query row: the second half of the dimensions sits 4 floats further on, so
  // the two half-warps' broadcast reads fall in different banks
  constexpr int QROW = D + 4;
  __shared__ __align__(16) float s_q[MQ][QROW];   // scaled queries
  __shared__ float s_p[kWarps][MQ][kBlock];       // one block's weights per warp
  __shared__ float s_m[kWarps][MQ], s_l[kWarps][MQ];
  __shared__ float s_o[kWarps][MQ][D];

  const int ngroups = (p.qpk + MQ - 1) / MQ;
  const int seq = blockIdx.x / (p.num_kv_heads * ngroups);
  const int rem = blockIdx.x - seq * p.num_kv_heads * ngroups;
  const int g = rem / ngroups;
  const int h0 = g * p.qpk + (rem - g * ngroups) * MQ;   // first query head of the CTA
  const int nq = min(MQ, g * p.qpk + p.qpk - h0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* q = static_cast<const T*>(p.query) + ((size_t)seq * p.num_query_heads + h0) * D;
  T* out = static_cast<T*>(p.out) + ((size_t)seq * p.num_query_heads + h0) * D;

  int L = p.seq_lens[seq];
  if (L > p.max_blocks * kBlock) L = p.max_blocks * kBlock;  // the table holds no more
  if (L <= 0) {
    for (int i = threadIdx.x; i < nq * D; i += blockDim.x) out[i] = from_f32<T>(0.f);
    return;
  }
  const int tok = lane & 15, half = lane >> 4;
  const int nblk = (L + kBlock - 1) / kBlock;
  const int32_t* table = p.block_tables + (size_t)seq * p.max_blocks;
  // One block's keys (this lane's token, half of the dimensions) and values
  // (this lane's dimensions, 16 tokens) in registers.  A block id outside
  // [0, num_blocks) is never dereferenced: it is reported and skipped.
  uint4 kc[HCH], vc[2 * DPL];
  auto load_block = [&](int b) -> bool {
    if (b < 0 || b >= p.num_blocks) {
      if (lane == 0) atomicOr(p.status, kPagedStatusBadBlock);
      return false;
    }
    const uint4* kb = reinterpret_cast<const uint4*>(static_cast<const T*>(p.k_cache) +
                                                     ((size_t)b * p.num_kv_heads + g) * D * kBlock);
#pragma unroll
    for (int c = 0; c < HCH; ++c) kc[c] = __ldg(kb + (half * HCH + c) * kBlock + tok);
    const T* vb = static_cast<const T*>(p.v_cache) + ((size_t)b * p.num_kv_heads + g) * D * kBlock +
                  (size_t)lane * DPL * kBlock;
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      vc[2 * e] = __ldg(reinterpret_cast<const uint4*>(vb + e * kBlock));
      vc[2 * e + 1] = __ldg(reinterpret_cast<const uint4*>(vb + e * kBlock) + 1);
    }
    return true;
  };
  // The warp's first block is read before the query is staged, so its memory
  // round trip overlaps the query's; later blocks are read one iteration
  // ahead of their use, their ids one further.
  bool have = warp < nblk ? load_block(__ldg(table + warp)) : false;
  int b_next = warp + kWarps < nblk ? __ldg(table + warp + kWarps) : 0;
  for (int i = threadIdx.x; i < MQ * D; i += blockDim.x) {
    const int hh = i / D, d = i % D;
    s_q[hh][d + (d >= D / 2 ? 4 : 0)] = hh < nq ? to_f32<T>(q[i]) * p.scale_log2 : 0.f;
  }
  __syncthreads();

  float m[MQ], l[MQ], o[MQ][DPL];
#pragma unroll
  for (int hh = 0; hh < MQ; ++hh) {
    m[hh] = -INFINITY;
    l[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[hh][e] = 0.f;
  }
  for (int jb = warp; jb < nblk; jb += kWarps) {
    if (!have) {  // this block's id was bad: fetch the next one and go on
      if (jb + kWarps < nblk) {
        have = load_block(b_next);
        if (jb + 2 * kWarps < nblk) b_next = __ldg(table + jb + 2 * kWarps);
      }
      continue;
    }
    // scores of this lane's token for every query head (half the dimensions)
    float acc[MQ];
#pragma unroll
    for (int hh = 0; hh < MQ; ++hh) acc[hh] = 0.f;
#pragma unroll
    for (int c = 0; c < HCH; ++c) {
      float kf[8];
      unpack8<T>(kc[c], kf);
      const int d0 = (half * HCH + c) * 8 + half * 4;  // padded query row
#pragma unroll
      for (int hh = 0; hh < MQ; ++hh) {
        if (hh < nq) {
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[hh] = fmaf(s_q[hh][d0 + e], kf[e], acc[hh]);
        }
      }
    }
    const bool live = jb * kBlock + tok < L;
#pragma unroll
    for (int hh = 0; hh < MQ; ++hh) {
      if (hh >= nq) continue;
      float sc = acc[hh] + __shfl_xor_sync(0xffffffffu, acc[hh], 16);
      sc = live ? sc : -INFINITY;
      float bm = sc;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
      const float mn = fmaxf(m[hh], bm);  // finite: every block holds a live token
      const float alpha = fast_ex2(m[hh] - mn);
      const float pw = fast_ex2(sc - mn);
      float bs = pw;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) bs += __shfl_xor_sync(0xffffffffu, bs, off);
      l[hh] = l[hh] * alpha + bs;
      m[hh] = mn;
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[hh][e] *= alpha;
      if (half == 0) s_p[warp][hh][tok] = pw;
    }
    __syncwarp();
    // values: this lane's DPL dimensions, 16 tokens each
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      float v0[8], v1[8];
      unpack8<T>(vc[2 * e], v0);
      unpack8<T>(vc[2 * e + 1], v1);
#pragma unroll
      for (int hh = 0; hh < MQ; ++hh) {
        if (hh >= nq) continue;
        float a = o[hh][e];
#pragma unroll
        for (int t = 0; t < 8; ++t) a = fmaf(s_p[warp][hh][t], v0[t], a);
#pragma unroll
        for (int t = 0; t < 8; ++t) a = fmaf(s_p[warp][hh][8 + t], v1[t], a);
        o[hh][e] = a;
      }
    }
    __syncwarp();
    // the warp's next block: its keys and values into the same registers
    have = false;
    if (jb + kWarps < nblk) {
      have = load_block(b_next);
      if (jb + 2 * kWarps < nblk) b_next = __ldg(table + jb + 2 * kWarps);
    }
  }

  // merge the warps: O = sum_w 2^(m_w - m*) O_w, l likewise
  if (lane == 0) {
#pragma unroll
    for (int hh = 0; hh < MQ; ++hh) {
      s_m[warp][hh] = m[hh];
      s_l[warp][hh] = l[hh];
    }
  }
#pragma unroll
  for (int hh = 0; hh < MQ; ++hh)
#pragma unroll
    for (int e = 0; e < DPL; ++e) s_o[warp][hh][lane * DPL + e] = o[hh][e];
  __syncthreads();
  for (int i = threadIdx.x; i < nq * D; i += blockDim.x) {
    const int hh = i / D, d = i % D;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, s_m[w][hh]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      if (s_m[w][hh] == -INFINITY) continue;  // a warp that saw no block
      const float f = fast_ex2(s_m[w][hh] - mm);
      num += f * s_o[w][hh][d];
      den += f * s_l[w][hh];
    }
    out[i] = from_f32<T>(den > 0.f ? num / den : 0.f);
  }
}

template <int D, typename T, int MQ>
cudaError_t launch_mq(const PagedParams& p, cudaStream_t stream) {
  const int ngroups = (p.qpk + MQ - 1) / MQ;
  const long long grid = (long long)p.num_seqs * p.num_kv_heads * ngroups;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  paged_decode_kernel<D, T, MQ><<<(unsigned)grid, 32 * kWarps, 0, stream>>>(p);
  return cudaGetLastError();
}

// The head group is the smallest power of two (at most kMaxQ) covering the
// query heads of one KV head, halved while the grid would not fill the SMs:
// a smaller group gives more CTAs (each KV block is then read by several,
// mostly from L2) and shorter per-block work for the few that run.
template <int D, typename T>
cudaError_t launch_t(const PagedParams& p, cudaStream_t stream) {
  int mq = p.qpk <= 1 ? 1 : (p.qpk <= 2 ? 2 : (p.qpk <= 4 ? 4 : kMaxQ));
  const long long pairs = (long long)p.num_seqs * p.num_kv_heads;
  while (mq > 1 && pairs * ((p.qpk + mq - 1) / mq) < p.sm_count) mq >>= 1;
  if (mq == 1) return launch_mq<D, T, 1>(p, stream);
  if (mq == 2) return launch_mq<D, T, 2>(p, stream);
  if (mq == 4) return launch_mq<D, T, 4>(p, stream);
  return launch_mq<D, T, kMaxQ>(p, stream);
}

}  // namespace

bool paged_head_size_supported(int head_size) {
  return head_size == 64 || head_size == 128 || head_size == 256;
}

cudaError_t launch_paged_decode(const PagedParams& p, bool fp16, cudaStream_t stream) {
  switch (p.head_size) {
    case 64: return fp16 ? launch_t<64, __half>(p, stream) : launch_t<64, __nv_bfloat16>(p, stream);
    case 128: return fp16 ? launch_t<128, __half>(p, stream) : launch_t<128, __nv_bfloat16>(p, stream);
    case 256: return fp16 ? launch_t<256, __half>(p, stream) : launch_t<256, __nv_bfloat16>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace avp
