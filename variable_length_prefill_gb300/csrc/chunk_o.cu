// Chunked gated delta-rule output for sm_103a.
//
// What is computed: atrex-bench "chunk_delta_rule_output" (page #004,
// reference.py, Model.forward).  Tokens are cut into chunks of 64; for chunk
// c of batch b and value head hd (query/key head qh = min(hd / max(H / Hq, 1),
// Hq - 1)), with r, j the rows of the chunk,
//
//   out[r,:] = scale * ( exp(g_r) * q_r h_c
//                        + sum_{j <= r, g_r <= g_j} bf16(q_r . k_j * exp(g_r - g_j)) v_j )
//
// scale = key_dim^-1/2 unless given; rows past the last token are not
// written.  key_dim = value_dim = 128.
//
// The kernel is bound by HBM (80 KB of inputs per chunk and head against
// about 4 MFLOP), so the design goal is to keep bytes in flight while the
// products run on the 5th-generation tensor cores.  A work item is a pair of
// consecutive chunks (128 tokens) of one (batch, value head): stacking the
// pair makes every product M = 128, the tcgen05 shape whose accumulator row
// i is TMEM lane i.  Value heads that share a query/key head are adjacent in
// the item order, so concurrent CTAs read that q and k from HBM once.
//
// A persistent CTA per SM has six warps:
//   warp 5     producer: streams each item as five 32 KB TMA tiles -- Q and K
//              (128 tokens x 128 dims), h of the first and of the second
//              chunk (128 x 128), V (128 x 128) -- through a 7-slot ring
//              (128-byte swizzle; rows past a batch's last token zero-filled).
//   warp 4     MMA issuer (one elected lane): S = Q K^T, X = Q h_c0,
//              Y = Q h_c1 (all M = N = 128, K = 128, fp32 in TMEM), then,
//              once P is in TMEM, P V into S's columns.  Each tile's slot is
//              released by a tcgen05.commit as soon as its last product is
//              done.
//   warps 0-3  epilogue, one thread per row: reads its row of S for the 64
//              keys of its own chunk, gates, masks and rounds them to bf16
//              into TMEM as the A operand of P V (zeros for the other chunk's
//              keys, so the pair's P is block diagonal); then reads X (first
//              chunk) or Y (second chunk) and P V and stores
//              scale * (exp(g_r) X + P V) as bf16.  The gates of the chunk
//              live in two registers per lane (prefetched one item ahead) and
//              are broadcast with shuffles.
// TMEM columns: S and then P V [0, 128), X [128, 256), Y [256, 384), P (bf16
// pairs) [384, 448).
//
// Every mbarrier wait is bounded: after kWaitNs a wait sets
// kChunkStatusTimeout in the status word, raises the CTA's abort flag, and
// the CTA winds down (the producer waits for its loads in flight, the MMA
// warp for its MMAs) before TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "chunk_o_internal.h"
#include "ptx.cuh"

namespace avp {
namespace {

constexpr int kCs = 64;          // tokens per chunk
constexpr int kRows = 2 * kCs;   // tokens per item (a pair of chunks)
constexpr int kDim = 128;        // key_dim = value_dim
constexpr int kUnits = 5;        // Q, K, H0, H1, V
constexpr int kSlots = 7;        // ring depth (units)
constexpr int kBoxBytes = kRows * 64 * 2;    // one TMA box: 128 rows x 64 columns
constexpr int kUnitBytes = 2 * kBoxBytes;    // 32 KB
constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kProdWarp = 5;
constexpr int kThreads = 32 * 6;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColX = 128, kColY = 256, kColP = 384;
constexpr uint64_t kWaitNs = 4000000000ull;  // 4 s

enum : int { U_Q = 0, U_K = 1, U_H0 = 2, U_H1 = 3, U_V = 4 };
enum : int { B_FULL = 0, B_EMPTY = kSlots, B_S_DONE = 2 * kSlots, B_P_READY, B_PV_DONE, B_TFREE,
             B_DRAIN, kNumBars };

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kRingOff = 0;
constexpr int kBarOff = kRingOff + kSlots * kUnitBytes;
constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
constexpr int kFlagOff = kTmemSlotOff + 4;
constexpr int kSmemBytes = kFlagOff + 4 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "one CTA per SM within the 227 KB opt-in limit");

struct KParams {
  CUtensorMap mq, mk, mv, mh;
  const float* g;
  void* out;
  int* status;
  int tokens, num_q_heads, num_v_heads, nc, npairs, num_items;
  float scale;
};

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       int* status) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitNs) {
      atomicOr(status, kChunkStatusTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_full(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, status);
}

// Fixed bound, no abort check: used only while draining loads in flight.
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitNs) return;
}

struct Item {
  int b, cp, hd, qh;
};

__device__ __forceinline__ Item decode(const KParams& p, int item) {
  Item it;
  it.hd = item % p.num_v_heads;
  it.cp = (item / p.num_v_heads) % p.npairs;
  it.b = item / (p.num_v_heads * p.npairs);
  int hpq = p.num_v_heads / p.num_q_heads;
  if (hpq < 1) hpq = 1;
  it.qh = min(it.hd / hpq, p.num_q_heads - 1);
  return it;
}

__device__ __forceinline__ float load_g(const KParams& p, const Item& it, int t) {
  return t < p.tokens ? __ldg(p.g + ((size_t)it.b * p.tokens + t) * p.num_v_heads + it.hd) : 0.f;
}

__global__ void __launch_bounds__(kThreads, 1) chunk_o_kernel(const __grid_constant__ KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kFlagOff);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + kTmemSlotOff);
  auto bar = [&](int i) { return base + kBarOff + 8u * (uint32_t)i; };
  auto slot_addr = [&](int s) { return base + kRingOff + (uint32_t)s * kUnitBytes; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    mbar_init(bar(B_S_DONE), 1);
    mbar_init(bar(B_P_READY), kEpiWarps);
    mbar_init(bar(B_PV_DONE), 1);
    mbar_init(bar(B_TFREE), kEpiWarps);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(base + kTmemSlotOff, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tmap_prefetch(&p.mq);
      tmap_prefetch(&p.mk);
      tmap_prefetch(&p.mv);
      tmap_prefetch(&p.mh);
      int issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.num_items; item += gridDim.x) {
        const Item it = decode(p, item);
        const int t0 = it.cp * kRows;
        const int c0 = 2 * it.cp;
        const int hrow0 = (it.b * p.nc + c0) * p.num_v_heads + it.hd;
        // a pair without a second chunk computes Y from h_c0 and drops it
        const int hrow1 = c0 + 1 < p.nc ? hrow0 + p.num_v_heads : hrow0;
        for (int u = 0; u < kUnits; ++u) {
          const int j = issued, s = j % kSlots;
          const uint32_t lap = (uint32_t)(j / kSlots);
          if (!wait_full(bar(B_EMPTY + s), (lap & 1u) ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t dst = slot_addr(s), fb = bar(B_FULL + s);
          mbar_arrive_expect_tx(fb, kUnitBytes);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const uint32_t d = dst + (uint32_t)x * kBoxBytes;
            switch (u) {
              case U_Q: tma_load_4d(d, &p.mq, fb, 64 * x, it.qh, t0, it.b); break;
              case U_K: tma_load_4d(d, &p.mk, fb, 64 * x, it.qh, t0, it.b); break;
              case U_H0: tma_load_3d(d, &p.mh, fb, 64 * x, 0, hrow0); break;
              case U_H1: tma_load_3d(d, &p.mh, fb, 64 * x, 0, hrow1); break;
              default: tma_load_4d(d, &p.mv, fb, 64 * x, it.hd, t0, it.b); break;
            }
          }
          ++issued;
        }
      }
      // every issued load has landed before the CTA may exit
      const int first = issued > kSlots ? issued - kSlots : 0;
      for (int j = first; j < issued; ++j)
        wait_drain(bar(B_FULL + j % kSlots), (uint32_t)(j / kSlots) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs the loop (descriptors in uniform registers); one
    // elected lane issues every MMA and commit.
    const uint32_t leader = elect_one();
    constexpr uint32_t idesc_kk = idesc_bf16_f32(kRows, kDim, false, false);  // B K-major (K)
    constexpr uint32_t idesc_kn = idesc_bf16_f32(kRows, kDim, false, true);   // B MN-major (h, V)
    auto wait_ = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, wait_full(b, parity, abort_flag, p.status));
    };
    bool issued_any = false;
    int n = 0;
    for (int item = blockIdx.x; item < p.num_items; item += gridDim.x, ++n) {
      const int u0 = n * kUnits;
      const int sQ = (u0 + U_Q) % kSlots, sK = (u0 + U_K) % kSlots;
      const int sH0 = (u0 + U_H0) % kSlots, sH1 = (u0 + U_H1) % kSlots, sV = (u0 + U_V) % kSlots;
      auto par = [&](int u) { return (uint32_t)((u0 + u) / kSlots) & 1u; };
      // TMEM is free once the epilogue has read the previous item
      if (n > 0 && !wait_(bar(B_TFREE), (uint32_t)(n - 1) & 1u)) break;
      if (!wait_(bar(B_FULL + sQ), par(U_Q)) || !wait_(bar(B_FULL + sK), par(U_K))) break;
      tc_fence_after();
      issued_any = true;
      // K-major Q and K: 16-element k-steps walk 32 bytes along a 128-byte
      // swizzled row, then on to the second 64-column box
      const uint64_t aq = smem_desc(slot_addr(sQ), 16, 1024, kSwizzle128B);
      const uint64_t bk = smem_desc(slot_addr(sK), 16, 1024, kSwizzle128B);
#pragma unroll
      for (int k = 0; k < kDim / 16; ++k) {
        const uint32_t off = (uint32_t)((k >> 2) * kBoxBytes + (k & 3) * 32) >> 4;
        mma_ss_if(leader, tmem + kColS, aq + off, bk + off, idesc_kk, k > 0 ? 1u : 0u);
      }
      mma_commit_if(leader, bar(B_S_DONE));
      mma_commit_if(leader, bar(B_EMPTY + sK));
      // MN-major h: a k-step is 16 rows of 128 bytes; the second 64-column
      // half of N is the next box (leading byte offset)
      for (int half = 0; half < 2; ++half) {
        const int sh = half ? sH1 : sH0;
        if (!wait_(bar(B_FULL + sh), par(half ? U_H1 : U_H0))) {
          issued_any = true;
          goto mma_done;
        }
        tc_fence_after();
        const uint64_t bh = smem_desc(slot_addr(sh), kBoxBytes, 1024, kSwizzle128B);
#pragma unroll
        for (int k = 0; k < kDim / 16; ++k) {
          const uint32_t off = (uint32_t)((k >> 2) * kBoxBytes + (k & 3) * 32) >> 4;
          mma_ss_if(leader, tmem + (half ? kColY : kColX), aq + off,
                    bh + ((uint32_t)(k * 16 * 128) >> 4), idesc_kn, k > 0 ? 1u : 0u);
        }
        mma_commit_if(leader, bar(B_EMPTY + sh));
      }
      mma_commit_if(leader, bar(B_EMPTY + sQ));
      // P V into S's columns, A = P from TMEM (8 columns of bf16 pairs per
      // 16 keys), B = V MN-major
      if (!wait_(bar(B_P_READY), (uint32_t)n & 1u)) break;
      if (!wait_(bar(B_FULL + sV), par(U_V))) break;
      tc_fence_after();
      {
        const uint64_t bv = smem_desc(slot_addr(sV), kBoxBytes, 1024, kSwizzle128B);
#pragma unroll
        for (int k = 0; k < kRows / 16; ++k)
          mma_ts_if(leader, tmem + kColS, tmem + kColP + 8u * k,
                    bv + ((uint32_t)(k * 16 * 128) >> 4), idesc_kn, k > 0 ? 1u : 0u);
      }
      mma_commit_if(leader, bar(B_PV_DONE));
      mma_commit_if(leader, bar(B_EMPTY + sV));
    }
  mma_done:
    if (issued_any) {
      // every MMA of this warp has finished before TMEM is freed
      mma_commit_if(leader, bar(B_DRAIN));
      wait_drain(bar(B_DRAIN), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ch = warp >> 1;                 // chunk of the pair
    const int rr = 32 * (warp & 1) + lane;    // row within the chunk
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    // gates of the chunk of the next item: lane l holds keys l and l + 32
    float gn0 = 0.f, gn1 = 0.f;
    if ((int)blockIdx.x < p.num_items) {
      const Item it0 = decode(p, blockIdx.x);
      const int tc = (2 * it0.cp + ch) * kCs;
      gn0 = load_g(p, it0, tc + lane);
      gn1 = load_g(p, it0, tc + 32 + lane);
    }
    int n = 0;
    for (int item = blockIdx.x; item < p.num_items; item += gridDim.x, ++n) {
      const Item it = decode(p, item);
      const float gk0 = gn0, gk1 = gn1;
      if (item + (int)gridDim.x < p.num_items) {
        const Item nx = decode(p, item + gridDim.x);
        const int tc = (2 * nx.cp + ch) * kCs;
        gn0 = load_g(p, nx, tc + lane);
        gn1 = load_g(p, nx, tc + 32 + lane);
      }
      const float g_r = (warp & 1) ? gk1 : gk0;  // this row's own gate

      // S row (own chunk's 64 keys) -> gated, masked bf16 P in TMEM
      if (!__all_sync(0xffffffffu, wait_full(bar(B_S_DONE), (uint32_t)n & 1u, abort_flag, p.status)))
        break;
      tc_fence_after();
      uint32_t sv[2][32];
      tmem_ld32(tmem + lane_base + kColS + 64u * ch, sv[0]);
      tmem_ld32(tmem + lane_base + kColS + 64u * ch + 32u, sv[1]);
      tmem_wait_ld();
      uint32_t pk[32], zero[32];
#pragma unroll
      for (int j2 = 0; j2 < 32; ++j2) {
        float w[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = 2 * j2 + e;
          const float gj = __shfl_sync(0xffffffffu, j < 32 ? gk0 : gk1, j & 31);
          const float gd = g_r - gj;
          const float sj = __uint_as_float(sv[j >> 5][j & 31]);
          w[e] = (j <= rr && gd <= 0.f) ? sj * __expf(gd) : 0.f;
        }
        pk[j2] = pack_bf16(w[0], w[1]);
        zero[j2] = 0u;
      }
      tmem_st32(tmem + lane_base + kColP + 32u * ch, pk);
      tmem_st32(tmem + lane_base + kColP + 32u * (1 - ch), zero);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P_READY));

      // out = scale * (exp(g_r) * (X or Y) + P V)
      if (!__all_sync(0xffffffffu, wait_full(bar(B_PV_DONE), (uint32_t)n & 1u, abort_flag, p.status)))
        break;
      tc_fence_after();
      const float eg = __expf(g_r) * p.scale;
      const int t = (2 * it.cp + ch) * kCs + rr;
      __nv_bfloat16* orow = out + (((size_t)it.b * p.tokens + t) * p.num_v_heads + it.hd) * kDim;
      const uint32_t col_xy = ch ? kColY : kColX;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t xv[32], pv[32];
        tmem_ld32(tmem + lane_base + col_xy + 32u * q4, xv);
        tmem_ld32(tmem + lane_base + kColS + 32u * q4, pv);
        tmem_wait_ld();
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          o[i] = pack_bf16(eg * __uint_as_float(xv[2 * i]) + p.scale * __uint_as_float(pv[2 * i]),
                           eg * __uint_as_float(xv[2 * i + 1]) + p.scale * __uint_as_float(pv[2 * i + 1]));
        if (t < p.tokens) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * q4);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_TFREE));
    }
  }

  // all roles done (or given up, with their async work drained): free TMEM
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

int encode(EncodeTiledFn enc, CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
           const cuuint64_t* strides, const cuuint32_t* box) {
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return (int)enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

size_t chunk_o_smem_bytes() { return kSmemBytes; }

cudaError_t prepare_chunk_o() {
  return cudaFuncSetAttribute(chunk_o_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_chunk_o(const ChunkParams& p, EncodeTiledFn enc, cudaStream_t stream) {
  const long long nc = (p.tokens + kCs - 1) / kCs;
  const long long npairs = (nc + 1) / 2;
  const long long items = (long long)p.batch * p.num_v_heads * npairs;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL || (long long)p.batch * nc * p.num_v_heads * kDim > 0xffffffffLL)
    return cudaErrorInvalidValue;

  KParams k;
  const cuuint64_t row = kDim * 2;  // bytes per head row
  const cuuint64_t T = (cuuint64_t)p.tokens, B = (cuuint64_t)p.batch;
  const cuuint32_t box_t[4] = {64, 1, kRows, 1};
  {
    const cuuint64_t dims[4] = {kDim, (cuuint64_t)p.num_q_heads, T, B};
    const cuuint64_t str[3] = {row, row * p.num_q_heads, row * p.num_q_heads * T};
    if (encode(enc, &k.mq, p.q, 4, dims, str, box_t) || encode(enc, &k.mk, p.k, 4, dims, str, box_t))
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {kDim, (cuuint64_t)p.num_v_heads, T, B};
    const cuuint64_t str[3] = {row, row * p.num_v_heads, row * p.num_v_heads * T};
    if (encode(enc, &k.mv, p.v, 4, dims, str, box_t)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {kDim, kDim, (cuuint64_t)(B * nc * p.num_v_heads)};
    const cuuint64_t str[2] = {row, row * kDim};
    const cuuint32_t box[3] = {64, kDim, 1};
    if (encode(enc, &k.mh, p.h, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  k.g = p.g;
  k.out = p.out;
  k.status = p.status;
  k.tokens = p.tokens;
  k.num_q_heads = p.num_q_heads;
  k.num_v_heads = p.num_v_heads;
  k.nc = (int)nc;
  k.npairs = (int)npairs;
  k.num_items = (int)items;
  k.scale = p.scale;
  const int grid = (int)(items < p.sm_count ? items : p.sm_count);
  chunk_o_kernel<<<grid, kThreads, kSmemBytes, stream>>>(k);
  return cudaGetLastError();
}

}  // namespace avp
