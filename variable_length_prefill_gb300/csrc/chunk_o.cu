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
// Per chunk the work is three small products (64x128 by 128x64, 64x128 by
// 128x128, 64x64 by 64x128) on 80 KB of inputs: about 44 FLOP per byte, so the
// kernel is bound by HBM, not by the tensor pipe, and the design goal is to
// keep enough bytes in flight.  A persistent CTA per SM walks the work items
// (batch, chunk, value head) -- value heads that share a query/key head are
// adjacent, so concurrent CTAs read that q and k once from HBM.  One producer
// warp streams each item as five 16 KB units -- Q, K, h[:, 0:64], h[:, 64:128],
// V -- through a ring of 13 shared-memory slots with TMA tile loads (128-byte
// swizzle, zero fill past the last token of a batch).  Four consumer warps,
// warp w owning rows 16w..16w+15, release each unit as soon as its product is
// done (Q once its rows are in registers, K after S, each h half after its
// half of Q h, V after P V), so the next items' loads start while the current
// one is computed.  The products use the warp-level bf16 MMA (mma.sync
// m16n8k16) fed by ldmatrix; S = Q K^T is gated, masked and rounded to bf16 in
// registers and its accumulator fragments are reused as the A operand of P V
// (an m16n8 accumulator and an m16k16 A fragment have the same row/column
// ownership).  Each warp writes its 16 output rows to its own staging tile
// and stores them with one TMA tile store (rows past the batch's last token
// are clipped by the tensor map).  The 64 gates of an item live in two
// registers per lane of every consumer warp (prefetched one item ahead) and
// are read with warp shuffles, so the consumer warps share nothing but the
// ring's barriers.
//
// Every mbarrier wait is bounded: after kWaitNs a wait sets
// kChunkStatusTimeout in the status word, raises the CTA's abort flag, and
// the CTA winds down, the producer first waiting (bounded) for its loads in
// flight.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "chunk_o_internal.h"
#include "ptx.cuh"

namespace avp {
namespace {

constexpr int kCs = 64;        // tokens per chunk
constexpr int kDim = 128;      // key_dim = value_dim
constexpr int kUnits = 5;      // Q, K, H0, H1, V
constexpr int kSlots = 13;     // ring depth (units)
constexpr int kUnitBytes = 16384;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kStageBytes = 2 * 16 * 128;  // one warp's 16 output rows, two 64-column halves
constexpr uint64_t kWaitNs = 4000000000ull;  // 4 s

enum : int { U_Q = 0, U_K = 1, U_H0 = 2, U_H1 = 3, U_V = 4 };

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kRingOff = 0;
constexpr int kStageOff = kRingOff + kSlots * kUnitBytes;
constexpr int kBarOff = kStageOff + kConsumerWarps * kStageBytes;  // full[13], empty[13]
constexpr int kFlagOff = kBarOff + 2 * kSlots * 8;
constexpr int kSmemBytes = kFlagOff + 16 + 1024;  // + alignment slack

struct KParams {
  CUtensorMap mq, mk, mv, mh, mo;
  const float* g;
  int* status;
  int tokens, num_q_heads, num_v_heads, nc, num_items;
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

__device__ __forceinline__ void tma_store_4d(const void* tmap, uint32_t src, int c0, int c1, int c2,
                                             int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
          tmap),
      "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// Byte offset of 16-byte chunk `ch` (0..7) of row `row` in a tile of
// 128-byte rows written by TMA with the 128-byte swizzle (tile base 1024-byte
// aligned): the chunk index is XORed with the row index modulo 8.
__device__ __forceinline__ uint32_t sw128(int row, int ch) {
  return (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4));
}

// A [64 rows][128 columns] unit: two 64-column halves of 8 KB.
__device__ __forceinline__ uint32_t rows64_addr(uint32_t base, int row, int col) {
  return base + (uint32_t)(col >> 6) * 8192u + sw128(row, (col & 63) >> 3);
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

// Hand a ring slot back to the producer after this warp's ldmatrix reads of
// it.  The reads went through the generic proxy and the next fill is a TMA
// write (async proxy): each lane orders its reads before async-proxy accesses
// with a proxy fence, then one lane arrives (release) for the warp.  Without
// the fence a refill was seen to land under reads still in flight.
__device__ __forceinline__ void release(uint32_t empty_bar, int lane) {
  fence_async_smem();
  __syncwarp();
  if (lane == 0) mbar_arrive(empty_bar);
}

struct Item {
  int b, c, hd, qh;
};

__device__ __forceinline__ Item decode(const KParams& p, int item) {
  Item it;
  it.hd = item % p.num_v_heads;
  it.c = (item / p.num_v_heads) % p.nc;
  it.b = item / (p.num_v_heads * p.nc);
  int hpq = p.num_v_heads / p.num_q_heads;
  if (hpq < 1) hpq = 1;
  it.qh = min(it.hd / hpq, p.num_q_heads - 1);
  return it;
}

__device__ __forceinline__ float load_g(const KParams& p, const Item& it, int r) {
  const int t = it.c * kCs + r;
  return t < p.tokens ? __ldg(p.g + ((size_t)it.b * p.tokens + t) * p.num_v_heads + it.hd) : 0.f;
}

__global__ void __launch_bounds__(kThreads, 1) chunk_o_kernel(const __grid_constant__ KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kFlagOff);
  auto full = [&](int s) { return base + kBarOff + 8u * s; };
  auto empty = [&](int s) { return base + kBarOff + 8u * (kSlots + s); };
  auto slot_addr = [&](int s) { return base + kRingOff + (uint32_t)s * kUnitBytes; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
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
        const int t0 = it.c * kCs;
        const int hrow = ((it.b * p.nc + it.c) * p.num_v_heads + it.hd);
        for (int u = 0; u < kUnits; ++u) {
          const int j = issued, s = j % kSlots;
          const uint32_t lap = (uint32_t)(j / kSlots);
          if (!wait_full(empty(s), (lap & 1u) ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t dst = slot_addr(s), bar = full(s);
          mbar_arrive_expect_tx(bar, kUnitBytes);
          switch (u) {
            case U_Q:
              tma_load_4d(dst, &p.mq, bar, 0, it.qh, t0, it.b);
              tma_load_4d(dst + 8192, &p.mq, bar, 64, it.qh, t0, it.b);
              break;
            case U_K:
              tma_load_4d(dst, &p.mk, bar, 0, it.qh, t0, it.b);
              tma_load_4d(dst + 8192, &p.mk, bar, 64, it.qh, t0, it.b);
              break;
            case U_H0:
              tma_load_3d(dst, &p.mh, bar, 0, 0, hrow);
              break;
            case U_H1:
              tma_load_3d(dst, &p.mh, bar, 64, 0, hrow);
              break;
            default:
              tma_load_4d(dst, &p.mv, bar, 0, it.hd, t0, it.b);
              tma_load_4d(dst + 8192, &p.mv, bar, 64, it.hd, t0, it.b);
              break;
          }
          ++issued;
        }
      }
      // every issued load has landed before the CTA may exit (on the normal
      // path the consumers waited for all of them already)
      const int first = issued > kSlots ? issued - kSlots : 0;
      for (int j = first; j < issued; ++j) wait_drain(full(j % kSlots), (uint32_t)(j / kSlots) & 1u);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int r0 = warp * 16;                       // this warp's first row
  const int fr = lane >> 2, fc = (lane & 3) * 2;  // fragment row / column pair
  const int row_lo = r0 + fr, row_hi = row_lo + 8;
  const uint32_t stage = base + kStageOff + (uint32_t)warp * kStageBytes;
  // ldmatrix row/column offsets of this lane
  const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8;  // A (Q) and B^T (h, V) rows
  const int a_col = (lane >> 4) * 8;
  const int b_row = (lane & 7) + (lane >> 4) * 8;        // B (K) rows = keys
  const int b_col = ((lane >> 3) & 1) * 8;

  // gates of the next item: lane l holds rows l and l + 32
  float gn0 = 0.f, gn1 = 0.f;
  if ((int)blockIdx.x < p.num_items) {
    const Item it0 = decode(p, blockIdx.x);
    gn0 = load_g(p, it0, lane);
    gn1 = load_g(p, it0, lane + 32);
  }
  int unit0 = 0;  // ring index of the item's first unit
  bool ok = true;
  for (int item = blockIdx.x; item < p.num_items; item += gridDim.x, unit0 += kUnits) {
    const Item it = decode(p, item);
    const float gv0 = gn0, gv1 = gn1;
    if (item + (int)gridDim.x < p.num_items) {
      const Item nx = decode(p, item + gridDim.x);
      gn0 = load_g(p, nx, lane);
      gn1 = load_g(p, nx, lane + 32);
    }

    auto slot_of = [&](int u) { return (unit0 + u) % kSlots; };
    auto par_of = [&](int u) { return (uint32_t)((unit0 + u) / kSlots) & 1u; };

    // Q rows of this warp -> registers; Q slot free
    uint32_t qa[8][4];
    {
      const int s = slot_of(U_Q);
      if (!(ok = wait_full(full(s), par_of(U_Q), abort_flag, p.status))) break;
      const uint32_t q0 = slot_addr(s);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) ldsm_x4(rows64_addr(q0, r0 + a_row, ks * 16 + a_col), qa[ks]);
      release(empty(s), lane);
    }

    // S = Q K^T (8 tiles of 8 keys)
    float sacc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
    {
      const int s = slot_of(U_K);
      if (!(ok = wait_full(full(s), par_of(U_K), abort_flag, p.status))) break;
      const uint32_t k0 = slot_addr(s);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int n2 = 0; n2 < 4; ++n2) {
          uint32_t bk[4];
          ldsm_x4(rows64_addr(k0, n2 * 16 + b_row, ks * 16 + b_col), bk);
          mma_bf16(sacc[2 * n2], qa[ks], bk[0], bk[1]);
          mma_bf16(sacc[2 * n2 + 1], qa[ks], bk[2], bk[3]);
        }
      }
      release(empty(s), lane);
    }

    // gate, mask, round to bf16 -> A fragments of P (4 k-steps of 16 keys)
    // rows row_lo, row_hi are both in one 32-row half (r0 is a multiple of 16)
    const float g_lo = __shfl_sync(0xffffffffu, r0 < 32 ? gv0 : gv1, row_lo & 31);
    const float g_hi = __shfl_sync(0xffffffffu, r0 < 32 ? gv0 : gv1, row_hi & 31);
    uint32_t pa[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      // key columns nt*8 + fc and nt*8 + fc + 1
      const float gc0 = __shfl_sync(0xffffffffu, nt < 4 ? gv0 : gv1, (nt * 8 + fc) & 31);
      const float gc1 = __shfl_sync(0xffffffffu, nt < 4 ? gv0 : gv1, (nt * 8 + fc + 1) & 31);
      float w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = e < 2 ? row_lo : row_hi;
        const int col = nt * 8 + fc + (e & 1);
        const float gd = (e < 2 ? g_lo : g_hi) - ((e & 1) ? gc1 : gc0);
        w[e] = (col <= row && gd <= 0.f) ? sacc[nt][e] * __expf(gd) : 0.f;
      }
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(w[0], w[1]);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(w[2], w[3]);
    }

    // O = Q h, one 64-column half of h per unit
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int u = U_H0 + half, s = slot_of(u);
      if (!(ok = wait_full(full(s), par_of(u), abort_flag, p.status))) break;
      const uint32_t h0 = slot_addr(s);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int n2 = 0; n2 < 4; ++n2) {
          uint32_t bh[4];
          ldsm_x4_t(h0 + sw128(ks * 16 + a_row, n2 * 2 + (a_col >> 3)), bh);
          mma_bf16(o[half * 8 + 2 * n2], qa[ks], bh[0], bh[1]);
          mma_bf16(o[half * 8 + 2 * n2 + 1], qa[ks], bh[2], bh[3]);
        }
      }
      release(empty(s), lane);
    }
    if (!ok) break;
    const float eg_lo = __expf(g_lo), eg_hi = __expf(g_hi);
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= eg_lo;
      o[nt][1] *= eg_lo;
      o[nt][2] *= eg_hi;
      o[nt][3] *= eg_hi;
    }

    // O += P V
    {
      const int s = slot_of(U_V);
      if (!(ok = wait_full(full(s), par_of(U_V), abort_flag, p.status))) break;
      const uint32_t v0 = slot_addr(s);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
        for (int n2 = 0; n2 < 8; ++n2) {
          uint32_t bv[4];
          ldsm_x4_t(rows64_addr(v0, ks * 16 + a_row, n2 * 16 + a_col), bv);
          mma_bf16(o[2 * n2], pa[ks], bv[0], bv[1]);
          mma_bf16(o[2 * n2 + 1], pa[ks], bv[2], bv[3]);
        }
      }
      release(empty(s), lane);
    }

    // out = scale * O: staging tile (after the previous store has read it),
    // then one TMA store per 64-column half
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int col = nt * 8 + fc;
      const uint32_t half = (uint32_t)(col >> 6) * 2048u;
      const int ch = (col & 63) >> 3, byte = (col & 7) * 2;
      asm volatile("st.shared.b32 [%0], %1;" ::"r"(stage + half + sw128(fr, ch) + byte),
                   "r"(pack_bf16(o[nt][0] * p.scale, o[nt][1] * p.scale)));
      asm volatile("st.shared.b32 [%0], %1;" ::"r"(stage + half + sw128(fr + 8, ch) + byte),
                   "r"(pack_bf16(o[nt][2] * p.scale, o[nt][3] * p.scale)));
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0 && it.c * kCs + r0 < p.tokens) {
      tma_store_4d(&p.mo, stage, 0, it.hd, it.c * kCs + r0, it.b);
      tma_store_4d(&p.mo, stage + 2048, 64, it.hd, it.c * kCs + r0, it.b);
      bulk_commit();
    }
  }
  if (lane == 0) bulk_wait0();
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

cudaError_t launch_chunk_o(const ChunkParams& p, EncodeTiledFn enc, cudaStream_t stream) {
  static bool attr_set = false;  // per process; the attribute is per function, not per device
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(chunk_o_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long nc = (p.tokens + kCs - 1) / kCs;
  const long long items = (long long)p.batch * p.num_v_heads * nc;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL || (long long)p.batch * nc * p.num_v_heads * kDim > 0xffffffffLL)
    return cudaErrorInvalidValue;

  KParams k;
  const cuuint64_t row = kDim * 2;  // bytes per head row
  const cuuint64_t T = (cuuint64_t)p.tokens, B = (cuuint64_t)p.batch;
  {
    const cuuint64_t dims[4] = {kDim, (cuuint64_t)p.num_q_heads, T, B};
    const cuuint64_t str[3] = {row, row * p.num_q_heads, row * p.num_q_heads * T};
    const cuuint32_t box[4] = {64, 1, kCs, 1};
    if (encode(enc, &k.mq, p.q, 4, dims, str, box) || encode(enc, &k.mk, p.k, 4, dims, str, box))
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {kDim, (cuuint64_t)p.num_v_heads, T, B};
    const cuuint64_t str[3] = {row, row * p.num_v_heads, row * p.num_v_heads * T};
    const cuuint32_t box_v[4] = {64, 1, kCs, 1};
    const cuuint32_t box_o[4] = {64, 1, 16, 1};
    if (encode(enc, &k.mv, p.v, 4, dims, str, box_v) ||
        encode(enc, &k.mo, p.out, 4, dims, str, box_o))
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {kDim, kDim, (cuuint64_t)(B * nc * p.num_v_heads)};
    const cuuint64_t str[2] = {row, row * kDim};
    const cuuint32_t box[3] = {64, kDim, 1};
    if (encode(enc, &k.mh, p.h, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  k.g = p.g;
  k.status = p.status;
  k.tokens = p.tokens;
  k.num_q_heads = p.num_q_heads;
  k.num_v_heads = p.num_v_heads;
  k.nc = (int)nc;
  k.num_items = (int)items;
  k.scale = p.scale;
  const int grid = (int)(items < p.sm_count ? items : p.sm_count);
  chunk_o_kernel<<<grid, kThreads, kSmemBytes, stream>>>(k);
  return cudaGetLastError();
}

}  // namespace avp
