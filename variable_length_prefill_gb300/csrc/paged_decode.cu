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
// (block, KV head) holds D x 16 contiguous keys and D x 16 contiguous values
// (4 KB each for D = 128), so the kernel is bound by HBM, or for the page's
// small shapes by latency.  No tensor cores:
//   grid  = persistent CTAs, each walking (sequence, KV head, group of up to
//           MQ query heads) pairs with a stride of gridDim.x; MQ is the power
//           of two (at most 8) that covers the query heads per KV head,
//           halved while the pairs would not fill the SMs;
//   warp 4 (producer) streams each block's keys and values with two
//           cp.async.bulk copies into a ring of stages, across pair
//           boundaries, so many blocks are in flight per SM;
//   warps 0-3 (consumers) take the blocks round-robin (block i of the CTA's
//           stream goes to warp i mod 4, stage i mod STAGES), each with an
//           exp2 online softmax per head; keys: lane = (token, half of the
//           dimensions), one shuffle to add the halves; values: lane = the
//           dimensions lane, lane + 32, ...; per pair the four warps' (m, l,
//           O) merge through shared memory.
// Short block tables (at most kWppMaxBlocks blocks) with at least one pair
// per consumer warp run warp-per-pair instead: consumer warp w takes the
// CTA's pairs w, w + 4, ... whole, from its own quarter of the ring (stages
// w, w + 4, ...), which the producer fills round-robin over the four warps;
// no merge, no barrier between the warps.
// Every wait is bounded like the attention kernels'.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "attn_varlen_device.cuh"
#include "paged_decode_internal.h"
#include "ptx.cuh"

namespace avp {
namespace {

constexpr int kConsumers = 4;                    // consumer warps
constexpr int kThreads = 32 * (kConsumers + 1);  // + the producer warp
constexpr int kBlock = 16;   // tokens per cache block
constexpr int kMaxQ = 8;     // query heads per CTA at most
constexpr int kMaxDevices = 64;
// Ring stages per CTA (D <= 128; half as many for D = 256): a multiple of
// the four consumer warps.
#ifndef ATTN_VARLEN_PAGED_STAGES
#define ATTN_VARLEN_PAGED_STAGES 8
#endif
// Ring stages of the warp-per-pair form (D <= 128; half as many for D = 256)
#ifndef ATTN_VARLEN_PAGED_STAGES_WPP
#define ATTN_VARLEN_PAGED_STAGES_WPP 8
#endif
// Longest block table (blocks) the warp-per-pair form takes
constexpr int kWppMaxBlocks = 8;

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

// Shared-memory layout of one kernel instance.
template <int D, int MQ, bool WPP>
struct PagedSmem {
  static constexpr uint32_t KV_BYTES = D * kBlock * 2;    // one block's keys (or values)
  static constexpr uint32_t STAGE = 2 * KV_BYTES;          // keys, then values
  static constexpr int RING = WPP ? ATTN_VARLEN_PAGED_STAGES_WPP : ATTN_VARLEN_PAGED_STAGES;
  static constexpr int STAGES = D == 256 ? (RING / 2 + 3) / 4 * 4 : RING;
  static_assert(STAGES % kConsumers == 0, "stage i mod STAGES belongs to warp i mod 4");
  static constexpr int SPW = STAGES / kConsumers;  // stages of each consumer warp
  static_assert(SPW >= 1, "every consumer warp owns a stage");
  static constexpr int QROW = D + 4;  // second half of a query row 4 floats on
  static constexpr int QROWS = WPP ? kConsumers * MQ : MQ;  // warp-private rows with WPP
  static constexpr uint32_t RING_OFF = 0;
  static constexpr uint32_t Q_OFF = RING_OFF + STAGES * STAGE;
  static constexpr uint32_t P_OFF = Q_OFF + QROWS * QROW * 4;
  static constexpr uint32_t M_OFF = P_OFF + kConsumers * MQ * kBlock * 4;
  static constexpr uint32_t L_OFF = M_OFF + kConsumers * MQ * 4;
  static constexpr uint32_t O_OFF = L_OFF + kConsumers * MQ * 4;
  static constexpr uint32_t BAR_OFF = (O_OFF + kConsumers * MQ * D * 4 + 7u) & ~7u;
  static constexpr uint32_t OK_OFF = BAR_OFF + 2 * STAGES * 8;  // int per stage: block id valid
  static constexpr uint32_t ABORT_OFF = OK_OFF + STAGES * 4;
  static constexpr uint32_t BYTES = ABORT_OFF + 16 + 128;       // + alignment slack
};

template <int D, typename T, int MQ, bool WPP>
__global__ void __launch_bounds__(kThreads) paged_decode_kernel(const __grid_constant__ PagedParams p) {
  using S = PagedSmem<D, MQ, WPP>;
  constexpr int NCH = D / 8;        // 16-byte chunks of a key row
  constexpr int HCH = NCH / 2;      // chunks per lane (one half of the row)
  constexpr int DPL = D / 32;       // value dimensions per lane
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 127u) & ~127u;
  uint8_t* bp = smem_raw + (base - raw);
  float (*s_q)[S::QROW] = reinterpret_cast<float (*)[S::QROW]>(bp + S::Q_OFF);
  float (*s_p)[MQ][kBlock] = reinterpret_cast<float (*)[MQ][kBlock]>(bp + S::P_OFF);
  float (*s_m)[MQ] = reinterpret_cast<float (*)[MQ]>(bp + S::M_OFF);
  float (*s_l)[MQ] = reinterpret_cast<float (*)[MQ]>(bp + S::L_OFF);
  float (*s_o)[MQ][D] = reinterpret_cast<float (*)[MQ][D]>(bp + S::O_OFF);
  volatile int* blk_ok = reinterpret_cast<volatile int*>(bp + S::OK_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bp + S::ABORT_OFF);
  auto full = [&](int s) -> uint32_t { return base + S::BAR_OFF + 8u * (uint32_t)s; };
  auto empty = [&](int s) -> uint32_t { return base + S::BAR_OFF + 8u * (uint32_t)(S::STAGES + s); };

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int ngroups = (p.qpk + MQ - 1) / MQ;
  const int pairs = p.num_seqs * p.num_kv_heads * ngroups;
  // pair -> sequence, KV head, first query head, query heads, blocks
  auto decode = [&](int pr, int& seq, int& g, int& h0, int& nq, int& nblk) {
    seq = pr / (p.num_kv_heads * ngroups);
    const int rem = pr - seq * p.num_kv_heads * ngroups;
    g = rem / ngroups;
    h0 = g * p.qpk + (rem - g * ngroups) * MQ;
    nq = min(MQ, g * p.qpk + p.qpk - h0);
    int L = p.seq_lens[seq];
    if (L > p.max_blocks * kBlock) L = p.max_blocks * kBlock;  // the table holds no more
    nblk = L > 0 ? (L + kBlock - 1) / kBlock : 0;
    return L;
  };

  // One block of stage `s` for the MQ query rows `qr` (pre-scaled by
  // scale_log2): scores, running max and sum, O.  Lane = (token, half) for
  // the keys, lane = dimensions lane, lane + 32, ... for the values.
  const int tok = lane & 15, half = lane >> 4;
  auto block_step = [&](int s, const float (*qr)[S::QROW], int jb, int L, float (&m)[MQ],
                        float (&l)[MQ], float (&o)[MQ][DPL]) {
    const uint8_t* stage = bp + S::RING_OFF + (size_t)s * S::STAGE;
    // scores of this lane's token for every query head (half the dimensions)
    const uint4* kb = reinterpret_cast<const uint4*>(stage);
    float acc[MQ];
#pragma unroll
    for (int hh = 0; hh < MQ; ++hh) acc[hh] = 0.f;
#pragma unroll
    for (int c = 0; c < HCH; ++c) {
      float kf[8];
      unpack8<T>(kb[(half * HCH + c) * kBlock + tok], kf);
      const int d0 = (half * HCH + c) * 8 + half * 4;  // padded query row
      // every head of the group, also past nq (zero queries, results
      // unused): branch-free, so the heads' chains interleave
#pragma unroll
      for (int hh = 0; hh < MQ; ++hh) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[hh] = fmaf(qr[hh][d0 + e], kf[e], acc[hh]);
      }
    }
    const bool live = jb * kBlock + tok < L;
#pragma unroll
    for (int hh = 0; hh < MQ; ++hh) {
      float sc = acc[hh] + __shfl_xor_sync(0xffffffffu, acc[hh], 16);
      sc = live ? sc : -INFINITY;
      float bm = sc;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
      const float mn = fmaxf(m[hh], bm);  // finite: every block holds a live token
      const float alpha = ex2(m[hh] - mn);
      const float pw = ex2(sc - mn);
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
    // values: dimensions lane, lane + 32, ...; 16 tokens each (32 bytes)
    const uint4* vb = reinterpret_cast<const uint4*>(stage + S::KV_BYTES);
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      float v0[8], v1[8];
      const int d = e * 32 + lane;
      unpack8<T>(vb[2 * d], v0);
      unpack8<T>(vb[2 * d + 1], v1);
#pragma unroll
      for (int hh = 0; hh < MQ; ++hh) {
        float a = o[hh][e];
#pragma unroll
        for (int t = 0; t < 8; ++t) a = fmaf(s_p[warp][hh][t], v0[t], a);
#pragma unroll
        for (int t = 0; t < 8; ++t) a = fmaf(s_p[warp][hh][8 + t], v1[t], a);
        o[hh][e] = a;
      }
    }
    // the stage's shared-memory reads come before its next bulk copy, and
    // s_p is read by every lane before the next block overwrites it
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  };
  // issue one block's two copies into stage s (lane 0); a bad id marks it
  auto issue_block = [&](int s, int b, int g) {
    if (lane == 0) {
      if (b < 0 || b >= p.num_blocks) {  // never dereference a bad block id
        atomicOr(p.status, kPagedStatusBadBlock);
        blk_ok[s] = 0;
        mbar_arrive(full(s));
      } else {
        blk_ok[s] = 1;
        const size_t off = ((size_t)b * p.num_kv_heads + g) * D * kBlock;
        const uint32_t dst = base + S::RING_OFF + (uint32_t)s * S::STAGE;
        mbar_arrive_expect_tx(full(s), S::STAGE);
        bulk_copy_g2s(dst, static_cast<const T*>(p.k_cache) + off, S::KV_BYTES, full(s));
        bulk_copy_g2s(dst + S::KV_BYTES, static_cast<const T*>(p.v_cache) + off, S::KV_BYTES,
                      full(s));
      }
    }
    __syncwarp();
  };
  // query rows of pair pr for consumer lane slots e = idx0 + stride i
  constexpr int QSTRIDE = WPP ? 32 : 32 * kConsumers;
  constexpr int QPT = (MQ * D + QSTRIDE - 1) / QSTRIDE;
  auto load_q = [&](int pr, int idx0, float (&qn)[QPT]) {
    int seq, g, h0, nq, nblk;
    if (pr < pairs) decode(pr, seq, g, h0, nq, nblk);
#pragma unroll
    for (int i = 0; i < QPT; ++i) {
      const int e = idx0 + i * QSTRIDE;
      qn[i] = 0.f;
      if (pr < pairs && e < MQ * D && e / D < nq)
        qn[i] = to_f32<T>(static_cast<const T*>(p.query)[((size_t)seq * p.num_query_heads + h0) * D + e]) *
                p.scale_log2;
    }
  };

  if constexpr (WPP) {
    if (warp == kConsumers) {
      // -------------------------------------------- producer, warp per pair
      // Stream w = the pairs of consumer warp w; round-robin over the four
      // streams, one block each turn, into stage w + 4 (pos_w mod SPW).
      // A pair's block ids (at most kWppMaxBlocks) are one coalesced read.
      int kk[kConsumers], nb[kConsumers], jj[kConsumers], gg[kConsumers], ids[kConsumers];
      uint32_t pos[kConsumers];
      bool ok = true;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        kk[w] = w - kConsumers;
        nb[w] = jj[w] = gg[w] = ids[w] = 0;
        pos[w] = 0;
      }
      // next pair of stream w with blocks; nb = -1 once the stream has none
      auto advance = [&](int& k, int& n, int& j, int& g, int& id) {
        for (;;) {
          k += kConsumers;
          const int pr = (int)blockIdx.x + k * (int)gridDim.x;
          if (pr >= pairs) { n = -1; return; }
          // the pair's table row (at most kWppMaxBlocks entries) is read
          // together with its length, not after it
          const int sq = pr / (p.num_kv_heads * ngroups);
          const int idl =
              lane < p.max_blocks ? __ldg(p.block_tables + (size_t)sq * p.max_blocks + lane) : 0;
          int seq, h0, nq;
          decode(pr, seq, g, h0, nq, n);
          if (n > 0) {
            j = 0;
            id = idl;
            return;
          }
        }
      };
      for (bool any = true; ok && any;) {
        any = false;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
          if (!ok || nb[w] < 0) continue;
          if (jj[w] == nb[w]) advance(kk[w], nb[w], jj[w], gg[w], ids[w]);
          if (nb[w] < 0) continue;
          any = true;
          const int s = w + kConsumers * (int)(pos[w] % S::SPW);
          const uint32_t use = pos[w] / S::SPW;
          const bool wt = wait_bounded(empty(s), (use & 1u) ^ 1u, abort_flag, p.status,
                                       kStatusTimeoutLoad);
          if (!__all_sync(0xffffffffu, wt)) { ok = false; break; }
          issue_block(s, __shfl_sync(0xffffffffu, ids[w], jj[w]), gg[w]);
          ++jj[w];
          ++pos[w];
        }
      }
      if (!ok) {
        // let every copy already issued land before the CTA can exit
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
          const uint32_t first = pos[w] > (uint32_t)S::SPW ? pos[w] - S::SPW : 0;
          for (uint32_t it = first; it < pos[w]; ++it)
            wait_drain(full(w + kConsumers * (int)(it % S::SPW)), (it / S::SPW) & 1u);
        }
      }
      return;
    }
    // ----------------------------------------- consumer warp, whole pairs
    // Pairs k = warp, warp + 4, ... of the CTA; the next pair's query rows
    // are read into registers while this pair runs.
    float (*qw)[S::QROW] = s_q + warp * MQ;
    bool ok = true;
    uint32_t pos = 0;
    float qn[QPT];
    load_q((int)blockIdx.x + warp * (int)gridDim.x, lane, qn);
    for (int k = warp;; k += kConsumers) {
      const int pr = (int)blockIdx.x + k * (int)gridDim.x;
      if (pr >= pairs) break;
      int seq, g, h0, nq, nblk;
      const int L = decode(pr, seq, g, h0, nq, nblk);
      T* out = static_cast<T*>(p.out) + ((size_t)seq * p.num_query_heads + h0) * D;
      __syncwarp();  // the previous pair's reads of qw are done
#pragma unroll
      for (int i = 0; i < QPT; ++i) {
        const int e = lane + i * 32;
        if (e < MQ * D) qw[e / D][e % D + (e % D >= D / 2 ? 4 : 0)] = qn[i];
      }
      __syncwarp();
      load_q(pr + kConsumers * (int)gridDim.x, lane, qn);
      float m[MQ], l[MQ], o[MQ][DPL];
#pragma unroll
      for (int hh = 0; hh < MQ; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[hh][e] = 0.f;
      }
      for (int jb = 0; jb < nblk; ++jb, ++pos) {
        const int s = warp + kConsumers * (int)(pos % S::SPW);
        if (ok) {
          const bool w = wait_bounded(full(s), (pos / S::SPW) & 1u, abort_flag, p.status,
                                      kStatusTimeoutSoftmax);
          ok = __all_sync(0xffffffffu, w);
        }
        if (!ok || !blk_ok[s]) {
          __syncwarp();
          if (lane == 0 && ok) mbar_arrive(empty(s));
          continue;
        }
        block_step(s, qw, jb, L, m, l, o);
      }
      // a pair with no block (ctx_len <= 0) or whose blocks were all bad
      // gets zero rows
#pragma unroll
      for (int hh = 0; hh < MQ; ++hh) {
        if (hh >= nq) break;
        const float inv = l[hh] > 0.f ? 1.0f / l[hh] : 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) out[hh * D + e * 32 + lane] = from_f32<T>(o[hh][e] * inv);
      }
    }
    return;
  }

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    // The CTA's blocks in stream order, 32 at a time: one coalesced read of
    // 32 block-table entries per chunk, the next chunk's read (possibly the
    // next pair's) issued before the current chunk's copies, so no copy
    // waits for its block id.  Pairs with no block add no item.
    struct Chunk {
      int pr, seq, g, nblk, jb0;
    };
    auto first_from = [&](int pr) -> Chunk {
      for (; pr < pairs; pr += gridDim.x) {
        int seq, g, h0, nq, nblk;
        decode(pr, seq, g, h0, nq, nblk);
        if (nblk > 0) return Chunk{pr, seq, g, nblk, 0};
      }
      return Chunk{pairs, 0, 0, 0, 0};
    };
    auto advance = [&](const Chunk& c) -> Chunk {
      if (c.jb0 + 32 < c.nblk) return Chunk{c.pr, c.seq, c.g, c.nblk, c.jb0 + 32};
      return first_from(c.pr + (int)gridDim.x);
    };
    auto ids_of = [&](const Chunk& c) -> int {
      if (c.pr >= pairs || c.jb0 + lane >= c.nblk) return 0;
      return __ldg(p.block_tables + (size_t)c.seq * p.max_blocks + c.jb0 + lane);
    };
    uint32_t item = 0;
    bool ok = true;
    Chunk cur = first_from(blockIdx.x);
    int ids = ids_of(cur);
    while (ok && cur.pr < pairs) {
      const Chunk nxt = advance(cur);
      const int ids_next = ids_of(nxt);
      const int n = min(32, cur.nblk - cur.jb0);
      for (int j = 0; j < n; ++j, ++item) {
        const int s = item % S::STAGES;
        const uint32_t use = item / S::STAGES;
        const bool w = wait_bounded(empty(s), (use & 1u) ^ 1u, abort_flag, p.status,
                                    kStatusTimeoutLoad);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        issue_block(s, __shfl_sync(0xffffffffu, ids, j), cur.g);
      }
      cur = nxt;
      ids = ids_next;
    }
    if (!ok) {
      // let every copy already issued land before the CTA can exit
      const uint32_t first = item > (uint32_t)S::STAGES ? item - S::STAGES : 0;
      for (uint32_t it = first; it < item; ++it) wait_drain(full(it % S::STAGES), (it / S::STAGES) & 1u);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // Control flow is the same in every consumer warp (the named barrier below
  // counts all four); a warp whose wait gave up only skips its arithmetic.
  bool ok = true;
  uint32_t item = 0;
  // The query rows of a pair are read one pair ahead into registers (element
  // threadIdx.x + 128 i of the group's MQ x D), so no pair waits for them.
  float qn[QPT];
  load_q(blockIdx.x, threadIdx.x, qn);
  for (int pr = blockIdx.x; pr < pairs; pr += gridDim.x) {
    int seq, g, h0, nq, nblk;
    const int L = decode(pr, seq, g, h0, nq, nblk);
    T* out = static_cast<T*>(p.out) + ((size_t)seq * p.num_query_heads + h0) * D;
    named_bar_sync(1, 32 * kConsumers);  // the previous pair's merge has read shared memory
#pragma unroll
    for (int i = 0; i < QPT; ++i) {
      const int e = threadIdx.x + i * 32 * kConsumers;
      if (e < MQ * D) s_q[e / D][e % D + (e % D >= D / 2 ? 4 : 0)] = qn[i];
    }
    named_bar_sync(1, 32 * kConsumers);
    load_q(pr + (int)gridDim.x, threadIdx.x, qn);  // the next pair's query, in flight now
    float m[MQ], l[MQ], o[MQ][DPL];
#pragma unroll
    for (int hh = 0; hh < MQ; ++hh) {
      m[hh] = -INFINITY;
      l[hh] = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[hh][e] = 0.f;
    }
    // this warp's blocks: stream items item + jb with (item + jb) mod 4 == warp
    const int jb0 = (warp - (int)(item % kConsumers) + kConsumers) % kConsumers;
    for (int jb = jb0; jb < nblk; jb += kConsumers) {
      const uint32_t it = item + (uint32_t)jb;
      const int s = it % S::STAGES;
      if (ok) {
        const bool w = wait_bounded(full(s), (it / S::STAGES) & 1u, abort_flag, p.status,
                                    kStatusTimeoutSoftmax);
        ok = __all_sync(0xffffffffu, w);
      }
      if (!ok || !blk_ok[s]) {
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(empty(s));
        continue;
      }
      block_step(s, s_q, jb, L, m, l, o);
    }
    item += (uint32_t)nblk;

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
      for (int e = 0; e < DPL; ++e) s_o[warp][hh][e * 32 + lane] = o[hh][e];
    named_bar_sync(1, 32 * kConsumers);
    for (int i = threadIdx.x; i < nq * D; i += 32 * kConsumers) {
      const int hh = i / D, d = i % D;
      float mm = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) mm = fmaxf(mm, s_m[w][hh]);
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        if (s_m[w][hh] == -INFINITY) continue;  // a warp that saw no block
        const float f = ex2(s_m[w][hh] - mm);
        num += f * s_o[w][hh][d];
        den += f * s_l[w][hh];
      }
      out[i] = from_f32<T>(den > 0.f ? num / den : 0.f);
    }
  }
}

template <int D, typename T, int MQ, bool WPP>
cudaError_t launch_form(const PagedParams& p, cudaStream_t stream) {
  const int ngroups = (p.qpk + MQ - 1) / MQ;
  const long long pairs = (long long)p.num_seqs * p.num_kv_heads * ngroups;
  using S = PagedSmem<D, MQ, WPP>;
  auto kern = paged_decode_kernel<D, T, MQ, WPP>;
  // per device: the shared-memory opt-in and the resident CTAs per SM
  static int resident[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (resident[dev] == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::BYTES);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, S::BYTES);
    if (e != cudaSuccess) return e;
    resident[dev] = n > 0 ? n : 1;
  }
  const long long grid = std::min<long long>(WPP ? (pairs + kConsumers - 1) / kConsumers : pairs,
                                             (long long)p.sm_count * resident[dev]);
  kern<<<(unsigned)grid, kThreads, S::BYTES, stream>>>(p);
  return cudaGetLastError();
}

// Warp per pair when the block table is short and every consumer warp of a
// full grid gets a pair; otherwise the four consumer warps share each pair.
template <int D, typename T, int MQ>
cudaError_t launch_mq(const PagedParams& p, cudaStream_t stream) {
  const int ngroups = (p.qpk + MQ - 1) / MQ;
  const long long pairs = (long long)p.num_seqs * p.num_kv_heads * ngroups;
  if (pairs <= 0) return cudaSuccess;
  if (pairs > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (p.max_blocks <= kWppMaxBlocks && pairs >= (long long)kConsumers * p.sm_count &&
      pairs < (1LL << 30))
    return launch_form<D, T, MQ, true>(p, stream);
  return launch_form<D, T, MQ, false>(p, stream);
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
