// head_dim 256: the packed variable-length attention forward of
// attn_varlen_kernels.cu (the same operation, plan, work units, workspace and
// status word) with a schedule that fits a 256-column accumulator.
//
// Two 128-row Q tiles need 2 x 256 TMEM columns for O alone, so a CTA
// computes the two Q tiles of a unit one after the other.  TMEM (512
// columns) holds, for the current tile:
//   Qt [0, 128)    the Q tile (bf16 pairs), the A operand of S = Q K^T
//   O  [128, 384)  the fp32 output accumulator
//   S0 [384, 448), S1 [448, 512)  two score buffers of 64 keys; P(j) (bf16
//                  pairs) overwrites the first 32 columns of its S buffer
// With Q in TMEM both products read only their B operand from shared memory
// (S: K, 64 x 16 per step; P.V: V, 16 x 256 per step), so the tensor pipe,
// not shared memory, bounds them.  The MMA warp issues
//   S(0) S(1) | P(0).V(0) S(2) | P(1).V(1) S(3) | ...
// S(j + 2) reuses the buffer of S(j)/P(j) and is issued right behind
// P(j).V(j) (tcgen05.mma from one thread executes in issue order), so the
// softmax of key tile j + 1 overlaps P(j).V(j).
//
// Warps: 0-3 softmax (one row per thread; they also copy each Q tile from
// shared memory into TMEM), 4 TMA producer, 5 MMA issuer and TMEM owner.
// Every wait is bounded like in the other kernel.  Units are never split
// along keys (the partial rows would not fit the split region).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_varlen_device.cuh"
#include "attn_varlen_internal.h"
#include "ptx.cuh"

namespace avp {

namespace {

namespace d256 {
constexpr int D = 256;
constexpr int KN = 64;                         // keys per K/V tile
#ifndef ATTN_VARLEN_KV_STAGES_256
#define ATTN_VARLEN_KV_STAGES_256 4
#endif
constexpr int STAGES = ATTN_VARLEN_KV_STAGES_256;
constexpr int kLoadWarp = 4, kMmaWarp = 5;
constexpr int THREADS = 32 * 6;
constexpr uint32_t BOX_COLS = 64;              // 128-byte swizzled boxes of 64 columns
constexpr uint32_t Q_BOX = kBlockM * BOX_COLS * 2;   // 16 KB
constexpr uint32_t Q_BYTES = 4 * Q_BOX;              // 64 KB
constexpr uint32_t KV_BOX = KN * BOX_COLS * 2;       // 8 KB
constexpr uint32_t KV_BYTES = 4 * KV_BOX;            // 32 KB
constexpr uint32_t Q_OFF = 0;
constexpr uint32_t KV_OFF = Q_BYTES;
constexpr uint32_t BAR_OFF = KV_OFF + STAGES * KV_BYTES;
constexpr int B_Q_FULL = 0, B_Q_EMPTY = 1, B_QT_FULL = 2, B_KV_FULL = 3,
              B_KV_EMPTY = B_KV_FULL + STAGES, B_S_FULL = B_KV_EMPTY + STAGES,
              B_P_FULL = B_S_FULL + 2, B_PV_DONE = B_P_FULL + 1, B_O_FREE = B_PV_DONE + 1,
              B_DRAIN = B_O_FREE + 1, B_ITEM_FULL = B_DRAIN + 1,
              B_ITEM_EMPTY = B_ITEM_FULL + kItemDepth, NUM_BARS = B_ITEM_EMPTY + kItemDepth;
constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;
constexpr uint32_t SMEM_BYTES = MISC_OFF + 8 + 4 * kItemDepth + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory above the sm_103 per-block limit");
constexpr int ITEM_CONSUMERS = 5;              // 4 softmax warps + the MMA warp
constexpr uint32_t QT_COL = 0, O_COL = 128, S_COL = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t SBO = 8 * BOX_COLS * 2;     // 8-row group stride of a 128B-swizzled box

// The i-th K/V tile (of 2n) a Q tile with n key tiles puts into the ring, in
// the order the MMA warp uses them: K0 K1 | V0 K2 | V1 K3 | ... | V(n-2) V(n-1)
// (n = 1: K0 V0).  Returns true for a V tile; j = key tile.
__device__ __forceinline__ bool kv_tile(int i, int n, int& j) {
  if (i == 0) { j = 0; return false; }
  if (n == 1) { j = 0; return true; }
  if (i == 1) { j = 1; return false; }
  if (i >= 2 * n - 2) { j = i - n; return true; }
  const int u = i - 2;
  if (u & 1) { j = (u >> 1) + 2; return false; }
  j = u >> 1;
  return true;
}
}  // namespace d256

}  // namespace

__global__ void __launch_bounds__(d256::THREADS, 1)
    attn_varlen_fwd_d256_kernel(const __grid_constant__ FwdParams p) {
  using namespace d256;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  const uint32_t sQ = base + Q_OFF;
  const uint32_t sKV = base + KV_OFF;
  auto bar = [&](int i) -> uint32_t { return base + BAR_OFF + 8u * (uint32_t)i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base_ptr + MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + MISC_OFF + 4);
  volatile int* item_ring = reinterpret_cast<volatile int*>(base_ptr + MISC_OFF + 8);
  auto next_item = [&](int k) -> int {
    const uint32_t islot = k % kItemDepth, iuse = k / kItemDepth;
    const bool w = wait_bounded(bar(B_ITEM_FULL + islot), iuse & 1u, abort_flag, p.status,
                                kStatusTimeoutItem);
    if (!__all_sync(0xffffffffu, w)) return -1;
    const int u = item_ring[islot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar(B_ITEM_EMPTY + islot));
    return u;
  };
  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);

  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    mbar_init(bar(B_Q_EMPTY), kBlockM);
    mbar_init(bar(B_QT_FULL), kBlockM);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(B_KV_FULL + s), 1);
      mbar_init(bar(B_KV_EMPTY + s), 1);
    }
    mbar_init(bar(B_S_FULL + 0), 1);
    mbar_init(bar(B_S_FULL + 1), 1);
    mbar_init(bar(B_P_FULL), kBlockM);
    mbar_init(bar(B_PV_DONE), 1);
    mbar_init(bar(B_O_FREE), kBlockM);
    mbar_init(bar(B_DRAIN), 1);
    for (int i = 0; i < kItemDepth; ++i) {
      mbar_init(bar(B_ITEM_FULL + i), 1);
      mbar_init(bar(B_ITEM_EMPTY + i), ITEM_CONSUMERS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(base + MISC_OFF, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  grid_wait_prerequisite();
  const WsLayout L = ws_layout(p.num_seqs);
  const int num_units = reinterpret_cast<const int*>(p.ws)[1];
  const int num_items = reinterpret_cast<const int*>(p.ws)[2];
  const int split_start = reinterpret_cast<const int*>(p.ws)[3];
  const int32_t* order = reinterpret_cast<const int32_t*>(p.ws + L.order);
  const int32_t* prefix = reinterpret_cast<const int32_t*>(p.ws + L.prefix);
  auto decode = [&](int u) {
    return decode_item(u, order, prefix, p.num_seqs, p.cu_q, p.cu_k, KN, split_start, num_units,
                       nullptr, p.causal != 0, p.head_begin);
  };
  // key tiles of Q tile t of a unit (0: the tile has no row or sees no key)
  auto tile_steps = [](const UnitInfo& ui, int t) { return t == 0 ? ui.nkv0 : (ui.t1 ? ui.nkv : 0); };

  if (warp == kLoadWarp) {
    // ------------------------------------------------------ TMA producer
    const uint32_t leader = elect_one();
    const int leader_lane = __ffs(__ballot_sync(0xffffffffu, leader != 0)) - 1;
    uint32_t kv_item = 0, q_use = 0;
    bool ok = true;
    auto wait_ = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu,
                        wait_bounded(b, parity, abort_flag, p.status, kStatusTimeoutLoad));
    };
    int pending = 0;
    for (int k = 0; ok; ++k) {
      const int u = k == 0 ? (int)blockIdx.x
                           : (int)gridDim.x + __shfl_sync(0xffffffffu, pending, leader_lane);
      const uint32_t islot = k % kItemDepth, iuse = k / kItemDepth;
      if (!(ok = wait_(bar(B_ITEM_EMPTY + islot), (iuse & 1u) ^ 1u))) break;
      if (leader) item_ring[islot] = u;
      __syncwarp();
      if (leader) mbar_arrive(bar(B_ITEM_FULL + islot));
      if (u >= num_items) break;
#if !ATTN_VARLEN_LATE_CLAIM
      if (leader) pending = atomicAdd(p.status + kHdrNextItem, 1);
#endif
      const UnitInfo ui = decode(u);
      if (ui.nkv == 0) {
#if ATTN_VARLEN_LATE_CLAIM
        if (leader) pending = atomicAdd(p.status + kHdrNextItem, 1);
#endif
        continue;
      }
      const uint8_t* mq = p.ws + L.maps + (size_t)ui.seq * kMapsPerSeq * kMapBytes;
      const uint8_t* mk = mq + kMapBytes;
      const uint8_t* mv = mq + 2 * kMapBytes;
      if (leader) {
        tmap_acquire(mq);
        tmap_acquire(mk);
        tmap_acquire(mv);
      }
      __syncwarp();
      for (int t = 0; ok && t < 2; ++t) {
        const int n = tile_steps(ui, t);
        if (n == 0) continue;
        if (!(ok = wait_(bar(B_Q_EMPTY), (q_use & 1u) ^ 1u))) break;
        ++q_use;
        mbar_arrive_expect_tx_if(leader, bar(B_Q_FULL), Q_BYTES);
#pragma unroll
        for (int b = 0; b < 4; ++b)
          tma_load_3d_if(leader, sQ + b * Q_BOX, mq, bar(B_Q_FULL), b * BOX_COLS, ui.head,
                         ui.q0 + t * kBlockM);
        for (int i = 0; i < 2 * n; ++i) {
          int j;
          const bool is_v = kv_tile(i, n, j);
          const uint32_t stage = kv_item % STAGES, use = kv_item / STAGES;
          if (!(ok = wait_(bar(B_KV_EMPTY + stage), (use & 1u) ^ 1u))) break;
#if ATTN_VARLEN_TEST_HOOKS
          const uint32_t issue = (p.test_withhold && blockIdx.x == 0 && kv_item == 0) ? 0u : leader;
#else
          const uint32_t issue = leader;
#endif
          mbar_arrive_expect_tx_if(issue, bar(B_KV_FULL + stage), KV_BYTES);
          const uint32_t dst = sKV + stage * KV_BYTES;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            tma_load_3d_if(issue, dst + b * KV_BOX, is_v ? mv : mk, bar(B_KV_FULL + stage),
                           b * BOX_COLS, ui.head, (ui.jb + j) * KN);
          ++kv_item;
        }
      }
#if ATTN_VARLEN_LATE_CLAIM
      // the next item is claimed once this one's last K/V load is out
      if (leader) pending = atomicAdd(p.status + kHdrNextItem, 1);
#endif
    }
    if (!ok) {
      // let every copy already issued land before the CTA can exit
      if (q_use > 0) wait_drain(bar(B_Q_FULL), (q_use - 1) & 1u);
      const uint32_t first = kv_item > (uint32_t)STAGES ? kv_item - STAGES : 0;
      for (uint32_t it = first; it < kv_item; ++it)
        wait_drain(bar(B_KV_FULL + it % STAGES), (it / STAGES) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------- MMA issuer
    const uint32_t leader = elect_one();
    constexpr uint32_t idesc_s = idesc_bf16_f32(kBlockM, KN, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kBlockM, D, false, true);
    const uint64_t dk0 = smem_desc(sKV, 16, SBO, kSwizzle128B);
    const uint64_t dv0 = smem_desc(sKV, KV_BOX, SBO, kSwizzle128B);
    uint32_t kv_item = 0, qt_use = 0, p_use = 0, s_cnt = 0, tiles = 0;
    bool ok = true, issued = false;
    auto wait_ = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu,
                        wait_bounded(b, parity, abort_flag, p.status, kStatusTimeoutMma));
    };
    auto kv_full = [&]() -> bool {
      return wait_(bar(B_KV_FULL + kv_item % STAGES), (kv_item / STAGES) & 1u);
    };
    // S(j) into buffer s_cnt % 2: Q from TMEM (A), K from the ring (B)
    auto issue_s = [&]() -> bool {
      if (!kv_full()) return false;
      tc_fence_after();
      const uint32_t stage = kv_item % STAGES;
      const uint64_t kb = dk0 + ((stage * KV_BYTES) >> 4);
      const uint32_t d = tmem + S_COL + 64u * (s_cnt & 1u);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t box = (uint32_t)(k / 4), col_b = (uint32_t)(k % 4) * 32u;
        mma_ts_if(leader, d, tmem + QT_COL + 8u * k, kb + ((box * KV_BOX + col_b) >> 4), idesc_s,
                  k > 0 ? 1u : 0u);
      }
      mma_commit_if(leader, bar(B_S_FULL + (s_cnt & 1u)));
      mma_commit_if(leader, bar(B_KV_EMPTY + stage));
      ++s_cnt;
      ++kv_item;
      return true;
    };
    // O (+)= P(j) V(j): P from the first 32 columns of S buffer `buf`
    auto issue_pv = [&](uint32_t buf, bool acc) -> bool {
      if (!wait_(bar(B_P_FULL), p_use & 1u)) return false;
      ++p_use;
      if (!kv_full()) return false;
      tc_fence_after();
      const uint32_t stage = kv_item % STAGES;
      const uint64_t vb = dv0 + ((stage * KV_BYTES) >> 4);
      const uint32_t a = tmem + S_COL + 64u * buf;
#pragma unroll
      for (int k = 0; k < KN / 16; ++k)
        mma_ts_if(leader, tmem + O_COL, a + 8u * k, vb + ((k * 16 * BOX_COLS * 2) >> 4), idesc_pv,
                  (acc || k > 0) ? 1u : 0u);
      mma_commit_if(leader, bar(B_PV_DONE));
      mma_commit_if(leader, bar(B_KV_EMPTY + stage));
      ++kv_item;
      return true;
    };
    for (int k = 0; ok; ++k) {
      const int u = next_item(k);
      if (u < 0 || u >= num_items) break;
      const UnitInfo ui = decode(u);
      for (int t = 0; ok && t < 2; ++t) {
        const int n = tile_steps(ui, t);
        if (n == 0) continue;
        // the tile's Q in TMEM; O read out by the softmax after the last tile
        if (!(ok = wait_(bar(B_QT_FULL), qt_use & 1u))) break;
        ++qt_use;
        if (tiles > 0 && !(ok = wait_(bar(B_O_FREE), (tiles - 1) & 1u))) break;
        ++tiles;
        issued = true;
        const uint32_t buf0 = s_cnt & 1u;  // buffer of S(0) of this tile
        if (!(ok = issue_s())) break;
        if (n > 1 && !(ok = issue_s())) break;
        for (int j = 0; ok && j < n; ++j) {
          if (!(ok = issue_pv((buf0 + (uint32_t)j) & 1u, j > 0))) break;
          if (j + 2 < n && !(ok = issue_s())) break;
        }
      }
    }
    if (issued) {
      mma_commit_if(leader, bar(B_DRAIN));
      wait_drain(bar(B_DRAIN), 0);
    }
  } else {
    // --------------------------------------------------------- softmax
    const int r = threadIdx.x & 127;  // row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + lane_off + O_COL;
    const float sl2 = p.scale_log2;
    uint32_t q_use = 0, s_cnt = 0, p_cnt = 0, tiles = 0;
    bool ok = true;
    auto wait_ = [&](uint32_t b, uint32_t parity) -> bool {
      bool w = wait_bounded(b, parity, abort_flag, p.status, kStatusTimeoutSoftmax);
      return __all_sync(0xffffffffu, w);
    };
    for (int k = 0; ok; ++k) {
      const int u = next_item(k);
      if (u < 0 || u >= num_items) break;
      const UnitInfo ui = decode(u);
      for (int t = 0; ok && t < 2; ++t) {
        if (t == 1 && !ui.t1) break;
        const int row = ui.q0 + kBlockM * t + r;
        const bool valid = row < ui.lq;
        uint16_t* orow = p.out + ((size_t)(ui.qbase + row) * p.num_heads + ui.head) * D;
        const int n = tile_steps(ui, t);
        if (n == 0) {
          if (valid) {
#pragma unroll
            for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
          }
          continue;
        }
        const int klim = p.causal ? min(ui.lk, row + 1 + ui.coff) : ui.lk;
        // ---- Q tile: shared memory (four 128B-swizzled boxes) -> TMEM
        if (!(ok = wait_(bar(B_Q_FULL), q_use & 1u))) break;
        ++q_use;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint8_t* rowp = base_ptr + Q_OFF + b * Q_BOX + r * 128;
          uint32_t qv[32];
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            // 16-byte chunk ch of the row sits at chunk ch ^ (row mod 8)
            const uint4 v = *reinterpret_cast<const uint4*>(rowp + ((ch ^ (r & 7)) << 4));
            qv[4 * ch] = v.x;
            qv[4 * ch + 1] = v.y;
            qv[4 * ch + 2] = v.z;
            qv[4 * ch + 3] = v.w;
          }
          tmem_st32(tmem + lane_off + QT_COL + 32u * b, qv);
        }
        // the reads above come before the next TMA write of the Q buffer
        fence_proxy_async_smem();
        mbar_arrive(bar(B_Q_EMPTY));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_QT_FULL));
        float m = 0.f, l = 0.f;
        for (int j = 0; j < n; ++j) {
          const uint32_t buf = s_cnt & 1u;
          if (!(ok = wait_(bar(B_S_FULL + buf), (s_cnt >> 1) & 1u))) break;
          ++s_cnt;
          tc_fence_after();
          const uint32_t tS = tmem + lane_off + S_COL + 64u * buf;
          uint32_t s[KN];
          tmem_ld_cols<KN>(tS, s);
          tmem_wait_ld();
          reg_fence(s, 0, KN);
          const int lim = klim - (ui.jb + j) * KN;
          if (__any_sync(0xffffffffu, lim < KN)) {
#pragma unroll
            for (int c = 0; c < KN; ++c)
              if (c >= lim) s[c] = __float_as_uint(-INFINITY);
          }
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
          for (int c = 0; c < KN; c += 8) {
            mx0 = fmax3(mx0, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
            mx1 = fmax3(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
            mx2 = fmax3(mx2, __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
            mx3 = fmax3(mx3, __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
          }
          const float mxs = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
          if (j == 0) {
            m = mxs == -INFINITY ? 0.f : mxs;
          } else {
            const bool need = mxs > m + kRescaleThreshold;
            if (__any_sync(0xffffffffu, need)) {
              // O must hold P(j-1) V(j-1) before it is rescaled
              if (!(ok = wait_(bar(B_PV_DONE), (p_cnt - 1) & 1u))) break;
              tc_fence_after();
              const float alpha = need ? ex2(m - mxs) : 1.0f;
              if (need) m = mxs;
              l *= alpha;
#pragma unroll 4
              for (int c = 0; c < D; c += 16) {
                uint32_t o[16];
                tmem_ld16(tO + c, o);
                tmem_wait_ld();
                reg_fence(o, 0, 16);
#pragma unroll
                for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tmem_st16(tO + c, o);
              }
              tmem_wait_st();
            }
          }
          // P(j) overwrites the first 32 columns of its S buffer: S(j) is in
          // registers, and P(j-2), which lived there, was read by P(j-2).V(j-2)
          // before S(j) was written (the MMAs of one thread run in order)
          const float2 c2 = make_float2(sl2, sl2);
          const float2 nm2 = make_float2(-m, -m);
          float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
          uint32_t pk[KN / 2];
#pragma unroll
          for (int c = 0; c < KN / 2; c += 2) {
            float2 a = __ffma2_rn(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])),
                                  c2, nm2);
            float2 b = __ffma2_rn(make_float2(__uint_as_float(s[2 * c + 2]),
                                              __uint_as_float(s[2 * c + 3])), c2, nm2);
            a.x = ex2(a.x);
            a.y = ex2(a.y);
            b.x = ex2(b.x);
            b.y = ex2(b.y);
            acc0 = __fadd2_rn(acc0, a);
            acc1 = __fadd2_rn(acc1, b);
            pk[c] = pack_bf16x2(a.x, a.y);
            pk[c + 1] = pack_bf16x2(b.x, b.y);
          }
          // Observe the completion of P(j-1).V(j-1) before P(j) is handed
          // over: every PV_DONE phase is then waited for in order, so a
          // parity wait can never match a phase two completions old (the
          // epilogue's and the rescale's waits rely on it).
          if (j > 0) {
            if (!(ok = wait_(bar(B_PV_DONE), (p_cnt - 1) & 1u))) break;
            tc_fence_after();
          }
          tmem_st32(tS, pk);
          tmem_wait_st();
          l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
          tc_fence_before();
          mbar_arrive(bar(B_P_FULL));
          ++p_cnt;
        }
        if (!ok) break;
        // epilogue: O / l -> bf16 -> out, then O is free for the next tile
        if (!(ok = wait_(bar(B_PV_DONE), (p_cnt - 1) & 1u))) break;
        tc_fence_after();
        const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll 4
        for (int c = 0; c < D; c += 16) {
          uint32_t o[16];
          tmem_ld16(tO + c, o);
          tmem_wait_ld();
          reg_fence(o, 0, 16);
          if (valid) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
            uint4* o4 = reinterpret_cast<uint4*>(orow + c);
            o4[0] = make_uint4(w[0], w[1], w[2], w[3]);
            o4[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(B_O_FREE));
        ++tiles;
      }
    }
    (void)tiles;
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Launched as a programmatic dependent of the plan kernel, like the other
// head dims.
cudaError_t launch_fwd_d256(const FwdParams& p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)d256::THREADS);
  cfg.dynamicSmemBytes = d256::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_varlen_fwd_d256_kernel, p);
}

cudaError_t prepare_fwd_d256() {
  return cudaFuncSetAttribute(attn_varlen_fwd_d256_kernel,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)d256::SMEM_BYTES);
}

int fwd_threads_d256() { return d256::THREADS; }
size_t fwd_smem_bytes_d256() { return d256::SMEM_BYTES; }
int kv_tile_rows_d256() { return d256::KN; }

}  // namespace avp
