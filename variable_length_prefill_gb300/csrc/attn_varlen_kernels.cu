// Packed variable-length, non-causal attention forward for sm_103a.
//
// What is computed: atrex-bench "attention_forward" (page #001, reference.py,
// Model.forward) -- per non-empty query sequence and head,
// softmax(Q K^T * head_dim^-1/2) V over that sequence's keys, bf16 in, bf16
// out, fp32 accumulation.
//
// Two kernels run back to back on the caller's stream:
//
//  1. plan (one CTA): reads cu_seqlens on the device, counts the work units
//     of every sequence (a unit is one head x 256 query rows), orders the
//     sequences longest-key-range first, writes the prefix sums of the units
//     in that order, and writes the q, k, v and out tensor maps of every
//     sequence (box A and box B) by patching host-encoded templates (global
//     address = the sequence's first row, row extent = the sequence length)
//     so that TMA zero-fills every row past the end of a sequence and clips
//     stores there.  The template is chosen by the sequence's byte size (see
//     kMapLargeBytes), which makes each patched map identical to the one the
//     host encoder would produce.  It then plans the key-range split of the
//     units at the end of the schedule (step 4 of the kernel).
//
//  2. fwd (persistent, one CTA per SM): the first item of a CTA is its
//     blockIdx.x, later ones come from a workspace counter, whole units in
//     longest-first order and then the split units' chunks.  Warp roles:
//       warps 0-3  softmax for Q tile 0 (TMEM lanes 0-127 = its 128 rows)
//       warps 4-7  softmax for Q tile 1
//       warp  8    TMA producer: Q tiles, then a ring of K and V tiles
//       warp  9    TMEM owner and tcgen05.mma issuer (head_dim 128: both
//                  tiles; head_dim 64-96: tile 0)
//       warp 10    head_dim 64-96 only: tcgen05.mma issuer for tile 1
//     Softmax is an online exp2 softmax, one row per thread, with a lazy
//     rescale: the running max is only raised (and O rescaled in TMEM) when a
//     row's new max exceeds it by more than kRescaleThreshold (log2 units).
//     P (bf16, packed in pairs) is the A operand of the P.V MMA straight from
//     TMEM.
//
//     head_dim 128 (TMEM: S0 [0,128), S1 [128,256), O0 [256,384),
//     O1 [384,512)): key tiles of 128; P overwrites the first 64 columns of
//     its S; one issuer alternates the tiles,
//       S0(0) S1(0) | PV0(j) S0(j+1) PV1(j) S1(j+1) | ...
//     so each softmax warpgroup has the other tile's two MMAs to hide behind;
//     the tensor pipe is the bound.
//
//     head_dim 72 (TMEM: S0 [0,112), S1 [112,224), P0 [224,280),
//     P1 [288,344), O0 [352,432), O1 [432,512)): key tiles of 112 so that P
//     fits in columns of its own; S_t(j+1) is issued as soon as the softmax
//     has read S_t(j) into registers (S_FREE), not after P_t(j).V(j); each
//     tile has its own issuer, so neither tile's S waits in one in-order
//     program behind the other tile's P.V.
//
// Head dims 64, 72, 80, 96 and 128 run here (256 has a kernel of its own).
// Box A holds columns 0-63 with 128-byte swizzle.  For 72, box B is an
// unswizzled 8-column box (columns 64-71); a zero region in shared memory
// supplies columns 72-79 of Q and K to the K = 80 MMA step, and a ones region
// makes V's padding column 72 read 1.0, so P.V also sums each row of P.  For
// 80, 96 and 128 box B is a second 64-column swizzled box (zero-filled past
// head_dim).  Padded output columns are never stored.  The scale always uses
// the true head_dim.
//
// Every mbarrier wait is bounded in time; a wait that runs out records a bit
// in the workspace status word, raises a CTA-wide abort flag, and the CTA
// drains its outstanding copies and MMAs (again with a bound), frees TMEM
// and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "attn_varlen_device.cuh"
#include "attn_varlen_internal.h"
#include "ptx.cuh"

namespace avp {

namespace {

constexpr uint32_t kTmemCols = 512;
// S(j+1) of a tile overwrites the TMEM columns that P(j) of the same tile
// occupies.  tcgen05.mma operations issued by one thread execute in issue
// order, so S(j+1) is queued right behind P(j).V(j); with kStrictPvWait the
// MMA warp instead waits for P(j).V(j) to complete before issuing S(j+1).
#ifndef ATTN_VARLEN_STRICT_PV_WAIT
#define ATTN_VARLEN_STRICT_PV_WAIT 0
#endif
constexpr bool kStrictPvWait = ATTN_VARLEN_STRICT_PV_WAIT != 0;
// Test builds only (never the product library): with FwdParams::test_withhold
// set, CTA 0's producer neither issues nor announces its first K/V tile, so
// the MMA warp's wait on that slot runs out and the give-up path (status
// bit, abort flag, drain, TMEM free) runs with no copy in flight on it.
#ifndef ATTN_VARLEN_TEST_HOOKS
#define ATTN_VARLEN_TEST_HOOKS 0
#endif
// The plan kernel is itself a programmatic dependent of the previous
// attention kernel on the stream: it may be resident before that kernel ends
// and waits for it (griddepcontrol.wait) before it reads or writes anything.
#ifndef ATTN_VARLEN_PLAN_PDL
#define ATTN_VARLEN_PLAN_PDL 1
#endif
#ifndef ATTN_VARLEN_TAIL_SPLIT
#define ATTN_VARLEN_TAIL_SPLIT 1
#endif
// The tail is found by simulating the list schedule (else: the grid's last
// partial wave).
#ifndef ATTN_VARLEN_SIM_TAIL
#define ATTN_VARLEN_SIM_TAIL 1
#endif
#ifndef ATTN_VARLEN_MIN_CHUNK
#define ATTN_VARLEN_MIN_CHUNK 32
#endif
// A split pays off only if it shortens the tail by more than the partial
// write and merge cost, counted in key tiles of work.
constexpr int kMergeTiles = 8;
// A chunk of a split unit holds at least this many key tiles (its partial
// write and the merge cost several).
constexpr int kMinChunkTiles = ATTN_VARLEN_MIN_CHUNK;
// A tail with at least this many key tiles per CTA is cut into up to
// kSplitWaves chunks per CTA; a shorter one into at most one per CTA.
#ifndef ATTN_VARLEN_FINE_TAIL
#define ATTN_VARLEN_FINE_TAIL 192
#endif
constexpr int kFineTailTiles = ATTN_VARLEN_FINE_TAIL;
// The plan's model of a unit's cost beyond its key tiles (Q load, epilogue),
// in key tiles.
constexpr int kUnitCostTiles = 2;
// Limits of the plan's list-schedule simulation (steps, CTAs).
constexpr int kSimMaxSteps = 128;
constexpr int kSimMaxGrid = 256;


// K/V ring depth per head_dim (shared memory: head_dim 72 holds 2 x 18 KB of
// Q and 16 KB per stage, head_dim 128 2 x 32 KB and 32 KB per stage)
// head_dim 72: the row sum of P comes out of the P.V product as O column 72
// (V's padding column 72 reads 1.0 from a "ones" region), instead of being
// added up by the softmax threads.
#ifndef ATTN_VARLEN_SUM_IN_O
#define ATTN_VARLEN_SUM_IN_O 1
#endif
#ifndef ATTN_VARLEN_KV_STAGES_72
#define ATTN_VARLEN_KV_STAGES_72 8
#endif
#ifndef ATTN_VARLEN_KV_STAGES_128
#define ATTN_VARLEN_KV_STAGES_128 4
#endif

// Share of the softmax's exponentials computed on the FMA pipe
// (exp2_poly2) instead of the MUFU unit: POLY of every 7 groups of four
// columns.  Off by default: on GB300 the MUFU unit retires ex2 fast enough
// that the softmax is bound by issue slots, and each polynomial costs about
// six instructions against one; 2/7, 3/7 and 4/7 made the head_dim-72
// kernel 13, 21 and 35 % slower.
#ifndef ATTN_VARLEN_POLY_SMALL
#define ATTN_VARLEN_POLY_SMALL 0
#endif
#ifndef ATTN_VARLEN_POLY_128
#define ATTN_VARLEN_POLY_128 0
#endif
constexpr int kPolyDen = 7;

// Per head_dim configuration.  Every head_dim other than 128 runs the
// separate-P, two-issuer schedule; the key tile is the largest multiple of 16
// whose S, P and O columns for two Q tiles fit the 512 TMEM columns
// (2 KN + 2 KN/2 + 2 DP <= 512, with P placed at 2 KN + 64 t).
template <int D>
struct Cfg;
template <>
struct Cfg<64> {
  static constexpr int DP = 64;
  static constexpr int BW = 64;    // one 64-column box
  static constexpr int WB = 0;    // one box
  static constexpr int KN = 128;
  static constexpr bool PSEP = true;
  static constexpr int ISSUERS = 2;
  static constexpr int STAGES = 6;  // 16 KB per K or V tile
  static constexpr uint32_t SWZ = kSwizzle128B;
  static constexpr int POLY = ATTN_VARLEN_POLY_SMALL;
};
template <>
struct Cfg<80> {
  static constexpr int DP = 80;
  static constexpr int BW = 64;    // second box: columns 64-79 and zero fill
  static constexpr int WB = 64;   // box B: columns 64-127, 128-byte swizzle
  static constexpr int KN = 112;
  static constexpr bool PSEP = true;
  static constexpr int ISSUERS = 2;
  static constexpr int STAGES = 4;
  static constexpr uint32_t SWZ = kSwizzle128B;
  static constexpr int POLY = ATTN_VARLEN_POLY_SMALL;
};
template <>
struct Cfg<96> {
  static constexpr int DP = 96;
  static constexpr int BW = 64;    // second box: columns 64-95 and zero fill
  static constexpr int WB = 64;   // box B: columns 64-127, 128-byte swizzle
  static constexpr int KN = 96;
  static constexpr bool PSEP = true;
  static constexpr int ISSUERS = 2;
  static constexpr int STAGES = 4;
  static constexpr uint32_t SWZ = kSwizzle128B;
  static constexpr int POLY = ATTN_VARLEN_POLY_SMALL;
};
template <>
struct Cfg<72> {
  static constexpr int DP = 80;    // padded head_dim (MMA K and N multiple of 16)
  static constexpr int BW = 64;    // box A: columns 0-63, 128-byte swizzle
  static constexpr int WB = 8;     // box B: columns 64-71, unswizzled; the MMAs take
                                   // columns 72-79 from a zero region in shared memory
  static constexpr int KN = 112;   // keys per K/V tile
  static constexpr bool PSEP = true;  // P in TMEM columns of its own
  static constexpr int ISSUERS = 2;   // one MMA-issuing warp per Q tile
  static constexpr int STAGES = ATTN_VARLEN_KV_STAGES_72;
  static constexpr uint32_t SWZ = kSwizzle128B;
  static constexpr int POLY = ATTN_VARLEN_POLY_SMALL;
};
template <>
struct Cfg<128> {
  static constexpr int DP = 128;
  static constexpr int BW = 64;
  static constexpr int WB = 64;   // box B: columns 64-127, 128-byte swizzle
  static constexpr int KN = 128;
  static constexpr bool PSEP = false;  // P overwrites the first half of S
  static constexpr int ISSUERS = 1;    // one MMA-issuing warp for both Q tiles
  static constexpr int STAGES = ATTN_VARLEN_KV_STAGES_128;
  static constexpr uint32_t SWZ = kSwizzle128B;
  static constexpr int POLY = ATTN_VARLEN_POLY_128;
};

template <int D>
struct Geometry {
  static constexpr int DP = Cfg<D>::DP;
  static constexpr int BW = Cfg<D>::BW;
  static constexpr int KN = Cfg<D>::KN;
  static constexpr bool PSEP = Cfg<D>::PSEP;
  static constexpr int ISSUERS = Cfg<D>::ISSUERS;
  static_assert(PSEP || ISSUERS == 1, "two issuers need P in columns of its own");
  static constexpr int SM_WARPS = 8;             // softmax warps: 2 Q tiles x 4
  static constexpr int LOAD_WARP = SM_WARPS;     // TMA producer
  static constexpr int MMA_WARP = SM_WARPS + 1;  // first MMA issuer (and TMEM owner)
  static constexpr int THREADS = 32 * (MMA_WARP + ISSUERS);
  static constexpr int NB = (DP + BW - 1) / BW;             // boxes per tile
  static constexpr int STAGES = Cfg<D>::STAGES;
  static constexpr uint32_t SWZ = Cfg<D>::SWZ;
  static constexpr int POLY = Cfg<D>::POLY;
  static_assert(POLY >= 0 && POLY <= kPolyDen, "polynomial share");
  // Box B (columns 64 and up) is either a second 64-column, 128-byte
  // swizzled box (ZB false) or, for head_dim 72, an unswizzled 8-column box
  // (ZB true) whose 16-byte rows form the core matrices of the MMAs' last
  // 16-column step together with a 16-byte-wide zero region (ZERO_OFF):
  // every copied byte is a real input byte, and no TMA zero fill is used.
  static constexpr int WB = Cfg<D>::WB;
  static constexpr bool ZB = WB == 8;
  static_assert(NB == 1 ? WB == 0 : (WB == BW || (ZB && DP == BW + 16)), "box B");
  static constexpr uint32_t Q_BOX_BYTES = kBlockM * BW * 2;  // box A: 128 rows x BW
  static constexpr uint32_t Q_BOXB_BYTES = NB == 1 ? 0u : kBlockM * WB * 2;
  static constexpr uint32_t Q_LOAD_BYTES = Q_BOX_BYTES + Q_BOXB_BYTES;  // bytes one Q tile copies
  static constexpr uint32_t Q_TILE_BYTES = (Q_LOAD_BYTES + 1023u) / 1024u * 1024u;
  static constexpr uint32_t KV_BOX_BYTES = KN * BW * 2;      // box A: KN keys x BW
  static constexpr uint32_t KV_BOXB_BYTES = NB == 1 ? 0u : KN * WB * 2;
  static constexpr uint32_t KV_LOAD_BYTES = KV_BOX_BYTES + KV_BOXB_BYTES;
  static constexpr uint32_t KV_TILE_BYTES = (KV_LOAD_BYTES + 1023u) / 1024u * 1024u;
  static_assert(KV_BOX_BYTES % 1024 == 0, "128B-swizzled boxes start on 1024-byte boundaries");
  static constexpr uint32_t SBO = 8 * BW * 2;               // 8-row group stride
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t KV_OFF = 2 * Q_TILE_BYTES;
  // zero region: 128 rows x 16 bytes (ZB only)
  static constexpr uint32_t ZERO_OFF = KV_OFF + STAGES * KV_TILE_BYTES;
  static constexpr uint32_t ZERO_BYTES = ZB ? kBlockM * 16u : 0u;
  // LO: O column D (= 72) accumulates sum_k P[r, k], the row sum, because
  // V's padding column 72 reads 1.0 from the ones region (128 rows x 16 B,
  // each row 1.0 then seven zeros) instead of the zero region.
  static constexpr bool LO = ZB && ATTN_VARLEN_SUM_IN_O != 0;
  static constexpr uint32_t ONES_OFF = ZERO_OFF + ZERO_BYTES;
  static constexpr uint32_t ONES_BYTES = LO ? kBlockM * 16u : 0u;
  // Epilogue staging, one region per softmax warp (its 32 output rows): box
  // A as 32 rows x 128 bytes in the 128-byte swizzle of the out map (1024-
  // byte aligned), then, for head_dim 72, box B as 32 rows x 16 bytes.  With
  // a 64-column box B the box-A region is reused once box A's store has read
  // it.
  static constexpr uint32_t STG_A_BYTES = kStoreRows * 128u;
  static constexpr uint32_t STG_B_BYTES = ZB ? kStoreRows * 16u : 0u;
  static constexpr uint32_t STG_WARP = (STG_A_BYTES + STG_B_BYTES + 1023u) / 1024u * 1024u;
  static constexpr uint32_t STG_OFF = (ONES_OFF + ONES_BYTES + 1023u) / 1024u * 1024u;
  static constexpr uint32_t STG_BYTES = SM_WARPS * STG_WARP;
  static constexpr uint32_t BAR_OFF = STG_OFF + STG_BYTES;
  // barrier slots (8 bytes each)
  static constexpr int B_Q_FULL = 0, B_Q_EMPTY = 1, B_KV_FULL = 2, B_KV_EMPTY = 2 + STAGES,
                       B_S_FULL = 2 + 2 * STAGES, B_P_FULL = B_S_FULL + 2,
                       B_PV_DONE = B_P_FULL + 2, B_S_FREE = B_PV_DONE + 2,
                       B_DRAIN = B_S_FREE + 2, B_ITEM_FULL = B_DRAIN + 2,
                       B_ITEM_EMPTY = B_ITEM_FULL + kItemDepth,
                       NUM_BARS = B_ITEM_EMPTY + kItemDepth;
  // tmem slot, abort flag, then the item ring (kItemDepth int32)
  static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = MISC_OFF + 8 + 4 * kItemDepth + 1024;  // + alignment slack
  static constexpr int ITEM_CONSUMERS = SM_WARPS + ISSUERS;  // warps that read each ring entry
  static_assert(SMEM_BYTES <= 232448, "shared memory above the sm_103 per-block limit");
  static constexpr int NK_S = DP / 16;  // K-steps of S = Q K^T
  static constexpr int NK_PV = KN / 16; // K-steps of O += P V
  static_assert(KN % 32 == 0 || KN == 112, "key tile rows: 64, 96, 112 or 128");
  static_assert(KN >= 64 && KN <= 128, "key tile rows");
  static_assert(DP + 2 <= kPartRowMax, "partial row");
  // TMEM columns of S_t, P_t (bf16 pairs) and O_t
  __host__ __device__ static constexpr uint32_t s_col(int t) { return PSEP ? (uint32_t)(t * KN) : 128u * t; }
  __host__ __device__ static constexpr uint32_t p_col(int t) { return PSEP ? 2u * KN + 64u * t : s_col(t); }
  __host__ __device__ static constexpr uint32_t o_col(int t) { return PSEP ? 2u * KN + 128u + DP * t : 256u + 128u * t; }
  static_assert(o_col(1) + DP <= 512, "TMEM columns");
};

// The i-th K/V tile a unit with n key tiles puts into the ring, in the order
// the MMA warp first uses them.  Returns true for a V tile; j = key tile.
//   P aliasing S:  K0 V0 K1 V1 ...            (P_t(j).V(j) precedes S_t(j+1))
//   P separate:    K0 K1 V0 K2 V1 ... K(n-1) V(n-2) V(n-1)
//                  (S_t(j+1) is issued before P_t(j).V(j))
template <bool kPSep>
__device__ __forceinline__ bool kv_item_tile(int i, int n, int& j) {
  if constexpr (!kPSep) {
    j = i >> 1;
    return (i & 1) != 0;
  } else {
    if (i == 0) { j = 0; return false; }
    if (i == 2 * n - 1) { j = n - 1; return true; }
    if (i & 1) { j = (i + 1) >> 1; return false; }
    j = (i - 2) >> 1;
    return true;
  }
}

}  // namespace

// ------------------------------------------------------------------- plan
__global__ void __launch_bounds__(1024, 1) attn_varlen_plan_kernel(const __grid_constant__ PlanParams p) {
  // the attention kernel may start launching now; it waits for this grid to
  // complete before it reads the workspace
  grid_launch_dependents();
#if ATTN_VARLEN_PLAN_PDL
  // the previous attention kernel on the stream (if any) still reads the
  // workspace: nothing is read or written before it has finished
  grid_wait_prerequisite();
#endif
  __shared__ int s_key[kLptMaxSeqs];
  // with at most kLptMaxSeqs sequences the per-sequence lengths, the order
  // and the prefix sums stay in shared memory, so the plan costs one round
  // of global loads (the global copies are written for the attention kernel)
  __shared__ int s_lq[kLptMaxSeqs];
  __shared__ int s_lk[kLptMaxSeqs];
  __shared__ int s_order[kLptMaxSeqs];
  __shared__ int s_pref[kLptMaxSeqs + 1];
  __shared__ int s_warp[32];
  __shared__ int s_carry;
  const int N = p.num_seqs;
  const WsLayout L = ws_layout(N);
  int* hdr = reinterpret_cast<int*>(p.ws);
  // read now, so that the load's latency overlaps the map writes
  const int counters_dirty = p.split_cap > 0 ? hdr[kHdrCountersDirty] : 0;
  int* order = reinterpret_cast<int*>(p.ws + L.order);
  int* prefix = reinterpret_cast<int*>(p.ws + L.prefix);
  const bool lpt = N <= kLptMaxSeqs;
  const int tid = threadIdx.x, nt = blockDim.x;
  auto lq_of = [&](int i) { return lpt ? s_lq[i] : p.cu_q[i + 1] - p.cu_q[i]; };
  auto lk_of = [&](int i) { return lpt ? s_lk[i] : p.cu_k[i + 1] - p.cu_k[i]; };
  auto order_at = [&](int r) { return lpt ? s_order[r] : order[r]; };
  auto prefix_at = [&](int r) { return lpt ? s_pref[r] : prefix[r]; };
  auto units_of = [&](int i) {
    const int lq = lq_of(i);
    return lq > 0 ? p.num_heads * ((lq + kUnitRows - 1) / kUnitRows) : 0;
  };

  // 1. per sequence: lengths, sort key, tensor maps
  bool wrote_map = false;
  if (lpt) {
    for (int i = tid; i < N; i += nt) {
      const int lq = p.cu_q[i + 1] - p.cu_q[i];
      const int lk = p.cu_k[i + 1] - p.cu_k[i];
      s_lq[i] = lq;
      s_lk[i] = lk;
      s_key[i] = lq > 0 ? (lk > 0 ? lk : 0) : -1;
    }
  }
  // one thread per (sequence, map): the q, k, v and out maps of box A and box B
  for (int idx = tid; idx < N * kMapsPerSeq; idx += nt) {
    const int i = idx / kMapsPerSeq, m = idx - i * kMapsPerSeq, t = m % kTensors;
    const int q0 = p.cu_q[i], lq = p.cu_q[i + 1] - q0;
    const int k0 = p.cu_k[i], lk = p.cu_k[i + 1] - k0;
    if (lq > 0 && lk > 0) {
      uint8_t* dst = p.ws + L.maps + (size_t)idx * kMapBytes;
      const bool qrows = t == 0 || t == kOut;  // q and out: the sequence's query rows
      const int row0 = qrows ? q0 : k0;
      const int len = qrows ? lq : lk;
      const int cls = (uint64_t)len * (uint64_t)p.row_bytes >= kMapLargeBytes ? 1 : 0;
      const uint4* src = reinterpret_cast<const uint4*>(&p.tmpl[cls][m]);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int w = 0; w < kMapBytes / 16; ++w) d4[w] = src[w];
      tmap_set_address(dst, p.base[t] + (size_t)row0 * p.row_bytes);
      tmap_set_dim2(dst, (uint32_t)len);
      wrote_map = true;
    }
  }
  if (wrote_map) tmap_release();
  __syncthreads();

  // 2. rank = position in longest-key-range-first order (stable)
  for (int i = tid; i < N; i += nt) {
    int rank = i;
    if (lpt) {
      const int ki = s_key[i];
      rank = 0;
      for (int j = 0; j < N; ++j) {
        const int kj = s_key[j];
        rank += (kj > ki) || (kj == ki && j < i);
      }
      s_order[rank] = i;
    }
    order[rank] = i;
  }
  __syncthreads();

  // 3. exclusive prefix sums of the unit counts in rank order
  const int chunk = (N + nt - 1) / nt;
  const int r0 = tid * chunk, r1 = min(N, r0 + chunk);
  int local = 0;
  for (int r = r0; r < r1; ++r) local += units_of(order_at(r));
  // block-wide exclusive scan of `local`
  const int lane = tid & 31, warp = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = nt >> 5;
    int w = lane < nw ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) s_warp[lane] = wi - w;  // exclusive warp offsets
    if (lane == nw - 1) s_carry = wi;      // total
  }
  __syncthreads();
  int run = s_warp[warp] + incl - local;
  for (int r = r0; r < r1; ++r) {
    prefix[r] = run;
    if (lpt) s_pref[r] = run;
    run += units_of(order_at(r));
  }
  if (tid == 0) {
    prefix[N] = s_carry;
    if (lpt) s_pref[N] = s_carry;
  }
  __syncthreads();

  // 4. tail split.  The plan first finds where the tail starts: it runs the
  //    attention kernel's list schedule (units longest first, each to the
  //    CTA that frees up first; a unit costs its key tiles plus
  //    kUnitCostTiles) over groups of CTAs that free up at the same time.
  //    The first unit that would end past 31/32 of the balanced time per
  //    CTA starts the tail (a unit of the first wave only if it alone runs
  //    past 33/32 of it); every unit from there on may be cut along the key
  //    range.  (Without the longest-first order, past kSimMaxSteps steps or
  //    a grid above kSimMaxGrid, the tail is the grid's last partial wave.)
  //    Chunk count of tail unit i: ceil(nkv_i / T) with the smallest key-tile
  //    budget T (at least kMinChunkTiles) whose total fits the split region.
  //    Everything runs on chip: the tail units' key-tile counts go to shared
  //    memory (s_key is free now), one warp simulates (the first rank in
  //    closed form) and searches T with warp reductions.
  const int U = s_carry;
  auto nkv_of = [&](int i) {
    const int lk = lk_of(i);
    return lk > 0 ? (lk + p.kv_rows - 1) / p.kv_rows : 0;
  };
  __shared__ unsigned s_gt[kSimMaxGrid];   // simulated CTA groups: time they free up
  __shared__ int s_gc[kSimMaxGrid];        // and their CTA count
  __shared__ int s_t0;                     // first tail unit (U: none)
  // (rank 0 holds the most key tiles: if even its units are too short to cut
  // into two chunks, nothing is split and the schedule is not simulated)
  const bool try_split = ATTN_VARLEN_TAIL_SPLIT && !p.causal && lpt && p.split_cap >= p.grid &&
                         p.grid > 0 && U > 0 &&
                         nkv_of(order_at(0)) > kMinChunkTiles + kMergeTiles;
  if (warp == 0) {
    int t0 = U;
    if (try_split) {
      t0 = U - U % p.grid;  // the grid's last partial wave
      if (ATTN_VARLEN_SIM_TAIL && p.grid <= kSimMaxGrid) {
        long long tot = 0;
        for (int r = lane; r < N; r += 32) {
          const int i = order_at(r), k = units_of(i);
          if (k > 0) tot += (long long)k * (nkv_of(i) + kUnitCostTiles);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        const long long bal = tot / p.grid;
        const long long late = bal - bal / 32;  // a unit ending past this starts the tail
        const long long big = bal + bal / 32;   // a first-wave unit this long is late too
        int found = U;
        bool done_all = bal < (1ll << 29);  // simulated times fit 32 bits
        if (done_all) {
          // rank 0 in closed form (every CTA is free at time 0, so its unit d
          // starts at (d / grid) n0): the first late wave is the first w >= 1
          // with (w + 1) n0 > late, or wave 0 for a unit longer than `big`
          const int k0 = units_of(order_at(0));
          const long long n0 = nkv_of(order_at(0)) + kUnitCostTiles;
          const long long w = n0 > big ? 0 : max(1ll, late / n0);
          if (w * p.grid < k0) {
            found = (int)(w * p.grid);
          } else {
            const int W = k0 / p.grid, rem = k0 - W * p.grid;
            if (lane == 0) {
              s_gt[0] = (unsigned)(W * n0);
              s_gc[0] = p.grid - rem;
              s_gt[1] = (unsigned)((W + 1) * n0);
              s_gc[1] = rem;
            }
            int ng = rem > 0 ? 2 : 1, steps = 0;
            __syncwarp();
            // later ranks step by step, one group of CTAs at a time
            for (int r = 1; r < N && found == U && done_all; ++r) {
              const int i = order_at(r), k = units_of(i);
              if (k == 0) break;  // ranks without units come last
              const unsigned n = (unsigned)(nkv_of(i) + kUnitCostTiles);
              for (int d = 0; d < k;) {
                if (++steps > kSimMaxSteps) {
                  done_all = false;
                  break;
                }
                // the group that frees up first
                unsigned mt = 0xffffffffu;
                int mi = 0;
                for (int g = lane; g < ng; g += 32)
                  if (s_gt[g] < mt) {
                    mt = s_gt[g];
                    mi = g;
                  }
                const unsigned bt = __reduce_min_sync(0xffffffffu, mt);
                const int src = __ffs(__ballot_sync(0xffffffffu, mt == bt)) - 1;
                const int bi = __shfl_sync(0xffffffffu, mi, src);
                // late: it ends past the mark; a unit of the first wave only
                // if it alone runs longer than `big` (else splitting it
                // cannot shorten the schedule)
                if ((long long)bt + n > late && (bt > 0 || n > big)) {
                  found = prefix_at(r) + d;
                  break;
                }
                const int c = s_gc[bi];
                const int j = min(k - d, c);
                __syncwarp();
                if (lane == 0) {
                  if (j == c) {
                    s_gt[bi] = bt + n;
                  } else {  // j of the group's CTAs take one unit each
                    s_gc[bi] = c - j;
                    s_gt[ng] = bt + n;
                    s_gc[ng] = j;
                  }
                }
                if (j != c) ++ng;
                __syncwarp();
                d += j;
              }
            }
          }
        }
        if (done_all) t0 = found;
      }
      // the split region holds at most split_cap tail units (and items)
      if (U - t0 > p.split_cap) t0 = U - U % p.grid;
    }
    if (lane == 0) s_t0 = t0;
  }
  __syncthreads();
  const int t0 = s_t0;  // first tail unit
  const int R = U - t0;  // tail units
  if (warp == 0) {
    int split_start = U, items = U;
    if (R > 0) {
      // The tail, rank by rank: ranks rt .. N-1, rank r holding cnt(r) tail
      // units of s_key[r] key tiles each (units of a rank are consecutive).
      int before = 0;
      for (int r = lane; r < N; r += 32) before += s_pref[r + 1] <= t0;
      const int rt = __reduce_add_sync(0xffffffffu, before);
      auto cnt = [&](int r) { return s_pref[r + 1] - max(s_pref[r], t0); };
      int maxn = 0, minn = 0x7fffffff;
      long long work = 0;
      for (int r = rt + lane; r < N; r += 32) {
        const int cr = cnt(r);
        const int nk = cr > 0 ? nkv_of(order_at(r)) : 0;
        s_key[r] = nk;
        if (cr > 0) {
          maxn = max(maxn, nk);
          minn = min(minn, nk);
          work += (long long)cr * nk;
        }
      }
      __syncwarp();
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        maxn = max(maxn, __shfl_xor_sync(0xffffffffu, maxn, o));
        minn = min(minn, __shfl_xor_sync(0xffffffffu, minn, o));
        work += __shfl_xor_sync(0xffffffffu, work, o);
      }
      // Items the tail may take.  Equal units in a short tail: one chunk per
      // CTA, all of about the same length.  Unequal units, or a long tail
      // (kFineTailTiles key tiles per CTA and more): up to split_cap, so that
      // the longest-first hand-out of smaller chunks evens out the CTAs'
      // ends (chunks still hold at least kMinChunkTiles key tiles, enough to
      // pay for their partial writes and merges).
      const bool coarse = minn == maxn && work < (long long)kFineTailTiles * p.grid;
      const int cap = coarse ? p.grid : p.split_cap;
      auto chunks_of = [&](int nk, int t) { return nk > t ? (nk + t - 1) / t : 1; };
      int lo = 1, hi = maxn > 1 ? maxn : 1;
      if (minn == maxn && maxn > 0) {
        // equal tail units (every single-sequence call): each may take
        // cap / R chunks, so the smallest budget is ceil(nkv / that)
        const int per = max(cap / R, 1);
        lo = hi = (maxn + per - 1) / per;
      }
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        int sum = 0;
        for (int r = rt + lane; r < N; r += 32) {
          const int cr = cnt(r);
          if (cr > 0) sum += cr * chunks_of(s_key[r], mid);
        }
        sum = __reduce_add_sync(0xffffffffu, sum);
        if (sum <= cap) hi = mid; else lo = mid + 1;
      }
      lo = max(lo, kMinChunkTiles);
      if (lo + kMergeTiles < maxn) {
        // chunk counts -> exclusive prefix per tail unit: each lane takes a
        // contiguous block of ranks, and a rank's units follow one another
        const SplitLayout SL = split_layout(p.split_cap);
        int* tp = reinterpret_cast<int*>(p.split + SL.prefix);
        const int per = (N - rt + 31) / 32, r0 = rt + lane * per, r1 = min(N, r0 + per);
        int mine = 0;
        for (int r = r0; r < r1; ++r) {
          const int cr = cnt(r);
          if (cr > 0) mine += cr * chunks_of(s_key[r], lo);
        }
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        int run_items = incl - mine;
        for (int r = r0; r < r1; ++r) {
          const int cr = cnt(r);
          if (cr == 0) continue;
          const int q = chunks_of(s_key[r], lo), f = max(s_pref[r], t0) - t0;
          for (int j = 0; j < cr; ++j) tp[f + j] = run_items + j * q;
          run_items += cr * q;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (lane == 0) tp[R] = total;
        split_start = t0;
        items = t0 + total;
      }
    }
    if (lane == 0) {
      hdr[1] = U;
      hdr[2] = items;
      hdr[3] = split_start;
      hdr[kHdrNextItem] = 0;
    }
  }
  // The split region's row counters: every merge leaves its counter at zero,
  // so they are zeroed only when marked dirty (a new workspace, or a call in
  // which a CTA gave up a wait), 16 bytes at a time (the region is 256-byte
  // aligned).
  if (counters_dirty != 0) {
    uint4* c4 = reinterpret_cast<uint4*>(p.split + split_layout(p.split_cap).counters);
    for (int i = tid; i < p.split_cap * 2 * kBlockM / 4; i += nt) c4[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (tid == 0) hdr[kHdrCountersDirty] = 0;
  }
}

// Epilogue of one chunk of a split unit (a softmax warp of Q tile t; lane =
// row r).  The chunk's unnormalised O row, m and l go to its partial slot,
// and the chunk is counted in with an acquire-release add on a counter per
// (row, Q tile).  The last chunk of the unit to finish a row merges,
//   m* = max_c m_c,  O = sum_c 2^(m_c - m*) O_c,  l = sum_c 2^(m_c - m*) l_c,
// always in chunk order (the result does not depend on which chunk came
// last), and writes O / l as bf16.  Its own chunk is read back from TMEM, so
// each other chunk costs one batch of loads per pass over the columns (one
// pass up to 80 columns, two above).  TMEM loads are warp-collective: a warp
// takes part in the merge if any of its lanes merges.  A slot is
// column-major ([column][128 rows]) so that a warp's stores and loads of one
// column are one 128-byte line; partials bypass L1.  No thread waits for
// another CTA.
constexpr size_t kSlot = (size_t)kPartRowMax * kBlockM;  // floats per (chunk, tile) slot

template <int D>
__device__ __noinline__ void split_epilogue(uint8_t* parts_base, int* counters, uint32_t tO, int t,
                                            int r, float m, float l, uint16_t* orow, bool valid,
                                            int part, int part0, int tail, int chunks) {
  using G = Geometry<D>;
  constexpr int NB = (D + 15) / 16;                 // 16-column TMEM blocks holding O's columns
  constexpr int PB = D <= 80 ? NB : NB / 2;          // blocks per pass
  constexpr int PC = D <= 80 ? D : D / 2;            // columns per pass
  static_assert(D <= 80 || (D % 32 == 0), "two passes of whole 16-column blocks");
  float* parts = reinterpret_cast<float*>(parts_base);
  float* mine = parts + (size_t)(part * 2 + t) * kSlot + r;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    uint32_t o[16];
    tmem_ld16(tO + 16 * b, o);
    tmem_wait_ld();
    reg_fence(o, 0, 16);
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (16 * b + e < D) __stcg(mine + (size_t)(16 * b + e) * kBlockM, __uint_as_float(o[e]));
  }
  __stcg(mine + (size_t)G::DP * kBlockM, m);
  __stcg(mine + (size_t)(G::DP + 1) * kBlockM, l);
  int* cnt = counters + ((size_t)(2 * tail + t) * kBlockM + r);
  const bool last = atom_add_acq_rel_gpu(cnt, 1) == chunks - 1;
  if (!__any_sync(0xffffffffu, last)) return;  // warp-uniform from here on
  const float* first = parts + (size_t)(part0 * 2 + t) * kSlot + r;
  const size_t cstride = 2 * kSlot;  // next chunk, same tile and row
  const int own = part - part0;      // this warp's chunk (the same for all lanes)
  auto mval = [&](int cc) -> float {
    if (cc == own) return m;
    return last ? __ldcg(first + cc * cstride + (size_t)G::DP * kBlockM) : 0.f;
  };
  float mm = -INFINITY;
  for (int cc = 0; cc < chunks; ++cc) mm = fmaxf(mm, mval(cc));
  float ll = 0.f;
  for (int cc = 0; cc < chunks; ++cc) {
    const float lc = cc == own ? l : (last ? __ldcg(first + cc * cstride + (size_t)(G::DP + 1) * kBlockM) : 0.f);
    ll += ex2(mval(cc) - mm) * lc;
  }
  const float inv_l = ll > 0.f ? 1.0f / ll : 0.f;
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += PC) {
    float acc[PC];
#pragma unroll
    for (int e = 0; e < PC; ++e) acc[e] = 0.f;
    for (int cc = 0; cc < chunks; ++cc) {
      const float w = ex2(mval(cc) - mm);
      if (cc == own) {
#pragma unroll
        for (int b = 0; b < PB; ++b) {
          uint32_t o[16];
          tmem_ld16(tO + (uint32_t)c0 + 16 * b, o);
          tmem_wait_ld();
          reg_fence(o, 0, 16);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (16 * b + e < PC) acc[16 * b + e] += w * __uint_as_float(o[e]);
        }
      } else if (last) {
        const float* src = first + cc * cstride + (size_t)c0 * kBlockM;
        float v[PC];
#pragma unroll
        for (int e = 0; e < PC; ++e) v[e] = __ldcg(src + (size_t)e * kBlockM);
#pragma unroll
        for (int e = 0; e < PC; ++e) acc[e] += w * v[e];
      }
    }
    if (last && valid) {
#pragma unroll
      for (int e = 0; e < PC; e += 8)
        *reinterpret_cast<uint4*>(orow + c0 + e) = make_uint4(
            pack_bf16x2(acc[e] * inv_l, acc[e + 1] * inv_l),
            pack_bf16x2(acc[e + 2] * inv_l, acc[e + 3] * inv_l),
            pack_bf16x2(acc[e + 4] * inv_l, acc[e + 5] * inv_l),
            pack_bf16x2(acc[e + 6] * inv_l, acc[e + 7] * inv_l));
    }
  }
  if (last) *cnt = 0;  // ready for the next call
}

// -------------------------------------------------------------------- fwd
template <int D>
__global__ void __launch_bounds__(Geometry<D>::THREADS, 1)
    attn_varlen_fwd_kernel(const __grid_constant__ FwdParams p) {
  using G = Geometry<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_u32);
  const uint32_t sQ = base + G::Q_OFF;
  const uint32_t sKV = base + G::KV_OFF;
  auto bar = [&](int i) -> uint32_t { return base + G::BAR_OFF + 8u * (uint32_t)i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base_ptr + G::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + G::MISC_OFF + 4);
  volatile int* item_ring = reinterpret_cast<volatile int*>(base_ptr + G::MISC_OFF + 8);
  // Consumer side of the item ring (MMA issuers, softmax warps): the k-th
  // item of this CTA, or -1 if a wait gave up.  Lane 0 of every consumer
  // warp releases the entry once the warp has read it.
  auto next_item = [&](int k) -> int {
    const uint32_t islot = k % kItemDepth, iuse = k / kItemDepth;
    const bool w = wait_bounded(bar(G::B_ITEM_FULL + islot), iuse & 1u, abort_flag, p.status,
                                kStatusTimeoutItem);
    if (!__all_sync(0xffffffffu, w)) return -1;
    const int u = item_ring[islot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar(G::B_ITEM_EMPTY + islot));
    return u;
  };

  // warp index made warp-uniform for the compiler (role branches below)
  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);

  if (threadIdx.x == 0) {
    mbar_init(bar(G::B_Q_FULL), 1);
    mbar_init(bar(G::B_Q_EMPTY), G::ISSUERS);
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(bar(G::B_KV_FULL + s), 1);
      mbar_init(bar(G::B_KV_EMPTY + s), G::ISSUERS);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(G::B_S_FULL + t), 1);
      mbar_init(bar(G::B_P_FULL + t), kBlockM);
      mbar_init(bar(G::B_PV_DONE + t), 1);
      mbar_init(bar(G::B_S_FREE + t), kBlockM);
    }
    mbar_init(bar(G::B_DRAIN + 0), 1);
    mbar_init(bar(G::B_DRAIN + 1), 1);
    for (int i = 0; i < kItemDepth; ++i) {
      mbar_init(bar(G::B_ITEM_FULL + i), 1);
      mbar_init(bar(G::B_ITEM_EMPTY + i), G::ITEM_CONSUMERS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == G::MMA_WARP) {
    tmem_alloc(base + G::MISC_OFF, kTmemCols);
    tmem_relinquish();
  }
  if constexpr (G::ZB) {
    // the zero (and ones) regions, read by the MMAs (async proxy) from now on
    if (threadIdx.x < G::ZERO_BYTES / 16u)
      reinterpret_cast<uint4*>(base_ptr + G::ZERO_OFF)[threadIdx.x] = make_uint4(0, 0, 0, 0);
    if (G::LO && threadIdx.x < G::ONES_BYTES / 16u)  // bf16 1.0 in column 0 of each row
      reinterpret_cast<uint4*>(base_ptr + G::ONES_OFF)[threadIdx.x] = make_uint4(0x3F80u, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // everything above overlaps the plan kernel; the workspace is read below
  grid_wait_prerequisite();
#if ATTN_VARLEN_PLAN_PDL
  // the next call's plan kernel may launch now; it waits for this grid to
  // finish before it touches the workspace
  grid_launch_dependents();
#endif
  const WsLayout L = ws_layout(p.num_seqs);
  const int num_units = reinterpret_cast<const int*>(p.ws)[1];
  const int num_items = reinterpret_cast<const int*>(p.ws)[2];
  const int split_start = reinterpret_cast<const int*>(p.ws)[3];
  const SplitLayout SL = split_layout(p.split_cap);
  const int32_t* tail_prefix = reinterpret_cast<const int32_t*>(p.split + SL.prefix);
  const int32_t* order = reinterpret_cast<const int32_t*>(p.ws + L.order);
  const int32_t* prefix = reinterpret_cast<const int32_t*>(p.ws + L.prefix);

  if (warp == G::LOAD_WARP) {
    // ------------------------------------------------------ TMA producer
    // The whole warp runs the loop (uniform control flow); one elected lane
    // issues each TMA and expect-tx.  K and V tiles enter the ring in the
    // order the MMA warp first uses them (kv_item_tile).
    const uint32_t leader = elect_one();
    uint32_t kv_item = 0, q_use = 0;
    bool ok = true;
    auto wait_ = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu,
                        wait_bounded(b, parity, abort_flag, p.status, kStatusTimeoutLoad));
    };
    // Items are handed out dynamically, longest first: the CTA's first item
    // is blockIdx.x, every later one comes from the workspace counter.  The
    // producer publishes each item (or a past-the-end index) in the ring.
    // The next item is claimed once the current item's last K/V load is out,
    // so the counter's round trip overlaps that item's last key tiles.
    const int leader_lane = __ffs(__ballot_sync(0xffffffffu, leader != 0)) - 1;
    int pending = 0;
    for (int k = 0; ok; ++k) {
      const int u = k == 0 ? (int)blockIdx.x
                           : (int)gridDim.x + __shfl_sync(0xffffffffu, pending, leader_lane);
      const uint32_t islot = k % kItemDepth, iuse = k / kItemDepth;
      if (!(ok = wait_(bar(G::B_ITEM_EMPTY + islot), (iuse & 1u) ^ 1u))) break;
      if (leader) item_ring[islot] = u;
      __syncwarp();
      if (leader) mbar_arrive(bar(G::B_ITEM_FULL + islot));
      if (u >= num_items) break;
#if !ATTN_VARLEN_LATE_CLAIM
      if (leader) pending = atomicAdd(p.status + kHdrNextItem, 1);
#endif
      const UnitInfo ui = decode_item(u, order, prefix, p.num_seqs, p.cu_q, p.cu_k, G::KN,
                                        split_start, num_units, tail_prefix, p.causal != 0,
                                        p.head_begin);
      if (ui.nkv == 0) {
#if ATTN_VARLEN_LATE_CLAIM
        if (leader) pending = atomicAdd(p.status + kHdrNextItem, 1);
#endif
        continue;
      }
      // maps of this sequence: box A of q, k, v, then box B of q, k, v
      const uint8_t* mq = p.ws + L.maps + (size_t)ui.seq * kMapsPerSeq * kMapBytes;
      const uint8_t* mk = mq + kMapBytes;
      const uint8_t* mv = mq + 2 * kMapBytes;
      const uint8_t* mqb = G::ZB ? mq + kTensors * kMapBytes : mq;
      const uint8_t* mkb = G::ZB ? mk + kTensors * kMapBytes : mk;
      const uint8_t* mvb = G::ZB ? mv + kTensors * kMapBytes : mv;
      if (leader) {
        tmap_acquire(mq);
        tmap_acquire(mk);
        tmap_acquire(mv);
        if (G::ZB) {
          tmap_acquire(mqb);
          tmap_acquire(mkb);
          tmap_acquire(mvb);
        }
      }
      __syncwarp();
      if (!(ok = wait_(bar(G::B_Q_EMPTY), (q_use & 1u) ^ 1u))) break;
      ++q_use;
      mbar_arrive_expect_tx_if(leader, bar(G::B_Q_FULL), (ui.t1 ? 2u : 1u) * G::Q_LOAD_BYTES);
      // box A at x = 0; box B at x = 64, right after box A (the whole tile
      // for ZB, the second 64-column box otherwise)
      for (int t = 0; t < (ui.t1 ? 2 : 1); ++t) {
        const uint32_t dq = sQ + t * G::Q_TILE_BYTES;
        tma_load_3d_if(leader, dq, mq, bar(G::B_Q_FULL), 0, ui.head, ui.q0 + t * kBlockM);
        if (G::NB == 2)
          tma_load_3d_if(leader, dq + G::Q_BOX_BYTES, mqb, bar(G::B_Q_FULL), G::BW, ui.head,
                         ui.q0 + t * kBlockM);
      }
      for (int i = 0; i < 2 * ui.nkv; ++i) {
        int j;
        const bool is_v = kv_item_tile<G::PSEP>(i, ui.nkv, j);
        const uint32_t stage = kv_item % G::STAGES;
        const uint32_t use = kv_item / G::STAGES;
        if (!(ok = wait_(bar(G::B_KV_EMPTY + stage), (use & 1u) ^ 1u))) break;
#if ATTN_VARLEN_TEST_HOOKS
        const uint32_t issue = (p.test_withhold && blockIdx.x == 0 && kv_item == 0) ? 0u : leader;
#else
        const uint32_t issue = leader;
#endif
        mbar_arrive_expect_tx_if(issue, bar(G::B_KV_FULL + stage), G::KV_LOAD_BYTES);
        const uint32_t dst = sKV + stage * G::KV_TILE_BYTES;
        const int row = (ui.jb + j) * G::KN;
        tma_load_3d_if(issue, dst, is_v ? mv : mk, bar(G::B_KV_FULL + stage), 0, ui.head, row);
        if (G::NB == 2)
          tma_load_3d_if(issue, dst + G::KV_BOX_BYTES, is_v ? mvb : mkb, bar(G::B_KV_FULL + stage),
                         G::BW, ui.head, row);
        ++kv_item;
      }
#if ATTN_VARLEN_LATE_CLAIM
      // the next item is claimed only once this one's last K/V load is out,
      // a few key tiles before its compute ends: the claim's round trip is
      // still hidden, and the longest-first order holds (claimed at the start
      // of an item, a long item's successor was taken one whole item early)
      if (leader) pending = atomicAdd(p.status + kHdrNextItem, 1);
#endif
    }
    if (!ok) {
      // let every copy already issued land before the CTA can exit
      if (q_use > 0) wait_drain(bar(G::B_Q_FULL), (q_use - 1) & 1u);
      const uint32_t first = kv_item > (uint32_t)G::STAGES ? kv_item - G::STAGES : 0;
      for (uint32_t it = first; it < kv_item; ++it)
        wait_drain(bar(G::B_KV_FULL + it % G::STAGES), (it / G::STAGES) & 1u);
    }
  } else if (warp >= G::MMA_WARP) {
    // ------------------------------------------------------- MMA issuer
    // The whole warp runs the loop; descriptors are computed once per tile
    // base and advanced by constants, and one elected lane issues each
    // tcgen05.mma and commit (commits track that lane's MMAs).  With two
    // issuers, warp MMA_WARP + t issues every MMA of Q tile t, so neither
    // tile's S waits behind the other tile's P.V in one in-order program;
    // K/V slots and the Q buffer are released by both.
    const int mi = warp - G::MMA_WARP;
    const uint32_t leader = elect_one();
    constexpr uint32_t idesc_s = idesc_bf16_f32(kBlockM, G::KN, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kBlockM, G::DP, false, true);
    // K-major (Q, K) and MN-major (V) descriptors of the first tile of each
    // region; a byte offset `o` inside shared memory adds o >> 4.
    const uint64_t dq0 = smem_desc(sQ, 16, G::SBO, G::SWZ);
    const uint64_t dk0 = smem_desc(sKV, 16, G::SBO, G::SWZ);
    const uint64_t dv0 = smem_desc(sKV, G::KV_BOX_BYTES, G::SBO, G::SWZ);
    uint32_t kv_item = 0, q_use = 0;
    uint32_t p_wait[2] = {0, 0};  // p_full phases consumed per tile
    uint32_t pv_cnt[2] = {0, 0};  // P.V groups committed per tile
    uint32_t s_cnt[2] = {0, 0};   // S groups committed per tile
    bool ok = true;
    bool issued = false;

    auto wait_ = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu,
                        wait_bounded(b, parity, abort_flag, p.status, kStatusTimeoutMma));
    };
    // Box B with a zero chunk (ZB): unswizzled core matrices of 8 rows x 16
    // bytes.  K-major (Q, K): the K-direction step to the second 8-column
    // chunk (LBO) lands in the zero region, 8-row groups are 128 bytes apart
    // (SBO).  MN-major (V): 8-key groups 128 bytes apart (LBO), the second
    // 8-column chunk of N (SBO) in the zero region.
    const uint32_t sZero = base + G::ZERO_OFF;
    auto desc_kb = [&](uint32_t addr) { return smem_desc(addr, sZero - addr, 128, kSwizzleNone); };
    // S_t = Q_t K^T : K from stage `ks`
    auto issue_s = [&](int t, uint32_t ks) {
      const uint64_t qa = dq0 + ((t * G::Q_TILE_BYTES) >> 4);
      const uint64_t kb = dk0 + ((ks * G::KV_TILE_BYTES) >> 4);
      const uint32_t d = tmem + G::s_col(t);
#pragma unroll
      for (int k = 0; k < G::NK_S; ++k) {
        const uint32_t box = (uint32_t)(k * 16 / G::BW);
        const uint32_t col_b = (uint32_t)((k * 16) % G::BW) * 2;
        if (G::ZB && box == 1) {
          mma_ss_if(leader, d, desc_kb(sQ + t * G::Q_TILE_BYTES + G::Q_BOX_BYTES),
                    desc_kb(sKV + ks * G::KV_TILE_BYTES + G::KV_BOX_BYTES), idesc_s, 1u);
        } else {
          mma_ss_if(leader, d, qa + ((box * G::Q_BOX_BYTES + col_b) >> 4),
                    kb + ((box * G::KV_BOX_BYTES + col_b) >> 4), idesc_s, k > 0 ? 1u : 0u);
        }
      }
    };
    // O_t (+)= P_t V : V from stage `vs`, P from TMEM.  With ZB, columns
    // 0-63 (box A) and 64-79 (box B and the zero chunk) are two products of
    // N = 64 and N = 16 per 16-key step.
    constexpr uint32_t idesc_pv_a = idesc_bf16_f32(kBlockM, G::BW, false, true);
    constexpr uint32_t idesc_pv_b = idesc_bf16_f32(kBlockM, 16, false, true);
    auto issue_pv = [&](int t, uint32_t vs, bool acc) {
      const uint64_t vb = dv0 + ((vs * G::KV_TILE_BYTES) >> 4);
      const uint32_t d = tmem + G::o_col(t);
      const uint32_t a = tmem + G::p_col(t);
      if constexpr (G::ZB) {
        const uint32_t vbb = sKV + vs * G::KV_TILE_BYTES + G::KV_BOX_BYTES;
        const uint32_t pad = G::LO ? base + G::ONES_OFF : sZero;  // V columns 72-79
        const uint64_t dvb = smem_desc(vbb, 128, pad - vbb, kSwizzleNone);
#pragma unroll
        for (int k = 0; k < G::NK_PV; ++k) {
          const uint32_t acc_k = (acc || k > 0) ? 1u : 0u;
          mma_ts_if(leader, d, a + 8u * k, vb + ((k * 16 * G::BW * 2) >> 4), idesc_pv_a, acc_k);
          mma_ts_if(leader, d + G::BW, a + 8u * k, dvb + ((k * 16 * 16) >> 4), idesc_pv_b, acc_k);
        }
      } else {
#pragma unroll
        for (int k = 0; k < G::NK_PV; ++k)
          mma_ts_if(leader, d, a + 8u * k, vb + ((k * 16 * G::BW * 2) >> 4), idesc_pv,
                    (acc || k > 0) ? 1u : 0u);
      }
    };
    // S_t overwrites P_t: the P.V MMA that reads P_t must be finished
    // (issue order guarantees it unless kStrictPvWait asks for the wait)
    auto wait_pv_idle = [&](int t) -> bool {
      if (!kStrictPvWait || pv_cnt[t] == 0) return true;
      return wait_(bar(G::B_PV_DONE + t), (pv_cnt[t] - 1) & 1u);
    };
    auto stage_of = [](uint32_t it) { return it % G::STAGES; };
    auto kv_full = [&](uint32_t it) -> bool {
      return wait_(bar(G::B_KV_FULL + it % G::STAGES), (it / G::STAGES) & 1u);
    };

    for (int k = 0; ok; ++k) {
      const int u = next_item(k);
      if (u < 0 || u >= num_items) break;
      const UnitInfo ui = decode_item(u, order, prefix, p.num_seqs, p.cu_q, p.cu_k, G::KN,
                                        split_start, num_units, tail_prefix, p.causal != 0,
                                        p.head_begin);
      if (ui.nkv == 0) continue;
      if (!(ok = wait_(bar(G::B_Q_FULL), q_use & 1u))) break;
      ++q_use;
      issued = true;
      const int nt = ui.t1 ? 2 : 1;
      if constexpr (G::PSEP) {
        // Tile t = mi.  Order per key tile j:  S_t(j) | P_t(j-1).V(j-1).
        // S_t(j) only needs the softmax to have read S_t(j-1) (S_FREE), so
        // it runs while that softmax is still in its exp2 phase.  A unit
        // without a second Q tile still has issuer 1 take part in the slot
        // releases, after each slot has filled, so no barrier runs ahead.
        // Under the causal mask tile 0 may need fewer key tiles (nkv0) than
        // the unit loads; its issuer then only takes part in the releases.
        const int t = mi;
        const bool has = t == 0 || ui.t1;
        const int n_t = has ? (t == 0 ? ui.nkv0 : ui.nkv) : 0;
        bool mine = false;  // this issuer has MMAs on the slot being released
        auto release = [&](uint32_t b) {
          if (mine)
            mma_commit_if(leader, b);
          else if (leader)
            mbar_arrive(b);
        };
        const int n = ui.nkv;
        for (int j = 0; ok && j <= n; ++j) {
          if (j < n) {
            const uint32_t itk = kv_item + (j == 0 ? 0u : 2u * j - 1u);
            if (!(ok = kv_full(itk))) break;
            mine = j < n_t;
            if (mine) {
              if (s_cnt[t] > 0 && !(ok = wait_(bar(G::B_S_FREE + t), (s_cnt[t] - 1) & 1u))) break;
              tc_fence_after();
              issue_s(t, stage_of(itk));
              mma_commit_if(leader, bar(G::B_S_FULL + t));
              ++s_cnt[t];
            }
            release(bar(G::B_KV_EMPTY + stage_of(itk)));
            mine = n_t > 0;  // commit after this issuer's last MMA on Q
            if (j == n - 1) release(bar(G::B_Q_EMPTY));
          }
          if (j >= 1) {
            const uint32_t itv = kv_item + (j == n ? 2u * n - 1u : 2u * j);
            if (!(ok = kv_full(itv))) break;
            mine = j - 1 < n_t;
            if (mine) {
              if (!(ok = wait_(bar(G::B_P_FULL + t), p_wait[t] & 1u))) break;
              ++p_wait[t];
              tc_fence_after();
              issue_pv(t, stage_of(itv), j > 1);
              mma_commit_if(leader, bar(G::B_PV_DONE + t));
            }
            release(bar(G::B_KV_EMPTY + stage_of(itv)));
          }
        }
        (void)nt;
      } else {
        // Order:  S0(0) S1(0) | PV0(j) S0(j+1) PV1(j) S1(j+1) | ...
        // S_t(j+1) overwrites P_t(j) and is queued right behind P_t(j).V(j).
        {
          const uint32_t it = kv_item;
          if (!(ok = kv_full(it))) break;
          if (ui.nkv0 > 0) {
            ok = wait_pv_idle(0);
            if (!ok) break;
            tc_fence_after();
            issue_s(0, stage_of(it));
            mma_commit_if(leader, bar(G::B_S_FULL + 0));
          }
          if (ui.t1) {
            ok = wait_pv_idle(1);
          if (!ok) break;
            tc_fence_after();
            issue_s(1, stage_of(it));
            mma_commit_if(leader, bar(G::B_S_FULL + 1));
          }
          mma_commit_if(leader, bar(G::B_KV_EMPTY + stage_of(it)));
          if (ui.nkv == 1) mma_commit_if(leader, bar(G::B_Q_EMPTY));
        }
        for (int j = 0; ok && j < ui.nkv; ++j) {
          const uint32_t itv = kv_item + 2 * j + 1;
          const uint32_t itk = itv + 1;
          const bool more = j + 1 < ui.nkv;
          if (!(ok = kv_full(itv))) break;
          // tile 0 (for its nkv0 key tiles): O0 += P0 V_j, then S0 = Q0 K_{j+1}^T
          if (j < ui.nkv0) {
            if (!(ok = wait_(bar(G::B_P_FULL + 0), p_wait[0] & 1u))) break;
            ++p_wait[0];
            tc_fence_after();
            issue_pv(0, stage_of(itv), j > 0);
            mma_commit_if(leader, bar(G::B_PV_DONE + 0));
            ++pv_cnt[0];
          }
          if (more) {
            if (!(ok = kv_full(itk))) break;
          }
          if (more && j + 1 < ui.nkv0) {
            ok = wait_pv_idle(0);
            if (!ok) break;
            tc_fence_after();
            issue_s(0, stage_of(itk));
            mma_commit_if(leader, bar(G::B_S_FULL + 0));
          }
          // tile 1: O1 += P1 V_j, then S1 = Q1 K_{j+1}^T
          if (ui.t1) {
            if (!(ok = wait_(bar(G::B_P_FULL + 1), p_wait[1] & 1u))) break;
            ++p_wait[1];
            tc_fence_after();
            issue_pv(1, stage_of(itv), j > 0);
            mma_commit_if(leader, bar(G::B_PV_DONE + 1));
            ++pv_cnt[1];
          }
          mma_commit_if(leader, bar(G::B_KV_EMPTY + stage_of(itv)));
          if (more) {
            if (ui.t1) {
              ok = wait_pv_idle(1);
          if (!ok) break;
              tc_fence_after();
              issue_s(1, stage_of(itk));
              mma_commit_if(leader, bar(G::B_S_FULL + 1));
            }
            mma_commit_if(leader, bar(G::B_KV_EMPTY + stage_of(itk)));
            if (j + 2 == ui.nkv) mma_commit_if(leader, bar(G::B_Q_EMPTY));
          }
        }
      }
      kv_item += 2u * (uint32_t)ui.nkv;
    }
    if (issued) {
      // every MMA this warp issued must be finished before TMEM is freed
      mma_commit_if(leader, bar(G::B_DRAIN + mi));
      wait_drain(bar(G::B_DRAIN + mi), 0);
    }
  } else {
    // --------------------------------------------------------- softmax
    // Warp w: Q tile t = w / 4, TMEM lane quarter w mod 4; each thread owns
    // row r of its tile (TMEM lane r) and all KN key columns of every tile.
    constexpr int KN = G::KN, KC = KN;
    const int t = warp >> 2;                       // Q tile of this warpgroup
    const int qq = warp & 3;                       // TMEM lane quarter
    const int r = threadIdx.x & 127;               // row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const uint32_t tS = tmem + lane_off + G::s_col(t);
    const uint32_t tP = tmem + lane_off + G::p_col(t);
    const uint32_t tO = tmem + lane_off + G::o_col(t);
    const float sl2 = p.scale_log2;
    uint32_t s_wait = 0, p_cnt = 0;
    bool ok = true;

    auto wait_ = [&](uint32_t b, uint32_t parity) -> bool {
      bool w = wait_bounded(b, parity, abort_flag, p.status, kStatusTimeoutSoftmax);
      return __all_sync(0xffffffffu, w);
    };

    for (int k = 0; ok; ++k) {
      const int u = next_item(k);
      if (u < 0 || u >= num_items) break;
      const UnitInfo ui = decode_item(u, order, prefix, p.num_seqs, p.cu_q, p.cu_k, KN,
                                        split_start, num_units, tail_prefix, p.causal != 0,
                                        p.head_begin);
      if (t == 1 && !ui.t1) continue;
      const int row = ui.q0 + kBlockM * t + r;
      const bool valid = row < ui.lq;
      uint16_t* orow = p.out + ((size_t)(ui.qbase + row) * p.num_heads + ui.head) * D;
      const int nsteps = t == 0 ? ui.nkv0 : ui.nkv;  // key tiles of this Q tile
      // keys this row may see: all L_k, or under the causal mask
      // min(L_k, row + 1 + L_k - L_q) (<= 0: none, the row is zero)
      const int klim = p.causal ? min(ui.lk, row + 1 + ui.coff) : ui.lk;
      // this sequence's out maps: acquired and prefetched now, so the
      // epilogue's stores do not wait for their descriptors
      const uint8_t* mo = p.ws + L.maps + ((size_t)ui.seq * kMapsPerSeq + kOut) * kMapBytes;
      const uint8_t* mob = mo + kTensors * kMapBytes;
      if ((threadIdx.x & 31) == 0 && ui.part < 0 && nsteps > 0) {
        tmap_acquire(mo);
        tmap_prefetch(mo);
        if (G::NB == 2) {
          tmap_acquire(mob);
          tmap_prefetch(mob);
        }
      }
      if (nsteps == 0) {
        if (valid) {
#pragma unroll
          for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      float m = 0.f, l = 0.f;
      for (int j = 0; j < nsteps; ++j) {
        if (!(ok = wait_(bar(G::B_S_FULL + t), s_wait & 1u))) break;
        ++s_wait;
        tc_fence_after();
        uint32_t s[KC];
        // keys past the end of the sequence (or past this row's causal
        // limit) in this tile are masked
        const int lim = klim - (ui.jb + j) * KN;
        // warp-uniform: both branches below hold tcgen05.wait::ld, which the
        // whole warp must execute together; masking at lim >= KC is a no-op
        const bool tail = __any_sync(0xffffffffu, lim < KC);
        float mx0, mx1, mx2, mx3;
        auto max_cols = [&](int c0, int c1) {
#pragma unroll
          for (int c = c0; c < c1; c += 8) {
            mx0 = fmax3(mx0, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
            mx1 = fmax3(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
            mx2 = fmax3(mx2, __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
            mx3 = fmax3(mx3, __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
          }
        };
        mx0 = mx1 = mx2 = mx3 = -INFINITY;
        if constexpr (KC > 64) {
          // the first 64 columns, then the rest while their max is taken
          tmem_ld_cols<64>(tS, s);
          tmem_wait_ld();
          reg_fence(s, 0, 64);
          tmem_ld_cols<KC - 64>(tS + 64, s + 64);
          if (!tail) {
            max_cols(0, 64);
            tmem_wait_ld();
            reg_fence(s, 64, KC - 64);
          } else {
            tmem_wait_ld();
            reg_fence(s, 64, KC - 64);
#pragma unroll
            for (int c = 0; c < KC; ++c)
              if (c >= lim) s[c] = __float_as_uint(-INFINITY);
            max_cols(0, 64);
          }
        } else {
          tmem_ld_cols<KC>(tS, s);
          tmem_wait_ld();
          reg_fence(s, 0, KC);
          if (tail) {
#pragma unroll
            for (int c = 0; c < KC; ++c)
              if (c >= lim) s[c] = __float_as_uint(-INFINITY);
          }
          max_cols(0, KC);
        }
        if constexpr (G::PSEP) {
          // S_t is in registers: the MMA warp may compute the next S_t now
          tc_fence_before();
          mbar_arrive(bar(G::B_S_FREE + t));
        }
        if constexpr (KC > 64) max_cols(64, KC);
        const float mxs = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
        if (j == 0) {
          // a row that sees no key keeps m = 0: all its weights are 0
          m = mxs == -INFINITY ? 0.f : mxs;
        } else {
          const bool need = mxs > m + kRescaleThreshold;
          if (__any_sync(0xffffffffu, need)) {
            // O_t must hold P(j-1) V(j-1) before it is rescaled
            if (!(ok = wait_(bar(G::B_PV_DONE + t), (p_cnt - 1) & 1u))) break;
            tc_fence_after();
            const float alpha = need ? ex2(m - mxs) : 1.0f;
            if (need) m = mxs;
            l *= alpha;
#pragma unroll
            for (int c = 0; c < G::DP; c += 16) {
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
        // p = 2^(s * scale * log2(e) - m), packed two lanes per FMA/add;
        // exp_pairs(c0, c1, pk) fills pk[0, c1 - c0) with packed columns
        // [c0, c1) (keys 2 c0 ... 2 c1 - 1 of this thread's columns)
        const float2 c2 = make_float2(sl2, sl2);
        const float2 nm2 = make_float2(-m, -m);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
        auto exp_pairs = [&](int c0, int c1, uint32_t* pk) {
#pragma unroll
          for (int c = c0; c < c1; c += 2) {
            float2 a = __ffma2_rn(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])),
                                  c2, nm2);
            float2 b = __ffma2_rn(make_float2(__uint_as_float(s[2 * c + 2]),
                                              __uint_as_float(s[2 * c + 3])), c2, nm2);
            // group c / 2 of four columns: FMA-pipe polynomial or MUFU
            // (a compile-time choice once the loop is unrolled)
            if (((c >> 1) * G::POLY) % kPolyDen < G::POLY) {
              a = exp2_poly2(a);
              b = exp2_poly2(b);
            } else {
              a.x = ex2(a.x);
              a.y = ex2(a.y);
              b.x = ex2(b.x);
              b.y = ex2(b.y);
            }
            if constexpr (!G::LO) {
              acc0 = __fadd2_rn(acc0, a);
              acc1 = __fadd2_rn(acc1, b);
            }
            pk[c - c0] = pack_bf16x2(a.x, a.y);
            pk[c - c0 + 1] = pack_bf16x2(b.x, b.y);
          }
        };
        if constexpr (G::PSEP) {
          uint32_t pk[KC / 2];
          exp_pairs(0, KC / 2, pk);
          // P_t(j-1) must have been read by its P.V before it is overwritten
          if (p_cnt > 0 && !(ok = wait_(bar(G::B_PV_DONE + t), (p_cnt - 1) & 1u))) break;
          tc_fence_after();
          tmem_st_cols<KC / 2>(tP, pk);
        } else {
          // P_t overwrites the first half of S_t, already in registers
#pragma unroll
          for (int hh = 0; hh < KN / 64; ++hh) {
            uint32_t pk[32];
            exp_pairs(32 * hh, 32 * hh + 32, pk);
            tmem_st32(tP + 32 * hh, *reinterpret_cast<const uint32_t(*)[32]>(pk));
          }
        }
        tmem_wait_st();
        if constexpr (!G::LO) l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
        tc_fence_before();
        mbar_arrive(bar(G::B_P_FULL + t));
        ++p_cnt;
      }
      if (!ok) break;
      // epilogue: O / l -> bf16 -> out (rows of this sequence only)
      if (!(ok = wait_(bar(G::B_PV_DONE + t), (p_cnt - 1) & 1u))) break;
      tc_fence_after();
      if constexpr (G::LO) {
        // the row sum is O column D (the ones column of V)
        uint32_t o[16];
        tmem_ld16(tO + (D / 16) * 16, o);
        tmem_wait_ld();
        reg_fence(o, 0, 16);
        l = __uint_as_float(o[D % 16]);
      }
      if (ui.part >= 0) {
        split_epilogue<D>(p.split + SL.parts, reinterpret_cast<int*>(p.split + SL.counters), tO, t,
                          r, m, l, orow, valid, ui.part, ui.part0, ui.tail, ui.chunks);
        continue;
      }
      // TMEM -> registers (O / l, bf16) -> shared memory -> TMA store.  Each
      // warp stages its 32 rows in the out map's box layout and its lane 0
      // stores them; rows at or past L_q are outside the map's extent and are
      // not written.
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      const int wrow = ui.q0 + kBlockM * t + kStoreRows * qq;  // warp's first row in the sequence
      const bool any_row = wrow < ui.lq;                        // warp-uniform
      const int rr = threadIdx.x & 31;                          // row within the box
      const uint32_t stg = base + G::STG_OFF + (uint32_t)warp * G::STG_WARP;
      uint8_t* stg_ptr = base_ptr + G::STG_OFF + (size_t)warp * G::STG_WARP;
      // the warp's stores of the previous unit have read the staging region
      if (rr == 0) bulk_wait_read_all();
      __syncwarp();
      // 16-byte chunk ch (columns 8 ch .. 8 ch + 7) of this thread's row: box
      // A (chunks 0-7, 128-byte swizzle), box B after it (head_dim 72, one
      // unswizzled chunk) or, for a 64-column box B, in box A's region
      auto put = [&](int ch, uint4 v) {
        uint32_t off;
        if (ch < 8)
          off = (uint32_t)rr * 128u + (uint32_t)((ch ^ (rr & 7)) * 16);
        else if constexpr (G::ZB)
          off = G::STG_A_BYTES + (uint32_t)rr * 16u;
        else
          off = (uint32_t)rr * 128u + (uint32_t)(((ch - 8) ^ (rr & 7)) * 16);
        *reinterpret_cast<uint4*>(stg_ptr + off) = v;
      };
      auto store_box = [&](const uint8_t* map, int col0) {
        fence_proxy_async_smem();  // this thread's staging writes, to the async proxy
        __syncwarp();
        if (rr == 0 && any_row) {
          tma_store_3d(map, stg, col0, ui.head, wrow);
          bulk_commit();
        }
      };
#pragma unroll
      for (int c = 0; c < G::DP; c += 16) {
        if (c == 64 && !G::ZB) {
          // box A's columns are staged: store them, then reuse the region
          store_box(mo, 0);
          if (rr == 0) bulk_wait_read_all();
          __syncwarp();
        }
        uint32_t o[16];
        tmem_ld16(tO + c, o);
        tmem_wait_ld();
        reg_fence(o, 0, 16);
        if (c < D) {
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
          put(c / 8, make_uint4(w[0], w[1], w[2], w[3]));
          if (c + 8 < D) put(c / 8 + 1, make_uint4(w[4], w[5], w[6], w[7]));
        }
      }
      if constexpr (G::NB == 1) {
        store_box(mo, 0);
      } else if constexpr (G::ZB) {
        store_box(mo, 0);
        // box B from its own region
        if (rr == 0 && any_row) {
          tma_store_3d(mob, stg + G::STG_A_BYTES, G::BW, ui.head, wrow);
          bulk_commit();
        }
      } else {
        store_box(mob, G::BW);
      }
      (void)orow;
      (void)valid;
    }
    // every store of this warp has read its staging region before the CTA
    // exits (the global writes complete on their own)
    if ((threadIdx.x & 31) == 0) bulk_wait_read_all();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // a CTA that gave up may have left split-region row counters counted in
  if (threadIdx.x == 0 && *abort_flag && p.split_cap > 0) p.status[kHdrCountersDirty] = 1;
  if (warp == G::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- launch
// A small batch plans in four warps, a larger one in eight or 32 (fewer
// threads to launch and to synchronise; four warps still spread the map
// writes and, when they are dirty, the zeroing of the split region's row
// counters); the kernel's loops take any multiple of 32 threads.
cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream) {
  const int threads = p.num_seqs <= 128 ? 128 : (p.num_seqs <= 256 ? 256 : 1024);
#if ATTN_VARLEN_PLAN_PDL
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_varlen_plan_kernel, p);
#else
  attn_varlen_plan_kernel<<<1, threads, 0, stream>>>(p);
  return cudaGetLastError();
#endif
}

// Launched as a programmatic dependent of the plan kernel: its CTAs start
// (barrier init, TMEM allocation) while the plan kernel still runs.
template <int D>
static cudaError_t launch_fwd_t(const FwdParams& p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)Geometry<D>::THREADS);
  cfg.dynamicSmemBytes = Geometry<D>::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_varlen_fwd_kernel<D>, p);
}

// head_dim dispatch: calls f(std::integral_constant<int, D>) for a built D.
template <typename F>
static auto with_head_dim(int head_dim, F&& f) -> decltype(f(std::integral_constant<int, 72>{})) {
  switch (head_dim) {
    case 64: return f(std::integral_constant<int, 64>{});
    case 72: return f(std::integral_constant<int, 72>{});
    case 80: return f(std::integral_constant<int, 80>{});
    case 96: return f(std::integral_constant<int, 96>{});
    default: return f(std::integral_constant<int, 128>{});
  }
}

bool head_dim_supported(int head_dim) {
  return head_dim == 64 || head_dim == 72 || head_dim == 80 || head_dim == 96 ||
         head_dim == 128 || head_dim == 256;
}

// head_dim 256 runs its own kernel (attn_varlen_d256.cu); every other
// supported head_dim an instance of attn_varlen_fwd_kernel.
cudaError_t prepare_fwd(int head_dim) {
  if (!head_dim_supported(head_dim)) return cudaErrorInvalidValue;
  if (head_dim == 256) return prepare_fwd_d256();
  return with_head_dim(head_dim, [](auto d) {
    constexpr int D = decltype(d)::value;
    return cudaFuncSetAttribute(attn_varlen_fwd_kernel<D>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Geometry<D>::SMEM_BYTES);
  });
}

cudaError_t launch_fwd(int head_dim, const FwdParams& p, int grid, cudaStream_t stream) {
  if (!head_dim_supported(head_dim)) return cudaErrorInvalidValue;
  if (head_dim == 256) return launch_fwd_d256(p, grid, stream);
  return with_head_dim(head_dim, [&](auto d) { return launch_fwd_t<decltype(d)::value>(p, grid, stream); });
}

int fwd_threads(int head_dim) {
  if (head_dim == 256) return fwd_threads_d256();
  return with_head_dim(head_dim, [](auto d) { return Geometry<decltype(d)::value>::THREADS; });
}

size_t fwd_smem_bytes(int head_dim) {
  if (head_dim == 256) return fwd_smem_bytes_d256();
  return with_head_dim(head_dim,
                       [](auto d) { return (size_t)Geometry<decltype(d)::value>::SMEM_BYTES; });
}

int box_cols(int head_dim) {
  if (head_dim == 256) return 64;
  return with_head_dim(head_dim, [](auto d) { return Cfg<decltype(d)::value>::BW; });
}

int kv_tile_rows(int head_dim) {
  if (head_dim == 256) return kv_tile_rows_d256();
  return with_head_dim(head_dim, [](auto d) { return Cfg<decltype(d)::value>::KN; });
}

int box_b_cols(int head_dim) {
  if (head_dim == 256) return 64;  // four 64-column boxes of the box-A map
  return with_head_dim(head_dim, [](auto d) {
    using G = Geometry<decltype(d)::value>;
    return G::NB == 1 ? G::BW : G::WB;  // one box: box B is never loaded
  });
}

bool box_b_swizzle_128(int head_dim) {
  if (head_dim == 256) return true;
  return with_head_dim(head_dim, [](auto d) { return !Geometry<decltype(d)::value>::ZB; });
}

bool tail_split_supported(int head_dim) { return head_dim != 256; }

}  // namespace avp
