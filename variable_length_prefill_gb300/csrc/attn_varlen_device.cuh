// Device-side pieces shared by the attention kernels (attn_varlen_kernels.cu
// and attn_varlen_d256.cu): work-unit decoding and the bounded waits.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "attn_varlen_internal.h"
#include "ptx.cuh"

namespace avp {

namespace {

constexpr int kItemDepth = 4;  // work items handed from the producer to the other roles
// The producer claims a CTA's next work item once the current item's last
// K/V load is issued (else: when the current item starts).
#ifndef ATTN_VARLEN_LATE_CLAIM
#define ATTN_VARLEN_LATE_CLAIM 1
#endif
// Lazy rescale: a row's running max is only raised when the new maximum
// exceeds it by more than this (log2 units), so exponentials stay <= 2^8.
constexpr float kRescaleThreshold = 8.0f;
// Time after which a wait gives up.  The product build waits 4 s; a test
// build shortens it to run the give-up path (see ATTN_VARLEN_TEST_HOOKS).
#ifndef ATTN_VARLEN_WAIT_LIMIT_NS
#define ATTN_VARLEN_WAIT_LIMIT_NS 4000000000ull
#endif
constexpr uint64_t kWaitLimitNs = ATTN_VARLEN_WAIT_LIMIT_NS;

struct UnitInfo {
  int seq, head, q0, lq, lk, qbase;
  int jb, nkv;     // this item's key tiles: [jb, jb + nkv) (Q tile 1, or 0 alone)
  int nkv0;        // key tiles Q tile 0 needs (< nkv only with the causal mask)
  int coff;        // causal mask: row r sees keys <= r + coff (coff = L_k - L_q)
  int chunks;      // items the unit is split into (1: not split)
  int part, part0, tail;  // split items: partial slot, the unit's first slot, tail unit
  bool t1;  // second Q tile holds at least one row
};

// Unit u -> sequence, head (offset by head_begin: the call may cover a
// sub-range of the tensors' heads), 256-row block and key-tile range.
__device__ __forceinline__ UnitInfo decode_unit(int u, const int32_t* __restrict__ order,
                                                const int32_t* __restrict__ prefix, int num_seqs,
                                                const int32_t* __restrict__ cu_q,
                                                const int32_t* __restrict__ cu_k, int kn,
                                                bool causal, int head_begin) {
  // largest rank r in [0, num_seqs) with prefix[r] <= u
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(prefix + mid) <= u) lo = mid; else hi = mid - 1;
  }
  UnitInfo ui;
  ui.seq = __ldg(order + lo);
  const int local = u - __ldg(prefix + lo);
  ui.qbase = __ldg(cu_q + ui.seq);
  ui.lq = __ldg(cu_q + ui.seq + 1) - ui.qbase;
  const int kb = __ldg(cu_k + ui.seq);
  ui.lk = __ldg(cu_k + ui.seq + 1) - kb;
  if (ui.lk < 0) ui.lk = 0;
  const int pairs = (ui.lq + kUnitRows - 1) / kUnitRows;
  const int hl = local / pairs;
  ui.head = head_begin + hl;
  const int qb = local - hl * pairs;
  // causal: the last row blocks see the most keys, so they go first
  ui.q0 = (causal ? pairs - 1 - qb : qb) * kUnitRows;
  ui.t1 = ui.q0 + kBlockM < ui.lq;
  ui.nkv = (ui.lk + kn - 1) / kn;
  ui.nkv0 = ui.nkv;
  ui.coff = ui.lk - ui.lq;
  if (causal) {
    // keys visible to the last row of each tile: min(L_k, row + 1 + coff)
    const int last1 = min(ui.q0 + kUnitRows, ui.lq) - 1;
    const int last0 = min(ui.q0 + kBlockM, ui.lq) - 1;
    const int k1 = max(0, min(ui.lk, last1 + 1 + ui.coff));
    const int k0 = max(0, min(ui.lk, last0 + 1 + ui.coff));
    ui.nkv = (k1 + kn - 1) / kn;
    ui.nkv0 = (k0 + kn - 1) / kn;
  }
  ui.jb = 0;
  ui.chunks = 1;
  ui.part = ui.part0 = ui.tail = -1;
  return ui;
}

// Work item -> unit and key-tile range.  Items below split_start are whole
// units; the others are chunks of the tail units (tail_prefix).
__device__ __forceinline__ UnitInfo decode_item(int it, const int32_t* __restrict__ order,
                                                const int32_t* __restrict__ prefix, int num_seqs,
                                                const int32_t* __restrict__ cu_q,
                                                const int32_t* __restrict__ cu_k, int kn,
                                                int split_start, int num_units,
                                                const int32_t* __restrict__ tail_prefix,
                                                bool causal, int head_begin) {
  if (it < split_start)
    return decode_unit(it, order, prefix, num_seqs, cu_q, cu_k, kn, causal, head_begin);
  const int k = it - split_start;
  int lo = 0, hi = num_units - split_start - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(tail_prefix + mid) <= k) lo = mid; else hi = mid - 1;
  }
  // (split units are never causal: the plan does not split under the mask)
  UnitInfo ui =
      decode_unit(split_start + lo, order, prefix, num_seqs, cu_q, cu_k, kn, causal, head_begin);
  const int c0 = __ldg(tail_prefix + lo);
  const int chunks = __ldg(tail_prefix + lo + 1) - c0;
  if (chunks > 1) {
    const int c = k - c0;
    const int jb = (int)(((long long)c * ui.nkv) / chunks);
    const int je = (int)(((long long)(c + 1) * ui.nkv) / chunks);
    ui.jb = jb;
    ui.nkv = je - jb;
    ui.nkv0 = ui.nkv;
    ui.chunks = chunks;
    ui.part = k;
    ui.part0 = c0;
    ui.tail = lo;
  }
  return ui;
}

// Bounded wait: spins on the barrier, gives up after kWaitLimitNs or as soon
// as another role of the CTA has given up.  Returns false on give-up.
__device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int* status, int code) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, code);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             int* status, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bounded_slow(bar, parity, abort_flag, status, code);
}

// Wait with a fixed bound and no abort check (used only while draining).
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
}

}  // namespace

}  // namespace avp
