// Definitions shared by the scan, merge and selection kernels: problem constants, the
// 64-bit selection key, the work-unit and ticket records, and the thread-group primitives
// (named-barrier sync, radix digit pick, aggregated appends).
//
// Operation: flashinfer PR #8691 ("perf(cake_dsa_indexer_det): ticket scheduling on
// sm_107a, no fill kernel in eager entry"), opening description -- BF16 q/k, FP32 w and
// scores, top-k key ids per query, ties to the larger id, ids and scores independent of
// partition or chunking.
//
// Selection key: the FP32 score is mapped to an unsigned word whose integer order is the
// float order (sign bit flipped for positives, all bits flipped for negatives), and the
// key id fills the low 32 bits. Comparing these 64-bit keys compares (score, id), so the
// order is total (larger id first among equal scores) and the top-k set and its order
// are unique.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "itk_ptx.cuh"

namespace itk {

constexpr int kHeads = 64;
constexpr int kDim = 128;
constexpr int kQB = 4;                       // queries per work unit
constexpr int kBlockKeys = 128;              // keys per tile (MMA M)
constexpr int kMaxTopK = 2048;
constexpr int kCap = 4096;                   // candidates per query handed from the scan to the selection
constexpr int kBinShift = 21;                // histogram bin = top 11 bits of the 32-bit score key
constexpr int kBins = 1 << (32 - kBinShift); // 2048 bins
constexpr int kMaxMergeChunks = 256;         // chunks (units) a split query's keys may span

constexpr uint32_t kStatusTimeout = 10u;   // matches ITK_ERR_DEVICE_TIMEOUT
constexpr uint32_t kStatusInternal = 11u;  // matches ITK_ERR_INTERNAL

struct UnitDesc {
  int32_t q_row0;    // first query row of the unit
  int32_t nq;        // queries in the unit (1..4)
  int32_t key_row0;  // first key row of the unit's segment
  int32_t pos0;      // causal position of the first query within its segment
  int32_t tile0;     // key tiles [tile0, tile1) of the segment that this unit scans
  int32_t tile1;     //   (all visible tiles, or one chunk of a split query block)
};

// A query whose visible keys were split over several units: its candidates sit in the
// store slots (unit u, query j) for u in [first_unit, first_unit + n_chunks); the merge
// selects its top_k from their union and writes output row `row`.
struct MergeDesc {
  int32_t first_unit;
  int32_t n_chunks;
  int32_t j;    // query index within the units (0..3)
  int32_t row;  // output row of the query
};

// Self-resetting work counter: CTAs draw items with atomicAdd on `next`; the last CTA to
// finish drawing (counted in `done`) puts both words back to zero for the next launch.
struct TicketBlock {
  unsigned long long next;
  unsigned long long done;
};

__device__ __forceinline__ uint32_t ord_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t o) {
  const uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(b);
}
__device__ __forceinline__ uint32_t bin_of(unsigned long long key) {
  return static_cast<uint32_t>(key >> (32 + kBinShift));
}

__device__ __forceinline__ void record_timeout(uint32_t* status, volatile uint32_t* abort_flag, uint32_t role) {
  *abort_flag = 1u;
  atomicOr(status, kStatusTimeout | (role << 8));
}

// Ends a persistent launch's use of its ticket block: called once per CTA after its last
// draw; the last CTA resets the block.
__device__ __forceinline__ void ticket_release(TicketBlock* t) {
  __threadfence();
  const unsigned long long prev = atomicAdd(&t->done, 1ull);
  if (prev == static_cast<unsigned long long>(gridDim.x) - 1ull) {
    atomicExch(&t->next, 0ull);
    atomicExch(&t->done, 0ull);
  }
}

// ------------------------------------------------------------------ 128-thread groups
struct GroupCtx {
  int gtid;        // 0 .. nthr - 1
  int gwarp;       // warp within the group
  int lane;
  uint32_t bar;    // named barrier id
  uint32_t nthr = 128;  // threads in the group
  uint32_t* radix; // 256 words of radix-select scratch
  uint32_t* sel;   // 8 words of scratch
};

__device__ __forceinline__ void gsync(const GroupCtx& c) { named_bar_sync(c.bar, c.nthr); }

// Warp-aggregated append: lanes with `pred` get consecutive slots from *counter.
__device__ __forceinline__ uint32_t warp_append_slot(bool pred, uint32_t* counter, int lane) {
  const uint32_t m = __ballot_sync(0xFFFFFFFFu, pred);
  uint32_t base = 0;
  if (m) {
    const int leader = __ffs(m) - 1;
    if (lane == leader) base = atomicAdd(counter, static_cast<uint32_t>(__popc(m)));
    base = __shfl_sync(0xFFFFFFFFu, base, leader);
  }
  return base + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
}

// Warp 0 of the group finds the radix digit that holds the K-th largest remaining key:
// cnt = c.radix (256 digit counts); writes sel[0] = digit, sel[1] = rank within the
// digit, sel[2] = keys in the digit.
__device__ __forceinline__ void group_pick_digit(const GroupCtx& c, uint32_t k_rem) {
  if (c.gwarp != 0) return;
  uint32_t cnt[8];
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    cnt[i] = c.radix[255 - 8 * c.lane - i];
    s += cnt[i];
  }
  uint32_t incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (c.lane >= off) incl += t;
  }
  const uint32_t excl = incl - s;
  if (excl < k_rem && k_rem <= incl) {
    uint32_t above = excl;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (above < k_rem && k_rem <= above + cnt[i]) {
        c.sel[0] = static_cast<uint32_t>(255 - 8 * c.lane - i);
        c.sel[1] = k_rem - above;
        c.sel[2] = cnt[i];
      }
      above += cnt[i];
    }
  }
}

}  // namespace itk
