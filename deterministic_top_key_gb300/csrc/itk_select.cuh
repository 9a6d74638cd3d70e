// The selection kernel: exact top-k of each query's candidate list (written by the scan
// kernel), sorted by the total order of the 64-bit selection key, written as the query's
// output row of ids and scores.
//
// Operation: flashinfer PR #8691, opening description -- top-k key ids and scores per
// query, ties to the larger id; the candidate lists hold every key of the query's top-k
// (the scan's filter only drops keys below top_k keys already seen), so selecting within
// them gives the exact answer.
//
// Work distribution: a persistent grid; each 128-thread group draws one query at a time
// from a self-resetting ticket word (same page, commit note on drawing work units from
// the ticket word and the TicketWord note).
//
// Per query (n candidates, keff = min(n, top_k) outputs): the candidates are counted into
// the 2048 bins of their score's top 11 bits; the bins that reach the first top_k
// positions are kept, and each kept bin b with c_b keys is spread over c_b sub-buckets by
// linear position inside the bin, so sub-buckets hold about one key each. Counting, a
// prefix sum and a scatter put every key into its sub-bucket's slot range, in descending
// order of sub-bucket; sorting each (tiny) sub-bucket in place finishes the order. Two
// exact fallbacks handle heavy ties: a radix select inside an oversized sub-bucket that
// crosses position top_k, and a full bitonic sort when some sub-bucket is large.
#pragma once

#include "itk_common.cuh"

namespace itk {

constexpr int kSelGroups = 4;                 // 128-thread groups per selection CTA
constexpr int kSelThreads = kSelGroups * 128;
constexpr int kStageSlack = 256;              // staging slots past top_k
constexpr int kBigBucket = 32;                // sub-buckets above this size take the full sort

// Per-group shared memory of the selection kernel (offsets within the group's slice).
// The bin and sub-bucket arrays carry one pad word per run of entries that one thread
// scans (16 bins, 32 sub-buckets), so that the 32 lanes of a warp, each walking its own
// run, hit 32 different banks.
constexpr uint32_t kSgBins = 0;                                        // 2048 + 128 x u32
constexpr uint32_t kSgSub = kSgBins + (kBins + kBins / 16) * 4;        // 4096 + 128 x u32
constexpr uint32_t kSgStage = kSgSub + (kCap + kCap / 32) * 4;         // (2048 + 256) x u64
constexpr uint32_t kSgRadix = kSgStage + (kMaxTopK + kStageSlack) * 8; // 256 x u32
constexpr uint32_t kSgSel = kSgRadix + 256 * 4;                        // 8 x u32
constexpr uint32_t kSgFlags = kSgSel + 8 * 4;                          // 4 x u32
constexpr uint32_t kSgItem = kSgFlags + 4 * 4;                         // 4 x u32 (drawn item)
constexpr uint32_t kSgBytes = (kSgItem + 16 + 127) / 128 * 128;
constexpr uint32_t kSelSmemBytes = kSelGroups * kSgBytes;
static_assert(kSgStage % 16 == 0, "alignment");
static_assert(kSelSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t bin_pad(uint32_t b) { return b + (b >> 4); }
__device__ __forceinline__ uint32_t sub_pad(uint32_t i) { return i + (i >> 5); }

struct SelectParams {
  const int32_t* item_rows;           // per store slot: output row, or -1 (nothing to select there)
  int32_t n_items;                    // store slots
  int32_t top_k;
  TicketBlock* ticket;
  uint32_t* status;
  const unsigned long long* store;    // [n_items][kCap] candidate keys
  const uint32_t* counts;             // [n_items] candidates per slot
  int32_t* out_ids;                   // [T, top_k]
  float* out_scores;                  // [T, top_k]
};

// Exclusive prefix sum of the padded array a (entry i at a[sub_pad(i)], i < n <= 128 *
// kPerThread) in place, 128 threads, each scanning a run of kPerThread entries.
__device__ __forceinline__ void group_exclusive_scan_padded(const GroupCtx& c, uint32_t* a, uint32_t n) {
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    const uint32_t idx = c.gtid * kPerThread + i;
    s += idx < n ? a[sub_pad(idx)] : 0u;
  }
  uint32_t incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (c.lane >= off) incl += t;
  }
  if (c.lane == 31) c.sel[4 + c.gwarp] = incl;
  gsync(c);
  uint32_t run = incl - s;
#pragma unroll
  for (int wv = 0; wv < 4; ++wv) run += wv < c.gwarp ? c.sel[4 + wv] : 0u;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {  // second pass: the run is read again, not held
    const uint32_t idx = c.gtid * kPerThread + i;
    if (idx < n) {
      const uint32_t x = a[sub_pad(idx)];
      a[sub_pad(idx)] = run;
      run += x;
    }
  }
  gsync(c);
}

// Bitonic sort (descending) of a[0..np2) in shared memory, np2 a power of two.
__device__ void group_bitonic_desc(const GroupCtx& c, unsigned long long* a, uint32_t np2) {
  for (uint32_t size = 2; size <= np2; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t i = c.gtid; i < np2 / 2; i += 128) {
        const uint32_t lo = 2 * i - (i & (stride - 1));
        const uint32_t hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long x = a[lo], y = a[hi];
        if ((x < y) == desc) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      gsync(c);
    }
  }
}

// Slot-range index (in descending key order) of a kept candidate with score key h (the
// high word of its 64-bit key). ge[bin_pad(b)] counts kept candidates in bins >= b; bin
// b's keys own sub-buckets [ge(b+1), ge(b)) by linear position inside the bin (higher key
// first).
__device__ __forceinline__ uint32_t sub_bucket(const uint32_t* ge, uint32_t h) {
  const uint32_t b = h >> kBinShift;
  const uint32_t above = b + 1 < static_cast<uint32_t>(kBins) ? ge[bin_pad(b + 1)] : 0u;
  const uint32_t cb = ge[bin_pad(b)] - above;
  const uint32_t frac = h & ((1u << kBinShift) - 1u);         // position inside the bin
  const uint32_t sub = ((frac >> 9) * cb) >> (kBinShift - 9);  // 0 .. cb-1
  return above + (cb - 1u - sub);
}

// Exact fallback for the one sub-bucket that crosses position keff and is too large to
// sort in place (heavy ties): its `need` largest keys (bit r of in_b marks this thread's
// members, entry gtid + 128 r of buf) go to stage[start ..), unsorted. Kept out of line so
// that its 64-bit key registers do not weigh on the common path.
__device__ __noinline__ void sel_crossing_fallback(const GroupCtx& c, const unsigned long long* buf, uint32_t n,
                                                   uint32_t in_b, uint32_t need, uint32_t start,
                                                   unsigned long long* stage, uint32_t* flags) {
  unsigned long long v[kPerThread];
  group_load(c, buf, n, v);
  const unsigned long long pfx = group_select(c, v, in_b, need);
  if (c.gtid == 0) flags[3] = start;
  gsync(c);
#pragma unroll
  for (int r = 0; r < kPerThread; ++r) {
    const bool take = ((in_b >> r) & 1u) && v[r] >= pfx;
    const uint32_t slot = warp_append_slot(take, &flags[3], c.lane);
    if (take && slot < start + need) stage[slot] = v[r];  // exactly `need` keys qualify: keys are distinct
  }
  gsync(c);
}

// Exact top-k of one query's n candidates (buf[0..n), n <= kCap), sorted by the total
// order, written as one output row. Each thread holds the score keys (high words) of
// candidates gtid + 128 r in registers; full 64-bit keys are read again from buf only to
// place them.
__device__ __forceinline__ void sel_finish(const GroupCtx& c, const unsigned long long* buf, uint32_t n,
                                           uint32_t top_k, uint32_t* ge, uint32_t* sub, unsigned long long* stage,
                                           uint32_t* flags, int32_t* out_ids, float* out_scores) {
  const uint32_t* buf_hi = reinterpret_cast<const uint32_t*>(buf) + 1;  // high word of entry i at buf_hi[2 i]
  uint32_t hk[kPerThread];
  uint32_t valid = 0;
#pragma unroll
  for (int r = 0; r < kPerThread; ++r) {
    const uint32_t idx = c.gtid + 128u * r;
    hk[r] = idx < n ? buf_hi[2 * idx] : 0u;
    valid |= (idx < n ? 1u : 0u) << r;
  }
  const uint32_t keff = n < top_k ? n : top_k;
  // count the candidates per bin
  for (int i = c.gtid; i < kBins + kBins / 16; i += 128) ge[i] = 0u;
  if (c.gtid == 0) {
    flags[0] = kBins - 1;    // first kept bin
    flags[1] = 0u;           // large sub-bucket seen
    flags[2] = 0xFFFFFFFFu;  // sub-bucket that crosses top_k and overflows the staging area
  }
  gsync(c);
#pragma unroll
  for (int r = 0; r < kPerThread; ++r)
    if ((valid >> r) & 1u) atomicAdd(&ge[bin_pad(hk[r] >> kBinShift)], 1u);
  gsync(c);
  // ge(b) = candidates in bins >= b (suffix sums, 16 bins per thread, highest bins first)
  {
    uint32_t loc[16];
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      loc[i] = ge[bin_pad(kBins - 1 - (16 * c.gtid + i))];
      s += loc[i];
    }
    uint32_t incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (c.lane >= off) incl += t;
    }
    if (c.lane == 31) c.sel[4 + c.gwarp] = incl;
    gsync(c);
    uint32_t run = incl - s;
#pragma unroll
    for (int wv = 0; wv < 4; ++wv) run += wv < c.gwarp ? c.sel[4 + wv] : 0u;
    uint32_t first_kept = kBins - 1;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t b = kBins - 1 - (16 * c.gtid + i);
      // run = candidates in bins above b; bin b reaches a position below top_k iff run < top_k
      if (run < top_k) first_kept = b;
      run += loc[i];
      ge[bin_pad(b)] = run;
    }
    atomicMin(&flags[0], first_kept);
  }
  gsync(c);
  const uint32_t tstar = flags[0];
  const uint32_t m_keep = ge[bin_pad(tstar)];  // candidates in kept bins
  for (uint32_t i = c.gtid; i < m_keep; i += 128) sub[sub_pad(i)] = 0u;
  gsync(c);
  uint32_t kept = 0;  // bit r: candidate r lies in a kept bin
#pragma unroll
  for (int r = 0; r < kPerThread; ++r) {
    if (((valid >> r) & 1u) && (hk[r] >> kBinShift) >= tstar) {
      kept |= 1u << r;
      atomicAdd(&sub[sub_pad(sub_bucket(ge, hk[r]))], 1u);
    }
  }
  gsync(c);
  group_exclusive_scan_padded(c, sub, m_keep);  // sub(i) = first slot of sub-bucket i
  const uint32_t cap = top_k + kStageSlack;
#pragma unroll
  for (int r = 0; r < kPerThread; ++r) {
    if ((kept >> r) & 1u) {
      const uint32_t pos = atomicAdd(&sub[sub_pad(sub_bucket(ge, hk[r]))], 1u);
      if (pos < cap) stage[pos] = buf[c.gtid + 128u * r];
    }
  }
  gsync(c);
  // sub(i) is now the end of sub-bucket i; sort every sub-bucket that reaches a slot below
  // top_k, in place (they hold about one key each)
  for (uint32_t i = c.gtid; i < m_keep; i += 128) {
    const uint32_t start = i ? sub[sub_pad(i - 1)] : 0u;
    const uint32_t end = sub[sub_pad(i)];
    if (start >= keff || end - start < 2) continue;
    if (end > keff && (end > cap || end - start > static_cast<uint32_t>(kBigBucket))) {
      flags[2] = i;  // the one sub-bucket that crosses position keff, too large to sort here
      continue;
    }
    if (end - start > static_cast<uint32_t>(kBigBucket)) {
      flags[1] = 1u;
      continue;
    }
    for (uint32_t a = start + 1; a < end; ++a) {
      const unsigned long long x = stage[a];
      uint32_t b = a;
      while (b > start && stage[b - 1] < x) {
        stage[b] = stage[b - 1];
        --b;
      }
      stage[b] = x;
    }
  }
  gsync(c);
  const uint32_t over = flags[2];
  if (over != 0xFFFFFFFFu) {
    const uint32_t start = over ? sub[sub_pad(over - 1)] : 0u;
    uint32_t in_b = 0;
#pragma unroll
    for (int r = 0; r < kPerThread; ++r)
      if (((kept >> r) & 1u) && sub_bucket(ge, hk[r]) == over) in_b |= 1u << r;
    sel_crossing_fallback(c, buf, n, in_b, keff - start, start, stage, flags);
    if (c.gtid == 0) flags[1] = 1u;  // the refilled range is unsorted
    gsync(c);
  }
  if (flags[1]) {
    uint32_t np2 = 2;
    while (np2 < keff) np2 <<= 1;
    for (uint32_t i = keff + c.gtid; i < np2; i += 128) stage[i] = 0ull;
    gsync(c);
    group_bitonic_desc(c, stage, np2);
  }
  for (uint32_t r = c.gtid; r < top_k; r += 128) {
    if (r < keff) {
      const unsigned long long x = stage[r];
      st_stream_s32(out_ids + r, static_cast<int32_t>(static_cast<uint32_t>(x & 0xFFFFFFFFull)));
      st_stream_f32(out_scores + r, key_to_float(static_cast<uint32_t>(x >> 32)));
    } else {
      st_stream_s32(out_ids + r, -1);
      st_stream_f32(out_scores + r, -__int_as_float(0x7F800000));
    }
  }
  gsync(c);
}

__global__ void __launch_bounds__(kSelThreads, 1) indexer_topk_select_kernel(const SelectParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int g = threadIdx.x >> 7;
  uint8_t* gs = smem + g * kSgBytes;
  GroupCtx c;
  c.gtid = threadIdx.x & 127;
  c.gwarp = c.gtid >> 5;
  c.lane = threadIdx.x & 31;
  c.bar = 1 + g;
  c.radix = reinterpret_cast<uint32_t*>(gs + kSgRadix);
  c.sel = reinterpret_cast<uint32_t*>(gs + kSgSel);
  uint32_t* ge = reinterpret_cast<uint32_t*>(gs + kSgBins);
  uint32_t* sub = reinterpret_cast<uint32_t*>(gs + kSgSub);
  unsigned long long* stage = reinterpret_cast<unsigned long long*>(gs + kSgStage);
  uint32_t* flags = reinterpret_cast<uint32_t*>(gs + kSgFlags);
  volatile unsigned long long* s_item = reinterpret_cast<volatile unsigned long long*>(gs + kSgItem);
  const unsigned long long n_items = static_cast<unsigned long long>(p.n_items);

  while (true) {
    if (c.gtid == 0) *s_item = atomicAdd(&p.ticket->next, 1ull);
    gsync(c);
    const unsigned long long item = *s_item;
    gsync(c);  // every thread has read the item before the next draw overwrites it
    if (item >= n_items) break;
    const int32_t out_row = p.item_rows[item];
    if (out_row < 0) continue;
    const size_t row = static_cast<size_t>(out_row);
    uint32_t n = p.counts[item];
    if (n > static_cast<uint32_t>(kCap)) {  // cannot happen: the scan hands off at most kCap keys
      if (c.gtid == 0) atomicOr(p.status, kStatusInternal | (20u << 8));
      n = kCap;
    }
    sel_finish(c, p.store + item * kCap, n, static_cast<uint32_t>(p.top_k), ge, sub, stage, flags,
               p.out_ids + row * p.top_k, p.out_scores + row * p.top_k);
  }
  __syncthreads();
  if (threadIdx.x == 0) ticket_release(p.ticket);
}

// ------------------------------------------------------------------ split-query merge
// A query whose visible keys were scanned by several units (a split tail) has one
// candidate list per unit. One 256-thread CTA per such query histograms the union over
// the 2048 score bins, keeps every key in the bins that reach the first top_k positions
// when that fits in kCap, and otherwise keeps exactly the top_k keys (a radix select on
// the bits below the bin inside the crossing bin). The result goes to the query's own
// store slot, which the selection kernel then sorts like any other.
constexpr int kMergeThreads = 256;

struct MergeParams {
  const MergeDesc* merges;
  int32_t n_merges;
  int32_t top_k;
  const UnitDesc* units;
  unsigned long long* store;
  uint32_t* counts;
  uint32_t* status;
};

__global__ void __launch_bounds__(kMergeThreads) indexer_topk_merge_kernel(const MergeParams p) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t radix[256];
  __shared__ uint32_t sel[8];
  __shared__ uint32_t wsum[kMergeThreads / 32];
  __shared__ uint32_t s_cursor;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const MergeDesc m = p.merges[blockIdx.x];
  const uint32_t K = static_cast<uint32_t>(p.top_k);
  GroupCtx c;  // warp 0 picks radix digits, as in a 128-thread group
  c.gtid = tid;
  c.gwarp = warp;
  c.lane = lane;
  c.bar = 0;
  c.radix = radix;
  c.sel = sel;
  auto chunk_slot = [&](int ch) { return static_cast<size_t>(m.first_unit + ch) * kQB + m.j; };
  auto chunk_count = [&](int ch) {
    const uint32_t n = p.counts[chunk_slot(ch)];
    return n < static_cast<uint32_t>(kCap) ? n : static_cast<uint32_t>(kCap);
  };
  for (int i = tid; i < kBins; i += kMergeThreads) hist[i] = 0u;
  __syncthreads();
  for (int ch = 0; ch < m.n_chunks; ++ch) {
    const unsigned long long* src = p.store + chunk_slot(ch) * kCap;
    const uint32_t n = chunk_count(ch);
    for (uint32_t i = tid; i < n; i += kMergeThreads) atomicAdd(&hist[bin_of(src[i])], 1u);
  }
  __syncthreads();
  // ge(b) = keys in bins >= b: each thread sums 8 bins, highest bins first
  constexpr int kPer = kBins / kMergeThreads;
  uint32_t loc[kPer];
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    loc[i] = hist[kBins - 1 - (kPer * tid + i)];
    s += loc[i];
  }
  uint32_t incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) wsum[warp] = incl;
  if (tid == 0) sel[3] = 0u;  // tstar: the lowest bin kept (0 when fewer than K keys in all)
  __syncthreads();
  uint32_t run = incl - s;
  for (int wv = 0; wv < warp; ++wv) run += wsum[wv];
  __syncthreads();  // every thread has its run before hist is rewritten
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t b = kBins - 1 - (kPer * tid + i);
    const uint32_t above = run;  // keys in bins > b
    run += loc[i];
    hist[b] = run;               // now ge(b)
    if (above < K && run >= K) sel[3] = b;  // the bin that reaches position K (at most one)
  }
  __syncthreads();
  const uint32_t tstar = sel[3];
  const uint32_t ge_t = hist[tstar];
  const uint32_t ge_above = tstar + 1 < static_cast<uint32_t>(kBins) ? hist[tstar + 1] : 0u;
  __syncthreads();
  unsigned long long thr_key = static_cast<unsigned long long>(tstar) << (32 + kBinShift);
  if (ge_t > static_cast<uint32_t>(kCap)) {
    // exactly K: keys above bin tstar plus the (K - ge_above) largest inside bin tstar,
    // found by a radix select on the 53 bits below the bin (shifted to the top)
    unsigned long long prefix = 0ull;
    uint32_t k_rem = K - ge_above;
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kMergeThreads) radix[i] = 0u;
      __syncthreads();
      const unsigned long long hi_mask = (shift == 56) ? 0ull : (~0ull << (shift + 8));
      for (int ch = 0; ch < m.n_chunks; ++ch) {
        const unsigned long long* src = p.store + chunk_slot(ch) * kCap;
        const uint32_t n = chunk_count(ch);
        for (uint32_t i = tid; i < n; i += kMergeThreads) {
          const unsigned long long x = src[i];
          const unsigned long long y = x << (32 - kBinShift);  // the bits below the bin
          if (bin_of(x) == tstar && (y & hi_mask) == (prefix & hi_mask)) atomicAdd(&radix[(y >> shift) & 0xFFu], 1u);
        }
      }
      __syncthreads();
      group_pick_digit(c, k_rem);
      __syncthreads();
      prefix |= static_cast<unsigned long long>(sel[0]) << shift;
      k_rem = sel[1];
      const uint32_t cnt = sel[2];
      __syncthreads();
      if (cnt == k_rem) break;  // uniform
    }
    thr_key |= prefix >> (32 - kBinShift);
  }
  // keep every key at or above the threshold key
  if (tid == 0) s_cursor = 0u;
  __syncthreads();
  unsigned long long* dst = p.store + static_cast<size_t>(m.out_slot) * kCap;
  for (int ch = 0; ch < m.n_chunks; ++ch) {
    const unsigned long long* src = p.store + chunk_slot(ch) * kCap;
    const uint32_t n = chunk_count(ch);
    for (uint32_t base = 0; base < n; base += kMergeThreads) {
      const uint32_t i = base + tid;
      const unsigned long long x = i < n ? src[i] : 0ull;
      const bool keep = i < n && x >= thr_key;
      const uint32_t slot = warp_append_slot(keep, &s_cursor, lane);
      if (keep && slot < static_cast<uint32_t>(kCap)) dst[slot] = x;
    }
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t n = s_cursor;
    if (n > static_cast<uint32_t>(kCap)) {  // cannot happen: at most max(ge_t, K) <= kCap keys qualify
      atomicOr(p.status, kStatusInternal | (22u << 8));
      n = kCap;
    }
    p.counts[m.out_slot] = n;
  }
}

}  // namespace itk

