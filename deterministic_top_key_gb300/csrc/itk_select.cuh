// The selection kernel: exact top-k of each query's candidate list (written by the scan
// kernel), sorted by the total order of the 64-bit selection key, written as the query's
// output row of ids and scores.
//
// Operation: flashinfer PR #8691, opening description -- top-k key ids and scores per
// query, ties to the larger id; the candidate lists hold every key of the query's top-k
// (the scan's filter only drops keys below top_k keys already seen), so selecting within
// them gives the exact answer.
//
// Work distribution: a persistent grid; each 256-thread group draws one query at a time
// from a self-resetting ticket word (same page, commit note on drawing work units from
// the ticket word and the TicketWord note).
//
// Per query (n candidates, keff = min(n, top_k) outputs): the candidates are counted into
// the 2048 bins of their score's top 11 bits; the bins that reach the first top_k
// positions are kept, and each kept bin b with c_b keys is spread over c_b sub-buckets by
// linear position inside the bin, so sub-buckets hold about one key each. Counting, a
// prefix sum and a scatter put every key into its sub-bucket's slot range, in descending
// order of sub-bucket; a key's place in the row is then its sub-bucket's start plus the
// number of keys above it in the same (tiny) sub-bucket, and it is written there
// directly. Heavy ties take exact fallbacks: in-place sorts of the sub-buckets, a radix
// select inside an oversized sub-bucket that crosses position top_k, and a full bitonic
// sort when some sub-bucket is large.
#pragma once

#include "itk_common.cuh"

namespace itk {

constexpr int kSG = 256;                      // threads of a selection group (one query at a time)
constexpr int kSelGroups = 3;                 // groups per selection CTA (80 registers a thread)
constexpr int kSelThreads = kSelGroups * kSG;
constexpr int kSelWarps = kSG / 32;           // warps of a group
constexpr int kSelPer = kCap / kSG;           // candidates a thread holds (entry gtid + kSG r)
constexpr int kBinsPer = kBins / kSG;         // bins a thread scans in the suffix sums
static_assert(kSelPer <= 32, "candidate masks are 32-bit");
constexpr int kStageSlack = 256;              // staging slots past top_k
constexpr int kBigBucket = 32;                // sub-buckets above this size take the full sort

// Per-group shared memory of the selection kernel (offsets within the group's slice).
// The bin and sub-bucket arrays carry one pad word per run of entries that one thread
// scans (kBinsPer bins, kSelPer sub-buckets), so that the 32 lanes of a warp, each
// walking its own run, hit 32 different banks.
constexpr uint32_t kSgBins = 0;                                        // 2048 + 256 x u32
constexpr uint32_t kSgSub = kSgBins + (kBins + kBins / kBinsPer) * 4;  // 4096 + 256 x u32
constexpr uint32_t kSgStage = kSgSub + (kCap + kCap / kSelPer) * 4;    // (2048 + 256) x u64
constexpr uint32_t kSgRadix = kSgStage + (kMaxTopK + kStageSlack) * 8; // 256 x u32
constexpr uint32_t kSgSel = kSgRadix + 256 * 4;                        // 16 x u32
constexpr uint32_t kSgFlags = kSgSel + 16 * 4;                         // 4 x u32
constexpr uint32_t kSgItem = kSgFlags + 4 * 4;                         // drawn item (u64), its row and count
constexpr uint32_t kSgBkt = kSgItem + 16;                              // (2048 + 256) x u16: sub-bucket of each staged key
constexpr uint32_t kSgBytes = (kSgBkt + (kMaxTopK + kStageSlack) * 2 + 127) / 128 * 128;
constexpr uint32_t kSelSmemBytes = kSelGroups * kSgBytes;
static_assert(kSgStage % 16 == 0, "alignment");
static_assert(kSelSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t bin_pad(uint32_t b) { return b + b / kBinsPer; }
__device__ __forceinline__ uint32_t sub_pad(uint32_t i) { return i + i / kSelPer; }

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
  uint32_t key_id_base;               // added to every written id (the keys hold global key rows)
};

// Exclusive prefix sum of the padded array a (entry i at a[sub_pad(i)], i < n <= kSG *
// kSelPer) in place, kSG threads, each scanning a run of kSelPer entries.
__device__ __forceinline__ void group_exclusive_scan_padded(const GroupCtx& c, uint32_t* a, uint32_t n) {
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < kSelPer; ++i) {
    const uint32_t idx = c.gtid * kSelPer + i;
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
  for (int wv = 0; wv < kSelWarps; ++wv) run += wv < c.gwarp ? c.sel[4 + wv] : 0u;
#pragma unroll
  for (int i = 0; i < kSelPer; ++i) {  // second pass: the run is read again, not held
    const uint32_t idx = c.gtid * kSelPer + i;
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
      for (uint32_t i = c.gtid; i < np2 / 2; i += kSG) {
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

// Radix select over the group's register-held keys (entry r valid iff bit r of `valid`):
// returns `prefix` with #{valid x : x >= prefix} == K (1 <= K <= valid keys; keys are
// distinct). Digits of 8 bits from the top; stops as soon as the digit holding the K-th
// largest key is selected whole.
__device__ unsigned long long sel_group_select(const GroupCtx& c, const unsigned long long (&v)[kSelPer],
                                               uint32_t valid, uint32_t K) {
  unsigned long long prefix = 0ull;
  uint32_t k_rem = K;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = c.gtid; i < 256; i += kSG) c.radix[i] = 0u;
    gsync(c);
    const unsigned long long hi_mask = (shift == 56) ? 0ull : (~0ull << (shift + 8));
#pragma unroll
    for (int r = 0; r < kSelPer; ++r) {
      if (((valid >> r) & 1u) && ((v[r] & hi_mask) == (prefix & hi_mask)))
        atomicAdd(&c.radix[(v[r] >> shift) & 0xFFu], 1u);
    }
    gsync(c);
    group_pick_digit(c, k_rem);
    gsync(c);
    const uint32_t b = c.sel[0];
    k_rem = c.sel[1];
    const uint32_t bucket = c.sel[2];
    prefix |= static_cast<unsigned long long>(b) << shift;
    if (bucket == k_rem) break;  // uniform across the group
  }
  gsync(c);  // c.sel may be reused right after
  return prefix;
}

// Exact fallback for the one sub-bucket that crosses position keff and is too large to
// sort in place (heavy ties): its `need` largest keys (bit r of in_b marks this thread's
// members, entry gtid + kSG r of buf) go to stage[start ..), unsorted. Kept out of line so
// that its 64-bit key registers do not weigh on the common path.
__device__ __noinline__ void sel_crossing_fallback(const GroupCtx& c, const unsigned long long* buf, uint32_t n,
                                                   uint32_t in_b, uint32_t need, uint32_t start,
                                                   unsigned long long* stage, uint32_t* flags) {
  unsigned long long v[kSelPer];
#pragma unroll
  for (int r = 0; r < kSelPer; ++r) {
    const uint32_t idx = c.gtid + static_cast<uint32_t>(kSG) * r;
    v[r] = idx < n ? buf[idx] : 0ull;
  }
  const unsigned long long pfx = sel_group_select(c, v, in_b, need);
  if (c.gtid == 0) flags[3] = start;
  gsync(c);
#pragma unroll
  for (int r = 0; r < kSelPer; ++r) {
    const bool take = ((in_b >> r) & 1u) && v[r] >= pfx;
    const uint32_t slot = warp_append_slot(take, &flags[3], c.lane);
    if (take && slot < start + need) stage[slot] = v[r];  // exactly `need` keys qualify: keys are distinct
  }
  gsync(c);
}

// Exact top-k of one query's n candidates (buf[0..n), n <= kCap), sorted by the total
// order, written as one output row. Each thread holds the 64-bit keys of candidates
// gtid + kSG r in registers.
__device__ __forceinline__ void sel_finish(const GroupCtx& c, const unsigned long long* buf, uint32_t n,
                                           uint32_t top_k, uint32_t* ge, uint32_t* sub, unsigned long long* stage,
                                           uint16_t* bkt, uint32_t* flags, int32_t* out_ids, float* out_scores,
                                           uint32_t id_base) {
  unsigned long long vk[kSelPer];  // full 64-bit keys; the score word is the high half
  // entry r of this thread is candidate gtid + kSG r: it exists for r < ceil((n - gtid) / kSG)
  const uint32_t n_mine = n > static_cast<uint32_t>(c.gtid) ? (n - c.gtid + kSG - 1u) / kSG : 0u;
#pragma unroll
  for (int r = 0; r < kSelPer; ++r) vk[r] = 0ull;
#pragma unroll
  for (int r = 0; r < kSelPer; ++r) {  // entries past this thread's count are skipped one by one
    if (r >= static_cast<int>(n_mine)) break;
    {
      vk[r] = buf[c.gtid + static_cast<uint32_t>(kSG) * r];
    }
  }
  const uint32_t keff = n < top_k ? n : top_k;
  // count the candidates per bin
  for (int i = c.gtid; i < kBins + kBins / kBinsPer; i += kSG) ge[i] = 0u;
  if (c.gtid == 0) {
    flags[0] = kBins - 1;    // first kept bin
    flags[1] = 0u;           // large sub-bucket seen
    flags[2] = 0xFFFFFFFFu;  // sub-bucket that crosses top_k and overflows the staging area
  }
  gsync(c);
#pragma unroll
  for (int r = 0; r < kSelPer; ++r) {  // entries past this thread's count are skipped one by one
    if (r >= static_cast<int>(n_mine)) break;
    {
      atomicAdd(&ge[bin_pad(static_cast<uint32_t>(vk[r] >> 32) >> kBinShift)], 1u);
    }
  }
  gsync(c);
  // ge(b) = candidates in bins >= b (suffix sums, kBinsPer bins per thread, highest bins first)
  {
    uint32_t loc[kBinsPer];
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < kBinsPer; ++i) {
      loc[i] = ge[bin_pad(kBins - 1 - (kBinsPer * c.gtid + i))];
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
    for (int wv = 0; wv < kSelWarps; ++wv) run += wv < c.gwarp ? c.sel[4 + wv] : 0u;
    uint32_t first_kept = kBins - 1;
#pragma unroll
    for (int i = 0; i < kBinsPer; ++i) {
      const uint32_t b = kBins - 1 - (kBinsPer * c.gtid + i);
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
  for (uint32_t i = c.gtid; i < m_keep; i += kSG) sub[sub_pad(i)] = 0u;
  gsync(c);
  uint32_t kept = 0;  // bit r: candidate r lies in a kept bin
#pragma unroll
  for (int r = 0; r < kSelPer; ++r) {  // entries past this thread's count are skipped one by one
    if (r >= static_cast<int>(n_mine)) break;
    {
      if ((static_cast<uint32_t>(vk[r] >> 32) >> kBinShift) >= tstar) {
        kept |= 1u << r;
        atomicAdd(&sub[sub_pad(sub_bucket(ge, static_cast<uint32_t>(vk[r] >> 32)))], 1u);
      }
    }
  }
  gsync(c);
  group_exclusive_scan_padded(c, sub, m_keep);  // sub(i) = first slot of sub-bucket i
  const uint32_t cap = top_k + kStageSlack;
#pragma unroll
  for (int r = 0; r < kSelPer; ++r) {  // entries past this thread's count are skipped one by one
    if (r >= static_cast<int>(n_mine)) break;
    {
      if (!((kept >> r) & 1u)) continue;
      const uint32_t b = sub_bucket(ge, static_cast<uint32_t>(vk[r] >> 32));
      const uint32_t pos = atomicAdd(&sub[sub_pad(b)], 1u);
      if (pos < cap) {
        stage[pos] = vk[r];
        bkt[pos] = static_cast<uint16_t>(b);
      }
    }
  }
  gsync(c);
  // sub(i) is now the end of sub-bucket i. Common case: every sub-bucket that reaches a
  // slot below keff is small and inside the staging area; each staged key's position is
  // then its sub-bucket's start plus the number of keys above it in that sub-bucket. A
  // thread that meets a large sub-bucket (or one that runs past the staging area) skips
  // it and raises flags[1]; the exact path below then rewrites the whole row.
  {  // optimistic placement: a heavy sub-bucket sets flags[1], and the exact path below rewrites the row
    bool heavy = false;
    const uint32_t staged = m_keep < cap ? m_keep : cap;
    constexpr int kSlots = 1;  // staged keys a thread places per pass (2 and 4 measured 0.2-1 % slower)
    for (uint32_t j0 = c.gtid; j0 < staged; j0 += kSG * kSlots) {
      uint32_t start[kSlots], end[kSlots];
      unsigned long long x[kSlots];
#pragma unroll
      for (int u = 0; u < kSlots; ++u) {
        const uint32_t j = j0 + static_cast<uint32_t>(kSG) * u;
        const bool v = j < staged;
        const uint32_t b = v ? bkt[j] : 0u;
        start[u] = v && b ? sub[sub_pad(b - 1)] : 0u;
        end[u] = v ? sub[sub_pad(b)] : 0u;
        if (start[u] >= keff) end[u] = start[u];  // lands at or past keff: nothing to place
        x[u] = v ? stage[j] : 0ull;
        if (end[u] - start[u] > static_cast<uint32_t>(kBigBucket) || (end[u] > keff && end[u] > cap)) {
          heavy = true;
          end[u] = start[u];
        }
      }
#pragma unroll
      for (int u = 0; u < kSlots; ++u) {
        uint32_t pos = start[u];
        for (uint32_t i = start[u]; i < end[u]; ++i) pos += stage[i] > x[u] ? 1u : 0u;
        if (end[u] > start[u] && pos < keff) {
          st_stream_s32(out_ids + pos, static_cast<int32_t>(static_cast<uint32_t>(x[u] & 0xFFFFFFFFull) + id_base));
          st_stream_f32(out_scores + pos, key_to_float(static_cast<uint32_t>(x[u] >> 32)));
        }
      }
    }
    for (uint32_t r = keff + c.gtid; r < top_k; r += kSG) {
      st_stream_s32(out_ids + r, -1);
      st_stream_f32(out_scores + r, -__int_as_float(0x7F800000));
    }
    if (heavy) flags[1] = 1u;
  }
  gsync(c);
  if (flags[1] == 0u) {  // uniform: read by every thread before anyone writes it again
    gsync(c);
    return;
  }
  gsync(c);  // every thread has read flags[1]
  if (c.gtid == 0) flags[1] = 0u;
  gsync(c);
  // Heavy ties: sort every sub-bucket that reaches a slot below top_k in place, resolve
  // an oversized crossing sub-bucket exactly, and sort the whole range when needed.
  for (uint32_t i = c.gtid; i < m_keep; i += kSG) {
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
    for (int r = 0; r < kSelPer; ++r)
      if (((kept >> r) & 1u) && sub_bucket(ge, static_cast<uint32_t>(vk[r] >> 32)) == over) in_b |= 1u << r;
    sel_crossing_fallback(c, buf, n, in_b, keff - start, start, stage, flags);
    if (c.gtid == 0) flags[1] = 1u;  // the refilled range is unsorted
    gsync(c);
  }
  if (flags[1]) {
    uint32_t np2 = 2;
    while (np2 < keff) np2 <<= 1;
    for (uint32_t i = keff + c.gtid; i < np2; i += kSG) stage[i] = 0ull;
    gsync(c);
    group_bitonic_desc(c, stage, np2);
  }
  for (uint32_t r = c.gtid; r < top_k; r += kSG) {
    if (r < keff) {
      const unsigned long long x = stage[r];
      st_stream_s32(out_ids + r, static_cast<int32_t>(static_cast<uint32_t>(x & 0xFFFFFFFFull) + id_base));
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
  const int g = threadIdx.x / kSG;
  uint8_t* gs = smem + g * kSgBytes;
  GroupCtx c;
  c.gtid = threadIdx.x % kSG;
  c.gwarp = c.gtid >> 5;
  c.nthr = kSG;
  c.lane = threadIdx.x & 31;
  c.bar = 1 + g;
  c.radix = reinterpret_cast<uint32_t*>(gs + kSgRadix);
  c.sel = reinterpret_cast<uint32_t*>(gs + kSgSel);
  uint32_t* ge = reinterpret_cast<uint32_t*>(gs + kSgBins);
  uint32_t* sub = reinterpret_cast<uint32_t*>(gs + kSgSub);
  unsigned long long* stage = reinterpret_cast<unsigned long long*>(gs + kSgStage);
  uint16_t* bkt = reinterpret_cast<uint16_t*>(gs + kSgBkt);
  uint32_t* flags = reinterpret_cast<uint32_t*>(gs + kSgFlags);
  volatile unsigned long long* s_item = reinterpret_cast<volatile unsigned long long*>(gs + kSgItem);
  const unsigned long long n_items = static_cast<unsigned long long>(p.n_items);
  grid_dep_wait();  // the scan (and merge) that wrote the candidates is complete

  // Items are drawn one ahead: thread 0 draws the next item (and reads its output row and
  // candidate count) while the group works on the current one, hiding those latencies.
  volatile uint32_t* s_meta = reinterpret_cast<volatile uint32_t*>(gs + kSgItem + 8);  // [0] row, [1] count
  auto publish = [&](unsigned long long it) {  // thread 0 only
    int32_t r = -1;
    uint32_t cnt = 0;
    if (it < n_items) {
      r = p.item_rows[it];
      cnt = p.counts[it];
    }
    *s_item = it;
    s_meta[0] = static_cast<uint32_t>(r);
    s_meta[1] = cnt;
  };
  if (c.gtid == 0) publish(atomicAdd(&p.ticket->next, 1ull));
  gsync(c);
  unsigned long long item = *s_item;
  int32_t out_row = static_cast<int32_t>(s_meta[0]);
  uint32_t n = s_meta[1];
  gsync(c);  // every thread has read the item before the next one is published
  while (item < n_items) {
    unsigned long long next = 0ull;
    if (c.gtid == 0) next = atomicAdd(&p.ticket->next, 1ull);  // used after this item's work
    if (out_row >= 0) {
      if (n > static_cast<uint32_t>(kCap)) {  // cannot happen: the scan hands off at most kCap keys
        if (c.gtid == 0) atomicOr(p.status, kStatusInternal | (20u << 8));
        n = kCap;
      }
      const size_t row = static_cast<size_t>(out_row);
      sel_finish(c, p.store + item * kCap, n, static_cast<uint32_t>(p.top_k), ge, sub, stage, bkt, flags,
                 p.out_ids + row * p.top_k, p.out_scores + row * p.top_k, p.key_id_base);
    }
    if (c.gtid == 0) publish(next);
    gsync(c);
    item = *s_item;
    out_row = static_cast<int32_t>(s_meta[0]);
    n = s_meta[1];
    gsync(c);  // every thread has read the item before the next one is published
  }
  __syncthreads();
  if (threadIdx.x == 0) ticket_release(p.ticket);
}

// ------------------------------------------------------------------ split-query merge
// A query whose visible keys were scanned by several units (a split tail) has one
// candidate list per unit. A cluster of kMergeCluster CTAs per such query selects its
// top_k from the union and writes the output row; the selection kernel never sees it.
// 1. Threshold: the cluster looks for the key t with #{x >= t} in [top_k, kCap] by a
//    radix search on the 64-bit selection key, 11 bits (2048 digits) per level from the
//    top. At each level every CTA counts the digits of its share of the keys that match
//    the prefix fixed so far, the cluster adds the counts through distributed shared
//    memory (every CTA sums all of them, so all take the same decision), and the digit
//    that reaches position top_k is fixed. The search stops at the first level where the
//    keys at or above the digit fit in kCap: the first level already, unless the score
//    bin that crosses position top_k is crowded.
// 2. Every CTA keeps its own keys >= t in shared memory and sorts them (bitonic,
//    descending: shuffles inside a warp, shared memory across warps).
// 3. Every CTA copies the cluster's sorted blocks into its shared memory. A key's
//    position in the row is its index in its own block plus, for every other block, the
//    number of keys above it there (a binary search). Keys are distinct, so the positions
//    are those of the sorted union, whichever CTA holds which key.
constexpr int kMergeCluster = 8;
constexpr int kMergeThreads = 512;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeBatch = 8;     // chunks from which a thread loads a key before using any
constexpr int kDigitBits = 11;
constexpr int kDigits = 1 << kDigitBits;
static_assert(kDigits == 4 * kMergeThreads, "each thread sums four digits");
static_assert(kDigits == kBins, "the first level's digit is the score bin");

// own sorted keys, then a copy of every CTA's (kCap keys each: all kept keys may sit in one CTA)
constexpr uint32_t kMergeSmemBytes = 2 * kCap * sizeof(unsigned long long);

struct MergeParams {
  const MergeDesc* merges;
  int32_t n_merges;
  int32_t top_k;
  const unsigned long long* store;
  const uint32_t* counts;
  uint32_t* status;
  int32_t* out_ids;     // [T, top_k]
  float* out_scores;    // [T, top_k]
  uint32_t key_id_base; // added to every written id
};

// Adds one to h[d] for every lane with v; lanes with the same digit share one atomic.
__device__ __forceinline__ void hist_add_aggregated(uint32_t* h, uint32_t d, bool v, int lane) {
  const uint32_t act = __ballot_sync(0xFFFFFFFFu, v);
  if (v) {
    const uint32_t peers = __match_any_sync(act, d);
    if (lane == __ffs(peers) - 1) atomicAdd(&h[d], static_cast<uint32_t>(__popc(peers)));
  }
}

// Sorts the first n (<= 512 * E) keys of buf in descending order, in place, with the
// whole CTA: element e = 512 r + t sits in register v[r] of thread t; partners at index
// distance j < 32 are exchanged by shuffles, 32 <= j < 512 through buf, j >= 512 inside
// the thread. Entries n .. 512 E - 1 of buf are overwritten with zero keys (below every
// key) and sort last.
template <int E>
__device__ void cta_sort_desc(unsigned long long* buf, uint32_t n) {
  constexpr uint32_t kN = kMergeThreads * E;
  const uint32_t t = threadIdx.x;
  unsigned long long v[E];
#pragma unroll
  for (int r = 0; r < E; ++r) {
    const uint32_t e = kMergeThreads * r + t;
    v[r] = e < n ? buf[e] : 0ull;
  }
  for (uint32_t k = 2; k <= kN; k <<= 1) {
    for (uint32_t j = k >> 1; j > 0; j >>= 1) {
      if (j >= static_cast<uint32_t>(kMergeThreads)) {  // partner in the same thread
#pragma unroll
        for (int rj = 1; rj < E; rj <<= 1) {  // register indices stay compile-time constants
          if (static_cast<uint32_t>(rj) * kMergeThreads != j) continue;
#pragma unroll
          for (int r = 0; r < E; ++r) {
            if (r & rj) continue;
            const uint32_t e = kMergeThreads * r + t;
            const bool desc = (e & k) == 0;
            const unsigned long long a = v[r], b = v[r | rj];
            if ((a < b) == desc) {
              v[r] = b;
              v[r | rj] = a;
            }
          }
        }
      } else {
        unsigned long long pv[E];
        if (j < 32) {
#pragma unroll
          for (int r = 0; r < E; ++r) pv[r] = __shfl_xor_sync(0xFFFFFFFFu, v[r], static_cast<int>(j));
        } else {
#pragma unroll
          for (int r = 0; r < E; ++r) buf[kMergeThreads * r + t] = v[r];
          __syncthreads();
#pragma unroll
          for (int r = 0; r < E; ++r) pv[r] = buf[kMergeThreads * r + (t ^ j)];
          __syncthreads();
        }
#pragma unroll
        for (int r = 0; r < E; ++r) {
          const uint32_t e = kMergeThreads * r + t;
          const bool keep_max = ((e & j) == 0) == ((e & k) == 0);  // lower index of a descending pair, or upper of an ascending one
          const unsigned long long a = v[r], b = pv[r];
          v[r] = keep_max ? (a > b ? a : b) : (a < b ? a : b);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < E; ++r) buf[kMergeThreads * r + t] = v[r];
  __syncthreads();
}

__global__ void __cluster_dims__(kMergeCluster, 1, 1) __launch_bounds__(kMergeThreads, 1)
    indexer_topk_merge_kernel(const MergeParams p) {
  extern __shared__ __align__(16) unsigned long long s_own[];  // kCap own keys, then kCap of the cluster's
  unsigned long long* s_all = s_own + kCap;
  __shared__ __align__(16) uint32_t hist[2][kDigits];            // per level, alternating
  __shared__ uint32_t s_cnt[kMaxMergeChunks];
  __shared__ uint32_t wsum[kMergeWarps];
  __shared__ uint32_t sel[4];
  __shared__ uint32_t s_cursor;  // own keys kept in s_own
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const MergeDesc m = p.merges[blockIdx.x / kMergeCluster];
  grid_dep_wait();  // the scan that wrote the chunks' candidates is complete
  int n_chunks = m.n_chunks;
  if (n_chunks > kMaxMergeChunks) {  // the host never builds one; keep the walk in bounds
    if (rank == 0 && tid == 0) atomicOr(p.status, kStatusInternal | (21u << 8));
    n_chunks = kMaxMergeChunks;
  }
  auto chunk_slot = [&](int ch) { return static_cast<size_t>(m.first_unit + ch) * kQB + m.j; };
  for (int ch = tid; ch < n_chunks; ch += kMergeThreads) {
    const uint32_t n = p.counts[chunk_slot(ch)];
    s_cnt[ch] = n < static_cast<uint32_t>(kCap) ? n : static_cast<uint32_t>(kCap);
  }
  if (tid == 0) s_cursor = 0u;
  __syncthreads();

  // Visits this CTA's share of the union (chunk ch belongs to CTA ch % kMergeCluster),
  // loading one key from each of up to kMergeBatch chunks before using any of them.
  // f(x, v) is called by every thread of the CTA the same number of times.
  auto for_union = [&](auto&& f) {
    for (int c0 = static_cast<int>(rank); c0 < n_chunks; c0 += kMergeBatch * kMergeCluster) {
      uint32_t cmax = 0;
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const int ch = c0 + u * kMergeCluster;
        if (ch < n_chunks) cmax = max(cmax, s_cnt[ch]);
      }
      for (uint32_t base = 0; base < cmax; base += kMergeThreads) {
        const uint32_t off = base + static_cast<uint32_t>(tid);
        unsigned long long x[kMergeBatch];
        bool v[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          const int ch = c0 + u * kMergeCluster;
          v[u] = ch < n_chunks && off < s_cnt[ch];
          x[u] = v[u] ? __ldcg(p.store + chunk_slot(ch) * kCap + off) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) f(x[u], v[u]);
      }
    }
  };

  const uint32_t K = static_cast<uint32_t>(p.top_k);
  uint32_t k_rem = K;             // positions still to fill from the keys that match prefix
  uint32_t above = 0;             // keys above the prefix's range (all kept)
  unsigned long long prefix = 0;  // bits [hi, 64) fixed so far
  unsigned long long thr = 0;
  uint32_t kept = 0;
  int hi = 64;
  for (int level = 0;; ++level) {
    const int shift = hi > kDigitBits ? hi - kDigitBits : 0;
    uint32_t* h = hist[level & 1];
    for (int i = tid; i < kDigits; i += kMergeThreads) h[i] = 0u;
    __syncthreads();
    for_union([&](unsigned long long x, bool v) {
      const bool match = v && (hi >= 64 || (x >> hi) == (prefix >> hi));
      hist_add_aggregated(h, static_cast<uint32_t>(x >> shift) & (kDigits - 1), match, lane);
    });
    cluster_sync_all();  // every CTA's counts for this level are complete
    // Cluster-wide counts of the digits 2047-4t .. 2044-4t (thread t, descending).
    uint32_t c4[4];
    {
      const uint32_t addr = smem_u32(h + (kDigits - 4 - 4 * tid));
      uint4 acc = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int r = 0; r < kMergeCluster; ++r) {
        const uint4 t = ld_dsmem_v4(mapa_shared(addr, static_cast<uint32_t>(r)));
        acc.x += t.x;
        acc.y += t.y;
        acc.z += t.z;
        acc.w += t.w;
      }
      c4[0] = acc.w;
      c4[1] = acc.z;
      c4[2] = acc.y;
      c4[3] = acc.x;
    }
    const uint32_t s = c4[0] + c4[1] + c4[2] + c4[3];
    uint32_t incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    uint32_t run = incl - s;  // matching keys in digits above this thread's four
    uint32_t total = 0;
    for (int wv = 0; wv < kMergeWarps; ++wv) {
      if (wv < warp) run += wsum[wv];
      total += wsum[wv];
    }
    if (tid == 0) {  // fewer matching keys than positions left (first level only): keep all
      sel[0] = 0u;
      sel[1] = total;
      sel[2] = total;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t a = run;  // matching keys in digits above d
      run += c4[i];
      if (a < k_rem && run >= k_rem) {  // the digit that reaches position k_rem (at most one)
        sel[0] = static_cast<uint32_t>(kDigits - 1 - (4 * tid + i));
        sel[1] = run;
        sel[2] = a;
      }
    }
    __syncthreads();
    const uint32_t dstar = sel[0], ge_d = sel[1], ge_above = sel[2];
    if (above + ge_d <= static_cast<uint32_t>(kCap) || shift == 0) {
      thr = prefix | (static_cast<unsigned long long>(dstar) << shift);
      kept = above + ge_d;
      break;
    }
    above += ge_above;
    k_rem -= ge_above;
    prefix |= static_cast<unsigned long long>(dstar) << shift;
    hi = shift;
  }

  if (kept > static_cast<uint32_t>(kCap)) {  // cannot happen: keys are distinct
    if (rank == 0 && tid == 0) atomicOr(p.status, kStatusInternal | (22u << 8));
    kept = kCap;
  }
  // keep this CTA's keys at or above the threshold key
  for_union([&](unsigned long long x, bool v) {
    const bool keep = v && x >= thr;
    const uint32_t slot = warp_append_slot(keep, &s_cursor, lane);
    if (keep && slot < static_cast<uint32_t>(kCap)) s_own[slot] = x;
  });
  __syncthreads();
  const uint32_t n_own = min(s_cursor, static_cast<uint32_t>(kCap));
  if (n_own <= kMergeThreads) cta_sort_desc<1>(s_own, n_own);
  else if (n_own <= 2 * kMergeThreads) cta_sort_desc<2>(s_own, n_own);
  else if (n_own <= 4 * kMergeThreads) cta_sort_desc<4>(s_own, n_own);
  else cta_sort_desc<8>(s_own, n_own);
  cluster_sync_all();  // every CTA's block is sorted and its count final

  // copy the cluster's blocks (block r at offset off[r]) into s_all
  uint32_t off[kMergeCluster + 1];
  off[0] = 0;
  const uint32_t cur_addr = smem_u32(&s_cursor);
#pragma unroll
  for (int r = 0; r < kMergeCluster; ++r) {
    const uint32_t c = ld_dsmem_u32(mapa_shared(cur_addr, static_cast<uint32_t>(r)));
    off[r + 1] = min(off[r] + min(c, static_cast<uint32_t>(kCap)), static_cast<uint32_t>(kCap));
  }
  const uint32_t own_addr = smem_u32(s_own);
#pragma unroll
  for (int r = 0; r < kMergeCluster; ++r) {
    const uint32_t base = mapa_shared(own_addr, static_cast<uint32_t>(r));
    for (uint32_t i = off[r] + tid; i < off[r + 1]; i += kMergeThreads)
      s_all[i] = ld_dsmem_u64(base + (i - off[r]) * 8u);
  }
  cluster_sync_all();  // no CTA reads another's shared memory after this
  // positions of this CTA's keys in the merged row
  const uint32_t keff = kept < K ? kept : K;
  int32_t* out_ids = p.out_ids + static_cast<size_t>(m.row) * K;
  float* out_scores = p.out_scores + static_cast<size_t>(m.row) * K;
  for (uint32_t e = tid; e < n_own; e += kMergeThreads) {
    const unsigned long long x = s_own[e];
    uint32_t pos = e;
#pragma unroll
    for (int r = 0; r < kMergeCluster; ++r) {
      if (r == static_cast<int>(rank)) continue;
      uint32_t lo = off[r], hi2 = off[r + 1];  // block r: s_all[lo, hi2), descending
      const uint32_t first = lo;
      while (lo < hi2) {
        const uint32_t mid = (lo + hi2) >> 1;
        if (s_all[mid] > x) lo = mid + 1;
        else hi2 = mid;
      }
      pos += lo - first;
    }
    if (pos < keff) {
      st_stream_s32(out_ids + pos, static_cast<int32_t>(static_cast<uint32_t>(x & 0xFFFFFFFFull) + p.key_id_base));
      st_stream_f32(out_scores + pos, key_to_float(static_cast<uint32_t>(x >> 32)));
    }
  }
  if (rank == 0) {
    for (uint32_t r = keff + tid; r < K; r += kMergeThreads) {  // fewer visible keys than top_k
      st_stream_s32(out_ids + r, -1);
      st_stream_f32(out_scores + r, -__int_as_float(0x7F800000));
    }
  }
}

}  // namespace itk

