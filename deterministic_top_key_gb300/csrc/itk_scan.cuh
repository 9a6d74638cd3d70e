// The scan kernel: persistent CTAs draw work units from a self-resetting ticket word;
// each unit (up to 4 consecutive queries of one segment) streams its visible key tiles
// through a tcgen05 GEMM with the keys as the M side, a fused ReLU * w head reduction and
// a streaming candidate filter. At the end of a unit each query's candidates (a superset
// of its top-k, at most kCap keys) go to the query's slot of the candidate store, where
// the selection kernel picks and sorts the top-k.
//
// Operation: flashinfer PR #8691 ("perf(cake_dsa_indexer_det): ticket scheduling on
// sm_107a, no fill kernel in eager entry"), opening description -- BF16 q/k, FP32 w and
// scores, top-k key ids per query, ties to the larger id, ids and scores independent of
// partition or chunking -- with the lightning-indexer score
//     I[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . k[s,:]).
// Work distribution: same page, commit note on drawing work units from the ticket word
// (each running CTA takes the next unit, so a CTA that cannot start does not hold back a
// second wave) and the TicketWord note (every completed scan leaves the word at zero).
//
// CTA layout (576 threads, one CTA per SM):
//   warp 0        ticket draws, TMA loads of the Q block and of the K tile ring
//   warp 1        TMEM allocation, tcgen05.mma issue (one thread)
//   warps 2..17   epilogue: four groups of four warps; group g owns query g of the unit;
//                 the four warps of a group cover the 128 TMEM lanes (keys), so every
//                 SM sub-partition runs four epilogue warps. Per key tile: scores,
//                 candidate filter, appends to the query's working buffer, histogram of
//                 the appended score keys; at the end of the unit, the hand-off to the
//                 candidate store.
//
// Score arithmetic (fixed, so a score depends only on q[t], k[s] and w[t], never on
// tiling, unit or CTA): the tensor core forms the FP32 dot products x_h = q[t,h,:].k[s,:]
// over D = 128 in eight K = 16 steps in a fixed order; the epilogue forms eight partial
// sums p_m (m = 0..7), p_m = fma(w[t,h], max(x_h, 0), p_m) over h = m, m+8, ..., m+56 in
// that order, and returns
//     ((p0 + p1) + (p2 + p3)) + ((p4 + p5) + (p6 + p7)) + 0
// (the "+ 0" turns a -0 into +0). The four threads of a quad share four keys: thread c
// (c = 0..3) holds the head columns of chains 2c and 2c + 1 of all four (one 16x256b
// tensor-memory load per half of the warp's 32 keys) and keeps the head weights of those
// chains in registers; it forms P_c = p_2c + p_2c+1 for each key, and two shuffle rounds
// over the quad add (P0 + P1) + (P2 + P3), leaving key c's score with thread c. Each FMA
// is evaluated as fma(w/2, x + |x|, p) (relu_fma below): the same exact product, so the
// same bits, with the ReLU as one add on the FMA pipe.
//
// Candidate filter: a query's working buffer holds keys whose score key lies in a bin
// (top 11 bits of the order-preserving score key) at or above a threshold bin; the
// threshold bin is the highest bin whose bins-at-or-above hold at least top_k appended
// keys. It only rises, and every key it rejects is below top_k keys already seen, so the
// buffer always contains the exact top-k of the keys seen so far. The filter compares
// the score itself with the lowest score of the threshold bin, and forms the 64-bit key
// only for the keys it appends. A unit whose queries see at most kCap keys of its tile
// range skips the filter: every visible key goes straight to the store slot (no
// histogram, no sync points, no hand-off copy). A unit whose queries see at most kQCap
// keys has no sync points: every visible key goes to the working buffer and the
// threshold is applied once, at the hand-off. In both, key j of the unit's tile range
// has slot j (no slot reservation). A longer unit does the same over its first kQCap
// keys, then raises the threshold, compacts, and filters from there on with sync
// points. The tile loop is compiled for the three kinds.
// Scores are taken to be finite (inputs whose dot products overflow FP32 are out of scope).
#pragma once

#include <type_traits>

#include "itk_common.cuh"

namespace itk {

constexpr int kN = kQB * kHeads;             // MMA N = 256 (query, head) columns
constexpr int kStages = 2;                   // K tile ring depth (a third stage measured no faster)
constexpr int kQCap = 16384;                 // working buffer entries per query while a unit runs
constexpr int kDenseTiles = kQCap / 128;     // tiles a filtered unit appends densely before its first sync
constexpr int kSyncEvery = 32;               // epilogue group synchronizes every this many tiles
constexpr uint32_t kCompactAt = kQCap - kSyncEvery * kBlockKeys;  // buffer fill that triggers a compaction
constexpr int kEpiGroups = kQB;              // one 4-warp epilogue group per query of the unit
constexpr int kEpiWarps = 4 * kEpiGroups;
constexpr int kNumWarps = 2 + kEpiWarps;
constexpr int kNumThreads = kNumWarps * 32;
constexpr int kFirstEpiWarp = 2;
constexpr uint32_t kTmemCols = 512;          // two accumulator buffers of 256 columns

constexpr uint32_t kQHalfBytes = kN * 64 * 2;           // 256 rows x 128 B = 32 KB
constexpr uint32_t kQBytes = 2 * kQHalfBytes;            // 64 KB
constexpr uint32_t kKHalfBytes = kBlockKeys * 64 * 2;    // 128 rows x 128 B = 16 KB
constexpr uint32_t kKStageBytes = 2 * kKHalfBytes;       // 32 KB

// Shared memory layout (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffHist = kOffK + kStages * kKStageBytes;          // 4 queries x 2048 u32 bins
constexpr uint32_t kOffW = kOffHist + kQB * kBins * 4;                 // 4 queries x 64 floats
constexpr uint32_t kOffRadix = kOffW + kQB * kHeads * 4;               // 4 groups x 256 x u32
constexpr uint32_t kOffQState = kOffRadix + kEpiGroups * 256 * 4;      // 4 queries x 4 x u32
constexpr uint32_t kOffSel = kOffQState + kQB * 16;                    // 4 groups x 8 x u32
constexpr uint32_t kOffUnit = kOffSel + kEpiGroups * 8 * 4;            // 2 slots x (int4 unit, int unit index)
constexpr uint32_t kOffBar = kOffUnit + 2 * 32;                        // mbarriers
constexpr uint32_t kNumBars = 2 * kStages + 2 + 2 + 2 + 2 + 2 + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;                  // tmem base, abort, flags
constexpr uint32_t kSmemUsed = kOffMisc + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;                      // slack for 1024-byte alignment

static_assert(kOffK % 1024 == 0 && kKStageBytes % 1024 == 0 && kQHalfBytes % 1024 == 0,
              "SW128 tiles need 1 KB alignment");
static_assert(kOffBar % 8 == 0 && kOffW % 16 == 0 && kOffUnit % 16 == 0, "alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kMaxTopK <= static_cast<int>(kCompactAt), "a compaction to top_k must leave room for the next tiles");

struct ScanParams {
  const UnitDesc* units;
  int32_t n_units;
  int32_t top_k;
  TicketBlock* ticket;
  uint32_t* status;              // device status word (0 = ok)
  const float* w;                // [T,64]
  unsigned long long* cand;      // per CTA: 4 x kQCap working keys, then 4 x kMaxTopK exact-select scratch
  unsigned long long* store;     // [n_units * 4][kCap] candidate keys handed to the selection kernel
  uint32_t* counts;              // [n_slots] keys in each store slot
  int32_t static_schedule;       // benchmark aid: 1 = CTA b takes units b, b + grid, ... (no ticket)
  int32_t withhold_first_tile;   // test hook: 1 = CTA 0 never loads the first key tile of its first unit
  long long wait_limit;          // SM clocks after which an in-kernel wait gives up (kWaitLimitCycles)
};

constexpr size_t kCandKeysPerCta = static_cast<size_t>(kQB) * kQCap + kEpiGroups * kMaxTopK;
__host__ __device__ constexpr size_t candidate_bytes_per_cta() { return kCandKeysPerCta * sizeof(unsigned long long); }
// Candidate store bytes per work unit (four query slots of kCap keys, then the counts live apart).
__host__ __device__ constexpr size_t store_bytes_per_unit() {
  return static_cast<size_t>(kQB) * kCap * sizeof(unsigned long long);
}

struct Bars {
  uint32_t kfull, kempty, qfull, qempty, accfull, accempty, unitfull, unitempty, mmadone;
  __device__ uint32_t kf(int s) const { return kfull + 8u * s; }
  __device__ uint32_t ke(int s) const { return kempty + 8u * s; }
  __device__ uint32_t af(int b) const { return accfull + 8u * b; }
  __device__ uint32_t ae(int b) const { return accempty + 8u * b; }
  __device__ uint32_t uf(int s) const { return unitfull + 8u * s; }
  __device__ uint32_t ue(int s) const { return unitempty + 8u * s; }
};


// Two FP32 fused multiply-adds in one instruction: (d0, d1) = (a0*b0 + d0, a1*b1 + d1),
// each rounded once, exactly as two fmaf calls.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b, c;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %5};\n\t"
      "mov.b64 c, {%0, %1};\n\t"
      "fma.rn.f32x2 c, a, b, c;\n\t"
      "mov.b64 {%0, %1}, c;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// One step of two head chains, (p0, p1) = (fma(w0, max(x0, 0), p0), fma(w1, max(x1, 0), p1)),
// given the halved weights hw = w / 2: x + |x| is 2 max(x, 0) exactly for every finite x
// (2x or +0), so hw (x + |x|) is the exact product w max(x, 0) whenever w / 2 is exact
// (w = 0 or |w| >= 2^-125), and each fused multiply-add rounds the same exact value as the
// plain form. The ReLU becomes one FP32 add with an absolute-value operand, on the FMA
// pipe (a max runs on the ALU pipe at half rate).
__device__ __forceinline__ void relu_fma2(float& p0, float& p1, float hw0, float hw1, float x0, float x1) {
  ffma2(p0, p1, hw0, hw1, x0 + fabsf(x0), x1 + fabsf(x1));
}

// Per-query histogram of appended score keys: one 32-bit counter per bin.
__device__ __forceinline__ uint32_t hist_get(const uint32_t* h, uint32_t b) { return h[b]; }
__device__ __forceinline__ void hist_inc(uint32_t* h, uint32_t b) { atomicAdd(&h[b], 1u); }

// Radix select streamed from global memory, one byte per pass: returns `prefix` with
// #{x in buf[0..n) : x >= prefix} == K (K <= n, keys distinct). Used when the score bin at
// the threshold is crowded (more than kCap keys at or above it at a hand-off, or a
// compaction that cannot drop enough).
__device__ __noinline__ unsigned long long group_select_stream(const GroupCtx& c, const unsigned long long* buf,
                                                               uint32_t n, uint32_t K) {
  constexpr int kChunk = 8;  // keys a thread loads before counting them
  unsigned long long prefix = 0ull;
  uint32_t k_rem = K;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = c.gtid; i < 256; i += 128) c.radix[i] = 0u;
    gsync(c);
    const unsigned long long hi_mask = (shift == 56) ? 0ull : (~0ull << (shift + 8));
    for (uint32_t base = 0; base < n; base += 128 * kChunk) {
      unsigned long long x[kChunk];
#pragma unroll
      for (int r = 0; r < kChunk; ++r) {
        const uint32_t idx = base + c.gtid + 128u * r;
        x[r] = idx < n ? buf[idx] : 0ull;
      }
#pragma unroll
      for (int r = 0; r < kChunk; ++r) {
        const uint32_t idx = base + c.gtid + 128u * r;
        if (idx < n && (x[r] & hi_mask) == (prefix & hi_mask)) atomicAdd(&c.radix[(x[r] >> shift) & 0xFFu], 1u);
      }
    }
    gsync(c);
    group_pick_digit(c, k_rem);
    gsync(c);
    prefix |= static_cast<unsigned long long>(c.sel[0]) << shift;
    k_rem = c.sel[1];
    const uint32_t bucket = c.sel[2];
    gsync(c);
    if (bucket == k_rem) break;  // uniform across the group
  }
  return prefix;
}

// Copies the keys x of buf[0..n) with keep(x) to dst[0..limit) (dst may be buf itself:
// every key of a chunk is read before any slot of it is rewritten, and no more keys are
// kept than read); returns the number that qualified. A thread loads kChunk keys, then
// writes its kept ones to consecutive slots; a warp reserves its slots with one atomic.
template <typename Keep>
__device__ __forceinline__ uint32_t group_copy_if(const GroupCtx& c, const unsigned long long* buf, uint32_t n,
                                                  Keep keep, unsigned long long* dst, uint32_t limit, uint32_t* s_pos,
                                                  uint64_t pol_src, uint64_t pol_dst) {
  constexpr int kChunk = 16;  // keys per thread per pass
  if (c.gtid == 0) *s_pos = 0u;
  gsync(c);
  for (uint32_t base = 0; base < n; base += 128 * kChunk) {
    unsigned long long x[kChunk];
#pragma unroll
    for (int r = 0; r < kChunk; ++r) {
      const uint32_t idx = base + c.gtid + 128u * r;
      x[r] = idx < n ? ld_hint_u64(buf + idx, pol_src) : 0ull;
    }
    gsync(c);
    uint32_t km = 0;
#pragma unroll
    for (int r = 0; r < kChunk; ++r) {
      const uint32_t idx = base + c.gtid + 128u * r;
      km |= (idx < n && keep(x[r]) ? 1u : 0u) << r;
    }
    const uint32_t cnt = static_cast<uint32_t>(__popc(km));
    uint32_t incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (c.lane >= off) incl += t;
    }
    uint32_t wbase = 0;
    if (c.lane == 31 && incl) wbase = atomicAdd(s_pos, incl);
    wbase = __shfl_sync(0xFFFFFFFFu, wbase, 31);
    uint32_t pos = wbase + incl - cnt;
#pragma unroll
    for (int r = 0; r < kChunk; ++r) {
      if ((km >> r) & 1u) {
        if (pos < limit) st_hint_u64(dst + pos, x[r], pol_dst);
        ++pos;
      }
    }
  }
  gsync(c);
  const uint32_t m = *s_pos;
  gsync(c);
  return m;
}

// Appends the keys of buf[0..n) at or above `prefix` to dst[0..limit); returns the number
// appended.
__device__ __forceinline__ uint32_t group_keep_at_or_above(const GroupCtx& c, const unsigned long long* buf,
                                                           uint32_t n, unsigned long long prefix,
                                                           unsigned long long* dst, uint32_t limit,
                                                           uint32_t* s_cursor) {
  const uint64_t pol = policy_evict_last();
  const uint32_t m = group_copy_if(c, buf, n, [prefix](unsigned long long x) { return x >= prefix; }, dst, limit,
                                   s_cursor, pol, pol);
  return m < limit ? m : limit;  // exactly `limit` keys qualify: keys are distinct
}

// Keeps exactly the K largest of the n keys in buf (n > K): they go through `scratch`
// back to buf[0..K), and the histogram is rebuilt from them. Returns their lowest bin.
__device__ uint32_t group_exact_in_place(const GroupCtx& c, unsigned long long* buf, uint32_t n, uint32_t* hist,
                                         uint32_t K, uint32_t* s_cursor, unsigned long long* scratch) {
  const unsigned long long prefix = group_select_stream(c, buf, n, K);
  for (int i = c.gtid; i < kBins; i += 128) hist[i] = 0u;
  group_keep_at_or_above(c, buf, n, prefix, scratch, K, s_cursor);
  for (uint32_t i = c.gtid; i < K; i += 128) {
    const unsigned long long x = scratch[i];
    buf[i] = x;
    hist_inc(hist, bin_of(x));
  }
  gsync(c);
  return bin_of(prefix);
}

// Drops the keys of buf[0..n) whose bin is below thr, writing the survivors to dst[0..limit)
// (dst may be buf itself); returns the number that qualified (callers make sure it is <= limit).
__device__ __forceinline__ uint32_t group_drop_below(const GroupCtx& c, unsigned long long* buf, uint32_t n,
                                                     uint32_t thr, unsigned long long* dst, uint32_t limit,
                                                     uint32_t* s_pos, uint64_t pol_src, uint64_t pol_dst) {
  return group_copy_if(c, buf, n, [thr](unsigned long long x) { return bin_of(x) >= thr; }, dst, limit, s_pos,
                       pol_src, pol_dst);
}

// Mid-unit compaction of one working buffer, so that at most `limit` keys remain: drops
// the keys below the threshold bin; if more than `limit` remain (ties crowd the threshold
// bin), keeps exactly the K largest. Updates the query state qs: [0] count, [1] count at
// the last raise, [2] threshold bin, [3] keys at or above the threshold bin.
__device__ __forceinline__ void epi_compact(const GroupCtx& c, unsigned long long* buf, uint32_t* qs, uint32_t* hist,
                                            uint32_t K, uint32_t* s_pos, uint64_t pol, uint32_t limit,
                                            unsigned long long* scratch) {
  uint32_t m = group_drop_below(c, buf, qs[0], qs[2], buf, kQCap, s_pos, pol, pol);
  if (m > limit) {
    const uint32_t t = group_exact_in_place(c, buf, m, hist, K, s_pos, scratch);
    m = K;
    if (c.gtid == 0) qs[2] = t;
  }
  if (c.gtid == 0) {
    qs[0] = m;
    qs[1] = m;
    qs[3] = m;  // every kept key lies at or above the threshold bin
  }
  gsync(c);
}

// End of a unit for one query: its candidates (every key of the working buffer in a bin
// at or above the threshold, or exactly the K largest when more than kCap of those
// remain) go to its store slot, and their number to *count.
__device__ __forceinline__ void epi_handoff(const GroupCtx& c, unsigned long long* buf, const uint32_t* qs, uint32_t K,
                                            uint32_t* s_pos, uint64_t pol_src, uint64_t pol_dst, unsigned long long* dst,
                                            uint32_t* count, uint32_t* status) {
  const uint32_t n = qs[0];
  uint32_t m;
  if (qs[3] > static_cast<uint32_t>(kCap)) {  // uniform; qs[3] counts the keys at or above the threshold bin
    const unsigned long long prefix = group_select_stream(c, buf, n, K);
    m = group_keep_at_or_above(c, buf, n, prefix, dst, K, s_pos);
  } else {
    m = group_drop_below(c, buf, n, qs[2], dst, kCap, s_pos, pol_src, pol_dst);
  }
  if (c.gtid == 0) {
    if (m > static_cast<uint32_t>(kCap)) {  // cannot happen: qs[3] is the exact number kept
      atomicOr(status, kStatusInternal | (21u << 8));
      m = kCap;
    }
    *count = m;
  }
}

// Raise a query's threshold bin as far as its histogram allows, by one warp: afterwards
// thr is the highest bin with at least K appended keys at or above it (it stays put while
// fewer than K keys have been appended). qs: [0] count, [1] count at the last raise,
// [2] threshold bin, [3] appended keys at or above the threshold bin.
__device__ __forceinline__ void warp_raise_threshold(uint32_t* qs, const uint32_t* hist, uint32_t K, int lane) {
  const uint32_t n = qs[0];
  uint32_t ge = qs[3] + (n - qs[1]);
  uint32_t thr = qs[2];
  if (ge >= K) {
    // fast skip over empty runs of 32 bins (one counter per lane, conflict-free)
    while (thr + 32 < static_cast<uint32_t>(kBins)) {
      const uint32_t word = hist[thr + static_cast<uint32_t>(lane)];
      if (__any_sync(0xFFFFFFFFu, word != 0u)) break;
      thr += 32;
    }
    while (true) {
      const uint32_t b = thr + static_cast<uint32_t>(lane);
      const uint32_t h = b < static_cast<uint32_t>(kBins) ? hist_get(hist, b) : 0u;
      uint32_t incl = h;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += t;
      }
      // moving the threshold past bins thr..b keeps ge - incl keys at or above it
      const bool ok = b + 1 < static_cast<uint32_t>(kBins) && incl + K <= ge;
      const uint32_t adv = static_cast<uint32_t>(__popc(__ballot_sync(0xFFFFFFFFu, ok)));
      if (adv == 0) break;
      ge -= __shfl_sync(0xFFFFFFFFu, incl, adv - 1);
      thr += adv;
      if (adv < 32) break;
    }
  }
  __syncwarp();
  if (lane == 0) {
    qs[1] = n;
    qs[2] = thr;
    qs[3] = ge;
  }
}

// Raise a query's threshold bin as far as its histogram allows, by the whole group:
// afterwards thr is the highest bin with at least K keys at or above it (it stays put while
// fewer than K keys lie at or above it). qs: [0] count, [1] count at the last raise,
// [2] threshold bin, [3] keys at or above the threshold bin. The histogram counts exactly
// the buffer's keys in every bin at or above the current threshold: appends reach only
// those bins, a compaction drops keys below it, and the exact path rebuilds the histogram.
// Thread t holds bins [16 t, 16 t + 16) (bins below the threshold read as empty); a
// reversed warp scan of the run sums and the four warp totals give the keys above each
// run, and the one thread whose run crosses K walks its own bins. Called by every thread
// of the group; the caller synchronizes the group before reading qs. It serves the first
// raise of a unit, a walk from bin 0 across about a thousand bins; the later raises move
// the threshold by a few bins and stay with warp_raise_threshold (one warp, faster there).
__device__ __forceinline__ void group_raise_threshold(const GroupCtx& c, uint32_t* qs, const uint32_t* hist,
                                                      uint32_t K) {
  const uint32_t n = qs[0];
  const uint32_t thr0 = qs[2];
  const uint32_t ge0 = qs[3] + (n - qs[1]);  // keys at or above bin thr0
  if (ge0 < K) {  // uniform: the threshold stays
    gsync(c);     // every thread has read qs
    if (c.gtid == 0) {
      qs[1] = n;
      qs[3] = ge0;
    }
    return;
  }
  const uint32_t b0 = 16u * static_cast<uint32_t>(c.gtid);
  uint32_t h[16];
  const uint4* run16 = reinterpret_cast<const uint4*>(hist + b0);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 x = run16[v];
    h[4 * v + 0] = x.x;
    h[4 * v + 1] = x.y;
    h[4 * v + 2] = x.z;
    h[4 * v + 3] = x.w;
  }
  uint32_t sum = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (b0 + static_cast<uint32_t>(i) < thr0) h[i] = 0u;
    sum += h[i];
  }
  uint32_t incl = sum;  // keys in this thread's run and the higher runs of its warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, incl, off);
    if (c.lane + off < 32) incl += t;
  }
  if (c.lane == 0) c.radix[c.gwarp] = incl;  // the warp's total
  gsync(c);                                  // (every thread has also read qs)
  uint32_t above = incl - sum;               // keys in bins >= b0 + 16
#pragma unroll
  for (int w = 1; w < 4; ++w) above += w > c.gwarp ? c.radix[w] : 0u;
  if (above < K && above + sum >= K) {  // exactly one thread: its run holds the new threshold
    uint32_t run = above, thr = thr0, ge = ge0;
    bool found = false;
#pragma unroll
    for (int i = 15; i >= 0; --i) {
      run += h[i];
      if (!found && run >= K) {
        found = true;
        thr = b0 + static_cast<uint32_t>(i);
        ge = run;
      }
    }
    qs[1] = n;
    qs[2] = thr;
    qs[3] = ge;
  }
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kNumThreads, 1)
    indexer_topk_scan_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                             const ScanParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // per-query epilogue state: [j][0] count, [1] count at the last threshold raise,
  // [2] threshold bin, [3] keys appended at or above the threshold bin
  uint32_t* s_qs = reinterpret_cast<uint32_t*>(smem + kOffQState);
  int4* s_unit = reinterpret_cast<int4*>(smem + kOffUnit);            // [slot * 2]: unit; [slot * 2 + 1].x: index
  float* s_w = reinterpret_cast<float*>(smem + kOffW);
  uint32_t* s_misc = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  uint32_t* s_tmem = s_misc + 0;
  volatile uint32_t* s_abort = s_misc + 1;
  uint32_t* s_gfail = s_misc + 2;  // [4] per-group failure flags
  uint32_t* s_pos = s_misc + 6;    // [4] epilogue-group cursors

  const uint32_t bar0 = smem_u32(smem + kOffBar);
  Bars bars;
  bars.kfull = bar0;
  bars.kempty = bars.kfull + 8 * kStages;
  bars.qfull = bars.kempty + 8 * kStages;
  bars.qempty = bars.qfull + 8;
  bars.accfull = bars.qempty + 8;
  bars.accempty = bars.accfull + 16;
  bars.unitfull = bars.accempty + 16;
  bars.unitempty = bars.unitfull + 16;
  bars.mmadone = bars.unitempty + 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bars.kf(s), 1);
      mbar_init(bars.ke(s), 1);
    }
    mbar_init(bars.qfull, 1);
    mbar_init(bars.qempty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.af(b), 1);
      mbar_init(bars.ae(b), kEpiWarps);
      mbar_init(bars.uf(b), 1);
      mbar_init(bars.ue(b), 1 + kEpiWarps);
    }
    mbar_init(bars.mmadone, 1);
    for (int i = 1; i < 16; ++i) s_misc[i] = 0u;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&q_map);
    tma_prefetch_desc(&k_map);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *s_tmem;
  grid_dep_wait();  // the kernel that wrote q, k and w (if launched as its dependent) is complete

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_k = policy_evict_last();
      const uint64_t pol_q = policy_evict_first();
      uint32_t it = 0, kc = 0, qloads = 0;
      bool ok = true;
      while (ok) {
        const unsigned long long u = p.static_schedule
                                         ? static_cast<unsigned long long>(blockIdx.x) + it * gridDim.x
                                         : atomicAdd(&p.ticket->next, 1ull);
        const int slot = it & 1;
        if (!mbar_wait(bars.ue(slot), ((it >> 1) & 1) ^ 1, s_abort, p.wait_limit)) {
          record_timeout(p.status, s_abort, 1);
          break;
        }
        int4 unit, range;
        if (u < static_cast<unsigned long long>(p.n_units)) {
          const UnitDesc d = p.units[u];
          unit = make_int4(d.q_row0, d.nq, d.key_row0, d.pos0);
          range = make_int4(static_cast<int>(u), d.tile0, d.tile1, 0);
        } else {
          unit = make_int4(-1, 0, 0, 0);
          range = make_int4(0, 0, 0, 0);
        }
        s_unit[2 * slot] = unit;
        s_unit[2 * slot + 1] = range;  // unit index, key tiles [tile0, tile1)
        mbar_arrive(bars.uf(slot));
        if (unit.x < 0) {
          grid_dep_launch_dependents();  // no unit left for this CTA: the next kernel may launch
          break;
        }
        if (!mbar_wait(bars.qempty, (it & 1) ^ 1, s_abort, p.wait_limit)) {
          record_timeout(p.status, s_abort, 2);
          break;
        }
        mbar_arrive_expect_tx(bars.qfull, kQBytes);
        const uint32_t qdst = smem_u32(smem + kOffQ);
        tma_load_2d(qdst, &q_map, bars.qfull, 0, unit.x * kHeads, pol_q);
        tma_load_2d(qdst + kQHalfBytes, &q_map, bars.qfull, 64, unit.x * kHeads, pol_q);
        ++qloads;
        for (int tile = range.y; tile < range.z; ++tile, ++kc) {
          const int s = kc % kStages;
          if (!mbar_wait(bars.ke(s), ((kc / kStages) & 1) ^ 1, s_abort, p.wait_limit)) {
            record_timeout(p.status, s_abort, 3);
            ok = false;
            break;
          }
          // test hook: the tile's barrier phase never completes, as if its load never arrived
          if (p.withhold_first_tile && blockIdx.x == 0 && it == 0 && tile == range.y) continue;
          mbar_arrive_expect_tx(bars.kf(s), kKStageBytes);
          const uint32_t kdst = smem_u32(smem + kOffK + s * kKStageBytes);
          const int row = unit.z + tile * kBlockKeys;
          tma_load_2d(kdst, &k_map, bars.kf(s), 0, row, pol_k);
          tma_load_2d(kdst + kKHalfBytes, &k_map, bars.kf(s), 64, row, pol_k);
        }
        ++it;
      }
      // Drain: no TMA write into this CTA's shared memory may still be in flight (these
      // waits ignore the abort flag but keep their time limit).
      for (uint32_t j = (kc > kStages ? kc - kStages : 0); j < kc; ++j)
        mbar_wait(bars.kf(j % kStages), (j / kStages) & 1, nullptr, p.wait_limit);
      if (qloads > 0) mbar_wait(bars.qfull, (qloads - 1) & 1, nullptr, p.wait_limit);
      ticket_release(p.ticket);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBlockKeys, kN);
      const uint32_t qbase = smem_u32(smem + kOffQ);
      uint32_t it = 0, kc = 0, ac = 0;
      bool ok = true;
      while (ok) {
        const int slot = it & 1;
        if (!mbar_wait(bars.uf(slot), (it >> 1) & 1, s_abort, p.wait_limit)) {
          record_timeout(p.status, s_abort, 4);
          break;
        }
        const int4 unit = s_unit[2 * slot];
        if (unit.x < 0) break;
        if (!mbar_wait(bars.qfull, it & 1, s_abort, p.wait_limit)) {
          record_timeout(p.status, s_abort, 5);
          break;
        }
        const int nt = s_unit[2 * slot + 1].z - s_unit[2 * slot + 1].y;
        for (int tile = 0; tile < nt; ++tile, ++kc, ++ac) {
          const int ab = ac & 1;
          if (!mbar_wait(bars.ae(ab), ((ac >> 1) & 1) ^ 1, s_abort, p.wait_limit)) {
            record_timeout(p.status, s_abort, 6);
            ok = false;
            break;
          }
          const int s = kc % kStages;
          if (!mbar_wait(bars.kf(s), (kc / kStages) & 1, s_abort, p.wait_limit)) {
            record_timeout(p.status, s_abort, 7);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t kbase = smem_u32(smem + kOffK + s * kKStageBytes);
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(ab * kN);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t half = kk >> 2;
            const uint32_t koff = (kk & 3) * 32u;
            const uint64_t a_desc = sw128_kmajor_desc(kbase + half * kKHalfBytes + koff);
            const uint64_t b_desc = sw128_kmajor_desc(qbase + half * kQHalfBytes + koff);
            mma_bf16(d_tmem, a_desc, b_desc, idesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(bars.ke(s));
          mma_commit(bars.af(ab));
        }
        if (!ok) break;
        mma_commit(bars.qempty);
        mbar_arrive(bars.ue(slot));
        ++it;
      }
      // Every MMA this thread issued completes before TMEM is released (ignores the
      // abort flag, keeps the time limit).
      mma_commit(bars.mmadone);
      mbar_wait(bars.mmadone, 0, nullptr, p.wait_limit);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - kFirstEpiWarp;
    const int g = ew >> 2;  // the query of the unit this group owns
    GroupCtx c;
    c.gwarp = ew & 3;
    c.lane = lane;
    c.gtid = c.gwarp * 32 + lane;
    c.bar = 1 + g;
    c.radix = reinterpret_cast<uint32_t*>(smem + kOffRadix) + 256 * g;
    c.sel = reinterpret_cast<uint32_t*>(smem + kOffSel) + 8 * g;
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    // quad layout: thread (qd, qc) = (lane / 4, lane % 4) reads the head columns 8j + 2 qc
    // and 8j + 2 qc + 1 (j = 0..7) of the key rows qd and qd + 8 of each half (16 rows) of
    // the quarter, and after the quad's reduction owns key qc of its four: half qc / 2,
    // row qd + 8 (qc % 2)
    const int qd = lane >> 2, qc = lane & 3;
    const int key_lane = quarter * 32 + 16 * (qc >> 1) + 8 * (qc & 1) + qd;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    float hw[16];  // the halved weights of this thread's chains: hw[2j + e] = w[t, 8j + 2 qc + e] / 2
    const uint32_t K = static_cast<uint32_t>(p.top_k);
    const uint64_t pol_cand = policy_evict_last();   // working buffers: reused unit after unit
    const uint64_t pol_store = policy_evict_first();  // candidate store: read only by the next kernel
    uint32_t* hist_g = reinterpret_cast<uint32_t*>(smem + kOffHist) + g * kBins;
    uint32_t* qs = s_qs + g * 4;
    unsigned long long* cand = p.cand + static_cast<size_t>(blockIdx.x) * kCandKeysPerCta + static_cast<size_t>(g) * kQCap;
    unsigned long long* exact_scratch =
        p.cand + static_cast<size_t>(blockIdx.x) * kCandKeysPerCta + static_cast<size_t>(kQB) * kQCap + g * kMaxTopK;
    // The groups' sync points are spread over the kSyncEvery tiles, so that the MMA never
    // waits for all four groups at once.
    const int sync_phase = g * (kSyncEvery / kEpiGroups);

    uint32_t it = 0, ac = 0;
    while (true) {
      const int slot = it & 1;
      // Every decision to leave the loop is taken by the whole group at once (flag set
      // before a group barrier, read after it), so no warp is left waiting at a barrier.
      if (!mbar_wait(bars.uf(slot), (it >> 1) & 1, s_abort, p.wait_limit)) {
        record_timeout(p.status, s_abort, 8);
        atomicOr(&s_gfail[g], 1u);
      }
      gsync(c);
      if (s_gfail[g]) break;
      const int4 unit = s_unit[2 * slot];
      if (unit.x < 0) break;
      const bool active = g < unit.y;  // uniform across the group
      const int4 range = s_unit[2 * slot + 1];
      const size_t uidx = static_cast<size_t>(range.x);
      if (c.gtid < kHeads) s_w[g * kHeads + c.gtid] = active ? p.w[static_cast<size_t>(unit.x + g) * kHeads + c.gtid] : 0.f;
      // A unit whose queries see at most kCap keys of its tile range hands every visible
      // key over: the appends go straight to the store slots, with no histogram, no sync
      // points and no copy at the end (uniform across the CTA).
      const int visible = min(unit.w + unit.y, range.z * kBlockKeys) - range.y * kBlockKeys;  // most keys a query sees
      const bool direct = visible <= kCap;
      // Sync points raise the threshold and make room in the working buffer. A unit whose
      // queries see at most kQCap keys can never overflow its buffer, and its sync points
      // cost more than the appends they save: it raises the threshold once, at the end.
      const bool no_sync = visible <= kQCap;
      if (!direct)
        for (int i = c.gtid; i < kBins; i += 128) hist_g[i] = 0u;
      const int tile0 = range.y, nt = range.z - range.y;
      const int last_key = unit.w + g;  // causal bound: local keys 0..last_key are visible
      // units without sync points append every visible key, key j of the unit's range at
      // slot j: the count is known from the start
      const int mine = min(last_key + 1 - tile0 * kBlockKeys, nt * kBlockKeys);
      // (a filtered unit's first kDenseTiles tiles are appended the same way, so at most
      // kQCap keys before its first sync point)
      if (c.gtid < 4) qs[c.gtid] = (c.gtid == 0 && active) ? static_cast<uint32_t>(min(max(mine, 0), kQCap)) : 0u;
      gsync(c);
  #pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 wp = *reinterpret_cast<const float2*>(s_w + g * kHeads + 8 * j + 2 * qc);
        hw[2 * j] = 0.5f * wp.x;
        hw[2 * j + 1] = 0.5f * wp.y;
      }
      // The tile loop, compiled for three kinds of unit: direct (every visible key to the
      // store), dense (every visible key to the working buffer, no sync points) and
      // filtered (threshold raised at sync points).
      auto scan_tiles = [&](auto mode_tag) -> bool {
        constexpr int kMode = decltype(mode_tag)::value;
        constexpr bool kDirect = kMode == 0;
        constexpr bool kDense = kMode < 2;  // key j of the unit's tile range goes to slot j
        unsigned long long* app = kDirect ? p.store + (uidx * kQB + g) * kCap : cand;
        const uint64_t pol_app = kDirect ? pol_store : pol_cand;
        bool failed = false;
        uint32_t thr = 0u;  // threshold bin, refreshed at every sync point
        float thr_f = -__int_as_float(0x7F800000);  // the lowest score of bin thr (bins below 4 hold no finite score)
        for (int tile = 0; tile < nt; ++tile, ++ac) {
          const int ab = ac & 1;
          // A filtered unit appends its first kDenseTiles tiles densely (slot = key index,
          // no sync points), then raises the threshold and compacts once, then filters.
          if (!kDense && (tile == kDenseTiles || (tile > kDenseTiles && tile % kSyncEvery == sync_phase))) {
            // Group sync point (the only barriers inside a unit): every append of the
            // earlier tiles is done, so the count and the histogram are final.
            gsync(c);
            if (s_gfail[g]) {  // uniform: read after the barrier
              failed = true;
              break;
            }
            if (active) {
              if (tile == kDenseTiles)  // the unit's first raise (uniform)
                group_raise_threshold(c, qs, hist_g, K);
              else if (c.gwarp == 0)
                warp_raise_threshold(qs, hist_g, K, lane);
              gsync(c);
              // make room for the appends of the next kSyncEvery tiles (uniform decision)
              if (qs[0] > kCompactAt)
                epi_compact(c, cand, qs, hist_g, K, &s_pos[g], pol_cand, kCompactAt, exact_scratch);
              thr = qs[2];
              thr_f = thr < 4u ? -__int_as_float(0x7F800000) : key_to_float(thr << kBinShift);
            }
          }
          // The warp enters this wait converged (every branch above is uniform or closes
          // before it), so each try_wait, abort-flag read and clock read of the wait is one
          // instruction for all 32 lanes and returns them the same value: the warp leaves
          // the wait as one, as the warp-wide tensor-memory loads and shuffles below need.
          if (!mbar_wait(bars.af(ab), (ac >> 1) & 1, s_abort, p.wait_limit)) {
            record_timeout(p.status, s_abort, 10);
            atomicOr(&s_gfail[g], 1u);  // the group leaves at its next sync point
            continue;
          }
          tc_fence_after_sync();
          const int jl = (tile0 + tile) * kBlockKeys + key_lane;  // local key index within the segment
          float score = 0.f;
          if (active) {
            const uint32_t col = static_cast<uint32_t>(ab * kN + g * kHeads);
            float P[4];  // P_qc of the quad's keys: [2 half] row qd, [2 half + 1] row qd + 8
  #pragma unroll
            for (int half = 0; half < 2; ++half) {  // key rows 16 half .. 16 half + 15 of the quarter
              uint32_t x[32];
              tmem_ld16x256b_x8(lane_addr + (static_cast<uint32_t>(16 * half) << 16) + col, x);
              tmem_ld_wait();
              if (half == 1) {  // every column is in registers: hand the accumulator back now
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.ae(ab));
              }
              float pa0 = 0.f, pa1 = 0.f, pb0 = 0.f, pb1 = 0.f;
  #pragma unroll
              for (int j = 0; j < 8; ++j) {  // heads 8j + 2 qc and 8j + 2 qc + 1
                relu_fma2(pa0, pa1, hw[2 * j], hw[2 * j + 1], __uint_as_float(x[4 * j + 0]),
                          __uint_as_float(x[4 * j + 1]));
                relu_fma2(pb0, pb1, hw[2 * j], hw[2 * j + 1], __uint_as_float(x[4 * j + 2]),
                          __uint_as_float(x[4 * j + 3]));
              }
              P[2 * half] = pa0 + pa1;
              P[2 * half + 1] = pb0 + pb1;
            }
            // (P0 + P1) + (P2 + P3) over the quad; a + b and b + a are the same bits, so each
            // key's sum is the fixed tree whichever thread adds it. Round 1 (threads c, c ^ 1):
            // keep the keys k with k % 2 == c % 2. Round 2 (c, c ^ 2): keep key c.
            const bool odd = (qc & 1) != 0;
            const float q0 = (odd ? P[1] : P[0]) + __shfl_xor_sync(0xFFFFFFFFu, odd ? P[0] : P[1], 1);
            const float q1 = (odd ? P[3] : P[2]) + __shfl_xor_sync(0xFFFFFFFFu, odd ? P[2] : P[3], 1);
            const bool hi = (qc & 2) != 0;
            score = ((hi ? q1 : q0) + __shfl_xor_sync(0xFFFFFFFFu, hi ? q0 : q1, 2)) + 0.0f;
          }
          if (!active) {  // this group reads no columns of the buffer
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.ae(ab));
          }
          if (kDense || tile < kDenseTiles) {  // every visible key, at the slot of its index (scores are finite)
            if (active && jl <= last_key) {
              const uint32_t key32 = ord_key(score);
              st_hint_u64(app + tile * kBlockKeys + key_lane,
                          (static_cast<unsigned long long>(key32) << 32) | static_cast<uint32_t>(unit.z + jl), pol_app);
              if (!kDirect) hist_inc(hist_g, key32 >> kBinShift);
            }
          } else {
            // append the keys that pass the filter
            const bool ins = active && jl <= last_key && score >= thr_f;  // == bin(score) >= thr for finite scores
            const uint32_t m = __ballot_sync(0xFFFFFFFFu, ins);
            if (m) {
              const int lead = __ffs(m) - 1;
              uint32_t base = 0u;
              if (lane == lead) base = atomicAdd(&qs[0], static_cast<uint32_t>(__popc(m)));
              base = __shfl_sync(0xFFFFFFFFu, base, lead);
              if (ins) {
                const uint32_t key32 = ord_key(score);
                st_hint_u64(app + base + __popc(m & ((1u << lane) - 1u)),
                            (static_cast<unsigned long long>(key32) << 32) | static_cast<uint32_t>(unit.z + jl), pol_app);
                if (!kDirect) hist_inc(hist_g, key32 >> kBinShift);
              }
            }
          }
        }
        return failed;
      };
      const bool failed = direct    ? scan_tiles(std::integral_constant<int, 0>{})
                          : no_sync ? scan_tiles(std::integral_constant<int, 1>{})
                                    : scan_tiles(std::integral_constant<int, 2>{});
      if (failed) break;
      // Hand-off: every candidate of the unit's query goes to the store.
      gsync(c);  // every append of the unit is done
      if (active) {
        const size_t item = uidx * kQB + g;
        if (direct) {
          if (c.gtid == 0) p.counts[item] = qs[0];  // every visible key, at most kCap
        } else {
          if (no_sync)  // a unit without sync points: its first raise (uniform)
            group_raise_threshold(c, qs, hist_g, K);
          else if (c.gwarp == 0)
            warp_raise_threshold(qs, hist_g, K, lane);
          gsync(c);
          epi_handoff(c, cand, qs, K, &s_pos[g], pol_cand, pol_store, p.store + item * kCap, p.counts + item, p.status);
        }
      }
      gsync(c);
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.ue(slot));
      ++it;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace itk
