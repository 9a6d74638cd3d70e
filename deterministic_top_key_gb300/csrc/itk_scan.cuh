// The scan kernel: persistent CTAs draw work units from a self-resetting ticket word;
// each unit (up to 4 consecutive queries of one segment) streams its visible key tiles
// through a tcgen05 GEMM with the keys as the M side, a fused ReLU * w head reduction and
// an exact streaming top-k selection.
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
// CTA layout (320 threads):
//   warp 0      ticket draws, TMA loads of the Q block and of the K tile ring
//   warp 1      TMEM allocation, tcgen05.mma issue (one thread)
//   warps 2..9  epilogue: two groups of four warps; group g owns queries 2g and 2g+1 of
//               the unit; the four warps of a group cover the 128 TMEM lanes (keys).
//
// Score arithmetic (fixed, so the result does not depend on tiling or on which CTA runs
// a unit): the tensor core forms the FP32 dot products q[t,h,:].k[s,:] over D = 128 in
// eight K = 16 steps in a fixed order; the epilogue thread that owns key s then computes
//     acc = 0; for h = 0..63: acc = fma(w[t,h], max(dot_h, 0), acc);  score = acc + 0
// (the "+ 0" turns a -0 into +0). Selection compares (score, id) pairs packed into one
// 64-bit key (order-preserving score bits above the id), so the order is total and the
// selected set and its order are unique.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "itk_ptx.cuh"

namespace itk {

constexpr int kHeads = 64;
constexpr int kDim = 128;
constexpr int kQB = 4;                       // queries per work unit
constexpr int kBlockKeys = 128;              // keys per tile (MMA M)
constexpr int kN = kQB * kHeads;             // MMA N = 256 (query, head) columns
constexpr int kStages = 3;                   // K tile ring depth
constexpr int kMaxTopK = 2048;
constexpr int kCap = 4096;                   // candidate buffer entries per query
constexpr int kPerThread = kCap / 128;       // candidate entries a group thread holds in compaction
constexpr int kNumThreads = 320;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;          // two accumulator buffers of 256 columns

constexpr uint32_t kQHalfBytes = kN * 64 * 2;           // 256 rows x 128 B = 32 KB
constexpr uint32_t kQBytes = 2 * kQHalfBytes;            // 64 KB
constexpr uint32_t kKHalfBytes = kBlockKeys * 64 * 2;    // 128 rows x 128 B = 16 KB
constexpr uint32_t kKStageBytes = 2 * kKHalfBytes;       // 32 KB

// Shared memory layout (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffSort = kOffK + kStages * kKStageBytes;          // 2 groups x 2048 x 8 B
constexpr uint32_t kOffW = kOffSort + 2 * kMaxTopK * 8;                // 4 queries x 64 floats
constexpr uint32_t kOffHist = kOffW + kQB * kHeads * 4;                // 2 groups x 256 x 4 B
constexpr uint32_t kOffThr = kOffHist + 2 * 256 * 4;                   // 4 x u64
constexpr uint32_t kOffCnt = kOffThr + kQB * 8;                        // 4 x u32
constexpr uint32_t kOffSel = kOffCnt + kQB * 4;                        // 2 groups x 4 x u32
constexpr uint32_t kOffUnit = kOffSel + 2 * 4 * 4;                     // 2 slots x int4
constexpr uint32_t kOffBar = kOffUnit + 2 * 16;                        // mbarriers
constexpr uint32_t kNumBars = 2 * kStages + 2 + 2 + 2 + 2 + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;                  // tmem base, abort, fail flags
constexpr uint32_t kSmemUsed = kOffMisc + 32;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;                      // slack for 1024-byte alignment

static_assert(kOffK % 1024 == 0 && kKStageBytes % 1024 == 0 && kQHalfBytes % 1024 == 0, "SW128 tiles need 1 KB alignment");
static_assert(kOffBar % 8 == 0, "mbarrier alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct UnitDesc {
  int32_t q_row0;    // first query row of the unit
  int32_t nq;        // queries in the unit (1..4)
  int32_t key_row0;  // first key row of the unit's segment
  int32_t pos0;      // causal position of the first query within its segment
};

struct TicketBlock {
  unsigned long long next;  // next unit to hand out
  unsigned long long done;  // CTAs that finished drawing
};

struct ScanParams {
  const UnitDesc* units;
  int32_t n_units;
  int32_t top_k;
  TicketBlock* ticket;
  uint32_t* status;              // device status word (0 = ok)
  const float* w;                // [T,64]
  int32_t* out_ids;              // [T,top_k]
  float* out_scores;             // [T,top_k]
  unsigned long long* cand;      // workspace: gridDim.x x 4 x kCap candidate keys
};

constexpr uint32_t kStatusTimeout = 10u;  // matches ITK_ERR_DEVICE_TIMEOUT

__device__ __forceinline__ uint32_t ord_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t o) {
  const uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(b);
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

__device__ __forceinline__ int n_tiles_of(const int4& u) {
  return (u.w + u.y + kBlockKeys - 1) / kBlockKeys;  // ceil((pos0 + nq) / 128)
}

__device__ __forceinline__ void record_timeout(const ScanParams& p, volatile uint32_t* abort_flag, uint32_t role) {
  *abort_flag = 1u;
  atomicOr(p.status, kStatusTimeout | (role << 8));
}

// ------------------------------------------------------------------ group selection
// The 128 threads of an epilogue group select, among `n` candidate keys, the `K`
// largest. Keys are held in registers (entry gtid + 128*r). Radix select from the top
// byte down; stops as soon as the bucket that holds the K-th largest key is taken whole.
// Returns `prefix` with #{valid x : x >= prefix} == K.
struct GroupCtx {
  int g;          // group 0/1
  int gtid;       // 0..127
  int gwarp;      // 0..3
  int lane;
  uint32_t bar;   // named barrier id
  uint32_t* hist; // 256 bins
  uint32_t* sel;  // 4 words of scratch
};

__device__ __forceinline__ void gsync(const GroupCtx& c) { named_bar_sync(c.bar, 128); }

__device__ unsigned long long group_select(const GroupCtx& c, const unsigned long long (&v)[kPerThread], uint32_t n,
                                           uint32_t K) {
  unsigned long long prefix = 0ull;
  uint32_t k_rem = K;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = c.gtid; i < 256; i += 128) c.hist[i] = 0u;
    gsync(c);
    const unsigned long long hi_mask = (shift == 56) ? 0ull : (~0ull << (shift + 8));
#pragma unroll
    for (int r = 0; r < kPerThread; ++r) {
      const uint32_t idx = c.gtid + 128u * r;
      if (idx < n && ((v[r] & hi_mask) == (prefix & hi_mask)))
        atomicAdd(&c.hist[(v[r] >> shift) & 0xFFu], 1u);
    }
    gsync(c);
    if (c.gwarp == 0) {
      // lane L scans bins 255-8L .. 248-8L (highest bins first)
      uint32_t cnt[8];
      uint32_t s = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = c.hist[255 - 8 * c.lane - i];
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
    gsync(c);
    const uint32_t b = c.sel[0];
    const uint32_t rem = c.sel[1];
    const uint32_t bucket = c.sel[2];
    prefix |= static_cast<unsigned long long>(b) << shift;
    k_rem = rem;
    if (bucket == k_rem) break;  // the whole bucket is selected; uniform across the group
  }
  return prefix;
}

// Load the candidate buffer into registers (invalid slots are 0, below every real key).
__device__ __forceinline__ void group_load(const GroupCtx& c, const unsigned long long* buf, uint32_t n,
                                           unsigned long long (&v)[kPerThread]) {
#pragma unroll
  for (int r = 0; r < kPerThread; ++r) {
    const uint32_t idx = c.gtid + 128u * r;
    v[r] = idx < n ? buf[idx] : 0ull;
  }
}

// Keep the K largest of the n candidates in buf (n > K): afterwards buf[0..K) holds them
// (in no particular order) and the return value is a key threshold t such that every
// kept key is >= t and every dropped key is < t.
__device__ unsigned long long group_compact(const GroupCtx& c, unsigned long long* buf, uint32_t n, uint32_t K,
                                            uint32_t* s_pos) {
  unsigned long long v[kPerThread];
  group_load(c, buf, n, v);
  if (c.gtid == 0) *s_pos = 0u;
  const unsigned long long prefix = group_select(c, v, n, K);  // contains barriers after the loads
#pragma unroll
  for (int r = 0; r < kPerThread; ++r) {
    const uint32_t idx = c.gtid + 128u * r;
    const bool keep = idx < n && v[r] >= prefix;
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, keep);
    if (m) {
      uint32_t base = 0;
      const int leader = __ffs(m) - 1;
      if (c.lane == leader) base = atomicAdd(s_pos, static_cast<uint32_t>(__popc(m)));
      base = __shfl_sync(0xFFFFFFFFu, base, leader);
      if (keep) buf[base + __popc(m & ((1u << c.lane) - 1u))] = v[r];
    }
  }
  gsync(c);
  return prefix;
}

// Final selection, sort and output of one query row.
__device__ void group_finish(const GroupCtx& c, const unsigned long long* buf, uint32_t n, uint32_t top_k,
                             unsigned long long* sbuf, uint32_t* s_pos, int32_t* out_ids, float* out_scores) {
  unsigned long long v[kPerThread];
  group_load(c, buf, n, v);
  const uint32_t keff = n < top_k ? n : top_k;
  unsigned long long prefix = 0ull;
  if (c.gtid == 0) *s_pos = 0u;
  if (n > top_k) {
    prefix = group_select(c, v, n, top_k);
  } else {
    gsync(c);
  }
  // gather the kept keys into shared memory
#pragma unroll
  for (int r = 0; r < kPerThread; ++r) {
    const uint32_t idx = c.gtid + 128u * r;
    const bool keep = idx < n && v[r] >= prefix;
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, keep);
    if (m) {
      uint32_t base = 0;
      const int leader = __ffs(m) - 1;
      if (c.lane == leader) base = atomicAdd(s_pos, static_cast<uint32_t>(__popc(m)));
      base = __shfl_sync(0xFFFFFFFFu, base, leader);
      if (keep) sbuf[base + __popc(m & ((1u << c.lane) - 1u))] = v[r];
    }
  }
  uint32_t np2 = 2;
  while (np2 < keff) np2 <<= 1;
  gsync(c);
  for (uint32_t i = keff + c.gtid; i < np2; i += 128) sbuf[i] = 0ull;
  gsync(c);
  // bitonic sort, descending
  for (uint32_t size = 2; size <= np2; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t i = c.gtid; i < np2 / 2; i += 128) {
        const uint32_t lo = 2 * i - (i & (stride - 1));
        const uint32_t hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long a = sbuf[lo];
        const unsigned long long b = sbuf[hi];
        if ((a < b) == desc) {
          sbuf[lo] = b;
          sbuf[hi] = a;
        }
      }
      gsync(c);
    }
  }
  for (uint32_t r = c.gtid; r < top_k; r += 128) {
    if (r < keff) {
      const unsigned long long x = sbuf[r];
      out_ids[r] = static_cast<int32_t>(static_cast<uint32_t>(x & 0xFFFFFFFFull));
      out_scores[r] = key_to_float(static_cast<uint32_t>(x >> 32));
    } else {
      out_ids[r] = -1;
      out_scores[r] = -__int_as_float(0x7F800000);
    }
  }
  gsync(c);
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kNumThreads, 1)
    indexer_topk_scan_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                             const ScanParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  unsigned long long* s_thr = reinterpret_cast<unsigned long long*>(smem + kOffThr);
  uint32_t* s_cnt = reinterpret_cast<uint32_t*>(smem + kOffCnt);
  int4* s_unit = reinterpret_cast<int4*>(smem + kOffUnit);
  float* s_w = reinterpret_cast<float*>(smem + kOffW);
  uint32_t* s_misc = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  uint32_t* s_tmem = s_misc + 0;
  volatile uint32_t* s_abort = s_misc + 1;
  uint32_t* s_gfail = s_misc + 2;  // [2] per-group failure flags
  uint32_t* s_pos = s_misc + 4;    // [2] per-group compaction cursors

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
    s_misc[1] = 0u;
    s_misc[2] = 0u;
    s_misc[3] = 0u;
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

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_k = policy_evict_last();
      const uint64_t pol_q = policy_evict_first();
      uint32_t it = 0, kc = 0, qloads = 0;
      bool ok = true;
      while (ok) {
        const unsigned long long u = atomicAdd(&p.ticket->next, 1ull);
        const int slot = it & 1;
        if (!mbar_wait(bars.ue(slot), ((it >> 1) & 1) ^ 1, s_abort)) {
          record_timeout(p, s_abort, 1);
          break;
        }
        int4 unit;
        if (u < static_cast<unsigned long long>(p.n_units)) {
          const UnitDesc d = p.units[u];
          unit = make_int4(d.q_row0, d.nq, d.key_row0, d.pos0);
        } else {
          unit = make_int4(-1, 0, 0, 0);
        }
        s_unit[slot] = unit;
        mbar_arrive(bars.uf(slot));
        if (unit.x < 0) break;
        if (!mbar_wait(bars.qempty, (it & 1) ^ 1, s_abort)) {
          record_timeout(p, s_abort, 2);
          break;
        }
        mbar_arrive_expect_tx(bars.qfull, kQBytes);
        const uint32_t qdst = smem_u32(smem + kOffQ);
        tma_load_2d(qdst, &q_map, bars.qfull, 0, unit.x * kHeads, pol_q);
        tma_load_2d(qdst + kQHalfBytes, &q_map, bars.qfull, 64, unit.x * kHeads, pol_q);
        ++qloads;
        const int nt = n_tiles_of(unit);
        for (int tile = 0; tile < nt; ++tile, ++kc) {
          const int s = kc % kStages;
          if (!mbar_wait(bars.ke(s), ((kc / kStages) & 1) ^ 1, s_abort)) {
            record_timeout(p, s_abort, 3);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bars.kf(s), kKStageBytes);
          const uint32_t kdst = smem_u32(smem + kOffK + s * kKStageBytes);
          const int row = unit.z + tile * kBlockKeys;
          tma_load_2d(kdst, &k_map, bars.kf(s), 0, row, pol_k);
          tma_load_2d(kdst + kKHalfBytes, &k_map, bars.kf(s), 64, row, pol_k);
        }
        ++it;
      }
      // Drain: make sure no TMA write into this CTA's shared memory is still in flight
      // (these waits ignore the abort flag but keep their time limit).
      for (uint32_t j = (kc > kStages ? kc - kStages : 0); j < kc; ++j)
        mbar_wait(bars.kf(j % kStages), (j / kStages) & 1, nullptr);
      if (qloads > 0) mbar_wait(bars.qfull, (qloads - 1) & 1, nullptr);
      // The last CTA to finish drawing resets the ticket block for the next scan.
      __threadfence();
      const unsigned long long prev = atomicAdd(&p.ticket->done, 1ull);
      if (prev == static_cast<unsigned long long>(gridDim.x) - 1ull) {
        atomicExch(&p.ticket->next, 0ull);
        atomicExch(&p.ticket->done, 0ull);
      }
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
        if (!mbar_wait(bars.uf(slot), (it >> 1) & 1, s_abort)) {
          record_timeout(p, s_abort, 4);
          break;
        }
        const int4 unit = s_unit[slot];
        if (unit.x < 0) break;
        if (!mbar_wait(bars.qfull, it & 1, s_abort)) {
          record_timeout(p, s_abort, 5);
          break;
        }
        const int nt = n_tiles_of(unit);
        for (int tile = 0; tile < nt; ++tile, ++kc, ++ac) {
          const int ab = ac & 1;
          if (!mbar_wait(bars.ae(ab), ((ac >> 1) & 1) ^ 1, s_abort)) {
            record_timeout(p, s_abort, 6);
            ok = false;
            break;
          }
          const int s = kc % kStages;
          if (!mbar_wait(bars.kf(s), (kc / kStages) & 1, s_abort)) {
            record_timeout(p, s_abort, 7);
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
      // Wait until every MMA this thread issued has completed before TMEM is released
      // (ignores the abort flag, keeps the time limit).
      mma_commit(bars.mmadone);
      mbar_wait(bars.mmadone, 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - 2;
    GroupCtx c;
    c.g = ew >> 2;
    c.gwarp = ew & 3;
    c.lane = lane;
    c.gtid = c.gwarp * 32 + lane;
    c.bar = 1 + c.g;
    c.hist = reinterpret_cast<uint32_t*>(smem + kOffHist) + 256 * c.g;
    c.sel = reinterpret_cast<uint32_t*>(smem + kOffSel) + 4 * c.g;
    unsigned long long* sbuf = reinterpret_cast<unsigned long long*>(smem + kOffSort) + kMaxTopK * c.g;
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int key_lane = quarter * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    unsigned long long* cand_base = p.cand + static_cast<size_t>(blockIdx.x) * kQB * kCap;

    uint32_t it = 0, ac = 0;
    while (true) {
      const int slot = it & 1;
      // Every decision to leave the loop is taken by the whole group at once (flag set
      // before a group barrier, read after it), so no warp is left waiting at a barrier.
      if (!mbar_wait(bars.uf(slot), (it >> 1) & 1, s_abort)) {
        record_timeout(p, s_abort, 8);
        atomicOr(&s_gfail[c.g], 1u);
      }
      gsync(c);
      if (s_gfail[c.g]) break;
      const int4 unit = s_unit[slot];
      if (unit.x < 0) break;
      // per-unit state of this group's two queries
      for (int i = c.gtid; i < 2 * kHeads; i += 128) {
        const int jj = i / kHeads, h = i % kHeads;
        const int j = 2 * c.g + jj;
        s_w[j * kHeads + h] = j < unit.y ? p.w[static_cast<size_t>(unit.x + j) * kHeads + h] : 0.f;
      }
      if (c.gtid < 2) {
        s_cnt[2 * c.g + c.gtid] = 0u;
        s_thr[2 * c.g + c.gtid] = 0ull;
      }
      gsync(c);
      const int nt = n_tiles_of(unit);
      bool failed = false;
      for (int tile = 0; tile < nt; ++tile, ++ac) {
        const int ab = ac & 1;
        if (!mbar_wait(bars.af(ab), (ac >> 1) & 1, s_abort)) {
          record_timeout(p, s_abort, 9);
          atomicOr(&s_gfail[c.g], 1u);
        }
        gsync(c);
        if (s_gfail[c.g]) {
          failed = true;
          break;
        }
        tc_fence_after_sync();
        const int jl = tile * kBlockKeys + key_lane;  // local key index within the segment
#pragma unroll 1
        for (int jj = 0; jj < 2; ++jj) {
          const int j = 2 * c.g + jj;
          if (j >= unit.y) continue;  // uniform across the group
          uint32_t r0[32], r1[32];
          const uint32_t col = static_cast<uint32_t>(ab * kN + j * kHeads);
          tmem_ld32(lane_addr + col, r0);
          tmem_ld32(lane_addr + col + 32, r1);
          tmem_ld_wait();
          const float4* wv = reinterpret_cast<const float4*>(s_w + j * kHeads);
          float acc = 0.f;
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 w4 = wv[h4];
            acc = fmaf(w4.x, fmaxf(__uint_as_float(r0[4 * h4 + 0]), 0.f), acc);
            acc = fmaf(w4.y, fmaxf(__uint_as_float(r0[4 * h4 + 1]), 0.f), acc);
            acc = fmaf(w4.z, fmaxf(__uint_as_float(r0[4 * h4 + 2]), 0.f), acc);
            acc = fmaf(w4.w, fmaxf(__uint_as_float(r0[4 * h4 + 3]), 0.f), acc);
          }
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 w4 = wv[8 + h4];
            acc = fmaf(w4.x, fmaxf(__uint_as_float(r1[4 * h4 + 0]), 0.f), acc);
            acc = fmaf(w4.y, fmaxf(__uint_as_float(r1[4 * h4 + 1]), 0.f), acc);
            acc = fmaf(w4.z, fmaxf(__uint_as_float(r1[4 * h4 + 2]), 0.f), acc);
            acc = fmaf(w4.w, fmaxf(__uint_as_float(r1[4 * h4 + 3]), 0.f), acc);
          }
          const float score = acc + 0.0f;
          const bool vis = jl <= unit.w + j;
          const unsigned long long key = (static_cast<unsigned long long>(ord_key(score)) << 32) |
                                         static_cast<uint32_t>(unit.z + jl);
          const bool ins = vis && key >= s_thr[j];
          const uint32_t m = __ballot_sync(0xFFFFFFFFu, ins);
          if (m) {
            uint32_t base = 0;
            const int leader = __ffs(m) - 1;
            if (lane == leader) base = atomicAdd(&s_cnt[j], static_cast<uint32_t>(__popc(m)));
            base = __shfl_sync(0xFFFFFFFFu, base, leader);
            if (ins) cand_base[static_cast<size_t>(j) * kCap + base + __popc(m & ((1u << lane) - 1u))] = key;
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.ae(ab));
        gsync(c);
        // make room when the next tile could overflow a buffer
#pragma unroll 1
        for (int jj = 0; jj < 2; ++jj) {
          const int j = 2 * c.g + jj;
          if (j >= unit.y) continue;
          const uint32_t n = s_cnt[j];
          if (n > static_cast<uint32_t>(kCap - kBlockKeys)) {
            const unsigned long long t =
                group_compact(c, cand_base + static_cast<size_t>(j) * kCap, n, p.top_k, &s_pos[c.g]);
            if (c.gtid == 0) {
              s_cnt[j] = static_cast<uint32_t>(p.top_k);
              s_thr[j] = t;
            }
            gsync(c);
          }
        }
      }
      if (failed) break;
#pragma unroll 1
      for (int jj = 0; jj < 2; ++jj) {
        const int j = 2 * c.g + jj;
        if (j >= unit.y) continue;
        const size_t row = static_cast<size_t>(unit.x + j);
        group_finish(c, cand_base + static_cast<size_t>(j) * kCap, s_cnt[j], static_cast<uint32_t>(p.top_k), sbuf,
                     &s_pos[c.g], p.out_ids + row * p.top_k, p.out_scores + row * p.top_k);
      }
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
