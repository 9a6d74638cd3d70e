// Host side of the C ABI declared in include/indexer_topk.h: descriptor validation,
// work-unit planning, the plan's device block (unit table + two ticket blocks + status
// word), workspace layout, tensor-map encoding and the two kernel launches per run (the
// scan, then the selection).
//
// Prepared runner and eager entry: flashinfer PR #8691, commit notes "prepare now
// decides ... before it issues its first device operation", "zero_region ... ABI
// dsa_indexer_v3", "TicketWord ... ABI dsa_indexer_v4" and the "Changes" table row
// "Runner entry points and validation".
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "../../include/indexer_topk.h"
#include "itk_scan.cuh"
#include "itk_select.cuh"

namespace {

using itk::TicketBlock;
using itk::UnitDesc;

thread_local char g_last_error[256] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ITK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Validated copy of a descriptor plus its work tables.
struct Layout {
  int32_t T = 0, Tkv = 0, top_k = 0, B = 0;
  int32_t key_id_base = 0;         // added to every returned id
  std::vector<UnitDesc> units;     // ticket order: most key tiles first
  std::vector<int32_t> item_rows;  // per store slot: output row, or -1 (empty or merged elsewhere)
  std::vector<itk::MergeDesc> merges;
  size_t select_rows = 0;          // item rows >= 0: queries the selection kernel finishes
  size_t n_slots() const { return item_rows.size(); }  // units * 4
};

// Split tails: a descriptor with at most kSplitMaxBlocks query blocks cannot fill the
// GPU with one unit per block, so every block with at least 2 * kSplitTiles key tiles is
// split into chunks of about kSplitTiles tiles (at most kSplitUnits units in all); the
// chunks' candidates are merged per query before the selection.
constexpr int kSplitMaxBlocks = 64;
constexpr int kSplitTiles = 4;
constexpr int kSplitUnits = 256;
static_assert(kSplitUnits <= itk::kMaxMergeChunks, "a split query's chunks fit the merge's count table");

int build_layout(const itk_desc* d, Layout* out) {
  if (!d) return fail(ITK_ERR_INVALID_ARGUMENT, "descriptor is NULL");
  if (d->T < 0 || d->Tkv < 0 || d->num_segments < 0)
    return fail(ITK_ERR_INVALID_ARGUMENT, "negative size (T=%d Tkv=%d B=%d)", d->T, d->Tkv, d->num_segments);
  if (d->top_k < 1) return fail(ITK_ERR_INVALID_ARGUMENT, "top_k=%d must be >= 1", d->top_k);
  if (d->H != itk::kHeads || d->D != itk::kDim)
    return fail(ITK_ERR_UNSUPPORTED, "H=%d D=%d: only H=64, D=128 are supported", d->H, d->D);
  if (d->top_k > itk::kMaxTopK) return fail(ITK_ERR_UNSUPPORTED, "top_k=%d exceeds %d", d->top_k, itk::kMaxTopK);
  if (static_cast<int64_t>(d->T) * itk::kHeads >= (int64_t(1) << 31))
    return fail(ITK_ERR_UNSUPPORTED, "T=%d too large (T*H must stay below 2^31)", d->T);
  if (d->key_id_base < 0 || static_cast<int64_t>(d->key_id_base) + d->Tkv > INT32_MAX)
    return fail(ITK_ERR_INVALID_ARGUMENT, "key_id_base=%d: ids key_id_base .. key_id_base + Tkv - 1 must lie in 0 .. 2^31-1",
                d->key_id_base);
  const int B = d->num_segments;
  if (B == 0) {
    if (d->T != 0) return fail(ITK_ERR_INVALID_SEQLENS, "no segments but T=%d", d->T);
  } else if (!d->cu_seqlens_q || !d->cu_seqlens_k) {
    return fail(ITK_ERR_NULL_POINTER, "cu_seqlens pointer is NULL");
  }
  Layout L;
  L.T = d->T;
  L.Tkv = d->Tkv;
  L.top_k = d->top_k;
  L.B = B;
  L.key_id_base = d->key_id_base;
  if (B > 0) {
    const int32_t* cq = d->cu_seqlens_q;
    const int32_t* ck = d->cu_seqlens_k;
    if (cq[0] != 0 || ck[0] != 0) return fail(ITK_ERR_INVALID_SEQLENS, "cu_seqlens must start at 0");
    for (int b = 0; b < B; ++b)
      if (cq[b + 1] < cq[b] || ck[b + 1] < ck[b])
        return fail(ITK_ERR_INVALID_SEQLENS, "cu_seqlens decrease at segment %d", b);
    if (cq[B] != d->T) return fail(ITK_ERR_INVALID_SEQLENS, "cu_seqlens_q[B]=%d != T=%d", cq[B], d->T);
    if (ck[B] > d->Tkv) return fail(ITK_ERR_INVALID_SEQLENS, "cu_seqlens_k[B]=%d > Tkv=%d", ck[B], d->Tkv);
    struct Item {
      UnitDesc u;
      int64_t tiles;
    };
    std::vector<Item> items;
    for (int b = 0; b < B; ++b) {
      const int32_t tq = cq[b + 1] - cq[b];
      const int32_t tk = ck[b + 1] - ck[b];
      if (tq == 0) continue;
      const int64_t off = d->q_causal_offsets ? d->q_causal_offsets[b] : int64_t(tk) - tq;
      if (off < 0 || off + tq > tk)
        return fail(ITK_ERR_INVALID_OFFSETS, "segment %d: offset %lld with %d queries and %d keys", b,
                    static_cast<long long>(off), tq, tk);
      for (int32_t i0 = 0; i0 < tq; i0 += itk::kQB) {
        Item it;
        it.u.q_row0 = cq[b] + i0;
        it.u.nq = std::min<int32_t>(itk::kQB, tq - i0);
        it.u.key_row0 = ck[b];
        it.u.pos0 = static_cast<int32_t>(off + i0);
        it.tiles = (int64_t(it.u.pos0) + it.u.nq + itk::kBlockKeys - 1) / itk::kBlockKeys;
        it.u.tile0 = 0;
        it.u.tile1 = static_cast<int32_t>(it.tiles);
        items.push_back(it);
      }
    }
    // Longest first: the heaviest units are handed out first so the short ones fill the tail.
    std::stable_sort(items.begin(), items.end(), [](const Item& a, const Item& b) { return a.tiles > b.tiles; });
    const int64_t n_blocks = static_cast<int64_t>(items.size());
    const int64_t chunk_budget = n_blocks > 0 ? std::max<int64_t>(1, kSplitUnits / n_blocks) : 1;
    for (const Item& it : items) {
      int64_t chunks = 1;
      if (n_blocks <= kSplitMaxBlocks && it.tiles >= 2 * kSplitTiles)
        chunks = std::min<int64_t>((it.tiles + kSplitTiles - 1) / kSplitTiles, chunk_budget);
      const int32_t first = static_cast<int32_t>(L.units.size());
      for (int64_t c = 0; c < chunks; ++c) {
        UnitDesc u = it.u;
        u.tile0 = static_cast<int32_t>(it.tiles * c / chunks);
        u.tile1 = static_cast<int32_t>(it.tiles * (c + 1) / chunks);
        L.units.push_back(u);
        for (int j = 0; j < itk::kQB; ++j) {
          const bool own = chunks == 1 && j < u.nq;  // split queries are finished by the merge
          L.item_rows.push_back(own ? u.q_row0 + j : -1);
          L.select_rows += own ? 1 : 0;
        }
      }
      if (chunks > 1)
        for (int j = 0; j < it.u.nq; ++j) {
          itk::MergeDesc m;
          m.first_unit = first;
          m.n_chunks = static_cast<int32_t>(chunks);
          m.j = j;
          m.row = it.u.q_row0 + j;
          L.merges.push_back(m);
        }
    }
  }
  *out = std::move(L);
  return ITK_OK;
}

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
};

int query_device(DeviceInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ITK_ERR_NO_DEVICE, "cudaGetDevice: %s", cudaGetErrorString(e));
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(ITK_ERR_NO_DEVICE, "device attributes: %s", cudaGetErrorString(e));
  if (major != 10 || minor != 3)
    return fail(ITK_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
  info->device = dev;
  info->sm_count = sms;
  return ITK_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time libcuda).
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// Row-major BF16 [rows, 128] as a 2-D tensor map with a 64-column x box_rows box and the
// 128-byte swizzle (the layout the tcgen05 shared-memory descriptors expect).
int encode_rows(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  EncodeFn enc = get_encode();
  if (!enc) return fail(ITK_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(itk::kDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(itk::kDim) * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ITK_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return ITK_OK;
}

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int grid_for(size_t n_units, int sm_count) {
  return static_cast<int>(std::min<size_t>(n_units, static_cast<size_t>(sm_count)));
}

// Device block layout shared by the plan and the eager entry:
// [units | item rows | merges | scan ticket | selection ticket | status].
struct BlockLayout {
  size_t units_off = 0, items_off = 0, merges_off = 0, ticket_off = 0, sel_ticket_off = 0, status_off = 0, bytes = 0;
};
BlockLayout block_layout(const Layout& L) {
  BlockLayout b;
  b.units_off = 0;
  b.items_off = align_up(L.units.size() * sizeof(UnitDesc), 64);
  b.merges_off = align_up(b.items_off + L.item_rows.size() * sizeof(int32_t), 64);
  b.ticket_off = align_up(b.merges_off + L.merges.size() * sizeof(itk::MergeDesc), 64);
  b.sel_ticket_off = b.ticket_off + sizeof(TicketBlock);
  b.status_off = b.sel_ticket_off + sizeof(TicketBlock);
  b.bytes = b.status_off + 16;
  return b;
}
// The block's initial contents: the tables, then zeroed ticket blocks and status word.
std::vector<unsigned char> block_image(const Layout& L, const BlockLayout& b) {
  std::vector<unsigned char> host(b.bytes, 0);
  std::memcpy(host.data() + b.units_off, L.units.data(), L.units.size() * sizeof(UnitDesc));
  std::memcpy(host.data() + b.items_off, L.item_rows.data(), L.item_rows.size() * sizeof(int32_t));
  std::memcpy(host.data() + b.merges_off, L.merges.data(), L.merges.size() * sizeof(itk::MergeDesc));
  return host;
}

// Workspace layout of one run: per-CTA working buffers of the scan, then the candidate
// store (kCap keys per slot, four slots per unit), then the per-slot counts.
struct WorkLayout {
  size_t cand_off = 0, store_off = 0, counts_off = 0, bytes = 0;
};
constexpr WorkLayout work_layout(int grid, size_t n_slots) {
  WorkLayout w;
  w.cand_off = 0;
  w.store_off = align_up(static_cast<size_t>(grid) * itk::candidate_bytes_per_cta(), 256);
  w.counts_off = w.store_off + align_up(n_slots * itk::kCap * sizeof(unsigned long long), 256);
  w.bytes = w.counts_off + align_up(n_slots * sizeof(uint32_t), 256);
  return w;
}

// Device addresses of one run's tables.
struct RunTables {
  const UnitDesc* units = nullptr;
  size_t n_units = 0;
  const int32_t* item_rows = nullptr;
  size_t n_slots = 0;
  const itk::MergeDesc* merges = nullptr;
  size_t n_merges = 0;
  bool select = true;              // some slot has an output row (else no selection launch)
  TicketBlock* tickets = nullptr;  // two adjacent blocks: scan, selection
  uint32_t* status = nullptr;
};
RunTables block_tables(const Layout& L, const BlockLayout& b, char* blk) {
  RunTables t;
  t.units = reinterpret_cast<const UnitDesc*>(blk + b.units_off);
  t.n_units = L.units.size();
  t.item_rows = reinterpret_cast<const int32_t*>(blk + b.items_off);
  t.n_slots = L.item_rows.size();
  t.merges = reinterpret_cast<const itk::MergeDesc*>(blk + b.merges_off);
  t.n_merges = L.merges.size();
  t.select = L.select_rows > 0;
  t.tickets = reinterpret_cast<TicketBlock*>(blk + b.ticket_off);
  t.status = reinterpret_cast<uint32_t*>(blk + b.status_off);
  return t;
}

constexpr size_t kSelSmemLaunch = itk::kSelSmemBytes + 128;  // slack for 128-byte alignment

int ensure_kernel_attributes() {
  static cudaError_t err = cudaErrorUnknown;
  static std::once_flag once;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(itk::indexer_topk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(itk::kSmemBytes));
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(itk::indexer_topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSelSmemLaunch));
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(itk::indexer_topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(itk::kMergeSmemBytes));
  });
  if (err != cudaSuccess) return cuda_fail(err, "cudaFuncSetAttribute");
  return ITK_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Launches `kernel` on `stream` as a programmatic dependent of the stream's previous kernel:
// its CTAs may start (and run their set-up) while that kernel's last CTAs finish; each
// kernel waits (griddepcontrol.wait) before it reads anything the previous one wrote.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), int grid, int block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  const cudaError_t last = cudaGetLastError();  // clears the launch error, as after a <<<>>> launch
  return e != cudaSuccess ? e : last;
}

int check_run_buffers(const Layout& L, const void* q, const void* k, const float* w, int32_t* ids, float* scores) {
  if (!q || !k || !w || !ids || !scores) return fail(ITK_ERR_NULL_POINTER, "q, k, w, out_ids or out_scores is NULL");
  if (!aligned(q, 16) || !aligned(k, 16)) return fail(ITK_ERR_MISALIGNED, "q and k must be 16-byte aligned");
  if (!aligned(w, 4) || !aligned(ids, 4) || !aligned(scores, 4))
    return fail(ITK_ERR_MISALIGNED, "w, out_ids and out_scores must be 4-byte aligned");
  (void)L;
  return ITK_OK;
}

// Encode maps and launch the scan over the units of `t`, then the merge of split queries
// (if any) and the selection of every slot with an output row (if any). `work` is laid
// out by work_layout(grid, t.n_slots).
// Test hooks of one run (indexer_topk_debug_inject).
struct RunHooks {
  bool force_launch_failure = false;  // the scan launch is refused by the runtime
  bool static_schedule = false;       // fixed units per CTA instead of the ticket
  bool withhold_timeout = false;      // CTA 0 withholds a key-tile load; waits limited to kShortWaitCycles
};
constexpr long long kShortWaitCycles = 1ll << 21;  // about 1 ms at 2 GHz

int launch_run(const Layout& L, int grid, int sm_count, const RunTables& t, const void* q, const void* k,
               const float* w, int32_t* ids, float* scores, void* work, cudaStream_t stream,
               const RunHooks& hooks = RunHooks(), cudaEvent_t split_event = nullptr) {
  CUtensorMap qmap, kmap;
  int rc = encode_rows(&qmap, q, static_cast<uint64_t>(L.T) * itk::kHeads, itk::kN);
  if (rc) return rc;
  rc = encode_rows(&kmap, k, static_cast<uint64_t>(std::max(L.Tkv, 1)), itk::kBlockKeys);
  if (rc) return rc;
  rc = ensure_kernel_attributes();
  if (rc) return rc;
  const WorkLayout wl = work_layout(grid, t.n_slots);
  char* wb = static_cast<char*>(work);
  itk::ScanParams prm;
  prm.units = t.units;
  prm.n_units = static_cast<int32_t>(t.n_units);
  prm.top_k = L.top_k;
  prm.ticket = t.tickets;
  prm.status = t.status;
  prm.w = w;
  prm.cand = reinterpret_cast<unsigned long long*>(wb + wl.cand_off);
  prm.store = reinterpret_cast<unsigned long long*>(wb + wl.store_off);
  prm.counts = reinterpret_cast<uint32_t*>(wb + wl.counts_off);
  prm.static_schedule = hooks.static_schedule ? 1 : 0;
  prm.withhold_first_tile = hooks.withhold_timeout ? 1 : 0;
  prm.wait_limit = hooks.withhold_timeout ? kShortWaitCycles : itk::kWaitLimitCycles;
  // A test hook asks for a launch the runtime must refuse: a dynamic shared-memory request
  // above the device limit is rejected at launch time and no work reaches the GPU.
  const size_t smem = hooks.force_launch_failure ? size_t(1) << 30 : itk::kSmemBytes;
  cudaError_t e = launch_dependent(itk::indexer_topk_scan_kernel, grid, itk::kNumThreads, smem, stream, qmap, kmap, prm);
  if (e != cudaSuccess) return cuda_fail(e, "scan launch");
  if (split_event) {
    e = cudaEventRecord(split_event, stream);
    if (e != cudaSuccess) return cuda_fail(e, "recording the split event");
  }
  if (t.n_merges > 0) {
    itk::MergeParams mp;
    mp.merges = t.merges;
    mp.n_merges = static_cast<int32_t>(t.n_merges);
    mp.top_k = L.top_k;
    mp.store = prm.store;
    mp.counts = prm.counts;
    mp.status = t.status;
    mp.out_ids = ids;
    mp.out_scores = scores;
    mp.key_id_base = static_cast<uint32_t>(L.key_id_base);
    e = launch_dependent(itk::indexer_topk_merge_kernel, static_cast<int>(t.n_merges) * itk::kMergeCluster,
                         itk::kMergeThreads, itk::kMergeSmemBytes, stream, mp);
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  }
  if (!t.select) return ITK_OK;
  itk::SelectParams sp;
  sp.item_rows = t.item_rows;
  sp.n_items = static_cast<int32_t>(t.n_slots);
  sp.top_k = L.top_k;
  sp.ticket = t.tickets + 1;
  sp.status = t.status;
  sp.store = prm.store;
  sp.counts = prm.counts;
  sp.out_ids = ids;
  sp.out_scores = scores;
  sp.key_id_base = static_cast<uint32_t>(L.key_id_base);
  const size_t items = t.n_slots;
  const int sel_grid = static_cast<int>(
      std::max<size_t>(1, std::min<size_t>(static_cast<size_t>(sm_count), (items + itk::kSelGroups - 1) / itk::kSelGroups)));
  e = launch_dependent(itk::indexer_topk_select_kernel, sel_grid, itk::kSelThreads, kSelSmemLaunch, stream, sp);
  if (e != cudaSuccess) return cuda_fail(e, "selection launch");
  return ITK_OK;
}

// Waits for `stream`, reads the device status word at d_status and clears it; maps a
// nonzero word to ITK_ERR_INTERNAL or ITK_ERR_DEVICE_TIMEOUT (and sets *dirty). Allocates
// nothing: the word goes to a host stack variable through a pageable copy.
int read_status_word(uint32_t* d_status, cudaStream_t s, bool* dirty) {
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, d_status, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (word == 0) return ITK_OK;
  e = cudaMemsetAsync(d_status, 0, sizeof word, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (dirty) *dirty = true;
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
  if ((word & 0xFFu) == itk::kStatusInternal)
    return fail(ITK_ERR_INTERNAL, "device status word 0x%x (check %u failed)", word, (word >> 8) & 0xFFu);
  return fail(ITK_ERR_DEVICE_TIMEOUT, "device status word 0x%x (wait in role %u gave up)", word, (word >> 8) & 0xFFu);
}

// debug_inject 5 with no plan: the next call without a plan (eager or no-allocation) on
// this thread runs with the withheld key tile and short wait limit.
thread_local bool g_planless_timeout_next = false;

}  // namespace

struct itk_plan_s {
  Layout layout;
  DeviceInfo dev;
  int grid = 0;
  void* block = nullptr;  // device: [units | ticket | status]
  BlockLayout bl;
  bool ticket_dirty = false;
  bool fail_next_launch = false;  // test hook
  bool timeout_next_run = false;  // test hook (debug_inject 5)
  cudaEvent_t split_event = nullptr;  // recorded between the two launches when set
  bool static_schedule = false;       // benchmark aid (debug_inject 3 / 4)
};

extern "C" {

const char* indexer_topk_version(void) { return "0.1.0"; }

const char* indexer_topk_last_error(void) { return g_last_error; }

const char* indexer_topk_status_string(int status) {
  switch (status) {
    case ITK_OK: return "ok";
    case ITK_ERR_INVALID_ARGUMENT: return "invalid argument";
    case ITK_ERR_UNSUPPORTED: return "unsupported shape or top_k";
    case ITK_ERR_INVALID_SEQLENS: return "invalid cu_seqlens";
    case ITK_ERR_INVALID_OFFSETS: return "invalid causal offsets";
    case ITK_ERR_NULL_POINTER: return "null pointer";
    case ITK_ERR_MISALIGNED: return "misaligned buffer";
    case ITK_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case ITK_ERR_CUDA: return "CUDA error";
    case ITK_ERR_NO_DEVICE: return "no supported CUDA device";
    case ITK_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case ITK_ERR_INTERNAL: return "internal device check failed";
    default: return "unknown status";
  }
}

int indexer_topk_validate(const itk_desc* desc) {
  Layout L;
  return build_layout(desc, &L);
}

int64_t indexer_topk_num_units(const itk_desc* desc) {
  Layout L;
  const int rc = build_layout(desc, &L);
  return rc ? -static_cast<int64_t>(rc) : static_cast<int64_t>(L.units.size());
}

int64_t indexer_topk_unit_table(const itk_desc* desc, int32_t* units, int64_t capacity) {
  Layout L;
  const int rc = build_layout(desc, &L);
  if (rc) return -static_cast<int64_t>(rc);
  const int64_t n = static_cast<int64_t>(L.units.size());
  if (units && capacity > 0) {
    const int64_t m = std::min(n, capacity);
    for (int64_t i = 0; i < m; ++i) {
      units[6 * i + 0] = L.units[i].q_row0;
      units[6 * i + 1] = L.units[i].nq;
      units[6 * i + 2] = L.units[i].key_row0;
      units[6 * i + 3] = L.units[i].pos0;
      units[6 * i + 4] = L.units[i].tile0;
      units[6 * i + 5] = L.units[i].tile1;
    }
  }
  return n;
}

int indexer_topk_prepare(const itk_desc* desc, void* stream, itk_plan* out_plan) {
  if (!out_plan) return fail(ITK_ERR_INVALID_ARGUMENT, "out_plan is NULL");
  *out_plan = nullptr;
  itk_plan_s* plan = new (std::nothrow) itk_plan_s();
  if (!plan) return fail(ITK_ERR_INVALID_ARGUMENT, "out of host memory");
  int rc = build_layout(desc, &plan->layout);
  if (!rc) rc = query_device(&plan->dev);
  if (rc) {
    delete plan;
    return rc;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t n_units = plan->layout.units.size();
  plan->grid = grid_for(n_units, plan->dev.sm_count);
  plan->bl = block_layout(plan->layout);
  cudaError_t e = cudaMalloc(&plan->block, plan->bl.bytes);
  if (e != cudaSuccess) {
    delete plan;
    return cuda_fail(e, "cudaMalloc of the plan block");
  }
  // Tables plus zeroed ticket blocks and status word in one copy. The runtime passes a
  // pageable source through a staging buffer, so the image may be freed right away.
  const std::vector<unsigned char> image = block_image(plan->layout, plan->bl);
  e = cudaMemcpyAsync(plan->block, image.data(), image.size(), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) {
    cudaFree(plan->block);
    delete plan;
    return cuda_fail(e, "uploading the plan block");
  }
  *out_plan = plan;
  return ITK_OK;
}

size_t indexer_topk_workspace_bytes(itk_plan plan) {
  if (!plan) return 0;
  return plan->grid > 0 ? work_layout(plan->grid, plan->layout.n_slots()).bytes : 0;
}

int indexer_topk_run(itk_plan plan, const void* q, const void* k, const float* w, int32_t* out_ids,
                     float* out_scores, void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan) return fail(ITK_ERR_INVALID_ARGUMENT, "plan is NULL");
  const Layout& L = plan->layout;
  if (L.T == 0) return ITK_OK;
  int rc = check_run_buffers(L, q, k, w, out_ids, out_scores);
  if (rc) return rc;
  const size_t need = indexer_topk_workspace_bytes(plan);
  if (workspace_bytes < need) return fail(ITK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, need);
  if (need && !workspace) return fail(ITK_ERR_NULL_POINTER, "workspace is NULL");
  if (!aligned(workspace, 16)) return fail(ITK_ERR_MISALIGNED, "workspace must be 16-byte aligned");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* blk = static_cast<char*>(plan->block);
  TicketBlock* ticket = reinterpret_cast<TicketBlock*>(blk + plan->bl.ticket_off);
  if (plan->ticket_dirty) {
    cudaError_t e = cudaMemsetAsync(ticket, 0, 2 * sizeof(TicketBlock), s);
    if (e != cudaSuccess) return cuda_fail(e, "zeroing the ticket blocks");
  }
  RunHooks hooks;
  hooks.force_launch_failure = plan->fail_next_launch;
  hooks.static_schedule = plan->static_schedule;
  hooks.withhold_timeout = plan->timeout_next_run;
  plan->fail_next_launch = false;
  plan->timeout_next_run = false;
  rc = launch_run(L, plan->grid, plan->dev.sm_count, block_tables(L, plan->bl, blk), q, k, w, out_ids, out_scores,
                  workspace, s, hooks, plan->split_event);
  plan->ticket_dirty = (rc != ITK_OK);
  return rc;
}

size_t indexer_topk_eager_workspace_bytes(const itk_desc* desc) {
  Layout L;
  if (build_layout(desc, &L)) return 0;
  DeviceInfo dev;
  if (query_device(&dev)) return 0;
  const int grid = grid_for(L.units.size(), dev.sm_count);
  return work_layout(grid, L.n_slots()).bytes + block_layout(L).bytes;
}

int indexer_topk_eager(const itk_desc* desc, const void* q, const void* k, const float* w, int32_t* out_ids,
                       float* out_scores, void* workspace, size_t workspace_bytes, void* stream) {
  Layout L;
  int rc = build_layout(desc, &L);
  if (rc) return rc;
  if (L.T == 0) return ITK_OK;
  DeviceInfo dev;
  rc = query_device(&dev);
  if (rc) return rc;
  rc = check_run_buffers(L, q, k, w, out_ids, out_scores);
  if (rc) return rc;
  const int grid = grid_for(L.units.size(), dev.sm_count);
  const size_t cand = work_layout(grid, L.n_slots()).bytes;
  const BlockLayout bl = block_layout(L);
  if (!workspace) return fail(ITK_ERR_NULL_POINTER, "workspace is NULL");
  if (workspace_bytes < cand + bl.bytes)
    return fail(ITK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, cand + bl.bytes);
  if (!aligned(workspace, 256)) return fail(ITK_ERR_MISALIGNED, "eager workspace must be 256-byte aligned");
  // Tables, zeroed ticket blocks and status word go up in one copy.
  const std::vector<unsigned char> host = block_image(L, bl);
  char* blk = static_cast<char*>(workspace) + cand;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(blk, host.data(), bl.bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "uploading the eager unit table");
  RunHooks hooks;
  hooks.withhold_timeout = g_planless_timeout_next;
  g_planless_timeout_next = false;
  return launch_run(L, grid, dev.sm_count, block_tables(L, bl, blk), q, k, w, out_ids, out_scores, workspace, s, hooks);
}

int indexer_topk_eager_device_status(const itk_desc* desc, void* workspace, size_t workspace_bytes, void* stream) {
  Layout L;
  int rc = build_layout(desc, &L);
  if (rc) return rc;
  if (L.T == 0) return ITK_OK;  // such a call ran nothing
  DeviceInfo dev;
  rc = query_device(&dev);
  if (rc) return rc;
  if (!workspace) return fail(ITK_ERR_NULL_POINTER, "workspace is NULL");
  const size_t cand = work_layout(grid_for(L.units.size(), dev.sm_count), L.n_slots()).bytes;
  const BlockLayout bl = block_layout(L);
  if (workspace_bytes < cand + bl.bytes)
    return fail(ITK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, cand + bl.bytes);
  return read_status_word(reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + cand + bl.status_off),
                          static_cast<cudaStream_t>(stream), nullptr);
}

void indexer_topk_destroy(itk_plan plan) {
  if (!plan) return;
  if (plan->block) cudaFree(plan->block);
  delete plan;
}

int indexer_topk_device_status(itk_plan plan, void* stream) {
  if (!plan) return fail(ITK_ERR_INVALID_ARGUMENT, "plan is NULL");
  uint32_t* d_status = reinterpret_cast<uint32_t*>(static_cast<char*>(plan->block) + plan->bl.status_off);
  // a run that gave up may have left the ticket blocks nonzero: the next run zeroes them
  return read_status_word(d_status, static_cast<cudaStream_t>(stream), &plan->ticket_dirty);
}

// ---------------------------------------------------------------- test hooks
// Not part of the operation; used by the recovery tests and the benchmark.
//   what = 1: the next run's launch is refused by the runtime (oversized shared-memory
//             request), as after a run that raised while launching.
//   what = 2: write a nonzero value into the plan's two ticket blocks on `stream`, as a
//             run that stopped midway would leave them.
//   what = 3 / 4: fixed units per scan CTA / the ticket again.
//   what = 5: the next run (plan NULL: the next eager or no-allocation call of this thread) has
//             CTA 0 withhold one key-tile load and every wait limited to kShortWaitCycles,
//             so that the bounded waits run out and report a timeout.
int indexer_topk_set_split_event(itk_plan plan, void* event) {
  if (!plan) return fail(ITK_ERR_INVALID_ARGUMENT, "plan is NULL");
  plan->split_event = static_cast<cudaEvent_t>(event);
  return ITK_OK;
}

int indexer_topk_debug_inject(itk_plan plan, int what, void* stream) {
  if (what == 5 && !plan) {
    g_planless_timeout_next = true;
    return ITK_OK;
  }
  if (!plan) return fail(ITK_ERR_INVALID_ARGUMENT, "plan is NULL");
  if (what == 1) {
    plan->fail_next_launch = true;
    return ITK_OK;
  }
  if (what == 2) {
    TicketBlock* t = reinterpret_cast<TicketBlock*>(static_cast<char*>(plan->block) + plan->bl.ticket_off);
    cudaError_t e = cudaMemsetAsync(t, 0x11, 2 * sizeof(TicketBlock), static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ITK_OK : cuda_fail(e, "poisoning the ticket block");
  }
  if (what == 3 || what == 4) {
    plan->static_schedule = (what == 3);
    return ITK_OK;
  }
  if (what == 5) {
    plan->timeout_next_run = true;
    return ITK_OK;
  }
  return fail(ITK_ERR_INVALID_ARGUMENT, "unknown injection %d", what);
}

}  // extern "C"

// ---------------------------------------------------------------- residency holder
// Benchmark aid, not part of the operation: a kernel that keeps n SMs busy, as a kernel
// of another stream would, to show that the scan's ticket grid does not run a second wave
// of work units when some of its CTAs cannot start (flashinfer PR #8691, the side-stream
// table and its opening description, issue #7548). Each holder CTA claims enough shared
// memory that no scan CTA fits beside it, then sleeps in a clock-limited loop.
namespace {

constexpr size_t kHoldSmem = 128 * 1024;
constexpr long long kHoldMaxCycles = 200000000ll;  // about 0.1 s at 2 GHz, whatever is asked

__global__ void itk_hold_kernel(long long cycles) {
  extern __shared__ uint8_t hold_smem[];
  if (threadIdx.x == 0) {
    const long long t0 = clock64();
    while (clock64() - t0 < cycles) __nanosleep(2000);
    hold_smem[0] = 1;
  }
}

}  // namespace

extern "C" int indexer_topk_bench_hold(int n_ctas, int microseconds, void* stream) {
  if (n_ctas < 0 || microseconds < 0) return fail(ITK_ERR_INVALID_ARGUMENT, "negative holder size or time");
  if (n_ctas == 0 || microseconds == 0) return ITK_OK;
  int dev = 0, khz = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
  if (e != cudaSuccess) return cuda_fail(e, "reading the SM clock rate");
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(itk_hold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kHoldSmem));
  });
  if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute (holder)");
  const long long cycles = std::min<long long>(static_cast<long long>(microseconds) * khz / 1000, kHoldMaxCycles);
  itk_hold_kernel<<<n_ctas, 32, kHoldSmem, static_cast<cudaStream_t>(stream)>>>(cycles);
  e = cudaGetLastError();
  return e == cudaSuccess ? ITK_OK : cuda_fail(e, "holder launch");
}

// ---------------------------------------------------------------- no-allocation entry
// For callers that cannot allocate device memory at call time: a serving runtime or a
// framework that has already reserved the device's memory for its own pool (a
// cudaMalloc would fail or fight that pool), or a latency-critical path where an
// allocation -- which can synchronize the device -- is not acceptable. The run's scratch
// (working buffers, candidate store, unit table, ticket blocks, status word) lives in
// this file-scope device array instead of a plan block and a caller workspace. The
// candidate store holds kNoAllocChunkUnits work units, so larger inputs run as several
// scan + selection launch pairs over consecutive ranges of the unit table. Every GPU
// that loads this library holds the array until the process exits.
namespace {

constexpr int kNoAllocMaxCtas = 152;          // CTAs whose working buffers fit
constexpr size_t kNoAllocChunkUnits = 512;    // work units per launch pair (2048 queries)
constexpr int64_t kNoAllocMaxUnits = 65536;   // work units (4 queries each) the unit table holds
// Split queries (and so merges) exist only for descriptors of at most kSplitMaxBlocks
// query blocks, whose at most kSplitUnits + kSplitMaxBlocks units fit one launch pair.
constexpr size_t kNoAllocMaxMerges = static_cast<size_t>(kSplitMaxBlocks) * itk::kQB;
static_assert(kSplitUnits + kSplitMaxBlocks <= static_cast<int>(kNoAllocChunkUnits), "split runs fit one chunk");
constexpr size_t kNoAllocChunkSlots = kNoAllocChunkUnits * itk::kQB;
constexpr size_t kNoAllocWorkBytes = work_layout(kNoAllocMaxCtas, kNoAllocChunkSlots).bytes;
constexpr size_t kNoAllocUnitsOff = kNoAllocWorkBytes;
constexpr size_t kNoAllocItemsOff = kNoAllocUnitsOff + align_up(kNoAllocMaxUnits * sizeof(UnitDesc), 256);
constexpr size_t kNoAllocMergesOff =
    kNoAllocItemsOff + align_up(kNoAllocMaxUnits * itk::kQB * sizeof(int32_t), 256);
constexpr size_t kNoAllocTicketOff = kNoAllocMergesOff + align_up(kNoAllocMaxMerges * sizeof(itk::MergeDesc), 256);
constexpr size_t kNoAllocStatusOff = kNoAllocTicketOff + 256;
constexpr size_t kNoAllocBytes = kNoAllocStatusOff + 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device
// (the host-side symbol is only a stand-in and must never reach a kernel).
int noalloc_scratch(int device, unsigned char** out) {
  if (device < 0 || device >= kNoAllocMaxDevices)
    return fail(ITK_ERR_NO_DEVICE, "device ordinal %d out of range", device);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[device]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static scratch");
    g_noalloc_ptr[device] = ptr;
  }
  *out = static_cast<unsigned char*>(g_noalloc_ptr[device]);
  return ITK_OK;
}

}  // namespace

extern "C" {

size_t indexer_topk_noalloc_scratch_bytes(void) { return kNoAllocBytes; }

int indexer_topk_run_noalloc(const itk_desc* desc, const void* q, const void* k, const float* w, int32_t* out_ids,
                             float* out_scores, void* stream) {
  Layout L;
  int rc = build_layout(desc, &L);
  if (rc) return rc;
  if (L.T == 0) return ITK_OK;
  if (static_cast<int64_t>(L.units.size()) > kNoAllocMaxUnits)
    return fail(ITK_ERR_UNSUPPORTED, "%zu work units exceed the static scratch limit of %lld (about %lld queries)",
                L.units.size(), static_cast<long long>(kNoAllocMaxUnits),
                static_cast<long long>(kNoAllocMaxUnits) * itk::kQB);
  DeviceInfo dev;
  rc = query_device(&dev);
  if (rc) return rc;
  rc = check_run_buffers(L, q, k, w, out_ids, out_scores);
  if (rc) return rc;
  unsigned char* scratch = nullptr;
  rc = noalloc_scratch(dev.device, &scratch);
  if (rc) return rc;
  RunHooks hooks;
  hooks.withhold_timeout = g_planless_timeout_next;
  g_planless_timeout_next = false;
  // The tables, then the ticket blocks and status word, which must start at zero: three
  // copies and one memset on the call's stream (the array keeps the previous call's
  // contents otherwise). Working buffers, store and counts need no clearing.
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(scratch + kNoAllocUnitsOff, L.units.data(), L.units.size() * sizeof(UnitDesc),
                                  cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(scratch + kNoAllocItemsOff, L.item_rows.data(), L.item_rows.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && !L.merges.empty())
    e = cudaMemcpyAsync(scratch + kNoAllocMergesOff, L.merges.data(), L.merges.size() * sizeof(itk::MergeDesc),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch + kNoAllocTicketOff, 0, kNoAllocBytes - kNoAllocTicketOff, s);
  if (e != cudaSuccess) return cuda_fail(e, "staging the tables into the static scratch");
  for (size_t u0 = 0; u0 < L.units.size(); u0 += kNoAllocChunkUnits) {
    const size_t n = std::min(kNoAllocChunkUnits, L.units.size() - u0);
    const bool whole = (u0 == 0 && n == L.units.size());  // merges only ever occur then
    RunTables t;
    t.units = reinterpret_cast<const UnitDesc*>(scratch + kNoAllocUnitsOff) + u0;
    t.n_units = n;
    t.item_rows = reinterpret_cast<const int32_t*>(scratch + kNoAllocItemsOff) + u0 * itk::kQB;
    t.n_slots = n * itk::kQB;
    t.merges = reinterpret_cast<const itk::MergeDesc*>(scratch + kNoAllocMergesOff);
    t.n_merges = whole ? L.merges.size() : 0;
    t.select = !whole || L.select_rows > 0;
    t.tickets = reinterpret_cast<TicketBlock*>(scratch + kNoAllocTicketOff);
    t.status = reinterpret_cast<uint32_t*>(scratch + kNoAllocStatusOff);
    // work_layout(grid, t.n_slots) of a chunk fits inside work_layout(kNoAllocMaxCtas, kNoAllocChunkSlots)
    const int grid = std::min(grid_for(n, dev.sm_count), kNoAllocMaxCtas);
    rc = launch_run(L, grid, std::min(dev.sm_count, kNoAllocMaxCtas), t, q, k, w, out_ids, out_scores, scratch, s,
                    hooks);
    if (rc) return rc;
    hooks.withhold_timeout = false;  // the hook covers the first launch pair
  }
  return ITK_OK;
}

int indexer_topk_noalloc_device_status(void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ITK_ERR_NO_DEVICE, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(ITK_ERR_NO_DEVICE, "device ordinal %d out of range", dev);
  unsigned char* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    scratch = static_cast<unsigned char*>(g_noalloc_ptr[dev]);
  }
  if (!scratch) return ITK_OK;  // no call has run on this device
  return read_status_word(reinterpret_cast<uint32_t*>(scratch + kNoAllocStatusOff), static_cast<cudaStream_t>(stream),
                          nullptr);
}

}  // extern "C"
