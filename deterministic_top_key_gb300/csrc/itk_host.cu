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
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
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

// Validated copy of a descriptor plus its unit table.
struct Layout {
  int32_t T = 0, Tkv = 0, top_k = 0, B = 0;
  std::vector<UnitDesc> units;  // ticket order: most key tiles first
};

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
      int64_t order;
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
        it.order = static_cast<int64_t>(items.size());
        items.push_back(it);
      }
    }
    // Longest first: the heaviest units are handed out first so the short ones fill the tail.
    std::stable_sort(items.begin(), items.end(), [](const Item& a, const Item& b) { return a.tiles > b.tiles; });
    L.units.reserve(items.size());
    for (const Item& it : items) L.units.push_back(it.u);
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
// [units | scan ticket | selection ticket | status].
struct BlockLayout {
  size_t units_off = 0, ticket_off = 0, sel_ticket_off = 0, status_off = 0, bytes = 0;
};
BlockLayout block_layout(size_t n_units) {
  BlockLayout b;
  b.units_off = 0;
  b.ticket_off = align_up(n_units * sizeof(UnitDesc), 64);
  b.sel_ticket_off = b.ticket_off + sizeof(TicketBlock);
  b.status_off = b.sel_ticket_off + sizeof(TicketBlock);
  b.bytes = b.status_off + 16;
  return b;
}

// Workspace layout of one run: per-CTA working buffers of the scan, then the candidate
// store (kCap keys per query slot, four slots per unit), then the per-slot counts.
struct WorkLayout {
  size_t cand_off = 0, store_off = 0, counts_off = 0, bytes = 0;
};
constexpr WorkLayout work_layout(int grid, size_t n_units) {
  WorkLayout w;
  w.cand_off = 0;
  w.store_off = align_up(static_cast<size_t>(grid) * itk::candidate_bytes_per_cta(), 256);
  w.counts_off = w.store_off + align_up(n_units * itk::store_bytes_per_unit(), 256);
  w.bytes = w.counts_off + align_up(n_units * itk::kQB * sizeof(uint32_t), 256);
  return w;
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
  });
  if (err != cudaSuccess) return cuda_fail(err, "cudaFuncSetAttribute");
  return ITK_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_run_buffers(const Layout& L, const void* q, const void* k, const float* w, int32_t* ids, float* scores) {
  if (!q || !k || !w || !ids || !scores) return fail(ITK_ERR_NULL_POINTER, "q, k, w, out_ids or out_scores is NULL");
  if (!aligned(q, 16) || !aligned(k, 16)) return fail(ITK_ERR_MISALIGNED, "q and k must be 16-byte aligned");
  if (!aligned(w, 4) || !aligned(ids, 4) || !aligned(scores, 4))
    return fail(ITK_ERR_MISALIGNED, "w, out_ids and out_scores must be 4-byte aligned");
  (void)L;
  return ITK_OK;
}

// Encode maps and launch the scan over units [0, n_units) of d_units, then the selection
// of the same units' queries. d_ticket points at two adjacent ticket blocks (scan,
// selection); `work` is laid out by work_layout(grid, n_units).
int launch_run(const Layout& L, int grid, int sm_count, const UnitDesc* d_units, size_t n_units, TicketBlock* d_ticket,
               uint32_t* d_status, const void* q, const void* k, const float* w, int32_t* ids, float* scores,
               void* work, cudaStream_t stream, bool force_launch_failure, cudaEvent_t split_event = nullptr) {
  CUtensorMap qmap, kmap;
  int rc = encode_rows(&qmap, q, static_cast<uint64_t>(L.T) * itk::kHeads, itk::kN);
  if (rc) return rc;
  rc = encode_rows(&kmap, k, static_cast<uint64_t>(std::max(L.Tkv, 1)), itk::kBlockKeys);
  if (rc) return rc;
  rc = ensure_kernel_attributes();
  if (rc) return rc;
  const WorkLayout wl = work_layout(grid, n_units);
  char* wb = static_cast<char*>(work);
  itk::ScanParams prm;
  prm.units = d_units;
  prm.n_units = static_cast<int32_t>(n_units);
  prm.top_k = L.top_k;
  prm.ticket = d_ticket;
  prm.status = d_status;
  prm.w = w;
  prm.cand = reinterpret_cast<unsigned long long*>(wb + wl.cand_off);
  prm.store = reinterpret_cast<unsigned long long*>(wb + wl.store_off);
  prm.counts = reinterpret_cast<uint32_t*>(wb + wl.counts_off);
  // A test hook asks for a launch the runtime must refuse: a dynamic shared-memory request
  // above the device limit is rejected at launch time and no work reaches the GPU.
  const size_t smem = force_launch_failure ? size_t(1) << 30 : itk::kSmemBytes;
  itk::indexer_topk_scan_kernel<<<grid, itk::kNumThreads, smem, stream>>>(qmap, kmap, prm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "scan launch");
  if (split_event) {
    e = cudaEventRecord(split_event, stream);
    if (e != cudaSuccess) return cuda_fail(e, "recording the split event");
  }
  itk::SelectParams sp;
  sp.units = d_units;
  sp.n_units = static_cast<int32_t>(n_units);
  sp.top_k = L.top_k;
  sp.ticket = d_ticket + 1;
  sp.status = d_status;
  sp.store = prm.store;
  sp.counts = prm.counts;
  sp.out_ids = ids;
  sp.out_scores = scores;
  const size_t items = n_units * itk::kQB;
  const int sel_grid = static_cast<int>(
      std::max<size_t>(1, std::min<size_t>(static_cast<size_t>(sm_count), (items + itk::kSelGroups - 1) / itk::kSelGroups)));
  itk::indexer_topk_select_kernel<<<sel_grid, itk::kSelThreads, kSelSmemLaunch, stream>>>(sp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "selection launch");
  return ITK_OK;
}

}  // namespace

struct itk_plan_s {
  Layout layout;
  DeviceInfo dev;
  int grid = 0;
  void* block = nullptr;  // device: [units | ticket | status]
  BlockLayout bl;
  bool ticket_dirty = false;
  bool fail_next_launch = false;  // test hook
  cudaEvent_t split_event = nullptr;  // recorded between the two launches when set
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
      units[4 * i + 0] = L.units[i].q_row0;
      units[4 * i + 1] = L.units[i].nq;
      units[4 * i + 2] = L.units[i].key_row0;
      units[4 * i + 3] = L.units[i].pos0;
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
  plan->bl = block_layout(n_units);
  cudaError_t e = cudaMalloc(&plan->block, plan->bl.bytes);
  if (e != cudaSuccess) {
    delete plan;
    return cuda_fail(e, "cudaMalloc of the plan block");
  }
  char* blk = static_cast<char*>(plan->block);
  if (n_units)
    e = cudaMemcpyAsync(blk + plan->bl.units_off, plan->layout.units.data(), n_units * sizeof(UnitDesc),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(blk + plan->bl.ticket_off, 0, plan->bl.bytes - plan->bl.ticket_off, s);
  if (e != cudaSuccess) {
    cudaFree(plan->block);
    delete plan;
    return cuda_fail(e, "uploading the plan block");
  }
  // The host copy of the unit table is passed by the runtime through a staging buffer, so
  // the vector may be read again or freed right away.
  *out_plan = plan;
  return ITK_OK;
}

size_t indexer_topk_workspace_bytes(itk_plan plan) {
  if (!plan) return 0;
  return plan->grid > 0 ? work_layout(plan->grid, plan->layout.units.size()).bytes : 0;
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
  const bool inject = plan->fail_next_launch;
  plan->fail_next_launch = false;
  rc = launch_run(L, plan->grid, plan->dev.sm_count, reinterpret_cast<const UnitDesc*>(blk + plan->bl.units_off),
                  L.units.size(), ticket, reinterpret_cast<uint32_t*>(blk + plan->bl.status_off), q, k, w, out_ids,
                  out_scores, workspace, s, inject, plan->split_event);
  plan->ticket_dirty = (rc != ITK_OK);
  return rc;
}

size_t indexer_topk_eager_workspace_bytes(const itk_desc* desc) {
  Layout L;
  if (build_layout(desc, &L)) return 0;
  DeviceInfo dev;
  if (query_device(&dev)) return 0;
  const int grid = grid_for(L.units.size(), dev.sm_count);
  return work_layout(grid, L.units.size()).bytes + block_layout(L.units.size()).bytes;
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
  const size_t cand = work_layout(grid, L.units.size()).bytes;
  const BlockLayout bl = block_layout(L.units.size());
  if (!workspace) return fail(ITK_ERR_NULL_POINTER, "workspace is NULL");
  if (workspace_bytes < cand + bl.bytes)
    return fail(ITK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, cand + bl.bytes);
  if (!aligned(workspace, 256)) return fail(ITK_ERR_MISALIGNED, "eager workspace must be 256-byte aligned");
  // Unit table, zeroed ticket block and status word go up in one copy.
  std::vector<unsigned char> host(bl.bytes, 0);
  std::memcpy(host.data() + bl.units_off, L.units.data(), L.units.size() * sizeof(UnitDesc));
  char* blk = static_cast<char*>(workspace) + cand;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(blk, host.data(), bl.bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "uploading the eager unit table");
  return launch_run(L, grid, dev.sm_count, reinterpret_cast<const UnitDesc*>(blk + bl.units_off), L.units.size(),
                    reinterpret_cast<TicketBlock*>(blk + bl.ticket_off),
                    reinterpret_cast<uint32_t*>(blk + bl.status_off), q, k, w, out_ids, out_scores, workspace, s,
                    false);
}

void indexer_topk_destroy(itk_plan plan) {
  if (!plan) return;
  if (plan->block) cudaFree(plan->block);
  delete plan;
}

int indexer_topk_device_status(itk_plan plan, void* stream) {
  if (!plan) return fail(ITK_ERR_INVALID_ARGUMENT, "plan is NULL");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  uint32_t* d_status = reinterpret_cast<uint32_t*>(static_cast<char*>(plan->block) + plan->bl.status_off);
  cudaError_t e = cudaMemcpyAsync(&word, d_status, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (word == 0) return ITK_OK;
  e = cudaMemsetAsync(d_status, 0, sizeof word, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  plan->ticket_dirty = true;  // a run that gave up may have left the ticket blocks nonzero
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
  if ((word & 0xFFu) == itk::kStatusInternal)
    return fail(ITK_ERR_INTERNAL, "device status word 0x%x (check %u failed)", word, (word >> 8) & 0xFFu);
  return fail(ITK_ERR_DEVICE_TIMEOUT, "device status word 0x%x (wait in role %u gave up)", word, (word >> 8) & 0xFFu);
}

// ---------------------------------------------------------------- test hooks
// Not part of the operation; used by the host-side recovery tests.
//   what = 1: the next run's launch is refused by the runtime (oversized shared-memory
//             request), as after a run that raised while launching.
//   what = 2: write a nonzero value into the plan's two ticket blocks on `stream`, as a
//             run that stopped midway would leave them.
int indexer_topk_set_split_event(itk_plan plan, void* event) {
  if (!plan) return fail(ITK_ERR_INVALID_ARGUMENT, "plan is NULL");
  plan->split_event = static_cast<cudaEvent_t>(event);
  return ITK_OK;
}

int indexer_topk_debug_inject(itk_plan plan, int what, void* stream) {
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
  return fail(ITK_ERR_INVALID_ARGUMENT, "unknown injection %d", what);
}

}  // extern "C"

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
constexpr size_t kNoAllocWorkBytes = work_layout(kNoAllocMaxCtas, kNoAllocChunkUnits).bytes;
constexpr size_t kNoAllocUnitsOff = kNoAllocWorkBytes;
constexpr size_t kNoAllocTicketOff = kNoAllocUnitsOff + kNoAllocMaxUnits * sizeof(UnitDesc);
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
  // Unit table, then the ticket blocks and status word, which must start at zero: one
  // copy and one memset on the call's stream (the array keeps the previous call's
  // contents otherwise). Working buffers, store and counts need no clearing.
  const size_t unit_bytes = L.units.size() * sizeof(UnitDesc);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(scratch + kNoAllocUnitsOff, L.units.data(), unit_bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch + kNoAllocTicketOff, 0, kNoAllocBytes - kNoAllocTicketOff, s);
  if (e != cudaSuccess) return cuda_fail(e, "staging the unit table into the static scratch");
  const UnitDesc* d_units = reinterpret_cast<const UnitDesc*>(scratch + kNoAllocUnitsOff);
  for (size_t u0 = 0; u0 < L.units.size(); u0 += kNoAllocChunkUnits) {
    const size_t n = std::min(kNoAllocChunkUnits, L.units.size() - u0);
    // work_layout(grid, n) of a chunk fits inside work_layout(kNoAllocMaxCtas, kNoAllocChunkUnits)
    const int grid = std::min(grid_for(n, dev.sm_count), kNoAllocMaxCtas);
    rc = launch_run(L, grid, std::min(dev.sm_count, kNoAllocMaxCtas), d_units + u0, n,
                    reinterpret_cast<TicketBlock*>(scratch + kNoAllocTicketOff),
                    reinterpret_cast<uint32_t*>(scratch + kNoAllocStatusOff), q, k, w, out_ids, out_scores,
                    scratch, s, false);
    if (rc) return rc;
  }
  return ITK_OK;
}

}  // extern "C"
