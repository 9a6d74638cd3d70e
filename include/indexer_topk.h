/*
 * indexer_topk.h -- C ABI of the GB300 (sm_103a) deterministic lightning-indexer top-k scan.
 *
 * Operation (flashinfer PR #8691, "perf(cake_dsa_indexer_det): ticket scheduling on
 * sm_107a, no fill kernel in eager entry", opening description and the vendoring note
 * "lightning-indexer scores and deterministic exact top-k"):
 *
 *   For every query row t and every key row s that t may see,
 *       I[t,s] = sum_{h=0}^{H-1} w[t,h] * max(q[t,h,:] . k[s,:], 0)
 *   with BF16 q and k, FP32 w and FP32 scores. Each query returns the top_k key ids and
 *   their scores. Ties go to the larger id. Ids and scores do not depend on how the work
 *   is partitioned or chunked.
 *
 * Visibility (varlen segments, causal): segment b owns query rows [cu_q[b], cu_q[b+1])
 * and key rows [cu_k[b], cu_k[b+1]). Local query i of segment b sits at causal position
 * p = off_b + i and sees the keys at local positions 0..p, i.e. p + 1 keys. off_b is
 * q_causal_offsets[b] when given, else Tk_b - Tq_b (the queries end at the segment's
 * last key). The page makes the offsets optional (commit note on the q_offsets
 * placeholder: a call without q_causal_offsets reads no offsets); the bottom-right
 * default is this library's reading.
 *
 * Output of row t (our reading where the page is silent): k_eff = min(top_k, p + 1)
 * entries sorted by score descending, equal scores by id descending; slots k_eff ..
 * top_k-1 hold id -1 and score -INFINITY. The id of key row s is key_id_base + s
 * (key_id_base = 0: global row indices into k). A score of -0.0 is returned as +0.0.
 *
 * Supported: H == 64, D == 128, 1 <= top_k <= 2048, any number of segments.
 *
 * Prepared-runner contract (same page, commit note "TicketWord ... ABI dsa_indexer_v4" and
 * the review comment on stream ordering of prepared runners): prepare once per shape / segment layout / top_k, then run many
 * times with any buffers. The plan owns its 16-byte ticket blocks (one for the scan, one
 * for the selection), zeroed once at prepare on the prepare stream; every completed run
 * leaves them at zero again, so a run issues no memset. Prepare and run on the same stream, or order the two streams yourself:
 * the zeroing is queued on the prepare stream and nothing orders it before a run on
 * another stream. After a run whose launch failed, the next run zeroes the block on its
 * stream before the scan.
 *
 * Errors: every function returns an ITK_* status (0 = success); no exception, abort or
 * exit crosses this ABI. indexer_topk_last_error() gives a one-line detail of the last
 * failure on the calling thread.
 *
 * Streams are passed as void* and must be a cudaStream_t (NULL = legacy default stream).
 * All device pointers are device (or managed) memory of the current CUDA device. A run's
 * kernels are launched as programmatic dependents of the kernel before them on the
 * stream: their CTAs may start while that kernel finishes, and wait for it to complete
 * (griddepcontrol.wait) before they read any of its results, so stream order holds.
 */
#ifndef DTK_INDEXER_TOPK_H_
#define DTK_INDEXER_TOPK_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ITK_API __attribute__((visibility("default")))
#else
#define ITK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
  ITK_OK = 0,
  ITK_ERR_INVALID_ARGUMENT = 1,   /* null descriptor/plan, negative size, top_k < 1 */
  ITK_ERR_UNSUPPORTED = 2,        /* H != 64, D != 128, top_k > 2048, T*H too large */
  ITK_ERR_INVALID_SEQLENS = 3,    /* cu_seqlens not starting at 0, decreasing, or not ending at T / beyond Tkv */
  ITK_ERR_INVALID_OFFSETS = 4,    /* off_b < 0 or off_b + Tq_b > Tk_b */
  ITK_ERR_NULL_POINTER = 5,       /* a required buffer pointer is NULL */
  ITK_ERR_MISALIGNED = 6,         /* q or k not 16-byte aligned, w/outputs not 4-byte aligned */
  ITK_ERR_WORKSPACE_TOO_SMALL = 7,/* workspace_bytes below indexer_topk_workspace_bytes() */
  ITK_ERR_CUDA = 8,               /* a CUDA runtime call or the kernel launch failed */
  ITK_ERR_NO_DEVICE = 9,          /* no CUDA device, or the device is not sm_103 */
  ITK_ERR_DEVICE_TIMEOUT = 10,    /* a bounded wait inside the kernel ran out (see indexer_topk_device_status) */
  ITK_ERR_INTERNAL = 11           /* a kernel found one of its own invariants broken (see indexer_topk_device_status) */
};

typedef struct itk_plan_s* itk_plan;

/* Shape and segment layout; all pointers are host memory, read during prepare only. */
typedef struct {
  int32_t T;                /* query rows */
  int32_t Tkv;              /* key rows */
  int32_t H;                /* heads; must be 64 */
  int32_t D;                /* head dim; must be 128 */
  int32_t top_k;            /* 1..2048 */
  int32_t num_segments;     /* B >= 0 (B == 0 requires T == 0) */
  const int32_t* cu_seqlens_q;     /* [B+1], cu_q[0] = 0, non-decreasing, cu_q[B] = T */
  const int32_t* cu_seqlens_k;     /* [B+1], cu_k[0] = 0, non-decreasing, cu_k[B] <= Tkv */
  const int32_t* q_causal_offsets; /* [B] or NULL (bottom-right: off_b = Tk_b - Tq_b) */
  int32_t key_id_base;      /* added to every returned key id; 0 = global row ids into k.
                               0 <= key_id_base <= 2^31 - 1 - Tkv, so ids stay non-negative
                               int32 and keep their order (ITK_ERR_INVALID_ARGUMENT otherwise) */
} itk_desc;

/*
 * Validate `desc`, build the work-unit table (blocks of 4 consecutive queries of one
 * segment, ordered longest-first), and allocate the plan's device block (unit table,
 * two 16-byte ticket blocks (scan, selection), device status word) on the current device.
 * The ticket blocks and status word are zeroed and the unit table uploaded on `stream` (see the stream-ordering
 * note above). On success *out_plan owns that memory until indexer_topk_destroy().
 * Reference: flashinfer PR #8691, commit note "prepare now decides ... before it issues its
 * first device operation" and commit note "TicketWord ... ABI dsa_indexer_v4" (a runner's
 * own ticket block, zeroed once at prepare).
 */
ITK_API int indexer_topk_prepare(const itk_desc* desc, void* stream, itk_plan* out_plan);

/* Bytes of caller-owned device workspace a run of this plan needs (0 if plan is NULL).
 * The workspace holds the scan's per-CTA working buffers (about 0.56 MB per CTA), the
 * candidate store (32 KB per query slot, four slots per work unit) and its counts; it
 * need not be zeroed and its contents are scratch after a run. Reference: same page, commit note "zero_region ... ABI dsa_indexer_v3" (caller-owned
 * workspace). */
ITK_API size_t indexer_topk_workspace_bytes(itk_plan plan);

/*
 * One scan on `stream`: two kernel launches -- the scan, which leaves each query's
 * candidates (a superset of its top-k, at most 4096 keys) in the workspace, then the
 * selection, which writes the sorted top-k rows. A split-tail descriptor (see
 * indexer_topk_unit_table) launches, in place of the selection, the merge, which selects
 * and writes the rows of its split queries from their chunks' candidates; a descriptor
 * with both split and whole query blocks launches both (three kernels). The scan
 * is always the first launch. No copy and no memset is issued, except one 32-byte memset
 * right after a failed launch. (The page's scan is one kernel; here the selection is a
 * kernel of its own, because run inside the scan kernel its warps took issue slots from
 * the score epilogue.) Arguments:
 *   q          device, BF16 [T,H,D] row-major, 16-byte aligned
 *   k          device, BF16 [Tkv,D] row-major, 16-byte aligned
 *   w          device, FP32 [T,H] row-major
 *   out_ids    device, INT32 [T,top_k] row-major (written)
 *   out_scores device, FP32 [T,top_k] row-major (written)
 *   workspace  device, >= indexer_topk_workspace_bytes(plan) bytes (may be NULL if that is 0)
 * Buffers may change from run to run; a shape change needs a new plan. Runs of one plan
 * must not overlap in time (they share the plan's ticket blocks): issue them on one stream
 * or order them. The call is asynchronous; launch errors are returned, in-kernel wait
 * timeouts are reported by indexer_topk_device_status().
 * Reference: same page, commit note "TicketWord ... ABI dsa_indexer_v4" (ticket word, the
 * recovery after a run that raised while launching).
 */
ITK_API int indexer_topk_run(itk_plan plan, const void* q, const void* k, const float* w, int32_t* out_ids,
                     float* out_scores, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Eager entry: prepare + run + destroy in one call, for a one-shot scan. It allocates no
 * device memory: the unit table and the ticket blocks live at the end of the caller's
 * workspace, which must hold indexer_topk_eager_workspace_bytes(desc) bytes. Device work
 * on `stream`: one host-to-device copy of the unit table with zeroed ticket blocks, then
 * the kernels of indexer_topk_run (the scan first). Reference: same page, "Changes" table row "Runner entry points and
 * validation" (the eager entry uses a one-shot runner) and the TicketWord commit note (the
 * eager entry zeroes its ticket word on the launch stream).
 */
ITK_API size_t indexer_topk_eager_workspace_bytes(const itk_desc* desc);
ITK_API int indexer_topk_eager(const itk_desc* desc, const void* q, const void* k, const float* w, int32_t* out_ids,
                       float* out_scores, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Device status of eager calls that used this workspace: waits for `stream`, then reads and
 * clears the status word that the eager entry keeps in the caller's workspace (at an offset
 * that depends on `desc`, so pass the descriptor and workspace of the call). Returns ITK_OK,
 * ITK_ERR_DEVICE_TIMEOUT or ITK_ERR_INTERNAL as indexer_topk_device_status does; a call that
 * reported either has undefined outputs. Each eager call clears the word before it runs, so
 * read it after the call whose outcome you need. ITK_ERR_WORKSPACE_TOO_SMALL if the
 * workspace cannot be one of `desc`'s.
 */
ITK_API int indexer_topk_eager_device_status(const itk_desc* desc, void* workspace, size_t workspace_bytes,
                                             void* stream);

/* Release the plan's device block (synchronizes nothing; the caller must not destroy a
 * plan while one of its runs may still execute). NULL is ignored. */
ITK_API void indexer_topk_destroy(itk_plan plan);

/*
 * Wait for `stream`, then read the plan's device status word: ITK_OK, or
 * ITK_ERR_DEVICE_TIMEOUT if a bounded wait inside an earlier run of this plan gave up, or
 * ITK_ERR_INTERNAL if a kernel found one of its own invariants broken (outputs of that
 * run are then undefined; the next run re-zeroes the ticket blocks). Reading clears the
 * word.
 */
ITK_API int indexer_topk_device_status(itk_plan plan, void* stream);

/* Validate a descriptor on the host only (no CUDA call). */
ITK_API int indexer_topk_validate(const itk_desc* desc);

/* Number of work units of a descriptor (host only; -status on an invalid descriptor). */
ITK_API int64_t indexer_topk_num_units(const itk_desc* desc);

/*
 * Host-only view of the work-unit table, in ticket order (longest query block first): for
 * each unit {first query row, number of queries (1..4), first key row of the segment,
 * causal position of the first query, first key tile, end key tile} -- the unit scans key
 * tiles [first, end) of 128 keys. A descriptor with at most 64 query blocks (a "split
 * tail") has every block of at least 8 visible key tiles split into consecutive units of
 * about 4 tiles (at most 256 units in all), whose candidates are merged per query into
 * its output row; otherwise a unit covers all visible tiles of its block. Writes min(capacity, n)
 * units to `units` (int32 [capacity][6]) and returns n, or -status on an invalid
 * descriptor. Reference: flashinfer PR #8691, benchmark rows A1-A3 ("split tail: 4
 * queries in one segment").
 */
ITK_API int64_t indexer_topk_unit_table(const itk_desc* desc, int32_t* units, int64_t capacity);

/* Static text for a status code. */
ITK_API const char* indexer_topk_status_string(int status);

/* One-line detail of the last failure on the calling thread ("" if none). */
ITK_API const char* indexer_topk_last_error(void);

/* Library version, e.g. "0.1.0". */
ITK_API const char* indexer_topk_version(void);

/*
 * Scan without any device allocation: same operation, arguments and output as
 * indexer_topk_prepare + indexer_topk_run, but every byte of scratch (working buffers,
 * candidate store, work-unit table, ticket blocks, status word) lives in one static
 * device array of indexer_topk_noalloc_scratch_bytes() bytes (about 159 MB) that every
 * GPU loading this library holds until the process exits. The store holds 512 work units
 * (2048 queries); larger inputs run as one scan + selection launch pair per 512 units. The
 * flashinfer PR page has no counterpart of this entry point: it exists for
 * callers that must not call cudaMalloc at call time -- a serving runtime or framework
 * that has already reserved the device memory for its own pool, or a latency-critical
 * path where an allocation, which can synchronize the device, is not acceptable.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call. The
 *     work-unit table is copied from host memory and the ticket blocks and status word
 *     are zeroed on `stream` before the scan; working buffers and store need no clearing.
 *   - Limit: at most 65536 work units (4 consecutive queries of one segment each, so
 *     about 262144 queries); a larger descriptor is rejected with ITK_ERR_UNSUPPORTED and
 *     a message from indexer_topk_last_error(). The grids are capped at 152 CTAs, because
 *     the static working buffers hold 152 scan CTAs; on a device with more SMs the calls
 *     still run, on 152 of them.
 *   - In-kernel wait timeouts and failed internal checks of a call are reported by
 *     indexer_topk_noalloc_device_status(); the next call clears the word first.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current) -- make that first call before any stream capture.
 *   - Every call shares the one array and leaves its contents behind: calls that overlap
 *     on the GPU race with each other. Issue them on one stream, or order them.
 */
ITK_API int indexer_topk_run_noalloc(const itk_desc* desc, const void* q, const void* k, const float* w,
                                     int32_t* out_ids, float* out_scores, void* stream);

/*
 * Per-kernel timing: from now on, every indexer_topk_run of this plan records `event` (a
 * cudaEvent_t owned by the caller, created on the plan's device) on the run's stream
 * right after the scan launch (before the merge and selection launches), so that events
 * recorded by the caller before and after the run bracket the scan and the rest. NULL stops the recording. Host only;
 * returns ITK_ERR_INVALID_ARGUMENT for a NULL plan. Not part of the operation.
 */
ITK_API int indexer_topk_set_split_event(itk_plan plan, void* event);

/*
 * Benchmark aid, not part of the operation: launch on `stream` a kernel of n_ctas CTAs
 * that each claim 128 KB of shared memory (so no scan CTA fits on the same SM) and stay
 * resident for `microseconds` (capped at about 0.1 s), the way a kernel of another
 * stream holds SMs. Used to show that the ticket grid runs no second wave of work units
 * when some of its CTAs cannot start (flashinfer PR #8691, opening description and the
 * side-stream table). 0 CTAs or 0 us launch nothing.
 */
ITK_API int indexer_topk_bench_hold(int n_ctas, int microseconds, void* stream);

/* Size in bytes of the static scratch array used by indexer_topk_run_noalloc. */
ITK_API size_t indexer_topk_noalloc_scratch_bytes(void);

/*
 * Device status of the last indexer_topk_run_noalloc call on the current device: waits for
 * `stream`, then reads and clears the status word in the static scratch array. ITK_OK, or
 * ITK_ERR_DEVICE_TIMEOUT / ITK_ERR_INTERNAL as indexer_topk_device_status reports them (the
 * outputs of that call are then undefined). Allocates nothing. ITK_OK if no call has run on
 * this device yet.
 */
ITK_API int indexer_topk_noalloc_device_status(void* stream);

/*
 * Test and benchmark hook; not part of the operation.
 *   what = 1: the next indexer_topk_run's launch is refused by the CUDA runtime (an
 *             oversized shared-memory request; no work reaches the GPU), as after a run
 *             that raised while launching. The run returns ITK_ERR_CUDA.
 *   what = 2: write a nonzero pattern into the plan's ticket blocks on `stream` and wait
 *             for it, as a scan that stopped midway would leave them.
 *   what = 3: later runs of the plan give scan CTA b the fixed units b, b + grid, ...
 *             instead of drawing them from the ticket word (the schedule the ticket
 *             replaces; results are the same, but a CTA that cannot start delays its
 *             units). what = 4 restores the ticket.
 */
ITK_API int indexer_topk_debug_inject(itk_plan plan, int what, void* stream);
/*   what = 5: the next run of `plan` -- or, with plan NULL, the next indexer_topk_eager or
 *             indexer_topk_run_noalloc call on this thread -- runs with every in-kernel wait
 *             limited to about 1 ms (2^21 SM clocks), and scan CTA 0 withholds the first
 *             key-tile load of its first unit, so that the waits on it run out as a load
 *             that never arrives would make them: the CTA records ITK_ERR_DEVICE_TIMEOUT in the status word,
 *             waits for its own copies and tensor-core work, frees its tensor memory and
 *             returns. The call itself returns ITK_OK with undefined outputs; the status
 *             readers report the timeout, and the next run is correct again. */

#ifdef __cplusplus
}
#endif

#endif /* DTK_INDEXER_TOPK_H_ */
