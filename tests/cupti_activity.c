/*
 * Test helper: records the device activities (kernels, memory copies, memsets) that a
 * process issues between dtk_activity_start() and dtk_activity_stop(), through the CUPTI
 * activity API. The launch-count tests use it to check how many kernels, copies and
 * memsets one call of the library puts on the GPU, and in which order.
 */
#include <cupti.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#define DTK_MAX_RECORDS 4096
#define DTK_NAME_LEN 160

typedef struct {
  uint64_t start;
  int kind; /* 0 kernel, 1 memcpy, 2 memset */
  char name[DTK_NAME_LEN];
} dtk_record;

static dtk_record g_records[DTK_MAX_RECORDS];
static int g_count = 0;
static int g_dropped = 0;

static void CUPTIAPI buffer_requested(uint8_t** buffer, size_t* size, size_t* max_records) {
  *size = (size_t)1 << 20;
  *buffer = (uint8_t*)aligned_alloc(8, *size);
  *max_records = 0;
}

static void add(uint64_t start, int kind, const char* name) {
  if (g_count >= DTK_MAX_RECORDS) {
    ++g_dropped;
    return;
  }
  dtk_record* r = &g_records[g_count++];
  r->start = start;
  r->kind = kind;
  snprintf(r->name, DTK_NAME_LEN, "%s", name ? name : "?");
}

static void CUPTIAPI buffer_completed(CUcontext ctx, uint32_t stream, uint8_t* buffer, size_t size, size_t valid) {
  (void)ctx;
  (void)stream;
  (void)size;
  CUpti_Activity* rec = NULL;
  while (cuptiActivityGetNextRecord(buffer, valid, &rec) == CUPTI_SUCCESS) {
    if (rec->kind == CUPTI_ACTIVITY_KIND_CONCURRENT_KERNEL || rec->kind == CUPTI_ACTIVITY_KIND_KERNEL) {
      const CUpti_ActivityKernel10* k = (const CUpti_ActivityKernel10*)rec;
      add(k->start, 0, k->name);
    } else if (rec->kind == CUPTI_ACTIVITY_KIND_MEMCPY) {
      const CUpti_ActivityMemcpy6* m = (const CUpti_ActivityMemcpy6*)rec;
      char name[64];
      snprintf(name, sizeof name, "memcpy (copy kind %u, %llu bytes)", (unsigned)m->copyKind,
               (unsigned long long)m->bytes);
      add(m->start, 1, name);
    } else if (rec->kind == CUPTI_ACTIVITY_KIND_MEMSET) {
      const CUpti_ActivityMemset4* m = (const CUpti_ActivityMemset4*)rec;
      char name[64];
      snprintf(name, sizeof name, "memset (%llu bytes)", (unsigned long long)m->bytes);
      add(m->start, 2, name);
    }
  }
  free(buffer);
}

/* Start recording (clears earlier records). Returns 0 or a CUPTI error code. */
int dtk_activity_start(void) {
  g_count = 0;
  g_dropped = 0;
  CUptiResult r = cuptiActivityRegisterCallbacks(buffer_requested, buffer_completed);
  if (r == CUPTI_SUCCESS) r = cuptiActivityEnable(CUPTI_ACTIVITY_KIND_CONCURRENT_KERNEL);
  if (r == CUPTI_SUCCESS) r = cuptiActivityEnable(CUPTI_ACTIVITY_KIND_MEMCPY);
  if (r == CUPTI_SUCCESS) r = cuptiActivityEnable(CUPTI_ACTIVITY_KIND_MEMSET);
  return (int)r;
}

/* Stop recording and flush; returns the number of records (or -1 if some were dropped). */
int dtk_activity_stop(void) {
  cuptiActivityFlushAll(1);
  cuptiActivityDisable(CUPTI_ACTIVITY_KIND_CONCURRENT_KERNEL);
  cuptiActivityDisable(CUPTI_ACTIVITY_KIND_MEMCPY);
  cuptiActivityDisable(CUPTI_ACTIVITY_KIND_MEMSET);
  cuptiActivityFlushAll(1);
  return g_dropped ? -1 : g_count;
}

/* Record i: its start time (ns), kind (0 kernel, 1 memcpy, 2 memset) and name. */
int dtk_activity_get(int i, uint64_t* start, int* kind, char* name, int cap) {
  if (i < 0 || i >= g_count || cap <= 0) return -1;
  *start = g_records[i].start;
  *kind = g_records[i].kind;
  snprintf(name, (size_t)cap, "%s", g_records[i].name);
  return 0;
}
