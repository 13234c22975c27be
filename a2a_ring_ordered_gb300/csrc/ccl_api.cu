// ccl_api.cu -- the C ABI (include/ccl.h): argument checks, aliasing rules,
// kernel selection, and the literal ring engine's step loop.
//
// Everything here is host code.  Invalid arguments are rejected before any
// CUDA call, so the checks run (and are tested) on machines without a GPU.
#include <stdarg.h>
#include <stdlib.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include <cuda.h>  // driver types only (CUcontext, CUresult); nothing links the driver
#include <nvtx3/nvToolsExt.h>

#include "ccl_internal.h"

namespace ccl {

// An NVTX range named after the entry point, so that a profiler's timeline
// (ncu --nvtx, Nsight Systems) groups each call's kernels under its name.
// Without an attached tool a push/pop costs a few nanoseconds.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define CCL_TRACE() ::ccl::NvtxRange ccl_trace_range_(__func__)

static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int current_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

int first_wave_ctas(const void* kernel) {
  struct Entry {
    const void* kernel;
    int dev, ctas;
  };
  constexpr int kEntries = 64;
  static thread_local Entry cache[kEntries];
  static thread_local int used = 0, next = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  for (int i = 0; i < used; ++i)
    if (cache[i].kernel == kernel && cache[i].dev == dev) return cache[i].ctas;
  int per_sm = 0;
  // every kernel launched through launch_kernel runs 256 threads per CTA
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess) {
    (void)cudaGetLastError();  // not sticky; prefetch is then simply off
    per_sm = 0;
  }
  const Entry e{kernel, dev, per_sm * current_sm_count()};
  if (used < kEntries) {
    cache[used++] = e;
  } else {
    cache[next] = e;
    next = (next + 1) % kEntries;
  }
  return e.ctas;
}

namespace {

thread_local char t_error[512];

void clear_error() { t_error[0] = '\0'; }

ccl_status_t fail(ccl_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_error, sizeof(t_error), fmt, ap);
  va_end(ap);
  return st;
}

ccl_status_t cuda_fail(cudaError_t err, const char* what) {
  return fail(CCL_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(err), cudaGetErrorName(err));
}

constexpr uint64_t kMaxElems = 1ull << 48;

size_t elem_bytes(int dt) {
  switch (dt) {
    case CCL_F32: return 4;
    case CCL_BF16: return 2;
    case CCL_I32: return 4;
    default: return 0;
  }
}

bool valid_op(int op) { return op == CCL_SUM || op == CCL_MAX || op == CCL_MIN; }

void chunk(int p, uint64_t n, int c, uint64_t* off, uint64_t* len) {
  const uint64_t q = n / static_cast<uint64_t>(p), rem = n % static_cast<uint64_t>(p);
  const uint64_t uc = static_cast<uint64_t>(c);
  *off = uc * q + (uc < rem ? uc : rem);
  *len = q + (uc < rem ? 1 : 0);
}

struct Span {
  uintptr_t lo, hi;  // [lo, hi); empty when lo == hi
  bool empty() const { return lo == hi; }
};
Span span(const void* p, uint64_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Span{a, a + bytes};
}
bool overlaps(const Span& a, const Span& b) {
  return !a.empty() && !b.empty() && a.lo < b.hi && b.lo < a.hi;
}

ccl_status_t check_p(int p) {
  if (p < 1 || p > CCL_MAX_RANKS) return fail(CCL_ERR_INVALID_ARG, "p=%d outside 1..%d", p, CCL_MAX_RANKS);
  return CCL_OK;
}

// Per-buffer checks: a buffer that holds bytes needs a non-NULL pointer
// aligned to its element size.
ccl_status_t check_buffers(const char* name, const void* const* ptrs, int p,
                           const uint64_t* bytes, size_t align) {
  if (ptrs == nullptr) return fail(CCL_ERR_INVALID_ARG, "%s is NULL", name);
  for (int r = 0; r < p; ++r) {
    if (bytes[r] == 0) continue;
    if (ptrs[r] == nullptr) return fail(CCL_ERR_INVALID_ARG, "%s[%d] is NULL", name, r);
    if (reinterpret_cast<uintptr_t>(ptrs[r]) % align != 0)
      return fail(CCL_ERR_INVALID_ARG, "%s[%d] is not aligned to its %zu-byte elements", name, r, align);
  }
  return CCL_OK;
}

// Aliasing: outputs must not overlap one another; an output may overlap an
// input only in the one in-place form the call allows (in_place[k] true when
// recv[k] sits exactly where that form puts it relative to send[k]).
ccl_status_t check_aliasing(const Span* in, const Span* out, const bool* in_place, int p) {
  for (int i = 0; i < p; ++i) {
    for (int j = i + 1; j < p; ++j)
      if (overlaps(out[i], out[j]))
        return fail(CCL_ERR_INVALID_ARG, "output buffers %d and %d overlap", i, j);
    for (int j = 0; j < p; ++j) {
      if (!overlaps(out[i], in[j])) continue;
      if (i == j && in_place != nullptr && in_place[i]) continue;
      return fail(CCL_ERR_INVALID_ARG, "output buffer %d overlaps input buffer %d", i, j);
    }
  }
  return CCL_OK;
}

bool all_aligned16(const void* const* a, int p, const void* const* b) {
  for (int r = 0; r < p; ++r) {
    if (reinterpret_cast<uintptr_t>(a[r]) & 15) return false;
    if (reinterpret_cast<uintptr_t>(b[r]) & 15) return false;
  }
  return true;
}

// Shared front half of the reducing calls: argument checks for AR / RS.
// kind: 0 all-reduce, 1 reduce-scatter.
ccl_status_t check_reduce(int kind, const void* const* send, void* const* recv, int p, size_t n,
                          int dt, int op) {
  ccl_status_t st = check_p(p);
  if (st != CCL_OK) return st;
  const size_t e = elem_bytes(dt);
  if (e == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (!valid_op(op)) return fail(CCL_ERR_INVALID_ARG, "unknown op %d", op);
  if (n > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "n=%zu too large", n);
  if (send == nullptr || recv == nullptr) return fail(CCL_ERR_INVALID_ARG, "send or recv array is NULL");
  uint64_t in_bytes[CCL_MAX_RANKS], out_bytes[CCL_MAX_RANKS];
  Span in[CCL_MAX_RANKS], out[CCL_MAX_RANKS];
  bool in_place[CCL_MAX_RANKS];
  for (int r = 0; r < p; ++r) {
    uint64_t off, len;
    chunk(p, n, r, &off, &len);
    in_bytes[r] = n * e;
    out_bytes[r] = (kind == 0 ? n : len) * e;
    in[r] = span(send[r], in_bytes[r]);
    out[r] = span(recv[r], out_bytes[r]);
    const uintptr_t where = reinterpret_cast<uintptr_t>(send[r]) + (kind == 0 ? 0 : off * e);
    in_place[r] = reinterpret_cast<uintptr_t>(recv[r]) == where;
  }
  if ((st = check_buffers("send", send, p, in_bytes, e)) != CCL_OK) return st;
  if ((st = check_buffers("recv", const_cast<const void* const*>(recv), p, out_bytes, e)) != CCL_OK) return st;
  return check_aliasing(in, out, in_place, p);
}

ccl_status_t check_gather(const void* const* send, void* const* recv, int p, size_t n, int dt) {
  ccl_status_t st = check_p(p);
  if (st != CCL_OK) return st;
  const size_t e = elem_bytes(dt);
  if (e == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (n > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "n=%zu too large", n);
  if (send == nullptr || recv == nullptr) return fail(CCL_ERR_INVALID_ARG, "send or recv array is NULL");
  uint64_t in_bytes[CCL_MAX_RANKS], out_bytes[CCL_MAX_RANKS];
  Span in[CCL_MAX_RANKS], out[CCL_MAX_RANKS];
  bool in_place[CCL_MAX_RANKS];
  for (int r = 0; r < p; ++r) {
    uint64_t off, len;
    chunk(p, n, r, &off, &len);
    in_bytes[r] = len * e;
    out_bytes[r] = n * e;
    in[r] = span(send[r], in_bytes[r]);
    out[r] = span(recv[r], out_bytes[r]);
    in_place[r] = reinterpret_cast<uintptr_t>(send[r]) == reinterpret_cast<uintptr_t>(recv[r]) + off * e;
  }
  if ((st = check_buffers("send", send, p, in_bytes, e)) != CCL_OK) return st;
  if ((st = check_buffers("recv", const_cast<const void* const*>(recv), p, out_bytes, e)) != CCL_OK) return st;
  return check_aliasing(in, out, in_place, p);
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

void clear_last_error() { clear_error(); }

ccl_status_t report_error(ccl_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_error, sizeof(t_error), fmt, ap);
  va_end(ap);
  return st;
}

}  // namespace ccl

using namespace ccl;

// ================================================================ utilities
extern "C" int ccl_abi_version(void) { return CCL_ABI_VERSION; }

extern "C" const char* ccl_status_string(ccl_status_t status) {
  switch (status) {
    case CCL_OK: return "CCL_OK";
    case CCL_ERR_INVALID_ARG: return "CCL_ERR_INVALID_ARG: invalid argument";
    case CCL_ERR_UNSUPPORTED: return "CCL_ERR_UNSUPPORTED: not implemented for these arguments";
    case CCL_ERR_CUDA: return "CCL_ERR_CUDA: a CUDA call failed";
    case CCL_ERR_TIMEOUT: return "CCL_ERR_TIMEOUT: a bounded wait gave up";
    default: return "unknown ccl_status_t";
  }
}

extern "C" const char* ccl_last_error(void) { return t_error; }

extern "C" uint64_t ccl_kernel_launch_count(void) {
  return g_launches.load(std::memory_order_relaxed);
}

extern "C" ccl_status_t ccl_device_error_flag(unsigned int* flag, int clear) {
  clear_error();
  if (flag == nullptr) return fail(CCL_ERR_INVALID_ARG, "flag is NULL");
  cudaError_t err = read_device_error(flag, clear != 0);
  if (err != cudaSuccess) return cuda_fail(err, "reading the device error word");
  return CCL_OK;
}

extern "C" ccl_status_t ccl_stream_check(void* stream) {
  clear_error();
  cudaError_t err = cudaStreamSynchronize(as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "synchronizing the stream");
  unsigned int flag = 0;
  if ((err = read_device_error(&flag, true)) != cudaSuccess) return cuda_fail(err, "reading the device error word");
  if (flag != 0)
    return fail(CCL_ERR_TIMEOUT, "a bounded device-side wait ran out (error word %u)", flag);
  return CCL_OK;
}

extern "C" ccl_status_t ccl_selftest_bounded_wait(void* stream) {
  CCL_TRACE();
  clear_error();
  cudaError_t err = launch_bounded_wait_probe(as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "bounded-wait probe launch");
  return CCL_OK;
}

extern "C" ccl_status_t ccl_chunk_bounds(int p, size_t n, int c, size_t* off, size_t* len) {
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK) return st;
  if (c < 0 || c >= p) return fail(CCL_ERR_INVALID_ARG, "chunk %d outside 0..%d", c, p - 1);
  if (off == nullptr || len == nullptr) return fail(CCL_ERR_INVALID_ARG, "NULL output pointer");
  uint64_t o, l;
  chunk(p, n, c, &o, &l);
  *off = static_cast<size_t>(o);
  *len = static_cast<size_t>(l);
  return CCL_OK;
}

extern "C" ccl_status_t ccl_fold_plan(ccl_fold_kind_t kind, ccl_dtype_t dt, ccl_op_t op, int p, size_t n,
                                      int aligned, int sm_count, int* batch, int* vectors) {
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK) return st;
  if (elem_bytes(dt) == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (!valid_op(op)) return fail(CCL_ERR_INVALID_ARG, "unknown op %d", op);
  int mode = 0;
  switch (kind) {
    case CCL_FOLD_ALLREDUCE: mode = kModeAllReduce; break;
    case CCL_FOLD_REDUCE_SCATTER: mode = kModeReduceScatter; break;
    case CCL_FOLD_BUCKET: mode = kModeBucket; break;
    case CCL_FOLD_REDUCE: mode = kModeReduce; break;
    default: return fail(CCL_ERR_INVALID_ARG, "unknown call kind %d", kind);
  }
  const bool bucket = mode == kModeBucket;
  if (bucket && (dt != CCL_F32 || op != CCL_SUM))
    return fail(CCL_ERR_INVALID_ARG, "the bucket call folds fp32 sums only");
  if (batch == nullptr || vectors == nullptr) return fail(CCL_ERR_INVALID_ARG, "NULL output pointer");
  const int sms = sm_count > 0 ? sm_count : current_sm_count();
  const FoldPlan pl = fold_plan(dt, bucket ? CCL_BF16 : dt, op, mode, p, n / static_cast<uint64_t>(p),
                                aligned != 0, sms);
  *batch = pl.batch;
  *vectors = pl.vectors;
  return CCL_OK;
}

// ====================================================== fused single-pass calls
namespace {
ccl_status_t fused_reduce(int mode, const void* const* send, void* const* recv, int p, size_t n,
                          int dt, int op, void* stream) {
  FoldArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) {
    a.send[r] = send[r];
    a.recv[r] = recv[r];
  }
  a.p = p;
  a.q = n / static_cast<uint64_t>(p);
  a.rem = n % static_cast<uint64_t>(p);
  a.scale = 1.0f;
  const bool vec = all_aligned16(send, p, const_cast<const void* const*>(recv));
  cudaError_t err = launch_fold(mode, dt, op, vec, a, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "fold kernel launch");
  return CCL_OK;
}
}  // namespace

extern "C" ccl_status_t ccl_allreduce(const void* const* send, void* const* recv, int p, size_t n,
                                      ccl_dtype_t dt, ccl_op_t op, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_reduce(0, send, recv, p, n, dt, op);
  if (st != CCL_OK || n == 0) return st;
  return fused_reduce(kModeAllReduce, send, recv, p, n, dt, op, stream);
}

extern "C" ccl_status_t ccl_allreduce_schedule(const void* const* send, void* const* recv, int p,
                                               size_t n, ccl_dtype_t dt, ccl_op_t op,
                                               ccl_schedule_t schedule, void* stream) {
  CCL_TRACE();
  clear_error();
  if (schedule == CCL_SCHEDULE_RING) return ccl_allreduce(send, recv, p, n, dt, op, stream);
  if (schedule < CCL_SCHEDULE_RECURSIVE_DOUBLING || schedule > CCL_SCHEDULE_NAIVE)
    return fail(CCL_ERR_INVALID_ARG, "unknown schedule %d", static_cast<int>(schedule));
  ccl_status_t st = check_reduce(0, send, recv, p, n, dt, op);
  if (st != CCL_OK) return st;
  if (op != CCL_SUM)
    return fail(CCL_ERR_UNSUPPORTED, "schedules other than the ring are implemented for SUM only");
  if ((schedule == CCL_SCHEDULE_RECURSIVE_DOUBLING || schedule == CCL_SCHEDULE_RABENSEIFNER) &&
      (p & (p - 1)) != 0)
    return fail(CCL_ERR_INVALID_ARG, "this schedule needs p to be a power of two (p=%d)", p);
  if (n == 0) return CCL_OK;
  FoldArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) {
    a.send[r] = send[r];
    a.recv[r] = recv[r];
  }
  a.p = p;
  a.q = n / static_cast<uint64_t>(p);
  a.rem = n % static_cast<uint64_t>(p);
  a.scale = 1.0f;
  const bool vec = all_aligned16(send, p, const_cast<const void* const*>(recv));
  cudaError_t err = launch_schedule_fold(dt, schedule == CCL_SCHEDULE_NAIVE,
                                         schedule == CCL_SCHEDULE_RABENSEIFNER, vec, a, n,
                                         as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "schedule kernel launch");
  return CCL_OK;
}

namespace {
ccl_status_t wire_reduce(int mode, const void* const* send, void* const* recv, int p, size_t n,
                         void* stream) {
  FoldArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) {
    a.send[r] = send[r];
    a.recv[r] = recv[r];
  }
  a.p = p;
  a.q = n / static_cast<uint64_t>(p);
  a.rem = n % static_cast<uint64_t>(p);
  a.scale = 1.0f;
  const bool vec = all_aligned16(send, p, const_cast<const void* const*>(recv));
  cudaError_t err = launch_wire_fold(mode, vec, a, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "bf16-wire fold kernel launch");
  return CCL_OK;
}
}  // namespace

extern "C" ccl_status_t ccl_allreduce_bf16_wire(const void* const* send, void* const* recv, int p,
                                                size_t n, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_reduce(0, send, recv, p, n, CCL_BF16, CCL_SUM);
  if (st != CCL_OK || n == 0) return st;
  return wire_reduce(kModeAllReduce, send, recv, p, n, stream);
}

extern "C" ccl_status_t ccl_reduce_scatter_bf16_wire(const void* const* send, void* const* recv, int p,
                                                     size_t n, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_reduce(1, send, recv, p, n, CCL_BF16, CCL_SUM);
  if (st != CCL_OK || n == 0) return st;
  return wire_reduce(kModeReduceScatter, send, recv, p, n, stream);
}

extern "C" ccl_status_t ccl_allreduce_hierarchical(const void* const* send, void* const* recv, int p,
                                                   int group, size_t n, ccl_dtype_t dt, ccl_op_t op,
                                                   void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_reduce(0, send, recv, p, n, dt, op);
  if (st != CCL_OK) return st;
  if (group < 1 || p % group != 0)
    return fail(CCL_ERR_INVALID_ARG, "group=%d must divide p=%d", group, p);
  if (op != CCL_SUM)
    return fail(CCL_ERR_UNSUPPORTED, "the hierarchical fold is implemented for SUM only");
  if (n == 0) return CCL_OK;
  FoldArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) {
    a.send[r] = send[r];
    a.recv[r] = recv[r];
  }
  a.p = p;
  a.q = n / static_cast<uint64_t>(group);
  a.rem = n % static_cast<uint64_t>(group);
  a.scale = 1.0f;
  const bool vec = all_aligned16(send, p, const_cast<const void* const*>(recv));
  cudaError_t err = launch_hier_fold(dt, vec, a, group, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "hierarchical fold kernel launch");
  return CCL_OK;
}

extern "C" ccl_status_t ccl_reduce_scatter(const void* const* send, void* const* recv, int p,
                                           size_t n, ccl_dtype_t dt, ccl_op_t op, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_reduce(1, send, recv, p, n, dt, op);
  if (st != CCL_OK || n == 0) return st;
  return fused_reduce(kModeReduceScatter, send, recv, p, n, dt, op, stream);
}

namespace {
// The bulk-copy fan-out (bulk_fanout.cu) is an alternative to the thread-store
// all-gather and broadcast kernels, taken when the environment variable
// CCL_FORCE_VARIANT is "tma" and the call is large, all device memory and
// meets the bulk copies' 16-byte rule.  It is not the default: on GB300 the
// thread stores reach 0.99 of the copy bandwidth at p = 16 and the best bulk
// pipeline (two 64 KB stages) 0.95.
#ifndef CCL_FANOUT_MIN_CHUNK
#define CCL_FANOUT_MIN_CHUNK (1ull << 20)
#endif
constexpr uint64_t kFanoutMinChunk = CCL_FANOUT_MIN_CHUNK;

// Memory of the current device (not host memory, not another GPU's).
bool device_memory(const void* ptr) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    cudaGetLastError();  // clear the (non-sticky) error of a failed query
    return false;
  }
  int dev = -1;
  return at.type == cudaMemoryTypeDevice && cudaGetDevice(&dev) == cudaSuccess && at.device == dev;
}

bool use_fanout(const FanoutArgs& f) {
  const char* variant = getenv("CCL_FORCE_VARIANT");
  if (variant == nullptr || strcmp(variant, "tma") != 0) return false;
  if (f.chunk_bytes < kFanoutMinChunk || !fanout_supported(f)) return false;
  for (int r = 0; r < f.p; ++r)
    if (!device_memory(f.recv[r])) return false;
  for (uint64_t c = 0; c < f.nchunks; ++c)
    if (!device_memory(f.send[c])) return false;
  return true;
}
}  // namespace

extern "C" ccl_status_t ccl_all_gather(const void* const* send, void* const* recv, int p, size_t n,
                                       ccl_dtype_t dt, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_gather(send, recv, p, n, dt);
  if (st != CCL_OK || n == 0) return st;
  GatherArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) {
    a.send[r] = send[r];
    a.recv[r] = recv[r];
  }
  a.p = p;
  a.q = n / static_cast<uint64_t>(p);
  a.rem = n % static_cast<uint64_t>(p);
  if (a.rem == 0) {
    FanoutArgs f;
    memset(&f, 0, sizeof(f));
    for (int r = 0; r < p; ++r) {
      f.send[r] = send[r];
      f.recv[r] = recv[r];
    }
    f.p = p;
    f.chunk_bytes = a.q * elem_bytes(dt);
    f.nchunks = static_cast<uint64_t>(p);
    if (use_fanout(f)) {
      cudaError_t err = launch_fanout(f, as_stream(stream));
      if (err != cudaSuccess) return cuda_fail(err, "all-gather bulk fan-out launch");
      return CCL_OK;
    }
  }
  const bool vec = all_aligned16(send, p, const_cast<const void* const*>(recv));
  cudaError_t err = launch_gather(dt, vec, a, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "all-gather kernel launch");
  return CCL_OK;
}

extern "C" ccl_status_t ccl_bucket_allreduce_scale_cast(const float* const* grads,
                                                        void* const* out_bf16, int p, size_t n,
                                                        float scale, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK) return st;
  if (n > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "n=%zu too large", n);
  if (grads == nullptr || out_bf16 == nullptr)
    return fail(CCL_ERR_INVALID_ARG, "grads or out_bf16 array is NULL");
  if (n == 0) return CCL_OK;
  const void* const* send = reinterpret_cast<const void* const*>(grads);
  uint64_t in_bytes[CCL_MAX_RANKS], out_bytes[CCL_MAX_RANKS];
  Span in[CCL_MAX_RANKS] = {}, out[CCL_MAX_RANKS] = {};
  for (int r = 0; r < p; ++r) {
    in_bytes[r] = n * 4;
    out_bytes[r] = n * 2;
    in[r] = span(send[r], in_bytes[r]);
    out[r] = span(out_bf16[r], out_bytes[r]);
  }
  if ((st = check_buffers("grads", send, p, in_bytes, 4)) != CCL_OK) return st;
  if ((st = check_buffers("out_bf16", const_cast<const void* const*>(out_bf16), p, out_bytes, 2)) != CCL_OK)
    return st;
  if ((st = check_aliasing(in, out, nullptr, p)) != CCL_OK) return st;
  FoldArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) {
    a.send[r] = send[r];
    a.recv[r] = out_bf16[r];
  }
  a.p = p;
  a.q = n / static_cast<uint64_t>(p);
  a.rem = n % static_cast<uint64_t>(p);
  a.scale = scale;
  const bool vec = all_aligned16(send, p, const_cast<const void* const*>(out_bf16));
  cudaError_t err = launch_fold(kModeBucket, CCL_F32, CCL_SUM, vec, a, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "bucket kernel launch");
  return CCL_OK;
}

// ========================================= broadcast / reduce / scatter / gather
namespace {

ccl_status_t check_root(int p, int root) {
  if (root < 0 || root >= p) return fail(CCL_ERR_INVALID_ARG, "root %d outside 0..%d", root, p - 1);
  return CCL_OK;
}

ccl_status_t copy_transfers(int dt, const char* const* src, char* const* dst, const uint64_t* len,
                            int p, void* stream) {
  XferArgs x;
  memset(&x, 0, sizeof(x));
  x.p = p;
  for (int r = 0; r < p; ++r) {
    x.src[r] = src[r];
    x.dst[r] = dst[r];
    x.len[r] = len[r];
  }
  cudaError_t err = launch_xfer(kXferCopy, dt, CCL_SUM, x, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "copy kernel launch");
  return CCL_OK;
}

}  // namespace

extern "C" ccl_status_t ccl_broadcast(const void* send, void* const* recv, int p, size_t n,
                                      ccl_dtype_t dt, int root, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK || (st = check_root(p, root)) != CCL_OK) return st;
  const size_t e = elem_bytes(dt);
  if (e == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (n > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "n=%zu too large", n);
  if (recv == nullptr) return fail(CCL_ERR_INVALID_ARG, "recv array is NULL");
  if (n == 0) return CCL_OK;
  const void* sends[1] = {send};
  uint64_t in_b[1] = {n * e}, out_b[CCL_MAX_RANKS];
  Span in[CCL_MAX_RANKS], out[CCL_MAX_RANKS];
  bool in_place[CCL_MAX_RANKS];
  for (int r = 0; r < p; ++r) {
    out_b[r] = n * e;
    out[r] = span(recv[r], out_b[r]);
    in[r] = (r == root) ? span(send, n * e) : Span{0, 0};
    in_place[r] = (r == root) && recv[r] == send;
  }
  if ((st = check_buffers("send", sends, 1, in_b, e)) != CCL_OK) return st;
  if ((st = check_buffers("recv", const_cast<const void* const*>(recv), p, out_b, e)) != CCL_OK) return st;
  for (int r = 0; r < p; ++r)  // the root's data must not overlap any other output
    if (r != root && overlaps(out[r], span(send, n * e)))
      return fail(CCL_ERR_INVALID_ARG, "output buffer %d overlaps the root's input", r);
  if ((st = check_aliasing(in, out, in_place, p)) != CCL_OK) return st;
  GatherArgs a;
  memset(&a, 0, sizeof(a));
  a.send[0] = send;
  for (int r = 0; r < p; ++r) a.recv[r] = recv[r];
  a.p = p;
  {
    FanoutArgs f;
    memset(&f, 0, sizeof(f));
    f.send[0] = send;
    for (int r = 0; r < p; ++r) f.recv[r] = recv[r];
    f.p = p;
    f.chunk_bytes = n * e;
    f.nchunks = 1;
    if (use_fanout(f)) {
      cudaError_t err = launch_fanout(f, as_stream(stream));
      if (err != cudaSuccess) return cuda_fail(err, "broadcast bulk fan-out launch");
      return CCL_OK;
    }
  }
  bool vec = (reinterpret_cast<uintptr_t>(send) & 15) == 0;
  for (int r = 0; r < p; ++r) vec = vec && (reinterpret_cast<uintptr_t>(recv[r]) & 15) == 0;
  cudaError_t err = launch_broadcast(dt, vec, a, n, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "broadcast kernel launch");
  return CCL_OK;
}

extern "C" ccl_status_t ccl_reduce(const void* const* send, void* recv, int p, size_t n,
                                   ccl_dtype_t dt, ccl_op_t op, int root, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK || (st = check_root(p, root)) != CCL_OK) return st;
  // validate as an all-reduce whose only output is the root's
  if (recv == nullptr && n != 0) return fail(CCL_ERR_INVALID_ARG, "recv is NULL");
  const size_t e = elem_bytes(dt);
  if (e == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (!valid_op(op)) return fail(CCL_ERR_INVALID_ARG, "unknown op %d", op);
  if (n > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "n=%zu too large", n);
  if (send == nullptr) return fail(CCL_ERR_INVALID_ARG, "send array is NULL");
  if (n == 0) return CCL_OK;
  uint64_t in_b[CCL_MAX_RANKS], out_b[1] = {n * e};
  Span in[CCL_MAX_RANKS], out[CCL_MAX_RANKS];
  bool in_place[CCL_MAX_RANKS];
  for (int r = 0; r < p; ++r) {
    in_b[r] = n * e;
    in[r] = span(send[r], in_b[r]);
    out[r] = (r == root) ? span(recv, n * e) : Span{0, 0};
    in_place[r] = (r == root) && send[r] == recv;
  }
  const void* const recvs[1] = {recv};
  if ((st = check_buffers("send", send, p, in_b, e)) != CCL_OK) return st;
  if ((st = check_buffers("recv", recvs, 1, out_b, e)) != CCL_OK) return st;
  if ((st = check_aliasing(in, out, in_place, p)) != CCL_OK) return st;
  FoldArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) a.send[r] = send[r];
  a.recv[0] = recv;
  a.p = p;
  a.q = n / static_cast<uint64_t>(p);
  a.rem = n % static_cast<uint64_t>(p);
  a.scale = 1.0f;
  bool vec = (reinterpret_cast<uintptr_t>(recv) & 15) == 0;
  for (int r = 0; r < p; ++r) vec = vec && (reinterpret_cast<uintptr_t>(send[r]) & 15) == 0;
  cudaError_t err = launch_fold(kModeReduce, dt, op, vec, a, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "reduce kernel launch");
  return CCL_OK;
}

extern "C" ccl_status_t ccl_scatter(const void* send, void* const* recv, int p, size_t n,
                                    ccl_dtype_t dt, int root, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK || (st = check_root(p, root)) != CCL_OK) return st;
  const size_t e = elem_bytes(dt);
  if (e == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (n > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "n=%zu too large", n);
  if (recv == nullptr) return fail(CCL_ERR_INVALID_ARG, "recv array is NULL");
  if (n == 0) return CCL_OK;
  const void* sends[1] = {send};
  uint64_t in_b[1] = {n * e}, out_b[CCL_MAX_RANKS], len[CCL_MAX_RANKS];
  const char* src[CCL_MAX_RANKS];
  char* dst[CCL_MAX_RANKS];
  Span in[CCL_MAX_RANKS], out[CCL_MAX_RANKS];
  bool in_place[CCL_MAX_RANKS];
  for (int r = 0; r < p; ++r) {
    uint64_t off, ln;
    chunk(p, n, r, &off, &ln);
    out_b[r] = ln * e;
    len[r] = ln;
    out[r] = span(recv[r], out_b[r]);
    in[r] = (r == root) ? span(send, n * e) : Span{0, 0};
    in_place[r] = (r == root) && static_cast<const char*>(send) + off * e == recv[r];
    src[r] = static_cast<const char*>(send) + off * e;
    dst[r] = static_cast<char*>(recv[r]);
  }
  if ((st = check_buffers("send", sends, 1, in_b, e)) != CCL_OK) return st;
  if ((st = check_buffers("recv", const_cast<const void* const*>(recv), p, out_b, e)) != CCL_OK) return st;
  for (int r = 0; r < p; ++r)
    if (r != root && overlaps(out[r], span(send, n * e)))
      return fail(CCL_ERR_INVALID_ARG, "output buffer %d overlaps the root's input", r);
  if ((st = check_aliasing(in, out, in_place, p)) != CCL_OK) return st;
  return copy_transfers(dt, src, dst, len, p, stream);
}

extern "C" ccl_status_t ccl_gather(const void* const* send, void* recv, int p, size_t n,
                                   ccl_dtype_t dt, int root, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK || (st = check_root(p, root)) != CCL_OK) return st;
  const size_t e = elem_bytes(dt);
  if (e == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (n > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "n=%zu too large", n);
  if (send == nullptr) return fail(CCL_ERR_INVALID_ARG, "send array is NULL");
  if (n == 0) return CCL_OK;
  const void* const recvs[1] = {recv};
  uint64_t in_b[CCL_MAX_RANKS], out_b[1] = {n * e}, len[CCL_MAX_RANKS];
  const char* src[CCL_MAX_RANKS];
  char* dst[CCL_MAX_RANKS];
  for (int r = 0; r < p; ++r) {
    uint64_t off, ln;
    chunk(p, n, r, &off, &ln);
    in_b[r] = ln * e;
    len[r] = ln;
    src[r] = static_cast<const char*>(send[r]);
    dst[r] = static_cast<char*>(recv) + off * e;
  }
  if ((st = check_buffers("send", send, p, in_b, e)) != CCL_OK) return st;
  if ((st = check_buffers("recv", recvs, 1, out_b, e)) != CCL_OK) return st;
  const Span whole = span(recv, n * e);
  for (int r = 0; r < p; ++r) {  // only the root's own block may sit in place
    if (!overlaps(whole, span(send[r], in_b[r]))) continue;
    if (r == root && src[r] == dst[r]) continue;
    return fail(CCL_ERR_INVALID_ARG, "input buffer %d overlaps the root's output", r);
  }
  return copy_transfers(dt, src, dst, len, p, stream);
}

// ==================================================== MoE route / dispatch / combine
namespace {

ccl_status_t check_moe(int p, size_t tokens, int k, int num_experts, size_t hidden) {
  if (p < 1 || p > kMoeMaxRanks) return fail(CCL_ERR_INVALID_ARG, "p=%d outside 1..%d", p, kMoeMaxRanks);
  if (k < 1 || k > kMoeMaxK) return fail(CCL_ERR_INVALID_ARG, "k=%d outside 1..%d", k, kMoeMaxK);
  if (num_experts < p || num_experts % p != 0)
    return fail(CCL_ERR_INVALID_ARG, "num_experts=%d must be a positive multiple of p=%d", num_experts, p);
  if (tokens * static_cast<uint64_t>(k) > 0x7FFFFFFFull || tokens > (1ull << 40))
    return fail(CCL_ERR_INVALID_ARG, "tokens * k must stay below 2^31");
  if (hidden == 0 || hidden % 128 != 0 || hidden > (1ull << 30))
    return fail(CCL_ERR_INVALID_ARG, "hidden=%zu must be a positive multiple of 128", hidden);
  return CCL_OK;
}

ccl_status_t check_ptrs(const char* name, const void* const* a, int p, size_t align, bool need) {
  if (!need) return CCL_OK;
  if (a == nullptr) return fail(CCL_ERR_INVALID_ARG, "%s array is NULL", name);
  for (int r = 0; r < p; ++r) {
    if (a[r] == nullptr) return fail(CCL_ERR_INVALID_ARG, "%s[%d] is NULL", name, r);
    if (reinterpret_cast<uintptr_t>(a[r]) % align)
      return fail(CCL_ERR_INVALID_ARG, "%s[%d] is not %zu-byte aligned", name, r, align);
  }
  return CCL_OK;
}

}  // namespace

extern "C" ccl_status_t ccl_moe_route(const int32_t* const* expert_ids, int p, size_t tokens, int k,
                                      int num_experts, int64_t* counts, int32_t* const* slots,
                                      void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_moe(p, tokens, k, num_experts, 128);
  if (st != CCL_OK) return st;
  if (counts == nullptr || (reinterpret_cast<uintptr_t>(counts) & 7))
    return fail(CCL_ERR_INVALID_ARG, "counts is NULL or not 8-byte aligned");
  const bool any = tokens > 0;
  if ((st = check_ptrs("expert_ids", reinterpret_cast<const void* const*>(expert_ids), p, 4, any)) != CCL_OK ||
      (st = check_ptrs("slots", reinterpret_cast<const void* const*>(slots), p, 4, any)) != CCL_OK)
    return st;
  MoeRouteArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) {
    a.ids[r] = any ? expert_ids[r] : nullptr;
    a.slots[r] = any ? slots[r] : nullptr;
  }
  a.counts = counts;
  a.items = tokens * static_cast<uint64_t>(k);
  a.p = p;
  a.epr = num_experts / p;
  a.num_experts = num_experts;
  cudaError_t err = launch_moe_route(a, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "MoE route kernel launch");
  return CCL_OK;
}

extern "C" ccl_status_t ccl_moe_dispatch(const void* const* x, const int32_t* const* expert_ids,
                                         const int64_t* counts, const int32_t* const* slots, int p,
                                         size_t tokens, int k, int num_experts, size_t hidden,
                                         int fp8, void* const* recv, const size_t* recv_rows,
                                         float* const* recv_scales, int32_t* const* recv_expert,
                                         void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_moe(p, tokens, k, num_experts, hidden);
  if (st != CCL_OK) return st;
  if (counts == nullptr || recv_rows == nullptr) return fail(CCL_ERR_INVALID_ARG, "counts or recv_rows is NULL");
  if (tokens == 0) return CCL_OK;
  if ((st = check_ptrs("x", x, p, 16, true)) != CCL_OK ||
      (st = check_ptrs("expert_ids", reinterpret_cast<const void* const*>(expert_ids), p, 4, true)) != CCL_OK ||
      (st = check_ptrs("slots", reinterpret_cast<const void* const*>(slots), p, 4, true)) != CCL_OK)
    return st;
  MoeDispatchArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) {
    a.cap[r] = recv_rows[r];
    if (recv_rows[r] != 0) {
      if (recv == nullptr || recv[r] == nullptr || (reinterpret_cast<uintptr_t>(recv[r]) & 15))
        return fail(CCL_ERR_INVALID_ARG, "recv[%d] is NULL or not 16-byte aligned", r);
      if (fp8 && (recv_scales == nullptr || recv_scales[r] == nullptr ||
                  (reinterpret_cast<uintptr_t>(recv_scales[r]) & 3)))
        return fail(CCL_ERR_INVALID_ARG, "recv_scales[%d] is NULL or misaligned", r);
      a.recv[r] = recv[r];
      a.scales[r] = fp8 ? recv_scales[r] : nullptr;
      a.rexp[r] = recv_expert != nullptr ? recv_expert[r] : nullptr;
    }
    a.x[r] = x[r];
    a.ids[r] = expert_ids[r];
    a.slots[r] = slots[r];
  }
  a.counts = counts;
  a.tokens = tokens;
  a.hidden = hidden;
  a.p = p;
  a.k = k;
  a.epr = num_experts / p;
  a.num_experts = num_experts;
  a.rexp_given = recv_expert != nullptr ? 1 : 0;
  cudaError_t err = launch_moe_dispatch(a, fp8 != 0, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "MoE dispatch kernel launch");
  return CCL_OK;
}

extern "C" ccl_status_t ccl_moe_combine(const void* const* y, const size_t* y_rows,
                                        const int32_t* const* expert_ids, const float* const* weights,
                                        const int64_t* counts, const int32_t* const* slots, int p,
                                        size_t tokens, int k, int num_experts, size_t hidden,
                                        void* const* out, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_moe(p, tokens, k, num_experts, hidden);
  if (st != CCL_OK) return st;
  if (counts == nullptr || y_rows == nullptr) return fail(CCL_ERR_INVALID_ARG, "counts or y_rows is NULL");
  if (tokens == 0) return CCL_OK;
  if ((st = check_ptrs("expert_ids", reinterpret_cast<const void* const*>(expert_ids), p, 4, true)) != CCL_OK ||
      (st = check_ptrs("weights", reinterpret_cast<const void* const*>(weights), p, 4, true)) != CCL_OK ||
      (st = check_ptrs("slots", reinterpret_cast<const void* const*>(slots), p, 4, true)) != CCL_OK ||
      (st = check_ptrs("out", const_cast<const void* const*>(out), p, 16, true)) != CCL_OK)
    return st;
  MoeCombineArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) {
    a.cap[r] = y_rows[r];
    if (y_rows[r] != 0) {
      if (y == nullptr || y[r] == nullptr || (reinterpret_cast<uintptr_t>(y[r]) & 15))
        return fail(CCL_ERR_INVALID_ARG, "y[%d] is NULL or not 16-byte aligned", r);
      a.y[r] = y[r];
    }
    a.ids[r] = expert_ids[r];
    a.slots[r] = slots[r];
    a.weights[r] = weights[r];
    a.out[r] = out[r];
  }
  a.counts = counts;
  a.tokens = tokens;
  a.hidden = hidden;
  a.p = p;
  a.k = k;
  a.epr = num_experts / p;
  a.num_experts = num_experts;
  cudaError_t err = launch_moe_combine(a, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "MoE combine kernel launch");
  return CCL_OK;
}

// ============================================= Ulysses head <-> sequence all-to-all
extern "C" ccl_status_t ccl_all_to_all_heads(const void* const* send, void* const* recv, int p,
                                             size_t seq_per_rank, size_t heads, size_t head_dim,
                                             ccl_dtype_t dt, int inverse, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK) return st;
  const size_t e = elem_bytes(dt);
  if (e == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (heads == 0 || heads % static_cast<size_t>(p) != 0)
    return fail(CCL_ERR_INVALID_ARG, "heads=%zu must be a positive multiple of p=%d", heads, p);
  if (seq_per_rank > (1ull << 32) || heads > (1ull << 20) || head_dim > (1ull << 20))
    return fail(CCL_ERR_INVALID_ARG, "sizes too large");
  if (send == nullptr || recv == nullptr) return fail(CCL_ERR_INVALID_ARG, "send or recv array is NULL");
  const uint64_t n = seq_per_rank * heads * head_dim;  // elements per rank, both layouts
  if (n == 0) return CCL_OK;
  uint64_t b[CCL_MAX_RANKS] = {};
  Span in[CCL_MAX_RANKS] = {}, out[CCL_MAX_RANKS] = {};
  for (int r = 0; r < p; ++r) {
    b[r] = n * e;
    in[r] = span(send[r], b[r]);
    out[r] = span(recv[r], b[r]);
  }
  if ((st = check_buffers("send", send, p, b, e)) != CCL_OK) return st;
  if ((st = check_buffers("recv", const_cast<const void* const*>(recv), p, b, e)) != CCL_OK) return st;
  if ((st = check_aliasing(in, out, nullptr, p)) != CCL_OK) return st;
  UlyssesArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < p; ++r) {
    a.x[r] = send[r];
    a.y[r] = recv[r];
  }
  a.seq_per_rank = seq_per_rank;
  a.heads = heads;
  a.head_dim = head_dim;
  a.segments = static_cast<uint64_t>(p) * p * seq_per_rank;
  a.p = p;
  a.inverse = inverse ? 1 : 0;
  const uint64_t seg_bytes = heads / p * head_dim * e;
  const bool vec = all_aligned16(send, p, const_cast<const void* const*>(recv)) &&
                   seg_bytes % 16 == 0 && (heads * head_dim * e) % 16 == 0;
  cudaError_t err = launch_ulysses(dt, vec, a, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "Ulysses all-to-all kernel launch");
  return CCL_OK;
}

// ============================================================== all-to-allv
namespace {

// Destination tiles of one launch: tile0[c] = tiles before destination
// j0 + c; returns the launch's total.  The tile follows the launch's bytes
// per SM (b): 4 KB below 5 KiB, 8 KB below 24 KiB, 16 KB below 64 KiB, else
// 32 KB.  Measured on GB300 with each tile forced (us per call, back to
// back, fp32; bf16 alike), the chosen tile against the next larger one and
// against the rule before (4 KB tiles while they fit one wave, else 32 KB):
//   p = 2 at 512 KiB per rank (b = 6.7 KiB)    8 KB 1.61, 16 KB 1.86, before 1.80
//   p = 8 at 256 KiB (b = 13.5)                8 KB 2.14, 16 KB 2.01, before 2.56
//   p = 72 at 32 KiB (b = 15.2)                8 KB 5.00, 16 KB 5.17, before 8.07
//   p = 16 at 256 KiB (b = 27)                 16 KB 2.50, 32 KB 3.14, before 3.14
//   p = 72 at 64 KiB (b = 30)                  16 KB 5.44, 32 KB 7.21, before 7.21
//   p = 72 at 128 KiB (b = 61)                 16 KB 6.59, 32 KB 7.41
//   p = 16 at 512 KiB (b = 54)                 16 KB 3.46, 32 KB 3.32
//   p = 40 at 256 KiB (b = 67)                 32 KB 7.72 (16 KB 8.60)
//   p = 40 at 16 KiB (b = 4.2)                 4 KB 3.04 (8 KB 3.31)
// Fewer, larger tiles cost a round of latency per tile; more, smaller ones
// the per-tile set-up (block bounds, barriers); from 64 KiB per SM on the
// 32 KB tiles' grid is several waves deep.
template <class P>
uint64_t fill_tiles(P& a, void* const* recv, const uint64_t* out_bytes, int sms) {
  auto fill = [&](uint64_t tile) {
    a.tile_bytes = static_cast<uint32_t>(tile);
    uint64_t total = 0;
    for (int c = 0; c < a.ndest; ++c) {
      a.tile0[c] = total;
      total += a2a_tiles_for(static_cast<const char*>(recv[a.j0 + c]), out_bytes[a.j0 + c], tile);
    }
    a.tile0[a.ndest] = total;
    return total;
  };
  uint64_t bytes = 0;
  for (int c = 0; c < a.ndest; ++c) bytes += out_bytes[a.j0 + c];
  const uint64_t per_sm = bytes / static_cast<uint64_t>(sms > 0 ? sms : 1);
  if (per_sm < 5 * 1024) return fill(kA2ASmallTileBytes);
  if (per_sm < 24 * 1024) return fill(kA2AMidTileBytes[0]);
  if (per_sm < 64 * 1024) return fill(kA2AMidTileBytes[1]);
  return fill(kA2ATileBytes);
}

// What an all-to-all(v) call launches (ccl_a2a_plan_t): filled instead of
// launching when a plan is asked for.
struct A2APlanOut {
  int form = 0, shift = 0, stage = 0, launches = 0;
  uint32_t tile_bytes = 0;
};

template <class P>
void fill_pointers(P& a, const void* const* send, void* const* recv, int p) {
  for (int r = 0; r < p; ++r) {
    a.send[r] = static_cast<const char*>(send[r]);
    a.recv[r] = static_cast<char*>(recv[r]);
  }
}

// The all-to-allv through row-prefix tables, as many destinations per launch
// as the parameter block holds (all of them for p <= 85).
template <class P>
ccl_status_t a2a_table_launches(P& a, const void* const* send, void* const* recv, const size_t* counts,
                                int p, uint64_t row_bytes, size_t e, const uint64_t* out_bytes,
                                bool shift, bool stage, cudaStream_t s, int sms, A2APlanOut* plan) {
  const int per_launch = P::kTableCap / p - 1;
  for (int j0 = 0; j0 < p; j0 += per_launch) {
    memset(static_cast<void*>(&a), 0, sizeof(a));
    fill_pointers(a, send, recv, p);
    a.p = p;
    a.j0 = j0;
    a.ndest = (p - j0 < per_launch) ? p - j0 : per_launch;
    a.plain = 0;
    a.row_bytes = row_bytes;
    a.elem = static_cast<int>(e);
    const int stride = a.ndest + 1;
    for (int i = 0; i < p; ++i) {
      uint64_t rows = 0;
      for (int d = 0; d < j0; ++d) rows += counts[static_cast<size_t>(i) * p + d];
      for (int c = 0; c <= a.ndest; ++c) {
        a.table[i * stride + c] = static_cast<typename P::Entry>(rows);
        if (j0 + c < p) rows += counts[static_cast<size_t>(i) * p + j0 + c];
      }
    }
    if (fill_tiles(a, recv, out_bytes, sms) == 0) continue;
    if (plan != nullptr) {
      if (plan->launches++ == 0) plan->tile_bytes = a.tile_bytes;
      continue;
    }
    cudaError_t err = launch_a2a(a, shift, stage, s);
    if (err != cudaSuccess) return cuda_fail(err, "all-to-all kernel launch");
  }
  return CCL_OK;
}

ccl_status_t a2a_table(const void* const* send, const size_t* counts, void* const* recv, int p,
                       uint64_t row_bytes, size_t e, const uint64_t* in_rows, cudaStream_t s, int sms,
                       A2APlanOut* plan) {
  uint64_t out_bytes[CCL_MAX_RANKS] = {0};
  uint64_t max_rows = 0;
  for (int i = 0; i < p; ++i) {
    max_rows = in_rows[i] > max_rows ? in_rows[i] : max_rows;
    for (int d = 0; d < p; ++d) out_bytes[d] += counts[static_cast<size_t>(i) * p + d] * row_bytes;
  }
  // some block's source and destination differ in 16-byte phase
  bool shift = false;
  uint64_t col[CCL_MAX_RANKS] = {0};  // rows of destination d before source i's block
  for (int i = 0; i < p && !shift; ++i) {
    uint64_t row = 0;
    for (int d = 0; d < p; ++d) {
      const uint64_t c = counts[static_cast<size_t>(i) * p + d];
      if (c != 0) {
        const uintptr_t src = reinterpret_cast<uintptr_t>(send[i]) + row * row_bytes;
        const uintptr_t dst = reinterpret_cast<uintptr_t>(recv[d]) + col[d] * row_bytes;
        shift = shift || ((src - dst) & 15) != 0;
      }
      row += c;
      col[d] += c;
    }
  }
  // the small-block stage: some block edge or destination end off the
  // 16-byte grid, and blocks of kA2AStageMaxBlockBytes or less on average
  bool off_grid = false;
  uint64_t blocks = 0, total = 0;
  for (int d = 0; d < p; ++d) {
    if (out_bytes[d] == 0) continue;
    const uintptr_t dst = reinterpret_cast<uintptr_t>(recv[d]);
    uint64_t rows = 0;
    for (int i = 0; i < p; ++i) {
      const uint64_t c = counts[static_cast<size_t>(i) * p + d];
      off_grid = off_grid || ((dst + rows * row_bytes) & 15) != 0;
      blocks += c != 0 ? 1 : 0;
      rows += c;
    }
    off_grid = off_grid || ((dst + out_bytes[d]) & 15) != 0;
    total += out_bytes[d];
  }
  const bool stage = off_grid && total <= kA2AStageMaxBlockBytes * blocks;
  if (plan != nullptr) {
    plan->shift = shift;
    plan->stage = stage;
  }
  // uint32 table entries hold every row prefix only while each source has
  // fewer than 2^32 rows
  if (max_rows >= (1ull << 32)) {
    static thread_local A2ATable64 a;  // 32 KB: kept off the stack
    if (plan != nullptr) plan->form = CCL_A2A_TABLE64;
    return a2a_table_launches(a, send, recv, counts, p, row_bytes, e, out_bytes, shift, stage, s, sms, plan);
  }
  if (p <= A2ASmall::kCap) {
    static thread_local A2ASmall a;
    if (plan != nullptr) plan->form = CCL_A2A_SMALL;
    return a2a_table_launches(a, send, recv, counts, p, row_bytes, e, out_bytes, shift, stage, s, sms, plan);
  }
  static thread_local A2ATable32 a;
  if (plan != nullptr) plan->form = CCL_A2A_TABLE32;
  return a2a_table_launches(a, send, recv, counts, p, row_bytes, e, out_bytes, shift, stage, s, sms, plan);
}

// Rows each rank sends and receives, with the size checks of an
// all-to-allv (CCL_OK, or the failure already recorded).
ccl_status_t a2av_rows(const size_t* counts, int p, uint64_t row_bytes, uint64_t* in_rows, uint64_t* out_rows) {
  for (int r = 0; r < p; ++r) in_rows[r] = out_rows[r] = 0;
  for (int s = 0; s < p; ++s) {
    for (int d = 0; d < p; ++d) {
      const uint64_t c = counts[s * p + d];
      if (c > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "counts[%d][%d] too large", s, d);
      in_rows[s] += c;
      out_rows[d] += c;
    }
  }
  for (int r = 0; r < p; ++r)
    if (row_bytes != 0 && (in_rows[r] > kMaxElems / row_bytes || out_rows[r] > kMaxElems / row_bytes))
      return fail(CCL_ERR_INVALID_ARG, "rank %d buffer too large", r);
  return CCL_OK;
}

}  // namespace

extern "C" ccl_status_t ccl_all_to_allv(const void* const* send, const size_t* counts,
                                        void* const* recv, int p, size_t row_elems,
                                        ccl_dtype_t dt, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK) return st;
  const size_t e = elem_bytes(dt);
  if (e == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (send == nullptr || recv == nullptr || counts == nullptr)
    return fail(CCL_ERR_INVALID_ARG, "send, recv or counts is NULL");
  if (row_elems > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "row_elems=%zu too large", row_elems);
  const uint64_t row_bytes = row_elems * e;
  uint64_t in_rows[CCL_MAX_RANKS], out_rows[CCL_MAX_RANKS];
  if ((st = a2av_rows(counts, p, row_bytes, in_rows, out_rows)) != CCL_OK) return st;
  uint64_t in_bytes[CCL_MAX_RANKS], out_bytes[CCL_MAX_RANKS];
  Span in[CCL_MAX_RANKS], out[CCL_MAX_RANKS];
  for (int r = 0; r < p; ++r) {
    in_bytes[r] = in_rows[r] * row_bytes;
    out_bytes[r] = out_rows[r] * row_bytes;
    in[r] = span(send[r], in_bytes[r]);
    out[r] = span(recv[r], out_bytes[r]);
  }
  if ((st = check_buffers("send", send, p, in_bytes, e)) != CCL_OK) return st;
  if ((st = check_buffers("recv", const_cast<const void* const*>(recv), p, out_bytes, e)) != CCL_OK) return st;
  if ((st = check_aliasing(in, out, nullptr, p)) != CCL_OK) return st;
  if (row_bytes == 0) return CCL_OK;

  return a2a_table(send, counts, recv, p, row_bytes, e, in_rows, as_stream(stream), current_sm_count(), nullptr);
}

namespace {

// The plain all-to-all of n elements per rank (block d of every source is
// chunk d, the chunk rule): its kernel choice, and its launch unless a plan
// is asked for.
ccl_status_t a2a_plain(const void* const* send, void* const* recv, int p, uint64_t n, size_t e,
                       cudaStream_t s, int sms, A2APlanOut* plan) {
  uint64_t out_bytes[CCL_MAX_RANKS], off[CCL_MAX_RANKS], len[CCL_MAX_RANKS];
  for (int r = 0; r < p; ++r) {
    chunk(p, n, r, &off[r], &len[r]);
    out_bytes[r] = static_cast<uint64_t>(p) * len[r] * e;
  }
  bool shift = false;  // some block's source and destination differ in 16-byte phase
  for (int d = 0; d < p && !shift; ++d) {
    if (len[d] == 0) continue;
    for (int i = 0; i < p && !shift; ++i) {
      const uintptr_t src = reinterpret_cast<uintptr_t>(send[i]) + off[d] * e;
      const uintptr_t dst = reinterpret_cast<uintptr_t>(recv[d]) + static_cast<uint64_t>(i) * len[d] * e;
      shift = ((src - dst) & 15) != 0;
    }
  }
  // the small-block stage: some block edge or destination end off the
  // 16-byte grid, and blocks of kA2AStageMaxBlockBytes or less on average
  bool off_grid = false;
  for (int d = 0; d < p && !off_grid; ++d) {
    if (len[d] == 0) continue;
    for (int i = 0; i <= p && !off_grid; ++i)
      off_grid = ((reinterpret_cast<uintptr_t>(recv[d]) + static_cast<uint64_t>(i) * len[d] * e) & 15) != 0;
  }
  const bool stage = off_grid && n * e <= kA2AStageMaxBlockBytes * static_cast<uint64_t>(p);
  if (plan != nullptr) {
    plan->form = p <= A2ASmall::kCap ? CCL_A2A_SMALL : CCL_A2A_PLAIN;
    plan->shift = shift;
    plan->stage = stage;
  }
  auto fill = [&](auto& a) -> ccl_status_t {
    memset(static_cast<void*>(&a), 0, sizeof(a));
    fill_pointers(a, send, recv, p);
    a.p = p;
    a.j0 = 0;
    a.ndest = p;
    a.plain = 1;
    a.row_bytes = e;
    a.elem = static_cast<int>(e);
    a.q = n / static_cast<uint64_t>(p);
    a.rem = n % static_cast<uint64_t>(p);
    if (fill_tiles(a, recv, out_bytes, sms) == 0) return CCL_OK;
    if (plan != nullptr) {
      plan->launches = 1;
      plan->tile_bytes = a.tile_bytes;
      return CCL_OK;
    }
    cudaError_t err = launch_a2a(a, shift, stage, s);
    if (err != cudaSuccess) return cuda_fail(err, "all-to-all kernel launch");
    return CCL_OK;
  };
  if (p <= A2ASmall::kCap) {
    A2ASmall a;
    return fill(a);
  }
  A2APlain a;
  return fill(a);
}

ccl_status_t put_plan(const A2APlanOut& pl, ccl_a2a_plan_t* plan) {
  plan->form = static_cast<ccl_a2a_form_t>(pl.form);
  plan->shift = pl.shift;
  plan->stage = pl.stage;
  plan->launches = pl.launches;
  plan->tile_bytes = pl.tile_bytes;
  return CCL_OK;
}

}  // namespace

extern "C" ccl_status_t ccl_all_to_all(const void* const* send, void* const* recv, int p, size_t n,
                                       ccl_dtype_t dt, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK) return st;
  const size_t e = elem_bytes(dt);
  if (e == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (send == nullptr || recv == nullptr) return fail(CCL_ERR_INVALID_ARG, "send or recv is NULL");
  if (n > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "n=%zu too large", n);
  // destination d receives p blocks of len(d) elements in source order
  uint64_t in_bytes[CCL_MAX_RANKS], out_bytes[CCL_MAX_RANKS];
  Span in[CCL_MAX_RANKS], out[CCL_MAX_RANKS];
  for (int r = 0; r < p; ++r) {
    uint64_t off, len;
    chunk(p, n, r, &off, &len);
    in_bytes[r] = n * e;
    out_bytes[r] = static_cast<uint64_t>(p) * len * e;
    in[r] = span(send[r], in_bytes[r]);
    out[r] = span(recv[r], out_bytes[r]);
  }
  if ((st = check_buffers("send", send, p, in_bytes, e)) != CCL_OK) return st;
  if ((st = check_buffers("recv", const_cast<const void* const*>(recv), p, out_bytes, e)) != CCL_OK) return st;
  if ((st = check_aliasing(in, out, nullptr, p)) != CCL_OK) return st;
  if (n == 0) return CCL_OK;
  return a2a_plain(send, recv, p, n, e, as_stream(stream), current_sm_count(), nullptr);
}

extern "C" ccl_status_t ccl_all_to_all_plan(const void* const* send, void* const* recv, int p, size_t n,
                                            ccl_dtype_t dt, int sm_count, ccl_a2a_plan_t* plan) {
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK) return st;
  const size_t e = elem_bytes(dt);
  if (e == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (send == nullptr || recv == nullptr || plan == nullptr)
    return fail(CCL_ERR_INVALID_ARG, "send, recv or plan is NULL");
  if (n > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "n=%zu too large", n);
  A2APlanOut pl;
  if (n != 0) {
    st = a2a_plain(send, recv, p, n, e, nullptr, sm_count > 0 ? sm_count : current_sm_count(), &pl);
    if (st != CCL_OK) return st;
  }
  return put_plan(pl, plan);
}

extern "C" ccl_status_t ccl_all_to_allv_plan(const void* const* send, const size_t* counts, void* const* recv,
                                             int p, size_t row_elems, ccl_dtype_t dt, int sm_count,
                                             ccl_a2a_plan_t* plan) {
  clear_error();
  ccl_status_t st = check_p(p);
  if (st != CCL_OK) return st;
  const size_t e = elem_bytes(dt);
  if (e == 0) return fail(CCL_ERR_INVALID_ARG, "unknown dtype %d", dt);
  if (send == nullptr || recv == nullptr || counts == nullptr || plan == nullptr)
    return fail(CCL_ERR_INVALID_ARG, "send, recv, counts or plan is NULL");
  if (row_elems > kMaxElems) return fail(CCL_ERR_INVALID_ARG, "row_elems=%zu too large", row_elems);
  const uint64_t row_bytes = row_elems * e;
  uint64_t in_rows[CCL_MAX_RANKS], out_rows[CCL_MAX_RANKS];
  if ((st = a2av_rows(counts, p, row_bytes, in_rows, out_rows)) != CCL_OK) return st;
  A2APlanOut pl;
  if (row_bytes != 0) {
    st = a2a_table(send, counts, recv, p, row_bytes, e, in_rows, nullptr,
                   sm_count > 0 ? sm_count : current_sm_count(), &pl);
    if (st != CCL_OK) return st;
  }
  return put_plan(pl, plan);
}

// ====================================================== literal ring engine
namespace {

// Byte pointers to each rank's working buffer of n elements.
struct Work {
  char* b[CCL_MAX_RANKS];
};

ccl_status_t run_xfer(int kind, int dt, int op, const XferArgs& x, cudaStream_t s) {
  cudaError_t err = launch_xfer(kind, dt, op, x, s);
  if (err != cudaSuccess) return cuda_fail(err, "ring step launch");
  return CCL_OK;
}

// Reduce-scatter phase: p-1 steps on working buffers of the accumulator type
// (4-byte fp32 or int32).  Step s: rank r sends its partial of chunk
// (r-s-1) mod p to rank r+1, which combines it with its own.
ccl_status_t rs_phase(const Work& w, int p, uint64_t n, int acc_dt, int op, uint64_t* sent,
                      cudaStream_t s) {
  for (int step = 0; step < p - 1; ++step) {
    XferArgs x;
    memset(&x, 0, sizeof(x));
    x.p = p;
    for (int r = 0; r < p; ++r) {
      const int c = ((r - step - 1) % p + p) % p;
      uint64_t off, len;
      chunk(p, n, c, &off, &len);
      x.src[r] = w.b[r] + off * 4;
      x.dst[r] = w.b[(r + 1) % p] + off * 4;
      x.len[r] = len;
      sent[r] += len * 4;
    }
    ccl_status_t st = run_xfer(kXferCombine, acc_dt, op, x, s);
    if (st != CCL_OK) return st;
  }
  return CCL_OK;
}

// All-gather phase: p-1 steps on the output buffers.  Step s: rank r sends
// chunk (r-s) mod p to rank r+1.
ccl_status_t ag_phase(const Work& w, int p, uint64_t n, int dt, uint64_t* sent, cudaStream_t s) {
  const size_t e = elem_bytes(dt);
  for (int step = 0; step < p - 1; ++step) {
    XferArgs x;
    memset(&x, 0, sizeof(x));
    x.p = p;
    for (int r = 0; r < p; ++r) {
      const int c = ((r - step) % p + p) % p;
      uint64_t off, len;
      chunk(p, n, c, &off, &len);
      x.src[r] = w.b[r] + off * e;
      x.dst[r] = w.b[(r + 1) % p] + off * e;
      x.len[r] = len;
      sent[r] += len * e;
    }
    ccl_status_t st = run_xfer(kXferCopy, dt, CCL_SUM, x, s);
    if (st != CCL_OK) return st;
  }
  return CCL_OK;
}

// One launch of p per-rank moves: src[r] + src_off(r) -> dst[r] + dst_off(r).
// `whole` true: n elements at offset 0; false: rank r's own chunk r.
ccl_status_t per_rank_move(int kind, int dt, const char* const* src, bool src_chunk_off,
                           char* const* dst, bool dst_chunk_off, bool whole, int p, uint64_t n,
                           size_t src_e, size_t dst_e, cudaStream_t s) {
  XferArgs x;
  memset(&x, 0, sizeof(x));
  x.p = p;
  for (int r = 0; r < p; ++r) {
    uint64_t off, len;
    chunk(p, n, r, &off, &len);
    x.src[r] = src[r] + (src_chunk_off ? off * src_e : 0);
    x.dst[r] = dst[r] + (dst_chunk_off ? off * dst_e : 0);
    x.len[r] = whole ? n : len;
  }
  return run_xfer(kind, dt, CCL_SUM, x, s);
}

ccl_status_t check_workspace(void* ws, size_t ws_bytes, size_t need, const void* const* send,
                             const uint64_t* in_bytes, void* const* recv, const uint64_t* out_bytes,
                             int p) {
  if (need == 0) return CCL_OK;
  if (ws == nullptr) return fail(CCL_ERR_INVALID_ARG, "workspace is NULL (%zu bytes needed)", need);
  if (ws_bytes < need)
    return fail(CCL_ERR_INVALID_ARG, "workspace has %zu bytes, %zu needed", ws_bytes, need);
  if (reinterpret_cast<uintptr_t>(ws) % 4 != 0)
    return fail(CCL_ERR_INVALID_ARG, "workspace is not 4-byte aligned");
  const Span w = span(ws, need);
  for (int r = 0; r < p; ++r) {
    if (overlaps(w, span(send[r], in_bytes[r])) || overlaps(w, span(recv[r], out_bytes[r])))
      return fail(CCL_ERR_INVALID_ARG, "workspace overlaps the buffers of rank %d", r);
  }
  return CCL_OK;
}

void write_sent(uint64_t* out, const uint64_t* sent, int p) {
  if (out == nullptr) return;
  for (int r = 0; r < p; ++r) out[r] = sent[r];
}

size_t literal_ws(int kind, int p, size_t n, int dt) {
  if (p < 1 || p > CCL_MAX_RANKS || elem_bytes(dt) == 0 || n > kMaxElems) return 0;
  if (kind == CCL_KIND_ALLREDUCE) return dt == CCL_BF16 ? static_cast<size_t>(p) * n * 4 : 0;
  if (kind == CCL_KIND_REDUCE_SCATTER) return static_cast<size_t>(p) * n * 4;
  return 0;
}

}  // namespace

extern "C" size_t ccl_ring_literal_workspace_bytes(ccl_kind_t kind, int p, size_t n,
                                                   ccl_dtype_t dt) {
  return literal_ws(kind, p, n, dt);
}

extern "C" ccl_status_t ccl_ring_allreduce_literal(const void* const* send, void* const* recv,
                                                   int p, size_t n, ccl_dtype_t dt, ccl_op_t op,
                                                   uint64_t* bytes_sent, void* workspace,
                                                   size_t workspace_bytes, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_reduce(0, send, recv, p, n, dt, op);
  if (st != CCL_OK) return st;
  uint64_t sent[CCL_MAX_RANKS] = {0};
  if (n == 0) {
    write_sent(bytes_sent, sent, p);
    return CCL_OK;
  }
  const size_t e = elem_bytes(dt);
  uint64_t nb[CCL_MAX_RANKS];
  for (int r = 0; r < p; ++r) nb[r] = n * e;
  const size_t need = literal_ws(CCL_KIND_ALLREDUCE, p, n, dt);
  if ((st = check_workspace(workspace, workspace_bytes, need, send, nb, recv, nb, p)) != CCL_OK) return st;
  cudaStream_t s = as_stream(stream);
  Work out;
  for (int r = 0; r < p; ++r) out.b[r] = static_cast<char*>(recv[r]);
  const char* const* src = reinterpret_cast<const char* const*>(send);

  if (dt == CCL_BF16) {
    // partials travel in fp32: widen into the workspace, reduce there, then the
    // owner of each chunk rounds it once into its output buffer
    Work ws;
    for (int r = 0; r < p; ++r) ws.b[r] = static_cast<char*>(workspace) + static_cast<size_t>(r) * n * 4;
    if ((st = per_rank_move(kXferWiden, CCL_BF16, src, false, ws.b, false, true, p, n, 2, 4, s)) != CCL_OK) return st;
    if ((st = rs_phase(ws, p, n, CCL_F32, op, sent, s)) != CCL_OK) return st;
    if ((st = per_rank_move(kXferNarrow, CCL_BF16, ws.b, true, out.b, true, false, p, n, 4, 2, s)) != CCL_OK) return st;
  } else {
    bool in_place = true;
    for (int r = 0; r < p; ++r) in_place = in_place && (send[r] == recv[r]);
    if (!in_place) {
      if ((st = per_rank_move(kXferCopy, dt, src, false, out.b, false, true, p, n, e, e, s)) != CCL_OK) return st;
    }
    if ((st = rs_phase(out, p, n, dt, op, sent, s)) != CCL_OK) return st;
  }
  if ((st = ag_phase(out, p, n, dt, sent, s)) != CCL_OK) return st;
  write_sent(bytes_sent, sent, p);
  return CCL_OK;
}

extern "C" ccl_status_t ccl_ring_reduce_scatter_literal(const void* const* send, void* const* recv,
                                                        int p, size_t n, ccl_dtype_t dt,
                                                        ccl_op_t op, uint64_t* bytes_sent,
                                                        void* workspace, size_t workspace_bytes,
                                                        void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_reduce(1, send, recv, p, n, dt, op);
  if (st != CCL_OK) return st;
  uint64_t sent[CCL_MAX_RANKS] = {0};
  if (n == 0) {
    write_sent(bytes_sent, sent, p);
    return CCL_OK;
  }
  const size_t e = elem_bytes(dt);
  uint64_t in_b[CCL_MAX_RANKS] = {}, out_b[CCL_MAX_RANKS] = {};
  for (int r = 0; r < p; ++r) {
    uint64_t off, len;
    chunk(p, n, r, &off, &len);
    in_b[r] = n * e;
    out_b[r] = len * e;
  }
  const size_t need = literal_ws(CCL_KIND_REDUCE_SCATTER, p, n, dt);
  if ((st = check_workspace(workspace, workspace_bytes, need, send, in_b, recv, out_b, p)) != CCL_OK) return st;
  cudaStream_t s = as_stream(stream);
  Work ws;
  for (int r = 0; r < p; ++r) ws.b[r] = static_cast<char*>(workspace) + static_cast<size_t>(r) * n * 4;
  char* out[CCL_MAX_RANKS];
  for (int r = 0; r < p; ++r) out[r] = static_cast<char*>(recv[r]);
  const char* const* src = reinterpret_cast<const char* const*>(send);
  const int acc_dt = (dt == CCL_I32) ? CCL_I32 : CCL_F32;
  if (dt == CCL_BF16) {
    if ((st = per_rank_move(kXferWiden, CCL_BF16, src, false, ws.b, false, true, p, n, 2, 4, s)) != CCL_OK) return st;
  } else {
    if ((st = per_rank_move(kXferCopy, dt, src, false, ws.b, false, true, p, n, 4, 4, s)) != CCL_OK) return st;
  }
  if ((st = rs_phase(ws, p, n, acc_dt, op, sent, s)) != CCL_OK) return st;
  // rank k's finished chunk k -> its shard
  const int finish = (dt == CCL_BF16) ? kXferNarrow : kXferCopy;
  if ((st = per_rank_move(finish, dt, ws.b, true, out, false, false, p, n, 4, e, s)) != CCL_OK) return st;
  write_sent(bytes_sent, sent, p);
  return CCL_OK;
}

extern "C" ccl_status_t ccl_ring_all_gather_literal(const void* const* send, void* const* recv,
                                                    int p, size_t n, ccl_dtype_t dt,
                                                    uint64_t* bytes_sent, void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_gather(send, recv, p, n, dt);
  if (st != CCL_OK) return st;
  uint64_t sent[CCL_MAX_RANKS] = {0};
  if (n == 0) {
    write_sent(bytes_sent, sent, p);
    return CCL_OK;
  }
  const size_t e = elem_bytes(dt);
  cudaStream_t s = as_stream(stream);
  Work out;
  for (int r = 0; r < p; ++r) out.b[r] = static_cast<char*>(recv[r]);
  bool in_place = true;
  for (int r = 0; r < p; ++r) {
    uint64_t off, len;
    chunk(p, n, r, &off, &len);
    in_place = in_place && (static_cast<const char*>(send[r]) == out.b[r] + off * e || len == 0);
  }
  if (!in_place) {
    const char* const* src = reinterpret_cast<const char* const*>(send);
    if ((st = per_rank_move(kXferCopy, dt, src, false, out.b, true, false, p, n, e, e, s)) != CCL_OK) return st;
  }
  if ((st = ag_phase(out, p, n, dt, sent, s)) != CCL_OK) return st;
  write_sent(bytes_sent, sent, p);
  return CCL_OK;
}

// ============================================ allocation-free reduce-scatter
// The literal reduce-scatter needs p*n*4 bytes of device scratch for the
// ranks' working buffers.  Some callers cannot allocate that themselves, so
// this entry point uses a fixed scratch array that lives inside the library
// (in this translation unit's module) instead of a caller workspace.

// File-scope scratch, CCL_STATIC_SCRATCH_BYTES on every GPU that loads the
// library, held until the process exits.  Host code must not use the
// symbol's host-side name as a device address; the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char ccl_static_scratch[CCL_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxScratchDevices = 256;
std::mutex g_scratch_mutex;
struct ScratchCache {
  unsigned long long ctx_id;  // the context the address belongs to
  void* address;              // NULL until looked up
};
ScratchCache g_scratch[kMaxScratchDevices];  // per device ordinal

// The process-unique id of the calling thread's current CUDA context, 0 when
// the thread has none yet.  The two driver calls are resolved through the
// runtime (cudaGetDriverEntryPointByVersion), so the library does not link
// the driver library itself.
ccl_status_t current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  if (get_current == nullptr || get_id == nullptr) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    cudaError_t err = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1);
    if (err == cudaSuccess)
      err = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
    if (err != cudaSuccess) return cuda_fail(err, "cudaGetDriverEntryPointByVersion");
    if (q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return fail(CCL_ERR_UNSUPPORTED, "the driver lacks cuCtxGetCurrent / cuCtxGetId");
    get_current = reinterpret_cast<GetCurrent>(f1);
    get_id = reinterpret_cast<GetId>(f2);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return fail(CCL_ERR_CUDA, "cuCtxGetCurrent failed");
  *id = 0;
  if (ctx != nullptr && get_id(ctx, id) != CUDA_SUCCESS) return fail(CCL_ERR_CUDA, "cuCtxGetId failed");
  return CCL_OK;
}

// Device address of the static scratch in the current device's context.
// Looked up on the first call made with that device current, and again
// whenever the current context is not the one the cached address came from
// (after cudaDeviceReset the primary context is re-created and the module,
// with its array, is loaded again at another address).
ccl_status_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxScratchDevices)
    return fail(CCL_ERR_UNSUPPORTED, "device %d beyond the %d devices the static scratch tracks",
                dev, kMaxScratchDevices);
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long ctx = 0;
  ccl_status_t st = current_context_id(&ctx);
  if (st != CCL_OK) return st;
  ScratchCache& c = g_scratch[dev];
  if (c.address == nullptr || ctx == 0 || ctx != c.ctx_id) {
    void* addr = nullptr;
    // makes the device's context current on this thread if it was not
    err = cudaGetSymbolAddress(&addr, ccl_static_scratch);
    if (err != cudaSuccess) return cuda_fail(err, "cudaGetSymbolAddress(static scratch)");
    if ((st = current_context_id(&ctx)) != CCL_OK) return st;
    c.address = addr;
    c.ctx_id = ctx;
  }
  *out = c.address;
  return CCL_OK;
}

}  // namespace

extern "C" ccl_status_t ccl_ring_reduce_scatter_literal_noalloc(const void* const* send,
                                                                void* const* recv, int p, size_t n,
                                                                ccl_dtype_t dt, ccl_op_t op,
                                                                uint64_t* bytes_sent,
                                                                void* stream) {
  CCL_TRACE();
  clear_error();
  ccl_status_t st = check_reduce(1, send, recv, p, n, dt, op);
  if (st != CCL_OK) return st;
  const size_t need = literal_ws(CCL_KIND_REDUCE_SCATTER, p, n, dt);
  if (need > CCL_STATIC_SCRATCH_BYTES)
    return fail(CCL_ERR_INVALID_ARG,
                "p*n*4 = %zu bytes of scratch needed; the static scratch holds %zu "
                "(p*n must not exceed %zu)",
                need, static_cast<size_t>(CCL_STATIC_SCRATCH_BYTES),
                static_cast<size_t>(CCL_STATIC_SCRATCH_BYTES / 4));
  if (n == 0) {
    uint64_t zero[CCL_MAX_RANKS] = {0};
    write_sent(bytes_sent, zero, p);
    return CCL_OK;
  }
  void* scratch = nullptr;
  if ((st = static_scratch_address(&scratch)) != CCL_OK) return st;
  // Nothing in the scratch has to start at zero: the call's first launch
  // overwrites every byte that later launches read.
  return ccl_ring_reduce_scatter_literal(send, recv, p, n, dt, op, bytes_sent, scratch,
                                         CCL_STATIC_SCRATCH_BYTES, stream);
}
