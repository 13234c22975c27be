// ring_step.cu -- one step of the literal ring schedule.
//
// "Networks and Collective Communication" section 5.1: at every step every
// device passes one chunk to the next device; in the reduce-scatter phase the
// receiver adds its own chunk to the partial it got, in the all-gather phase
// it stores the chunk.  One launch performs the p transfers of one step
// (blockIdx.y = sending rank).  Within a step no transfer reads a chunk that
// another transfer of the same step writes, so the p transfers run
// concurrently with no ordering between them; steps are ordered by the stream.
//
// The same kernel also does the engine's set-up and finishing moves: copying
// inputs into working buffers, widening bf16 inputs to fp32 partials, and
// rounding a finished fp32 chunk to bf16.
#include "device_common.cuh"

namespace ccl {
namespace {

template <int KIND, int DT>
struct XferTypes {
  static constexpr int kSrc = (KIND == kXferWiden) ? kBF16 : (KIND == kXferNarrow ? kF32 : DT);
  static constexpr int kDst = (KIND == kXferWiden) ? kF32 : (KIND == kXferNarrow ? kBF16 : DT);
  static constexpr int kVec = (Elem<kSrc>::kBytes == 2 || Elem<kDst>::kBytes == 2) ? 8 : 4;
};

template <int KIND, int DT, int OP, int VEC>
__device__ __forceinline__ void xfer_elems(const char* src, char* dst, uint64_t i) {
  using T = XferTypes<KIND, DT>;
  constexpr int WS = (VEC * Elem<T::kSrc>::kBytes + 3) / 4;
  constexpr int WD = (VEC * Elem<T::kDst>::kBytes + 3) / 4;
  uint32_t ws[WS];
  load_raw<T::kSrc, VEC>(src, i, ws);
  if constexpr (KIND == kXferCopy) {
    store_raw<T::kDst, VEC>(dst, i, ws);
  } else {
    using Acc = typename Elem<T::kSrc>::Acc;
    Acc acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = widen<T::kSrc>(ws, e);
    if constexpr (KIND == kXferCombine) {
      uint32_t wd[WD];
      load_raw<T::kDst, VEC>(dst, i, wd);  // the receiver's own value
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] = combine<OP>(acc[e], widen<T::kDst>(wd, e));
    }
    uint32_t wo[WD];
    pack_out<T::kDst, VEC>(acc, wo);
    store_raw<T::kDst, VEC>(dst, i, wo);
  }
}

// U vectors per thread (t, t + kThreads, ...): all their loads are issued
// before any store, so a thread keeps several 16-byte loads in flight.
template <int KIND, int DT, int OP, int U>
__global__ void __launch_bounds__(kThreads) xfer_kernel(const __grid_constant__ XferArgs a) {
  using T = XferTypes<KIND, DT>;
  constexpr int VEC = T::kVec;
  constexpr int WS = (VEC * Elem<T::kSrc>::kBytes + 3) / 4;
  constexpr int WD = (VEC * Elem<T::kDst>::kBytes + 3) / 4;
  pdl_enter();
  const int r = blockIdx.y;
  const char* src = a.src[r];
  char* dst = a.dst[r];
  const uint64_t len = a.len[r];
  const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
  const uint64_t nv = vec ? len / VEC : 0;
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * U;
  for (uint64_t base = static_cast<uint64_t>(blockIdx.x) * kSpan; base < nv;
       base += static_cast<uint64_t>(gridDim.x) * kSpan) {
    uint32_t ws[U][WS];
    uint32_t wd[U][WD];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
      if (v < nv) {
        load_raw<T::kSrc, VEC>(src, v * VEC, ws[u]);
        if constexpr (KIND == kXferCombine) load_raw<T::kDst, VEC>(dst, v * VEC, wd[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
      if (v >= nv) continue;
      if constexpr (KIND == kXferCopy) {
        store_raw<T::kDst, VEC>(dst, v * VEC, ws[u]);
      } else {
        using Acc = typename Elem<T::kSrc>::Acc;
        Acc acc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = widen<T::kSrc>(ws[u], e);
        if constexpr (KIND == kXferCombine) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[e] = combine<OP>(acc[e], widen<T::kDst>(wd[u], e));
        }
        uint32_t wo[WD];
        pack_out<T::kDst, VEC>(acc, wo);
        store_raw<T::kDst, VEC>(dst, v * VEC, wo);
      }
    }
  }
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  const uint64_t t0 = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x;
  for (uint64_t i = nv * VEC + t0; i < len; i += stride) xfer_elems<KIND, DT, OP, 1>(src, dst, i);
}

template <int KIND, int DT, int OP>
cudaError_t launch_one(const XferArgs& a, cudaStream_t s) {
  constexpr int VEC = XferTypes<KIND, DT>::kVec;
  constexpr int U = 4;
  uint64_t longest = 0;
  for (int r = 0; r < a.p; ++r) longest = a.len[r] > longest ? a.len[r] : longest;
  if (longest == 0) return cudaSuccess;
  uint64_t gx = (longest / VEC + kThreads * U - 1) / (kThreads * U);
  if (gx < 1) gx = 1;
  if (gx > (1u << 30)) gx = 1u << 30;
  cudaError_t err = launch_kernel(xfer_kernel<KIND, DT, OP, U>, dim3(static_cast<unsigned>(gx), a.p),
                                  dim3(kThreads), s, a);
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace

cudaError_t launch_xfer(int kind, int dt, int op, const XferArgs& a, cudaStream_t s) {
  switch (kind) {
    case kXferCopy:
      return (dt == kBF16) ? launch_one<kXferCopy, kBF16, CCL_SUM>(a, s)
                           : launch_one<kXferCopy, kF32, CCL_SUM>(a, s);
    case kXferCombine:
      if (dt == kF32 && op == CCL_SUM) return launch_one<kXferCombine, kF32, CCL_SUM>(a, s);
      if (dt == kF32 && op == CCL_MAX) return launch_one<kXferCombine, kF32, CCL_MAX>(a, s);
      if (dt == kF32 && op == CCL_MIN) return launch_one<kXferCombine, kF32, CCL_MIN>(a, s);
      if (dt == kI32 && op == CCL_SUM) return launch_one<kXferCombine, kI32, CCL_SUM>(a, s);
      if (dt == kI32 && op == CCL_MAX) return launch_one<kXferCombine, kI32, CCL_MAX>(a, s);
      if (dt == kI32 && op == CCL_MIN) return launch_one<kXferCombine, kI32, CCL_MIN>(a, s);
      return cudaErrorInvalidValue;
    case kXferWiden:
      return launch_one<kXferWiden, kBF16, CCL_SUM>(a, s);
    case kXferNarrow:
      return launch_one<kXferNarrow, kBF16, CCL_SUM>(a, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace ccl
