// schedule_fold.cu -- all-reduce in the fold order of the other schedules.
//
// "Networks and Collective Communication" section 5.2 gives recursive
// doubling, Rabenseifner (recursive halving + doubling), the binary
// (binomial) tree and the naive root algorithm.  Each fixes how the p values
// of an element are paired, and IEEE addition is commutative, so only that
// pairing decides the bits:
//
// * recursive doubling (step k pairs devices i and i XOR 2^k) and the
//   binomial tree (step k adds device i + 2^k into device i) both build the
//   left-complete pairwise tree over ranks 0, 1, ..., p-1;
// * Rabenseifner's halving pairs devices at distance p/2 first, then p/4,
//   ..., 1: the same pairwise tree over the ranks taken in bit-reversed order;
// * the naive root adds the arrivals one by one in rank order.
//
// The pairwise tree is evaluated as a binary counter over the ranks in that
// order: slot k holds a finished subtree of 2^k leaves, a new leaf carries
// through the occupied slots (slot k is occupied exactly when bit k of the
// number of leaves seen is set), and at the end the slots are combined from
// the smallest up.  For p a power of two that is the balanced tree; for other
// p it is the binomial tree's shape.  Every element uses the same order, so
// the grid is 1-D over 16-byte vectors; results go to all p outputs.
#include "device_common.cuh"

namespace ccl {
namespace {

constexpr int kMaxLevels = 8;  // p <= 128 = 2^7 leaves; one spare level

template <int DT, int VEC>
struct Counter {
  using Acc = typename Elem<DT>::Acc;
  Acc slot[kMaxLevels][VEC];

  // Add leaf number j (0-based) with values x.
  __device__ __forceinline__ void push(int j, const Acc* x) {
    Acc carry[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) carry[e] = x[e];
    bool chain = true;
#pragma unroll
    for (int k = 0; k < kMaxLevels; ++k) {
      if (chain) {
        if (j & (1 << k)) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) carry[e] = combine<CCL_SUM>(slot[k][e], carry[e]);
        } else {
#pragma unroll
          for (int e = 0; e < VEC; ++e) slot[k][e] = carry[e];
          chain = false;
        }
      }
    }
  }

  // Combine the finished subtrees of a p-leaf counter, smallest first.
  __device__ __forceinline__ void flush(int p, Acc* out) const {
    bool have = false;
#pragma unroll
    for (int k = 0; k < kMaxLevels; ++k) {
      if (p & (1 << k)) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) out[e] = have ? combine<CCL_SUM>(slot[k][e], out[e]) : slot[k][e];
        have = true;
      }
    }
  }
};

// Rank visited at position j: identity, or j's log2(p)-bit reversal.
__device__ __forceinline__ int rank_at(int j, int levels, bool reversed) {
  return reversed ? static_cast<int>(__brev(static_cast<unsigned>(j)) >> (32 - levels)) : j;
}

template <int DT, int VEC, int MODE>  // MODE 0: pairwise tree, 1: linear (naive)
__device__ __forceinline__ void fold_one(const FoldArgs& a, int p, int levels, bool reversed,
                                         uint64_t i, typename Elem<DT>::Acc* acc) {
  using Acc = typename Elem<DT>::Acc;
  constexpr int W = (VEC * Elem<DT>::kBytes + 3) / 4;
  constexpr int BATCH = 8;
  Counter<DT, VEC> ctr;
  for (int j0 = 0; j0 < p; j0 += BATCH) {
    uint32_t raw[BATCH][W];
#pragma unroll
    for (int b = 0; b < BATCH; ++b)
      if (j0 + b < p) load_raw<DT, VEC>(a.send[rank_at(j0 + b, levels, reversed)], i, raw[b]);
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (j0 + b < p) {
        Acc x[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) x[e] = widen<DT>(raw[b], e);
        if constexpr (MODE == 0) {
          ctr.push(j0 + b, x);
        } else {
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[e] = (j0 + b == 0) ? x[e] : combine<CCL_SUM>(x[e], acc[e]);
        }
      }
    }
  }
  if constexpr (MODE == 0) ctr.flush(p, acc);
}

template <int DT, int VEC, int MODE>
__global__ void __launch_bounds__(kThreads) schedule_kernel(const __grid_constant__ FoldArgs a,
                                                            uint64_t n, int levels, int reversed) {
  using Acc = typename Elem<DT>::Acc;
  pdl_enter();
  const int p = a.p;
  const uint64_t nv = n / VEC;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  const uint64_t t0 = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x;
  for (uint64_t v = t0; v < nv; v += stride) {
    Acc acc[VEC];
    fold_one<DT, VEC, MODE>(a, p, levels, reversed != 0, v * VEC, acc);
    uint32_t w[(VEC * Elem<DT>::kBytes + 3) / 4];
    pack_out<DT, VEC>(acc, w);
    for (int r = 0; r < p; ++r) store_raw<DT, VEC>(a.recv[r], v * VEC, w);
  }
  for (uint64_t i = nv * VEC + t0; i < n; i += stride) {  // tail (or everything when VEC == 1)
    Acc acc[1];
    fold_one<DT, 1, MODE>(a, p, levels, reversed != 0, i, acc);
    uint32_t w[1];
    pack_out<DT, 1>(acc, w);
    for (int r = 0; r < p; ++r) store_raw<DT, 1>(a.recv[r], i, w);
  }
}

template <int DT, int VEC, int MODE>
cudaError_t launch_one(const FoldArgs& a, uint64_t n, int levels, bool reversed, cudaStream_t s) {
  const uint64_t work = (VEC > 1) ? n / VEC : n;
  uint64_t gx = (work + 2 * kThreads - 1) / (2 * kThreads);
  if (gx < 1) gx = 1;
  if (gx > (1u << 30)) gx = 1u << 30;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(gx));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = CCL_PDL ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, schedule_kernel<DT, VEC, MODE>, a, n, levels,
                            reversed ? 1 : 0);
}

template <int DT, int MODE>
cudaError_t launch_typed(bool vec, const FoldArgs& a, uint64_t n, int levels, bool reversed,
                         cudaStream_t s) {
  if (vec) return launch_one<DT, 16 / Elem<DT>::kBytes, MODE>(a, n, levels, reversed, s);
  return launch_one<DT, 1, MODE>(a, n, levels, reversed, s);
}

}  // namespace

cudaError_t launch_schedule_fold(int dt, bool linear, bool reversed, bool vec, const FoldArgs& a,
                                 uint64_t n, cudaStream_t s) {
  int levels = 0;
  while ((1 << levels) < a.p) ++levels;
  cudaError_t err = cudaErrorInvalidValue;
  if (linear) {
    if (dt == kF32) err = launch_typed<kF32, 1>(vec, a, n, levels, false, s);
    else if (dt == kBF16) err = launch_typed<kBF16, 1>(vec, a, n, levels, false, s);
    else if (dt == kI32) err = launch_typed<kI32, 1>(vec, a, n, levels, false, s);
  } else {
    if (dt == kF32) err = launch_typed<kF32, 0>(vec, a, n, levels, reversed, s);
    else if (dt == kBF16) err = launch_typed<kBF16, 0>(vec, a, n, levels, reversed, s);
    else if (dt == kI32) err = launch_typed<kI32, 0>(vec, a, n, levels, reversed, s);
  }
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace ccl
