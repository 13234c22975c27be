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

// Binary counter of pairwise subtrees, LEVELS slots (enough for 2^(LEVELS-1)
// leaves plus the carry level), VEC lanes each.
template <int DT, int VEC, int LEVELS>
struct Counter {
  using Acc = typename Elem<DT>::Acc;
  Acc slot[LEVELS][VEC];

  // Add leaf number j (0-based) with values x.
  __device__ __forceinline__ void push(int j, const Acc* x) {
    Acc carry[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) carry[e] = x[e];
    bool chain = true;
#pragma unroll
    for (int k = 0; k < LEVELS; ++k) {
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
    for (int k = 0; k < LEVELS; ++k) {
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

// Fold U vectors (t, t + kThreads, ...) of VEC elements; the loads of BATCH
// ranks x U vectors are issued before any is folded.  MODE 0: pairwise tree,
// 1: linear (naive).
template <int DT, int VEC, int MODE, int LEVELS, int BATCH, int U>
__device__ __forceinline__ void fold_vectors(const FoldArgs& a, int p, int levels, bool reversed,
                                             uint64_t v0, uint64_t v_hi,
                                             typename Elem<DT>::Acc (&acc)[U][VEC]) {
  using Acc = typename Elem<DT>::Acc;
  constexpr int W = (VEC * Elem<DT>::kBytes + 3) / 4;
  Counter<DT, VEC, LEVELS> ctr[U];
  for (int j0 = 0; j0 < p; j0 += BATCH) {
    uint32_t raw[BATCH][U][W];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (j0 + b < p) {
        const void* src = a.send[rank_at(j0 + b, levels, reversed)];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const uint64_t v = v0 + static_cast<uint64_t>(u) * kThreads;
          if (v < v_hi) load_raw<DT, VEC>(src, v * VEC, raw[b][u]);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (j0 + b < p) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          Acc x[VEC];
#pragma unroll
          for (int e = 0; e < VEC; ++e) x[e] = widen<DT>(raw[b][u], e);
          if constexpr (MODE == 0) {
            ctr[u].push(j0 + b, x);
          } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e)
              acc[u][e] = (j0 + b == 0) ? x[e] : combine<CCL_SUM>(x[e], acc[u][e]);
          }
        }
      }
    }
  }
  if constexpr (MODE == 0) {
#pragma unroll
    for (int u = 0; u < U; ++u) ctr[u].flush(p, acc[u]);
  }
}

template <int DT, int VEC, int MODE, int LEVELS, int BATCH, int U>
__global__ void __launch_bounds__(kThreads) schedule_kernel(const __grid_constant__ FoldArgs a,
                                                            uint64_t n, int levels, int reversed) {
  using Acc = typename Elem<DT>::Acc;
  pdl_enter();
  const int p = a.p;
  const uint64_t nv = n / VEC;
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * U;
  for (uint64_t base = static_cast<uint64_t>(blockIdx.x) * kSpan; base < nv;
       base += static_cast<uint64_t>(gridDim.x) * kSpan) {
    Acc acc[U][VEC];
    fold_vectors<DT, VEC, MODE, LEVELS, BATCH, U>(a, p, levels, reversed != 0, base + threadIdx.x,
                                                   nv, acc);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
      if (v < nv) {
        uint32_t w[(VEC * Elem<DT>::kBytes + 3) / 4];
        pack_out<DT, VEC>(acc[u], w);
        for (int r = 0; r < p; ++r) store_raw<DT, VEC>(a.recv[r], v * VEC, w);
      }
    }
  }
  if (VEC > 1 && blockIdx.x == 0) {  // tail elements
    for (uint64_t i = nv * VEC + threadIdx.x; i < n; i += kThreads) {
      Acc acc[1][1];
      fold_vectors<DT, 1, MODE, LEVELS, BATCH, 1>(a, p, levels, reversed != 0, i, i + 1, acc);
      uint32_t w[1];
      pack_out<DT, 1>(acc[0], w);
      for (int r = 0; r < p; ++r) store_raw<DT, 1>(a.recv[r], i, w);
    }
  }
}

template <int DT, int VEC, int MODE, int LEVELS, int BATCH, int U>
cudaError_t launch_one(const FoldArgs& a, uint64_t n, int levels, bool reversed, cudaStream_t s) {
  const uint64_t nv = (VEC > 1) ? n / VEC : n;
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * U;
  uint64_t gx = (nv + kSpan - 1) / kSpan;
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
  return cudaLaunchKernelEx(&cfg, schedule_kernel<DT, VEC, MODE, LEVELS, BATCH, U>, a, n, levels,
                            reversed ? 1 : 0);
}

// Shapes by p, as in the small-p ring kernel: few ranks -> several vectors per
// thread so that about 256 bytes (fp32) / 128 bytes (bf16) of loads are in
// flight; counter slots sized to the ranks.
template <int DT, int MODE>
cudaError_t launch_typed(bool vec, const FoldArgs& a, uint64_t n, int levels, bool reversed,
                         cudaStream_t s) {
  if (!vec) return launch_one<DT, 1, MODE, 8, 8, 1>(a, n, levels, reversed, s);
  constexpr int VEC = 16 / Elem<DT>::kBytes;
  constexpr int H = (VEC > 4) ? 2 : 1;  // bf16: 8 accumulators per vector
  if (a.p <= 2) return launch_one<DT, VEC, MODE, 2, 2, 8 / H>(a, n, levels, reversed, s);
  if (a.p <= 4) return launch_one<DT, VEC, MODE, 3, 4, 4 / H>(a, n, levels, reversed, s);
  if (a.p <= 8) return launch_one<DT, VEC, MODE, 4, 8, 2 / H>(a, n, levels, reversed, s);
  // 16 ranks' loads in flight for bf16 and for p > 16; 8 for 32-bit data up to
  // p = 16 (measured on GB300 at 256 MiB per rank: 16 lifts bf16 p = 16 from
  // 1.00 to 1.03 of the copy bandwidth and p = 72 from 0.98 to 1.00, and
  // costs fp32 p = 16 0.5 %)
  if (a.p <= 16) {
    if constexpr (DT == kBF16) {
      return launch_one<DT, VEC, MODE, 5, 16, 1>(a, n, levels, reversed, s);
    } else {
      return launch_one<DT, VEC, MODE, 5, 8, 1>(a, n, levels, reversed, s);
    }
  }
  return launch_one<DT, VEC, MODE, 8, 16, 1>(a, n, levels, reversed, s);
}

}  // namespace

cudaError_t launch_schedule_fold(int dt, bool linear, bool reversed, bool vec, const FoldArgs& a,
                                 uint64_t n, cudaStream_t s) {
  int levels = 0;
  while ((1 << levels) < a.p) ++levels;
  // with p <= 3 the pairwise tree is ((x0 + x1) + x2), the rank-order fold
  // (Rabenseifner needs p a power of two, and for p = 2 x0 + x1 = x1 + x0)
  if (a.p <= 3) linear = true;
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
