// ulysses.cu -- the head <-> sequence all-to-all of sequence-parallel attention
// ("LLM Distributed Training Collectives", Sequence Parallelism / Ulysses: long
// sequences are split across devices, and attention needs an all-to-all that
// re-partitions the data by head).
//
// Rank r holds sequence shard r with every head, [S/p, H, D]; after the
// forward exchange it holds the whole sequence of head group r, [S, H/p, D]:
//   y_r[s * S/p + t, h, :] = x_s[t, r * H/p + h, :].
// The inverse exchange maps back.  A token row of a shard (H * D elements) is
// p contiguous segments of (H/p) * D elements, segment d going to rank d.  A
// CTA takes a block of token rows of one shard: thread x walks the row's
// 16-byte vectors o = x, x + blockDim.x, ...; the vector's segment d and
// offset e in it are worked out once per o and serve every row, and the
// rows (threadIdx.y + u * blockDim.y) are loaded together, kRows at a time,
// before they are stored -- a pure copy, bit-exact, with both sides read or
// written in runs of whole segments.
#include "device_common.cuh"

namespace ccl {
namespace {

constexpr int kRows = 8;  // rows per thread, loads in flight

template <int DT, int VEC>
__global__ void __launch_bounds__(kThreads) ulysses_kernel(const __grid_constant__ UlyssesArgs a) {
  constexpr int W = (VEC * Elem<DT>::kBytes + 3) / 4;
  pdl_enter();
  const uint64_t sp = a.seq_per_rank;
  const uint64_t R = a.heads * a.head_dim / VEC;             // vectors per shard row
  const uint64_t G = (a.heads / a.p) * a.head_dim / VEC;     // vectors per segment
  const uint64_t s = blockIdx.y;                              // sequence shard
  const uint64_t rows_per_cta = static_cast<uint64_t>(blockDim.y) * kRows;
  const uint64_t t0 = blockIdx.x * rows_per_cta + threadIdx.y;
  for (uint64_t o = threadIdx.x; o < R; o += blockDim.x) {
    const uint64_t d = o / G, e = o - d * G;
    // element offsets of row t0: in the [S/p, H, D] shard and in rank d's [S, H/p, D] group
    const uint64_t shard0 = (t0 * R + o) * VEC;
    const uint64_t group0 = ((s * sp + t0) * G + e) * VEC;
    const void* src = a.inverse ? a.x[d] : a.x[s];
    void* dst = a.inverse ? a.y[s] : a.y[d];
    const uint64_t src0 = a.inverse ? group0 : shard0, dst0 = a.inverse ? shard0 : group0;
    const uint64_t src_step = (a.inverse ? G : R) * VEC * blockDim.y;
    const uint64_t dst_step = (a.inverse ? R : G) * VEC * blockDim.y;
    uint32_t w[kRows][W];
#pragma unroll
    for (int u = 0; u < kRows; ++u)
      if (t0 + static_cast<uint64_t>(u) * blockDim.y < sp) load_raw<DT, VEC>(src, src0 + u * src_step, w[u]);
#pragma unroll
    for (int u = 0; u < kRows; ++u)
      if (t0 + static_cast<uint64_t>(u) * blockDim.y < sp) store_raw<DT, VEC>(dst, dst0 + u * dst_step, w[u]);
  }
}

template <int DT, int VEC>
cudaError_t launch_one(const UlyssesArgs& a, cudaStream_t s) {
  const uint64_t R = a.heads * a.head_dim / VEC;
  // x covers the row's vectors (whole warps), y the rows that fit beside them
  unsigned bx = kThreads;
  if (R < kThreads) bx = static_cast<unsigned>((R + 31) / 32 * 32);
  const unsigned by = kThreads / bx;
  const uint64_t rows_per_cta = static_cast<uint64_t>(by) * kRows;
  const uint64_t gx = (a.seq_per_rank + rows_per_cta - 1) / rows_per_cta;
  if (gx > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  return launch_kernel(ulysses_kernel<DT, VEC>, dim3(static_cast<unsigned>(gx), a.p), dim3(bx, by), s, a);
}

}  // namespace

cudaError_t launch_ulysses(int dt, bool vec, const UlyssesArgs& a, cudaStream_t s) {
  cudaError_t err = cudaErrorInvalidValue;
  if (dt == kF32 || dt == kI32) err = vec ? launch_one<kF32, 4>(a, s) : launch_one<kF32, 1>(a, s);
  else if (dt == kBF16) err = vec ? launch_one<kBF16, 8>(a, s) : launch_one<kBF16, 1>(a, s);
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace ccl
