// ulysses.cu -- the head <-> sequence all-to-all of sequence-parallel attention
// ("LLM Distributed Training Collectives", Sequence Parallelism / Ulysses: long
// sequences are split across devices, and attention needs an all-to-all that
// re-partitions the data by head).
//
// Rank r holds sequence shard r with every head, [S/p, H, D]; after the
// forward exchange it holds the whole sequence of head group r, [S, H/p, D]:
//   y_r[s * S/p + t, h, :] = x_s[t, r * H/p + h, :].
// The inverse exchange maps back.  Both are p * p * (S/p) contiguous segments
// of (H/p) * D elements; one 1-D grid strides over the 16-byte vectors of all
// segments (4 per thread in flight) -- a pure copy, bit-exact.
#include "device_common.cuh"

namespace ccl {
namespace {

constexpr int kUnroll = 4;

// Source and destination byte addresses of element offset `i` (in vectors of
// VEC elements) of segment `g`.
template <int DT>
__device__ __forceinline__ void segment_ends(const UlyssesArgs& a, uint64_t g, const char** src,
                                             char** dst) {
  constexpr int B = Elem<DT>::kBytes;
  const uint64_t sp = a.seq_per_rank, hp = a.heads / a.p, D = a.head_dim;
  const uint64_t t = g % sp;            // token within the shard
  const uint64_t pair = g / sp;
  const uint64_t d = pair % a.p;        // head group / destination rank
  const uint64_t s = pair / a.p;        // sequence shard / source rank
  const uint64_t shard_off = (t * a.heads + d * hp) * D;  // in the [S/p, H, D] shard
  const uint64_t group_off = ((s * sp + t) * hp) * D;     // in the [S, H/p, D] head group
  if (!a.inverse) {
    *src = static_cast<const char*>(a.x[s]) + shard_off * B;
    *dst = static_cast<char*>(a.y[d]) + group_off * B;
  } else {
    *src = static_cast<const char*>(a.x[d]) + group_off * B;
    *dst = static_cast<char*>(a.y[s]) + shard_off * B;
  }
}

template <int DT, int VEC>
__global__ void __launch_bounds__(kThreads) ulysses_kernel(const __grid_constant__ UlyssesArgs a) {
  constexpr int W = (VEC * Elem<DT>::kBytes + 3) / 4;
  pdl_enter();
  const uint64_t L = (a.heads / a.p) * a.head_dim;  // elements per segment
  const uint64_t vps = L / VEC;                      // vectors per segment
  const uint64_t total = a.segments * vps;
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * kUnroll;
  for (uint64_t base = static_cast<uint64_t>(blockIdx.x) * kSpan; base < total;
       base += static_cast<uint64_t>(gridDim.x) * kSpan) {
    uint32_t w[kUnroll][W];
    char* dst[kUnroll];
    uint64_t off[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
      dst[u] = nullptr;
      if (v < total) {
        const char* src;
        segment_ends<DT>(a, v / vps, &src, &dst[u]);
        off[u] = (v % vps) * VEC;
        load_raw<DT, VEC>(src, off[u], w[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (dst[u] != nullptr) store_raw<DT, VEC>(dst[u], off[u], w[u]);
  }
}

template <int DT, int VEC>
cudaError_t launch_one(const UlyssesArgs& a, cudaStream_t s) {
  const uint64_t L = (a.heads / a.p) * a.head_dim;
  const uint64_t total = a.segments * (L / VEC);
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * kUnroll;
  uint64_t gx = (total + kSpan - 1) / kSpan;
  if (gx < 1) gx = 1;
  if (gx > (1u << 30)) gx = 1u << 30;
  return launch_kernel(ulysses_kernel<DT, VEC>, dim3(static_cast<unsigned>(gx)), dim3(kThreads), s, a);
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
