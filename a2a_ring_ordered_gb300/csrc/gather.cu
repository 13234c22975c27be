// gather.cu -- all-gather: rank k's block is copied to offset off(k) of every
// rank's output ("Networks and Collective Communication" section 4.1: each
// device contributes one block and everyone gets the whole concatenation).
//
// The ring's all-gather phase forwards each finished chunk p-1 times; on one
// GPU the same result is one read of block k and p writes of it.  Grid:
// blockIdx.y = block k; vectors are aligned in output space, and the source
// side uses 16-byte loads too whenever off(k) keeps it aligned.
// HBM traffic: n reads + p*n writes of the element type.
#include "device_common.cuh"
#include "realign.cuh"

namespace ccl {
namespace {

// Load VEC elements one at a time into packed raw words (unaligned source).
template <int DT, int VEC>
__device__ __forceinline__ void load_elems(const void* base, uint64_t i, uint32_t* w) {
  constexpr int B = Elem<DT>::kBytes;
  if constexpr (B == 4) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) load_raw<DT, 1>(base, i + e, &w[e]);
  } else {
#pragma unroll
    for (int e = 0; e < VEC; e += 2) {
      uint32_t lo, hi;
      load_raw<DT, 1>(base, i + e, &lo);
      load_raw<DT, 1>(base, i + e + 1, &hi);
      w[e >> 1] = (lo & 0xFFFFu) | (hi << 16);
    }
  }
}

// REALIGN = false is launched only when every block starts on a whole vector
// of the outputs, and leaves the realigning path out.
template <int DT, int VEC, int U, bool REALIGN>
__global__ void __launch_bounds__(kThreads) gather_kernel(const __grid_constant__ GatherArgs a) {
  constexpr int W = (VEC * Elem<DT>::kBytes + 3) / 4;
  const int p = a.p;
  const int k = blockIdx.y;
  const Chunk ch = chunk_of(k, a.q, a.rem);
  const uint64_t end = ch.off + ch.len;
  const uint64_t v_lo = (ch.off + VEC - 1) / VEC;
  const uint64_t v_hi = end / VEC;
  const void* src = a.send[k];
  if (VEC > 1 && cta_rank() < a.pf_ctas) {  // this CTA's first source bytes, before waiting on the previous grid
    constexpr uint64_t kSpan0 = static_cast<uint64_t>(kThreads) * U;
    uint64_t b0 = (REALIGN ? (v_lo & ~static_cast<uint64_t>(31)) : v_lo) + static_cast<uint64_t>(blockIdx.x) * kSpan0;
    uint64_t e0 = b0 + kSpan0;
    b0 = b0 > v_lo ? b0 : v_lo;
    e0 = e0 < v_hi ? e0 : v_hi;
    if (b0 < e0) {
      constexpr uint64_t B = Elem<DT>::kBytes;
      prefetch_spans_l2(&src, 1, (b0 * VEC - ch.off) * B, (e0 - b0) * VEC * B);
    }
  }
  pdl_enter();
  const bool src_aligned = (ch.off % VEC) == 0;
  // Block k unaligned in the outputs (off(k) not a multiple of VEC): output
  // vector v takes the source bytes [((v - q) * VEC - s) * B, + 16), i.e.
  // aligned source granule v - q - 1 from byte `phase` on, continued in
  // granule v - q, which the next lane loads (s = off(k) mod VEC, q = off(k)
  // div VEC).  Every granule loaded holds at least one byte of block k.
  const uint64_t q = ch.off / VEC;
  const int phase = 16 - static_cast<int>(ch.off % VEC) * Elem<DT>::kBytes;
  const int lane = threadIdx.x & 31;
  // With REALIGN (blocks off the output vectors) vectors are counted from
  // v_lo rounded down to 32, so that every warp's 32 stores fill whole
  // 512-byte spans (whole 128-byte lines) of each output; lanes before v_lo
  // (the previous block's) stay idle.  Measured on GB300: the p = 72 bf16
  // all-gather 0.85 -> 0.99 of the copy bandwidth.  The aligned kernel keeps
  // v_lo: with the extra guards it compiled to 64 registers instead of 77
  // (4 CTAs per SM instead of 3) and ran the p = 16 all-gather 4 % slower.
  const uint64_t v_start = REALIGN ? (v_lo & ~static_cast<uint64_t>(31)) : v_lo;

  // U vectors per thread (t, t + kThreads, ...): their loads are issued
  // together, then each is stored to the p outputs
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * U;
  for (uint64_t base = v_start + static_cast<uint64_t>(blockIdx.x) * kSpan; base < v_hi;
       base += static_cast<uint64_t>(gridDim.x) * kSpan) {
    uint32_t w[U][W];
    if constexpr (!REALIGN || VEC == 1) {
      // (REALIGN = false is not launched with a block off the output vectors;
      // the element-wise loads are there so that no load could be misaligned)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
        if ((!REALIGN || v >= v_lo) && v < v_hi) {
          if (VEC == 1 || src_aligned) {
            load_raw<DT, VEC>(src, v * VEC - ch.off, w[u]);
          } else {
            load_elems<DT, VEC>(src, v * VEC - ch.off, w[u]);
          }
        }
      }
    } else if (src_aligned) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
        if (v >= v_lo && v < v_hi) load_raw<DT, VEC>(src, v * VEC - ch.off, w[u]);
      }
    } else {
      const char* g = static_cast<const char*>(src);
      uint4 cur[U], extra[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
        cur[u] = make_uint4(0, 0, 0, 0);
        extra[u] = make_uint4(0, 0, 0, 0);
        if (v >= v_lo && v <= v_hi) cur[u] = ld_once16(g + 16 * (v - q - 1));
        if (lane == 31 && v >= v_lo && v < v_hi) extra[u] = ld_once16(g + 16 * (v - q));
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint4 o = realign16(cur[u], next_lane(cur[u], extra[u], lane), phase);
        w[u][0] = o.x;
        w[u][1] = o.y;
        w[u][2] = o.z;
        w[u][3] = o.w;
      }
    }
    for (int r = 0; r < p; ++r) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
        if ((!REALIGN || v >= v_lo) && v < v_hi) store_raw<DT, VEC>(a.recv[r], v * VEC, w[u]);
      }
    }
  }

  if (VEC > 1 && blockIdx.x == 0) {
    const uint64_t head_end = (v_lo * VEC < end) ? v_lo * VEC : end;
    const uint64_t tail_begin = (v_hi * VEC > head_end) ? v_hi * VEC : head_end;
    const uint64_t n_head = head_end - ch.off;
    const uint64_t n_edge = n_head + (end - tail_begin);
    for (uint64_t t = threadIdx.x; t < n_edge; t += kThreads) {
      const uint64_t i = (t < n_head) ? ch.off + t : tail_begin + (t - n_head);
      uint32_t w[1];
      load_raw<DT, 1>(src, i - ch.off, w);
      for (int r = 0; r < p; ++r) store_raw<DT, 1>(a.recv[r], i, w);
    }
  }
}

template <int DT, int VEC, int U>
cudaError_t launch_one(const GatherArgs& a, cudaStream_t s) {
  const uint64_t per_chunk = (a.q + 1 + VEC - 1) / VEC + 31;  // + the lanes before v_lo
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * U;
  uint64_t gx = (per_chunk + kSpan - 1) / kSpan;
  if (gx < 1) gx = 1;
  if (gx > (1u << 30)) gx = 1u << 30;
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(a.p));
  bool realign = false;  // some block starts inside a vector of the outputs
  for (uint64_t k = 0; k < static_cast<uint64_t>(a.p) && VEC > 1 && !realign; ++k)
    realign = (k * a.q + (k < a.rem ? k : a.rem)) % VEC != 0;  // off(k), the chunk rule
  if (realign) return launch_kernel(gather_kernel<DT, VEC, U, true>, grid, dim3(kThreads), s, a);
  return launch_kernel(gather_kernel<DT, VEC, U, false>, grid, dim3(kThreads), s, a);
}

template <int DT>
cudaError_t launch_typed(bool vec, const GatherArgs& a, cudaStream_t s) {
  // 8 vectors (128 bytes) of loads in flight per thread before its p x 8
  // stores: at p = 16 that is 0.977 -> 1.022 of the copy bandwidth over 4
  // vectors, 8 outrunning 2 and 4 and matching 32-byte stores.  Two
  // exceptions, measured on GB300 (fraction of the copy bandwidth):
  //  * Mid-size calls whose grid would be under 8 CTAs per SM take fewer
  //    vectors per thread, as the fold kernels do: 1 while that grid stays
  //    within 20 CTAs per SM (2.5 waves of this 32-register kernel), else 2
  //    (2 vectors -> 1: p = 2 at 4 / 8 MiB per rank 0.66 -> 0.72 / 0.75 ->
  //    0.82, p = 8 at 4 / 8 MiB 0.64 -> 0.90 / 0.84 -> 0.88; at 16 MiB p = 2
  //    keeps 2, 0.94 against 0.91).  From p = 8 on, where every loaded
  //    vector is stored 8 times or more, 1 at any mid size (16 MiB, 2
  //    vectors -> 1: p = 8 0.91-0.93 -> 0.94, p = 16 0.93-0.95 -> 0.96,
  //    p = 32 0.96 -> 0.99, p = 72 0.95 -> 1.00).
  //  * From p = 8 on, blocks off the output vectors (the realigning kernel,
  //    whose two granules per vector cost registers) take 1 vector at every
  //    size: p = 72 at 64 / 256 MiB 0.98 / 0.98 -> 1.01 / 1.03, p = 48 0.98
  //    / 0.96 -> 1.01 / 1.02 against 8.  Aligned blocks keep 8 (p = 32 at
  //    64 MiB 1.06 against 0.99-1.01 with 1).
  if (!vec) return launch_one<DT, 1, 1>(a, s);
  constexpr int VEC = 16 / Elem<DT>::kBytes;
  const uint64_t per_chunk = (a.q + 1 + VEC - 1) / VEC;
  const int sms = current_sm_count();
  const uint64_t sm_count = static_cast<uint64_t>(sms > 0 ? sms : 1);
  auto ctas = [&](uint64_t u) { return (per_chunk + kThreads * u - 1) / (kThreads * u) * static_cast<uint64_t>(a.p); };
  const bool many = a.p >= 8;
  if (ctas(8) >= 8 * sm_count) {
    bool realign = false;  // some block starts inside a vector of the outputs
    for (uint64_t k = 0; k < static_cast<uint64_t>(a.p) && !realign; ++k)
      realign = (k * a.q + (k < a.rem ? k : a.rem)) % VEC != 0;  // off(k), the chunk rule
    if (many && realign) return launch_one<DT, VEC, 1>(a, s);
    return launch_one<DT, VEC, 8>(a, s);
  }
  if (many || ctas(1) <= 20 * sm_count) return launch_one<DT, VEC, 1>(a, s);
  return launch_one<DT, VEC, 2>(a, s);
}

// Broadcast: one 1-D pass over the root's buffer (send[0]); each of a
// thread's U vectors is loaded once and stored to all p outputs.
template <int DT, int VEC, int U>
__global__ void __launch_bounds__(kThreads) broadcast_kernel(const __grid_constant__ GatherArgs a,
                                                             uint64_t n) {
  constexpr int W = (VEC * Elem<DT>::kBytes + 3) / 4;
  pdl_enter();
  const int p = a.p;
  const void* src = a.send[0];
  const uint64_t nv = n / VEC;
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * U;
  for (uint64_t base = static_cast<uint64_t>(blockIdx.x) * kSpan; base < nv;
       base += static_cast<uint64_t>(gridDim.x) * kSpan) {
    uint32_t w[U][W];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
      if (v < nv) load_raw<DT, VEC>(src, v * VEC, w[u]);
    }
    for (int r = 0; r < p; ++r) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
        if (v < nv) store_raw<DT, VEC>(a.recv[r], v * VEC, w[u]);
      }
    }
  }
  if (blockIdx.x == 0) {  // tail elements
    for (uint64_t i = nv * VEC + threadIdx.x; i < n; i += kThreads) {
      uint32_t w[1];
      load_raw<DT, 1>(src, i, w);
      for (int r = 0; r < p; ++r) store_raw<DT, 1>(a.recv[r], i, w);
    }
  }
}

template <int DT, int VEC, int U>
cudaError_t launch_bcast(const GatherArgs& a, uint64_t n, cudaStream_t s) {
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
  return cudaLaunchKernelEx(&cfg, broadcast_kernel<DT, VEC, U>, a, n);
}

// 8 vectors per thread when that grid has 4 CTAs per SM or more; below it,
// 1 when the one-vector grid still fills a wave of this kernel (8 CTAs per
// SM), else 2.  Measured on GB300 (fp32, fraction of the copy bandwidth,
// 8 vectors -> this rule): p = 4 / 16 / 72 at 2 MiB 0.49 / 0.56 / 0.56 ->
// 0.76 / 0.96 / 0.94, p = 16 / 72 at 8 MiB 0.96 / 0.97 -> 0.95 / 1.00; from
// 32 MiB the vector counts came out within 2 % of one another.
template <int DT, int VEC>
cudaError_t launch_bcast_vec(const GatherArgs& a, uint64_t n, cudaStream_t s) {
  const uint64_t nv = n / VEC;
  const int sms = current_sm_count();
  const uint64_t sm_count = static_cast<uint64_t>(sms > 0 ? sms : 1);
  auto ctas = [&](uint64_t u) { return (nv + kThreads * u - 1) / (kThreads * u); };
  if (ctas(8) >= 4 * sm_count) return launch_bcast<DT, VEC, 8>(a, n, s);
  if (ctas(1) >= 8 * sm_count) return launch_bcast<DT, VEC, 1>(a, n, s);
  return launch_bcast<DT, VEC, 2>(a, n, s);
}

}  // namespace

cudaError_t launch_broadcast(int dt, bool vec, const GatherArgs& a, uint64_t n, cudaStream_t s) {
  cudaError_t err = cudaErrorInvalidValue;
  if (dt == kF32 || dt == kI32) {
    err = vec ? launch_bcast_vec<kF32, 4>(a, n, s) : launch_bcast<kF32, 1, 1>(a, n, s);
  } else if (dt == kBF16) {
    err = vec ? launch_bcast_vec<kBF16, 8>(a, n, s) : launch_bcast<kBF16, 1, 1>(a, n, s);
  }
  if (err == cudaSuccess) note_launch();
  return err;
}

cudaError_t launch_gather(int dt, bool vec, const GatherArgs& a, cudaStream_t s) {
  cudaError_t err = cudaErrorInvalidValue;
  // a copy only needs the element width: fp32 and int32 share one kernel
  if (dt == kF32 || dt == kI32) err = launch_typed<kF32>(vec, a, s);
  else if (dt == kBF16) err = launch_typed<kBF16>(vec, a, s);
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace ccl
