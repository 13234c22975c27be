// a2av.cu -- all-to-all(v) block transpose: MoE dispatch / combine
// ("Networks and Collective Communication" section 4.1: device i's block j
// goes to device j, a transpose; section 7.4: MoE dispatch and combine).
//
// The host turns the p x p row counts into a list of contiguous byte blocks
// (source s's block for d -> destination d's block from s).  Blocks are cut
// into 32 KB tiles measured in destination space, and one CTA copies one
// tile, so the work is balanced by bytes however skewed the counts are (a
// Zipf-hot expert receives far more rows than the others).
//
// Inside a tile, whole 16-byte destination units are copied with 16-byte
// loads and stores.  When source and destination differ in 16-byte phase
// (rows whose size is not a multiple of 16 bytes), each lane of a warp loads
// the aligned 16-byte source granule under its unit, takes the next granule
// from its neighbour with a warp shuffle, and funnel-shifts the pair into the
// destination's alignment; the few bytes before the first and after the last
// whole unit are copied one by one.  Every load touches only aligned granules
// that hold at least one source byte of the block.
// HBM traffic: one read and one write of every moved byte.
#include "device_common.cuh"
#include "realign.cuh"

namespace ccl {
namespace {

constexpr int kUnitsPerThread = static_cast<int>(kA2ATileBytes / 16 / kThreads);  // 8

__device__ __forceinline__ void copy_byte(uintptr_t dst, intptr_t shift) {
  const unsigned char b = __ldg(reinterpret_cast<const unsigned char*>(dst + shift));
  *reinterpret_cast<unsigned char*>(dst) = b;
}

// Copy destination bytes [lo, hi); the source byte of destination byte x is
// x + shift.  Called by all threads of the CTA with the same arguments.
// REALIGN = false is launched only when every block of the call has source
// and destination in the same 16-byte phase; it leaves out the realigning
// path and its registers (64 against 128), and any other phase would still
// be copied correctly, byte by byte.
template <bool REALIGN>
__device__ void copy_tile(uintptr_t lo, uintptr_t hi, intptr_t shift) {
  const int tid = threadIdx.x;
  const uintptr_t ua = (lo + 15) & ~static_cast<uintptr_t>(15);
  const uintptr_t ub = hi & ~static_cast<uintptr_t>(15);
  if (ua >= ub) {  // no whole destination unit: byte by byte
    for (uintptr_t x = lo + tid; x < hi; x += kThreads) copy_byte(x, shift);
    return;
  }
  // Units are counted from ua rounded down to 512 bytes, so that every warp's
  // 32 stores fill a whole 512-byte span (whole 128-byte lines); the units
  // before ua (u < u_first) stay idle.
  const uintptr_t uo = ua & ~static_cast<uintptr_t>(511);
  const uint64_t u_first = (ua - uo) / 16;
  const uint64_t m = (ub - uo) / 16;  // one past the last whole 16-byte destination unit
  const int delta = static_cast<int>(static_cast<uintptr_t>(shift) & 15);
  if (!REALIGN && delta != 0) {
    for (uintptr_t x = lo + tid; x < hi; x += kThreads) copy_byte(x, shift);
    return;
  }
  if (delta == 0) {
    for (uint64_t u0 = 0; u0 < m; u0 += static_cast<uint64_t>(kThreads) * kUnitsPerThread) {
      uint4 v[kUnitsPerThread];
#pragma unroll
      for (int j = 0; j < kUnitsPerThread; ++j) {
        const uint64_t u = u0 + static_cast<uint64_t>(j) * kThreads + tid;
        if (u >= u_first && u < m) v[j] = ld_once16(reinterpret_cast<const void*>(uo + 16 * u + shift));
      }
#pragma unroll
      for (int j = 0; j < kUnitsPerThread; ++j) {
        const uint64_t u = u0 + static_cast<uint64_t>(j) * kThreads + tid;
        if (u >= u_first && u < m) st_stream16(reinterpret_cast<void*>(uo + 16 * u), v[j]);
      }
    }
  } else if constexpr (REALIGN) {
    const int lane = tid & 31;
    const int warp = tid >> 5;
    // source granule under unit u: uo + 16u + shift - delta (16-byte aligned).
    // A warp takes 32 consecutive units per group, kUnitsPerThread groups
    // (kThreads units apart) with their loads issued together.
    const uintptr_t g0 = uo + shift - delta;
    for (uint64_t k0 = static_cast<uint64_t>(warp) * 32; k0 < m;
         k0 += static_cast<uint64_t>(kThreads) * kUnitsPerThread) {
      uint4 cur[kUnitsPerThread], extra[kUnitsPerThread];
#pragma unroll
      for (int j = 0; j < kUnitsPerThread; ++j) {
        const uint64_t u = k0 + static_cast<uint64_t>(j) * kThreads + lane;
        cur[j] = make_uint4(0, 0, 0, 0);
        extra[j] = make_uint4(0, 0, 0, 0);
        // granule u holds bytes of unit u (u < m) or the last bytes of unit u-1 (u == m)
        if (u >= u_first && u <= m) cur[j] = ld_once16(reinterpret_cast<const void*>(g0 + 16 * u));
        if (lane == 31 && u >= u_first && u < m)
          extra[j] = ld_once16(reinterpret_cast<const void*>(g0 + 16 * (u + 1)));
      }
#pragma unroll
      for (int j = 0; j < kUnitsPerThread; ++j) {
        const uint64_t u = k0 + static_cast<uint64_t>(j) * kThreads + lane;
        const uint4 nxt = next_lane(cur[j], extra[j], lane);
        if (u >= u_first && u < m)
          st_stream16(reinterpret_cast<void*>(uo + 16 * u), realign16(cur[j], nxt, delta));
      }
    }
  }
  // bytes before the first and after the last whole unit (at most 15 + 15)
  const int n_head = static_cast<int>(ua - lo);
  const int n_edge = n_head + static_cast<int>(hi - ub);
  if (tid < n_edge) copy_byte(tid < n_head ? lo + tid : ub + (tid - n_head), shift);
}

template <int CAP, bool REALIGN>
__global__ void __launch_bounds__(kThreads) a2av_kernel(const __grid_constant__ A2AArgsT<CAP> a) {
  pdl_enter();
  for (uint64_t t = blockIdx.x; t < a.total_tiles; t += gridDim.x) {
    // the block that owns tile t: the last one whose first tile is <= t
    int lo = 0, hi = a.ndesc - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.d[mid].tile0 <= t) lo = mid; else hi = mid - 1;
    }
    const A2ADesc& d = a.d[lo];
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(d.dst);
    const uintptr_t d_end = d0 + d.bytes;
    const uintptr_t base = d0 & ~static_cast<uintptr_t>(511);  // tiles on 512-byte boundaries
    const uint64_t k = t - d.tile0;
    uintptr_t tlo = base + k * kA2ATileBytes;
    uintptr_t thi = tlo + kA2ATileBytes;
    if (tlo < d0) tlo = d0;
    if (thi > d_end) thi = d_end;
    const intptr_t shift = reinterpret_cast<intptr_t>(d.src) - reinterpret_cast<intptr_t>(d.dst);
    copy_tile<REALIGN>(tlo, thi, shift);
  }
}

}  // namespace

uint64_t a2a_tiles_for(const char* dst, uint64_t bytes) {
  if (bytes == 0) return 0;
  const uint64_t lead = reinterpret_cast<uintptr_t>(dst) & 511;  // tiles start on 512-byte boundaries
  return (lead + bytes + kA2ATileBytes - 1) / kA2ATileBytes;
}

cudaError_t launch_a2av(const A2AArgs& a, cudaStream_t s) {
  if (a.total_tiles == 0 || a.ndesc == 0) return cudaSuccess;
  uint64_t g = a.total_tiles;
  if (g > (1u << 30)) g = 1u << 30;
  const dim3 grid(static_cast<unsigned>(g));
  bool phased = false;  // some block's source and destination differ in 16-byte phase
  for (int i = 0; i < a.ndesc && !phased; ++i)
    phased = ((reinterpret_cast<uintptr_t>(a.d[i].src) - reinterpret_cast<uintptr_t>(a.d[i].dst)) & 15) != 0;
  cudaError_t err;
  if (a.ndesc <= kA2ASmallDesc) {  // the common case: a 4 KB parameter block
    A2AArgsT<kA2ASmallDesc> small;
    small.total_tiles = a.total_tiles;
    small.ndesc = a.ndesc;
    for (int i = 0; i < a.ndesc; ++i) small.d[i] = a.d[i];
    err = phased ? launch_kernel(a2av_kernel<kA2ASmallDesc, true>, grid, dim3(kThreads), s, small)
                 : launch_kernel(a2av_kernel<kA2ASmallDesc, false>, grid, dim3(kThreads), s, small);
  } else {
    err = phased ? launch_kernel(a2av_kernel<kA2AMaxDesc, true>, grid, dim3(kThreads), s, a)
                 : launch_kernel(a2av_kernel<kA2AMaxDesc, false>, grid, dim3(kThreads), s, a);
  }
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace ccl
