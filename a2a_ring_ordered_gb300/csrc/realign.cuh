// realign.cuh -- moving 16-byte vectors between buffers whose 16-byte phases
// differ, with whole aligned loads and stores on both sides.
//
// A warp whose lanes hold consecutive aligned 16-byte granules of one side
// forms the other side's aligned vectors from two neighbouring granules: lane
// l takes granule l + 1 from its neighbour with a warp shuffle and funnel-
// shifts the 32-byte pair by the phase difference.  Used where a block starts
// at an offset that is not a multiple of 16 bytes: the all-gather's blocks
// (source aligned, destination not), the reduce-scatter's shards (the folded
// input vectors aligned, the shard not) and the all-to-allv's rows.
#pragma once

#include <cstdint>

#include "device_common.cuh"

namespace ccl {

// Bytes [delta, delta + 16) of the 32-byte pair (lo, hi), little-endian;
// 0 <= delta < 16.
__device__ __forceinline__ uint4 realign16(const uint4 lo, const uint4 hi, int delta) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const uint32_t sh = 8u * static_cast<uint32_t>(delta & 3);
  uint4 o;
#define CCL_REALIGN(Q)                             \
  o.x = __funnelshift_r(w[Q + 0], w[Q + 1], sh);   \
  o.y = __funnelshift_r(w[Q + 1], w[Q + 2], sh);   \
  o.z = __funnelshift_r(w[Q + 2], w[Q + 3], sh);   \
  o.w = __funnelshift_r(w[Q + 3], w[Q + 4], sh);
  switch (delta >> 2) {
    case 0: CCL_REALIGN(0) break;
    case 1: CCL_REALIGN(1) break;
    case 2: CCL_REALIGN(2) break;
    default: CCL_REALIGN(3) break;
  }
#undef CCL_REALIGN
  return o;
}

// The next lane's granule (lane 31 gets `own_next`, which it loaded itself).
__device__ __forceinline__ uint4 next_lane(const uint4 v, const uint4 own_next, int lane) {
  uint4 n;
  n.x = __shfl_down_sync(0xFFFFFFFFu, v.x, 1);
  n.y = __shfl_down_sync(0xFFFFFFFFu, v.y, 1);
  n.z = __shfl_down_sync(0xFFFFFFFFu, v.z, 1);
  n.w = __shfl_down_sync(0xFFFFFFFFu, v.w, 1);
  return lane == 31 ? own_next : n;
}

// Reduce-scatter shard store when the chunk's offset `off` is not a multiple
// of VEC (VEC * bytes == 16).  All 32 lanes of the warp call it together;
// lane l holds the packed outputs w of input vector v = v0 + l (elements
// [v * VEC, v * VEC + VEC) of the chunk, valid when v_lo <= v < v_hi).
// Element t of lane v lands at shard position (v - q) * VEC - s + t (q = off
// div VEC, s = off mod VEC), so shard vector J = v - q is lane v's elements
// [s, VEC) followed by lane v + 1's [0, s): the lane stores it whole when its
// neighbour is in the warp and valid.  Lane 31 and the last valid lane store
// their elements [s, VEC) one by one, lane 0 and the first valid lane their
// elements [0, s); the chunk's own head and tail edges are left to the
// element-wise edge path.
template <int DT_OUT, int VEC>
__device__ __forceinline__ void store_shard_realigned(void* shard, uint64_t off, uint64_t v, uint64_t v_lo,
                                                      uint64_t v_hi, int lane, const uint32_t* w) {
  static_assert(VEC * Elem<DT_OUT>::kBytes == 16, "one 16-byte vector per lane");
  const uint4 own = make_uint4(w[0], w[1], w[2], w[3]);
  const uint4 nxt = next_lane(own, own, lane);
  if (v < v_lo || v >= v_hi) return;
  const int s = static_cast<int>(off % VEC);
  const uint64_t J = v - off / VEC;
  const bool whole = lane < 31 && v + 1 < v_hi;
  const bool first = lane == 0 || v == v_lo;
  if (whole) st_stream16(static_cast<char*>(shard) + J * 16, realign16(own, nxt, s * Elem<DT_OUT>::kBytes));
  // element t lands at J * VEC - s + t (t fixed per unrolled step, so w stays in registers)
#pragma unroll
  for (int t = 0; t < VEC; ++t) {
    if ((t >= s && !whole) || (t < s && first)) store_one<DT_OUT>(shard, J * VEC - s + t, w, t);
  }
}

}  // namespace ccl
