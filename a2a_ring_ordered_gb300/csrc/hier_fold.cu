// hier_fold.cu -- all-reduce in the fold order of the hierarchical (two-level
// ring) all-reduce.
//
// "Networks and Collective Communication" section 6.3: with p = a * b devices
// in b nodes of a GPUs, a ring reduce-scatter inside every node, a ring
// all-reduce across the nodes among the GPUs with the same index inside their
// node, and a ring all-gather inside every node.  Section 6.1's
// two-dimensional all-reduce (reduce-scatter along the rows of an a x b grid,
// then along the columns, then the all-gathers in reverse) folds the same way.
//
// Groups are runs of a consecutive ranks (group g = ranks g*a .. g*a + a - 1).
// The buffer is cut into a chunks (chunk rule), chunk l into b sub-chunks
// (chunk rule again).  An element of sub-chunk (l, m) is first folded inside
// every group along that group's ring starting at local rank l + 1 and ending
// at l, then the b group partials are folded along the ring over the groups
// starting at group m + 1 and ending at m -- in fp32 (int32) throughout, bf16
// rounded once at the end.  As in the flat ring kernel, one thread performs
// the whole walk of one 16-byte vector in registers and writes the result to
// every rank: p reads and p writes per element, the all-reduce's minimum.
//
// Grid: blockIdx.y = l * b + m, so both starting points are uniform per CTA;
// blockIdx.x strides over the sub-chunk's aligned vectors; CTA (0, y) folds
// the sub-chunk's unaligned edges element by element.
#include "device_common.cuh"

namespace ccl {
namespace {


// Fold VEC elements at element i: rank sequence (group g0, local l0), then the
// rest of that group's ring, then the next group, ...; BATCH loads in flight.
template <int DT, int VEC, int BATCH>
__device__ __forceinline__ void fold_two_level(const FoldArgs& f, int a, int b, int g0, int l0,
                                               uint64_t i, typename Elem<DT>::Acc* tot) {
  using Acc = typename Elem<DT>::Acc;
  constexpr int W = (VEC * Elem<DT>::kBytes + 3) / 4;
  const int p = f.p;
  Acc part[VEC];
  int g = g0, loc = l0;  // next rank to load
  int li = 0;            // position of the next folded value inside its group's ring
  bool first_group = true;
  for (int k0 = 0; k0 < p; k0 += BATCH) {
    uint32_t raw[BATCH][W];
#pragma unroll
    for (int j = 0; j < BATCH; ++j) {
      if (k0 + j < p) {
        load_raw<DT, VEC>(f.send[g * a + loc], i, raw[j]);
        if (++loc == a) loc = 0;
        if (loc == l0) g = (g + 1 == b) ? 0 : g + 1;  // that group's ring is complete
      }
    }
#pragma unroll
    for (int j = 0; j < BATCH; ++j) {
      if (k0 + j < p) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const Acc x = widen<DT>(raw[j], e);
          part[e] = (li == 0) ? x : combine<CCL_SUM>(part[e], x);
        }
        if (++li == a) {  // group partial done: fold it into the ring over the groups
#pragma unroll
          for (int e = 0; e < VEC; ++e) tot[e] = first_group ? part[e] : combine<CCL_SUM>(tot[e], part[e]);
          first_group = false;
          li = 0;
        }
      }
    }
  }
}

template <int DT, int VEC>
__device__ __forceinline__ void write_all(const FoldArgs& f, uint64_t i, typename Elem<DT>::Acc* acc) {
  uint32_t w[(VEC * Elem<DT>::kBytes + 3) / 4];
  pack_out<DT, VEC>(acc, w);
  for (int r = 0; r < f.p; ++r) store_raw<DT, VEC>(f.recv[r], i, w);
}

// f.q, f.rem: the level-1 split, floor(n / a) and n mod a.
template <int DT, int VEC, int BATCH>
__global__ void __launch_bounds__(kThreads, 2) hier_fold_kernel(const __grid_constant__ FoldArgs f, int a, int b) {
  using Acc = typename Elem<DT>::Acc;
  pdl_enter();
  const int l = static_cast<int>(blockIdx.y) / b;
  const int m = static_cast<int>(blockIdx.y) - l * b;
  const Chunk c1 = chunk_of(l, f.q, f.rem);
  const Chunk c2 = chunk_of(m, c1.len / b, c1.len % b);
  const uint64_t off = c1.off + c2.off, end = off + c2.len;
  const uint64_t v_lo = (off + VEC - 1) / VEC, v_hi = end / VEC;
  const int l0 = (l + 1 == a) ? 0 : l + 1;
  const int g0 = (m + 1 == b) ? 0 : m + 1;

  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  // counted from v_lo rounded down to 32, so that a warp's 32 stores fill a
  // whole 512-byte span of every output; lanes before v_lo stay idle
  const uint64_t v_start = v_lo & ~static_cast<uint64_t>(31);
  for (uint64_t v = v_start + static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; v < v_hi; v += stride) {
    if (v < v_lo) continue;
    Acc acc[VEC];
    fold_two_level<DT, VEC, BATCH>(f, a, b, g0, l0, v * VEC, acc);
    write_all<DT, VEC>(f, v * VEC, acc);
  }
  if (VEC > 1 && blockIdx.x == 0) {
    const uint64_t head_end = (v_lo * VEC < end) ? v_lo * VEC : end;
    const uint64_t tail_begin = (v_hi * VEC > head_end) ? v_hi * VEC : head_end;
    const uint64_t n_head = head_end - off;
    const uint64_t n_edge = n_head + (end - tail_begin);
    for (uint64_t t = threadIdx.x; t < n_edge; t += kThreads) {
      const uint64_t i = (t < n_head) ? off + t : tail_begin + (t - n_head);
      Acc acc[1];
      fold_two_level<DT, 1, BATCH>(f, a, b, g0, l0, i, acc);
      write_all<DT, 1>(f, i, acc);
    }
  }
}

constexpr int kVectorsPerThread = 2;

template <int DT, int VEC, int BATCH>
cudaError_t launch_one(const FoldArgs& f, int a, cudaStream_t s) {
  const int b = f.p / a;
  const uint64_t longest = (f.q + 1) / static_cast<uint64_t>(b) + 1;  // elements of the largest sub-chunk
  const uint64_t per_sub = (longest + VEC - 1) / VEC + 31;  // + the lanes before v_lo
  uint64_t gx = (per_sub + kThreads * kVectorsPerThread - 1) / (kThreads * kVectorsPerThread);
  if (gx < 1) gx = 1;
  if (gx > (1u << 30)) gx = 1u << 30;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(f.p));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = CCL_PDL ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, hier_fold_kernel<DT, VEC, BATCH>, f, a, b);
}

// Loads in flight per thread: 16 ranks' worth from p = 9 on, 8 below (measured
// on GB300: 16 lifts p = 16 and p = 72 by 2-7 % and costs p = 8 4 %).
template <int DT, int VEC>
cudaError_t launch_batch(const FoldArgs& f, int a, cudaStream_t s) {
  return f.p > 8 ? launch_one<DT, VEC, 16>(f, a, s) : launch_one<DT, VEC, 8>(f, a, s);
}

}  // namespace

cudaError_t launch_hier_fold(int dt, bool vec, const FoldArgs& f, int a, cudaStream_t s) {
  cudaError_t err = cudaErrorInvalidValue;
  if (dt == kF32) err = vec ? launch_batch<kF32, 4>(f, a, s) : launch_batch<kF32, 1>(f, a, s);
  else if (dt == kBF16) err = vec ? launch_batch<kBF16, 8>(f, a, s) : launch_batch<kBF16, 1>(f, a, s);
  else if (dt == kI32) err = vec ? launch_batch<kI32, 4>(f, a, s) : launch_batch<kI32, 1>(f, a, s);
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace ccl
