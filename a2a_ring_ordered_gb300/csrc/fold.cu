// fold.cu -- fused single-pass ring-ordered reduction kernels.
//
// The ring all-reduce ("Networks and Collective Communication" section 5.1;
// "dist_train", Ring Algorithm) moves chunk c's partial sum once around the
// ring, starting at rank c+1 and ending at rank c, then copies the finished
// chunk to every rank.  On one GPU every rank's buffer is in the same HBM, so
// one thread can play the whole walk for its elements: it loads the p ranks'
// values of one 16-byte vector in ring order, folds them in that order in
// fp32 (int32) registers and writes the result once per output.  The fold
// order, and therefore every bit of the result, is the ring's.
//
// Grid: blockIdx.y = chunk c, so the starting rank is uniform per CTA;
// blockIdx.x strides over the chunk's 16-byte-aligned vectors.  The few
// elements of a chunk that do not fill a whole aligned vector (chunk edges
// when p does not divide n, or a ragged tail) are folded element by element
// by CTA (0, c).
//
// HBM traffic per element index: p reads of the input type, plus p writes
// (all-reduce, bucket) or 1 write (reduce-scatter) of the output type --
// exactly the primitives' minimum bytes.
#include "device_common.cuh"
#include "realign.cuh"

namespace ccl {
namespace {

template <int DT_IN, int DT_OUT>
__host__ __device__ constexpr int vec_width() {
  // 16 bytes of input per rank (two 16-byte loads when fp32 is cast to bf16,
  // so that the bf16 output is also a whole 16-byte store)
  return (DT_IN == kF32 && DT_OUT == kBF16) ? 8 : 16 / Elem<DT_IN>::kBytes;
}

__host__ __device__ constexpr int words_for(int vec, int bytes) { return (vec * bytes + 3) / 4; }

// Fold VEC elements starting at element i, in ring order from rank `first`.
// BATCH_IN: ranks whose loads are issued together before any of them is
// folded (0: 16, or 8 for 32-byte vectors).
template <int DT_IN, int VEC, int OP, int BATCH_IN = 0>
__device__ __forceinline__ void fold_elements(const FoldArgs& a, int p, int first, uint64_t i,
                                              typename Elem<DT_IN>::Acc* acc) {
  constexpr int WI = words_for(VEC, Elem<DT_IN>::kBytes);
  constexpr int BATCH = BATCH_IN > 0 ? BATCH_IN : ((WI >= 8) ? 8 : 16);
  int r = first;
  for (int j0 = 0; j0 < p; j0 += BATCH) {
    uint32_t raw[BATCH][WI];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (j0 + b < p) {
        load_raw<DT_IN, VEC>(a.send[r], i, raw[b]);
        r = (r + 1 == p) ? 0 : r + 1;
      }
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (j0 + b < p) {
        if (j0 + b == 0) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[e] = widen<DT_IN>(raw[b], e);
        } else {
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[e] = combine<OP>(acc[e], widen<DT_IN>(raw[b], e));
        }
      }
    }
  }
}

// Write the folded values of elements [i, i+VEC) of chunk c.
template <int DT_OUT, int VEC, int MODE, typename Acc>
__device__ __forceinline__ void emit(const FoldArgs& a, int p, int c, const Chunk& ch,
                                     uint64_t i, Acc* acc) {
  if constexpr (MODE == kModeBucket) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = __fmul_rn(acc[e], a.scale);
  }
  uint32_t w[words_for(VEC, Elem<DT_OUT>::kBytes)];
  pack_out<DT_OUT, VEC>(acc, w);
  if constexpr (MODE == kModeReduce) {
    store_raw<DT_OUT, VEC>(a.recv[0], i, w);
  } else if constexpr (MODE == kModeReduceScatter) {
    const uint64_t j = i - ch.off;  // position in rank c's shard
    if (VEC == 1 || (ch.off % VEC) == 0) {
      store_raw<DT_OUT, VEC>(a.recv[c], j, w);
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) store_one<DT_OUT>(a.recv[c], j + e, w, e);
    }
  } else {
    for (int r = 0; r < p; ++r) store_raw<DT_OUT, VEC>(a.recv[r], i, w);
  }
}

// REALIGN (reduce-scatter only) adds the realigned shard stores for chunks
// off the vector grid; the host picks it only when some chunk is, so that
// the aligned kernel keeps its registers (128 against 109 for bf16, which
// cost the p = 16 reduce-scatter 1 %).
template <int DT_IN, int DT_OUT, int VEC, int OP, int MODE, bool REALIGN, int BATCH = 0>
__global__ void __launch_bounds__(kThreads) fold_kernel(const __grid_constant__ FoldArgs a) {
  using Acc = typename Elem<DT_IN>::Acc;
  const int p = a.p;
  const int c = blockIdx.y;
  const Chunk ch = chunk_of(c, a.q, a.rem);
  const uint64_t end = ch.off + ch.len;
  const uint64_t v_lo = (ch.off + VEC - 1) / VEC;  // first whole vector inside chunk c
  const uint64_t v_hi = end / VEC;                 // one past the last
  const int first = (c + 1 == p) ? 0 : c + 1;      // the rank that starts chunk c
  if (VEC > 1 && cta_rank() < a.pf_ctas) {  // this CTA's first vectors of every rank, before waiting on the previous grid
    uint64_t b0 = ((MODE == kModeReduceScatter) ? v_lo : (v_lo & ~static_cast<uint64_t>(31))) +
                  static_cast<uint64_t>(blockIdx.x) * kThreads;
    uint64_t e0 = b0 + kThreads;
    b0 = b0 > v_lo ? b0 : v_lo;
    e0 = e0 < v_hi ? e0 : v_hi;
    if (b0 < e0)
      prefetch_spans_l2(a.send, p, b0 * VEC * Elem<DT_IN>::kBytes, (e0 - b0) * VEC * Elem<DT_IN>::kBytes);
  }
  pdl_enter();

  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  if (MODE == kModeReduceScatter && REALIGN && VEC > 1 && (ch.off % VEC) != 0) {
    // shard unaligned: whole warps step together so that neighbouring lanes
    // can hand each other the halves of the shard's aligned vectors
    const int lane = threadIdx.x & 31;
    for (uint64_t vb = v_lo + static_cast<uint64_t>(blockIdx.x) * kThreads + (threadIdx.x & ~31u); vb < v_hi;
         vb += stride) {
      const uint64_t v = vb + lane;
      Acc acc[VEC] = {};
      if (v < v_hi) fold_elements<DT_IN, VEC, OP, BATCH>(a, p, first, v * VEC, acc);
      uint32_t w[words_for(VEC, Elem<DT_OUT>::kBytes)];
      pack_out<DT_OUT, VEC>(acc, w);
      if constexpr (VEC * Elem<DT_OUT>::kBytes == 16)
        // (lanes start at v_lo here: 0 for v_lo spares the registers of the
        // check for lanes before it)
        store_shard_realigned<DT_OUT, VEC>(a.recv[c], ch.off, v, 0, v_hi, lane, w);
    }
  } else {
    // Vectors are counted from v_lo rounded down to 32, so that every warp's
    // 32 vectors fill whole 512-byte spans of the buffers (whole 128-byte
    // lines for the stores); lanes before v_lo (the previous chunk's) stay
    // idle.  Measured on GB300: the p = 72 all-reduce (chunks off the 512-byte
    // grid) 0.99 -> 1.03 of the copy bandwidth.  The reduce-scatter, whose
    // one output is a separate shard, keeps v_lo (1 % faster at p = 72).
    const uint64_t v_start = (MODE == kModeReduceScatter) ? v_lo : (v_lo & ~static_cast<uint64_t>(31));
    for (uint64_t v = v_start + static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; v < v_hi;
         v += stride) {
      if (v < v_lo) continue;
      Acc acc[VEC];
      fold_elements<DT_IN, VEC, OP, BATCH>(a, p, first, v * VEC, acc);
      emit<DT_OUT, VEC, MODE>(a, p, c, ch, v * VEC, acc);
    }
  }

  if (VEC > 1 && blockIdx.x == 0) {
    // element-wise edges: [off, head_end) and [tail_begin, end)
    const uint64_t head_end = (v_lo * VEC < end) ? v_lo * VEC : end;
    const uint64_t tail_begin = (v_hi * VEC > head_end) ? v_hi * VEC : head_end;
    const uint64_t n_head = head_end - ch.off;
    const uint64_t n_edge = n_head + (end - tail_begin);
    for (uint64_t t = threadIdx.x; t < n_edge; t += kThreads) {
      const uint64_t i = (t < n_head) ? ch.off + t : tail_begin + (t - n_head);
      Acc acc[1];
      fold_elements<DT_IN, 1, OP, BATCH>(a, p, first, i, acc);
      emit<DT_OUT, 1, MODE>(a, p, c, ch, i, acc);
    }
  }
}

// ------------------------------------------------------------- small p
// With few ranks a thread of fold_kernel has only p loads in flight, far too
// few to cover HBM latency at the occupancy its registers allow.  This kernel
// gives each thread U vectors (t, t + kThreads, ...) and issues the loads of
// all BATCH >= p ranks x U vectors before folding any of them, so a thread
// keeps about 256 bytes of loads in flight whatever p is.  The fold order of
// each element is the same ring walk as in fold_kernel.
template <int DT_IN, int VEC, int OP, int BATCH, int U>
__device__ __forceinline__ void fold_vectors(const FoldArgs& a, int p, int first, uint64_t v0,
                                             uint64_t v_lo, uint64_t v_hi,
                                             typename Elem<DT_IN>::Acc (&acc)[U][VEC]) {
  constexpr int WI = words_for(VEC, Elem<DT_IN>::kBytes);
  uint32_t raw[BATCH][U][WI];
  int r = first;
#pragma unroll
  for (int b = 0; b < BATCH; ++b) {
    if (b < p) {
      const void* src = a.send[r];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t v = v0 + static_cast<uint64_t>(u) * kThreads;
        if (v >= v_lo && v < v_hi) load_raw<DT_IN, VEC>(src, v * VEC, raw[b][u]);
      }
      r = (r + 1 == p) ? 0 : r + 1;
    }
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[u][e] = widen<DT_IN>(raw[0][u], e);
  }
#pragma unroll
  for (int b = 1; b < BATCH; ++b) {
    if (b < p) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[u][e] = combine<OP>(acc[u][e], widen<DT_IN>(raw[b][u], e));
      }
    }
  }
}

// Requires p <= BATCH and 16-byte aligned pointers; chunk edges are folded
// element-wise by CTA (0, c) exactly as in fold_kernel.
template <int DT_IN, int DT_OUT, int VEC, int OP, int MODE, int BATCH, int U>
__global__ void __launch_bounds__(kThreads) fold_unrolled_kernel(const __grid_constant__ FoldArgs a) {
  using Acc = typename Elem<DT_IN>::Acc;
  const int p = a.p;
  const int c = blockIdx.y;
  const Chunk ch = chunk_of(c, a.q, a.rem);
  const uint64_t end = ch.off + ch.len;
  const uint64_t v_lo = (ch.off + VEC - 1) / VEC;
  const uint64_t v_hi = end / VEC;
  const int first = (c + 1 == p) ? 0 : c + 1;

  // counted from v_lo rounded down to 32 (whole warps on 512-byte spans, as
  // in fold_kernel); lanes before v_lo stay idle
  const uint64_t v_start = v_lo & ~static_cast<uint64_t>(31);
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * U;
  if (cta_rank() < a.pf_ctas) {  // this CTA's first kSpan vectors of every rank, before waiting on the previous grid
    uint64_t b0 = v_start + static_cast<uint64_t>(blockIdx.x) * kSpan;
    uint64_t e0 = b0 + kSpan;
    b0 = b0 > v_lo ? b0 : v_lo;
    e0 = e0 < v_hi ? e0 : v_hi;
    if (b0 < e0)
      prefetch_spans_l2(a.send, p, b0 * VEC * Elem<DT_IN>::kBytes, (e0 - b0) * VEC * Elem<DT_IN>::kBytes);
  }
  pdl_enter();
  for (uint64_t base = v_start + static_cast<uint64_t>(blockIdx.x) * kSpan; base < v_hi;
       base += static_cast<uint64_t>(gridDim.x) * kSpan) {
    Acc acc[U][VEC];
    fold_vectors<DT_IN, VEC, OP, BATCH, U>(a, p, first, base + threadIdx.x, v_lo, v_hi, acc);
    if (MODE == kModeReduceScatter && (ch.off % VEC) != 0) {
      // shard unaligned: lanes hand each other the halves of its aligned
      // vectors (the loop is uniform over the CTA, so every lane is here)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
        uint32_t w[words_for(VEC, Elem<DT_OUT>::kBytes)];
        pack_out<DT_OUT, VEC>(acc[u], w);
        if constexpr (VEC * Elem<DT_OUT>::kBytes == 16)
          store_shard_realigned<DT_OUT, VEC>(a.recv[c], ch.off, v, v_lo, v_hi, threadIdx.x & 31, w);
      }
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
        if (v >= v_lo && v < v_hi) emit<DT_OUT, VEC, MODE>(a, p, c, ch, v * VEC, acc[u]);
      }
    }
  }

  if (blockIdx.x == 0) {
    const uint64_t head_end = (v_lo * VEC < end) ? v_lo * VEC : end;
    const uint64_t tail_begin = (v_hi * VEC > head_end) ? v_hi * VEC : head_end;
    const uint64_t n_head = head_end - ch.off;
    const uint64_t n_edge = n_head + (end - tail_begin);
    for (uint64_t t = threadIdx.x; t < n_edge; t += kThreads) {
      const uint64_t i = (t < n_head) ? ch.off + t : tail_begin + (t - n_head);
      Acc acc[1];
      fold_elements<DT_IN, 1, OP>(a, p, first, i, acc);
      emit<DT_OUT, 1, MODE>(a, p, c, ch, i, acc);
    }
  }
}

template <int DT_IN, int DT_OUT, int VEC, int OP, int MODE, int BATCH, int U>
cudaError_t launch_unrolled(const FoldArgs& a, cudaStream_t s) {
  const uint64_t per_chunk = (a.q + 1 + VEC - 1) / VEC + 31;  // + the lanes before v_lo
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * U;
  uint64_t gx = (per_chunk + kSpan - 1) / kSpan;
  if (gx < 1) gx = 1;
  if (gx > (1u << 30)) gx = 1u << 30;
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(a.p));
  return launch_kernel(fold_unrolled_kernel<DT_IN, DT_OUT, VEC, OP, MODE, BATCH, U>, grid,
                       dim3(kThreads), s, a);
}

// Programmatic dependent launch in two halves: wait for the previous grid,
// and let the next one be scheduled (a CTA that never does the second does
// it implicitly when it exits).
__device__ __forceinline__ void pdl_wait() {
#if CCL_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
__device__ __forceinline__ void pdl_trigger() {
#if CCL_PDL
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// Small chunks at large p: a CTA loads all p ranks' elements of a segment
// of chunk c at once (one round of loads, whatever p is) into shared
// memory, folds each element there in ring order from rank c + 1 (the same
// operations in the same order as fold_elements) and stores the results
// with all its threads.  The vector kernels load 16 ranks per round, p / 16
// dependent rounds.  Segments hold kSmallMaxItems / p elements; grid x =
// segments, grid y = chunks.
constexpr int kSmallMaxItems = 4096;  // p x segment held in shared memory
constexpr int kSmallMaxLen = 1536;    // chunks this kernel takes at p > 32

template <int DT_IN, int DT_OUT, int OP, int MODE>
__global__ void __launch_bounds__(kThreads) fold_small_kernel(const __grid_constant__ FoldArgs a) {
  using Acc = typename Elem<DT_IN>::Acc;
  __shared__ Acc s_in[kSmallMaxItems];  // ring position j, element e at j * len + e
  __shared__ Acc s_out[kSmallMaxItems / 17 + 1];
  const int p = a.p;
  const int c = blockIdx.y;
  const Chunk ch = chunk_of(c, a.q, a.rem);
  const int seg = kSmallMaxItems / p;
  const int e0 = static_cast<int>(blockIdx.x) * seg;
  const int len = static_cast<int>(ch.len) - e0 < seg ? static_cast<int>(ch.len) - e0 : seg;
  const uint64_t off = ch.off + static_cast<uint64_t>(e0);
  const int first = (c + 1 == p) ? 0 : c + 1;
  // A grid of more than half the device's resident CTAs (a.pf_ctas: one
  // wave) lets the next grid be scheduled only as its CTAs exit.  Scheduled
  // at entry, the next grid's CTAs took slots this grid's last CTAs needed:
  // measured on GB300, back-to-back calls, late against at entry (us per
  // call): all-reduce p = 72 with chunks of 455 (648 CTAs) 10.6 -> 8.2 fp32,
  // 11.0 -> 7.8 bf16; reduce-scatter 8.4 -> 6.1 and 8.0 -> 5.7; p = 48 with
  // chunks of 1024 (624 CTAs) 11.2 -> 8.4.  Grids within half a wave ran the
  // same either way and keep the early start.
  pdl_wait();
  if (static_cast<uint64_t>(gridDim.x) * gridDim.y * 2 <= a.pf_ctas) pdl_trigger();
  if (len <= 0) return;  // (uniform over the CTA)
  for (int t = threadIdx.x; t < p * len; t += kThreads) {
    const int j = t / len, e = t - j * len;
    const int r = first + j < p ? first + j : first + j - p;
    uint32_t w[1];
    load_raw<DT_IN, 1>(a.send[r], off + static_cast<uint64_t>(e), w);
    s_in[t] = widen<DT_IN>(w, 0);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < len; e += kThreads) {
    Acc acc = s_in[e];
    for (int j = 1; j < p; ++j) acc = combine<OP>(acc, s_in[j * len + e]);
    if constexpr (MODE == kModeBucket) acc = __fmul_rn(acc, a.scale);
    s_out[e] = acc;
  }
  __syncthreads();
  const int outputs = (MODE == kModeAllReduce || MODE == kModeBucket) ? p : 1;
  for (int t = threadIdx.x; t < outputs * len; t += kThreads) {
    const int r = t / len, e = t - r * len;
    Acc v = s_out[e];
    uint32_t w[1];
    pack_out<DT_OUT, 1>(&v, w);
    if constexpr (MODE == kModeReduceScatter) {
      store_raw<DT_OUT, 1>(a.recv[c], static_cast<uint64_t>(e0 + e), w);
    } else if constexpr (MODE == kModeReduce) {
      store_raw<DT_OUT, 1>(a.recv[0], off + static_cast<uint64_t>(e), w);
    } else {
      store_raw<DT_OUT, 1>(a.recv[r], off + static_cast<uint64_t>(e), w);
    }
  }
}

unsigned fold_small_segments(int p, uint64_t q) {
  const uint64_t seg = static_cast<uint64_t>(kSmallMaxItems / p);
  return static_cast<unsigned>((q + 1 + seg - 1) / seg);
}

// Whether a call takes fold_small_kernel.  The vector kernels load 16 ranks
// per round, ceil(p / 16) dependent rounds; this kernel loads every rank in
// one round.  It takes the call when
//  * 17 - 32 ranks (two rounds): a chunk holds at most 2048 of the ranks'
//    elements (p = 32 with chunks of 128 - 240 fp32 lost, 2.8 -> 4.0 us);
//  * more than 32 ranks: chunks of at most kSmallMaxLen elements and at
//    most 4 CTAs per SM for every two of the vector kernels' rounds (one
//    wave, 8 per SM, at p = 72; two waves at p = 128).
// Measured on GB300 against the vector kernels (us per call, one call after
// another; chunk = elements per chunk; the late dependent launch above in
// place):
//   all-reduce fp32 p = 72 at 1 / 16 / 64 KiB per rank  4.9 / 9.1 / 10.1 -> 2.2 / 5.6 / 6.8
//   all-reduce p = 72, chunk 300 / 455 / 768, fp32      9.9 / 10.1 / 11.5 -> 6.9 / 8.2 / 10.1
//                                             bf16      12.1 / 11.9 / 12.1 -> 6.5 / 7.8 / 9.8
//   reduce-scatter p = 72, chunk 300 / 455 / 768, fp32  8.6 / 8.8 / 9.1 -> 5.5 / 6.1 / 7.6
//                                                 bf16  9.4 / 9.4 / 9.6 -> 5.1 / 5.7 / 7.4
//   all-reduce fp32 p = 72, chunk 1024 (1,368 CTAs)     12.5 -> 15.5 (not taken)
//   all-reduce fp32 p = 128, chunk 300 / 512            18.4 / 20.6 -> 14.1 / 19.3
//   all-reduce fp32 p = 128, chunk 768 (3,200 CTAs)     23.5 -> 27.9 (not taken)
//   p = 48, chunk 768, all-reduce fp32 / bf16           7.3 / 7.9 -> 7.6 / 7.3
//   p = 48, chunk 1024 (624 CTAs), all-reduce fp32      7.9 -> 8.4 (not taken;
//                                  reduce-scatter bf16  6.4 -> 5.8)
//   all-reduce p = 33, chunk 1024, fp32 / bf16          6.6 / 7.1 -> 6.1 / 5.7
bool fold_small(int p, uint64_t q, int sms) {
  if (p <= 16) return false;
  if (p <= 32) return static_cast<uint64_t>(p) * (q + 1) <= 2048;
  if (q + 1 > static_cast<uint64_t>(kSmallMaxLen)) return false;
  const uint64_t rounds = static_cast<uint64_t>((p + 15) / 16);  // >= 3
  const uint64_t n_sms = static_cast<uint64_t>(sms > 0 ? sms : 1);
  return static_cast<uint64_t>(fold_small_segments(p, q)) * static_cast<uint64_t>(p) <= 4 * n_sms * (rounds / 2);
}

constexpr int kVectorsPerThread = 2;

// fold_kernel strides over a chunk's vectors, about kVectorsPerThread per
// thread; a call whose grid would then hold less than one wave takes one
// vector per thread (twice the CTAs) as long as that still fits one wave
// (the kernel's resident CTAs per SM x SMs).  Measured on GB300 (fraction
// of the copy bandwidth, 2 -> 1 vectors): reduce-scatter p = 72 fp32 at
// 1 MiB per rank 0.62 -> 0.93, all-reduce p = 16 fp32 at 1 MiB 0.66 -> 0.90,
// p = 72 at 256 KiB 0.36 -> 0.47; taking one vector also when its grid
// spills into a second wave lost at 2 MiB (reduce-scatter p = 72 0.97 ->
// 0.88).
//
// The reduce-scatter (and the reduce to the root) with 9..32 ranks and
// chunks of 128 KiB or more loads 8 ranks per batch instead of 16 (about 60 registers instead of 91-107: 4
// CTAs per SM instead of 2, each thread two dependent rounds of loads).
// Measured on GB300 against 16 (fraction of the copy bandwidth): p = 9 bf16
// at 8 / 64 / 256 MiB per rank 0.73 / 0.84 / 0.87 -> 0.85 / 0.98 / 0.98,
// p = 12 fp32 0.79 / 0.84 / 0.84 -> 0.91 / 1.02 / 1.03, p = 24 bf16 0.86 /
// 0.94 / 0.94 -> 0.99 / 1.05 / 1.04; p = 16 at 8 MiB 0.98 / 0.93 -> 1.08 /
// 1.07 (fp32 / bf16), p = 32 at 4 MiB 1.03 / 0.97 -> 1.06 / 1.05.  Smaller
// chunks lost (p = 16 at 1 MiB 0.83 -> 0.62: the second round of loads is
// latency there), p = 72 came out even, and the all-reduce, which stores
// every vector p times, lost 1-2 % at p = 16 - 72.
constexpr uint64_t kBatch8MinChunkBytes = 128 * 1024;

template <int DT_IN, int DT_OUT, int VEC, int OP, int MODE>
cudaError_t launch_one(const FoldArgs& a, cudaStream_t s) {
  auto kernel = fold_kernel<DT_IN, DT_OUT, VEC, OP, MODE, false>;
  if constexpr (MODE == kModeReduceScatter && VEC > 1) {
    bool realign = false;  // some chunk starts off the vector grid (off(c), the chunk rule)
    for (uint64_t c = 0; c < static_cast<uint64_t>(a.p) && !realign; ++c)
      realign = (c * a.q + (c < a.rem ? c : a.rem)) % VEC != 0;
    constexpr bool kWide = words_for(VEC, Elem<DT_IN>::kBytes) >= 8;  // 32-byte vectors batch 8 already
    const bool batch8 = !kWide && a.p >= 9 && a.p <= 32 && a.q * Elem<DT_IN>::kBytes >= kBatch8MinChunkBytes;
    if (batch8) {
      kernel = realign ? fold_kernel<DT_IN, DT_OUT, VEC, OP, MODE, true, 8>
                       : fold_kernel<DT_IN, DT_OUT, VEC, OP, MODE, false, 8>;
    } else if (realign) {
      kernel = fold_kernel<DT_IN, DT_OUT, VEC, OP, MODE, true>;
    }
  }
  if constexpr (MODE == kModeReduce && VEC > 1) {
    // the reduce to the root reads and writes what the reduce-scatter does
    // (fp32 p = 9 / 16 / 32 at 16 MiB per rank 0.96 / 1.05 / 1.09 -> 1.00 /
    // 1.09 / 1.10 of the copy bandwidth, bf16 p = 9 at 64 MiB 0.91 -> 1.03)
    constexpr bool kWide = words_for(VEC, Elem<DT_IN>::kBytes) >= 8;
    if (!kWide && a.p >= 9 && a.p <= 32 && a.q * Elem<DT_IN>::kBytes >= kBatch8MinChunkBytes)
      kernel = fold_kernel<DT_IN, DT_OUT, VEC, OP, MODE, false, 8>;
  }
  const uint64_t per_chunk = (a.q + 1 + VEC - 1) / VEC + 31;  // + the lanes before v_lo
  auto grid_x = [&](uint64_t vpt) { return (per_chunk + kThreads * vpt - 1) / (kThreads * vpt); };
  const uint64_t wave = static_cast<uint64_t>(first_wave_ctas(reinterpret_cast<const void*>(kernel)));
  const uint64_t p = static_cast<uint64_t>(a.p);
  uint64_t gx = grid_x(kVectorsPerThread);
  if (gx * p < wave && grid_x(1) * p <= wave) gx = grid_x(1);
  if (gx < 1) gx = 1;
  if (gx > (1u << 30)) gx = 1u << 30;
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(a.p));
  return launch_kernel(kernel, grid, dim3(kThreads), s, a);
}

// Instantiations of fold_unrolled_kernel per launch_typed; the choice among
// them is fold_plan's (below), so that one host function states it.
template <int DT_IN, int DT_OUT, int OP, int MODE>
cudaError_t launch_typed(bool vec, const FoldArgs& a, cudaStream_t s) {
  const FoldPlan pl = fold_plan(DT_IN, DT_OUT, OP, MODE, a.p, a.q, vec, current_sm_count());
  if (pl.batch < 0)
    return launch_kernel(fold_small_kernel<DT_IN, DT_OUT, OP, MODE>,
                         dim3(fold_small_segments(a.p, a.q), static_cast<unsigned>(a.p)), dim3(kThreads), s, a);
  if (!vec) return launch_one<DT_IN, DT_OUT, 1, OP, MODE>(a, s);
  constexpr int VEC = vec_width<DT_IN, DT_OUT>();
  if constexpr (OP == CCL_SUM) {
    constexpr bool kHalve = VEC > 4;
#define CCL_UNROLLED(B, U) \
  if (pl.batch == B && pl.vectors == U) return launch_unrolled<DT_IN, DT_OUT, VEC, OP, MODE, B, U>(a, s);
    CCL_UNROLLED(2, 2)
    CCL_UNROLLED(4, 1)
    CCL_UNROLLED(4, 2)
    if constexpr (MODE == kModeBucket) {
      CCL_UNROLLED(2, 4)
    } else {
      CCL_UNROLLED(8, 1)
      if constexpr (MODE == kModeAllReduce) {
        CCL_UNROLLED(2, 1)
      } else if constexpr (!kHalve) {
        CCL_UNROLLED(2, 8)
      }
    }
#undef CCL_UNROLLED
    if (pl.batch != 0) return cudaErrorInvalidConfiguration;  // a plan with no instantiation
  }
  return launch_one<DT_IN, DT_OUT, VEC, OP, MODE>(a, s);
}

template <int MODE>
cudaError_t launch_mode(int dt, int op, bool vec, const FoldArgs& a, cudaStream_t s) {
#define CCL_FOLD_CASE(DT, OP)                                     \
  if (dt == DT && op == OP) return launch_typed<DT, DT, OP, MODE>(vec, a, s);
  CCL_FOLD_CASE(kF32, CCL_SUM)
  CCL_FOLD_CASE(kF32, CCL_MAX)
  CCL_FOLD_CASE(kF32, CCL_MIN)
  CCL_FOLD_CASE(kBF16, CCL_SUM)
  CCL_FOLD_CASE(kBF16, CCL_MAX)
  CCL_FOLD_CASE(kBF16, CCL_MIN)
  CCL_FOLD_CASE(kI32, CCL_SUM)
  CCL_FOLD_CASE(kI32, CCL_MAX)
  CCL_FOLD_CASE(kI32, CCL_MIN)
#undef CCL_FOLD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

// Small p (sums only) goes to fold_unrolled_kernel with (ranks per batch,
// vectors per thread): a thread issues the loads of all its ranks' vectors
// before folding any.  The choice, measured on GB300 per call kind over
// 1 MiB - 256 MiB per rank (fractions of the copy bandwidth):
//  * Calls whose one-vector grid fits one wave (the one-vector kernels hold
//    4 CTAs per SM) take one vector per thread: all-reduce p = 2 at 2 MiB
//    0.57 -> 0.63 against two.  Above that, the reduce-scatter (and the
//    reduce to the root: the same bytes read and written) wants more loads in
//    flight than the all-reduce, which also stores every vector p times:
//  * p <= 2: all-reduce 2 x 2 (2 x 8 fp32 / 2 x 4 bf16 at 20 MiB and up ran
//    0.7-0.9 % slower); reduce-scatter 2 x 2, fp32 / int32 2 x 8 once that
//    grid has 8 CTAs per SM (bf16 2 x 4 there: 1.00 against 1.05 at 256 MiB).
//  * p = 3..4: 4 x 2 (reduce-scatter p = 3 fp32 at 8 MiB 0.75 -> 0.88 and at
//    16 MiB 0.84 -> 1.01 against 4 x 1, p = 4 0.94 -> 0.99; all-reduce p = 3
//    bf16 at 8 MiB 0.88 -> 0.93), except the all-reduce at p = 4, which
//    keeps 4 x 1 (0.93 against 0.87 at 8 MiB, 1.05 against 1.04 at 256 MiB).
//  * p = 5..8: 8 x 1 at every size (57 registers, 4 CTAs per SM: the loads
//    in flight per SM of 8 x 2 at 2 CTAs, in twice the CTAs): reduce-scatter
//    fp32 p = 5 0.90 -> 1.03 at 256 MiB and 0.75 -> 0.95 at 8 MiB, p = 6
//    0.82 -> 1.00 and p = 8 0.95 -> 1.09 at 8 MiB; all-reduce bf16 p = 5
//    0.87 -> 0.93 at 8 MiB; 1 KiB calls 1.7-2.4 -> 1.3-1.9 us.  8 x 2 had
//    replaced the general kernel for bf16 (all-reduce p = 6 0.92 -> 1.03,
//    reduce-scatter p = 8 0.94 -> 1.07 at 256 MiB - 1 GiB).
//  * The DDP bucket (fp32 in, 32-byte vectors of 8 accumulators): 2 x 4 at
//    p <= 2 and 4 x 2 at p <= 4 once that grid has 8 CTAs per SM, else 2 x 2
//    and 4 x 1; p > 4 stays on fold_kernel (8 ranks of 32-byte vectors
//    would need twice the registers).
// The general kernel ran 0.3-0.8 for p <= 4 at these sizes.  Calls of
// more than 16 ranks whose chunks fit shared memory (fold_small) take
// fold_small_kernel, whatever the op and alignment: (-1, 0).
FoldPlan fold_plan(int dt_in, int dt_out, int op, int mode, int p, uint64_t q, bool vec, int sms) {
  if (p < 1) return FoldPlan{0, 0};
  if (fold_small(p, q, sms)) return FoldPlan{-1, 0};  // fold_small_kernel, any op and alignment
  if (!vec || op != CCL_SUM) return FoldPlan{0, 0};
  const int in_bytes = (dt_in == kBF16) ? 2 : 4;
  const int v = (dt_in == kF32 && dt_out == kBF16) ? 8 : 16 / in_bytes;  // vec_width
  const bool halve = v > 4;
  const uint64_t per_chunk = (q + 1 + v - 1) / v;
  const uint64_t n_sms = static_cast<uint64_t>(sms > 0 ? sms : 1);
  const uint64_t want_ctas = 8 * n_sms;
  auto ctas = [&](int u) {
    return (per_chunk + static_cast<uint64_t>(kThreads) * u - 1) / (static_cast<uint64_t>(kThreads) * u) *
           static_cast<uint64_t>(p);
  };
  if (mode == kModeBucket) {
    if (p <= 2) return ctas(4) >= want_ctas ? FoldPlan{2, 4} : FoldPlan{2, 2};
    if (p <= 4) return ctas(2) >= want_ctas ? FoldPlan{4, 2} : FoldPlan{4, 1};
    return FoldPlan{0, 0};
  }
  const bool one_wave = ctas(1) <= 4 * n_sms;
  if (p <= 2) {
    if (mode == kModeAllReduce) return one_wave ? FoldPlan{2, 1} : FoldPlan{2, 2};
    return (!halve && ctas(8) >= want_ctas) ? FoldPlan{2, 8} : FoldPlan{2, 2};
  }
  if (p <= 4) {
    if (mode == kModeAllReduce && p == 4) return FoldPlan{4, 1};
    return one_wave ? FoldPlan{4, 1} : FoldPlan{4, 2};
  }
  if (p <= 8) return FoldPlan{8, 1};
  return FoldPlan{0, 0};
}

cudaError_t launch_fold(int mode, int dt, int op, bool vec, const FoldArgs& a, cudaStream_t s) {
  cudaError_t err = cudaErrorInvalidValue;
  if (mode == kModeAllReduce) {
    err = launch_mode<kModeAllReduce>(dt, op, vec, a, s);
  } else if (mode == kModeReduceScatter) {
    err = launch_mode<kModeReduceScatter>(dt, op, vec, a, s);
  } else if (mode == kModeBucket) {
    err = launch_typed<kF32, kBF16, CCL_SUM, kModeBucket>(vec, a, s);
  } else if (mode == kModeReduce) {
    err = launch_mode<kModeReduce>(dt, op, vec, a, s);
  }
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace ccl
