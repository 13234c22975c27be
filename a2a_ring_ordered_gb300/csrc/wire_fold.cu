// wire_fold.cu -- the ring all-reduce / reduce-scatter of bf16 data with bf16
// on the wire: every hop adds the received partial and its own value in fp32
// and rounds the new partial to bf16 (nearest-even) before it travels on, so
// chunk c's result is bf16(...bf16(bf16(x_{c+1} + x_{c+2}) + x_{c+3})... + x_c).
// The ring ("Networks and Collective Communication" section 5.1; "dist_train",
// Ring Algorithm) is the same as in fold.cu; only the partial's width differs
// (a bf16 message is half the bytes of an fp32 one).
//
// As in fold.cu, one thread performs a chunk's whole walk for one 16-byte
// vector (8 bf16) in registers, with the ring's start rank uniform per CTA
// (grid y = chunk) and each vector read once per rank and written once per
// output.  Small p takes several vectors per thread so that enough loads are
// in flight.  Chunk edges off the 16-byte grid are folded element-wise by
// CTA (0, c).
#include "device_common.cuh"
#include "realign.cuh"

namespace ccl {
namespace {

__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// Fold U vectors (t, t + kThreads, ...) of VEC bf16 elements starting at rank
// `first`; the loads of BATCH ranks x U vectors are issued before any is folded.
template <int VEC, int BATCH, int U>
__device__ __forceinline__ void fold_wire(const FoldArgs& a, int first, uint64_t v0, uint64_t v_hi,
                                          float (&acc)[U][VEC]) {
  constexpr int W = (VEC * 2 + 3) / 4;
  const int p = a.p;
  int r = first;
  for (int j0 = 0; j0 < p; j0 += BATCH) {
    uint32_t raw[BATCH][U][W];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (j0 + b < p) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const uint64_t v = v0 + static_cast<uint64_t>(u) * kThreads;
          if (v < v_hi) load_raw<kBF16, VEC>(a.send[r], v * VEC, raw[b][u]);
        }
        r = (r + 1 == p) ? 0 : r + 1;
      }
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (j0 + b < p) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const float x = widen<kBF16>(raw[b][u], e);
            acc[u][e] = (j0 + b == 0) ? x : round_bf16(__fadd_rn(acc[u][e], x));
          }
        }
      }
    }
  }
}

template <int VEC, int MODE>
__device__ __forceinline__ void emit_wire(const FoldArgs& a, int c, const Chunk& ch, uint64_t i,
                                          const float* acc) {
  uint32_t w[(VEC * 2 + 3) / 4];
  pack_out<kBF16, VEC>(acc, w);  // exact: every value is already a bf16
  if constexpr (MODE == kModeReduceScatter) {
    const uint64_t j = i - ch.off;
    if (VEC == 1 || (ch.off % VEC) == 0) {
      store_raw<kBF16, VEC>(a.recv[c], j, w);
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) store_one<kBF16>(a.recv[c], j + e, w, e);
    }
  } else {
    for (int r = 0; r < a.p; ++r) store_raw<kBF16, VEC>(a.recv[r], i, w);
  }
}

template <int VEC, int MODE, int BATCH, int U>
__global__ void __launch_bounds__(kThreads) wire_fold_kernel(const __grid_constant__ FoldArgs a) {
  pdl_enter();
  const int p = a.p;
  const int c = blockIdx.y;
  const Chunk ch = chunk_of(c, a.q, a.rem);
  const uint64_t end = ch.off + ch.len;
  const uint64_t v_lo = (ch.off + VEC - 1) / VEC, v_hi = end / VEC;
  const int first = (c + 1 == p) ? 0 : c + 1;
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * U;
  for (uint64_t base = v_lo + static_cast<uint64_t>(blockIdx.x) * kSpan; base < v_hi;
       base += static_cast<uint64_t>(gridDim.x) * kSpan) {
    float acc[U][VEC];
    fold_wire<VEC, BATCH, U>(a, first, base + threadIdx.x, v_hi, acc);
    if (MODE == kModeReduceScatter && VEC > 1 && (ch.off % VEC) != 0) {
      // shard unaligned: lanes hand each other the halves of its aligned
      // vectors (the loop is uniform over the CTA, so every lane is here)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
        uint32_t w[(VEC * 2 + 3) / 4];
        pack_out<kBF16, VEC>(acc[u], w);
        if constexpr (VEC == 8) store_shard_realigned<kBF16, VEC>(a.recv[c], ch.off, v, v_lo, v_hi, threadIdx.x & 31, w);
      }
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t v = base + threadIdx.x + static_cast<uint64_t>(u) * kThreads;
        if (v < v_hi) emit_wire<VEC, MODE>(a, c, ch, v * VEC, acc[u]);
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
      float acc[1][1];
      fold_wire<1, BATCH, 1>(a, first, i, i + 1, acc);
      emit_wire<1, MODE>(a, c, ch, i, acc[0]);
    }
  }
}

template <int VEC, int MODE, int BATCH, int U>
cudaError_t launch_one(const FoldArgs& a, cudaStream_t s) {
  const uint64_t per_chunk = (a.q + 1 + VEC - 1) / VEC;
  constexpr uint64_t kSpan = static_cast<uint64_t>(kThreads) * U;
  uint64_t gx = (per_chunk + kSpan - 1) / kSpan;
  if (gx < 1) gx = 1;
  if (gx > (1u << 30)) gx = 1u << 30;
  return launch_kernel(wire_fold_kernel<VEC, MODE, BATCH, U>, dim3(static_cast<unsigned>(gx), a.p),
                       dim3(kThreads), s, a);
}

// (ranks per load batch, vectors per thread): about 128 bytes of loads in
// flight per thread for small p, 8 ranks x 1 vector from p = 9 on.
template <int MODE>
cudaError_t launch_mode(bool vec, const FoldArgs& a, cudaStream_t s) {
  if (!vec) return launch_one<1, MODE, 8, 1>(a, s);
  if (a.p <= 2) return launch_one<8, MODE, 2, 4>(a, s);
  if (a.p <= 4) return launch_one<8, MODE, 4, 2>(a, s);
  return launch_one<8, MODE, 8, 1>(a, s);
}

}  // namespace

cudaError_t launch_wire_fold(int mode, bool vec, const FoldArgs& a, cudaStream_t s) {
  cudaError_t err = cudaErrorInvalidValue;
  if (mode == kModeAllReduce) err = launch_mode<kModeAllReduce>(vec, a, s);
  else if (mode == kModeReduceScatter) err = launch_mode<kModeReduceScatter>(vec, a, s);
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace ccl
