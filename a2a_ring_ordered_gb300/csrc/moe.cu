// moe.cu -- MoE expert-parallel routing, dispatch (bf16 or FP8) and combine.
//
// "Networks and Collective Communication" section 7.4: each MoE layer does an
// all-to-all dispatch (every token to the ranks holding the k experts it
// chose) and an all-to-all combine (the expert outputs come back); the
// DeepSeek-V3 recipe dispatches in FP8 and combines in BF16.
//
// Layout (shared with the oracle): expert e lives on rank e / (E / p); token t
// of source s sends one row per choice j; destination d holds its rows grouped
// by source, then token, then choice.  route() gives each (t, j) its slot --
// its rank among the rows the source sends to the same destination -- so the
// row lands at sum_{s' < s} counts[s'][d] + slot of d's buffer.
#include <cuda_fp8.h>

#include "device_common.cuh"

namespace ccl {
namespace {

constexpr int kRouteThreads = 1024;  // 32 warps

// One CTA per source.  Items (t, j) are taken in order, 1024 per tile; inside
// a warp __match_any_sync groups the lanes with the same destination, which
// gives each item its rank among earlier same-destination items of the warp;
// an exclusive scan over the 32 warps on top of the running per-destination
// count turns that into the slot.
__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(const __grid_constant__ MoeRouteArgs a) {
  __shared__ int warp_cnt[32][kMoeMaxRanks];
  __shared__ int run[kMoeMaxRanks];
  pdl_enter();
  const int s = blockIdx.x;
  const int p = a.p;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int d = tid; d < p; d += kRouteThreads) run[d] = 0;
  const int32_t* ids = a.ids[s];
  int32_t* slots = a.slots[s];
  for (uint64_t base = 0; base < a.items; base += kRouteThreads) {
    for (int i = tid; i < 32 * p; i += kRouteThreads) warp_cnt[i / p][i % p] = 0;
    __syncthreads();
    const uint64_t item = base + tid;
    int d = -1;
    if (item < a.items) {
      const int e = ids[item];
      if (e >= 0 && e < a.num_experts) d = e / a.epr;
    }
    const unsigned same = __match_any_sync(0xFFFFFFFFu, d);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (d >= 0 && rank == 0) warp_cnt[warp][d] = __popc(same);
    __syncthreads();
    if (tid < p) {
      int acc = run[tid];
      for (int w = 0; w < 32; ++w) {
        const int c = warp_cnt[w][tid];
        warp_cnt[w][tid] = acc;
        acc += c;
      }
      run[tid] = acc;
    }
    __syncthreads();
    if (item < a.items) slots[item] = (d >= 0) ? warp_cnt[warp][d] + rank : -1;
    __syncthreads();
  }
  if (tid < p) a.counts[static_cast<uint64_t>(s) * p + tid] = run[tid];
}

constexpr int kTokensPerCta = 8;

// base[d] = rows of destination d sent by sources before s.
__device__ __forceinline__ void row_bases(const int64_t* counts, int p, int s, int64_t* base) {
  for (int d = threadIdx.x; d < p; d += blockDim.x) {
    int64_t acc = 0;
    for (int q = 0; q < s; ++q) acc += counts[static_cast<uint64_t>(q) * p + d];
    base[d] = acc;
  }
}

// One CTA per (tile of tokens, source).  Each 16-byte vector of a token row
// (8 bf16) is loaded once and stored to the k destinations.  FP8: 16
// elements per thread, and the 8 threads holding a 128-element block (vectors
// are handed out so that 8 consecutive threads hold one block) reduce its amax
// with shuffles;
// inv = 448 / amax, code = e4m3(x * inv), round to nearest even, saturating;
// the block scale amax / 448 is stored for dequantisation.
template <bool FP8>
__global__ void __launch_bounds__(kThreads) moe_dispatch_kernel(const __grid_constant__ MoeDispatchArgs a) {
  __shared__ int64_t base[kMoeMaxRanks];
  __shared__ int64_t pos[kTokensPerCta][kMoeMaxK];
  __shared__ int dest[kTokensPerCta][kMoeMaxK];
  __shared__ int expert[kTokensPerCta][kMoeMaxK];
  pdl_enter();
  const int s = blockIdx.y;
  const int p = a.p, k = a.k;
  const uint64_t t0 = static_cast<uint64_t>(blockIdx.x) * kTokensPerCta;
  row_bases(a.counts, p, s, base);
  __syncthreads();
  for (int i = threadIdx.x; i < kTokensPerCta * k; i += kThreads) {
    const int tt = i / k, j = i % k;
    const uint64_t t = t0 + tt;
    int d = -1;
    int64_t row = -1;
    int e = -1;
    if (t < a.tokens) {
      e = a.ids[s][t * k + j];
      const int slot = a.slots[s][t * k + j];
      if (e >= 0 && e < a.num_experts && slot >= 0) {
        d = e / a.epr;
        row = base[d] + slot;
        if (static_cast<uint64_t>(row) >= a.cap[d]) d = -1;  // never write past a buffer
      }
    }
    dest[tt][j] = d;
    pos[tt][j] = row;
    expert[tt][j] = e;
  }
  __syncthreads();
  const uint64_t h = a.hidden;
  const uint64_t nvec = h / 8;
  for (int tt = 0; tt < kTokensPerCta; ++tt) {
    const uint64_t t = t0 + tt;
    if (t >= a.tokens) break;
    const char* src = static_cast<const char*>(a.x[s]) + t * h * 2;
    if constexpr (!FP8) {
      for (uint64_t v = threadIdx.x; v < nvec; v += kThreads) {
        uint32_t w[4];
        load_raw<kBF16, 8>(src, v * 8, w);
        for (int j = 0; j < k; ++j) {
          const int d = dest[tt][j];
          if (d >= 0) store_raw<kBF16, 8>(a.recv[d], static_cast<uint64_t>(pos[tt][j]) * h + v * 8, w);
        }
      }
    } else {
      // 16 elements (two 16-byte loads) per thread; the 8 consecutive threads
      // holding a 128-element block reduce its amax with shuffles; one
      // reciprocal per block, one multiply per element, one 16-byte store of
      // codes per destination row
      const uint64_t nv16 = h / 16;
      for (uint64_t v = threadIdx.x; v < nv16; v += kThreads) {
        uint32_t w[8];
        load_raw<kBF16, 8>(src, v * 16, w);
        load_raw<kBF16, 8>(src, v * 16 + 8, w + 4);
        float x[16];
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          x[e] = widen<kBF16>(w, e);
          amax = fmaxf(amax, fabsf(x[e]));
        }
        // the 8 lanes of this block are all active (hidden is a multiple of 128)
        const unsigned group = 0xFFu << (threadIdx.x & 24);
#pragma unroll
        for (int off = 4; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(group, amax, off));
        const float inv = (amax > 0.0f) ? __fdiv_rn(448.0f, amax) : 1.0f;
        const float scale = (amax > 0.0f) ? __fdiv_rn(amax, 448.0f) : 1.0f;
        uint32_t q[4] = {0, 0, 0, 0};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint32_t c = __nv_cvt_float_to_fp8(__fmul_rn(x[e], inv), __NV_SATFINITE, __NV_E4M3);
          q[e >> 2] |= (c & 0xFFu) << (8 * (e & 3));
        }
        const uint64_t blk = v / 8;  // 8 vectors of 16 = one 128-element block
        for (int j = 0; j < k; ++j) {
          const int d = dest[tt][j];
          if (d < 0) continue;
          const uint64_t row = static_cast<uint64_t>(pos[tt][j]);
          st_stream16(static_cast<char*>(a.recv[d]) + row * h + v * 16, make_uint4(q[0], q[1], q[2], q[3]));
          if ((threadIdx.x & 7) == 0) a.scales[d][row * (h / 128) + blk] = scale;
        }
      }
    }
    if (a.rexp_given && threadIdx.x < k) {
      const int d = dest[tt][threadIdx.x];
      if (d >= 0 && a.rexp[d] != nullptr) a.rexp[d][pos[tt][threadIdx.x]] = expert[tt][threadIdx.x];
    }
  }
}

// One CTA per (tile of tokens, source): token t's output is the bf16 of the
// fp32 sum over choices j of w[t][j] * y_j, in choice order (each product and
// each sum rounded; no fused multiply-add).  The k rows' loads are issued
// before any is combined.
__global__ void __launch_bounds__(kThreads) moe_combine_kernel(const __grid_constant__ MoeCombineArgs a) {
  __shared__ int64_t base[kMoeMaxRanks];
  __shared__ int64_t pos[kTokensPerCta][kMoeMaxK];
  __shared__ int dest[kTokensPerCta][kMoeMaxK];
  __shared__ float wt[kTokensPerCta][kMoeMaxK];
  pdl_enter();
  const int s = blockIdx.y;
  const int p = a.p, k = a.k;
  const uint64_t t0 = static_cast<uint64_t>(blockIdx.x) * kTokensPerCta;
  row_bases(a.counts, p, s, base);
  __syncthreads();
  for (int i = threadIdx.x; i < kTokensPerCta * k; i += kThreads) {
    const int tt = i / k, j = i % k;
    const uint64_t t = t0 + tt;
    int d = -1;
    int64_t row = -1;
    float wj = 0.0f;
    if (t < a.tokens) {
      const int e = a.ids[s][t * k + j];
      const int slot = a.slots[s][t * k + j];
      wj = a.weights[s][t * k + j];
      if (e >= 0 && e < a.num_experts && slot >= 0) {
        d = e / a.epr;
        row = base[d] + slot;
        if (static_cast<uint64_t>(row) >= a.cap[d]) d = -1;
      }
    }
    dest[tt][j] = d;
    pos[tt][j] = row;
    wt[tt][j] = wj;
  }
  __syncthreads();
  const uint64_t h = a.hidden;
  const uint64_t nvec = h / 8;
  for (int tt = 0; tt < kTokensPerCta; ++tt) {
    const uint64_t t = t0 + tt;
    if (t >= a.tokens) break;
    for (uint64_t v = threadIdx.x; v < nvec; v += kThreads) {
      float acc[8];
      bool have = false;
      for (int j0 = 0; j0 < k; j0 += 8) {
        uint32_t raw[8][4];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int j = j0 + b;
          if (j < k && dest[tt][j] >= 0)
            load_raw<kBF16, 8>(a.y[dest[tt][j]], static_cast<uint64_t>(pos[tt][j]) * h + v * 8, raw[b]);
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int j = j0 + b;
          if (j < k && dest[tt][j] >= 0) {
            const float wj = wt[tt][j];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float prod = __fmul_rn(wj, widen<kBF16>(raw[b], e));
              acc[e] = have ? __fadd_rn(acc[e], prod) : prod;
            }
            have = true;
          }
        }
      }
      if (!have) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
      }
      uint32_t w[4];
      pack_out<kBF16, 8>(acc, w);
      store_raw<kBF16, 8>(a.out[s], t * h + v * 8, w);
    }
  }
}

}  // namespace

cudaError_t launch_moe_route(const MoeRouteArgs& a, cudaStream_t s) {
  cudaError_t err = launch_kernel(moe_route_kernel, dim3(a.p), dim3(kRouteThreads), s, a);
  if (err == cudaSuccess) note_launch();
  return err;
}

cudaError_t launch_moe_dispatch(const MoeDispatchArgs& a, bool fp8, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((a.tokens + kTokensPerCta - 1) / kTokensPerCta), a.p);
  cudaError_t err = fp8 ? launch_kernel(moe_dispatch_kernel<true>, grid, dim3(kThreads), s, a)
                        : launch_kernel(moe_dispatch_kernel<false>, grid, dim3(kThreads), s, a);
  if (err == cudaSuccess) note_launch();
  return err;
}

cudaError_t launch_moe_combine(const MoeCombineArgs& a, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((a.tokens + kTokensPerCta - 1) / kTokensPerCta), a.p);
  cudaError_t err = launch_kernel(moe_combine_kernel, grid, dim3(kThreads), s, a);
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace ccl
