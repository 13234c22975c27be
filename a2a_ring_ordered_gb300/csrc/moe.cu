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
#include <cooperative_groups.h>
#include <cuda_fp8.h>

#include "device_common.cuh"

namespace ccl {
namespace {

constexpr int kRouteThreads = 1024;                  // 32 warps
constexpr int kRouteSub = 4;                         // items per thread per tile
constexpr int kRouteTile = kRouteThreads * kRouteSub;  // 4096 items
constexpr int kRouteRows = kRouteSub * 32;           // one count row per (sub-tile, warp)
constexpr int kRouteMaxCluster = 8;                  // portable cluster size

__device__ __forceinline__ int route_dest(const MoeRouteArgs& a, const int32_t* ids, uint64_t item,
                                          uint64_t hi) {
  if (item >= hi) return -1;
  const int e = ids[item];
  return (e >= 0 && e < a.num_experts) ? e / a.epr : -1;
}

// Routing of one source is split over a cluster of up to 8 CTAs (grid x =
// cluster rank, grid y = source); CTA c owns a contiguous segment of the
// (token, choice) items.
//
// 1. Each CTA counts its segment's items per destination (__match_any_sync
//    groups a warp's lanes by destination; one shared atomic per group).
// 2. After a cluster barrier, CTA c adds up the counts of CTAs 0..c-1 from
//    their shared memory (distributed shared memory), which is the number of
//    earlier same-destination items of the source: its base.  The last CTA
//    also writes the source's row of the p x p counts.
// 3. The segment is walked in tiles of 4096 items, thread t holding items
//    t, t + 1024, t + 2048, t + 3072 of the tile; in a warp, __match_any_sync
//    gives every item its rank among the earlier same-destination lanes, the
//    group leader stores the group's size in the (sub-tile, warp) row of a
//    count table, and a warp-shuffle scan down each destination's column (in
//    item order: sub-tile, then warp) on top of the running count turns the
//    table into the number of earlier same-destination items: item's slot =
//    table entry + its rank in the warp.
// A second cluster barrier keeps every CTA's counts alive until the others
// have read them.
__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(const __grid_constant__ MoeRouteArgs a,
                                                                 uint64_t seg) {
  namespace cg = cooperative_groups;
  __shared__ int table[kRouteRows][kMoeMaxRanks + 1];  // +1: conflict-free column scan
  __shared__ int hist[kMoeMaxRanks];
  __shared__ int run[kMoeMaxRanks];
  pdl_enter();
  cg::cluster_group cluster = cg::this_cluster();
  const int c = static_cast<int>(cluster.block_rank());
  const int s = blockIdx.y;
  const int p = a.p;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t* ids = a.ids[s];
  int32_t* slots = a.slots[s];
  const uint64_t lo = min(static_cast<uint64_t>(c) * seg, a.items);
  const uint64_t hi = min(lo + seg, a.items);
  for (int d = tid; d < p; d += kRouteThreads) hist[d] = 0;
  __syncthreads();

  // 1. per-destination counts of the segment
  for (uint64_t b = lo; b < hi; b += kRouteTile) {
    int d[kRouteSub];
#pragma unroll
    for (int j = 0; j < kRouteSub; ++j) d[j] = route_dest(a, ids, b + j * kRouteThreads + tid, hi);
#pragma unroll
    for (int j = 0; j < kRouteSub; ++j) {
      const unsigned same = __match_any_sync(0xFFFFFFFFu, d[j]);
      if (d[j] >= 0 && lane == __ffs(same) - 1) atomicAdd(&hist[d[j]], __popc(same));
    }
  }
  cluster.sync();

  // 2. base = items of the same source and destination in earlier segments
  if (tid < p) {
    int base = 0;
    for (int q = 0; q < c; ++q) base += cluster.map_shared_rank(hist, q)[tid];
    run[tid] = base;
    if (c == static_cast<int>(cluster.num_blocks()) - 1)
      a.counts[static_cast<uint64_t>(s) * p + tid] = base + hist[tid];
  }
  cluster.barrier_arrive();
  __syncthreads();

  // 3. slots, tile by tile
  for (uint64_t b = lo; b < hi; b += kRouteTile) {
    int d[kRouteSub], rank[kRouteSub];
#pragma unroll
    for (int j = 0; j < kRouteSub; ++j) d[j] = route_dest(a, ids, b + j * kRouteThreads + tid, hi);
    // this warp's rows are read only by this warp (slots of the previous
    // tile) and by the scan, which a __syncthreads has closed
    for (int i = lane; i < kRouteSub * p; i += 32) table[(i / p) * 32 + warp][i % p] = 0;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kRouteSub; ++j) {
      const unsigned same = __match_any_sync(0xFFFFFFFFu, d[j]);
      rank[j] = __popc(same & ((1u << lane) - 1u));
      if (d[j] >= 0 && rank[j] == 0) table[j * 32 + warp][d[j]] = __popc(same);
    }
    __syncthreads();
    for (int dd = warp; dd < p; dd += 32) {  // warp w scans columns w and w + 32
      int acc = run[dd];
#pragma unroll
      for (int j = 0; j < kRouteSub; ++j) {
        const int v = table[j * 32 + lane][dd];
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += t;
        }
        table[j * 32 + lane][dd] = acc + incl - v;
        acc += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (lane == 0) run[dd] = acc;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kRouteSub; ++j) {
      const uint64_t item = b + j * kRouteThreads + tid;
      if (item < hi) slots[item] = (d[j] >= 0) ? table[j * 32 + warp][d[j]] + rank[j] : -1;
    }
  }
  cluster.barrier_wait();
}

constexpr int kMaxTokensPerCta = 16;


// base[d] = rows of destination d sent by sources before s.
__device__ __forceinline__ void row_bases(const int64_t* counts, int p, int s, int64_t* base) {
  for (int d = threadIdx.x; d < p; d += blockDim.x) {
    int64_t acc = 0;
    for (int q = 0; q < s; ++q) acc += counts[static_cast<uint64_t>(q) * p + d];
    base[d] = acc;
  }
}

// Destination rank and row of each (token, choice) of the CTA's tokens; -1
// when the id is out of range, the item was not routed, or the row lies past
// the destination buffer's capacity (a short buffer loses rows, never memory).
// Combine also gathers each choice's gate weight (`weights` non-NULL).
template <typename Args>
__device__ __forceinline__ void token_rows(const Args& a, int s, uint64_t t0, int tpc, const int64_t* base,
                                           int (*dest)[kMoeMaxK], int64_t (*pos)[kMoeMaxK],
                                           int (*expert)[kMoeMaxK], const float* const* weights,
                                           float (*wt)[kMoeMaxK]) {
  const int k = a.k;
  for (int i = threadIdx.x; i < tpc * k; i += blockDim.x) {
    const int tt = i / k, j = i - (i / k) * k;
    const uint64_t t = t0 + tt;
    int d = -1, e = -1;
    int64_t row = -1;
    if (t < a.tokens) {
      e = a.ids[s][t * k + j];
      const int slot = a.slots[s][t * k + j];
      if (weights != nullptr) wt[tt][j] = weights[s][t * k + j];
      if (e >= 0 && e < a.num_experts && slot >= 0) {
        d = e / a.epr;
        row = base[d] + slot;
        if (static_cast<uint64_t>(row) >= a.cap[d]) d = -1;
      }
    }
    dest[tt][j] = d;
    pos[tt][j] = row;
    if (expert != nullptr) expert[tt][j] = e;
  }
}

// One CTA per (tpc tokens, source).  The CTA's (token, vector) items are one
// flat index range, U items per thread with their loads issued together; tpc
// is at most what one pass covers (see dispatch_tokens_per_cta).  Each vector of a token row is loaded once and stored to
// the token's k destination rows.  bf16: 8 elements (16 bytes) per item.
// FP8: 16 elements per item, and the 8 consecutive lanes holding a
// 128-element block reduce its amax with shuffles (a row is a multiple of 128
// elements, so an aligned group of 8 items never straddles two blocks or two
// tokens); the block's scaling factor scale = amax / 448 is stored for
// dequantisation and code = e4m3(x / scale), rounded to nearest even and
// saturating (the DeepSeek-V3 per-tile scaling that section 7.4 of
// "Networks and Collective Communication" points to).
template <bool FP8, int U>
__global__ void __launch_bounds__(kThreads) moe_dispatch_kernel(const __grid_constant__ MoeDispatchArgs a) {
  constexpr int EPI = FP8 ? 16 : 8;  // elements per item
  constexpr int WI = EPI / 2;        // 32-bit words of bf16 input per item
  __shared__ int64_t base[kMoeMaxRanks];
  __shared__ int64_t pos[kMaxTokensPerCta][kMoeMaxK];
  __shared__ int dest[kMaxTokensPerCta][kMoeMaxK];
  __shared__ int expert[kMaxTokensPerCta][kMoeMaxK];
  __shared__ char* rowp[kMaxTokensPerCta][kMoeMaxK];   // destination row, NULL if none
  __shared__ float* sclp[kMaxTokensPerCta][kMoeMaxK];  // its block scales (FP8)
  pdl_enter();
  const int s = blockIdx.y;
  const int k = a.k, tpc = a.tpc;
  const uint64_t h = a.hidden;
  const uint64_t t0 = static_cast<uint64_t>(blockIdx.x) * tpc;
  row_bases(a.counts, a.p, s, base);
  __syncthreads();
  token_rows(a, s, t0, tpc, base, dest, pos, expert, nullptr, static_cast<float (*)[kMoeMaxK]>(nullptr));
  __syncthreads();
  for (int i = threadIdx.x; i < tpc * k; i += kThreads) {
    const int tt = i / k, j = i - (i / k) * k;
    const int d = dest[tt][j];
    const uint64_t row = static_cast<uint64_t>(pos[tt][j]);
    rowp[tt][j] = (d >= 0) ? static_cast<char*>(a.recv[d]) + row * h * (FP8 ? 1 : 2) : nullptr;
    sclp[tt][j] = (FP8 && d >= 0) ? a.scales[d] + row * (h / 128) : nullptr;
    if (a.rexp_given && d >= 0 && a.rexp[d] != nullptr) a.rexp[d][row] = expert[tt][j];
  }
  __syncthreads();
  const uint32_t nv = static_cast<uint32_t>(h / EPI);  // items per token row
  const uint64_t left = a.tokens - t0;
  const uint32_t ntok = static_cast<uint32_t>(left < static_cast<uint64_t>(tpc) ? left : tpc);
  const uint32_t total = ntok * nv;
  const char* xs = static_cast<const char*>(a.x[s]);
  for (uint32_t f0 = threadIdx.x; f0 < total; f0 += kThreads * U) {
    uint32_t w[U][WI];
    uint32_t tt[U], v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t f = f0 + u * kThreads;
      tt[u] = f / nv;
      v[u] = f - tt[u] * nv;
      if (f < total) {
        const char* row = xs + (t0 + tt[u]) * h * 2;
        if constexpr (FP8) {
          // the item's 32 bytes are two 16-byte loads; they allocate in L1 so
          // that the second finds the sector the first brought in
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint4 g = ld_l1_16(row + static_cast<uint64_t>(v[u]) * 32 + 16 * q);
            w[u][4 * q] = g.x;
            w[u][4 * q + 1] = g.y;
            w[u][4 * q + 2] = g.z;
            w[u][4 * q + 3] = g.w;
          }
        } else {
          load_raw<kBF16, 8>(row, static_cast<uint64_t>(v[u]) * EPI, w[u]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (f0 + u * kThreads >= total) continue;  // whole aligned groups of 8 lanes drop out together
      if constexpr (!FP8) {
        const uint4 q = make_uint4(w[u][0], w[u][1], w[u][2], w[u][3]);
        for (int j = 0; j < k; ++j) {
          char* row = rowp[tt[u]][j];
          if (row != nullptr) st_stream16(row + static_cast<uint64_t>(v[u]) * 16, q);
        }
      } else {
        float x[16];
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          x[e] = widen<kBF16>(w[u], e);
          amax = fmaxf(amax, fabsf(x[e]));
        }
        const unsigned group = 0xFFu << (threadIdx.x & 24);
#pragma unroll
        for (int off = 4; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(group, amax, off));
        // the block's scaling factor; quantisation divides by it (one
        // correctly rounded fp32 division per element)
        const float scale = (amax > 0.0f) ? __fdiv_rn(amax, 448.0f) : 1.0f;
        // two codes per conversion (element 2e in the low byte, 2e+1 above it)
        uint32_t q[4] = {0, 0, 0, 0};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t c2 = __nv_cvt_float2_to_fp8x2(
              make_float2(__fdiv_rn(x[2 * e], scale), __fdiv_rn(x[2 * e + 1], scale)), __NV_SATFINITE, __NV_E4M3);
          q[e >> 1] |= (c2 & 0xFFFFu) << (16 * (e & 1));
        }
        const uint4 qv = make_uint4(q[0], q[1], q[2], q[3]);
        const uint64_t blk = v[u] / 8;  // 8 items of 16 = one 128-element block
        const bool lead = (threadIdx.x & 7) == 0;
        for (int j = 0; j < k; ++j) {
          char* row = rowp[tt[u]][j];
          if (row == nullptr) continue;
          st_stream16(row + static_cast<uint64_t>(v[u]) * 16, qv);
          if (lead) sclp[tt[u]][j][blk] = scale;
        }
      }
    }
  }
}

// One CTA per (tpc tokens, source), the (token, vector) items a flat range as
// in dispatch: token t's output is the bf16 of the fp32 sum over choices j of
// w[t][j] * y_j, in choice order (each product and each sum rounded; no fused
// multiply-add).  The k rows' loads are issued before any is combined.
__global__ void __launch_bounds__(kThreads) moe_combine_kernel(const __grid_constant__ MoeCombineArgs a) {
  __shared__ int64_t base[kMoeMaxRanks];
  __shared__ int64_t pos[kMaxTokensPerCta][kMoeMaxK];
  __shared__ int dest[kMaxTokensPerCta][kMoeMaxK];
  __shared__ float wt[kMaxTokensPerCta][kMoeMaxK];
  pdl_enter();
  const int s = blockIdx.y;
  const int k = a.k, tpc = a.tpc;
  const uint64_t t0 = static_cast<uint64_t>(blockIdx.x) * tpc;
  row_bases(a.counts, a.p, s, base);
  __syncthreads();
  token_rows(a, s, t0, tpc, base, dest, pos, static_cast<int (*)[kMoeMaxK]>(nullptr), a.weights, wt);
  __syncthreads();
  const uint64_t h = a.hidden;
  const uint32_t nv = static_cast<uint32_t>(h / 8);
  const uint64_t left = a.tokens - t0;
  const uint32_t ntok = static_cast<uint32_t>(left < static_cast<uint64_t>(tpc) ? left : tpc);
  const uint32_t total = ntok * nv;
  for (uint32_t f = threadIdx.x; f < total; f += kThreads) {
    const uint32_t tt = f / nv, v = f - (f / nv) * nv;
    float acc[8];
    bool have = false;
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint32_t raw[8][4];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int j = j0 + b;
        if (j < k && dest[tt][j] >= 0)
          load_raw<kBF16, 8>(a.y[dest[tt][j]], static_cast<uint64_t>(pos[tt][j]) * h + static_cast<uint64_t>(v) * 8, raw[b]);
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
    store_raw<kBF16, 8>(a.out[s], (t0 + tt) * h + static_cast<uint64_t>(v) * 8, w);
  }
}

// Combine's tokens per CTA: the fewest (at most 16) that make the CTA's items
// a whole number of passes of `per_pass` items.
__host__ int tokens_per_cta(uint64_t items_per_token, uint64_t per_pass) {
  for (int t = 1; t <= kMaxTokensPerCta; ++t)
    if ((items_per_token * static_cast<uint64_t>(t)) % per_pass == 0) return t;
  return 8;
}

// Dispatch's tokens per CTA: as many as fit in one pass of `per_pass` items
// (at least 1, at most 16), idle lanes in that pass notwithstanding.  Measured
// on GB300 (p=8 x 4096 tokens, hidden 7168, top-8 of 256): 1 / 2 / 4 / 8 / 16
// tokens per CTA ran the FP8 dispatch at 6.77 / 6.69 / 6.48 / 6.28 / 6.25
// TB/s and the bf16 one at 6.86 / 6.67 / 6.58 / 6.48 / 6.33 -- many short
// CTAs keep more token rows streaming at once and leave a shorter tail.  The
// combine went the other way (2 tokens 6.76, 1 token 6.52) and keeps whole
// passes.
__host__ int dispatch_tokens_per_cta(uint64_t items_per_token, uint64_t per_pass) {
  const uint64_t t = items_per_token == 0 ? kMaxTokensPerCta : per_pass / items_per_token;
  return static_cast<int>(t < 1 ? 1 : (t > kMaxTokensPerCta ? kMaxTokensPerCta : t));
}

}  // namespace

cudaError_t launch_moe_route(const MoeRouteArgs& a, cudaStream_t s) {
  // cluster size: one CTA per 4096-item tile, up to 8; segments whole tiles
  const uint64_t tiles = (a.items + kRouteTile - 1) / kRouteTile;
  const unsigned cl = static_cast<unsigned>(tiles < 1 ? 1 : (tiles > kRouteMaxCluster ? kRouteMaxCluster : tiles));
  const uint64_t seg = ((tiles + cl - 1) / cl) * kRouteTile;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cl, static_cast<unsigned>(a.p));
  cfg.blockDim = dim3(kRouteThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = CCL_PDL ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cl;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t err = cudaLaunchKernelEx(&cfg, moe_route_kernel, a, seg);
  if (err == cudaSuccess) note_launch();
  return err;
}

cudaError_t launch_moe_dispatch(const MoeDispatchArgs& args, bool fp8, cudaStream_t s) {
  // items per thread: FP8 (32-byte loads) 1, bf16 (16-byte) 4.  Measured on
  // GB300 for the FP8 dispatch of the MoE EP workload (one correctly rounded
  // division per element): 1 / 2 / 4 items 356 / 380 / 372 us.
  constexpr int kU8 = 1, kU16 = 4;
  MoeDispatchArgs a = args;
  a.tpc = dispatch_tokens_per_cta(a.hidden / (fp8 ? 16 : 8), static_cast<uint64_t>(kThreads) * (fp8 ? kU8 : kU16));
  const dim3 grid(static_cast<unsigned>((a.tokens + a.tpc - 1) / a.tpc), a.p);
  cudaError_t err = fp8 ? launch_kernel(moe_dispatch_kernel<true, kU8>, grid, dim3(kThreads), s, a)
                        : launch_kernel(moe_dispatch_kernel<false, kU16>, grid, dim3(kThreads), s, a);
  if (err == cudaSuccess) note_launch();
  return err;
}

cudaError_t launch_moe_combine(const MoeCombineArgs& args, cudaStream_t s) {
  MoeCombineArgs a = args;
  a.tpc = tokens_per_cta(a.hidden / 8, kThreads);
  const dim3 grid(static_cast<unsigned>((a.tokens + a.tpc - 1) / a.tpc), a.p);
  cudaError_t err = launch_kernel(moe_combine_kernel, grid, dim3(kThreads), s, a);
  if (err == cudaSuccess) note_launch();
  return err;
}

}  // namespace ccl
