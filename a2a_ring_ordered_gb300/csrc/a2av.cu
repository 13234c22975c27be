// a2av.cu -- all-to-all(v) block transpose: MoE dispatch / combine
// ("Networks and Collective Communication" section 4.1: device i's block j
// goes to device j, a transpose; section 7.4: MoE dispatch and combine).
//
// Destination j's buffer holds one block from every source i, in source
// order: block i is rows [cs_i, cs_{i+1}) of recv[j] and starts at row rs_i
// of send[i].  The plain all-to-all takes cs and rs from the chunk rule
// (cs_i = i * len(j), rs_i = off(j), one element per row); the all-to-allv
// takes rs from a row-prefix table in the kernel's parameter block and scans
// the table's column for cs on the device.  Nothing is allocated and any
// p <= 85 is one launch (the plain all-to-all: any p).
//
// Work is cut into tiles of destination space (4 - 32 KB by the call's
// size; boundaries on 512 bytes of the destination's address), one CTA per
// tile, so the work is balanced by bytes however skewed the counts are.
// The CTA puts the destination's block bounds in shared memory, and each
// thread writes whole aligned 16-byte destination units (a warp's 32 stores
// fill whole 128-byte lines):
//  * a unit inside one block is one aligned 16-byte source load when source
//    and destination share the 16-byte phase, else two aligned source
//    granules whose bytes are funnel-shifted into place;
//  * a unit that straddles blocks (block edges off the 16-byte grid) is
//    assembled from its elements and stored whole.  When blocks are small
//    (the host's choice: STAGE) this goes through the tile's small-block
//    stage: before the aligned units, the whole CTA issues asynchronous
//    copies of the elements of all such units at once (each element's
//    aligned source word, from the block holding it) into shared memory;
//    after them, each unit is assembled from the stage.  A unit not inside
//    one block holds one of the destination's p + 1 block edges, so the
//    stage holds at most p + 1 units.  With large blocks a tile holds one
//    such unit or none, and the thread that meets it loads its elements;
//  * only the units at the ends of the destination buffer, partly outside
//    it, are stored element by element.
// Every load touches only aligned granules (16 bytes, or the 4-byte words
// of the stage) that hold at least one byte of a block.  HBM traffic: one
// read and one write of every moved byte.
#include "device_common.cuh"
#include "realign.cuh"

namespace ccl {
namespace {


// Bounds of destination j's blocks, in bytes: block i covers destination
// bytes [dst0 + cs[i], dst0 + cs[i+1]) and its first byte comes from src[i].
struct Blocks {
  uint64_t* cs;       // p + 1 entries (shared memory)
  const char** src;   // p entries (shared memory)
  uintptr_t dst0;
  int p;
};

// The block holding destination byte offset `x` (x < cs[p]): the last i in
// [lo, hi] whose block starts at or before x (an empty block starts where
// the next one does, so the one found is never empty).
__device__ __forceinline__ int block_of(const Blocks& b, uint64_t x, int lo, int hi) {
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (b.cs[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ uint32_t load_elem(const char* p, int e) {
  return (e == 4) ? ld_once4(p) : ld_once2(p);
}

// Destination unit [ua, ua + 16) element by element: the valid bytes are
// [max(ua, vlo), min(ua + 16, vhi)); block i holds the first of them.
// Inside the buffer the elements are assembled and stored as one 16-byte
// unit; at the buffer's ends each element is stored on its own.
__device__ __noinline__ void unit_by_elements(const uint64_t* cs, const char* const* src, uintptr_t dst0,
                                              uintptr_t ua, uintptr_t vlo, uintptr_t vhi, int i, int e) {
  const uintptr_t x0 = ua > vlo ? ua : vlo;
  const uintptr_t x1 = ua + 16 < vhi ? ua + 16 : vhi;
  const bool whole = x0 == ua && x1 == ua + 16;
  uint32_t w[4] = {0, 0, 0, 0};
  for (uintptr_t x = x0; x < x1; x += e) {
    const uint64_t off = x - dst0;
    while (cs[i + 1] <= off) ++i;
    const uint32_t v = load_elem(src[i] + (off - cs[i]), e);
    if (whole) {
      const int k = static_cast<int>(x - ua);
      w[k >> 2] |= (e == 4) ? v : (v << (8 * (k & 3)));
    } else if (e == 4) {
      st_stream4(reinterpret_cast<void*>(x), v);
    } else {
      st_stream2(reinterpret_cast<void*>(x), v);
    }
  }
  if (whole) st_stream16(reinterpret_cast<void*>(ua), make_uint4(w[0], w[1], w[2], w[3]));
}

// The calling thread's units of a tile that lie inside one block whose
// source is off the destination's 16-byte phase, element by element (for a
// kernel launched without SHIFT, where no such block exists).
__device__ __noinline__ void shifted_units(const uint64_t* cs, const char* const* src, uintptr_t dst0,
                                           uintptr_t tlo, uintptr_t vlo, uintptr_t vhi, int ia, int ib,
                                           int units_per_thread, int e) {
  const Blocks b{const_cast<uint64_t*>(cs), const_cast<const char**>(src), dst0, 0};
  for (int w = 0; w < units_per_thread; ++w) {
    const uintptr_t ua = tlo + 16 * static_cast<uintptr_t>(w * kThreads + threadIdx.x);
    if (ua < vlo || ua + 16 > vhi) continue;
    const int i = block_of(b, ua - b.dst0, ia, ib);
    const uintptr_t bs = b.dst0 + b.cs[i], be = b.dst0 + b.cs[i + 1];
    if (ua + 16 > be || ((reinterpret_cast<uintptr_t>(b.src[i]) + (ua - bs)) & 15) == 0) continue;
    unit_by_elements(b.cs, b.src, b.dst0, ua, vlo, vhi, i, e);
  }
}

// The small-block stage.  The cuts of a tile whose bytes [vlo, vhi) touch
// blocks ia .. ib are, in ascending order, vlo, the starts of blocks
// ia + 1 .. ib and vhi.  A destination unit not inside one block holds a cut
// off the 16-byte grid (a block edge, or an end of the buffer), so staging
// the unit of every such cut, once, covers all of them: cut k stages unit
// at(k) & ~15 when at(k) is off the grid and cut k - 1 does not lie inside
// the same unit.  Staged unit k's bytes go to [16k, 16k + 16) of the stage.
struct Cuts {
  const uint64_t* cs;
  uintptr_t dst0, vlo, vhi;
  int ia, n;  // n = ib - ia + 2 cuts
  __device__ __forceinline__ uintptr_t at(int k) const {
    return k == 0 ? vlo : (k == n - 1 ? vhi : dst0 + cs[ia + k]);
  }
  __device__ __forceinline__ bool stages(int k) const {
    const uintptr_t x = at(k);
    return (x & 15) != 0 && (k == 0 || at(k - 1) <= (x & ~static_cast<uintptr_t>(15)));
  }
};

// 4-byte asynchronous copy global -> shared (no register holds the data,
// and the thread does not wait for it until cp_async_wait_all()).
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Slots of the stage: element m of staged unit k is the aligned 4-byte
// source word holding it, word[8k + m]; half[8k + m] says which half of the
// word a 2-byte element is.
constexpr int kStageSlots = 8;

// Issues the copies of the staged units' elements inside [vlo, vhi), the
// whole CTA over all staged units at once; returns whether this thread
// issued any.  Each copy reads the aligned 4-byte word that holds the
// element (a word holding one byte of a block lies in a mapped page).
__device__ __forceinline__ bool stage_issue(const Cuts& cu, const Blocks& b, int ib, int e, uint32_t* word,
                                            uint8_t* half) {
  const int lg = (e == 4) ? 2 : 3;  // log2 of the elements per unit
  const int items = cu.n << lg;
  bool issued = false;
  for (int it = threadIdx.x; it < items; it += kThreads) {
    const int k = it >> lg, m = it & ((1 << lg) - 1);
    if (!cu.stages(k)) continue;
    const uintptr_t x = (cu.at(k) & ~static_cast<uintptr_t>(15)) + static_cast<uintptr_t>(m * e);
    if (x < cu.vlo || x >= cu.vhi) continue;
    const uint64_t off = x - b.dst0;
    // the block holding x: a few steps from the block starting at cut k
    int i = cu.ia + k < ib ? cu.ia + k : ib;
    while (i > cu.ia && b.cs[i] > off) --i;
    while (i < ib && b.cs[i + 1] <= off) ++i;
    const uintptr_t src = reinterpret_cast<uintptr_t>(b.src[i]) + (off - b.cs[i]);
    cp_async4(word + kStageSlots * k + m, reinterpret_cast<const void*>(src & ~static_cast<uintptr_t>(3)));
    half[kStageSlots * k + m] = static_cast<uint8_t>((src >> 1) & 1);
    issued = true;
  }
  return issued;
}

// Stores the staged units (their copies complete and visible): whole where
// the unit lies inside [vlo, vhi), element by element at the destination
// buffer's ends.
__device__ __forceinline__ void stage_store(const Cuts& cu, int e, const uint32_t* word, const uint8_t* half) {
  for (int k = threadIdx.x; k < cu.n; k += kThreads) {
    if (!cu.stages(k)) continue;
    const uintptr_t ua = cu.at(k) & ~static_cast<uintptr_t>(15);
    const uintptr_t x0 = ua > cu.vlo ? ua : cu.vlo, x1 = ua + 16 < cu.vhi ? ua + 16 : cu.vhi;
    uint32_t w[4] = {0, 0, 0, 0};
    for (uintptr_t x = x0; x < x1; x += e) {
      const int kb = static_cast<int>(x - ua), m = kb / e;
      uint32_t v = word[kStageSlots * k + m];
      if (e == 2) v = (v >> (16 * half[kStageSlots * k + m])) & 0xFFFFu;
      if (x0 == ua && x1 == ua + 16) w[kb >> 2] |= v << (8 * (kb & 3));
      else if (e == 4) st_stream4(reinterpret_cast<void*>(x), v);
      else st_stream2(reinterpret_cast<void*>(x), v);
    }
    if (x0 == ua && x1 == ua + 16) st_stream16(reinterpret_cast<void*>(ua), make_uint4(w[0], w[1], w[2], w[3]));
  }
}

// SHIFT: some block's source and destination differ in 16-byte phase (the
// host checks); without it each thread keeps 8 units' loads in flight,
// with it 4 units' two granules.  STAGE: the units that straddle blocks go
// through the small-block stage, whose copies are issued before the tile's
// aligned units and land while those are in flight; without it (no block
// edge off the 16-byte grid, or blocks large enough that a tile holds few
// edges) the thread that meets such a unit assembles it from element
// loads.  64 registers, 4 CTAs per SM.
template <class P, bool SHIFT, bool STAGE, uint32_t TILE>
__global__ void __launch_bounds__(kThreads, 4) a2a_kernel(const __grid_constant__ P a) {
  __shared__ uint64_t s_cs[P::kCap + 1];
  __shared__ const char* s_src[P::kCap];
  // the stage: one unit per cut, at most p + 1
  constexpr int kStageWords = STAGE ? (P::kCap + 1) * kStageSlots : 1;
  __shared__ uint32_t s_word[kStageWords];
  __shared__ uint8_t s_half[kStageWords];
  bool entered = false;
  const int p = a.p;
  const uint64_t rb = a.row_bytes;
  const uint64_t total_tiles = a.tile0[a.ndest];
  // Tile size and 16-byte units per thread (8 for 32 KB tiles, 1 for 4 KB
  // ones, 2 and 4 between).  The phase-shifting kernels take it from the template (one
  // instantiation per tile size), the others from the parameters: measured
  // on GB300, the other way round cost up to 10 % (the template form of the
  // unshifted kernel spilled 16 bytes: p = 8 all-to-all at 8 MiB per rank
  // 1.01 -> 0.91 of the copy bandwidth; the parameter form of the shifted
  // one ran p = 72 at 0.98 instead of 1.01).
  const uint32_t tile = SHIFT ? TILE : a.tile_bytes;
  const int units_per_thread = static_cast<int>(tile / 16 / kThreads);
  for (uint64_t t = blockIdx.x; t < total_tiles; t += gridDim.x) {
    // this tile's destination (uniform over the CTA)
    int c = 0;
    {
      int lo = 0, hi = a.ndest - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.tile0[mid] <= t) lo = mid; else hi = mid - 1;
      }
      c = lo;
    }
    const int j = a.j0 + c;
    // block bounds of destination j, in bytes
    if (a.plain) {
      const uint64_t len = a.q + (static_cast<uint64_t>(j) < a.rem ? 1 : 0);
      const uint64_t off = static_cast<uint64_t>(j) * a.q + (static_cast<uint64_t>(j) < a.rem ? j : a.rem);
      for (int i = threadIdx.x; i <= p; i += kThreads) {
        s_cs[i] = static_cast<uint64_t>(i) * len * rb;
        if (i < p) s_src[i] = a.send[i] + off * rb;
      }
    } else if (threadIdx.x < 32) {
      // exclusive scan of the column's counts (rows of source i for j)
      const int stride = a.ndest + 1;
      uint64_t carry = 0;
      for (int i0 = 0; i0 < p; i0 += 32) {
        const int i = i0 + static_cast<int>(threadIdx.x);
        uint64_t rs = 0, cnt = 0;
        if (i < p) {
          rs = static_cast<uint64_t>(a.table[i * stride + c]);
          cnt = static_cast<uint64_t>(a.table[i * stride + c + 1]) - rs;
        }
        uint64_t incl = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
          if (static_cast<int>(threadIdx.x) >= d) incl += v;
        }
        if (i < p) {
          s_cs[i] = (carry + incl - cnt) * rb;
          s_src[i] = a.send[i] + rs * rb;
        }
        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (threadIdx.x == 0) s_cs[p] = carry * rb;
    }
    __syncthreads();

    Blocks b{s_cs, s_src, reinterpret_cast<uintptr_t>(a.recv[j]), p};
    const uintptr_t vlo0 = b.dst0, vhi0 = b.dst0 + s_cs[p];
    const uintptr_t tlo = (b.dst0 & ~static_cast<uintptr_t>(511)) + (t - a.tile0[c]) * tile;
    const uintptr_t vlo = tlo > vlo0 ? tlo : vlo0;
    const uintptr_t vhi = tlo + tile < vhi0 ? tlo + tile : vhi0;
    // the blocks this tile touches
    const int ia = block_of(b, vlo - b.dst0, 0, p - 1);
    const int ib = block_of(b, vhi - 1 - b.dst0, ia, p - 1);
    if (!entered) {
      // The CTA's first tile (one CTA per tile: its only one): its source
      // bytes are prefetched into L2 before waiting on the previous grid
      // (the block bounds come from the parameters alone), so that the loads
      // of the first wave overlap the previous grid's drain and every CTA's
      // second pass (SHIFT) finds its data on the way.  Measured on GB300
      // against no prefetch: MoE dispatch / combine (p = 8, 8 KiB rows)
      // 0.91 -> 1.05 of the copy bandwidth, p = 72 all-to-all 0.86 -> 1.01
      // at 8 MiB per rank.  The prefetch is a hint and cannot change a
      // result: L2 is the device's point of coherence, and the loads after
      // pdl_enter() read L2, not L1 (which a prefetch does not fill).
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
      for (int i = ia + warp; i <= ib; i += kThreads / 32) {
        const uintptr_t bs = b.dst0 + s_cs[i], be = b.dst0 + s_cs[i + 1];
        const uintptr_t lo = vlo > bs ? vlo : bs, hi = vhi < be ? vhi : be;
        if (lo >= hi) continue;
        const uintptr_t s0 = reinterpret_cast<uintptr_t>(s_src[i]) + (lo - bs), s1 = s0 + (hi - lo);
        for (uintptr_t line = (s0 & ~static_cast<uintptr_t>(127)) + 128 * lane; line < s1; line += 128 * 32)
          prefetch_l2(reinterpret_cast<const void*>(line));
      }
      pdl_enter();
      entered = true;
    }

    const Cuts cu{s_cs, b.dst0, vlo, vhi, ia, ib - ia + 2};
    const bool cut = ia < ib || ((vlo | vhi) & 15) != 0;  // the tile may hold a staged unit (uniform)
    bool issued = false;
    if constexpr (STAGE) {
      if (cut) issued = stage_issue(cu, b, ib, a.elem, s_word, s_half);
    }

    // units t, t + kThreads, ... of the tile, U at a time with their loads
    // issued together
    constexpr int U = SHIFT ? 4 : 8;
    bool odd = false;  // a unit inside one block off its source's 16-byte phase
#pragma unroll 1
    for (int w0 = 0; w0 < units_per_thread; w0 += U) {
      uint4 g0[U], g1[U];
      // per unit: -1 outside the tile's bytes, else (block << 5) | (whole << 4) | phase
      int code[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uintptr_t ua = tlo + 16 * static_cast<uintptr_t>((w0 + u) * kThreads + threadIdx.x);
        code[u] = -1;
        if (ua + 16 <= vlo || ua >= vhi) continue;
        const uintptr_t x0 = ua > vlo ? ua : vlo;
        const int i = (ia == ib) ? ia : block_of(b, x0 - b.dst0, ia, ib);
        code[u] = i << 5;
        const uintptr_t bs = b.dst0 + s_cs[i], be = b.dst0 + s_cs[i + 1];
        if (ua >= bs && ua + 16 <= be) {
          const uintptr_t src = reinterpret_cast<uintptr_t>(s_src[i]) + (ua - bs);
          const int dl = static_cast<int>(src & 15);
          const char* g = reinterpret_cast<const char*>(src - dl);
          if constexpr (SHIFT) {
            code[u] |= 16 | dl;
            g0[u] = ld_l1_16(g);
            if (dl != 0) g1[u] = ld_l1_16(g + 16);
          } else if (dl == 0) {
            code[u] |= 16;
            g0[u] = ld_once16(g);
          } else if constexpr (STAGE) {
            odd = true;  // (never: the host launches SHIFT then)
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uintptr_t ua = tlo + 16 * static_cast<uintptr_t>((w0 + u) * kThreads + threadIdx.x);
        if (code[u] < 0) continue;
        if (code[u] & 16) {
          uint4 o = g0[u];
          if constexpr (SHIFT) {
            if (code[u] & 15) o = realign16(g0[u], g1[u], code[u] & 15);
          }
          st_stream16(reinterpret_cast<void*>(ua), o);
        } else if constexpr (!STAGE) {
          unit_by_elements(s_cs, s_src, b.dst0, ua, vlo, vhi, code[u] >> 5, a.elem);
        }
        // else: not inside one block, stored by the stage below
      }
    }
    if constexpr (STAGE) {
      if constexpr (!SHIFT) {
        if (odd) shifted_units(s_cs, s_src, b.dst0, tlo, vlo, vhi, ia, ib, units_per_thread, a.elem);
      }
      if (cut) {
        cp_async_wait_all();
        if (__syncthreads_or(issued)) stage_store(cu, a.elem, s_word, s_half);
      }
    }
    __syncthreads();  // the block bounds and the stage are rewritten for the next tile
  }
  if (!entered) pdl_enter();
}

template <class P, bool STAGE>
cudaError_t launch_staged(const P& a, bool shift, const dim3& grid, cudaStream_t s) {
  constexpr uint32_t kBig = static_cast<uint32_t>(kA2ATileBytes), kSmall = static_cast<uint32_t>(kA2ASmallTileBytes);
  constexpr uint32_t k8 = static_cast<uint32_t>(kA2AMidTileBytes[0]), k16 = static_cast<uint32_t>(kA2AMidTileBytes[1]);
  if (!shift) return launch_kernel(a2a_kernel<P, false, STAGE, kBig>, grid, dim3(kThreads), s, a);  // tile size at run time
  if (a.tile_bytes == kSmall) return launch_kernel(a2a_kernel<P, true, STAGE, kSmall>, grid, dim3(kThreads), s, a);
  if (a.tile_bytes == k8) return launch_kernel(a2a_kernel<P, true, STAGE, k8>, grid, dim3(kThreads), s, a);
  if (a.tile_bytes == k16) return launch_kernel(a2a_kernel<P, true, STAGE, k16>, grid, dim3(kThreads), s, a);
  return launch_kernel(a2a_kernel<P, true, STAGE, kBig>, grid, dim3(kThreads), s, a);
}

template <class P>
cudaError_t launch_params(const P& a, bool shift, bool stage, cudaStream_t s) {
  const uint64_t tiles = a.tile0[a.ndest];
  if (tiles == 0) return cudaSuccess;
  const uint64_t g = tiles < (1ull << 31) - 1 ? tiles : (1ull << 31) - 1;
  const dim3 grid(static_cast<unsigned>(g));
  return stage ? launch_staged<P, true>(a, shift, grid, s) : launch_staged<P, false>(a, shift, grid, s);
}

}  // namespace

uint64_t a2a_tiles_for(const char* dst, uint64_t bytes, uint64_t tile_bytes) {
  if (bytes == 0) return 0;
  const uint64_t lead = reinterpret_cast<uintptr_t>(dst) & 511;  // tiles start on 512-byte boundaries
  return (lead + bytes + tile_bytes - 1) / tile_bytes;
}

cudaError_t launch_a2a(const A2ASmall& a, bool shift, bool stage, cudaStream_t s) {
  cudaError_t err = launch_params(a, shift, stage, s);
  if (err == cudaSuccess && a.tile0[a.ndest] != 0) note_launch();
  return err;
}
cudaError_t launch_a2a(const A2APlain& a, bool shift, bool stage, cudaStream_t s) {
  cudaError_t err = launch_params(a, shift, stage, s);
  if (err == cudaSuccess && a.tile0[a.ndest] != 0) note_launch();
  return err;
}
cudaError_t launch_a2a(const A2ATable32& a, bool shift, bool stage, cudaStream_t s) {
  cudaError_t err = launch_params(a, shift, stage, s);
  if (err == cudaSuccess && a.tile0[a.ndest] != 0) note_launch();
  return err;
}
cudaError_t launch_a2a(const A2ATable64& a, bool shift, bool stage, cudaStream_t s) {
  cudaError_t err = launch_params(a, shift, stage, s);
  if (err == cudaSuccess && a.tile0[a.ndest] != 0) note_launch();
  return err;
}

}  // namespace ccl
