// device_common.cuh -- element types, streaming memory access and the fold
// operator shared by the ring-ordered collective kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>
#include <utility>

#include "ccl_internal.h"

namespace ccl {

constexpr int kThreads = 256;  // threads per CTA for every streaming kernel

// ------------------------------------------------------------ element types
// Element type tags.  Acc is the register type partial sums travel in: fp32
// for fp32 and bf16 data, int32 for int32 data.
enum Dt : int { kF32 = CCL_F32, kBF16 = CCL_BF16, kI32 = CCL_I32 };

template <int DT> struct Elem;
template <> struct Elem<kF32> { using Acc = float; static constexpr int kBytes = 4; };
template <> struct Elem<kBF16> { using Acc = float; static constexpr int kBytes = 2; };
template <> struct Elem<kI32> { using Acc = int32_t; static constexpr int kBytes = 4; };

// ------------------------------------------------------- global memory access
// Every input element is read exactly once, so loads bypass L1 and use the
// read-only path; outputs are written once and never re-read, so stores are
// marked streaming (evict-first).
__device__ __forceinline__ uint4 ld_once16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}
// 16-byte read-only load that allocates in L1 (for data a thread reads as two
// halves of one sector).
__device__ __forceinline__ uint4 ld_l1_16(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_once4(const void* p) {
  uint32_t v;
  asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_once2(const void* p) {
  unsigned short v;
  asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_stream4(void* p, uint32_t v) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_stream2(void* p, uint32_t v) {
  unsigned short h = static_cast<unsigned short>(v);
  asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(p), "h"(h) : "memory");
}

// Load VEC consecutive elements starting at element `i` of `base` as raw
// 32-bit words (VEC * bytes / 4 words; a lone bf16 occupies the low half).
// VEC > 1 requires a 16-byte aligned address and VEC * bytes % 16 == 0.
template <int DT, int VEC>
__device__ __forceinline__ void load_raw(const void* base, uint64_t i, uint32_t* w) {
  constexpr int B = Elem<DT>::kBytes;
  const char* p = static_cast<const char*>(base) + i * B;
  if constexpr (VEC * B == 32) {
    // Two 16-byte halves of one 32-byte sector per thread: a warp's first
    // load touches every other 16 bytes of 32 sectors, so both loads allocate
    // in L1 and the second is served there.  In HBM the second would hit L2
    // anyway; from pinned host memory (zero-copy) it saves a second trip over
    // the host link, which doubles the kernel's host-memory throughput.
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      uint4 v = ld_l1_16(p + 16 * k);
      w[4 * k + 0] = v.x;
      w[4 * k + 1] = v.y;
      w[4 * k + 2] = v.z;
      w[4 * k + 3] = v.w;
    }
  } else if constexpr (VEC * B >= 16) {
#pragma unroll
    for (int k = 0; k < VEC * B / 16; ++k) {
      uint4 v = ld_once16(p + 16 * k);
      w[4 * k + 0] = v.x;
      w[4 * k + 1] = v.y;
      w[4 * k + 2] = v.z;
      w[4 * k + 3] = v.w;
    }
  } else {
    static_assert(VEC == 1, "sub-16-byte loads are element-wise");
    w[0] = (B == 4) ? ld_once4(p) : ld_once2(p);
  }
}

// Element e of a raw word array, widened exactly to the accumulator type.
template <int DT>
__device__ __forceinline__ typename Elem<DT>::Acc widen(const uint32_t* w, int e) {
  if constexpr (DT == kF32) {
    return __uint_as_float(w[e]);
  } else if constexpr (DT == kI32) {
    return static_cast<int32_t>(w[e]);
  } else {
    // bf16 is the top half of a binary32: append 16 zero bits.
    const uint32_t word = w[e >> 1];
    return __uint_as_float((e & 1) ? (word & 0xFFFF0000u) : (word << 16));
  }
}

// ---------------------------------------------------------------- the fold
// What a receiving rank computes from the partial it got (`acc`) and its own
// value (`x`).  SUM: IEEE fp32 add (round to nearest even) or wrapping int32
// add.  MAX / MIN: keep `x` only when strictly greater / smaller.
template <int OP, typename T>
__device__ __forceinline__ T combine(T acc, T x) {
  if constexpr (OP == CCL_SUM) {
    if constexpr (std::is_floating_point<T>::value) {
      return __fadd_rn(acc, x);
    } else {
      return static_cast<T>(static_cast<uint32_t>(acc) + static_cast<uint32_t>(x));
    }
  } else if constexpr (OP == CCL_MAX) {
    return (x > acc) ? x : acc;
  } else {
    return (x < acc) ? x : acc;
  }
}

// Pack accumulator values into output raw words (VEC * out_bytes / 4 words).
// bf16 output rounds each fp32 value to nearest even.
template <int DT_OUT, int VEC, typename Acc>
__device__ __forceinline__ void pack_out(const Acc* acc, uint32_t* w) {
  if constexpr (DT_OUT == kF32) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) w[e] = __float_as_uint(acc[e]);
  } else if constexpr (DT_OUT == kI32) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) w[e] = static_cast<uint32_t>(acc[e]);
  } else {
    if constexpr (VEC == 1) {
      w[0] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[0]));
    } else {
#pragma unroll
      for (int e = 0; e < VEC; e += 2) {
        __nv_bfloat162 h = __floats2bfloat162_rn(acc[e], acc[e + 1]);
        w[e >> 1] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
  }
}

// Store VEC elements (raw words) at element `i` of `base`.
template <int DT_OUT, int VEC>
__device__ __forceinline__ void store_raw(void* base, uint64_t i, const uint32_t* w) {
  constexpr int B = Elem<DT_OUT>::kBytes;
  char* p = static_cast<char*>(base) + i * B;
  if constexpr (VEC * B >= 16) {
#pragma unroll
    for (int k = 0; k < VEC * B / 16; ++k)
      st_stream16(p + 16 * k, make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]));
  } else {
    static_assert(VEC == 1, "sub-16-byte stores are element-wise");
    if constexpr (B == 4) st_stream4(p, w[0]); else st_stream2(p, w[0]);
  }
}

// Store element e of a raw word array (element-wise edge path).
template <int DT_OUT>
__device__ __forceinline__ void store_one(void* base, uint64_t i, const uint32_t* w, int e) {
  constexpr int B = Elem<DT_OUT>::kBytes;
  char* p = static_cast<char*>(base) + i * B;
  if constexpr (B == 4) {
    st_stream4(p, w[e]);
  } else {
    st_stream2(p, (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu));
  }
}

// ------------------------------------------------------- early L2 prefetch
// A kernel may prefetch its first inputs into L2 before pdl_enter(): while
// the previous grid in the stream drains, the lines are already on their way,
// which hides the first loads' DRAM latency of back-to-back calls.  This is
// only a hint: a prefetch returns no data, and L2 is the device's point of
// coherence, so a line the previous grid writes afterwards is updated in L2
// and the loads after pdl_enter() see the written value (they bypass or miss
// L1, which the prefetch does not fill).  Prefetched lines hold at least one
// byte of a buffer the kernel reads, so they lie in mapped pages.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// The byte spans [base[r] + off, base[r] + off + len), r < nspans, prefetched
// into L2 by the CTA's threads together, one prefetch per 128-byte line, at
// most kPrefetchCtaBytes in all (the spans cut short evenly).
constexpr uint64_t kPrefetchCtaBytes = 65536;
__device__ __forceinline__ void prefetch_spans_l2(const void* const* base, int nspans, uint64_t off,
                                                  uint64_t len) {
  if (len == 0) return;
  {
    const uint64_t cap = kPrefetchCtaBytes / static_cast<uint64_t>(nspans);
    len = len < cap ? len : (cap > 128 ? cap : 128);
  }
  const uint64_t lines = (len + 127) / 128 + 1;  // lines a span of len bytes can touch
  const uint64_t total = lines * static_cast<uint64_t>(nspans);
  for (uint64_t k = threadIdx.x; k < total; k += blockDim.x) {
    const uint64_t r = k / lines, l = k - r * lines;
    const uintptr_t first = reinterpret_cast<uintptr_t>(base[r]) + off;
    const uintptr_t line = (first & ~static_cast<uintptr_t>(127)) + 128 * l;
    if (line < first + len) prefetch_l2(reinterpret_cast<const void*>(line));
  }
}

// ------------------------------------------- programmatic dependent launch
// Kernels are launched with programmatic stream serialisation, so a kernel
// may be scheduled while the previous kernel in the stream is still draining.
// pdl_enter() must run before the kernel touches global memory: it waits
// until every earlier grid in the stream has completed and its writes are
// visible, then lets the next grid be scheduled.  When the previous work is
// not a programmatic launch both instructions cost nothing.
#ifndef CCL_PDL
#define CCL_PDL 1
#endif
__device__ __forceinline__ void pdl_enter() {
#if CCL_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

template <typename T, typename = void>
struct HasPfCtas : std::false_type {};
template <typename T>
struct HasPfCtas<T, std::void_t<decltype(std::declval<T&>().pf_ctas)>> : std::true_type {};

// The CTA's place in launch order (x fastest, then y).
__device__ __forceinline__ uint64_t cta_rank() {
  return static_cast<uint64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
}

template <typename Args>
cudaError_t launch_kernel(void (*kernel)(Args), dim3 grid, dim3 block, cudaStream_t s,
                          const Args& args_in) {
  // arguments with a pf_ctas field get the kernel's first wave there
  Args args = args_in;
  if constexpr (HasPfCtas<Args>::value)
    args.pf_ctas = static_cast<uint32_t>(first_wave_ctas(reinterpret_cast<const void*>(kernel)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = CCL_PDL ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

// ------------------------------------------------------------- chunk rule
// Chunk c of an n-element buffer split p ways: the first n mod p chunks hold
// one extra element (numpy's array_split).
struct Chunk {
  uint64_t off, len;
};
__device__ __forceinline__ Chunk chunk_of(int c, uint64_t q, uint64_t rem) {
  const uint64_t uc = static_cast<uint64_t>(c);
  return Chunk{uc * q + (uc < rem ? uc : rem), q + (uc < rem ? 1u : 0u)};
}

}  // namespace ccl
