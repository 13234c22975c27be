// bulk_fanout.cu -- all-gather and broadcast through the Tensor Memory
// Accelerator's bulk copies: one read of every source byte into shared
// memory, p bulk stores of it.
//
// All-gather ("Networks and Collective Communication" section 4.1: each
// device contributes one block and everyone gets the concatenation) and
// broadcast are one read and p writes per byte.  With thread stores every
// load feeds p 16-byte store instructions, and at p = 16 the store queue,
// not HBM, paces the warps.  Here a single thread per CTA drives the copy
// engine: it brings a tile of the source (64 KB) into shared memory with
// cp.async.bulk (completion counted on an mbarrier) and sends it to the p
// outputs with p cp.async.bulk stores, no SM load/store instruction touching
// the data.  Stages let the next tiles' loads run while a tile is stored.
// It is an alternative path (see use_fanout in ccl_api.cu), not the default:
// on GB300 the thread-store kernels of gather.cu are faster for these copies.
//
// Requirements (checked on the host): every pointer and every chunk's byte
// offset and length are multiples of 16 bytes -- the bulk copies' rule -- and
// all chunks have the same length (p divides n for the all-gather).  Waits
// are bounded: a wait that runs out sets a device error word (read with
// ccl_device_error_flag, or turned into CCL_ERR_TIMEOUT by ccl_stream_check),
// waits once more with a bound for the copies still in flight, and the CTA
// returns.
#include "device_common.cuh"

namespace ccl {

__device__ unsigned int g_device_error;  // nonzero: a bounded wait ran out

namespace {

// Pipeline shape (stages x tile bytes x CTAs per SM must fit the SM's 227 KB).
// Measured on GB300 (all-gather p=16 x 192 MiB bf16; broadcast p=16 x 64 MiB):
// 2 x 64 KB x 1 CTA 0.95 / 0.94 of the copy bandwidth, 3 x 64 KB 0.94 / 0.97,
// 4 x 16 KB x 3 0.91 / 0.93, 4 x 4 KB x 12 0.86 / 0.86 -- larger tiles win.
#ifndef CCL_FANOUT_STAGES
#define CCL_FANOUT_STAGES 2
#endif
#ifndef CCL_FANOUT_TILE
#define CCL_FANOUT_TILE 65536
#endif
#ifndef CCL_FANOUT_CTAS
#define CCL_FANOUT_CTAS 1
#endif
constexpr int kStages = CCL_FANOUT_STAGES;
constexpr uint32_t kTileBytes = CCL_FANOUT_TILE;
constexpr int kFanoutCtasPerSm = CCL_FANOUT_CTAS;
static_assert(kStages * kTileBytes * kFanoutCtasPerSm <= 227 * 1024, "fan-out stages exceed shared memory");
constexpr long long kWaitLimit = 1ll << 20;  // try_wait calls before giving up (well under a second)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// true once the barrier's phase `parity` has completed; false after `limit`
// tries
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit = kWaitLimit) {
  for (long long i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void bulk_load(uint32_t dst_smem, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst_smem),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src_smem), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// wait until at most N committed store groups are still reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Tiles are numbered over the chunks: chunk c holds tiles c*tpc .. c*tpc+tpc-1.
struct Tile {
  const char* src;
  uint64_t dst_off;  // byte offset in every output
  uint32_t bytes;
};

__device__ __forceinline__ Tile tile_at(const FanoutArgs& a, uint64_t t) {
  const uint64_t c = t / a.tiles_per_chunk;
  const uint64_t off = (t - c * a.tiles_per_chunk) * kTileBytes;
  const uint64_t left = a.chunk_bytes - off;
  Tile x;
  x.src = static_cast<const char*>(a.send[a.nchunks == 1 ? 0 : c]) + off;
  x.dst_off = c * a.chunk_bytes + off;
  x.bytes = static_cast<uint32_t>(left < kTileBytes ? left : kTileBytes);
  return x;
}

__global__ void __launch_bounds__(32) fanout_kernel(const __grid_constant__ FanoutArgs a) {
  extern __shared__ __align__(128) char stage[];  // kStages x kTileBytes
  __shared__ __align__(8) uint64_t full[kStages];
  pdl_enter();
  if (threadIdx.x != 0) return;  // one thread drives the copy engine
  const uint64_t ntiles = a.tiles_per_chunk * a.nchunks;
  const uint64_t first = blockIdx.x, step = gridDim.x;
  if (first >= ntiles) return;
  for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&full[s]), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");

  // this CTA's i-th tile is first + i * step; stage i % kStages
  const uint64_t mine = (ntiles - first + step - 1) / step;
  auto issue_load = [&](uint64_t i) {
    const int s = static_cast<int>(i % kStages);
    const Tile x = tile_at(a, first + i * step);
    const uint32_t bar = smem_addr(&full[s]);
    mbar_expect_tx(bar, x.bytes);
    bulk_load(smem_addr(stage + s * kTileBytes), x.src, x.bytes, bar);
  };
  const uint64_t prologue = mine < kStages ? mine : kStages;
  for (uint64_t i = 0; i < prologue; ++i) issue_load(i);

  uint64_t done_loads = prologue;  // loads issued
  uint64_t failed_at = mine;        // first tile whose load did not arrive in time
  for (uint64_t i = 0; i < mine; ++i) {
    const int s = static_cast<int>(i % kStages);
    if (!mbar_wait(smem_addr(&full[s]), static_cast<uint32_t>((i / kStages) & 1))) {
      failed_at = i;
      break;
    }
    const Tile x = tile_at(a, first + i * step);
    const uint32_t src = smem_addr(stage + s * kTileBytes);
    for (int r = 0; r < a.p; ++r) bulk_store(static_cast<char*>(a.recv[r]) + x.dst_off, src, x.bytes);
    bulk_commit();
    // refill the stage of tile i-1 once its stores have read it
    if (i >= 1 && done_loads < mine) {
      bulk_wait_read<1>();
      issue_load(done_loads);
      ++done_loads;
    }
  }
  if (failed_at < mine) {
    atomicExch(&g_device_error, 1u);
    // let the loads still in flight land (again with a bound) before the
    // shared memory goes away
    for (uint64_t i = failed_at; i < done_loads; ++i) {
      const int s = static_cast<int>(i % kStages);
      mbar_wait(smem_addr(&full[s]), static_cast<uint32_t>((i / kStages) & 1));
    }
  }
  bulk_wait_all();
}

// Self-test of the bounded-wait path: one thread waits on an mbarrier that no
// arrival or copy will ever complete, gives up after `limit` tries, records
// the error word as the fan-out does, and returns.  Nothing is in flight.
__global__ void __launch_bounds__(32) bounded_wait_probe_kernel(long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_addr(&bar), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (!mbar_wait(smem_addr(&bar), 0, limit)) atomicExch(&g_device_error, 2u);
}

}  // namespace

cudaError_t launch_bounded_wait_probe(cudaStream_t s) {
  bounded_wait_probe_kernel<<<1, 32, 0, s>>>(1ll << 14);
  cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) note_launch();
  return err;
}

bool fanout_supported(const FanoutArgs& a) {
  if (a.chunk_bytes == 0 || a.chunk_bytes % 16 != 0) return false;
  for (int r = 0; r < a.p; ++r)
    if (reinterpret_cast<uintptr_t>(a.recv[r]) % 16 != 0) return false;
  for (uint64_t c = 0; c < (a.nchunks == 1 ? 1 : a.nchunks); ++c)
    if (reinterpret_cast<uintptr_t>(a.send[c]) % 16 != 0) return false;
  return true;
}

cudaError_t launch_fanout(FanoutArgs a, cudaStream_t s) {
  a.tiles_per_chunk = (a.chunk_bytes + kTileBytes - 1) / kTileBytes;
  const uint64_t ntiles = a.tiles_per_chunk * a.nchunks;
  const int sms = current_sm_count();
  uint64_t g = static_cast<uint64_t>(sms > 0 ? sms : 1) * kFanoutCtasPerSm;
  if (g > ntiles) g = ntiles;
  if (g < 1) g = 1;
  const size_t smem = static_cast<size_t>(kStages) * kTileBytes;
  cudaError_t err = cudaFuncSetAttribute(fanout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(g));
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = CCL_PDL ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, fanout_kernel, a);
  if (err == cudaSuccess) note_launch();
  return err;
}

cudaError_t read_device_error(unsigned int* flag, bool clear) {
  cudaError_t err = cudaMemcpyFromSymbol(flag, g_device_error, sizeof(unsigned int));
  if (err == cudaSuccess && clear) {
    const unsigned int zero = 0;
    err = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
  }
  return err;
}

}  // namespace ccl
