// ccl_internal.h -- parameter blocks and kernel launchers behind the C ABI.
//
// Every kernel receives its rank pointers by value in a __grid_constant__
// parameter block (at most 4 KB), so a call needs no device memory of its own.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ccl.h"

namespace ccl {

// ------------------------------------------------ fused fold (AR / RS / bucket)
enum FoldMode : int {
  kModeAllReduce = 0,      // fold, write the result to every rank's buffer
  kModeReduceScatter = 1,  // fold, write chunk c only to rank c's shard
  kModeBucket = 2,         // fold fp32, scale, round to bf16, write to every rank
  kModeReduce = 3          // fold, write the result only to recv[0] (the root's buffer)
};

// pf_ctas (set by launch_kernel): CTAs of the launch's first wave, the ones
// that prefetch their first inputs into L2 before waiting on the previous
// grid (0: none); fold_small_kernel compares its grid with it.
struct FoldArgs {
  const void* send[CCL_MAX_RANKS];
  void* recv[CCL_MAX_RANKS];
  uint64_t q;    // floor(n / p)
  uint64_t rem;  // n mod p
  int p;
  float scale;   // bucket mode only
  uint32_t pf_ctas;
};

// `vec`: every pointer is 16-byte aligned, so 16-byte vectors may be used.
cudaError_t launch_fold(int mode, int dt, int op, bool vec, const FoldArgs& a, cudaStream_t s);

// The fold kernel a call takes: fold_unrolled_kernel with `batch` ranks'
// loads issued together and `vectors` vectors per thread, or fold_kernel
// when batch == 0.  dt_in / dt_out: element types (kF32 -> kBF16 is the
// bucket); mode: the call kind (kMode*); q = floor(n / p); sms = the
// device's SM count.
struct FoldPlan {
  int batch, vectors;
};
FoldPlan fold_plan(int dt_in, int dt_out, int op, int mode, int p, uint64_t q, bool vec, int sms);

// Fold in another schedule's order (schedule_fold.cu): `linear` = the naive
// root's rank-order fold; otherwise the pairwise tree over ranks in identity
// or (`reversed`) bit-reversed order.
// bf16 ring with bf16 partials (rounded at every hop); mode AR or RS.
cudaError_t launch_wire_fold(int mode, bool vec, const FoldArgs& a, cudaStream_t s);
// Two-level ring fold; f.q / f.rem = floor(n / a), n mod a (the level-1 split).
cudaError_t launch_hier_fold(int dt, bool vec, const FoldArgs& f, int a, cudaStream_t s);
cudaError_t launch_schedule_fold(int dt, bool linear, bool reversed, bool vec, const FoldArgs& a,
                                 uint64_t n, cudaStream_t s);

// ---------------------------------------------------------------- all-gather
struct GatherArgs {
  const void* send[CCL_MAX_RANKS];  // rank k's block (len(k) elements)
  void* recv[CCL_MAX_RANKS];        // full n-element outputs
  uint64_t q, rem;
  int p;
  uint32_t pf_ctas;                 // as in FoldArgs
};
cudaError_t launch_gather(int dt, bool vec, const GatherArgs& a, cudaStream_t s);
// Fan-out through bulk copies: chunk c (chunk_bytes from send[c], or from
// send[0] when nchunks == 1) goes to byte offset c * chunk_bytes of every
// recv[r].  All-gather: nchunks = p; broadcast: nchunks = 1.
struct FanoutArgs {
  const void* send[CCL_MAX_RANKS];
  void* recv[CCL_MAX_RANKS];
  uint64_t chunk_bytes, nchunks, tiles_per_chunk;
  int p;
};
bool fanout_supported(const FanoutArgs& a);  // alignment rules of the bulk copies
cudaError_t launch_fanout(FanoutArgs a, cudaStream_t s);
// The device error word set by a bounded wait that ran out (0 if none).
cudaError_t read_device_error(unsigned int* flag, bool clear);
// One-thread kernel whose mbarrier wait runs out by construction (self-test).
cudaError_t launch_bounded_wait_probe(cudaStream_t s);
// Broadcast: send[0] (n elements) copied to recv[0..p-1]; `vec`: all 16-byte aligned.
cudaError_t launch_broadcast(int dt, bool vec, const GatherArgs& a, uint64_t n, cudaStream_t s);

// ------------------------------------------------------------- all-to-allv
// Destination j's buffer holds one block per source i in source order; work
// is cut into tiles of tile_bytes of destination space (4, 8, 16 or 32 KB
// by the launch's bytes per SM; boundaries on 512 bytes of the
// destination's address), tile0[c] = first tile of destination j0 + c in
// this launch, tile0[ndest] = the launch's tiles.
//  plain = 1: the all-to-all of the chunk rule, one element per row:
//    block i of destination j has len(j) rows and starts at row off(j) of
//    send[i] (n = q * p + rem elements per rank).
//  plain = 0: table[i * (ndest + 1) + c] = rows of send[i] before its block
//    for destination j0 + c (c = 0..ndest; c = ndest gives the next
//    destination's start, or source i's total rows when j0 + ndest = p).
constexpr uint64_t kA2ATileBytes = 32768;
constexpr uint64_t kA2ASmallTileBytes = 4096;
constexpr uint64_t kA2AMidTileBytes[2] = {8192, 16384};
// Calls with a block edge off the 16-byte grid take the small-block stage
// while their blocks average at most this many bytes (larger blocks leave a
// tile one edge or none, which the element path handles at less cost).
constexpr uint64_t kA2AStageMaxBlockBytes = 8192;
template <int CAP, int TCAP, typename TT>
struct A2AParamsT {
  static constexpr int kCap = CAP;
  static constexpr int kTableCap = TCAP;
  using Entry = TT;
  const char* send[CAP];
  char* recv[CAP];
  uint64_t tile0[CAP + 1];
  uint64_t row_bytes;  // bytes per row (a multiple of elem)
  uint64_t q, rem;     // plain: the chunk rule of n
  int p, j0, ndest, plain;
  int elem;            // element bytes (2 or 4)
  uint32_t tile_bytes; // 4096, 8192, 16384 or 32768
  TT table[TCAP];
};
// p <= 16, any geometry (a table of 16 x 17 entries): under the classic 4 KB
using A2ASmall = A2AParamsT<16, 16 * 17, uint32_t>;
// plain all-to-all, any p
using A2APlain = A2AParamsT<128, 1, uint32_t>;
// tables in the 32 KB parameter space of CUDA 12.1+ drivers: p * (ndest + 1)
// entries per launch (uint32 while every row prefix fits in 32 bits)
using A2ATable32 = A2AParamsT<128, 7408, uint32_t>;
using A2ATable64 = A2AParamsT<128, 3704, uint64_t>;
static_assert(sizeof(A2ASmall) <= 4096, "all-to-allv parameters exceed 4 KB");
static_assert(sizeof(A2APlain) <= 4096, "all-to-all parameters exceed 4 KB");
static_assert(sizeof(A2ATable32) <= 32764, "all-to-allv parameters exceed 32,764 bytes");
static_assert(sizeof(A2ATable64) <= 32764, "all-to-allv parameters exceed 32,764 bytes");
uint64_t a2a_tiles_for(const char* dst, uint64_t bytes, uint64_t tile_bytes);
// shift: some block's source and destination differ in 16-byte phase;
// stage: the units that straddle blocks go through the small-block stage
cudaError_t launch_a2a(const A2ASmall& a, bool shift, bool stage, cudaStream_t s);
cudaError_t launch_a2a(const A2APlain& a, bool shift, bool stage, cudaStream_t s);
cudaError_t launch_a2a(const A2ATable32& a, bool shift, bool stage, cudaStream_t s);
cudaError_t launch_a2a(const A2ATable64& a, bool shift, bool stage, cudaStream_t s);

// ------------------------------------------------- literal ring engine steps
// One launch moves p independent transfers, transfer r: src[r] -> dst[r],
// len[r] elements.  Kinds:
enum XferKind : int {
  kXferCopy = 0,     // dst = src (element type dt)
  kXferCombine = 1,  // dst = combine(src, dst): received partial (+) own value
  kXferWiden = 2,    // bf16 src -> fp32 dst (exact)
  kXferNarrow = 3    // fp32 src -> bf16 dst (round to nearest even)
};
struct XferArgs {
  const char* src[CCL_MAX_RANKS];
  char* dst[CCL_MAX_RANKS];
  uint64_t len[CCL_MAX_RANKS];
  int p;
};
cudaError_t launch_xfer(int kind, int dt, int op, const XferArgs& a, cudaStream_t s);

// Reason text for ccl_last_error() (per calling thread), for entry points
// that live outside ccl_api.cu.
void clear_last_error();
ccl_status_t report_error(ccl_status_t st, const char* fmt, ...);

// ------------------------------------------------- Ulysses head <-> sequence
struct UlyssesArgs {
  const void* x[CCL_MAX_RANKS];  // inputs (sequence shards, or head groups when inverse)
  void* y[CCL_MAX_RANKS];        // outputs
  uint64_t seq_per_rank, heads, head_dim, segments;  // segments = p * p * seq_per_rank
  int p, inverse;
};
cudaError_t launch_ulysses(int dt, bool vec, const UlyssesArgs& a, cudaStream_t s);

// ------------------------------------------------------------------- MoE
constexpr int kMoeMaxRanks = 64;  // keeps every MoE parameter block under 4 KB
constexpr int kMoeMaxK = 16;
struct MoeRouteArgs {
  const int32_t* ids[kMoeMaxRanks];  // tokens * k expert ids per source
  int32_t* slots[kMoeMaxRanks];      // out: slot of each (token, choice), -1 if unrouted
  int64_t* counts;                   // out: p x p rows source -> destination (device)
  uint64_t items;                    // tokens * k
  int p, epr, num_experts;
};
struct MoeDispatchArgs {
  const void* x[kMoeMaxRanks];        // tokens x hidden bf16 per source
  const int32_t* ids[kMoeMaxRanks];
  const int32_t* slots[kMoeMaxRanks];
  void* recv[kMoeMaxRanks];           // rows x hidden, bf16 or e4m3
  float* scales[kMoeMaxRanks];        // FP8: rows x hidden/128 block scales
  int32_t* rexp[kMoeMaxRanks];        // optional: expert id of each received row
  const int64_t* counts;              // device p x p
  uint64_t cap[kMoeMaxRanks];         // rows each recv[d] holds
  uint64_t tokens, hidden;
  int p, k, epr, num_experts, rexp_given;
  int tpc;                            // tokens per CTA (set by the launcher)
};
struct MoeCombineArgs {
  const void* y[kMoeMaxRanks];        // rows x hidden bf16, dispatch layout
  const int32_t* ids[kMoeMaxRanks];
  const int32_t* slots[kMoeMaxRanks];
  const float* weights[kMoeMaxRanks]; // tokens * k gate weights per source
  void* out[kMoeMaxRanks];            // tokens x hidden bf16 per source
  const int64_t* counts;
  uint64_t cap[kMoeMaxRanks];         // rows each y[d] holds
  uint64_t tokens, hidden;
  int p, k, epr, num_experts;
  int tpc;                            // tokens per CTA (set by the launcher)
};
static_assert(sizeof(MoeDispatchArgs) <= 4096, "MoE dispatch parameters exceed 4 KB");
static_assert(sizeof(MoeCombineArgs) <= 4096, "MoE combine parameters exceed 4 KB");
cudaError_t launch_moe_route(const MoeRouteArgs& a, cudaStream_t s);
cudaError_t launch_moe_dispatch(const MoeDispatchArgs& a, bool fp8, cudaStream_t s);
cudaError_t launch_moe_combine(const MoeCombineArgs& a, cudaStream_t s);

// Records one successful kernel launch (ccl_kernel_launch_count).
void note_launch();

// Streaming multiprocessors of the current device (0 if unknown).
int current_sm_count();

// CTAs of `kernel` (kThreads threads each) resident on the current device at
// once -- a launch's first wave -- cached per host thread, kernel and device
// (0 if unknown).
int first_wave_ctas(const void* kernel);

}  // namespace ccl
