// cpu_ranks.cpp -- the literal ring run by CPU "ranks".  TEST INFRASTRUCTURE
// ONLY: called by tests/ and by the CPU baseline of bench.py through the
// ctypes shim oracle/cpu_ranks.py, never by the library, and sharing no code
// with it.
//
// The same schedule as oracle/ring.py ("Networks and Collective
// Communication" section 5.1 and Exercise 2; "dist_train", Ring Algorithm;
// "LLM Distributed Training Collectives", Ring AllReduce), but executed the way
// the pages' devices execute it: every virtual rank is driven by a host
// thread (one std::thread per rank, at most `max_threads`, ranks dealt
// round-robin to the threads), each rank keeps its own working buffer and an
// inbox, and the ranks move in lock step -- in every step each rank writes its
// one message into the next rank's inbox, all ranks meet at a barrier, each
// rank combines what it received with its own chunk, and all meet again.
//
//   reduce-scatter step s = 0..p-2: rank r sends its partial of chunk
//     (r - s - 1) mod p to rank r + 1, which adds its own chunk to it (fp32
//     partials for f32 and bf16, int32 with wraparound for i32; MAX / MIN keep
//     the receiver's value only when strictly greater / smaller);
//   all-gather step s = 0..p-2: rank r sends chunk (r - s) mod p;
//   chunk c = the numpy array_split rule (the first n mod p chunks one longer);
//   bf16: the owner rounds its finished chunk to bf16 once (nearest-even, by
//   the published bit method) and the all-gather moves bf16.
//
// Waits are bounded.  A barrier that is not complete within `timeout_s`
// aborts the collective with O3_TIMEOUT; a rank whose inbox does not hold the
// message of the current step aborts it with O3_LOST_MESSAGE.  Host-side
// fault injection drives both: a rank that stalls (stops taking part from a
// given step) or a rank that skips one send.
#include <chrono>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <thread>
#include <type_traits>
#include <vector>

namespace {

enum Status { kOk = 0, kInvalid = 1, kTimeout = 4, kLostMessage = 5 };
enum Dtype { kF32 = 0, kBF16 = 1, kI32 = 2 };
enum Op { kSum = 0, kMax = 1, kMin = 2 };
enum Kind { kAllReduce = 0, kReduceScatter = 1, kAllGather = 2, kBucket = 3 };
enum Fault { kNoFault = 0, kStall = 1, kSkipSend = 2 };

float bf16_to_f32(uint16_t b) {
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// nearest-even: add 0x7FFF plus the lowest kept bit, drop the low 16 bits; a
// NaN keeps its top bits with the quiet bit set
uint16_t f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if (f != f) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  const uint32_t lsb = (u >> 16) & 1u;
  return static_cast<uint16_t>((u + 0x7FFFu + lsb) >> 16);
}

struct Chunk {
  uint64_t off, len;
};

Chunk chunk(int p, uint64_t n, int c) {
  const uint64_t q = n / static_cast<uint64_t>(p), rem = n % static_cast<uint64_t>(p);
  const uint64_t uc = static_cast<uint64_t>(c);
  return {uc * q + (uc < rem ? uc : rem), q + (uc < rem ? 1 : 0)};
}

// A barrier whose waits end after a deadline or when the collective aborts.
class Barrier {
 public:
  Barrier(int parties, double timeout_s) : parties_(parties), timeout_(timeout_s) {}

  // true when every party arrived; false when the collective was aborted
  // (by this wait timing out or by another thread)
  bool wait() {
    std::unique_lock<std::mutex> lk(m_);
    if (status_ != kOk) return false;
    const uint64_t gen = gen_;
    if (++arrived_ == parties_) {
      arrived_ = 0;
      ++gen_;
      cv_.notify_all();
      return true;
    }
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::duration<double>(timeout_);
    while (gen_ == gen && status_ == kOk) {
      if (cv_.wait_until(lk, deadline) == std::cv_status::timeout && gen_ == gen && status_ == kOk) {
        status_ = kTimeout;
        cv_.notify_all();
      }
    }
    return gen_ != gen && status_ == kOk;
  }

  void abort(int st) {
    std::lock_guard<std::mutex> lk(m_);
    if (status_ == kOk) status_ = st;
    cv_.notify_all();
  }

  // a stalled rank waits here (bounded) until the others have given up
  void wait_for_abort() {
    std::unique_lock<std::mutex> lk(m_);
    cv_.wait_for(lk, std::chrono::duration<double>(2.0 * timeout_ + 1.0), [&] { return status_ != kOk; });
  }

  int status() {
    std::lock_guard<std::mutex> lk(m_);
    return status_;
  }

 private:
  std::mutex m_;
  std::condition_variable cv_;
  const int parties_;
  const double timeout_;
  int arrived_ = 0;
  uint64_t gen_ = 0;
  int status_ = kOk;
};

// Acc: the partial's type (float for f32 / bf16, int32_t for i32); Out: the
// element type the all-gather moves (float, uint16_t bf16 bits, int32_t).
template <typename Acc, typename Out>
struct Ring {
  int kind, p, dtype, op;
  uint64_t n;
  float scale;
  const void* const* send;
  void* const* recv;
  int fault, fault_rank, fault_step;
  std::vector<std::vector<Acc>> work;    // reduce-scatter working buffers
  std::vector<std::vector<Acc>> inbox;   // one reduce-scatter message per rank
  std::vector<std::vector<Out>> full;    // all-gather buffers
  std::vector<std::vector<Out>> inbox2;  // one all-gather message per rank
  std::vector<int64_t> tag;              // step whose message an inbox holds
  std::vector<uint64_t> sent;
  Barrier* bar;

  Acc widen(const void* base, uint64_t i) const {
    if (dtype == kBF16) return static_cast<Acc>(bf16_to_f32(static_cast<const uint16_t*>(base)[i]));
    Acc v;
    std::memcpy(&v, static_cast<const char*>(base) + i * sizeof(Acc), sizeof(Acc));
    return v;
  }

  Acc combine(Acc received, Acc own) const {
    if (op == kMax) return own > received ? own : received;
    if (op == kMin) return own < received ? own : received;
    if constexpr (std::is_integral<Acc>::value) {  // int32: two's-complement wraparound
      return static_cast<Acc>(static_cast<uint32_t>(received) + static_cast<uint32_t>(own));
    } else {
      return received + own;
    }
  }

  Out finish(Acc v) const {
    if constexpr (sizeof(Out) == 2) {
      return f32_to_bf16(static_cast<float>(v));
    } else {
      return static_cast<Out>(v);
    }
  }

  bool stalls(int r, int step) const { return fault == kStall && r == fault_rank && step == fault_step; }

  // Run the ranks of thread t (r = t, t + T, ...).  Steps are numbered over
  // both phases: 0 .. p-2 reduce-scatter, p-1 .. 2p-3 all-gather.
  void run(int t, int T) {
    const bool do_rs = kind != kAllGather, do_ag = kind != kReduceScatter;
    for (int r = t; r < p; r += T) {
      if (do_rs) {
        work[r].resize(n);
        for (uint64_t i = 0; i < n; ++i) work[r][i] = widen(send[r], i);
      }
    }
    if (!bar->wait()) return;
    if (do_rs) {
      for (int s = 0; s < p - 1; ++s) {
        for (int r = t; r < p; r += T) {
          if (stalls(r, s)) {
            bar->wait_for_abort();
            return;
          }
          if (fault == kSkipSend && r == fault_rank && s == fault_step) continue;
          const int dst = (r + 1) % p;
          const Chunk c = chunk(p, n, ((r - s - 1) % p + p) % p);
          std::copy(work[r].begin() + c.off, work[r].begin() + c.off + c.len, inbox[dst].begin());
          tag[dst] = s;
          sent[r] += c.len * sizeof(Acc);
        }
        if (!bar->wait()) return;
        for (int r = t; r < p; r += T) {
          const int src = (r - 1 + p) % p;
          if (tag[r] != s) {
            bar->abort(kLostMessage);
            return;
          }
          const Chunk c = chunk(p, n, ((src - s - 1) % p + p) % p);
          for (uint64_t i = 0; i < c.len; ++i) work[r][c.off + i] = combine(inbox[r][i], work[r][c.off + i]);
        }
        if (!bar->wait()) return;
      }
    }
    // the owner's finished chunk
    for (int r = t; r < p; r += T) {
      const Chunk c = chunk(p, n, r);
      if (kind == kReduceScatter) {
        Out* o = static_cast<Out*>(recv[r]);
        for (uint64_t i = 0; i < c.len; ++i) o[i] = finish(work[r][c.off + i]);
      } else {
        full[r].assign(n, Out{});
        if (kind == kAllGather) {
          std::memcpy(full[r].data() + c.off, send[r], c.len * sizeof(Out));
        } else {
          for (uint64_t i = 0; i < c.len; ++i) full[r][c.off + i] = finish(work[r][c.off + i]);
        }
      }
    }
    if (!bar->wait()) return;
    if (do_ag) {
      for (int s = 0; s < p - 1; ++s) {
        const int step = (do_rs ? p - 1 : 0) + s;
        for (int r = t; r < p; r += T) {
          if (stalls(r, step)) {
            bar->wait_for_abort();
            return;
          }
          if (fault == kSkipSend && r == fault_rank && step == fault_step) continue;
          const int dst = (r + 1) % p;
          const Chunk c = chunk(p, n, ((r - s) % p + p) % p);
          std::copy(full[r].begin() + c.off, full[r].begin() + c.off + c.len, inbox2[dst].begin());
          tag[dst] = step;
          sent[r] += c.len * sizeof(Out);
        }
        if (!bar->wait()) return;
        for (int r = t; r < p; r += T) {
          const int src = (r - 1 + p) % p;
          if (tag[r] != step) {
            bar->abort(kLostMessage);
            return;
          }
          const Chunk c = chunk(p, n, ((src - s) % p + p) % p);
          std::copy(inbox2[r].begin(), inbox2[r].begin() + c.len, full[r].begin() + c.off);
        }
        if (!bar->wait()) return;
      }
      for (int r = t; r < p; r += T) {
        if (kind == kBucket) {
          uint16_t* o = static_cast<uint16_t*>(recv[r]);
          for (uint64_t i = 0; i < n; ++i) {
            const float prod = static_cast<float>(full[r][i]) * scale;  // one fp32 rounding
            o[i] = f32_to_bf16(prod);
          }
        } else {
          std::memcpy(recv[r], full[r].data(), n * sizeof(Out));
        }
      }
    }
  }
};

template <typename Acc, typename Out>
int run_ring(int kind, const void* const* send, void* const* recv, int p, uint64_t n, int dtype, int op,
             float scale, int max_threads, double timeout_s, int fault, int fault_rank, int fault_step,
             uint64_t* bytes_sent, int* threads_used) {
  Ring<Acc, Out> R;
  R.kind = kind;
  R.p = p;
  R.dtype = dtype;
  R.op = op;
  R.n = n;
  R.scale = scale;
  R.send = send;
  R.recv = recv;
  R.fault = fault;
  R.fault_rank = fault_rank;
  R.fault_step = fault_step;
  const uint64_t maxlen = chunk(p, n, 0).len;
  R.work.resize(p);
  R.full.resize(p);
  R.inbox.assign(p, std::vector<Acc>(kind == kAllGather ? 0 : maxlen));
  R.inbox2.assign(p, std::vector<Out>(kind == kReduceScatter ? 0 : maxlen));
  R.tag.assign(p, -1);
  R.sent.assign(p, 0);
  const int T = p < max_threads ? p : max_threads;
  Barrier bar(T, timeout_s);
  R.bar = &bar;
  std::vector<std::thread> pool;
  pool.reserve(T);
  for (int t = 0; t < T; ++t) pool.emplace_back([&R, t, T] { R.run(t, T); });
  for (auto& th : pool) th.join();
  if (bytes_sent != nullptr)
    for (int r = 0; r < p; ++r) bytes_sent[r] = R.sent[r];
  if (threads_used != nullptr) *threads_used = T;
  return bar.status();
}

}  // namespace

extern "C" {

// One collective over p CPU ranks (see the file header).
//   kind        0 all-reduce, 1 reduce-scatter, 2 all-gather, 3 DDP bucket
//               (fp32 all-reduce, x scale in fp32, one bf16 rounding)
//   send/recv   host pointers per rank: all-reduce / bucket n -> n elements;
//               reduce-scatter n -> len(k); all-gather len(k) -> n
//   dtype       0 f32, 1 bf16 (uint16 bits), 2 i32; the bucket takes f32 in, bf16 out
//   op          0 sum, 1 max, 2 min (sum only for the bucket)
//   max_threads host threads (ranks dealt round-robin); timeout_s bounds every wait
//   fault       0 none, 1 rank fault_rank stalls from step fault_step on,
//               2 rank fault_rank skips its send of step fault_step (steps
//               count the reduce-scatter's p-1 first, then the all-gather's)
//   bytes_sent  p entries or NULL: bytes each rank sent (4 per partial element
//               in the reduce-scatter, the element size in the all-gather)
// Returns 0, 1 (bad arguments), 4 (a wait timed out) or 5 (a message was lost).
int o3_ring(int kind, const void* const* send, void* const* recv, int p, uint64_t n, int dtype, int op,
            float scale, int max_threads, double timeout_s, int fault, int fault_rank, int fault_step,
            uint64_t* bytes_sent, int* threads_used) {
  if (p < 1 || p > 4096 || max_threads < 1 || kind < 0 || kind > 3 || dtype < 0 || dtype > 2 || op < 0 ||
      op > 2 || !(timeout_s > 0) || send == nullptr || recv == nullptr)
    return kInvalid;
  if (kind == kBucket && (dtype != kF32 || op != kSum)) return kInvalid;
  for (int r = 0; r < p; ++r)
    if ((send[r] == nullptr || recv[r] == nullptr) && n > 0) return kInvalid;
  if (kind == kBucket)
    return run_ring<float, float>(kind, send, recv, p, n, dtype, op, scale, max_threads, timeout_s, fault,
                                  fault_rank, fault_step, bytes_sent, threads_used);
  if (dtype == kF32)
    return run_ring<float, float>(kind, send, recv, p, n, dtype, op, scale, max_threads, timeout_s, fault,
                                  fault_rank, fault_step, bytes_sent, threads_used);
  if (dtype == kBF16)
    return run_ring<float, uint16_t>(kind, send, recv, p, n, dtype, op, scale, max_threads, timeout_s, fault,
                                     fault_rank, fault_step, bytes_sent, threads_used);
  return run_ring<int32_t, int32_t>(kind, send, recv, p, n, dtype, op, scale, max_threads, timeout_s, fault,
                                    fault_rank, fault_step, bytes_sent, threads_used);
}

}  // extern "C"
