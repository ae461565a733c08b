// Split-phase dispatch: the sender and receiver halves of dispatch in one launch, the
// receiver starting on a peer's rows as soon as that peer has signalled their arrival.
//
// "Enabling trillion-parameter models on AWS EFA" (Perplexity), section "Dispatch and
// combine": dispatch and combine are split into sender and receiver halves so that they
// overlap; the sender fills the buffers and signals, and the receiver blocks until every
// transfer has arrived, then shuffles the tokens into the grouped-GEMM input. Section "MoE
// all-to-all over EFA": within a node, tokens are pushed straight into peers' buffers.
//
// On one GPU the two halves cannot be separate kernels that wait on each other (nothing
// guarantees they run at the same time), so both run in one cooperative launch, whose
// CTAs are all resident at once. The tokens are taken in nb batches (tokens
// [j*T/nb, (j+1)*T/nb) of every rank), and every warp runs the two halves pipelined: it
// pushes its (token, column chunk) units of batch j+1 into the owners' receive rows (the
// direct-push pack) and, once they have landed (one fence), signals each on the counter of
// (batch j+1, source s); then it takes its (pair, column chunk) units of batch j, waits with
// an acquire poll until the pair's source has signalled every chunk of batch j, and copies
// the row chunk into its expert's grouped row (codes and scales apart for fp8). A batch's
// rows are read back one batch after they were pushed, while they are still in L2.
// Waits in that loop are short (kSplitQuickNs): one that runs out leaves the rest of the
// batch's units for later, so a warp's pushes never wait behind a missing signal. After its
// last push a warp finishes the units it left, each wait now bounded by kSplitWaitNs; every
// push of the call has landed by then, so a wait that runs out means a signal that will
// never come: the status word gets the timeout bit, later waits of the call give up at once
// unless their counter is already complete, and the unfinished rows are skipped. The
// counters start at zero (moe_layout_init) and the last CTA of each call zeroes them again.
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

constexpr uint64_t kSplitWaitNs = 1000000000ull;   // 1 s: a signal that will not come
constexpr uint64_t kSplitQuickNs = 20000ull;         // 20 us: leave the batch for later
constexpr int kSplitThreads = 256;
// Pushed rows per token batch, about a quarter of L2. Measured on GB300 with the receive
// half's evict-first reads: EP8 73.5 us in 4 batches against 79.9 in 7 (16 MB each), EP16
// skew 254 us in 16 against 272 in 32, EP32 225 us in 16 against 232 in 29.
constexpr int64_t kSplitBatchBytes = 32ll << 20;

struct SplitArgs {
  const uint8_t* x;     // [N][T][B] token rows
  uint8_t* recv;        // [N][RB][B]
  uint8_t* ex;          // grouped rows: [N][L][cap][B] (bf16) or codes [N][L][cap][H] (fp8)
  uint8_t* exs;         // fp8 scales [N][L][cap][H/128]
  const int32_t* grecv;
  const int32_t* gslot;
  uint32_t* arrive;     // [nb][N]: arrive[j*N + s], token chunks of source s in batch j landed
  uint32_t* done;       // CTAs finished (the last one resets arrive[], done and abort)
  uint32_t* abort;      // set by the first wait that times out in this call
  int32_t* status;
  int chunks;           // column chunks of a row per unit
  int nb;               // token batches
  int drop_source;      // failure injection: the source rank whose signals are withheld, or -1
};

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Waits until *ctr >= target. quick: gives up after kSplitQuickNs and records nothing (the
// caller retries later). Otherwise gives up at once if a wait of this call already timed
// out, else after kSplitWaitNs, recording the timeout. Returns whether the target was reached.
__device__ __forceinline__ bool wait_arrival(const uint32_t* ctr, uint32_t target, uint32_t* abort,
                                             int32_t* status, bool quick) {
  if (ld_acquire(ctr) >= target) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (ld_acquire(ctr) >= target) return true;
    const uint64_t dt = global_ns() - t0;
    if (quick) {
      if (dt > kSplitQuickNs) return false;
    } else {
      if (*reinterpret_cast<volatile uint32_t*>(abort)) return false;
      if (dt > kSplitWaitNs) {
        atomicExch(abort, 1u);
        set_status(status, kBitTimeout);
        return false;
      }
    }
    __nanosleep(128);
  }
}

// Token rows are read-only during the kernel (non-coherent path is fine); receive rows
// were written by other CTAs of this kernel, so they are read at L2 (.cg), after the acquire.
template <typename V>
__device__ __forceinline__ V ldv(const uint8_t* p);
template <>
__device__ __forceinline__ uint4 ldv<uint4>(const uint8_t* p) {
  return ld_stream16(p);
}
template <>
__device__ __forceinline__ uint32_t ldv<uint32_t>(const uint8_t* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}
template <typename V>
__device__ __forceinline__ V ldv_l2(const uint8_t* p);
// The receive half reads each pushed row once, for the last time in the pass: evict-first in
// L2, so the rows still being pushed and shuffled stay there (GB300: EP8 and EP32 split-phase
// steps 3-4% faster).
template <>
__device__ __forceinline__ uint4 ldv_l2<uint4>(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.cg.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(l2_evict_first_policy()));
  return v;
}
template <>
__device__ __forceinline__ uint32_t ldv_l2<uint32_t>(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void stv(uint8_t* p, const uint4& v) { st16(p, v); }
__device__ __forceinline__ void stv(uint8_t* p, const uint32_t& v) { *reinterpret_cast<uint32_t*>(p) = v; }

__device__ __forceinline__ int batch_lo(const Geo& g, int nb, int j) { return (int)((int64_t)j * g.T / nb); }

// Pushes this warp's (token, column chunk) units of batch j into the owners' receive rows,
// then, once they have landed, signals each on its source's counter of the batch.
template <typename V>
__device__ __forceinline__ void send_batch(const Geo& g, const SplitArgs& a, int j, int64_t w0, int64_t nw,
                                           int lane) {
  constexpr int W = (int)sizeof(V);
  constexpr int U = 8;
  const int64_t nel = g.B / W;
  const int64_t cv = (nel + a.chunks - 1) / a.chunks;   // vectors per chunk
  const int lo = batch_lo(g, a.nb, j), nt = batch_lo(g, a.nb, j + 1) - lo;
  const int64_t per_rank = (int64_t)nt * a.chunks;
  const int64_t units = (int64_t)g.N * per_rank;
  if (w0 >= units) return;
  for (int64_t u = w0; u < units; u += nw) {
    const int s = (int)(u / per_rank);
    const int64_t r = u - s * per_rank;
    const int64_t tok = (int64_t)s * g.T + lo + r / a.chunks;
    const int64_t v_lo = (r % a.chunks) * cv;
    const int64_t v_hi = v_lo + cv < nel ? v_lo + cv : nel;
    const uint8_t* src = a.x + tok * g.B;
    const int myr = lane < g.R ? __ldg(a.grecv + tok * g.R + lane) : -1;   // R <= 32
    // The trip count is the same for every lane: the shuffles below need the whole warp.
    for (int64_t b0 = v_lo; b0 < v_hi; b0 += 32 * U) {
      const int64_t v0 = b0 + lane;
      V v[U];
#pragma unroll
      for (int k = 0; k < U; ++k)
        if (v0 + 32 * k < v_hi) v[k] = ldv<V>(src + (v0 + 32 * k) * W);
#pragma unroll 1
      for (int k = 0; k < g.R; ++k) {
        const int gr = __shfl_sync(0xffffffffu, myr, k);
        if (gr < 0) continue;
        uint8_t* d = a.recv + (int64_t)gr * g.B;
#pragma unroll
        for (int i = 0; i < U; ++i)
          if (v0 + 32 * i < v_hi) stv(d + (v0 + 32 * i) * W, v[i]);
      }
    }
  }
  // Every lane's stores of the batch, then one increment per unit on its source's counter.
  __threadfence();
  __syncwarp();
  if (lane == 0)
    for (int64_t u = w0; u < units; u += nw) {
      const int s = (int)(u / per_rank);
      if (s != a.drop_source) atomicAdd(a.arrive + (int64_t)j * g.N + s, 1u);
    }
}

// Copies this warp's (pair, column chunk) units of batch j, from unit index `from` on, into
// the grouped rows once their source's batch has landed. quick: a wait that runs out stops
// the batch there; returns the unit index to resume from (or a value >= units when done).
template <bool FP8, typename V>
__device__ __forceinline__ int64_t recv_batch(const Geo& g, const SplitArgs& a, int j, int64_t from, int64_t nw,
                                              int lane, bool quick) {
  constexpr int W = (int)sizeof(V);
  constexpr int U = 8;
  const int64_t nel = g.B / W;
  const int64_t cv = (nel + a.chunks - 1) / a.chunks;
  const int64_t split = g.H / W;   // fp8: codes are vectors [0, split), scales the rest
  const int lo = batch_lo(g, a.nb, j), nt = batch_lo(g, a.nb, j + 1) - lo;
  const int64_t per_rank = (int64_t)nt * g.R * a.chunks;
  const int64_t units = (int64_t)g.N * per_rank;
  const uint32_t target = (uint32_t)nt * (uint32_t)a.chunks;
  int ready_s = -1;
  for (int64_t u = from; u < units; u += nw) {
    const int s = (int)(u / per_rank);
    const int64_t r = u - s * per_rank;
    const int64_t q = ((int64_t)s * g.T + lo) * g.R + r / a.chunks;
    const int64_t v_lo = (r % a.chunks) * cv;
    const int64_t v_hi = v_lo + cv < nel ? v_lo + cv : nel;
    const int gl = __ldg(a.gslot + q);
    const int gr = __ldg(a.grecv + q);
    if (gl < 0) continue;
    if (s != ready_s) {
      bool ok = true;
      if (lane == 0) ok = wait_arrival(a.arrive + (int64_t)j * g.N + s, target, a.abort, a.status, quick);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      __syncwarp();   // orders every lane's loads below after lane 0's acquire
      if (!ok) {
        if (quick) return u;   // resume here later
        continue;              // timed out: the row stays unwritten
      }
      ready_s = s;
    }
    const uint8_t* src = a.recv + (int64_t)gr * g.B;
    for (int64_t b0 = v_lo; b0 < v_hi; b0 += 32 * U) {
      const int64_t v0 = b0 + lane;
      V v[U];
#pragma unroll
      for (int k = 0; k < U; ++k)
        if (v0 + 32 * k < v_hi) v[k] = ldv_l2<V>(src + (v0 + 32 * k) * W);
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int64_t e = v0 + 32 * k;
        if (e >= v_hi) continue;
        if (FP8) {
          if (e < split)
            stv(a.ex + (int64_t)gl * g.H + e * W, v[k]);
          else
            stv(a.exs + (int64_t)gl * (g.H / 32) + (e - split) * W, v[k]);
        } else {
          stv(a.ex + (int64_t)gl * g.B + e * W, v[k]);
        }
      }
    }
  }
  return units;
}

template <bool FP8, typename V>
__global__ void __launch_bounds__(kSplitThreads, 2) k_dispatch_split(Geo g, SplitArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // Units of batch j go to warps from a rotating start, so the pushes of successive batches
  // fall on different warps.
  auto mine = [&](int j) { return (w0 + (int64_t)j * 977) % nw; };
  int64_t resume[kMaxSplitBatches];
  uint32_t left = 0;   // batches with units left for the second pass
  send_batch<V>(g, a, 0, mine(0), nw, lane);
  for (int j = 0; j < a.nb; ++j) {
    if (j + 1 < a.nb) send_batch<V>(g, a, j + 1, mine(j + 1), nw, lane);
    const int64_t at = recv_batch<FP8, V>(g, a, j, mine(j), nw, lane, true);
    const int lo = batch_lo(g, a.nb, j), nt = batch_lo(g, a.nb, j + 1) - lo;
    if (at < (int64_t)g.N * nt * g.R * a.chunks) {
      resume[j] = at;
      left |= 1u << j;
    }
  }
  // Every push of this warp is out; finish what the short waits left.
  for (int j = 0; j < a.nb; ++j)
    if (left & (1u << j)) recv_batch<FP8, V>(g, a, j, resume[j], nw, lane, false);

  // The last CTA to finish zeroes the arrival counters for the next call.
  __shared__ int is_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    is_last = atomicAdd(a.done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (is_last) {
    for (int i = threadIdx.x; i < a.nb * g.N; i += blockDim.x) a.arrive[i] = 0u;
    if (threadIdx.x == 0) {
      *a.abort = 0u;
      *a.done = 0u;
    }
  }
}

template <bool FP8, typename V>
cudaError_t run_split(const Geo& g, const SplitArgs& a, Ctx& c) {
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_dispatch_split<FP8, V>, kSplitThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)c.num_sms * per_sm));
  cfg.blockDim = dim3(kSplitThreads);
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: waits can be satisfied
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_dispatch_split<FP8, V>, g, a);
}

}  // namespace

int split_batches(const Geo& g) {
  int64_t nb = (g.P * g.B + kSplitBatchBytes / 2) / kSplitBatchBytes;
  if (nb > kMaxSplitBatches) nb = kMaxSplitBatches;
  if (nb > g.T) nb = g.T;
  return nb < 1 ? 1 : (int)nb;
}

cudaError_t launch_dispatch_split(const Geo& g, const moe_layout_t* lay, const void* x, void* recv, void* ex,
                                  float* exs, int drop_source, Ctx& c) {
  SplitArgs a;
  a.x = static_cast<const uint8_t*>(x);
  a.recv = static_cast<uint8_t*>(recv);
  a.ex = static_cast<uint8_t*>(ex);
  a.exs = reinterpret_cast<uint8_t*>(exs);
  a.grecv = lay->grecv;
  a.gslot = lay->gslot;
  a.arrive = reinterpret_cast<uint32_t*>(lay->scratch + layout_scratch_arrive_offset(g));
  a.done = a.arrive + split_arrive_words(g);
  a.abort = a.done + 1;
  a.status = lay->status;
  a.drop_source = drop_source;
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  // Units are row chunks of about 4 KB: one round of eight vectors per lane.
  a.chunks = (int)((g.B + 4095) / 4096);
  a.nb = lay->batches > 0 ? (lay->batches < kMaxSplitBatches ? lay->batches : kMaxSplitBatches) : split_batches(g);
  if (a.nb > g.T) a.nb = g.T < 1 ? 1 : g.T;
  if ((int64_t)g.N * g.T == 0) return cudaSuccess;
  LaunchScope ls(c, MOE_K_DISPATCH_SPLIT);
  if (g.B % 16 == 0)
    return fp8 ? run_split<true, uint4>(g, a, c) : run_split<false, uint4>(g, a, c);
  return fp8 ? run_split<true, uint32_t>(g, a, c) : run_split<false, uint32_t>(g, a, c);
}

}  // namespace moe
