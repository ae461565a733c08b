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
// CTAs are all resident at once:
//  1. sender work: every (token, column chunk) unit is pushed into the owners' receive
//     rows (the direct-push pack); after a row chunk lands, the warp release-increments
//     the arrival counter of its (destination d, source s) slice;
//  2. receiver work: each (pair, column chunk) unit waits, with an acquire poll bounded
//     by kSplitWaitNs, until its slice's counter reaches C[s][d] * chunks, then copies the
//     row chunk into its expert's grouped row (codes and scales apart for fp8).
// A CTA finishes all its sender units before it takes receiver units, and no sender ever
// waits, so every wait ends unless a signal is missing; then the status word gets the
// timeout bit, later waits give up at once, and the unfinished rows are skipped. The
// counters start at zero (moe_layout_init) and the last CTA of each call zeroes them again.
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

constexpr uint64_t kSplitWaitNs = 1000000000ull;   // 1 s
constexpr int kSplitThreads = 256;

struct SplitArgs {
  const uint8_t* x;     // [N][T][B] token rows
  uint8_t* recv;        // [N][RB][B]
  uint8_t* ex;          // grouped rows: [N][L][cap][B] (bf16) or codes [N][L][cap][H] (fp8)
  uint8_t* exs;         // fp8 scales [N][L][cap][H/128]
  const int32_t* gsend;
  const int32_t* grecv;
  const int32_t* gslot;
  const int32_t* C;     // [N][N]: rows s sends to d
  uint32_t* arrive;     // [N][N]: arrive[d*N + s], row chunks of slice (d, s) landed
  uint32_t* done;       // CTAs finished (the last one resets arrive[], done and abort)
  uint32_t* abort;      // set by the first wait that times out in this call
  int32_t* status;
  int chunks;           // column chunks per row
  int64_t chunk_bytes;
  int drop_slice;       // failure injection: the slice d*N+s whose signals are withheld, or -1
};

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Waits until *ctr >= target. Gives up at once if a wait of this call already timed out,
// else after kSplitWaitNs, recording the timeout. Returns whether the target was reached.
__device__ __forceinline__ bool wait_arrival(const uint32_t* ctr, uint32_t target, uint32_t* abort,
                                             int32_t* status) {
  if (ld_acquire(ctr) >= target) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (ld_acquire(ctr) >= target) return true;
    if (*reinterpret_cast<volatile uint32_t*>(abort)) return false;
    if (global_ns() - t0 > kSplitWaitNs) {
      atomicExch(abort, 1u);
      set_status(status, kBitTimeout);
      return false;
    }
    __nanosleep(256);
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
template <>
__device__ __forceinline__ uint4 ldv_l2<uint4>(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
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

template <bool FP8, typename V>
__global__ void __launch_bounds__(kSplitThreads) k_dispatch_split(Geo g, SplitArgs a) {
  constexpr int W = (int)sizeof(V);
  constexpr int U = 8;
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t nel = a.chunk_bytes / W;

  // ---- sender half: push every token chunk into its owners' receive rows, then signal
  const int64_t send_units = (int64_t)g.N * g.T * a.chunks;
  for (int64_t u = warp0; u < send_units; u += nwarps) {
    const int64_t tok = u / a.chunks;
    const int64_t coff = (u - tok * a.chunks) * a.chunk_bytes;
    const int s = (int)(tok / g.T);
    const uint8_t* src = a.x + tok * g.B + coff;
    const int myr = lane < g.R ? __ldg(a.grecv + tok * g.R + lane) : -1;   // R <= 32
    // The trip count is the same for every lane: the shuffles below need the whole warp.
    for (int64_t b0 = 0; b0 < nel; b0 += 32 * U) {
      const int64_t v0 = b0 + lane;
      V r[U];
#pragma unroll
      for (int j = 0; j < U; ++j)
        if (v0 + 32 * j < nel) r[j] = ldv<V>(src + (v0 + 32 * j) * W);
#pragma unroll 1
      for (int k = 0; k < g.R; ++k) {
        const int gr = __shfl_sync(0xffffffffu, myr, k);
        if (gr < 0) continue;
        uint8_t* d = a.recv + (int64_t)gr * g.B + coff;
#pragma unroll
        for (int j = 0; j < U; ++j)
          if (v0 + 32 * j < nel) stv(d + (v0 + 32 * j) * W, r[j]);
      }
    }
    // Every lane's stores of this chunk, then one release increment per destination row.
    __threadfence();
    __syncwarp();
    if (myr >= 0) {
      const int d = myr / (int)g.RB;
      const int slice = d * g.N + s;
      if (slice != a.drop_slice) {
        __threadfence();
        atomicAdd(a.arrive + slice, 1u);
      }
    }
  }

  // ---- receiver half: wait for the slice of each pair's row, then shuffle it into place
  const int64_t recv_units = g.P * a.chunks;
  for (int64_t u = warp0; u < recv_units; u += nwarps) {
    const int64_t q = u / a.chunks;
    const int64_t coff = (u - q * a.chunks) * a.chunk_bytes;
    const int gl = __ldg(a.gslot + q);
    if (gl < 0) continue;
    const int gr = __ldg(a.grecv + q);
    const int s = (int)(q / g.TR);
    const int d = gr / (int)g.RB;
    const uint32_t target = (uint32_t)__ldg(a.C + s * g.N + d) * (uint32_t)a.chunks;
    bool ready = true;
    if (lane == 0) ready = wait_arrival(a.arrive + d * g.N + s, target, a.abort, a.status);
    ready = __shfl_sync(0xffffffffu, ready, 0);
    __syncwarp();   // orders every lane's loads below after lane 0's acquire
    if (!ready) continue;
    const uint8_t* src = a.recv + (int64_t)gr * g.B + coff;
    for (int64_t b0 = 0; b0 < nel; b0 += 32 * U) {
      const int64_t v0 = b0 + lane;
      V r[U];
#pragma unroll
      for (int j = 0; j < U; ++j)
        if (v0 + 32 * j < nel) r[j] = ldv_l2<V>(src + (v0 + 32 * j) * W);
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int64_t v = v0 + 32 * j;
        if (v >= nel) continue;
        if (FP8) {   // one chunk per row: codes [0, H), then the scales
          const int64_t split = g.H / W;
          if (v < split)
            stv(a.ex + (int64_t)gl * g.H + v * W, r[j]);
          else
            stv(a.exs + (int64_t)gl * (g.H / 32) + (v - split) * W, r[j]);
        } else {
          stv(a.ex + (int64_t)gl * g.B + coff + v * W, r[j]);
        }
      }
    }
  }

  // The last CTA to finish zeroes the arrival counters for the next call.
  __shared__ int is_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    is_last = atomicAdd(a.done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (is_last) {
    for (int i = threadIdx.x; i < g.N * g.N; i += blockDim.x) a.arrive[i] = 0u;
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

cudaError_t launch_dispatch_split(const Geo& g, const moe_layout_t* lay, const void* x, void* recv, void* ex,
                                  float* exs, int drop_slice, Ctx& c) {
  SplitArgs a;
  a.x = static_cast<const uint8_t*>(x);
  a.recv = static_cast<uint8_t*>(recv);
  a.ex = static_cast<uint8_t*>(ex);
  a.exs = reinterpret_cast<uint8_t*>(exs);
  a.gsend = lay->gsend;
  a.grecv = lay->grecv;
  a.gslot = lay->gslot;
  a.C = lay->C;
  a.arrive = reinterpret_cast<uint32_t*>(lay->scratch + layout_scratch_arrive_offset(g));
  a.done = a.arrive + (int64_t)g.N * g.N;
  a.abort = a.done + 1;
  a.status = lay->status;
  a.drop_slice = drop_slice;
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  a.chunks = (!fp8 && g.B >= 8192 && g.B % 32 == 0) ? 2 : 1;
  a.chunk_bytes = g.B / a.chunks;
  if ((int64_t)g.N * g.T == 0) return cudaSuccess;
  LaunchScope ls(c, MOE_K_DISPATCH_SPLIT);
  if (g.B % 16 == 0)
    return fp8 ? run_split<true, uint4>(g, a, c) : run_split<false, uint4>(g, a, c);
  return fp8 ? run_split<true, uint32_t>(g, a, c) : run_split<false, uint32_t>(g, a, c);
}

}  // namespace moe
