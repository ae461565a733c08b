// Split-phase dispatch with per-sender dedicated space and the routing information
// piggybacked on the first writes.
//
// "Enabling trillion-parameter models on AWS EFA" (Perplexity), section "Send and receive
// buffers": exchanging the routing information alone would make every rank wait before its
// writes; instead each receiver reserves a small dedicated space per sender, and the sender
// dispatches part of its tokens together with the routing-information write. Once the
// routes have been exchanged, the remaining tokens go with one write per peer. Section
// "Dispatch and combine": the receiver centralises the routing of all its peers and
// computes the offsets it needs; it blocks until every transfer has arrived and then
// shuffles the tokens into the grouped-GEMM input.
//
// On one GPU every rank is an address range and the whole exchange is one cooperative
// launch (all CTAs resident). A sender uses only its own routing (cnt[s][.], soff[s][.] and
// its pairs' send positions pos); a receiver computes its offsets only from the counts the
// senders piggybacked. Work items, taken by every warp in this order:
//  M. for each (receiver d, sender s): the counts of d's experts, meta[d][s][l] =
//     cnt[s][d*L + l], then mflag[d][s] (release);
//  P. for each receiver d: wait for every sender's counts (mflag), then C[s][d], the shared
//     region's offsets moff[d][s] = sum over s' < s of max(C[s'][d] - K, 0), the grouped
//     offsets eoffx[d][l][s] = sum over s' < s of meta[d][s'][l] and the slice-local
//     expert offsets spre[d][s][l]; then pflag[d] (release);
//  S. for each (token, column chunk of about 4 KB), one lane per pair: a pair whose place j
//     in the slice (d, s) is below K goes to ded[d][s][j] at once; the others wait for
//     pflag[d] and go to main[d][moff[d][s] + j - K]; each chunk is read once and stored R
//     times; once it has landed (one fence), each lane signals its row chunk on arrive[d][s]
//     (a slice is complete at C[s][d] x chunks);
//  C. for each item (a group of 8 places j of a slice (d, s) below its row count C[s][d],
//     from the reported counts, and a column chunk of about 4 KB): wait for pflag[d] and the
//     slice's C[s][d] rows; lanes 0..7 find their row's expert l from spre (the receiver
//     never reads the senders' routing arrays) and its grouped row eoffx[d][l][s] + j -
//     spre[d][s][l] (dropped at or beyond cap); the warp copies the chunk of each of the 8
//     rows from the dedicated or the shared region.
// A wait depends only on items of earlier letters, and items of M never wait, so every wait
// ends unless a signal is missing (withheld for a test); then the status word gets the
// timeout bit, later waits of the call give up at once, and their rows are skipped. The
// flags and counters are zeroed on the stream before each launch.
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

constexpr uint64_t kDedWaitNs = 1000000000ull;   // 1 s
constexpr int kDedThreads = 256;
constexpr int kRowsPerItem = 4;   // receive rows one warp item handles
constexpr int64_t kItemBytes = 4096;   // column chunk of a receive item

struct DedArgs {
  const uint8_t* x;       // [N][T][B] token rows
  const int32_t* idx;     // [N][T][R]
  const int32_t* pos;     // [N][T][R] send position of each pair (sender-local)
  const int32_t* soff;    // [N][E] send offsets (sender-local)
  const int32_t* cnt;     // [N][E] counts (sender-local)
  uint8_t* ded;           // [N][N][K][B]
  uint8_t* main;          // [N][RB][B]
  uint8_t* ex;            // grouped rows: [N][L][cap][B] (bf16) or codes [N][L][cap][H] (fp8)
  uint8_t* exs;           // fp8 scales [N][L][cap][H/128]
  int32_t* meta;          // [N][N][L]: counts sender s reports to receiver d
  int32_t* cx;            // [N][N]: C[s][d] as receiver d computed it, at d*N + s
  int32_t* moff;          // [N][N]
  int32_t* eoffx;         // [N][L][N]
  int32_t* spre;          // [N][N][L]
  uint32_t* mflag;        // [N][N]
  uint32_t* pflag;        // [N]
  uint32_t* arrive;       // [N][N]: row chunks of slice (d, s) landed, at d*N + s
  uint32_t* abort;        // a wait of this call timed out
  int32_t* status;
  int K;
  int drop_slice;
};

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits until *ctr >= target, bounded like the split-phase waits. The polls back off from
// 256 ns to 1 us, so that thousands of waiting warps leave the counters' lines to the
// senders' increments (a 4 us ceiling measured 0.5-2.3% slower on GB300: a warp woke up to
// 4 us after its slice had landed).
__device__ __forceinline__ bool wait_at_least(const uint32_t* ctr, uint32_t target, uint32_t* abort, int32_t* status) {
  if (ld_acquire(ctr) >= target) return true;
  const uint64_t t0 = global_ns();
  unsigned nap = 256;
  while (true) {
    if (ld_acquire(ctr) >= target) return true;
    if (*reinterpret_cast<volatile uint32_t*>(abort)) return false;
    if (global_ns() - t0 > kDedWaitNs) {
      atomicExch(abort, 1u);
      set_status(status, kBitTimeout);
      return false;
    }
    __nanosleep(nap);
    if (nap < 1024) nap <<= 1;
  }
}

template <typename V>
__device__ __forceinline__ V ld_nc(const uint8_t* p);
template <>
__device__ __forceinline__ uint4 ld_nc<uint4>(const uint8_t* p) {
  return ld_stream16(p);
}
template <>
__device__ __forceinline__ uint32_t ld_nc<uint32_t>(const uint8_t* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}
template <typename V>
__device__ __forceinline__ V ld_l2(const uint8_t* p);
template <>
__device__ __forceinline__ uint4 ld_l2<uint4>(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
template <>
__device__ __forceinline__ uint32_t ld_l2<uint32_t>(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_v(uint8_t* p, const uint4& v) { st16(p, v); }
__device__ __forceinline__ void st_v(uint8_t* p, const uint32_t& v) { *reinterpret_cast<uint32_t*>(p) = v; }


// Sends the column chunk [v_lo, v_hi) (in vectors) of token tok, lane k holding pair k: a
// place j < K in its slice goes to the dedicated rows, the rest to the shared region once the
// receiver's offsets are out. The chunk is read once and stored to its pairs' rows; after
// one fence every lane with a row signals the chunk on its slice.
template <typename V>
__device__ __forceinline__ void send_unit(const Geo& g, const DedArgs& a, int64_t tok, int64_t v_lo, int64_t v_hi,
                                          int lane) {
  constexpr int W = (int)sizeof(V);
  constexpr int U = 8;
  uint8_t* myrow = nullptr;
  int myslice = -1;
  if (lane < g.R) {
    const int s = (int)(tok / g.T);
    const int64_t q = tok * g.R + lane;
    const int e = __ldg(a.idx + q);
    if (e >= 0 && e < g.E) {
      const int d = e / g.L;
      const int j = __ldg(a.pos + q) - __ldg(a.soff + (int64_t)s * g.E + d * g.L);   // place in the slice
      const int slice = d * g.N + s;
      if (j < a.K) {
        myrow = a.ded + ((int64_t)slice * a.K + j) * g.B;
        myslice = slice;
      } else if (wait_at_least(a.pflag + d, 1u, a.abort, a.status)) {
        myrow = a.main + ((int64_t)d * g.RB + __ldcg(a.moff + slice) + (j - a.K)) * g.B;
        myslice = slice;
      }
    }
  }
  const unsigned any = __ballot_sync(0xffffffffu, myrow != nullptr);
  if (any) {
    const uint8_t* src = a.x + tok * g.B;
    for (int64_t b0 = v_lo; b0 < v_hi; b0 += 32 * U) {   // same trip count on every lane
      const int64_t v0 = b0 + lane;
      V r[U];
#pragma unroll
      for (int j = 0; j < U; ++j)
        if (v0 + 32 * j < v_hi) r[j] = ld_nc<V>(src + (v0 + 32 * j) * W);
#pragma unroll 1
      for (int k = 0; k < g.R; ++k) {
        if (!((any >> k) & 1u)) continue;
        uint8_t* dst = reinterpret_cast<uint8_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(myrow), k));
#pragma unroll
        for (int j = 0; j < U; ++j)
          if (v0 + 32 * j < v_hi) st_v(dst + (v0 + 32 * j) * W, r[j]);
      }
    }
  }
  __threadfence();
  __syncwarp();
  // One increment per slice: lanes whose rows share a slice add their count together.
  const int key = (myrow && myslice != a.drop_slice) ? myslice : -1;
  const unsigned same = __match_any_sync(0xffffffffu, key);
  if (key >= 0 && lane == __ffs(same) - 1) atomicAdd(a.arrive + key, (unsigned)__popc(same));
}

// Largest i in [0, n) with v[i] <= key (v ascending, v[0] <= key).
__device__ __forceinline__ int last_at_most(const int32_t* v, int n, int key) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldcg(v + mid) <= key)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

template <bool FP8, typename V>
__global__ void __launch_bounds__(kDedThreads, 2) k_dispatch_dedicated(Geo g, DedArgs a) {
  constexpr int W = (int)sizeof(V);
  constexpr int U = 8;
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int N = g.N, L = g.L;
  const int64_t tokens = (int64_t)N * g.T;

  // ---- M: the routing information
  for (int64_t it = warp0; it < (int64_t)N * N; it += nwarps) {   // it = d*N + s
    const int d = (int)(it / N), s = (int)(it - (int64_t)d * N);
    for (int l = lane; l < L; l += 32) a.meta[it * L + l] = __ldg(a.cnt + (int64_t)s * g.E + d * L + l);
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release(a.mflag + it, 1u);
  }

  // ---- P: each receiver's offsets from the counts its senders reported
  for (int64_t d = warp0; d < N; d += nwarps) {
    bool ok = true;
    for (int s = lane; s < N; s += 32) ok = ok && wait_at_least(a.mflag + d * N + s, 1u, a.abort, a.status);
    ok = __all_sync(0xffffffffu, ok);
    __syncwarp();   // every lane's acquires before any lane reads another sender's counts
    if (!ok) continue;
    const int32_t* m = a.meta + d * N * L;     // [s][l]
    int carry_m = 0;
    for (int s0 = 0; s0 < N; s0 += 32) {       // per sender: slice-local expert offsets and C
      const int s = s0 + lane;
      int c = 0;
      if (s < N)
        for (int l = 0; l < L; ++l) {
          a.spre[((int64_t)d * N + s) * L + l] = c;
          c += __ldcg(m + (int64_t)s * L + l);
        }
      const int vm = s < N ? (c > a.K ? c - a.K : 0) : 0;
      int im = vm;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int tm = __shfl_up_sync(0xffffffffu, im, o);
        if (lane >= o) im += tm;
      }
      if (s < N) {
        a.cx[d * N + s] = c;
        a.moff[d * N + s] = carry_m + im - vm;
      }
      carry_m += __shfl_sync(0xffffffffu, im, 31);
    }
    for (int l0 = 0; l0 < L; l0 += 32) {       // per expert: grouped offsets over senders
      const int l = l0 + lane;
      if (l < L) {
        int run = 0;
        for (int s = 0; s < N; ++s) {
          a.eoffx[((int64_t)d * L + l) * N + s] = run;
          run += __ldcg(m + (int64_t)s * L + l);
        }
      }
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release(a.pflag + d, 1u);
  }

  const int64_t nel = g.B / W;
  const int chunks = (int)((g.B + kItemBytes - 1) / kItemBytes);   // column chunks of a row
  const int64_t cv = (nel + chunks - 1) / chunks;

  // ---- S: every token row chunk once, to its dedicated and shared-region rows
  for (int64_t u = warp0; u < tokens * chunks; u += nwarps) {
    const int64_t tok = u / chunks, v_lo = (u - tok * chunks) * cv;
    send_unit<V>(g, a, tok, v_lo, v_lo + cv < nel ? v_lo + cv : nel, lane);
  }

  // ---- C: receive: items of up to kRowsPerItem places of one slice (d, s) and one column
  // chunk, each row chunk into its expert's grouped row
  const int64_t split = g.H / W;   // fp8: codes are vectors [0, split), scales the rest
  // Row groups per slice: enough for an average slice (P / N^2 rows); group m of a slice
  // takes the places m, m + per_slice, ... (in steps of kRowsPerItem rows), so a long
  // (skewed) slice is still covered.
  int64_t per_slice = (g.P + (int64_t)N * N * kRowsPerItem - 1) / ((int64_t)N * N * kRowsPerItem);
  const int64_t most = (g.TR + kRowsPerItem - 1) / kRowsPerItem;   // a slice has <= T*R rows
  per_slice = per_slice < 1 ? 1 : (per_slice > most ? most : per_slice);
  const int64_t items = (int64_t)N * N * per_slice * chunks;
  for (int64_t it = warp0; it < items; it += nwarps) {
    const int64_t sg = it / chunks;
    const int ch = (int)(it - sg * chunks);
    const int slice = (int)(sg / per_slice);
    const int d = slice / N, s = slice - d * N;
    const int j0 = (int)(sg - (int64_t)slice * per_slice) * kRowsPerItem;
    bool ok = lane == 0 ? wait_at_least(a.pflag + d, 1u, a.abort, a.status) : false;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    if (!ok) continue;
    const int c = __ldcg(a.cx + slice);   // rows of the slice, from the reported counts
    if (j0 >= c) continue;
    ok = lane == 0 ? wait_at_least(a.arrive + slice, (uint32_t)c * (uint32_t)chunks, a.abort, a.status) : false;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    if (!ok) continue;
    const int moff = __ldcg(a.moff + slice);
    const int64_t v_lo = ch * cv, v_hi = v_lo + cv < nel ? v_lo + cv : nel;
    for (int jg = j0; jg < c; jg += (int)per_slice * kRowsPerItem) {
      // lanes 0 .. kRowsPerItem-1: place jg + lane's expert, grouped row and source row
      const uint8_t* mysrc = nullptr;
      int64_t mygl = -1;
      if (lane < kRowsPerItem && jg + lane < c) {
        const int j = jg + lane;
        const int l = last_at_most(a.spre + (int64_t)slice * L, L, j);   // the slice is expert-major
        const int slot = __ldcg(a.eoffx + ((int64_t)d * L + l) * N + s) + j - __ldcg(a.spre + (int64_t)slice * L + l);
        if (slot < g.cap) {   // else dropped for capacity
          mygl = ((int64_t)d * L + l) * g.cap + slot;
          mysrc = j < a.K ? a.ded + ((int64_t)slice * a.K + j) * g.B
                          : a.main + ((int64_t)d * g.RB + moff + (j - a.K)) * g.B;
        }
      }
      for (int rr = 0; rr < kRowsPerItem; ++rr) {
        const int64_t gl = __shfl_sync(0xffffffffu, mygl, rr);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mysrc), rr));
        if (gl < 0) continue;
        for (int64_t b0 = v_lo; b0 < v_hi; b0 += 32 * U) {
          const int64_t v0 = b0 + lane;
          V r[U];
#pragma unroll
          for (int k = 0; k < U; ++k)
            if (v0 + 32 * k < v_hi) r[k] = ld_l2<V>(src + (v0 + 32 * k) * W);
#pragma unroll
          for (int k = 0; k < U; ++k) {
            const int64_t v = v0 + 32 * k;
            if (v >= v_hi) continue;
            if (FP8) {
              if (v < split)
                st_v(a.ex + gl * g.H + v * W, r[k]);
              else
                st_v(a.exs + gl * (g.H / 32) + (v - split) * W, r[k]);
            } else {
              st_v(a.ex + gl * g.B + v * W, r[k]);
            }
          }
        }
      }
    }
  }
}

template <bool FP8, typename V>
cudaError_t run_dedicated(const Geo& g, const DedArgs& a, Ctx& c) {
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_dispatch_dedicated<FP8, V>, kDedThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)c.num_sms * per_sm));
  cfg.blockDim = dim3(kDedThreads);
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: every wait can be satisfied
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_dispatch_dedicated<FP8, V>, g, a);
}

// Exchange buffer, int32 words: meta [N][N][L], cx, moff [N][N], eoffx [N][L][N],
// spre [N][N][L], then the flags and counters mflag [N][N], pflag [N], arrive [N][N],
// abort [1], zeroed at each call.
struct XchgPlan {
  int64_t meta, cx, moff, eoffx, spre, mflag, pflag, arrive, abort, total, flags_from;
};

XchgPlan xchg_plan(const Geo& g) {
  const int64_t N = g.N, E = g.E;
  XchgPlan p;
  p.meta = 0;
  p.cx = p.meta + N * E;
  p.moff = p.cx + N * N;
  p.eoffx = p.moff + N * N;
  p.spre = p.eoffx + N * E;
  p.mflag = p.spre + N * E;
  p.pflag = p.mflag + N * N;
  p.arrive = p.pflag + N;
  p.abort = p.arrive + N * N;
  p.total = p.abort + 1;
  p.flags_from = p.mflag;
  return p;
}

}  // namespace

size_t dedicated_exchange_bytes(const Geo& g) { return (size_t)(4 * xchg_plan(g).total + 255) & ~(size_t)255; }

cudaError_t launch_dispatch_dedicated(const Geo& g, const moe_layout_t* lay, const int32_t* idx, const void* x,
                                      int K, void* ded, void* xchg, void* main, void* ex, float* exs,
                                      int drop_slice, Ctx& c) {
  const XchgPlan p = xchg_plan(g);
  int32_t* w = static_cast<int32_t*>(xchg);
  cudaError_t e = cudaMemsetAsync(w + p.flags_from, 0, 4 * (size_t)(p.total - p.flags_from), c.stream);
  if (e != cudaSuccess || (int64_t)g.N * g.T == 0) return e;
  DedArgs a;
  a.x = static_cast<const uint8_t*>(x);
  a.idx = idx;
  a.pos = lay->pos;
  a.soff = lay->soff;
  a.cnt = lay->cnt;
  a.ded = static_cast<uint8_t*>(ded);
  a.main = static_cast<uint8_t*>(main);
  a.ex = static_cast<uint8_t*>(ex);
  a.exs = reinterpret_cast<uint8_t*>(exs);
  a.meta = w + p.meta;
  a.cx = w + p.cx;
  a.moff = w + p.moff;
  a.eoffx = w + p.eoffx;
  a.spre = w + p.spre;
  a.mflag = reinterpret_cast<uint32_t*>(w + p.mflag);
  a.pflag = reinterpret_cast<uint32_t*>(w + p.pflag);
  a.arrive = reinterpret_cast<uint32_t*>(w + p.arrive);
  a.abort = reinterpret_cast<uint32_t*>(w + p.abort);
  a.status = lay->status;
  a.K = K;
  a.drop_slice = drop_slice;
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  LaunchScope ls(c, MOE_K_DISPATCH_DEDICATED);
  if (g.B % 16 == 0) return fp8 ? run_dedicated<true, uint4>(g, a, c) : run_dedicated<false, uint4>(g, a, c);
  return fp8 ? run_dedicated<true, uint32_t>(g, a, c) : run_dedicated<false, uint32_t>(g, a, c);
}

}  // namespace moe
