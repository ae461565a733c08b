// Routing layout: the per-(source rank, expert) routing-count histogram, stable per-pair
// ranks, the exclusive scans that turn counts into collision-free contiguous offsets, and
// the per-pair placements every data kernel reads.
//
// "Enabling trillion-parameter models on AWS EFA" (Perplexity), section "Dispatch and
// combine": dispatch send first aggregates the routing with shared-memory atomics inside a
// single block into per-expert token counts, then takes their cumulative sum to get the
// offsets at which tokens fill the per-peer send buffers; the receiver centralises all
// ranks' routing and computes the offsets for dispatch and combine (on the host in the
// page's design, here on the GPU). Section "Send and receive buffers": senders can place
// their writes contiguously and without collisions once per-expert counts are known.
//
// Differences from the page's design, for sm_103a and bit-exact reproducibility:
//  - one 1024-thread CTA per source rank counts with warp __match_any_sync groups plus a
//    per-warp table in shared memory, so the rank of each pair among the same expert's
//    pairs is its (token, slot) order — deterministic, unlike an atomic slot grab;
//  - the last CTA to finish (completion counter, no spinning) runs every scan, so the
//    whole histogram + scan step is one launch.
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kCountThreads = 1024;
constexpr unsigned kFull = 0xffffffffu;

struct LayoutArgs {
  const int32_t* idx;
  int32_t *cnt, *C, *soff, *roff, *rtot, *ecnt, *eoff;
  int32_t *pos, *rrow, *slot, *slot_src, *recv_src;
  int32_t *gsend, *grecv, *gslot;
  int32_t* status;
  int32_t* done;
};

// Exclusive scans over the full count table; run by the last CTA of k_route_count.
// sm holds at least N*E + N*N ints.
__device__ __forceinline__ void layout_scans(const Geo& g, const LayoutArgs& a, int32_t* sm) {
  const int N = g.N, E = g.E, L = g.L;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* scnt = sm;          // [N][E]
  int32_t* sC = sm + N * E;    // [N][N], sC[s*N + d]

#pragma unroll 4
  for (int i = tid; i < N * E; i += kCountThreads) scnt[i] = __ldcg(a.cnt + i);
  __syncthreads();

  // C[s][d] = sum over d's experts of cnt[s][.]
  for (int i = tid; i < N * N; i += kCountThreads) {
    const int s = i / N, d = i - s * N;
    int c = 0;
    for (int l = 0; l < L; ++l) c += scnt[s * E + d * L + l];
    sC[i] = c;
    a.C[i] = c;
  }
  // soff[s][e]: exclusive scan over experts, one warp per source rank
  for (int s = warp; s < N; s += kCountThreads / 32) {
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? scnt[s * E + e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
      }
      if (e < E) a.soff[(int64_t)s * E + e] = carry + incl - v;
      carry += __shfl_sync(kFull, incl, 31);
    }
  }
  // eoff[d][l][s] (= eoff[e][s]) and ecnt[e]: exclusive scan over source ranks, per expert
  for (int e = tid; e < E; e += kCountThreads) {
    int r = 0;
    for (int s = 0; s < N; ++s) {
      a.eoff[(int64_t)e * N + s] = r;
      r += scnt[s * E + e];
    }
    a.ecnt[e] = r;
    if (r > g.cap) set_status(a.status, kBitCapacity);
  }
  __syncthreads();
  // roff[d][s] and rtot[d]: exclusive scan of C[.][d] over source ranks
  for (int d = tid; d < N; d += kCountThreads) {
    int r = 0;
    for (int s = 0; s < N; ++s) {
      a.roff[d * N + s] = r;
      r += sC[s * N + d];
    }
    a.rtot[d] = r;
    if ((int64_t)r > g.RB) set_status(a.status, kBitRecvBound);
  }
}

// One CTA per source rank s. Walks the rank's T*R pairs in (t,k) order, 1024 at a time.
// Writes cnt[s][.] and, into pos[], each pair's rank among rank s's pairs of the same
// expert (-1 for an id outside [0,E)).
__global__ void __launch_bounds__(kCountThreads, 1) k_route_count(Geo g, LayoutArgs a) {
  extern __shared__ int32_t sm[];
  __shared__ int is_last;
  const int E = g.E;
  int32_t* wtab = sm;            // [32][E]: per-warp counts, then per-warp exclusive offsets
  int32_t* run = sm + 32 * E;    // [E]: pairs of each expert in earlier chunks
  const int s = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t* idx_s = a.idx + (int64_t)s * g.TR;
  int32_t* rk_s = a.pos + (int64_t)s * g.TR;

  for (int e = tid; e < E; e += kCountThreads) run[e] = 0;
  for (int64_t base = 0; base < g.TR; base += kCountThreads) {
    for (int i = tid; i < 32 * E; i += kCountThreads) wtab[i] = 0;
    const int64_t pl = base + tid;
    const bool in = pl < g.TR;
    const int e = in ? __ldg(idx_s + pl) : -1;
    const bool ok = in && e >= 0 && e < E;
    if (in && !ok) set_status(a.status, kBitExpertRange);
    __syncthreads();
    const unsigned peers = __match_any_sync(kFull, ok ? e : -1);
    const int lrank = __popc(peers & ((1u << lane) - 1u));
    if (ok && lrank == 0) wtab[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int ee = tid; ee < E; ee += kCountThreads) {
      int r = run[ee];
#pragma unroll 8
      for (int w = 0; w < 32; ++w) {
        const int v = wtab[w * E + ee];
        wtab[w * E + ee] = r;
        r += v;
      }
      run[ee] = r;
    }
    __syncthreads();
    if (in) rk_s[pl] = ok ? wtab[warp * E + e] + lrank : -1;
    __syncthreads();
  }
  for (int e = tid; e < E; e += kCountThreads) a.cnt[(int64_t)s * E + e] = run[e];

  // The last CTA to finish computes the scans over all ranks' counts.
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = (atomicAdd(a.done, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  layout_scans(g, a, sm);
  if (tid == 0) *a.done = 0;  // ready for the next call
}

// Per-pair placements from ranks and scans, plus -1 padding of the inverse maps.
// Index space: [0,P) pairs, then E*cap grouped rows, then N*RB receive rows.
__global__ void __launch_bounds__(256) k_layout_maps(Geo g, LayoutArgs a) {
  const int64_t n_pairs = g.P;
  const int64_t n_slot = (int64_t)g.E * g.cap;
  const int64_t n_recv = (int64_t)g.N * g.RB;
  const int64_t total = n_pairs + n_slot + n_recv;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    if (i < n_pairs) {
      const int64_t q = i;
      const int e = __ldg(a.idx + q);
      if (e < 0 || e >= g.E) {  // pos[q] is already -1
        a.rrow[q] = -1;
        a.slot[q] = -1;
        a.gsend[q] = -1;
        a.grecv[q] = -1;
        a.gslot[q] = -1;
        continue;
      }
      const int s = (int)(q / g.TR);
      const int rk = a.pos[q];
      const int d = e / g.L;
      const int p = a.soff[(int64_t)s * g.E + e] + rk;
      const int rr = a.roff[d * g.N + s] + p - a.soff[(int64_t)s * g.E + d * g.L];
      const int sl = a.eoff[(int64_t)e * g.N + s] + rk;
      a.pos[q] = p;
      a.rrow[q] = rr;
      a.gsend[q] = (int32_t)((int64_t)s * g.TR + p);
      a.grecv[q] = (int32_t)((int64_t)d * g.RB + rr);
      a.recv_src[(int64_t)d * g.RB + rr] = (int32_t)q;
      if (sl < g.cap) {
        a.slot[q] = sl;
        a.gslot[q] = (int32_t)((int64_t)e * g.cap + sl);
        a.slot_src[(int64_t)e * g.cap + sl] = (int32_t)q;
      } else {
        a.slot[q] = -1;
        a.gslot[q] = -1;
      }
    } else if (i < n_pairs + n_slot) {
      const int64_t j = i - n_pairs;
      const int e = (int)(j / g.cap);
      const int r = (int)(j - (int64_t)e * g.cap);
      if (r >= a.ecnt[e]) a.slot_src[j] = -1;
    } else {
      const int64_t j = i - n_pairs - n_slot;
      const int d = (int)(j / g.RB);
      const int64_t r = j - (int64_t)d * g.RB;
      if (r >= a.rtot[d]) a.recv_src[j] = -1;
    }
  }
}

std::atomic<int> g_count_smem[64];

}  // namespace

size_t layout_smem_bytes(const Geo& g) {
  const size_t a = (size_t)33 * g.E;
  const size_t b = (size_t)g.N * g.E + (size_t)g.N * g.N;
  return 4 * (a > b ? a : b);
}

cudaError_t launch_layout(const Geo& g, const int32_t* idx, const moe_layout_t* lay, Ctx& c) {
  LayoutArgs a;
  a.idx = idx;
  a.cnt = lay->cnt;
  a.C = lay->C;
  a.soff = lay->soff;
  a.roff = lay->roff;
  a.rtot = lay->rtot;
  a.ecnt = lay->ecnt;
  a.eoff = lay->eoff;
  a.pos = lay->pos;
  a.rrow = lay->rrow;
  a.slot = lay->slot;
  a.slot_src = lay->slot_src;
  a.recv_src = lay->recv_src;
  a.gsend = lay->gsend;
  a.grecv = lay->grecv;
  a.gslot = lay->gslot;
  a.status = lay->status;
  a.done = lay->scratch;

  const size_t smem = layout_smem_bytes(g);
  if (smem + 1024 > (size_t)c.smem_optin) return cudaErrorInvalidValue;
  {
    cudaError_t e = ensure_dyn_smem(k_route_count, c.device, smem, g_count_smem);
    if (e != cudaSuccess) return e;
  }
  {
    LaunchScope ls(c, MOE_K_ROUTE_COUNT);
    k_route_count<<<g.N, kCountThreads, smem, c.stream>>>(g, a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int64_t total = g.P + (int64_t)g.E * g.cap + (int64_t)g.N * g.RB;
  if (total > 0) {
    int64_t blocks = (total + 255) / 256;
    const int64_t maxb = (int64_t)c.num_sms * 8;
    if (blocks > maxb) blocks = maxb;
    LaunchScope ls(c, MOE_K_LAYOUT_MAPS);
    k_layout_maps<<<(unsigned)blocks, 256, 0, c.stream>>>(g, a);
  }
  return cudaGetLastError();
}

}  // namespace moe
