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
//  - the histogram is split over 256-pair chunks, one 256-thread CTA each; warp
//    __match_any_sync groups plus a per-warp table in shared memory give each pair its
//    rank among the chunk's pairs of the same expert in (token, slot) order —
//    deterministic, unlike an atomic slot grab;
//  - one CTA then turns the chunk table into chunk offsets and totals and runs every
//    scan; the maps kernel adds a pair's chunk offset to its chunk-local rank. The three
//    kernels chain with programmatic dependent launch.
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kChunk = 256;          // pairs per histogram CTA (= its threads)
constexpr int kScanThreads = 1024;   // threads of the scan CTA
constexpr unsigned kFull = 0xffffffffu;

struct LayoutArgs {
  const int32_t* idx;
  int32_t *cnt, *C, *soff, *roff, *rtot, *ecnt, *eoff;
  int32_t *pos, *rrow, *slot, *slot_src, *recv_src;
  int32_t *gsend, *grecv, *gslot;
  int32_t* status;
  int32_t* ccnt;    // [N][nch][E]: per-chunk counts
  int nch;          // chunks per rank, ceil(T*R / kChunk)
};

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive scans over the full count table; run by the last CTA of k_route_count.
// The table is staged in shared memory with odd row strides (E|1, N|1) so that the
// column walks below are free of bank conflicts; every scan runs one warp per row with
// lanes along the scanned dimension, so the global stores are coalesced.
__device__ __forceinline__ void layout_scans(const Geo& g, const LayoutArgs& a, int32_t* sm) {
  const int N = g.N, E = g.E, L = g.L;
  const int E1 = E | 1, N1 = N | 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kScanThreads / 32;
  int32_t* scnt = sm;               // [N][E1]
  int32_t* sC = sm + N * E1;        // [N][N1], sC[s*N1 + d] = C[s][d]

  // cnt[s][e] = sum of the chunk counts, read kColBatch columns at a time so that their
  // loads are in flight together.
  constexpr int kColBatch = 8;
  const int nch = a.nch;
  const int NE = N * E;
  for (int i0 = tid; i0 < NE; i0 += kScanThreads * kColBatch) {
    int run[kColBatch];
#pragma unroll
    for (int j = 0; j < kColBatch; ++j) run[j] = 0;
    for (int c = 0; c < nch; ++c) {
      int v[kColBatch];
#pragma unroll
      for (int j = 0; j < kColBatch; ++j) {
        const int i = i0 + j * kScanThreads;
        v[j] = 0;
        if (i < NE) {
          const int s = i / E;
          v[j] = __ldcg(a.ccnt + ((int64_t)s * nch + c) * E + (i - s * E));
        }
      }
#pragma unroll
      for (int j = 0; j < kColBatch; ++j) run[j] += v[j];
    }
#pragma unroll
    for (int j = 0; j < kColBatch; ++j) {
      const int i = i0 + j * kScanThreads;
      if (i < NE) {
        const int s = i / E;
        scnt[s * E1 + (i - s * E)] = run[j];
        a.cnt[i] = run[j];
      }
    }
  }
  __syncthreads();

  // C[s][d] = sum over d's experts of cnt[s][.]
  for (int i = tid; i < N * N; i += kScanThreads) {
    const int s = i / N, d = i - s * N;
    int c = 0;
    for (int l = 0; l < L; ++l) c += scnt[s * E1 + d * L + l];
    sC[s * N1 + d] = c;
    a.C[i] = c;
  }
  // soff[s][e]: scan over experts, one warp per source rank
  for (int s = warp; s < N; s += kWarps) {
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? scnt[s * E1 + e] : 0;
      const int incl = warp_inclusive_scan(v, lane);
      if (e < E) a.soff[(int64_t)s * E + e] = carry + incl - v;
      carry += __shfl_sync(kFull, incl, 31);
    }
  }
  // eoff[d][l][s] (= eoff[e][s]) and ecnt[e]: scan over source ranks, one warp per expert
  for (int e = warp; e < E; e += kWarps) {
    int carry = 0;
    for (int s0 = 0; s0 < N; s0 += 32) {
      const int s = s0 + lane;
      const int v = s < N ? scnt[s * E1 + e] : 0;
      const int incl = warp_inclusive_scan(v, lane);
      if (s < N) a.eoff[(int64_t)e * N + s] = carry + incl - v;
      carry += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) {
      a.ecnt[e] = carry;
      if (carry > g.cap) set_status(a.status, kBitCapacity);
    }
  }
  __syncthreads();
  // roff[d][s] and rtot[d]: scan of C[.][d] over source ranks, one warp per destination
  for (int d = warp; d < N; d += kWarps) {
    int carry = 0;
    for (int s0 = 0; s0 < N; s0 += 32) {
      const int s = s0 + lane;
      const int v = s < N ? sC[s * N1 + d] : 0;
      const int incl = warp_inclusive_scan(v, lane);
      if (s < N) a.roff[d * N + s] = carry + incl - v;
      carry += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) {
      a.rtot[d] = carry;
      if ((int64_t)carry > g.RB) set_status(a.status, kBitRecvBound);
    }
  }
}

// One CTA per (chunk c, source rank s): the chunk's 256 pairs in (t,k) order, one per
// thread. Writes each pair's rank among the chunk's pairs of the same expert into pos[]
// (-1 for an id outside [0,E)) and the chunk's count of every expert into ccnt[s][c][.].
__global__ void __launch_bounds__(kChunk) k_route_count(Geo g, LayoutArgs a) {
  extern __shared__ int32_t wtab[];  // [kChunk/32][E]: per-warp counts, then exclusive offsets
  constexpr int kW = kChunk / 32;
  const int E = g.E;
  const int c = blockIdx.x, s = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kW * E; i += kChunk) wtab[i] = 0;
  const int64_t pl = (int64_t)c * kChunk + tid;
  const bool in = pl < g.TR;
  const int64_t q = (int64_t)s * g.TR + pl;
  pdl_wait();
  const int e = in ? __ldg(a.idx + q) : -1;
  const bool ok = in && e >= 0 && e < E;
  if (in && !ok) set_status(a.status, kBitExpertRange);
  const unsigned peers = __match_any_sync(kFull, ok ? e : -1);
  const int lrank = __popc(peers & ((1u << lane) - 1u));
  __syncthreads();
  if (ok && lrank == 0) wtab[warp * E + e] = __popc(peers);
  __syncthreads();
  int32_t* crow = a.ccnt + ((int64_t)s * a.nch + c) * E;
  for (int ee = tid; ee < E; ee += kChunk) {
    int r = 0;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const int v = wtab[w * E + ee];
      wtab[w * E + ee] = r;
      r += v;
    }
    crow[ee] = r;
  }
  __syncthreads();
  if (in) a.pos[q] = ok ? wtab[warp * E + e] + lrank : -1;
  pdl_trigger();
}

// One CTA: per-rank totals and every scan (see layout_scans).
__global__ void __launch_bounds__(kScanThreads, 1) k_route_scan(Geo g, LayoutArgs a) {
  extern __shared__ int32_t sm[];
  pdl_wait();
  layout_scans(g, a, sm);
  pdl_trigger();
}

// Per-pair placements from ranks and scans, plus -1 padding of the inverse maps.
// Blocks [0, pair_blocks) take one pair per thread; the next E blocks pad one expert's
// grouped rows each; the remaining blocks pad kRecvPadRows receive rows of a rank each.
constexpr int kMapThreads = 256;
constexpr int kRecvPadRows = 8192;

__global__ void __launch_bounds__(kMapThreads) k_layout_maps(Geo g, LayoutArgs a, int pair_blocks) {
  pdl_wait();
  const int b = blockIdx.x;
  if (b < pair_blocks) {
    const int q = b * kMapThreads + threadIdx.x;
    if (q < g.P) {
      const int e = __ldg(a.idx + q);
      if (e < 0 || e >= g.E) {  // pos[q] is already -1
        a.rrow[q] = -1;
        a.slot[q] = -1;
        a.gsend[q] = -1;
        a.grecv[q] = -1;
        a.gslot[q] = -1;
      } else {
        const int TR = (int)g.TR;
        const int s = q / TR;
        const int c = (q - s * TR) / kChunk;
        const int32_t* col = a.ccnt + (int64_t)s * a.nch * g.E + e;
        int rk = a.pos[q];
        for (int cc = 0; cc < c; ++cc) rk += col[(int64_t)cc * g.E];   // pairs of e in earlier chunks
        const int d = e / g.L;
        const int p = a.soff[s * g.E + e] + rk;
        const int rr = a.roff[d * g.N + s] + p - a.soff[s * g.E + d * g.L];
        const int sl = a.eoff[e * g.N + s] + rk;
        a.pos[q] = p;
        a.rrow[q] = rr;
        a.gsend[q] = s * TR + p;
        a.grecv[q] = (int32_t)(d * g.RB + rr);
        a.recv_src[d * g.RB + rr] = q;
        if (sl < g.cap) {
          a.slot[q] = sl;
          a.gslot[q] = e * g.cap + sl;
          a.slot_src[(int64_t)e * g.cap + sl] = q;
        } else {
          a.slot[q] = -1;
          a.gslot[q] = -1;
        }
      }
    }
  } else if (b < pair_blocks + g.E) {
    const int e = b - pair_blocks;
    int32_t* row = a.slot_src + (int64_t)e * g.cap;
    for (int j = a.ecnt[e] + threadIdx.x; j < g.cap; j += kMapThreads) row[j] = -1;
  } else {
    const int per_rank = (int)((g.RB + kRecvPadRows - 1) / kRecvPadRows);
    const int r = b - pair_blocks - g.E;
    const int d = r / per_rank;
    const int64_t lo = (int64_t)(r - d * per_rank) * kRecvPadRows;
    const int64_t hi = lo + kRecvPadRows < g.RB ? lo + kRecvPadRows : g.RB;
    int32_t* row = a.recv_src + (int64_t)d * g.RB;
    const int64_t from = a.rtot[d] > lo ? a.rtot[d] : lo;
    for (int64_t j = from + threadIdx.x; j < hi; j += kMapThreads) row[j] = -1;
  }
  pdl_trigger();
}

std::atomic<int> g_scan_smem[64];

}  // namespace

int layout_chunks(const Geo& g) { return (int)((g.TR + kChunk - 1) / kChunk); }

size_t layout_smem_bytes(const Geo& g) {
  return 4 * ((size_t)g.N * (g.E | 1) + (size_t)g.N * (g.N | 1));
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
  a.ccnt = lay->scratch;
  a.nch = layout_chunks(g);

  const size_t scan_smem = layout_smem_bytes(g);
  if (scan_smem + 1024 > (size_t)c.smem_optin) return cudaErrorInvalidValue;
  cudaError_t e = ensure_dyn_smem(k_route_scan, c.device, scan_smem, g_scan_smem);
  if (e != cudaSuccess) return e;
  if (a.nch > 0) {
    LaunchScope ls(c, MOE_K_ROUTE_COUNT);
    e = launch_kernel(k_route_count, dim3(a.nch, g.N), dim3(kChunk), (size_t)4 * (kChunk / 32) * g.E, c, g, a);
    if (e != cudaSuccess) return e;
  }
  {
    LaunchScope ls(c, MOE_K_ROUTE_SCAN);
    e = launch_kernel(k_route_scan, dim3(1), dim3(kScanThreads), scan_smem, c, g, a);
  }
  if (e != cudaSuccess) return e;
  const int pair_blocks = (int)((g.P + kMapThreads - 1) / kMapThreads);
  {
    LaunchScope ls(c, MOE_K_LAYOUT_MAPS);
    const int64_t pad_blocks = (int64_t)g.N * ((g.RB + kRecvPadRows - 1) / kRecvPadRows);
    e = launch_kernel(k_layout_maps, dim3((unsigned)(pair_blocks + g.E + pad_blocks)), dim3(kMapThreads), 0, c, g, a,
                      pair_blocks);
  }
  return e;
}

}  // namespace moe
