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
//  - the last chunk CTA of each source rank to finish (a completion counter, no waiting)
//    sums that rank's chunk counts into cnt[s][.]; a grid of independent scan CTAs (one
//    per source row, per 32-expert column tile and per destination) then runs every
//    scan, and the maps kernel adds a pair's earlier-chunk counts to its chunk-local rank.
//    The counting kernel's last CTA per rank also turns the rank's chunk counts into
//    exclusive prefixes over its chunks. The three kernels chain with programmatic
//    dependent launch.
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kChunk = 256;          // pairs per histogram CTA (= its threads)
constexpr unsigned kFull = 0xffffffffu;

struct LayoutArgs {
  const int32_t* idx;
  int32_t *cnt, *C, *soff, *roff, *rtot, *ecnt, *eoff;
  int32_t *pos, *rrow, *slot, *slot_src, *recv_src;
  int32_t *gsend, *grecv, *gslot;
  int32_t* status;
  int32_t* ccnt;    // [N][nch][E]: per-chunk counts, then exclusive prefixes over the chunks
  int32_t* done;    // [N]: chunk CTAs of each rank that have finished (reset by the last one)
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

// The scans, as one grid of independent CTAs (kScanThreads threads each), by role:
//   [0, N)              row CTA s:    soff[s][.] = exclusive scan of cnt[s][.] over experts,
//                                     C[s][d] = sum of cnt[s][.] over d's experts;
//   [N, N + ceil(E/32)) column CTA:   for 32 experts e, eoff[e][.] = exclusive scan of
//                                     cnt[.][e] over source ranks, ecnt[e] = its total;
//   [.., + N)           dest CTA d:   roff[d][.] = exclusive scan of C[.][d] over source
//                                     ranks, rtot[d] = its total.
// Every CTA reads the per-rank totals cnt[][] written by the counting kernel; lanes run
// along the scanned dimension, so global stores are coalesced.
constexpr int kScanThreads = 256;
// Shared staging of the scan CTAs: a 64 x 33 tile (column CTAs), a row of E counts (row
// CTAs), or E counts plus N sums (destination CTAs). The entry points accept E <= 1536,
// and N <= E since E is a multiple of N.
constexpr int kScanMaxE = 1536;
constexpr int kScanTileInts = 2 * kScanMaxE;
static_assert(kScanTileInts >= 64 * 33, "the column tile fits");

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int incl = warp_inclusive_scan(v, lane);
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int t = lane < kScanThreads / 32 ? warp_tot[lane] : 0;
    const int ti = warp_inclusive_scan(t, lane);
    if (lane < kScanThreads / 32) warp_tot[lane] = ti - t;
    if (lane == 31) warp_tot[kScanThreads / 32] = ti;
  }
  __syncthreads();
  total = warp_tot[kScanThreads / 32];
  const int r = warp_tot[warp] + incl - v;
  __syncthreads();
  return r;
}

// cnt[i], or 0 when there are no tokens (no counting kernel ran; the row CTAs write the 0s).
__device__ __forceinline__ int cnt_at(const LayoutArgs& a, int64_t i) {
  return a.nch > 0 ? __ldcg(a.cnt + i) : 0;
}

__global__ void __launch_bounds__(kScanThreads) k_route_scan(Geo g, LayoutArgs a) {
  __shared__ int warp_tot[kScanThreads / 32 + 1];
  __shared__ int tile[kScanTileInts];
  const int N = g.N, E = g.E, L = g.L;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_col = (E + 31) / 32;
  const int b = blockIdx.x;
  pdl_wait();
  if (b < N) {
    // ---- row CTA: soff[s][.] and C[s][.]
    const int s = b;
    const int k = (E + kScanThreads - 1) / kScanThreads;      // experts per thread, <= 6
    const int e0 = tid * k;
    int vals[6];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < 6; ++j) {
      vals[j] = (j < k && e0 + j < E) ? cnt_at(a, (int64_t)s * E + e0 + j) : 0;
      sum += vals[j];
    }
    int* row = tile;   // the row's counts (read once, summed from shared memory), E <= kScanMaxE
#pragma unroll
    for (int j = 0; j < 6; ++j)
      if (j < k && e0 + j < E) row[e0 + j] = vals[j];
    int total;
    int run = block_exclusive_scan(sum, warp_tot, total);   // its barriers also publish row[]
#pragma unroll
    for (int j = 0; j < 6; ++j)
      if (j < k && e0 + j < E) {
        a.soff[(int64_t)s * E + e0 + j] = run;
        run += vals[j];
        if (a.nch == 0) a.cnt[(int64_t)s * E + e0 + j] = 0;
      }
    for (int d = warp; d < N; d += kScanThreads / 32) {   // C[s][d]: lanes along d's experts
      int c = 0;
      for (int l = lane; l < L; l += 32) c += row[d * L + l];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
      if (lane == 0) a.C[s * N + d] = c;
    }
  } else if (b < N + n_col) {
    // ---- column CTA: eoff[e][.] and ecnt[e] for experts e0 .. e0+31. Tiles of 64 ranks
    // x 32 experts are staged in shared memory (coalesced rows, odd stride); warp w scans
    // experts w, w+8, w+16, w+24 down the ranks, carrying their totals across tiles.
    const int e0 = (b - N) * 32;
    int carry[4] = {0, 0, 0, 0};
    for (int s0 = 0; s0 < N; s0 += 64) {
      const int ns = N - s0 < 64 ? N - s0 : 64;
      for (int i = tid; i < ns * 32; i += kScanThreads) {
        const int ss = i >> 5, ee = i & 31;
        tile[ss * 33 + ee] = (e0 + ee < E) ? cnt_at(a, (int64_t)(s0 + ss) * E + e0 + ee) : 0;
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ee = warp + 8 * j, e = e0 + ee;
        for (int sc = 0; sc < ns; sc += 32) {
          const int sl = sc + lane;
          const int v = sl < ns ? tile[sl * 33 + ee] : 0;
          const int incl = warp_inclusive_scan(v, lane);
          if (sl < ns && e < E) a.eoff[(int64_t)e * N + s0 + sl] = carry[j] + incl - v;
          carry[j] += __shfl_sync(kFull, incl, 31);
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + warp + 8 * j;
      if (lane == 0 && e < E) {
        a.ecnt[e] = carry[j];
        if (carry[j] > g.cap) set_status(a.status, kBitCapacity);
      }
    }
  } else {
    // ---- destination CTA: roff[d][.] and rtot[d]
    const int d = b - N - n_col;
    // cnt[s][d*L + l] for every s and l (N * L = E values) in one round of loads, then the
    // per-source sums from shared memory.
    int* col = tile;                 // col[s * L + l]: E values
    int* cd = tile + E;              // cd[s] = C[s][d]: E + N <= 2 * kScanMaxE
    for (int i = tid; i < E; i += kScanThreads) {
      const int s = i / L, l = i - s * L;
      col[i] = cnt_at(a, (int64_t)s * E + d * L + l);
    }
    __syncthreads();
    for (int s = warp; s < N; s += kScanThreads / 32) {
      int c = 0;
      for (int l = lane; l < L; l += 32) c += col[s * L + l];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
      if (lane == 0) cd[s] = c;
    }
    __syncthreads();
    if (warp == 0) {
      int carry = 0;
      for (int sc = 0; sc < N; sc += 32) {
        const int s = sc + lane;
        const int v = s < N ? cd[s] : 0;
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
  pdl_trigger();
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

  // The last chunk CTA of rank s to finish sums the rank's chunk rows into cnt[s][.]
  // (completion counter per rank; no CTA waits for another).
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = (atomicAdd(a.done + s, 1) == a.nch - 1);
  __syncthreads();
  if (is_last) {
    // cnt[s][.] = sum over the chunks; each chunk's row becomes the exclusive prefix over
    // the rank's earlier chunks, so a pair's rank is its chunk-local rank plus one load.
    __threadfence();
    int32_t* base = a.ccnt + (int64_t)s * a.nch * E;
    for (int ee = tid; ee < E; ee += kChunk) {
      int r = 0;
      int cc = 0;
      for (; cc + 4 <= a.nch; cc += 4) {   // four independent loads in flight
        const int v0 = __ldcg(base + (int64_t)cc * E + ee), v1 = __ldcg(base + (int64_t)(cc + 1) * E + ee);
        const int v2 = __ldcg(base + (int64_t)(cc + 2) * E + ee), v3 = __ldcg(base + (int64_t)(cc + 3) * E + ee);
        base[(int64_t)cc * E + ee] = r;
        base[(int64_t)(cc + 1) * E + ee] = r + v0;
        base[(int64_t)(cc + 2) * E + ee] = r + v0 + v1;
        base[(int64_t)(cc + 3) * E + ee] = r + v0 + v1 + v2;
        r += v0 + v1 + v2 + v3;
      }
      for (; cc < a.nch; ++cc) {
        const int v = __ldcg(base + (int64_t)cc * E + ee);
        base[(int64_t)cc * E + ee] = r;
        r += v;
      }
      a.cnt[(int64_t)s * E + ee] = r;
    }
    if (tid == 0) a.done[s] = 0;  // ready for the next call
  }
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
        // chunk-local rank + pairs of e in the rank's earlier chunks (the counting kernel
        // left the chunk table as exclusive prefixes over the chunks)
        const int rk = a.pos[q] + a.ccnt[((int64_t)s * a.nch + c) * g.E + e];
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


}  // namespace

int layout_chunks(const Geo& g) { return (int)((g.TR + kChunk - 1) / kChunk); }

int64_t layout_scratch_done_offset(const Geo& g) { return (int64_t)g.N * layout_chunks(g) * g.E; }

int64_t layout_scratch_tgroups_offset(const Geo& g) { return layout_scratch_done_offset(g) + g.N; }

int64_t layout_scratch_arrive_offset(const Geo& g) { return layout_scratch_tgroups_offset(g) + (int64_t)g.N * g.T; }


std::atomic<int> g_count_smem[64];   // per device: dynamic shared memory k_route_count is set up for

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
  a.nch = layout_chunks(g);
  a.ccnt = lay->scratch;
  a.done = lay->scratch + layout_scratch_done_offset(g);

  cudaError_t e = cudaSuccess;
  if (a.nch > 0) {
    const size_t smem = (size_t)4 * (kChunk / 32) * g.E;   // per-warp tables: 48 KB at E = 1536
    if ((e = ensure_dyn_smem(k_route_count, c.device, smem, g_count_smem)) != cudaSuccess) return e;
    LaunchScope ls(c, MOE_K_ROUTE_COUNT);
    e = launch_kernel(k_route_count, dim3(a.nch, g.N), dim3(kChunk), smem, c, g, a);
    if (e != cudaSuccess) return e;
  }
  {
    LaunchScope ls(c, MOE_K_ROUTE_SCAN);
    e = launch_kernel(k_route_scan, dim3(2 * g.N + (g.E + 31) / 32), dim3(kScanThreads), 0, c, g, a);
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
