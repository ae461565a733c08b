// Row movers: every dispatch/combine step that moves whole token rows.
//
// "Enabling trillion-parameter models on AWS EFA" (Perplexity), section "Dispatch and
// combine": the sender shuffles tokens into its send buffer so that one RDMA write per
// peer suffices (pack); the TransferEngine "scatter" of section "MoE routing with
// TransferEngine" copies slices of one source buffer to offsets on every peer (here a
// device copy into the peer's receive region); the receiver shuffles received tokens into
// the grouped-GEMM input; combine runs the same moves backwards.
//
// Two implementations, same results:
//  - k_move_tma: kIssuers independent issuer warps per CTA. Lane 0 of each warp runs its
//    own ring of S row stages in shared memory: a 1-D TMA bulk copy (cp.async.bulk
//    global->shared, completion counted on the stage's mbarrier) brings a row in, and bulk
//    stores shared->global write it to its destination(s): R of them for pack, codes +
//    scales for the fp8 receive shuffle. A row is read from HBM once however many
//    destinations it has. While the oldest stage drains, S-1 loads stay in flight, and the
//    indices of the next row to load are fetched one refill ahead.
//  - k_move_ldg: one warp per unit with 16-byte (or, for rows that are not 16-byte
//    multiples, 4-byte) register loads and stores; also the path for misaligned shapes.
// Units are (token, column chunk) for pack and (token, expert) pairs for the rest; units
// are dealt round-robin over all issuers / warps, so skewed routing spreads evenly.
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kPackPrefetch = 16;  // send rows of a token kept in registers by the planner

struct MoveArgs {
  const uint8_t* src;
  uint8_t* dst;
  uint8_t* dst2;
  uint8_t* dst3;          // pack-all: the grouped rows
  const int32_t* gsend;   // per pair: global send row, or -1
  const int32_t* grecv;   // per pair: global receive row, or -1
  const int32_t* gslot;   // per pair: global grouped row, or -1
  const int32_t* fan;     // pack: per pair, the destination row (gsend, or grecv for direct push)
  int t0, nt;             // token range [t0, t0 + nt) of every rank that the move covers
  int32_t* status;
  int64_t units;
  uint32_t stage_bytes;
  int stages;
  int chunks;             // pack: column chunks per token row (1 elsewhere)
  uint32_t chunk_bytes;   // pack: bytes per chunk (B / chunks)
  // Rank window filter of the receive-side moves (mode 2): a pair is moved only when its
  // destination rank (its global receive row / fd_rows, or for the identity copy its grouped
  // row / fd_rows) is in [fd_lo, fd_lo + fd_n).
  int64_t fd_rows;
  int fd_lo, fd_n;
};

template <int MODE>
__device__ __forceinline__ bool dst_outside(const MoveArgs& a, int64_t row) {
  if (MODE != 2) return false;   // only rank-window launches filter (MODE 2)
  return (uint64_t)(row / a.fd_rows - a.fd_lo) >= (uint64_t)a.fd_n;
}

struct Plan {
  const uint8_t* src;
  uint8_t* dst;
  uint8_t* dst2;
  int64_t tok;                 // pack: token index s*T+t
  int32_t coff;                // pack: byte offset of the chunk in the row
  int32_t p[kPackPrefetch];    // pack: global send rows of the token's pairs
};

// Bytes one unit moves per destination: one column chunk of a row (the whole row when
// the move is not chunked).
template <int KIND>
__host__ __device__ __forceinline__ uint32_t unit_bytes(const Geo& g, const MoveArgs& a) {
  return a.chunk_bytes;
}

// Launch modes, a compile-time choice: 0 the whole pass, 1 a token range [t0, t0 + nt) of
// every rank (micro-batches), 2 a rank window (buffers window-local; the receive-side moves
// skip pairs whose destination is outside the window). Modes 0 and 1 compile no filter.
//
// The global index (token for per = 1, pair for per = R) of item v: in mode 1, item v of the
// token range of every rank, items rank-major; otherwise v itself.
template <int MODE>
__device__ __forceinline__ int64_t range_item(const Geo& g, const MoveArgs& a, int64_t v, int per) {
  if (MODE != 1) return v;
  const int64_t span = (int64_t)a.nt * per;
  const int64_t s = v / span;
  return (s * g.T + a.t0) * per + (v - s * span);
}

// Fills `pl` for unit u; false when the unit moves nothing (bad expert id, dropped pair, or a
// destination outside the rank window).
template <int KIND, bool FP8, int MODE, bool REV>
__device__ __forceinline__ bool make_plan(const Geo& g, const MoveArgs& a, int64_t u, Plan& pl) {
  if (REV) u = a.units - 1 - u;
  const int64_t H2 = 2 * (int64_t)g.H;
  if (is_pack_kind(KIND)) {
    const int64_t tv = u / a.chunks;
    const int64_t tok = range_item<MODE>(g, a, tv, 1);
    pl.tok = tok;
    pl.coff = (int32_t)((u - tv * a.chunks) * a.chunk_bytes);
    pl.src = a.src + tok * g.B + pl.coff;
#pragma unroll
    for (int k = 0; k < kPackPrefetch; ++k) pl.p[k] = (k < g.R) ? __ldg(a.fan + tok * g.R + k) : -1;
    return true;
  }
  // Non-pack kinds: unit u is column chunk (u % chunks) of pair u / chunks.
  const int64_t cq = u / a.chunks;
  const int64_t coff = (u - cq * a.chunks) * (int64_t)a.chunk_bytes;
  u = range_item<MODE>(g, a, cq, g.R);
  if (KIND == kMoveScatter) {
    const int gs = __ldg(a.gsend + u);
    const int gr = __ldg(a.grecv + u);
    if (gs < 0 || dst_outside<MODE>(a, gr)) return false;
    pl.src = a.src + (int64_t)gs * g.B + coff;
    pl.dst = a.dst + (int64_t)gr * g.B + coff;
    return true;
  }
  if (KIND == kMoveCopyEx) {
    const int gl = __ldg(a.gslot + u);
    if (gl < 0 || dst_outside<MODE>(a, gl)) return false;
    pl.src = a.src + (int64_t)gl * H2 + coff;
    pl.dst = a.dst + (int64_t)gl * H2 + coff;
    return true;
  }
  const int gl = __ldg(a.gslot + u);
  const int gr = __ldg(a.grecv + u);
  if (KIND == kMoveUnpack) {
    if (gl < 0 || dst_outside<MODE>(a, gr)) return false;
    pl.src = a.src + (int64_t)gr * g.B + coff;
    if (FP8) {
      pl.dst = a.dst + (int64_t)gl * g.H;
      pl.dst2 = a.dst2 + (int64_t)gl * (g.H / 32);
    } else {
      pl.dst = a.dst + (int64_t)gl * g.B + coff;
    }
    return true;
  }
  if (KIND == kMoveCPack) {
    if (gl < 0 || dst_outside<MODE>(a, gr)) return false;
    pl.src = a.src + (int64_t)gl * H2 + coff;
    pl.dst = a.dst + (int64_t)gr * H2 + coff;
    return true;
  }
  if (KIND == kMoveCPush) {
    const int gs = __ldg(a.gsend + u);
    if (gl < 0) return false;
    pl.src = a.src + (int64_t)gl * H2 + coff;
    pl.dst = a.dst + (int64_t)gs * H2 + coff;
    return true;
  }
  // kMoveCScatter
  const int gs = __ldg(a.gsend + u);
  if (gl < 0 || dst_outside<MODE>(a, gr)) return false;
  pl.src = a.src + (int64_t)gr * H2 + coff;
  pl.dst = a.dst + (int64_t)gs * H2 + coff;
  return true;
}

// Bulk stores of one staged row to its destination(s); the caller commits the group.
template <int KIND, bool FP8>
__device__ __forceinline__ void issue_stores(const Geo& g, const MoveArgs& a, const Plan& pl, const uint8_t* stage,
                                             uint32_t bytes) {
  if (is_pack_kind(KIND)) {
    if (KIND != kMovePackAllPush) {   // pack-all with direct push has no send rows
#pragma unroll
      for (int k = 0; k < kPackPrefetch; ++k)
        if (pl.p[k] >= 0) bulk_s2g(a.dst + (int64_t)pl.p[k] * g.B + pl.coff, stage, bytes);
      for (int k = kPackPrefetch; k < g.R; ++k) {
        const int p = __ldg(a.fan + pl.tok * g.R + k);
        if (p >= 0) bulk_s2g(a.dst + (int64_t)p * g.B + pl.coff, stage, bytes);
      }
    }
    if (is_pack_all_kind(KIND)) {   // the receive rows, and the grouped rows of the kept pairs
      for (int k = 0; k < g.R; ++k) {
        const int64_t q = pl.tok * g.R + k;
        if (__ldg(a.gsend + q) < 0) continue;
        bulk_s2g(a.dst2 + (int64_t)__ldg(a.grecv + q) * g.B + pl.coff, stage, bytes);
        const int gl = __ldg(a.gslot + q);
        if (gl >= 0) bulk_s2g(a.dst3 + (int64_t)gl * g.B + pl.coff, stage, bytes);
      }
    }
  } else if (KIND == kMoveUnpack && FP8) {
    bulk_s2g(pl.dst, stage, (uint32_t)g.H);
    bulk_s2g(pl.dst2, stage + g.H, (uint32_t)(g.H / 32));
  } else {
    bulk_s2g(pl.dst, stage, bytes);
  }
}

constexpr int kIssuers = 4;          // issuer warps per CTA
constexpr int kMaxStages = 8;        // stages per issuer
constexpr int kTmaHeader = kIssuers * kMaxStages * (8 + 128);  // mbarriers + plan slots

// One stage's plan, kept in shared memory until its stores are issued.
struct StagePlan {
  uint8_t* dst;
  uint8_t* dst2;
  int64_t tok;
  int32_t coff;
  int32_t p[kPackPrefetch];
};

__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

template <int KIND, bool FP8, int MODE, bool REV>
__global__ void __launch_bounds__(kIssuers * 32) k_move_tma(Geo g, MoveArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem) + warp * kMaxStages;
  StagePlan* sp = reinterpret_cast<StagePlan*>(smem + kIssuers * kMaxStages * 8) + warp * kMaxStages;
  uint8_t* ring = smem + kTmaHeader + (size_t)warp * S * a.stage_bytes;
  if (lane < S) mbar_init(&bar[lane], 1);
  fence_mbar_init();
  __syncwarp();
  pdl_wait();
  if (lane == 0) {
    const int64_t G = (int64_t)gridDim.x * kIssuers;
    const int64_t gi = (int64_t)blockIdx.x * kIssuers + warp;
    const int64_t n = a.units > gi ? (a.units - gi + G - 1) / G : 0;   // this issuer's units
    const uint32_t bytes = unit_bytes<KIND>(g, a);
    uint32_t vbits = 0, pbits = 0;   // per stage: a load is in flight; the barrier's parity
    Plan pl;
    for (int k = 0; k < S && k < n; ++k) {
      const bool ok = make_plan<KIND, FP8, MODE, REV>(g, a, gi + k * G, pl);
      sp[k] = StagePlan{pl.dst, pl.dst2, pl.tok, pl.coff, {}};
      if (is_pack_kind(KIND))
        for (int r = 0; r < kPackPrefetch; ++r) sp[k].p[r] = pl.p[r];
      if (ok) {
        mbar_arrive_expect_tx(&bar[k], bytes);
        bulk_g2s(ring + (size_t)k * a.stage_bytes, pl.src, bytes, &bar[k]);
        vbits |= 1u << k;
      }
    }
    Plan nx;
    bool nx_ok = (S < n) && make_plan<KIND, FP8, MODE, REV>(g, a, gi + S * G, nx);
    for (int64_t j = 0; j < n; ++j) {
      const int k = (int)(j % S);
      bool stored = false;
      if (vbits & (1u << k)) {
        if (!mbar_wait_bounded(&bar[k], (pbits >> k) & 1u, a.status)) break;  // status has the timeout
        pbits ^= 1u << k;
        Plan cur;
        cur.dst = sp[k].dst;
        cur.dst2 = sp[k].dst2;
        cur.tok = sp[k].tok;
        cur.coff = sp[k].coff;
        if (is_pack_kind(KIND))
          for (int r = 0; r < kPackPrefetch; ++r) cur.p[r] = sp[k].p[r];
        issue_stores<KIND, FP8>(g, a, cur, ring + (size_t)k * a.stage_bytes, bytes);
        bulk_commit();
        stored = true;
      }
      // Refill the stage of unit j-1 with unit j-1+S once its stores have read it.
      const int64_t jr = j - 1 + S;
      if (j >= 1 && jr < n) {
        const int kp = (int)((j - 1) % S);
        if (stored)
          bulk_wait_read_1();
        else
          bulk_wait_read_all();
        vbits &= ~(1u << kp);
        sp[kp] = StagePlan{nx.dst, nx.dst2, nx.tok, nx.coff, {}};
        if (is_pack_kind(KIND))
          for (int r = 0; r < kPackPrefetch; ++r) sp[kp].p[r] = nx.p[r];
        if (nx_ok) {
          mbar_arrive_expect_tx(&bar[kp], bytes);
          bulk_g2s(ring + (size_t)kp * a.stage_bytes, nx.src, bytes, &bar[kp]);
          vbits |= 1u << kp;
        }
        nx_ok = (jr + 1 < n) && make_plan<KIND, FP8, MODE, REV>(g, a, gi + (jr + 1) * G, nx);
      }
    }
    pdl_trigger();
    bulk_wait_all();
  }
}

template <typename V>
__device__ __forceinline__ V ld_vec(const uint8_t* p);
template <>
__device__ __forceinline__ uint4 ld_vec<uint4>(const uint8_t* p) {
  return ld_stream16(p);
}
template <>
__device__ __forceinline__ uint32_t ld_vec<uint32_t>(const uint8_t* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}
__device__ __forceinline__ void st_vec(uint8_t* p, const uint4& v) { st16(p, v); }
__device__ __forceinline__ void st_vec(uint8_t* p, const uint32_t& v) { *reinterpret_cast<uint32_t*>(p) = v; }

// The pack-all move keeps three destination rows per pair and takes 89 registers (two CTAs
// of 256 threads per SM): measured on GB300, bounding it to three CTAs per SM (79 registers)
// was 1-3% slower on every workload, and finer column chunks changed nothing.
template <int KIND, bool FP8, typename V, int MODE, bool REV>
__device__ __forceinline__ void move_ldg(const Geo& g, const MoveArgs& a) {
  constexpr int U = 8;
  constexpr int W = (int)sizeof(V);
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t nel = unit_bytes<KIND>(g, a) / W;
  const int64_t split = (KIND == kMoveUnpack && FP8) ? g.H / W : nel;
  pdl_wait();
  if (is_pack_kind(KIND)) {
    // Pack: lane k holds the destination row of the token's pair k and broadcasts it by
    // shuffle, so a warp keeps only its U loaded vectors live while it writes R copies.
    for (int64_t u0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u0 < a.units; u0 += nwarps) {
      const int64_t u = REV ? a.units - 1 - u0 : u0;
      const int64_t tv = u / a.chunks;
      const int64_t tok = range_item<MODE>(g, a, tv, 1);
      const int64_t coff = (u - tv * a.chunks) * (int64_t)a.chunk_bytes;
      const uint8_t* src = a.src + tok * g.B + coff;
      uint8_t* dst0 = KIND == kMovePackAllPush ? nullptr : a.dst + coff;
      const int32_t* fan = a.fan + tok * g.R;
      const int myp = lane < g.R ? __ldg(fan + lane) : -1;   // pairs 0..31 (R > 32: see below)
      // pack-all: the pair's receive row and grouped row (-1: dropped) as well. No later
      // kernel of the pass reads the receive rows (the combine gathers from the grouped
      // rows), so they go through L2 marked evict-first, which keeps the grouped rows and the
      // next micro-batch's rows there. Measured on GB300: direct-push steps 9-11% faster on
      // the bf16 workloads, default steps 1-4% (the send rows instead: the same; both: less).
      const uint64_t pol = is_pack_all_kind(KIND) ? l2_evict_first_policy() : 0;
      // Without direct push the grouped rows, which the combine of the same micro-batch reads,
      // are kept over other lines (1-1.5% faster default steps on GB300; with direct push,
      // where the combine runs from them alone, 2% slower, so not there).
      const uint64_t keep = KIND == kMovePackAll ? l2_evict_last_policy() : 0;
      const int myr = (is_pack_all_kind(KIND) && lane < g.R) ? __ldg(a.grecv + tok * g.R + lane) : -1;
      const int myl = (is_pack_all_kind(KIND) && lane < g.R) ? __ldg(a.gslot + tok * g.R + lane) : -1;
      // The trip count is the same for every lane: the shuffles below need the whole warp.
      for (int64_t b0 = 0; b0 < nel; b0 += 32 * U) {
        const int64_t v0 = b0 + lane;
        V r[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int64_t v = v0 + 32 * j;
          if (v < nel) r[j] = ld_vec<V>(src + v * W);
        }
#pragma unroll 1
        for (int k = 0; k < g.R; ++k) {
          const int p = k < 32 ? __shfl_sync(0xffffffffu, myp, k) : __ldg(fan + k);
          if (is_pack_all_kind(KIND)) {
            const int rr = k < 32 ? __shfl_sync(0xffffffffu, myr, k) : __ldg(a.grecv + tok * g.R + k);
            const int rl = k < 32 ? __shfl_sync(0xffffffffu, myl, k) : __ldg(a.gslot + tok * g.R + k);
            if (p < 0) continue;
            uint8_t* d = KIND == kMovePackAll ? dst0 + (int64_t)p * g.B : nullptr;   // no send rows with push
            uint8_t* d2 = a.dst2 + coff + (int64_t)rr * g.B;
            uint8_t* d3 = a.dst3 + coff + (int64_t)rl * g.B;
#pragma unroll
            for (int j = 0; j < U; ++j) {
              const int64_t v = v0 + 32 * j;
              if (v < nel) {
                if (KIND == kMovePackAll) st_vec(d + v * W, r[j]);   // no send rows with direct push
                if constexpr (sizeof(V) == 16)
                  st16_hint(d2 + v * W, r[j], pol);   // receive rows: nothing in the pass reads them
                else
                  st_vec(d2 + v * W, r[j]);
                if constexpr (KIND == kMovePackAll && sizeof(V) == 16) {
                  if (rl >= 0) st16_hint(d3 + v * W, r[j], keep);
                } else if (rl >= 0) {
                  st_vec(d3 + v * W, r[j]);
                }
              }
            }
            continue;
          }
          if (p < 0) continue;
          uint8_t* d = dst0 + (int64_t)p * g.B;
#pragma unroll
          for (int j = 0; j < U; ++j) {
            const int64_t v = v0 + 32 * j;
            if (v < nel) st_vec(d + v * W, r[j]);
          }
        }
      }
    }
    pdl_trigger();
    return;
  }
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < a.units; u += nwarps) {
    Plan pl;
    if (!make_plan<KIND, FP8, MODE, REV>(g, a, u, pl)) continue;
    for (int64_t v0 = lane; v0 < nel; v0 += 32 * U) {
      V r[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int64_t v = v0 + 32 * j;
        if (v < nel) r[j] = ld_vec<V>(pl.src + v * W);
      }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int64_t v = v0 + 32 * j;
        if (v >= nel) continue;
        if (KIND == kMoveUnpack && FP8) {
          if (v < split)
            st_vec(pl.dst + v * W, r[j]);
          else
            st_vec(pl.dst2 + (v - split) * W, r[j]);
        } else {
          st_vec(pl.dst + v * W, r[j]);
        }
      }
    }
  }
  pdl_trigger();
}

template <int KIND, bool FP8, typename V, int MODE, bool REV>
__global__ void __launch_bounds__(256) k_move_ldg(Geo g, MoveArgs a) {
  move_ldg<KIND, FP8, V, MODE, REV>(g, a);
}

// Direct-push pack-all held to two CTAs per SM: left to itself it takes 80 registers and
// three, and then leaves the concurrent combine of the previous micro-batch no room.
template <int KIND, bool FP8, typename V, int MODE, bool REV>
__global__ void __launch_bounds__(256, 2) k_move_ldg_b2(Geo g, MoveArgs a) {
  move_ldg<KIND, FP8, V, MODE, REV>(g, a);
}

template <int KIND, bool FP8, typename V, int MODE, bool REV>
constexpr auto ldg_kernel() {
  if constexpr (KIND == kMovePackAllPush)
    return k_move_ldg_b2<KIND, FP8, V, MODE, REV>;
  else
    return k_move_ldg<KIND, FP8, V, MODE, REV>;
}

// Largest dynamic shared memory limit set so far, per TMA instantiation and device.
std::atomic<int> g_tma_smem[10][2][3][2][64];

// Stages per issuer and CTAs per SM: as many CTAs as fit with 3 stages per issuer (at
// most 8 CTAs), then as many stages as the shared memory of each CTA holds (2..8). Each
// CTA also pays 1 KB of reserved shared memory and its mbarrier/plan header.
template <int KIND, bool FP8, int MODE, bool REV>
cudaError_t run_tma(const Geo& g, MoveArgs a, Ctx& c) {
  const uint32_t bytes = unit_bytes<KIND>(g, a);
  const int stage_bytes = (int)((bytes + 127u) & ~127u);
  const int per_cta_extra = 1024 + kTmaHeader;
  int cps = c.ctas_per_sm;
  if (cps <= 0) {
    cps = c.smem_per_sm / (kIssuers * 3 * stage_bytes + per_cta_extra);
    if (cps > 8) cps = 8;
    if (cps < 1) cps = 1;
  }
  while (cps > 1 && (c.smem_per_sm / cps - per_cta_extra) / (kIssuers * stage_bytes) < 2) --cps;
  int S = (c.smem_per_sm / cps - per_cta_extra) / (kIssuers * stage_bytes);
  const int S_blk = (c.smem_optin - kTmaHeader) / (kIssuers * stage_bytes);
  if (S > S_blk) S = S_blk;
  if (S > kMaxStages) S = kMaxStages;
  if (c.tma_stages > 0 && c.tma_stages < S) S = c.tma_stages;
  if (S < 2) return cudaErrorInvalidValue;
  const size_t smem = kTmaHeader + (size_t)kIssuers * S * stage_bytes;
  {
    cudaError_t e = ensure_dyn_smem(k_move_tma<KIND, FP8, MODE, REV>, c.device, smem,
                                    g_tma_smem[KIND][FP8 ? 1 : 0][MODE][REV ? 1 : 0]);
    if (e != cudaSuccess) return e;
  }
  a.stages = S;
  a.stage_bytes = stage_bytes;
  int64_t grid = (int64_t)c.num_sms * cps;
  const int64_t need = (a.units + kIssuers - 1) / kIssuers;
  if (grid > need) grid = need;
  return launch_kernel(k_move_tma<KIND, FP8, MODE, REV>, dim3((unsigned)grid), dim3(kIssuers * 32), smem, c, g, a);
}

template <int KIND, bool FP8, typename V, int MODE, bool REV>
cudaError_t run_ldg(const Geo& g, const MoveArgs& a, Ctx& c) {
  // Four waves of the CTAs the SMs hold at once (registers decide): warps that finish early
  // take later units, which measured faster on GB300 than one wave of grid-stride loops.
  static std::atomic<int> resident{0};
  int per_sm = resident.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ldg_kernel<KIND, FP8, V, MODE, REV>(), 256, 0) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    resident.store(per_sm, std::memory_order_relaxed);
  }
  per_sm = c.ctas_per_sm > 0 ? c.ctas_per_sm : 4 * per_sm;   // tuning override, else 4 waves
  int64_t blocks = (a.units + 7) / 8;
  const int64_t maxb = (int64_t)c.num_sms * per_sm;
  if (blocks > maxb) blocks = maxb;
  return launch_kernel(ldg_kernel<KIND, FP8, V, MODE, REV>(), dim3((unsigned)blocks), dim3(256), 0, c, g, a);
}

// True when two stages per issuer fit in one CTA's shared memory.
template <int KIND>
bool tma_fits(const Geo& g, const MoveArgs& a, const Ctx& c) {
  const int stage_bytes = (int)((unit_bytes<KIND>(g, a) + 127u) & ~127u);
  return (c.smem_optin - kTmaHeader) / (kIssuers * stage_bytes) >= 2;
}

// Default choice (measured on GB300): the TMA ring streams one-to-one moves at 95-98% of
// the copy bandwidth once every issuer has >= 40 rows (32K+ pairs), but its stages are held
// until the bulk stores have read them, which costs it the ramp on smaller problems and
// pack's R-fold stores; there the register mover, whose stores free their registers at
// issue, is as fast or faster.
template <int KIND>
bool tma_default(const MoveArgs& a, const Ctx& c) {
  if (is_pack_kind(KIND)) return false;
  return a.units / a.chunks >= 40LL * kIssuers * c.num_sms;
}

template <int KIND, bool FP8, int MODE, bool REV>
cudaError_t run_kind(const Geo& g, const MoveArgs& a, Ctx& c, bool row16) {
  const bool want_tma = (c.flags & MOE_FLAG_TMA_MOVER) ? true
                        : (c.flags & MOE_FLAG_LDG_MOVER) ? false
                                                          : tma_default<KIND>(a, c);
  if (row16 && want_tma && tma_fits<KIND>(g, a, c)) return run_tma<KIND, FP8, MODE, REV>(g, a, c);
  if (row16) return run_ldg<KIND, FP8, uint4, MODE, REV>(g, a, c);
  return run_ldg<KIND, FP8, uint32_t, MODE, REV>(g, a, c);
}

// Traversal direction. Each intermediate buffer of the pass is written by one move and read
// once by the next; a move that runs in the opposite unit order to its producer starts on
// the rows the producer wrote last, which are still in L2 (at 8K pairs of 14 KB rows,
// about 117 MB a buffer against 129 MB of L2). Pair-ordered moves therefore alternate:
// pack forward, scatter backward, unpack forward, identity expert forward, combine pack
// backward, combine scatter forward. With direct push the pack writes the receive rows
// forward, so the unpack and the identity expert run backward and the combine push forward.
// Only the order in which independent rows are copied changes, never a value.
template <int KIND, bool FP8, int MODE>
cudaError_t run_dir(const Geo& g, const MoveArgs& a, Ctx& c, bool row16) {
  if constexpr (KIND == kMoveUnpack || KIND == kMoveCopyEx) {
    if (c.flags & MOE_FLAG_DIRECT_PUSH) return run_kind<KIND, FP8, MODE, true>(g, a, c, row16);
    return run_kind<KIND, FP8, MODE, false>(g, a, c, row16);
  } else {
    return run_kind<KIND, FP8, MODE, KIND == kMoveScatter || KIND == kMoveCPack>(g, a, c, row16);
  }
}

}  // namespace

namespace {

template <int R>
cudaError_t run_move(MoveKind kind, const Geo& g, const MoveArgs& a, Ctx& c, bool fp8, bool rowB16) {
  if constexpr (R == 2) {   // the pack-all moves are whole-group moves only
    if (is_pack_all_kind(kind)) return cudaErrorInvalidValue;
  }
  switch (kind) {
    case kMovePack:
      return run_dir<kMovePack, false, R>(g, a, c, rowB16);
    case kMoveScatter:
      return run_dir<kMoveScatter, false, R>(g, a, c, rowB16);
    case kMoveUnpack:
      return fp8 ? run_dir<kMoveUnpack, true, R>(g, a, c, rowB16) : run_dir<kMoveUnpack, false, R>(g, a, c, rowB16);
    case kMoveCPack:
      return run_dir<kMoveCPack, false, R>(g, a, c, true);
    case kMoveCScatter:
      return run_dir<kMoveCScatter, false, R>(g, a, c, true);
    case kMoveCopyEx:
      return run_dir<kMoveCopyEx, false, R>(g, a, c, true);
    case kMovePackPush:
      return run_dir<kMovePackPush, false, R>(g, a, c, rowB16);
    case kMoveCPush:
      return run_dir<kMoveCPush, false, R>(g, a, c, true);
    case kMovePackAll:
      if constexpr (R != 2) return run_dir<kMovePackAll, false, R>(g, a, c, rowB16);
      break;
    case kMovePackAllPush:
      if constexpr (R != 2) return run_dir<kMovePackAllPush, false, R>(g, a, c, rowB16);
      break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace

namespace {

// A move on the rank window [lo, lo + n) of a layout (see moe_layout_t): buffers are
// window-local. Moves that start from the window's tokens or pairs (pack, scatter, combine
// scatter) run over the window's contiguous token / pair range as a group of n ranks, their
// index arrays advanced to it; moves into the window's receive or grouped rows (unpack,
// combine pack, identity copy) visit every pair and skip those whose destination is outside
// the window. Scatter and combine scatter move only the pairs whose both ends are in the
// window; the caller moves the others between windows.
cudaError_t launch_move_window(MoveKind kind, const Geo& g, const moe_layout_t* lay, MoveArgs a, Ctx& c) {
  const int64_t lo = c.win_lo, n = (int64_t)c.win_hi - c.win_lo;
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  const int64_t H2 = 2 * (int64_t)g.H, LC = (int64_t)g.L * g.cap;
  const int64_t q0 = lo * g.TR;   // the window's first pair
  Geo gw = g;                     // the window as a group of n ranks (source-side moves)
  gw.N = (int)n;
  gw.P = n * g.TR;
  const uint8_t* src = a.src;
  uint8_t* dst = a.dst;
  uint8_t* dst2 = a.dst2;
  const Geo* gp = &g;
  switch (kind) {
    case kMovePack:   // window tokens -> window send rows
      gp = &gw;
      a.fan = lay->gsend + q0;
      a.dst = rebase(dst, q0 * g.B);
      break;
    case kMoveScatter:   // window pairs with a window destination: send rows -> receive rows
      gp = &gw;
      a.gsend = lay->gsend + q0;
      a.grecv = lay->grecv + q0;
      a.gslot = lay->gslot + q0;
      a.src = rebase(src, q0 * g.B);
      a.dst = rebase(dst, lo * g.RB * g.B);
      a.fd_rows = g.RB;
      break;
    case kMoveUnpack:   // every pair with a window destination: receive rows -> grouped rows
      a.src = rebase(src, lo * g.RB * g.B);
      a.dst = rebase(dst, lo * LC * (fp8 ? (int64_t)g.H : g.B));
      a.dst2 = rebase(dst2, lo * LC * (int64_t)(g.H / 32));
      a.fd_rows = g.RB;
      break;
    case kMoveCPack:   // every pair with a window destination: grouped outputs -> receive order
      a.src = rebase(src, lo * LC * H2);
      a.dst = rebase(dst, lo * g.RB * H2);
      a.fd_rows = g.RB;
      break;
    case kMoveCScatter:   // window pairs with a window destination: receive order -> sources
      gp = &gw;
      a.gsend = lay->gsend + q0;
      a.grecv = lay->grecv + q0;
      a.gslot = lay->gslot + q0;
      a.src = rebase(src, lo * g.RB * H2);
      a.dst = rebase(dst, q0 * H2);
      a.fd_rows = g.RB;
      break;
    case kMoveCopyEx:   // the window's grouped rows (bf16 identity expert into another buffer)
      a.src = rebase(src, lo * LC * H2);
      a.dst = rebase(dst, lo * LC * H2);
      a.fd_rows = LC;
      break;
    default:   // direct push writes other ranks' rows: the whole group only
      return cudaErrorInvalidValue;
  }
  a.fd_lo = (int)lo;
  a.fd_n = (int)n;
  const Geo& gg = *gp;
  if (kind == kMovePack) {
    a.units = gg.N * (int64_t)gg.T * a.chunks;   // chunks were chosen for the whole group
  } else {
    a.units = gg.P * a.chunks;
  }
  if (a.units == 0) return cudaSuccess;
  static const moe_kernel_id ids[] = {MOE_K_PACK,         MOE_K_SCATTER,         MOE_K_UNPACK,
                                      MOE_K_COMBINE_PACK, MOE_K_COMBINE_SCATTER, MOE_K_EXPERT};
  LaunchScope ls(c, ids[kind]);
  return run_move<2>(kind, gg, a, c, fp8, (g.B % 16) == 0);
}

}  // namespace

cudaError_t launch_move(MoveKind kind, const Geo& g, const moe_layout_t* lay, const void* src, void* dst, void* dst2,
                        Ctx& c, void* dst3) {
  return launch_move_range(kind, g, lay, src, dst, dst2, 0, g.T, c, dst3);
}

cudaError_t launch_move_range(MoveKind kind, const Geo& g, const moe_layout_t* lay, const void* src, void* dst,
                              void* dst2, int t0, int nt, Ctx& c, void* dst3) {
  MoveArgs a;
  a.src = static_cast<const uint8_t*>(src);
  a.dst = static_cast<uint8_t*>(dst);
  a.dst2 = static_cast<uint8_t*>(dst2);
  a.dst3 = static_cast<uint8_t*>(dst3);
  a.gsend = lay->gsend;
  a.grecv = lay->grecv;
  a.gslot = lay->gslot;
  a.fan = kind == kMovePackPush ? lay->grecv : lay->gsend;
  a.t0 = 0;
  a.nt = g.T;
  a.status = lay->status;
  a.stages = 0;
  a.stage_bytes = 0;
  a.chunks = 1;
  a.chunk_bytes = (uint32_t)g.B;
  a.fd_rows = 0;
  a.fd_lo = 0;
  a.fd_n = 0;
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  const bool rowB16 = (g.B % 16) == 0;  // bf16 rows always; fp8 rows when H % 512 == 0
  if (is_pack_kind(kind)) {
    // Split token rows into column chunks (16-byte multiples, at most 8 per row) of at least
    // 2 KB, or 1.5 KB while this launch has fewer than ~16 units per SM: smaller units
    // balance the warps better (measured: 3.5 KB chunks of 14 KB rows and 2 KB chunks of 8 KB
    // rows were the fastest for whole passes; 1.75 KB chunks of 14 KB rows for micro-batches
    // of 256 tokens, while 1 KB chunks of 8 KB rows lost 1.6%) and give small batches
    // parallelism beyond one unit per token.
    const int64_t tokens = (int64_t)g.N * nt;   // of this launch
    while (a.chunks < 8 && g.B % (16 * 2 * a.chunks) == 0) {
      const int64_t half = g.B / (2 * a.chunks);
      if (half >= 2048 || (half >= 1536 && tokens * a.chunks < 16LL * c.num_sms))
        a.chunks *= 2;
      else
        break;
    }
    a.chunk_bytes = (uint32_t)(g.B / a.chunks);
    a.units = tokens * a.chunks;
  } else {
    // One-to-one moves: halve rows of >= 12 KB when this launch has fewer than 32 pairs per
    // issuer slot of the TMA ring, so that each issuer keeps more (smaller) rows in flight
    // (measured on micro-batches of 2048 pairs: 14 KB rows 6% faster halved, 8 KB rows 4.5%
    // slower). The fp8 receive split (codes | scales) is never chunked.
    const int64_t rowb = (kind == kMoveScatter || kind == kMoveUnpack) ? g.B : 2 * (int64_t)g.H;
    const bool splittable = !(kind == kMoveUnpack && fp8) && rowb >= 12288 && rowb % 32 == 0;
    const int64_t pairs = nt == g.T ? g.P : (int64_t)g.N * nt * g.R;   // of this launch
    if (splittable && pairs < 32LL * 4 * c.num_sms) a.chunks = 2;
    a.chunk_bytes = (uint32_t)(rowb / a.chunks);
    a.units = g.P * a.chunks;
  }
  if (windowed(g, c)) return nt == g.T ? launch_move_window(kind, g, lay, a, c) : cudaErrorInvalidValue;
  if (nt != g.T) {   // a token range of every rank: its tokens, or its pairs
    a.t0 = t0;
    a.nt = nt;
    a.units = (int64_t)g.N * nt * (is_pack_kind(kind) ? 1 : g.R) * a.chunks;
  }
  if (a.units == 0) return cudaSuccess;
  static const moe_kernel_id ids[] = {MOE_K_PACK,         MOE_K_SCATTER,         MOE_K_UNPACK,
                                      MOE_K_COMBINE_PACK, MOE_K_COMBINE_SCATTER, MOE_K_EXPERT,
                                      MOE_K_PACK_PUSH,    MOE_K_COMBINE_PUSH,    MOE_K_DISPATCH_FUSED,
                                      MOE_K_DISPATCH_FUSED};
  LaunchScope ls(c, ids[kind]);
  return nt != g.T ? run_move<1>(kind, g, a, c, fp8, rowB16) : run_move<0>(kind, g, a, c, fp8, rowB16);
}

}  // namespace moe
