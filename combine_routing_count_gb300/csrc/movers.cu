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
//  - k_move_tma: one warp per CTA; lane j owns pipeline stage j (one row of shared memory
//    and one mbarrier). Each lane plans its next row's addresses while its current row
//    streams in through a 1-D TMA bulk copy (cp.async.bulk global->shared, completion on
//    the mbarrier), then issues bulk stores shared->global to the row's destination(s):
//    R of them for pack, codes + scales for the fp8 receive shuffle. A row is read from
//    HBM once however many destinations it has.
//  - k_move_ldg: one warp per row with 16-byte (or, for rows that are not 16-byte
//    multiples, 4-byte) register loads and stores; also the path for misaligned shapes.
// Units are tokens (pack) or (token, expert) pairs (everything else); each CTA takes a
// contiguous range of units, so skewed routing spreads evenly over the grid.
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kPackPrefetch = 16;  // send rows of a token kept in registers by the planner

struct MoveArgs {
  const uint8_t* src;
  uint8_t* dst;
  uint8_t* dst2;
  const int32_t* gsend;   // per pair: global send row, or -1
  const int32_t* grecv;   // per pair: global receive row, or -1
  const int32_t* gslot;   // per pair: global grouped row, or -1
  int32_t* status;
  int64_t units;
  uint32_t stage_bytes;
  int stages;
};

struct Plan {
  const uint8_t* src;
  uint8_t* dst;
  uint8_t* dst2;
  int64_t tok;                 // pack: token index s*T+t
  int32_t p[kPackPrefetch];    // pack: global send rows of the token's pairs
};

template <int KIND>
__host__ __device__ __forceinline__ uint32_t load_bytes(const Geo& g) {
  if (KIND == kMovePack || KIND == kMoveScatter || KIND == kMoveUnpack) return (uint32_t)g.B;
  return (uint32_t)(2 * g.H);
}

// Fills `pl` for unit u; false when the unit moves nothing (bad expert id or dropped pair).
template <int KIND, bool FP8>
__device__ __forceinline__ bool make_plan(const Geo& g, const MoveArgs& a, int64_t u, Plan& pl) {
  const int64_t H2 = 2 * (int64_t)g.H;
  if (KIND == kMovePack) {
    pl.tok = u;
    pl.src = a.src + u * g.B;
#pragma unroll
    for (int k = 0; k < kPackPrefetch; ++k) pl.p[k] = (k < g.R) ? __ldg(a.gsend + u * g.R + k) : -1;
    return true;
  }
  if (KIND == kMoveScatter) {
    const int gs = __ldg(a.gsend + u);
    const int gr = __ldg(a.grecv + u);
    if (gs < 0) return false;
    pl.src = a.src + (int64_t)gs * g.B;
    pl.dst = a.dst + (int64_t)gr * g.B;
    return true;
  }
  if (KIND == kMoveCopyEx) {
    const int gl = __ldg(a.gslot + u);
    if (gl < 0) return false;
    pl.src = a.src + (int64_t)gl * H2;
    pl.dst = a.dst + (int64_t)gl * H2;
    return true;
  }
  const int gl = __ldg(a.gslot + u);
  const int gr = __ldg(a.grecv + u);
  if (KIND == kMoveUnpack) {
    if (gl < 0) return false;
    pl.src = a.src + (int64_t)gr * g.B;
    if (FP8) {
      pl.dst = a.dst + (int64_t)gl * g.H;
      pl.dst2 = a.dst2 + (int64_t)gl * (g.H / 32);
    } else {
      pl.dst = a.dst + (int64_t)gl * g.B;
    }
    return true;
  }
  if (KIND == kMoveCPack) {
    if (gl < 0) return false;
    pl.src = a.src + (int64_t)gl * H2;
    pl.dst = a.dst + (int64_t)gr * H2;
    return true;
  }
  // kMoveCScatter
  const int gs = __ldg(a.gsend + u);
  if (gl < 0) return false;
  pl.src = a.src + (int64_t)gr * H2;
  pl.dst = a.dst + (int64_t)gs * H2;
  return true;
}

// Bulk stores of one staged row to its destination(s); the caller commits the group.
template <int KIND, bool FP8>
__device__ __forceinline__ void issue_stores(const Geo& g, const MoveArgs& a, const Plan& pl, const uint8_t* stage,
                                             uint32_t bytes) {
  if (KIND == kMovePack) {
#pragma unroll
    for (int k = 0; k < kPackPrefetch; ++k)
      if (pl.p[k] >= 0) bulk_s2g(a.dst + (int64_t)pl.p[k] * g.B, stage, bytes);
    for (int k = kPackPrefetch; k < g.R; ++k) {
      const int p = __ldg(a.gsend + pl.tok * g.R + k);
      if (p >= 0) bulk_s2g(a.dst + (int64_t)p * g.B, stage, bytes);
    }
  } else if (KIND == kMoveUnpack && FP8) {
    bulk_s2g(pl.dst, stage, (uint32_t)g.H);
    bulk_s2g(pl.dst2, stage + g.H, (uint32_t)(g.H / 32));
  } else {
    bulk_s2g(pl.dst, stage, bytes);
  }
}

template <int KIND, bool FP8>
__global__ void __launch_bounds__(32) k_move_tma(Geo g, MoveArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  const int lane = threadIdx.x;
  const int S = a.stages;
  uint8_t* stage = smem + 256 + (size_t)lane * a.stage_bytes;
  if (lane < S) mbar_init(&bar[lane], 1);
  fence_mbar_init();
  __syncwarp();

  const int64_t u0 = a.units * blockIdx.x / gridDim.x;
  const int64_t u1 = a.units * (blockIdx.x + 1) / gridDim.x;
  const uint32_t bytes = load_bytes<KIND>(g);
  uint32_t phase = 0;
  bool alive = lane < S;

  Plan nxt;
  bool has_nxt = alive && (u0 + lane < u1) && make_plan<KIND, FP8>(g, a, u0 + lane, nxt);
  for (int64_t base = u0; base < u1; base += S) {
    const Plan cur = nxt;
    const bool has = has_nxt && alive;
    bulk_wait_read_all();  // the stage's previous stores have read it
    if (has) {
      mbar_arrive_expect_tx(&bar[lane], bytes);
      bulk_g2s(stage, cur.src, bytes, &bar[lane]);
    }
    const int64_t un = base + S + lane;
    has_nxt = alive && (un < u1) && make_plan<KIND, FP8>(g, a, un, nxt);
    if (has) {
      if (mbar_wait_bounded(&bar[lane], phase, a.status)) {
        phase ^= 1u;
        issue_stores<KIND, FP8>(g, a, cur, stage, bytes);
        bulk_commit();
      } else {
        alive = false;  // status carries the timeout; stop issuing
      }
    }
  }
  bulk_wait_all();
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

template <int KIND, bool FP8, typename V>
__global__ void __launch_bounds__(256) k_move_ldg(Geo g, MoveArgs a) {
  constexpr int U = 8;
  constexpr int W = (int)sizeof(V);
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t nel = load_bytes<KIND>(g) / W;
  const int64_t split = (KIND == kMoveUnpack && FP8) ? g.H / W : nel;
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < a.units; u += nwarps) {
    Plan pl;
    if (!make_plan<KIND, FP8>(g, a, u, pl)) continue;
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
        if (KIND == kMovePack) {
#pragma unroll
          for (int k = 0; k < kPackPrefetch; ++k)
            if (pl.p[k] >= 0) st_vec(a.dst + (int64_t)pl.p[k] * g.B + v * W, r[j]);
          for (int k = kPackPrefetch; k < g.R; ++k) {
            const int p = __ldg(a.gsend + pl.tok * g.R + k);
            if (p >= 0) st_vec(a.dst + (int64_t)p * g.B + v * W, r[j]);
          }
        } else if (KIND == kMoveUnpack && FP8) {
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
}

// Largest dynamic shared memory limit set so far, per TMA instantiation and device.
std::atomic<int> g_tma_smem[6][2][64];

// Stages per CTA and CTAs per SM: two CTAs per SM when each still holds >= 8 row stages,
// else one CTA with as many stages as shared memory allows (at most 32, one per lane).
// Each CTA also pays 1 KB of reserved shared memory and 256 bytes of mbarriers.
template <int KIND, bool FP8>
cudaError_t run_tma(const Geo& g, MoveArgs a, Ctx& c) {
  const uint32_t row = load_bytes<KIND>(g);
  const int stage_bytes = (int)((row + 127u) & ~127u);
  const int per_cta_extra = 1024 + 256;
  int cps = c.ctas_per_sm;
  if (cps <= 0) cps = ((c.smem_per_sm / 2 - per_cta_extra) / stage_bytes >= 8) ? 2 : 1;
  int S = (c.smem_per_sm / cps - per_cta_extra) / stage_bytes;
  const int S_blk = (c.smem_optin - 256) / stage_bytes;
  if (S > S_blk) S = S_blk;
  if (S > 32) S = 32;
  if (c.tma_stages > 0 && c.tma_stages < S) S = c.tma_stages;
  if (S < 1) return cudaErrorInvalidValue;
  const size_t smem = 256 + (size_t)S * stage_bytes;
  {
    cudaError_t e = ensure_dyn_smem(k_move_tma<KIND, FP8>, c.device, smem, g_tma_smem[KIND][FP8 ? 1 : 0]);
    if (e != cudaSuccess) return e;
  }
  a.stages = S;
  a.stage_bytes = stage_bytes;
  int64_t grid = (int64_t)c.num_sms * cps;
  if (grid > a.units) grid = a.units;
  k_move_tma<KIND, FP8><<<(unsigned)grid, 32, smem, c.stream>>>(g, a);
  return cudaGetLastError();
}

template <int KIND, bool FP8, typename V>
cudaError_t run_ldg(const Geo& g, const MoveArgs& a, Ctx& c) {
  int64_t blocks = (a.units + 7) / 8;
  const int64_t maxb = (int64_t)c.num_sms * 4;
  if (blocks > maxb) blocks = maxb;
  k_move_ldg<KIND, FP8, V><<<(unsigned)blocks, 256, 0, c.stream>>>(g, a);
  return cudaGetLastError();
}

template <int KIND, bool FP8>
cudaError_t run_kind(const Geo& g, const MoveArgs& a, Ctx& c, bool row16) {
  if (row16 && !(c.flags & MOE_FLAG_LDG_MOVER)) return run_tma<KIND, FP8>(g, a, c);
  if (row16) return run_ldg<KIND, FP8, uint4>(g, a, c);
  return run_ldg<KIND, FP8, uint32_t>(g, a, c);
}

}  // namespace

cudaError_t launch_move(MoveKind kind, const Geo& g, const moe_layout_t* lay, const void* src, void* dst, void* dst2,
                        Ctx& c) {
  MoveArgs a;
  a.src = static_cast<const uint8_t*>(src);
  a.dst = static_cast<uint8_t*>(dst);
  a.dst2 = static_cast<uint8_t*>(dst2);
  a.gsend = lay->gsend;
  a.grecv = lay->grecv;
  a.gslot = lay->gslot;
  a.status = lay->status;
  a.units = (kind == kMovePack) ? (int64_t)g.N * g.T : g.P;
  a.stages = 0;
  a.stage_bytes = 0;
  if (a.units == 0) return cudaSuccess;
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  const bool rowB16 = (g.B % 16) == 0;  // bf16 rows always; fp8 rows when H % 512 == 0
  static const moe_kernel_id ids[] = {MOE_K_PACK, MOE_K_SCATTER, MOE_K_UNPACK, MOE_K_COMBINE_PACK,
                                      MOE_K_COMBINE_SCATTER, MOE_K_EXPERT};
  LaunchScope ls(c, ids[kind]);
  switch (kind) {
    case kMovePack:
      return run_kind<kMovePack, false>(g, a, c, rowB16);
    case kMoveScatter:
      return run_kind<kMoveScatter, false>(g, a, c, rowB16);
    case kMoveUnpack:
      return fp8 ? run_kind<kMoveUnpack, true>(g, a, c, rowB16) : run_kind<kMoveUnpack, false>(g, a, c, rowB16);
    case kMoveCPack:
      return run_kind<kMoveCPack, false>(g, a, c, true);
    case kMoveCScatter:
      return run_kind<kMoveCScatter, false>(g, a, c, true);
    case kMoveCopyEx:
      return run_kind<kMoveCopyEx, false>(g, a, c, true);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
