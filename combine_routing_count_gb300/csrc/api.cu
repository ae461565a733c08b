// C ABI of libmoe_ep (declared in include/moe_ep.h): argument checks, workspace carving, the
// kernel sequence of each dispatch/combine step and the token batches of the batched passes.
// No memory allocation, no synchronisation (except moe_status_sync), no fallback: every step
// runs in this library's kernels.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>
#include <utility>
#include <vector>

#include "internal.h"

namespace moe {

std::atomic<uint64_t> g_launches{0};

namespace {

// Reads n16 16-byte words so that whatever L2 held before is evicted (dirty lines are
// written back during this kernel). The xor of everything read decides a store that never
// happens in practice, which keeps the loads from being dropped.
__global__ void __launch_bounds__(256) k_l2_flush(uint4* buf, int64_t n16) {
  uint4 acc = make_uint4(0, 0, 0, 0);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 v = buf[i];   // plain load: normal L2 allocation, so it displaces what was cached
    acc.x ^= v.x;
    acc.y ^= v.y;
    acc.z ^= v.z;
    acc.w ^= v.w;
  }
  if (acc.x == 0x6d6f6531u && acc.y == 0x6c326675u && acc.z == 0x73686f6eu && acc.w == 0x21212121u) buf[0] = acc;
}

}  // namespace

cudaError_t launch_l2_flush(const moe_prof_t* prof, cudaStream_t stream) {
  if (!prof->flush || prof->flush_bytes < 16 || (prof->flush_bytes & 15u)) return cudaSuccess;
  const int64_t n16 = (int64_t)(prof->flush_bytes / 16);
  int64_t blocks = (n16 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  k_l2_flush<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<uint4*>(prof->flush), n16);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxHostBatches = 24;
constexpr int kMaxMicroBatches = 32;
constexpr int64_t kMaxE = 1536;
constexpr int64_t kMaxN = 2048;           // ranks: the scan CTAs stage up to 64*33 per-rank values
constexpr int64_t kI32 = 0x7fffffff;

struct DevInfo {
  int num_sms = 0;
  int smem_optin = 0;
  int smem_per_sm = 0;
  int l2_bytes = 0;
  // The library's second stream (default priority), which takes the odd token batches of
  // the batched passes, and the mapped host pass's fork and join events; created on first
  // use and kept until exit. fork_mu makes a fork (record, then wait) atomic.
  cudaStream_t aux = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex fork_mu;
  // The copy-engine pipeline of the host pass: a stream for host-to-device and one for
  // device-to-host copies, with their events; p_lay and p_aux fork the second stream from
  // the caller's and join it back in every batched pass. pipe_mu makes one pass's enqueue
  // atomic.
  bool pipe_ready = false;
  cudaStream_t cin = nullptr, cout = nullptr;
  cudaEvent_t p_start = nullptr, p_idx = nullptr, p_done = nullptr, p_lay = nullptr, p_aux = nullptr;
  cudaEvent_t p_in[kMaxHostBatches] = {}, p_dev[kMaxHostBatches] = {};
  std::mutex pipe_mu;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

DevInfo* aux_for(int dev) {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& di = g_dev[dev];
  if (!di.aux) {
    // Default priority: batches on the two streams interleave their CTAs fairly (measured
    // with the second stream at the highest priority, its batches ran ahead and the step
    // was 3-7% slower).
    cudaStream_t s = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
      if (f) cudaEventDestroy(f);
      cudaStreamDestroy(s);
      return nullptr;
    }
    di.aux = s;
    di.fork = f;
    di.join = j;
  }
  return &di;
}

DevInfo* pipe_for(int dev) {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& di = g_dev[dev];
  if (!di.pipe_ready) {
    auto ev = [](cudaEvent_t* e) { return *e || cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
    if ((!di.cin && cudaStreamCreateWithFlags(&di.cin, cudaStreamNonBlocking) != cudaSuccess) ||
        (!di.cout && cudaStreamCreateWithFlags(&di.cout, cudaStreamNonBlocking) != cudaSuccess) ||
        !ev(&di.p_start) || !ev(&di.p_idx) || !ev(&di.p_done) || !ev(&di.p_lay) || !ev(&di.p_aux))
      return nullptr;
    for (int i = 0; i < kMaxHostBatches; ++i)
      if (!ev(&di.p_in[i]) || !ev(&di.p_dev[i])) return nullptr;
    di.pipe_ready = true;
  }
  return &di;
}

// The auxiliary stream starts after everything issued so far on `main`.
bool fork_to(DevInfo* di, cudaStream_t main) {
  std::lock_guard<std::mutex> lk(di->fork_mu);
  return cudaEventRecord(di->fork, main) == cudaSuccess && cudaStreamWaitEvent(di->aux, di->fork, 0) == cudaSuccess;
}

// `main` continues after everything issued so far on the auxiliary stream.
bool join_from(DevInfo* di, cudaStream_t main) {
  return cudaEventRecord(di->join, di->aux) == cudaSuccess && cudaStreamWaitEvent(main, di->join, 0) == cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The device buffers a whole pass uses, present and 16-byte aligned (x, idx, w and out only
// when `with_io`); send and csend may be NULL with direct push, which never touches them.
bool pass_buffers_ok(const moe_buffers_t* b, uint32_t flags, bool fp8, bool with_io) {
  const bool push = (flags & MOE_FLAG_DIRECT_PUSH) != 0;
  auto ok = [](const void* p) { return p && aligned16(p); };
  if (with_io && (!ok(b->x) || !b->idx || !b->w || !ok(b->out))) return false;
  if (!push && (!ok(b->send) || !ok(b->csend))) return false;
  return ok(b->recv) && ok(b->expert_x) && ok(b->expert_y) && ok(b->crecv) && (!fp8 || ok(b->expert_scale));
}

}  // namespace

moe_status make_geo(const moe_dims* d, Geo& g) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->N < 1 || d->T < 0 || d->E < 1 || d->R < 1 || d->cap < 0 || d->H < 8) return MOE_ERR_INVALID_ARG;
  if (d->E % d->N != 0 || d->H % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (d->payload != MOE_PAYLOAD_BF16 && d->payload != MOE_PAYLOAD_FP8_E4M3_B128) return MOE_ERR_INVALID_ARG;
  if (d->payload == MOE_PAYLOAD_FP8_E4M3_B128 && d->H % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (d->E > kMaxE) return MOE_ERR_INVALID_ARG;
  const int64_t N = d->N, T = d->T, E = d->E, R = d->R, L = E / N;
  if (N > kMaxN) return MOE_ERR_INVALID_ARG;
  const int64_t cap = d->cap > 0 ? d->cap : N * T;  // 0 only when there are no tokens
  const int64_t RB = N * T * (R > L ? R : L);
  if (N * T * R > kI32 || N * RB > kI32 || E * cap > kI32 || N * T * (int64_t)d->H > (int64_t)1 << 40)
    return MOE_ERR_INVALID_ARG;
  g.N = d->N;
  g.T = d->T;
  g.H = d->H;
  g.E = d->E;
  g.R = d->R;
  g.L = (int)L;
  g.cap = (int)cap;
  g.payload = d->payload;
  g.TR = T * R;
  g.RB = RB;
  g.P = N * T * R;
  g.B = d->payload == MOE_PAYLOAD_FP8_E4M3_B128 ? (int64_t)d->H + 4 * (int64_t)(d->H / 128) : 2 * (int64_t)d->H;
  return MOE_OK;
}

moe_status make_ctx(const moe_layout_t* lay, void* stream, Ctx& c) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo& di = g_dev[dev];
    if (di.num_sms == 0) {
      if (cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&di.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
        di.num_sms = 0;
        return MOE_ERR_CUDA;
      }
    }
    c.num_sms = di.num_sms;
    c.smem_optin = di.smem_optin;
    c.smem_per_sm = di.smem_per_sm;
    c.l2_bytes = di.l2_bytes;
  }
  c.device = dev;
  c.stream = static_cast<cudaStream_t>(stream);
  c.prof = lay->prof;
  c.flags = lay->flags;
  c.tma_stages = lay->tma_stages;
  c.ctas_per_sm = lay->ctas_per_sm;
  c.status = lay->status;
  c.win_lo = lay->win_lo;
  c.win_hi = lay->win_hi;
  return MOE_OK;
}

bool layout_ok(const moe_layout_t* l) {
  if (!l) return false;
  const void* ps[] = {l->cnt, l->C,        l->soff,     l->roff,  l->rtot,  l->ecnt,  l->eoff,   l->pos,
                      l->rrow, l->slot,    l->slot_src, l->recv_src, l->gsend, l->grecv, l->gslot, l->status,
                      l->scratch};
  for (const void* p : ps)
    if (!p) return false;
  return true;
}

namespace {

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// The layout's rank window: valid (0, 0 or 0 <= lo < hi <= N) and whether it is smaller than
// the group.
bool window_valid(const Geo& g, const moe_layout_t* l) {
  if (l->win_lo == 0 && l->win_hi == 0) return true;
  return l->win_lo >= 0 && l->win_lo < l->win_hi && l->win_hi <= g.N;
}
bool window_partial(const Geo& g, const moe_layout_t* l) {
  return l->win_hi > 0 && !(l->win_lo == 0 && l->win_hi == g.N);
}
// Entry points that work on the whole group only.
bool whole_group(const Geo& g, const moe_layout_t* l) { return l && window_valid(g, l) && !window_partial(g, l); }
// Entry points that accept a rank window: valid, and no direct push with a partial one.
bool window_ok(const Geo& g, const moe_layout_t* l) {
  return l && window_valid(g, l) && !(window_partial(g, l) && (l->flags & MOE_FLAG_DIRECT_PUSH));
}

// Byte sizes of the workspace arrays, in carving order.
struct WsPlan {
  size_t n[18];
  size_t total;
};

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

WsPlan ws_plan(const Geo& g) {
  WsPlan w;
  const size_t N = g.N, E = g.E, P = g.P;
  const size_t sizes[] = {N * E,           // cnt
                          N * N,           // C
                          N * E,           // soff
                          N * N,           // roff
                          N,               // rtot
                          E,               // ecnt
                          E * N,           // eoff
                          P,               // pos
                          P,               // rrow
                          P,               // slot
                          E * g.cap,       // slot_src
                          N * g.RB,        // recv_src
                          P,               // gsend
                          P,               // grecv
                          P,               // gslot
                          16,              // status
                          (size_t)(layout_scratch_arrive_offset(g) + split_arrive_words(g)) + 16};  // scratch: chunk table,
                                                                      // counters, token groups, arrivals
  w.total = 0;
  for (int i = 0; i < 17; ++i) {
    w.n[i] = al256(4 * sizes[i]);
    w.total += w.n[i];
  }
  return w;
}

// The device address of pinned host memory p (cudaHostAlloc / cudaHostRegister), if the
// current device can address it.
bool host_mapped(const void* p, void** dev) {
  if (!p) return false;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();   // not a CUDA-known pointer: clear the error
    return false;
  }
  if (attr.type != cudaMemoryTypeHost || !attr.devicePointer) return false;
  *dev = attr.devicePointer;
  return true;
}

}  // namespace
}  // namespace moe

using namespace moe;

namespace moe {
namespace {

// Dispatch: the send rows of the token range [t0, t0 + nt) of every rank written to their
// owners' receive rows, then shuffled into the grouped rows.
cudaError_t dispatch_recv_range(const Geo& g, const moe_layout_t* lay, const void* send, void* recv, void* ex,
                                float* exs, int t0, int nt, Ctx& c) {
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  cudaError_t e = launch_move_range(kMoveScatter, g, lay, send, recv, nullptr, t0, nt, c);
  if (e == cudaSuccess) e = launch_move_range(kMoveUnpack, g, lay, recv, ex, fp8 ? exs : nullptr, t0, nt, c);
  return e;
}

// Combine: the expert output rows of the pairs of the token range [t0, t0 + nt) of every
// rank written in receive order, then back to their sources' combine rows.
cudaError_t combine_send_range(const Geo& g, const moe_layout_t* lay, const uint16_t* ey, uint16_t* csend,
                               uint16_t* crecv, int t0, int nt, Ctx& c) {
  cudaError_t e = launch_move_range(kMoveCPack, g, lay, ey, csend, nullptr, t0, nt, c);
  if (e == cudaSuccess) e = launch_move_range(kMoveCScatter, g, lay, csend, crecv, nullptr, t0, nt, c);
  return e;
}

// The whole pass in two token batches (tokens [0, T/2) and [T/2, T) of every rank) so that
// the host-link-bound kernels of one batch overlap the HBM-bound moves of the other: the
// pack of batch B (reading tokens over the host link) runs while batch A is scattered and
// unpacked on the second stream, and the reduce of batch A (writing the output over the
// link) runs there while batch B's combine send runs. The two batches touch disjoint rows
// of every buffer (also when the combine buffers alias the dispatch ones).
moe_status forward_two_batches(const Geo& g, const moe_dims* dims, const moe_layout_t* lay, const moe_buffers_t* b,
                               void* stream) {
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  if (!layout_ok(lay) || !pass_buffers_ok(b, lay->flags, fp8, true)) return MOE_ERR_INVALID_ARG;
  moe_status st = moe_layout(dims, b->idx, lay, stream);
  if (st != MOE_OK) return st;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  DevInfo* di = aux_for(c.device);
  if (!di) return MOE_ERR_CUDA;
  Ctx ca = c;
  ca.stream = di->aux;
  const int ta = g.T / 2, tb = g.T - ta;
  auto pack = [&](int t0, int nt) {
    return fp8 ? launch_quant_pack(g, lay->gsend, b->x, static_cast<uint8_t*>(b->send), c, t0, nt)
               : launch_move_range(kMovePack, g, lay, b->x, b->send, nullptr, t0, nt, c);
  };
  auto recv_half = [&](int t0, int nt, Ctx& cc) {
    return dispatch_recv_range(g, lay, b->send, b->recv, b->expert_x, b->expert_scale, t0, nt, cc);
  };
  auto combine_send_half = [&](int t0, int nt) {
    return combine_send_range(g, lay, b->expert_y, b->csend, b->crecv, t0, nt, c);
  };
  if (pack(0, ta) != cudaSuccess || !fork_to(di, c.stream) || pack(ta, tb) != cudaSuccess ||
      recv_half(0, ta, ca) != cudaSuccess || recv_half(ta, tb, c) != cudaSuccess || !join_from(di, c.stream))
    return MOE_ERR_CUDA;
  if ((st = moe_expert_identity(dims, lay, b->expert_x, b->expert_scale, b->expert_y, stream)) != MOE_OK) return st;
  if (combine_send_half(0, ta) != cudaSuccess || !fork_to(di, c.stream) ||
      launch_combine_reduce(g, lay, b->crecv, b->w, b->out, ca, 0, ta) != cudaSuccess ||
      combine_send_half(ta, tb) != cudaSuccess ||
      launch_combine_reduce(g, lay, b->crecv, b->w, b->out, c, ta, tb) != cudaSuccess || !join_from(di, c.stream))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// Dispatch send and recv of the token range [t0, t0 + nt) of every rank: its tokens'
// rows packed (quantised for fp8) and written to their owners, then shuffled into the
// grouped rows.
cudaError_t dispatch_range(const Geo& g, const moe_layout_t* lay, const void* x, void* send, void* recv, void* ex,
                           float* exs, int t0, int nt, Ctx& c) {
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  cudaError_t e;
  const bool push = (c.flags & MOE_FLAG_DIRECT_PUSH) != 0;
  if (!(c.flags & MOE_FLAG_SEPARATE_MOVES)) {
    // pack, write and shuffle in one kernel: each token row read (and quantised) once; direct
    // push writes no send rows
    void* snd = push ? nullptr : send;
    return fp8 ? launch_quant_dispatch_fused(g, lay, static_cast<const uint16_t*>(x), static_cast<uint8_t*>(snd),
                                             static_cast<uint8_t*>(recv), static_cast<uint8_t*>(ex), exs, c, t0, nt)
               : launch_move_range(push ? kMovePackAllPush : kMovePackAll, g, lay, x, snd, recv, t0, nt, c, ex);
  }
  if (push) {
    e = fp8 ? launch_quant_pack(g, lay->grecv, static_cast<const uint16_t*>(x), static_cast<uint8_t*>(recv), c, t0,
                                nt)
            : launch_move_range(kMovePackPush, g, lay, x, recv, nullptr, t0, nt, c);
  } else {
    e = fp8 ? launch_quant_pack(g, lay->gsend, static_cast<const uint16_t*>(x), static_cast<uint8_t*>(send), c, t0,
                                nt)
            : launch_move_range(kMovePack, g, lay, x, send, nullptr, t0, nt, c);
    if (e == cudaSuccess) e = dispatch_recv_range(g, lay, send, recv, ex, exs, t0, nt, c);
    return e;
  }
  if (e == cudaSuccess) e = launch_move_range(kMoveUnpack, g, lay, recv, ex, fp8 ? exs : nullptr, t0, nt, c);
  return e;
}

// Combine send and recv of the token range [t0, t0 + nt) of every rank: its pairs' expert
// rows written back to their sources, then each token's weighted sum.
cudaError_t combine_range(const Geo& g, const moe_layout_t* lay, const uint16_t* ey, uint16_t* csend, uint16_t* crecv,
                          const float* w, uint16_t* out, int t0, int nt, Ctx& c) {
  cudaError_t e;
  const bool push = (c.flags & MOE_FLAG_DIRECT_PUSH) != 0;
  if (!(c.flags & MOE_FLAG_SEPARATE_MOVES)) {
    // combine pack, write and weighted sum in one kernel: each expert output row read once;
    // direct push writes no receive-order rows
    return launch_combine_fused(g, lay, ey, push ? nullptr : csend, crecv, w, out, c, t0, nt);
  }
  if (push) {
    e = launch_move_range(kMoveCPush, g, lay, ey, crecv, nullptr, t0, nt, c);
  } else {
    e = combine_send_range(g, lay, ey, csend, crecv, t0, nt, c);
  }
  if (e == cudaSuccess) e = launch_combine_reduce(g, lay, crecv, w, out, c, t0, nt);
  return e;
}

// Device work of one token batch [t0, t0 + nt) of every rank: dispatch send and recv, the
// identity expert and the combine, each on only the batch's tokens or pairs.
cudaError_t batch_chain(const Geo& g, const moe_layout_t* lay, const moe_buffers_t* b, int t0, int nt, Ctx& c) {
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  cudaError_t e = dispatch_range(g, lay, b->x, b->send, b->recv, b->expert_x, b->expert_scale, t0, nt, c);
  if (e == cudaSuccess) {
    if (fp8)
      e = launch_dequant_fp8(g, lay, static_cast<const uint8_t*>(b->expert_x), b->expert_scale, b->expert_y, c, t0,
                             nt);
    else if (static_cast<const void*>(b->expert_y) != b->expert_x)
      e = launch_move_range(kMoveCopyEx, g, lay, b->expert_x, b->expert_y, nullptr, t0, nt, c);
  }
  if (e == cudaSuccess) e = combine_range(g, lay, b->expert_y, b->csend, b->crecv, b->w, b->out, t0, nt, c);
  return e;
}

// Token batches of the copy-engine pipeline: the caller's choice, else about twice the
// square root of the token rows' MB. The first copy in and the last copy out are what no
// device work hides (X / nb each, X the token bytes), while every batch adds its launches'
// ramp and tail (about c); X / nb + c * nb is least at nb = sqrt(X / c). The factor fitted
// the measured optimum with batches alternating over two streams on GB300 and one kernel per
// phase (7 batches at 14.7 MB, 16 at 59 and 67 MB, 3.6-4.2% faster than 11).
int host_batch_count(const Geo& g, const moe_layout_t* lay) {
  if (lay->flags & MOE_FLAG_ONE_BATCH) return 1;
  if (g.payload == MOE_PAYLOAD_FP8_E4M3_B128 && (lay->flags & MOE_FLAG_STAGED_QUANT)) return 1;
  int nb = lay->batches;
  if (nb <= 0) nb = (int)std::lround(2.0 * std::sqrt((double)g.N * g.T * g.H * 2 / 1e6));
  if (nb > kMaxHostBatches) nb = kMaxHostBatches;
  if (nb > g.T) nb = (int)g.T;
  return nb < 1 ? 1 : nb;
}

// First token of batch j of nb (j = nb gives T): equal batches, or, when `shaped` and there
// are three or more, a first and a last batch of half the others' tokens (weights 1, 2, ...,
// 2, 1), since the first batch's copy in and the last batch's copy out are the parts of a
// one-stream pipeline that no device work hides.
int batch_start(int T, int nb, int j, bool shaped) {
  if (!shaped || nb < 3) return (int)((int64_t)j * T / nb);
  const int64_t wsum = 2 * (int64_t)nb - 2, wj = j == 0 ? 0 : (j == nb ? wsum : 2 * (int64_t)j - 1);
  return (int)((wj * T + wsum / 2) / wsum);
}

// Micro-batches of moe_forward: the caller's choice (at most 32 and T), else, for bf16 rows,
// about one per 55 MB of dispatch and combine rows (pairs x (B + 2H) bytes; at most 20 and
// T), and one per 60 MB (at most 16) for fp8 rows, with direct push or with
// MOE_FLAG_SEPARATE_MOVES; one with MOE_FLAG_ONE_BATCH or staged fp8 quantisation. Measured
// on GB300 with batches alternating over two equal-priority streams, each the best of the
// counts tried. One kernel per phase with its L2 policies: 4 batches of 235 MB of rows (EP8,
// 4% faster than 8), 20 of 940 MB and 1074 MB (EP32 and EP16 1.5-2% faster than 16 and 24,
// 7% faster than 12 and 32): while a batch's rows stay in L2, its combine reads the grouped
// rows the dispatch wrote, and rewrites its send and receive rows, before they reach DRAM (the
// combine buffers may alias them). With direct push 4 of 235 MB and 16 of 940 MB and 1074 MB
// (3-7% faster than 12 and 20). fp8, whose identity expert writes a bf16 row per pair inside
// the chain: 6 of 356 MB (10% faster than one; 12 no faster than one). Separate kernels: 4
// batches of 235 MB (EP8, 18% faster than one), 6 of 356 MB (fp8 EP64, expert included,
// 16%), 16 of 940 MB and 1074 MB (EP32 28%, EP16 24%). Under ~35 MB one batch is fastest.
// Even counts keep both streams equally loaded (EP8: 3 and 5 batches lose to 4 and 6), so an
// odd count of 3 or more rounds up.
int forward_batch_count(const Geo& g, const moe_layout_t* lay) {
  if (lay->flags & MOE_FLAG_ONE_BATCH) return 1;
  if (g.payload == MOE_PAYLOAD_FP8_E4M3_B128 && (lay->flags & MOE_FLAG_STAGED_QUANT)) return 1;
  int nb = lay->batches;
  if (nb <= 0) {
    const bool fine = !(lay->flags & (MOE_FLAG_SEPARATE_MOVES | MOE_FLAG_DIRECT_PUSH)) &&
                      g.payload != MOE_PAYLOAD_FP8_E4M3_B128;
    nb = (int)std::min(fine ? 20L : 16L, std::lround((double)g.P * (g.B + 2.0 * g.H) / (fine ? 55e6 : 60e6)));
    if (nb >= 3 && (nb & 1)) ++nb;   // even: both streams end together
  }
  if (nb > kMaxMicroBatches) nb = kMaxMicroBatches;
  if (nb > g.T) nb = (int)g.T;
  return nb < 1 ? 1 : nb;
}

// Token batches of moe_dispatch and moe_combine (each phase on its own, the expert between
// them a barrier): the caller's choice (at most 32 and T), else none up to 2048 tokens of
// all ranks and about one per 8 tokens of a rank beyond (at most 16); one with
// MOE_FLAG_ONE_BATCH. Measured on GB300 with batches alternating over two streams and one
// kernel per phase: 1024 tokens never gained; 64 ranks x 32 tokens (fp8) 2.5% faster in one
// batch than in 4; 16 x 512 tokens 1.5% faster in 16 than in one, slower in 24.
int phase_batch_count(const Geo& g, const moe_layout_t* lay) {
  if (lay->flags & MOE_FLAG_ONE_BATCH) return 1;
  int nb = lay->batches;
  if (nb <= 0) nb = (int64_t)g.N * g.T <= 2048 ? 1 : (int)std::min<int64_t>(16, g.T / 8);
  if (nb > kMaxMicroBatches) nb = kMaxMicroBatches;
  if (nb > g.T) nb = (int)g.T;
  return nb < 1 ? 1 : nb;
}

// Runs fn(t0, nt, ctx) for nb equal token ranges of every rank, odd ones on the library's
// second stream (which starts after everything issued so far on the caller's
// stream); the caller's stream waits for it at the end. One range on the caller's stream
// when nb is 1.
template <typename F>
cudaError_t run_batches(const Geo& g, Ctx& c, int nb, F&& fn) {
  if (nb <= 1) return fn(0, (int)g.T, c);
  DevInfo* di = pipe_for(c.device);
  DevInfo* da = aux_for(c.device);
  if (!di || !da) return cudaErrorUnknown;
  Ctx ca = c;
  ca.stream = da->aux;
  std::lock_guard<std::mutex> lk(di->pipe_mu);
  cudaError_t e = cudaEventRecord(di->p_lay, c.stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ca.stream, di->p_lay, 0);
  for (int j = 0; j < nb && e == cudaSuccess; ++j) {
    const int t0 = batch_start(g.T, nb, j, false), nt = batch_start(g.T, nb, j + 1, false) - t0;
    if (nt > 0) e = fn(t0, nt, (j & 1) ? ca : c);
  }
  if (e == cudaSuccess) e = cudaEventRecord(di->p_aux, ca.stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(c.stream, di->p_aux, 0);
  return e;
}

// moe_forward as nb micro-batches (tokens [j*T/nb, (j+1)*T/nb) of every rank), each running
// dispatch, identity expert and combine on its own rows, odd ones on the library's
// second stream: a micro-batch's rows of each buffer are still in L2 when its next
// move reads them, and one batch's first kernels fill the SMs its neighbour's last kernels
// leave idle. The batches touch disjoint rows of every buffer. The caller's stream waits for
// the auxiliary stream before the call returns.
moe_status forward_batched(const Geo& g, const moe_dims* dims, const moe_layout_t* lay, const moe_buffers_t* b,
                           int nb, void* stream) {
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  if (!pass_buffers_ok(b, lay->flags, fp8, true)) return MOE_ERR_INVALID_ARG;
  moe_status st = moe_layout(dims, b->idx, lay, stream);
  if (st != MOE_OK) return st;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  return cuda_status(
      run_batches(g, c, nb, [&](int t0, int nt, Ctx& cj) { return batch_chain(g, lay, b, t0, nt, cj); }));
}

// The host pass as a pipeline over nb token batches (tokens [t0, t0 + nt) of every rank):
// the library's input stream copies idx, w and then each batch's token rows into the device
// buffers; the caller's stream runs the layout once idx is there, then each batch's device
// work once its rows are there; the output stream copies each finished batch's output rows
// back. Copy engines move the host bytes, so batch j's copies in and out overlap the device
// work of its neighbours without taking SMs from it. When an average batch's combine rows
// take at most 40% of L2, odd batches run on the library's second stream, so one batch's
// first kernels fill the SMs its neighbour's last kernels leave idle (the batches touch
// disjoint rows of every buffer); with larger batches the two would evict each other's
// rows from L2 between consecutive moves, and one stream measured faster (GB300: 29 and
// 47 MB batches 8-13% faster on two streams, 59 and 67 MB batches 2.5% slower). On one
// stream the first and last batches are half-size (3-4% faster there; 5% slower on two
// streams, whose overlapping batches prefer equal sizes). The caller's stream waits for
// the auxiliary stream and for the last copy before the call returns.
moe_status forward_host_pipelined(const Geo& g, const moe_dims* dims, const moe_layout_t* lay,
                                  const moe_buffers_t* b, const uint16_t* h_x, const int32_t* h_idx,
                                  const float* h_w, uint16_t* h_out, int nb, void* stream) {
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  if (!pass_buffers_ok(b, lay->flags, fp8, true)) return MOE_ERR_INVALID_ARG;
  Ctx c;
  moe_status st = make_ctx(lay, stream, c);
  if (st != MOE_OK) return st;
  DevInfo* di = pipe_for(c.device);
  DevInfo* da = aux_for(c.device);
  if (!di || !da) return MOE_ERR_CUDA;
  Ctx ca = c;
  ca.stream = da->aux;
  const double batch_rows = (double)g.N * g.T * g.R / nb;   // pairs of one batch
  const bool two_streams = batch_rows * 2.0 * g.H <= 0.4 * c.l2_bytes;
  const size_t pitch = (size_t)g.T * g.H * 2, pb = (size_t)g.P * 4;
  std::lock_guard<std::mutex> lk(di->pipe_mu);
  // Nothing is overwritten before the caller's earlier work on `stream` is done with it.
  if (cudaEventRecord(di->p_start, c.stream) != cudaSuccess || cudaStreamWaitEvent(di->cin, di->p_start, 0) ||
      cudaStreamWaitEvent(di->cout, di->p_start, 0))
    return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(b->idx, h_idx, pb, cudaMemcpyHostToDevice, di->cin) != cudaSuccess ||
      cudaEventRecord(di->p_idx, di->cin) != cudaSuccess ||
      cudaMemcpyAsync(b->w, h_w, pb, cudaMemcpyHostToDevice, di->cin) != cudaSuccess)
    return MOE_ERR_CUDA;
  for (int j = 0; j < nb; ++j) {
    const int t0 = batch_start(g.T, nb, j, !two_streams), nt = batch_start(g.T, nb, j + 1, !two_streams) - t0;
    if (nt == 0) continue;
    if (cudaMemcpy2DAsync(b->x + (size_t)t0 * g.H, pitch, h_x + (size_t)t0 * g.H, pitch, (size_t)nt * g.H * 2, g.N,
                          cudaMemcpyHostToDevice, di->cin) != cudaSuccess ||
        cudaEventRecord(di->p_in[j], di->cin) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (cudaStreamWaitEvent(c.stream, di->p_idx, 0) != cudaSuccess) return MOE_ERR_CUDA;
  if ((st = moe_layout(dims, b->idx, lay, stream)) != MOE_OK) return st;
  if (cudaEventRecord(di->p_lay, c.stream) != cudaSuccess || cudaStreamWaitEvent(ca.stream, di->p_lay, 0))
    return MOE_ERR_CUDA;
  for (int j = 0; j < nb; ++j) {
    const int t0 = batch_start(g.T, nb, j, !two_streams), nt = batch_start(g.T, nb, j + 1, !two_streams) - t0;
    if (nt == 0) continue;
    Ctx& cj = (two_streams && (j & 1)) ? ca : c;
    if (cudaStreamWaitEvent(cj.stream, di->p_in[j], 0) != cudaSuccess) return MOE_ERR_CUDA;
    if (batch_chain(g, lay, b, t0, nt, cj) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaEventRecord(di->p_dev[j], cj.stream) != cudaSuccess || cudaStreamWaitEvent(di->cout, di->p_dev[j], 0) ||
        cudaMemcpy2DAsync(h_out + (size_t)t0 * g.H, pitch, b->out + (size_t)t0 * g.H, pitch, (size_t)nt * g.H * 2,
                          g.N, cudaMemcpyDeviceToHost, di->cout) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (cudaEventRecord(di->p_aux, ca.stream) != cudaSuccess || cudaStreamWaitEvent(c.stream, di->p_aux, 0) ||
      cudaEventRecord(di->p_done, di->cout) != cudaSuccess || cudaStreamWaitEvent(c.stream, di->p_done, 0))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_check_dims(const moe_dims* dims) {
  Geo g;
  return make_geo(dims, g);
}

size_t moe_recv_capacity_rows(const moe_dims* dims) {
  Geo g;
  return make_geo(dims, g) == MOE_OK ? (size_t)g.RB : 0;
}

size_t moe_row_bytes(const moe_dims* dims) {
  Geo g;
  return make_geo(dims, g) == MOE_OK ? (size_t)g.B : 0;
}

int32_t moe_capacity(const moe_dims* dims) {
  Geo g;
  return make_geo(dims, g) == MOE_OK ? g.cap : 0;
}

size_t moe_layout_workspace_bytes(const moe_dims* dims) {
  Geo g;
  if (make_geo(dims, g) != MOE_OK) return 0;
  return ws_plan(g).total;
}

moe_status moe_layout_init(const moe_dims* dims, void* d_ws, size_t ws_bytes, moe_layout_t* out, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!out || !d_ws || (reinterpret_cast<uintptr_t>(d_ws) & 255u)) return MOE_ERR_INVALID_ARG;
  const WsPlan w = ws_plan(g);
  if (ws_bytes < w.total) return MOE_ERR_INVALID_ARG;
  uint8_t* p = static_cast<uint8_t*>(d_ws);
  int32_t** slots[] = {&out->cnt,  &out->C,        &out->soff,     &out->roff,  &out->rtot,  &out->ecnt,
                       &out->eoff, &out->pos,      &out->rrow,     &out->slot,  &out->slot_src, &out->recv_src,
                       &out->gsend, &out->grecv,   &out->gslot,    &out->status, &out->scratch};
  for (int i = 0; i < 17; ++i) {
    *slots[i] = reinterpret_cast<int32_t*>(p);
    p += w.n[i];
  }
  out->flags = 0;
  out->prof = nullptr;
  out->tma_stages = 0;
  out->ctas_per_sm = 0;
  out->batches = 0;
  out->win_lo = 0;
  out->win_hi = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(out->status, 0, 64, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(out->scratch + layout_scratch_done_offset(g), 0, 4 * (size_t)g.N, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemsetAsync(out->scratch + layout_scratch_arrive_offset(g), 0, 4 * ((size_t)split_arrive_words(g) + 2), s) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_layout(const moe_dims* dims, const int32_t* d_idx, const moe_layout_t* lay, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!layout_ok(lay) || (!d_idx && g.P > 0)) return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  return cuda_status(launch_layout(g, d_idx, lay, c));
}

moe_status moe_quantize_fp8_b128(const moe_dims* dims, const uint16_t* d_x, uint8_t* d_xq, const moe_layout_t* lay,
                                 void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!window_ok(g, lay)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  if (g.payload != MOE_PAYLOAD_FP8_E4M3_B128 || !layout_ok(lay) || !d_x || !d_xq || !aligned16(d_x) ||
      !aligned16(d_xq))
    return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  return cuda_status(launch_quant_fp8(g, d_x, d_xq, c));
}

moe_status moe_dispatch_send(const moe_dims* dims, const moe_layout_t* lay, const void* d_x, void* d_send,
                             void* d_recv, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!window_ok(g, lay)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  const bool push = lay && (lay->flags & MOE_FLAG_DIRECT_PUSH);
  if (!layout_ok(lay) || !d_x || !d_recv || !aligned16(d_x) || !aligned16(d_recv) ||
      (!push && (!d_send || !aligned16(d_send))))
    return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  if (push) return cuda_status(launch_move(kMovePackPush, g, lay, d_x, d_recv, nullptr, c));
  cudaError_t e = launch_move(kMovePack, g, lay, d_x, d_send, nullptr, c);
  if (e == cudaSuccess) e = launch_move(kMoveScatter, g, lay, d_send, d_recv, nullptr, c);
  return cuda_status(e);
}

moe_status moe_quantize_dispatch_send(const moe_dims* dims, const moe_layout_t* lay, const uint16_t* d_x,
                                      void* d_send, void* d_recv, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!window_ok(g, lay)) return MOE_ERR_INVALID_ARG;
  if (g.payload != MOE_PAYLOAD_FP8_E4M3_B128) return MOE_ERR_INVALID_ARG;
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  const bool push = lay && (lay->flags & MOE_FLAG_DIRECT_PUSH);
  if (!layout_ok(lay) || !d_x || !d_recv || !aligned16(d_x) || !aligned16(d_recv) ||
      (!push && (!d_send || !aligned16(d_send))))
    return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  if (push) return cuda_status(launch_quant_pack(g, lay->grecv, d_x, static_cast<uint8_t*>(d_recv), c));
  cudaError_t e = launch_quant_pack(g, lay->gsend, d_x, static_cast<uint8_t*>(d_send), c);
  if (e == cudaSuccess) e = launch_move(kMoveScatter, g, lay, d_send, d_recv, nullptr, c);
  return cuda_status(e);
}

moe_status moe_dispatch_split(const moe_dims* dims, const moe_layout_t* lay, const void* d_x, void* d_recv,
                              void* d_expert_x, float* d_expert_scale, int32_t withhold_source, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!whole_group(g, lay)) return MOE_ERR_INVALID_ARG;   // a rank window is not supported here
  if (withhold_source < -1 || withhold_source >= g.N) return MOE_ERR_INVALID_ARG;
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  if (!layout_ok(lay) || !d_x || !d_recv || !d_expert_x || !aligned16(d_x) || !aligned16(d_recv) ||
      !aligned16(d_expert_x) || g.R > 32)
    return MOE_ERR_INVALID_ARG;
  if (fp8 && (!d_expert_scale || !aligned16(d_expert_scale))) return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  return cuda_status(launch_dispatch_split(g, lay, d_x, d_recv, d_expert_x, fp8 ? d_expert_scale : nullptr,
                                           withhold_source, c));
}

size_t moe_dedicated_exchange_bytes(const moe_dims* dims) {
  Geo g;
  if (make_geo(dims, g) != MOE_OK) return 0;
  return dedicated_exchange_bytes(g);
}

moe_status moe_dispatch_dedicated(const moe_dims* dims, const moe_layout_t* lay, const int32_t* d_idx,
                                  const void* d_x, int32_t K, void* d_ded, void* d_xchg, void* d_main,
                                  void* d_expert_x, float* d_expert_scale, int32_t withhold_slice, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!whole_group(g, lay)) return MOE_ERR_INVALID_ARG;   // a rank window is not supported here
  if (K < 0 || withhold_slice < -1 || withhold_slice >= (int64_t)g.N * g.N || g.R > 32) return MOE_ERR_INVALID_ARG;
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  if (!layout_ok(lay) || !d_xchg || !aligned16(d_xchg)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)g.N * g.T > 0 &&
      (!d_idx || !d_x || !d_main || !d_expert_x || !aligned16(d_x) || !aligned16(d_main) ||
       !aligned16(d_expert_x) || (K > 0 && (!d_ded || !aligned16(d_ded))) ||
       (fp8 && (!d_expert_scale || !aligned16(d_expert_scale)))))
    return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  return cuda_status(launch_dispatch_dedicated(g, lay, d_idx, d_x, K, d_ded, d_xchg, d_main, d_expert_x,
                                               fp8 ? d_expert_scale : nullptr, withhold_slice, c));
}

moe_status moe_dispatch_recv(const moe_dims* dims, const moe_layout_t* lay, const void* d_recv, void* d_expert_x,
                             float* d_expert_scale, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!window_ok(g, lay)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  if (!layout_ok(lay) || !d_recv || !d_expert_x || !aligned16(d_recv) || !aligned16(d_expert_x))
    return MOE_ERR_INVALID_ARG;
  if (fp8 && (!d_expert_scale || !aligned16(d_expert_scale))) return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  return cuda_status(launch_move(kMoveUnpack, g, lay, d_recv, d_expert_x, fp8 ? d_expert_scale : nullptr, c));
}

moe_status moe_expert_identity(const moe_dims* dims, const moe_layout_t* lay, const void* d_expert_x,
                               const float* d_expert_scale, uint16_t* d_expert_y, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!window_ok(g, lay)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  if (!layout_ok(lay) || !d_expert_x || !d_expert_y || !aligned16(d_expert_x) || !aligned16(d_expert_y))
    return MOE_ERR_INVALID_ARG;
  if (fp8 && (!d_expert_scale || !aligned16(d_expert_scale))) return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  if (fp8)
    return cuda_status(launch_dequant_fp8(g, lay, static_cast<const uint8_t*>(d_expert_x), d_expert_scale,
                                          d_expert_y, c));
  if (static_cast<const void*>(d_expert_y) == d_expert_x) return MOE_OK;  // identity by aliasing
  return cuda_status(launch_move(kMoveCopyEx, g, lay, d_expert_x, d_expert_y, nullptr, c));
}

moe_status moe_combine_send(const moe_dims* dims, const moe_layout_t* lay, const uint16_t* d_expert_y,
                            uint16_t* d_csend, uint16_t* d_crecv, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!window_ok(g, lay)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  const bool push = lay && (lay->flags & MOE_FLAG_DIRECT_PUSH);
  if (!layout_ok(lay) || !d_expert_y || !d_crecv || !aligned16(d_expert_y) || !aligned16(d_crecv) ||
      (!push && (!d_csend || !aligned16(d_csend))))
    return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  if (push) return cuda_status(launch_move(kMoveCPush, g, lay, d_expert_y, d_crecv, nullptr, c));
  cudaError_t e = launch_move(kMoveCPack, g, lay, d_expert_y, d_csend, nullptr, c);
  if (e == cudaSuccess) e = launch_move(kMoveCScatter, g, lay, d_csend, d_crecv, nullptr, c);
  return cuda_status(e);
}

moe_status moe_combine_recv(const moe_dims* dims, const moe_layout_t* lay, const uint16_t* d_crecv, const float* d_w,
                            uint16_t* d_out, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!window_ok(g, lay)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  if (!layout_ok(lay) || !d_crecv || !d_w || !d_out || !aligned16(d_crecv) || !aligned16(d_out))
    return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  return cuda_status(launch_combine_reduce(g, lay, d_crecv, d_w, d_out, c));
}

moe_status moe_dispatch(const moe_dims* dims, const moe_layout_t* lay, const void* d_x, void* d_send, void* d_recv,
                        void* d_expert_x, float* d_expert_scale, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!whole_group(g, lay)) return MOE_ERR_INVALID_ARG;   // a rank window is not supported here
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  const bool push = lay && (lay->flags & MOE_FLAG_DIRECT_PUSH);
  if (!layout_ok(lay) || !d_x || !d_recv || !d_expert_x || !aligned16(d_x) || !aligned16(d_recv) ||
      !aligned16(d_expert_x) || (!push && (!d_send || !aligned16(d_send))) ||
      (fp8 && (!d_expert_scale || !aligned16(d_expert_scale))))
    return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  return cuda_status(run_batches(g, c, phase_batch_count(g, lay), [&](int t0, int nt, Ctx& cj) {
    return dispatch_range(g, lay, d_x, d_send, d_recv, d_expert_x, d_expert_scale, t0, nt, cj);
  }));
}

moe_status moe_combine(const moe_dims* dims, const moe_layout_t* lay, const uint16_t* d_expert_y, uint16_t* d_csend,
                       uint16_t* d_crecv, const float* d_w, uint16_t* d_out, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!whole_group(g, lay)) return MOE_ERR_INVALID_ARG;   // a rank window is not supported here
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  const bool push = lay && (lay->flags & MOE_FLAG_DIRECT_PUSH);
  if (!layout_ok(lay) || !d_expert_y || !d_crecv || !d_w || !d_out || !aligned16(d_expert_y) ||
      !aligned16(d_crecv) || !aligned16(d_out) || (!push && (!d_csend || !aligned16(d_csend))))
    return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  return cuda_status(run_batches(g, c, phase_batch_count(g, lay), [&](int t0, int nt, Ctx& cj) {
    return combine_range(g, lay, d_expert_y, d_csend, d_crecv, d_w, d_out, t0, nt, cj);
  }));
}

moe_status moe_combine_send_partial(const moe_dims* dims, const moe_layout_t* lay, const uint16_t* d_expert_y,
                                    const float* d_w, uint16_t* d_cpart, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!whole_group(g, lay)) return MOE_ERR_INVALID_ARG;   // a rank window is not supported here
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  if (!layout_ok(lay) || !d_expert_y || !d_w || !d_cpart || !aligned16(d_expert_y) || !aligned16(d_cpart) ||
      g.R > 32)
    return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  return cuda_status(launch_combine_partial(g, lay, d_expert_y, d_w, d_cpart, c));
}

moe_status moe_combine_recv_partial(const moe_dims* dims, const moe_layout_t* lay, const uint16_t* d_cpart,
                                    uint16_t* d_out, void* stream) {
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!whole_group(g, lay)) return MOE_ERR_INVALID_ARG;   // a rank window is not supported here
  if ((int64_t)g.N * g.T == 0) return layout_ok(lay) ? MOE_OK : MOE_ERR_INVALID_ARG;  // nothing to move
  if (!layout_ok(lay) || !d_cpart || !d_out || !aligned16(d_cpart) || !aligned16(d_out) || g.R > 32)
    return MOE_ERR_INVALID_ARG;
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  return cuda_status(launch_combine_sum(g, lay, d_cpart, d_out, c));
}

moe_status moe_forward(const moe_dims* dims, const moe_layout_t* lay, const moe_buffers_t* b, void* stream) {
  if (!b) return MOE_ERR_INVALID_ARG;
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  const bool fp8 = g.payload == MOE_PAYLOAD_FP8_E4M3_B128;
  // Every buffer is checked before anything is launched (an empty batch needs none).
  if (!layout_ok(lay) || !whole_group(g, lay)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)g.N * g.T > 0 &&
      (!pass_buffers_ok(b, lay->flags, fp8, true) ||
       (fp8 && (lay->flags & MOE_FLAG_STAGED_QUANT) && (!b->xq || !aligned16(b->xq)))))
    return MOE_ERR_INVALID_ARG;
  {
    // One or more token batches of the whole chain; staged fp8 quantisation runs as a
    // separate pass over all tokens first, so it takes the phase by phase path below.
    const int nb = moe_batches(dims, lay, 0);
    const bool staged = fp8 && (lay->flags & MOE_FLAG_STAGED_QUANT);
    if (nb > 1 || ((int64_t)g.N * g.T > 0 && !staged)) return forward_batched(g, dims, lay, b, nb, stream);
  }
  if ((st = moe_layout(dims, b->idx, lay, stream)) != MOE_OK) return st;
  if (fp8 && !(lay->flags & MOE_FLAG_STAGED_QUANT)) {
    if ((st = moe_quantize_dispatch_send(dims, lay, b->x, b->send, b->recv, stream)) != MOE_OK) return st;
  } else {
    const void* xin = b->x;
    if (fp8) {
      if ((st = moe_quantize_fp8_b128(dims, b->x, b->xq, lay, stream)) != MOE_OK) return st;
      xin = b->xq;
    }
    if ((st = moe_dispatch_send(dims, lay, xin, b->send, b->recv, stream)) != MOE_OK) return st;
  }
  if ((st = moe_dispatch_recv(dims, lay, b->recv, b->expert_x, b->expert_scale, stream)) != MOE_OK) return st;
  if ((st = moe_expert_identity(dims, lay, b->expert_x, b->expert_scale, b->expert_y, stream)) != MOE_OK) return st;
  if ((st = moe_combine_send(dims, lay, b->expert_y, b->csend, b->crecv, stream)) != MOE_OK) return st;
  return moe_combine_recv(dims, lay, b->crecv, b->w, b->out, stream);
}

moe_status moe_forward_host(const moe_dims* dims, const moe_layout_t* lay, const moe_buffers_t* b, const uint16_t* h_x,
                            const int32_t* h_idx, const float* h_w, uint16_t* h_out, void* stream) {
  if (!b) return MOE_ERR_INVALID_ARG;
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  const size_t xb = (size_t)g.N * g.T * g.H * 2, pb = (size_t)g.P * 4;
  if ((xb && (!h_x || !h_out || !b->x || !b->out)) || (pb && (!h_idx || !h_w || !b->idx || !b->w)))
    return MOE_ERR_INVALID_ARG;
  if (!layout_ok(lay) || !whole_group(g, lay)) return MOE_ERR_INVALID_ARG;
  if (lay->flags & MOE_FLAG_HOST_MAPPED) {
    // Device-accessible host memory: run the pass on it directly.
    void *dx = nullptr, *didx = nullptr, *dw = nullptr, *dout = nullptr;
    if (host_mapped(h_x, &dx) && host_mapped(h_idx, &didx) && host_mapped(h_w, &dw) && host_mapped(h_out, &dout)) {
      moe_buffers_t m = *b;
      m.x = static_cast<uint16_t*>(dx);
      m.idx = static_cast<int32_t*>(didx);
      m.w = static_cast<float*>(dw);
      m.out = static_cast<uint16_t*>(dout);
      const bool two = g.T >= 2 && !(lay->flags & (MOE_FLAG_ONE_BATCH | MOE_FLAG_DIRECT_PUSH)) &&
                       !(g.payload == MOE_PAYLOAD_FP8_E4M3_B128 && (lay->flags & MOE_FLAG_STAGED_QUANT));
      return two ? forward_two_batches(g, dims, lay, &m, stream) : moe_forward(dims, lay, &m, stream);
    }
  }
  const int nb = moe_batches(dims, lay, 1);
  if (nb > 1) return forward_host_pipelined(g, dims, lay, b, h_x, h_idx, h_w, h_out, nb, stream);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (xb && cudaMemcpyAsync(b->x, h_x, xb, cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (pb && cudaMemcpyAsync(b->idx, h_idx, pb, cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (pb && cudaMemcpyAsync(b->w, h_w, pb, cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
  if ((st = moe_forward(dims, lay, b, stream)) != MOE_OK) return st;
  if (xb && cudaMemcpyAsync(h_out, b->out, xb, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

int64_t moe_exchange_plan(const moe_dims* dims, const int32_t* h_C, const int32_t* h_soff, const int32_t* h_roff,
                          int32_t nwin, const int32_t* h_bounds, int32_t me, int32_t direction, int32_t sending,
                          moe_slice_t* out, int64_t max_out) {
  Geo g;
  if (make_geo(dims, g) != MOE_OK || !h_bounds || nwin < 1 || me < 0 || me >= nwin || direction < 0 ||
      direction > 1 || sending < 0 || sending > 1 || max_out < 0)
    return -1;
  if (h_bounds[0] != 0 || h_bounds[nwin] != g.N) return -1;
  for (int w = 0; w < nwin; ++w)
    if (h_bounds[w] > h_bounds[w + 1]) return -1;
  const int N = g.N, L = g.L;
  if ((int64_t)N * g.T > 0 && (!h_C || !h_soff || !h_roff)) return -1;
  const int lo = h_bounds[me], hi = h_bounds[me + 1];
  // window of each rank
  std::vector<int32_t> win(N);
  for (int w = 0; w < nwin; ++w)
    for (int r = h_bounds[w]; r < h_bounds[w + 1]; ++r) win[r] = w;
  int64_t n = 0;
  if ((int64_t)N * g.T == 0) return 0;
  for (int s = 0; s < N; ++s)
    for (int d = 0; d < N; ++d) {
      const bool s_in = s >= lo && s < hi, d_in = d >= lo && d < hi;
      if (s_in == d_in) continue;   // inside the window (moved by the kernels) or not ours
      const int32_t rows = h_C[(int64_t)s * N + d];
      if (rows <= 0) continue;
      // Dispatch moves s -> d, combine d -> s: the side that sends is the one holding the
      // rows before the move.
      const bool mine_sends = direction == 0 ? s_in : d_in;
      if ((sending != 0) != mine_sends) continue;
      if (out && n < max_out) {
        moe_slice_t& sl = out[n];
        sl.peer = s_in ? win[d] : win[s];
        sl.s = s;
        sl.d = d;
        sl.rows = rows;
        const int64_t send_side = (int64_t)(s - lo) * g.TR + h_soff[(int64_t)s * g.E + (int64_t)d * L];
        const int64_t recv_side = (int64_t)(d - lo) * g.RB + h_roff[(int64_t)d * N + s];
        sl.local_row = s_in ? send_side : recv_side;
      }
      ++n;
    }
  return n;
}

int32_t moe_batches(const moe_dims* dims, const moe_layout_t* lay, int32_t which) {
  Geo g;
  if (make_geo(dims, g) != MOE_OK || !lay || which < 0 || which > 2) return 0;
  if ((int64_t)g.N * g.T == 0) return 1;
  return which == 1 ? host_batch_count(g, lay) : which == 2 ? phase_batch_count(g, lay) : forward_batch_count(g, lay);
}

moe_status moe_status_sync(const moe_layout_t* lay, void* stream, uint32_t* bits_out) {
  if (!lay || !lay->status) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t bits = 0;
  if (cudaMemcpy(&bits, lay->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(lay->status, 0, 4, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (bits_out) *bits_out = bits;
  for (int code = MOE_ERR_EXPERT_RANGE; code <= MOE_ERR_TIMEOUT; ++code)
    if (bits & (1u << code)) return static_cast<moe_status>(code);
  return MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_EXPERT_RANGE: return "expert id out of range (pair skipped)";
    case MOE_ERR_CAPACITY: return "expert capacity exceeded (pairs dropped)";
    case MOE_ERR_RECV_BOUND: return "receive bound N*T*max(R,E/N) exceeded";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "bounded in-kernel wait timed out";
  }
  return "unknown status";
}

uint64_t moe_launch_count(void) { return g_launches.load(); }

}  // extern "C"
