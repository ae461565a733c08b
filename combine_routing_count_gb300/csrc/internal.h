// Host-side internals of libmoe_ep: launch context, per-kernel profiling scope and the
// launchers each translation unit provides.
#pragma once

#include <atomic>
#include <utility>

#include "common.cuh"

namespace moe {

// Everything a launcher needs besides its operands.
struct Ctx {
  cudaStream_t stream;
  moe_prof_t* prof;
  int device;
  int num_sms;
  int smem_optin;     // max dynamic shared memory per block (opt-in), bytes
  int smem_per_sm;    // shared memory per SM, bytes
  int l2_bytes;       // L2 cache size, bytes
  uint32_t flags;
  int tma_stages;     // 0 = automatic
  int ctas_per_sm;    // 0 = automatic
  int32_t* status;
  int win_lo, win_hi; // rank window of the layout (0, 0: the whole group)
};

// True when the call works on a rank window smaller than the group (see moe_layout_t).
inline bool windowed(const Geo& g, const Ctx& c) { return c.win_hi > 0 && !(c.win_lo == 0 && c.win_hi == g.N); }

// A device pointer moved back by `bytes`: the base of a window-local buffer seen as a whole-
// group buffer, so that whole-group row indices of the window's ranks land in it. Only rows
// of the window are ever accessed through it.
template <typename P>
inline P rebase(P p, int64_t bytes) {
  return p ? reinterpret_cast<P>(reinterpret_cast<uintptr_t>(p) - (uintptr_t)bytes) : p;
}

extern std::atomic<uint64_t> g_launches;

// Reads prof->flush (prof->flush_bytes) on `stream`: the cold-cache option of moe_prof_t.
cudaError_t launch_l2_flush(const moe_prof_t* prof, cudaStream_t stream);

// Launches `kernel` on c.stream, with programmatic stream serialization unless
// MOE_FLAG_NO_PDL is set (every kernel calls pdl_wait() before touching memory).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, const Ctx& c,
                                 Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (c.flags & MOE_FLAG_NO_PDL) ? 0 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Brackets one kernel launch with the caller's profiling events (if any) and counts it.
struct LaunchScope {
  Ctx& c;
  int slot = -1;
  LaunchScope(Ctx& ctx, moe_kernel_id id) : c(ctx) {
    if (c.prof && c.prof->n < MOE_PROF_MAX) {
      launch_l2_flush(c.prof, c.stream);
      slot = c.prof->n++;
      c.prof->kernel[slot] = id;
      cudaEventRecord(static_cast<cudaEvent_t>(c.prof->events[2 * slot]), c.stream);
    }
  }
  ~LaunchScope() {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (slot >= 0) cudaEventRecord(static_cast<cudaEvent_t>(c.prof->events[2 * slot + 1]), c.stream);
  }
};

// Raises a kernel's dynamic shared memory limit to `bytes` (needed above 48 KB) once per
// device; `cache` holds the largest value set so far for each of 64 devices.
template <typename K>
inline cudaError_t ensure_dyn_smem(K kernel, int device, size_t bytes, std::atomic<int>* cache) {
  if (bytes + 1024 <= 48 * 1024) return cudaSuccess;   // room for up to 1 KB of static shared memory
  std::atomic<int>& c = cache[device & 63];
  if (c.load() >= (int)bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  int cur = c.load();
  while (cur < (int)bytes && !c.compare_exchange_weak(cur, (int)bytes)) {
  }
  return cudaSuccess;
}

// api.cu: argument checks shared by every entry point.
moe_status make_geo(const moe_dims* d, Geo& g);                       // dims -> geometry, or INVALID_ARG
moe_status make_ctx(const moe_layout_t* lay, void* stream, Ctx& c);   // launch context (device attributes cached)
bool layout_ok(const moe_layout_t* l);                                // every layout array present

// layout.cu
cudaError_t launch_layout(const Geo& g, const int32_t* idx, const moe_layout_t* lay, Ctx& c);
int layout_chunks(const Geo& g);
int64_t layout_scratch_done_offset(const Geo& g);  // ints from the scratch start to the counters
int64_t layout_scratch_tgroups_offset(const Geo& g);  // ... to the per-token group counts
int64_t layout_scratch_arrive_offset(const Geo& g);   // ... to the split-dispatch counters (+ 2)

// split.cu
constexpr int kMaxSplitBatches = 32;   // token batches of the split-phase dispatch
// Words of the split-dispatch arrival counters: one per (token batch, source rank).
inline int64_t split_arrive_words(const Geo& g) {
  const int64_t a = (int64_t)g.N * g.N, b = (int64_t)kMaxSplitBatches * g.N;
  return a > b ? a : b;
}
int split_batches(const Geo& g);

// dedicated.cu
size_t dedicated_exchange_bytes(const Geo& g);
cudaError_t launch_dispatch_dedicated(const Geo& g, const moe_layout_t* lay, const int32_t* idx, const void* x,
                                      int K, void* ded, void* xchg, void* main, void* ex, float* exs,
                                      int drop_slice, Ctx& c);

cudaError_t launch_dispatch_split(const Geo& g, const moe_layout_t* lay, const void* x, void* recv, void* ex,
                                  float* exs, int drop_source, Ctx& c);

// movers.cu: row movement kernels.
enum MoveKind : int {
  kMovePack = 0,      // token rows -> R send rows
  kMoveScatter = 1,   // send rows -> receive rows of the owner rank
  kMoveUnpack = 2,    // receive rows -> grouped expert rows (fp8: codes + scales)
  kMoveCPack = 3,     // grouped expert output rows -> receive order (combine send buffer)
  kMoveCScatter = 4,  // combine send rows -> the source rank's combine receive rows
  kMoveCopyEx = 5,    // grouped rows -> grouped rows (bf16 identity expert, distinct output)
  kMovePackPush = 6,  // direct push: token rows -> R receive rows of the owner ranks
  kMoveCPush = 7,     // direct push: grouped expert output rows -> source ranks' combine rows
  kMovePackAll = 8,   // pack, write and shuffle in one move: token row -> its R send rows (dst), the
                      // owners' receive rows (dst2) and the kept pairs' grouped rows (dst3), bf16
  kMovePackAllPush = 9,  // the same with direct push: no send rows (dst unused)
};

// Moves whose unit is a (token, column chunk) that fans out to the token's R pairs.
constexpr bool is_pack_kind(int kind) {
  return kind == kMovePack || kind == kMovePackPush || kind == kMovePackAll || kind == kMovePackAllPush;
}
constexpr bool is_pack_all_kind(int kind) { return kind == kMovePackAll || kind == kMovePackAllPush; }
cudaError_t launch_move(MoveKind kind, const Geo& g, const moe_layout_t* lay, const void* src, void* dst,
                        void* dst2, Ctx& c, void* dst3 = nullptr);
// The same move over the token range [t0, t0 + nt) of every rank only (its tokens for a
// pack, its pairs otherwise).
// dst3: the grouped rows of kMovePackAll; unused otherwise.
cudaError_t launch_move_range(MoveKind kind, const Geo& g, const moe_layout_t* lay, const void* src, void* dst,
                              void* dst2, int t0, int nt, Ctx& c, void* dst3 = nullptr);

// numerics.cu
cudaError_t launch_quant_fp8(const Geo& g, const uint16_t* x, uint8_t* xq, Ctx& c);
// Quantise bf16 token rows and write each one's fp8 row into dst rows fan[token][k] (k < R).
// t0, nt: only the token range [t0, t0 + nt) of every rank (nt < 0: all tokens).
cudaError_t launch_quant_pack(const Geo& g, const int32_t* fan, const uint16_t* x, uint8_t* dst, Ctx& c, int t0 = 0,
                              int nt = -1);
cudaError_t launch_dequant_fp8(const Geo& g, const moe_layout_t* lay, const uint8_t* exq, const float* exs,
                               uint16_t* ey, Ctx& c, int t0 = 0, int nt = -1);   // t0, nt as launch_quant_pack
cudaError_t launch_combine_partial(const Geo& g, const moe_layout_t* lay, const uint16_t* ey, const float* w,
                                   uint16_t* cpart, Ctx& c);
cudaError_t launch_combine_sum(const Geo& g, const moe_layout_t* lay, const uint16_t* cpart, uint16_t* out,
                               Ctx& c);
cudaError_t launch_combine_reduce(const Geo& g, const moe_layout_t* lay, const uint16_t* crecv, const float* w,
                                  uint16_t* out, Ctx& c, int t0 = 0, int nt = -1);   // t0, nt as launch_quant_pack
// fp8 quantisation, pack, write and shuffle in one kernel: each token row quantised once and
// stored to its R send rows (none when send is null: direct push), the owners' receive rows
// and the kept pairs' grouped codes and scales (whole group only).
cudaError_t launch_quant_dispatch_fused(const Geo& g, const moe_layout_t* lay, const uint16_t* x, uint8_t* send,
                                        uint8_t* recv, uint8_t* ex, float* exs, Ctx& c, int t0 = 0, int nt = -1);
// Combine pack, write and weighted sum in one kernel: each kept pair's expert output row read
// once, stored to its receive-order row (csend; none when csend is null: direct push) and its
// source's combine row (crecv), and summed into the token's output as launch_combine_reduce
// does (whole group only).
cudaError_t launch_combine_fused(const Geo& g, const moe_layout_t* lay, const uint16_t* ey, uint16_t* csend,
                                 uint16_t* crecv, const float* w, uint16_t* out, Ctx& c, int t0 = 0, int nt = -1);

}  // namespace moe
