// Dispatch send for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they dispatch: code running
// under a fixed memory plan set up before serving starts, allocator hooks and other code
// that must not re-enter the allocator, or hosts that hand this library only the tensors
// they already own. moe_dispatch_send needs a send buffer besides its input and output;
// this variant keeps that buffer in a file-scope device array instead, so the caller
// passes only the token rows and the receive buffer.
//
// The array (kNoAllocSendBytes, 64 MiB) is part of the library's device image: every GPU
// that loads the library holds it until the process exits. All calls share it and it
// keeps the last call's rows; every row a call reads was written earlier in the same
// call, so nothing needs clearing. Calls that overlap on the GPU (different streams,
// different threads) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace moe {
namespace {

constexpr size_t kNoAllocSendBytes = 64ull << 20;

static __device__ __align__(256) uint8_t g_noalloc_send[kNoAllocSendBytes];

// Device address of g_noalloc_send, looked up once per device with that device current.
void* g_send_addr[64];
std::mutex g_send_mu;

cudaError_t send_scratch(int device, void** out) {
  std::lock_guard<std::mutex> lk(g_send_mu);
  if (!g_send_addr[device & 63]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_send);
    if (e != cudaSuccess) return e;
    g_send_addr[device & 63] = p;
  }
  *out = g_send_addr[device & 63];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_dispatch_send_noalloc(const moe_dims* dims, const moe_layout_t* lay, const void* d_x,
                                                void* d_recv, void* stream) {
  if (moe_check_dims(dims) != MOE_OK || !lay || !lay->gsend || !lay->grecv || !lay->status)
    return MOE_ERR_INVALID_ARG;
  const int64_t N = dims->N, T = dims->T, R = dims->R, E = dims->E, H = dims->H, L = E / N;
  if (N * T == 0) return MOE_OK;
  if (!d_x || !d_recv || !aligned16(d_x) || !aligned16(d_recv)) return MOE_ERR_INVALID_ARG;
  const int64_t B = (int64_t)moe_row_bytes(dims);
  if ((size_t)(N * T * R * B) > kNoAllocSendBytes) return MOE_ERR_INVALID_ARG;  // beyond the static buffer

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  void* send = nullptr;
  if (send_scratch(dev, &send) != cudaSuccess) return MOE_ERR_CUDA;
  Ctx c;
  c.device = dev;
  c.stream = static_cast<cudaStream_t>(stream);
  c.prof = lay->prof;
  c.flags = lay->flags;
  c.tma_stages = lay->tma_stages;
  c.ctas_per_sm = lay->ctas_per_sm;
  c.status = lay->status;
  if (cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&c.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&c.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&c.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  Geo g;
  g.N = (int)N;
  g.T = (int)T;
  g.H = (int)H;
  g.E = (int)E;
  g.R = (int)R;
  g.L = (int)L;
  g.cap = moe_capacity(dims);
  g.payload = dims->payload;
  g.TR = T * R;
  g.RB = (int64_t)moe_recv_capacity_rows(dims);
  g.P = N * T * R;
  g.B = B;
  cudaError_t e = launch_move(kMovePack, g, lay, d_x, send, nullptr, c);
  if (e == cudaSuccess) e = launch_move(kMoveScatter, g, lay, send, d_recv, nullptr, c);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
