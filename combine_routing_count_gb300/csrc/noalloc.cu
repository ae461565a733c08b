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

// Device address of g_noalloc_send, looked up once per device with that device current (the
// set-up step of the first call on each device). The address belongs to the library's module
// as loaded in the device's primary context: after cudaDeviceReset, or when a caller makes
// another context of the device current, it is no longer valid, and this entry point must
// not be used there.
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
  Geo g;
  moe_status st = make_geo(dims, g);
  if (st != MOE_OK) return st;
  if (!layout_ok(lay) || (lay->win_hi > 0 && !(lay->win_lo == 0 && lay->win_hi == g.N)))
    return MOE_ERR_INVALID_ARG;   // the whole group only
  if ((int64_t)g.N * g.T == 0) return MOE_OK;   // nothing to move
  if (!d_x || !d_recv || !aligned16(d_x) || !aligned16(d_recv)) return MOE_ERR_INVALID_ARG;
  if ((size_t)(g.P * g.B) > kNoAllocSendBytes) return MOE_ERR_INVALID_ARG;   // beyond the static buffer
  Ctx c;
  if ((st = make_ctx(lay, stream, c)) != MOE_OK) return st;
  void* send = nullptr;
  if (send_scratch(c.device, &send) != cudaSuccess) return MOE_ERR_CUDA;
  // Always pack then scatter through the array (MOE_FLAG_DIRECT_PUSH, which needs no send
  // buffer, is what moe_dispatch_send offers without one).
  c.flags &= ~MOE_FLAG_DIRECT_PUSH;
  cudaError_t e = launch_move(kMovePack, g, lay, d_x, send, nullptr, c);
  if (e == cudaSuccess) e = launch_move(kMoveScatter, g, lay, send, d_recv, nullptr, c);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
