// ring_attn_bwd_noalloc: the backward pass with library-owned scratch, for
// callers that cannot allocate device memory.
//
// ring_attn_bwd takes its workspace (two float32 statistics per tile-padded
// query row, written by the prep phase and read by the gradient kernels)
// from the caller. Some callers have no way to provide one: a plugin whose
// host framework owns the device memory through its own pool and hands it no
// workspace, or a latency-critical path on which cudaMalloc / cudaFree may
// synchronise the device. For them this entry point keeps the workspace in a
// file-scope device array, so the call allocates nothing.
//
// The array is module memory: every GPU that loads the library holds it until
// the process exits. Its host-side name is only a stand-in for the symbol, so
// host code passes the kernels the device address that cudaGetSymbolAddress
// returns, looked up once per device with that device current.
#include <mutex>

#include "ra_internal.h"

namespace {

constexpr size_t kScratchFloats = RA_BWD_NOALLOC_MAX_BYTES / sizeof(float);

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) float g_bwd_scratch[kScratchFloats];

// Device address of g_bwd_scratch on the current device (cached per device).
ra_status scratch_address(float** ptr) {
  static std::mutex mu;
  static float* addr[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return RA_ERR_DEVICE;
  }
  if (dev < 0 || dev >= 64) return RA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return RA_ERR_LAUNCH;
    }
    addr[dev] = static_cast<float*>(p);
  }
  *ptr = addr[dev];
  return RA_OK;
}

}  // namespace

extern "C" ra_status ring_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                           const void* out, const float* lse, const void* dout,
                                           void* dq, void* dk, void* dv, int B, int H_q,
                                           int H_kv, int S, int D, int P, int causal,
                                           float scale, int dtype, int order, int* dev_status,
                                           void* stream) {
  // the size check is host arithmetic only: an oversized problem is refused
  // before the GPU is touched
  size_t need = 0;
  ra_status st = ring_attn_bwd_workspace(B, H_q, S, D, P, order, &need);
  if (st != RA_OK) return st;
  if (need > (size_t)RA_BWD_NOALLOC_MAX_BYTES) return RA_ERR_SCRATCH;
  int sms = 0;
  st = ra::check_device(&sms);
  if (st != RA_OK) return st;
  float* ws = nullptr;
  st = scratch_address(&ws);
  if (st != RA_OK) return st;
  // every remaining argument check, then the same three kernels as ring_attn_bwd
  return ring_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, H_q, H_kv, S, D, P, causal,
                       scale, dtype, order, ws, (size_t)RA_BWD_NOALLOC_MAX_BYTES, dev_status,
                       stream);
}
