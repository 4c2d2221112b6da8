// Bounds checks of the debug build (compiled with -DRA_DEBUG_CHECKS).
//
// Every global-memory access a kernel computes from indices (TMA copies are
// bounds-checked by the hardware) is tested against the extent of its
// tensor. A violation records RA_ERR_RANGE in the status word and the access
// is skipped: no trap, no fault, and the context stays usable. The release
// build compiles every check to `true`.
#pragma once

#include "ra_internal.h"

namespace ra {

// Rows of the q/k/v/out tensors in the call's layout: B*S (fixed length),
// total (packed sequences) or P*B*C (sequence-sharded).
__device__ __forceinline__ long long layout_rows(const Geometry& g) {
  if (g.cu_seqlens) return g.total;
  if (g.shard_rows > 0) return (long long)g.P * g.B * g.shard_rows;
  return (long long)g.B * g.S;
}
__device__ __forceinline__ long long extent_q(const Geometry& g) {
  return layout_rows(g) * g.H_q * g.D;
}
__device__ __forceinline__ long long extent_kv(const Geometry& g) {
  return layout_rows(g) * g.H_kv * g.D;
}
// lse holds one value per query row and head in every layout
__device__ __forceinline__ long long extent_lse(const Geometry& g) {
  return layout_rows(g) * g.H_q;
}

#ifdef RA_DEBUG_CHECKS
__device__ __forceinline__ bool in_range(long long first, long long count, long long extent,
                                         int* status) {
  if (first >= 0 && first + count <= extent) return true;
  if (status) atomicExch(status, (int)RA_ERR_RANGE);
  return false;
}
#else
__device__ __forceinline__ bool in_range(long long, long long, long long, int*) { return true; }
#endif

}  // namespace ra
