// Host-side planning: ring schedule table, tiling, argument checks, errors.
//
// Glossary "sequence parallelism transformers": §Sequence Parallelism
// Fundamentals (S cut into P chunks of S/P tokens), §Ring Attention (at step
// t rank r holds the block of rank (r - t) mod P), §Implementation
// Considerations (load balancing: the zig-zag order, 2P halves with rank r
// owning halves r and 2P-1-r).
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ra_internal.h"

namespace ra {

int tile_rows_for(int dtype, int D) {
  (void)D;
  return dtype == RA_BF16 ? 128 : 64;
}

ra_status make_geometry(int B, int H_q, int H_kv, int S, int D, int P,
                        int causal, float scale, int order, int step, int tile,
                        Geometry* g) {
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || S <= 0 || P <= 0) return RA_ERR_SHAPE;
  if (H_q % H_kv != 0) return RA_ERR_SHAPE;
  if (order != RA_ORDER_CONTIGUOUS && order != RA_ORDER_ZIGZAG) return RA_ERR_DTYPE;
  const int parts = order == RA_ORDER_ZIGZAG ? 2 * P : P;
  if (step < -1 || step >= P) return RA_ERR_RANGE;
  g->B = B; g->H_q = H_q; g->H_kv = H_kv; g->S = S; g->D = D; g->P = P;
  g->causal = causal ? 1 : 0;
  g->order = order;
  g->step = step;
  g->n_seg = parts;
  // S counts as padded to a multiple of `parts`; the padding holds no token
  g->seg_len = (S + parts - 1) / parts;
  g->segs_per_rank = order == RA_ORDER_ZIGZAG ? 2 : 1;
  g->tile = tile;
  g->nt = (g->seg_len + tile - 1) / tile;
  g->scale = scale > 0.f ? scale : 1.0f / __builtin_sqrtf((float)D);
  g->scale_log2 = g->scale * 1.4426950408889634f;
  g->cu_seqlens = nullptr;
  g->total = 0;
  g->shard_rows = 0;
  g->qb_major = 0;
  return RA_OK;
}

ra_status check_device(int* sm_count) {
  // Per-device cache of (compute capability ok, SM count).
  static std::mutex mu;
  static int cached_ok[64];
  static int cached_sms[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return RA_ERR_DEVICE;
  }
  if (dev < 0 || dev >= 64) return RA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (cached_ok[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return RA_ERR_DEVICE;
    }
    cached_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    cached_sms[dev] = sms;
  }
  if (cached_ok[dev] != 1) return RA_ERR_DEVICE;
  if (sm_count) *sm_count = cached_sms[dev];
  return RA_OK;
}

}  // namespace ra

using namespace ra;

namespace {

// Segment starts of rank r, ascending; returns how many (1 or 2).
int rank_segment_starts(int r, int P, int order, int seg_len, int out[2]) {
  if (order == RA_ORDER_CONTIGUOUS) {
    out[0] = r * seg_len;
    return 1;
  }
  out[0] = r * seg_len;
  out[1] = (2 * P - 1 - r) * seg_len;
  return 2;
}

// Class of all pairs (query in any q segment, key in any kv segment) under
// the causal rule key <= query. Segments start at multiples of L and hold
// their positions below S. One q range [a, a+n) and one kv range [c, c+m):
// all pairs allowed iff c+m-1 <= a; none iff c > a+n-1. Empty ranges hold no
// pair.
int classify_segments(const int* qs, int nq, const int* ks, int nk, int L, int S,
                      int causal) {
  if (!causal) return RA_CLASS_FULL;
  bool all_full = true, all_skip = true;
  for (int i = 0; i < nq; ++i)
    for (int j = 0; j < nk; ++j) {
      const int n = S - qs[i] < L ? S - qs[i] : L;
      const int m = S - ks[j] < L ? S - ks[j] : L;
      if (n <= 0 || m <= 0) continue;
      if (!(ks[j] + m - 1 <= qs[i])) all_full = false;
      if (!(ks[j] > qs[i] + n - 1)) all_skip = false;
    }
  if (all_skip) return RA_CLASS_SKIP;
  if (all_full) return RA_CLASS_FULL;
  return RA_CLASS_PARTIAL;
}

}  // namespace

extern "C" {

ra_status ring_attn_plan(int S, int P, int causal, int order, int* table,
                         size_t table_len) {
  if (!table) return RA_ERR_NULL;
  if (S <= 0 || P <= 0) return RA_ERR_SHAPE;
  if (order != RA_ORDER_CONTIGUOUS && order != RA_ORDER_ZIGZAG) return RA_ERR_DTYPE;
  const int parts = order == RA_ORDER_ZIGZAG ? 2 * P : P;
  if ((size_t)P * (size_t)P * RA_PLAN_COLS > table_len) return RA_ERR_BUFFER;
  const int L = (S + parts - 1) / parts;     // S padded to a multiple of parts
  int* row = table;
  for (int r = 0; r < P; ++r) {
    int qs[2] = {-1, -1};
    const int nq = rank_segment_starts(r, P, order, L, qs);
    for (int t = 0; t < P; ++t) {
      const int src = ((r - t) % P + P) % P;
      int ks[2] = {-1, -1};
      const int nk = rank_segment_starts(src, P, order, L, ks);
      row[0] = r;
      row[1] = t;
      row[2] = src;
      row[3] = classify_segments(qs, nq, ks, nk, L, S, causal);
      row[4] = L;
      row[5] = qs[0];
      row[6] = nq > 1 ? qs[1] : -1;
      row[7] = ks[0];
      row[8] = nk > 1 ? ks[1] : -1;
      row += RA_PLAN_COLS;
    }
  }
  return RA_OK;
}

ra_status ring_attn_visit_log_len(int B, int H_q, int S, int D, int P,
                                  int dtype, int order, int* tile_rows,
                                  int* tiles_per_segment, int* n_query_tiles,
                                  int* stride, long long* len) {
  if (dtype != RA_BF16 && dtype != RA_F32) return RA_ERR_DTYPE;
  if (D != 64 && D != 128) return RA_ERR_HEADDIM;
  Geometry g;
  ra_status st = make_geometry(B, H_q, 1, S, D, P, 0, 0.f, order, -1,
                               tile_rows_for(dtype, D), &g);
  if (st != RA_OK) return st;
  const long long nq = (long long)g.n_seg * g.nt;
  const long long strd = 1 + 4 * nq;    // a query tile visits at most every key tile
  if (tile_rows) *tile_rows = g.tile;
  if (tiles_per_segment) *tiles_per_segment = g.nt;
  if (n_query_tiles) *n_query_tiles = (int)nq;
  if (stride) *stride = (int)strd;
  if (len) *len = (long long)B * H_q * nq * strd;
  return RA_OK;
}

const char* ring_attn_strerror(int status) {
  switch (status) {
    case RA_OK: return "ok";
    case RA_ERR_NULL: return "a required pointer is NULL";
    case RA_ERR_SHAPE: return "invalid shape (sizes must be positive; H_q divisible by H_kv)";
    case RA_ERR_HEADDIM:
      return "unsupported head dimension (attention: D 64 or 128; merge: D 32, 64, 128 or 256)";
    case RA_ERR_ALIGN: return "misaligned pointer (tensors need 16-byte alignment, lse/log/status 4-byte)";
    case RA_ERR_DTYPE: return "unknown dtype or chunk order";
    case RA_ERR_DEVICE: return "no usable CUDA device of compute capability 10.3 (GB300)";
    case RA_ERR_LAUNCH: return "CUDA error while preparing or launching a kernel";
    case RA_ERR_TIMEOUT: return "a device-side bounded wait expired";
    case RA_ERR_BUFFER: return "caller buffer too small";
    case RA_ERR_RANGE: return "size out of range (32-bit indexing) or ring step outside [-1, P)";
    case RA_ERR_SCRATCH:
      return "problem too large for the library's built-in backward scratch "
             "(8 MiB: at most 2^20 tile-padded query rows; use ring_attn_bwd with a workspace)";
    default: return "unknown status";
  }
}

int ring_attn_version(void) { return 103; }   // 1.03: backward, packed variable lengths, Ulysses layout

}  // extern "C"
