// Internal declarations shared by the host entry points and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ring_attn.h"

namespace ra {

// Geometry of one ring-attention call, as every kernel role sees it.
// Segments are the contiguous token ranges a virtual rank owns: one chunk of
// S/P tokens (contiguous order) or two halves of S/(2P) tokens (zig-zag).
// Segment g (in position order) starts at g * seg_len. Each segment is cut
// into `nt` tiles of `tile` rows; the last may be shorter.
struct Geometry {
  int B, H_q, H_kv, S, D, P;
  int causal;
  int order;       // RA_ORDER_*
  int step;        // -1: all steps; else the single ring step to run
  int seg_len;     // tokens per segment
  int n_seg;       // P or 2P
  int segs_per_rank;
  int tile;        // tile rows of the kernel
  int nt;          // tiles per segment
  float scale;     // softmax scale
  float scale_log2;  // scale * log2(e)
  // Packed variable-length batches (null for fixed-length BSHD tensors):
  // sequence b occupies rows [cu_seqlens[b], cu_seqlens[b+1]) of tensors of
  // `total` rows; B is the number of sequences and S their maximum length,
  // which sizes the grid. Each sequence is its own ring problem.
  const int* cu_seqlens;
  int total;
  // > 0: tensors in the sequence-sharded layout of P virtual ranks,
  // [P, B, shard_rows, H, D] (rank p's rows [p * shard_rows, ...) of every
  // batch contiguous), chunks contiguous with shard_rows = seg_len.
  int shard_rows;
  // Forward grid order: 0 = (batch, kv head) outermost, so the CTAs resident
  // at one time share one head's keys and values in L2; 1 = query block
  // outermost (globally longest first), for problems whose keys and values
  // fit in L2 anyway.
  int qb_major;
};

// Host-side planning helpers (plan.cpp).
ra_status make_geometry(int B, int H_q, int H_kv, int S, int D, int P,
                        int causal, float scale, int order, int step, int tile,
                        Geometry* g);
int tile_rows_for(int dtype, int D);

// Per-device facts, cached (plan.cpp).
ra_status check_device(int* sm_count);

// Launchers (one per kernel family). They assume validated arguments.
ra_status launch_attn_simt(const Geometry& g, const float* q, const float* k,
                           const float* v, void* out, float* lse,
                           int* visit_log, int log_stride, int* dev_status,
                           cudaStream_t stream);
// Same kernel with the V load of key tile 0 withheld (expiry-path test).
ra_status launch_attn_tc_withheld(const Geometry& g, const void* q, const void* k,
                                  const void* v, void* out, float* lse, int* dev_status,
                                  cudaStream_t stream);
// Packed variable-length launches (g.cu_seqlens set, no visit log, all steps).
ra_status launch_attn_tc_varlen(const Geometry& g, const void* q, const void* k,
                                const void* v, void* out, float* lse, int* dev_status,
                                cudaStream_t stream);
ra_status launch_attn_simt_varlen(const Geometry& g, const float* q, const float* k,
                                  const float* v, float* out, float* lse, int* dev_status,
                                  cudaStream_t stream);
// Sequence-sharded layout launches (g.shard_rows set, no visit log, all steps).
ra_status launch_attn_tc_sharded(const Geometry& g, const void* q, const void* k,
                                 const void* v, void* out, float* lse, int* dev_status,
                                 cudaStream_t stream);
ra_status launch_attn_simt_sharded(const Geometry& g, const float* q, const float* k,
                                   const float* v, float* out, float* lse, int* dev_status,
                                   cudaStream_t stream);
ra_status launch_attn_tc(const Geometry& g, const void* q, const void* k,
                         const void* v, void* out, float* lse, int* visit_log,
                         int log_stride, int* dev_status, cudaStream_t stream);

// TMA map of a [B, S, H, D] bf16 tensor: box = 64 columns x 1 head x
// `box_rows` rows x 1 batch, 128-byte swizzle (tensor_map.cpp).
bool make_bshd_map(CUtensorMap* m, const void* ptr, int B, int S, int H, int D,
                   int box_rows);

// Backward pass (attn_bwd.cu). `workspace` holds bwd_workspace_floats(g)
// floats: per (b, h, query tile) 128 base-2 lse values, then as many deltas.
long long bwd_workspace_floats(const Geometry& g);
ra_status launch_attn_bwd(const Geometry& g, const void* q, const void* k, const void* v,
                          const void* out, const float* lse, const void* dout, void* dq,
                          void* dk, void* dv, float* workspace, int phases,
                          int* dev_status, cudaStream_t stream);

struct MergeArgs {
  const void* o[RA_MERGE_MAX_N];
  const float* lse[RA_MERGE_MAX_N];
  int n;
  void* out;
  float* out_lse;
  int B, H, S, D;
};
ra_status launch_merge(const MergeArgs& a, int dtype, int sm_count,
                       cudaStream_t stream);

}  // namespace ra
