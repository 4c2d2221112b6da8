// extern "C" entry points: argument checks, then dispatch to one kernel.
//
// Every check runs on the host before anything touches the GPU, so a bad
// call returns its status without launching work.
#include <cstdint>

#include "ra_internal.h"

using namespace ra;

namespace {

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

constexpr long long kMaxElems = 0x7fffffffLL;   // 32-bit element indexing

ra_status check_attn_args(const void* q, const void* k, const void* v,
                          const void* out, const float* lse, int B, int H_q,
                          int H_kv, int S, int D, int dtype, int step,
                          const int* visit_log, const int* dev_status) {
  if (!q || !k || !v || !out) return RA_ERR_NULL;
  if (step >= 0 && !lse) return RA_ERR_NULL;
  if (dtype != RA_BF16 && dtype != RA_F32) return RA_ERR_DTYPE;
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || S <= 0) return RA_ERR_SHAPE;
  if (D != 64 && D != 128) return RA_ERR_HEADDIM;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return RA_ERR_ALIGN;
  if ((lse && !aligned(lse, 4)) || (visit_log && !aligned(visit_log, 4)) ||
      (dev_status && !aligned(dev_status, 4)))
    return RA_ERR_ALIGN;
  const long long nq = (long long)B * S * H_q * D;
  const long long nk = (long long)B * S * H_kv * D;
  if (nq > kMaxElems || nk > kMaxElems) return RA_ERR_RANGE;
  return RA_OK;
}

}  // namespace

extern "C" {

ra_status ring_attn_fwd_ex(const void* q, const void* k, const void* v,
                           void* out, float* lse, int B, int H_q, int H_kv,
                           int S, int D, int P, int causal, float scale,
                           int dtype, int order, int step, int* visit_log,
                           int* dev_status, void* stream) {
  ra_status st = check_attn_args(q, k, v, out, lse, B, H_q, H_kv, S, D, dtype,
                                 step, visit_log, dev_status);
  if (st != RA_OK) return st;
  Geometry g;
  st = make_geometry(B, H_q, H_kv, S, D, P, causal, scale, order, step,
                     tile_rows_for(dtype, D), &g);
  if (st != RA_OK) return st;
  int log_stride = 0;
  if (visit_log) {
    long long len = 0;
    st = ring_attn_visit_log_len(B, H_q, S, D, P, dtype, order, nullptr,
                                 nullptr, nullptr, &log_stride, &len);
    if (st != RA_OK) return st;
    if (len > kMaxElems) return RA_ERR_RANGE;
  }
  int sms = 0;
  st = check_device(&sms);
  if (st != RA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == RA_F32)
    return launch_attn_simt(g, static_cast<const float*>(q),
                            static_cast<const float*>(k),
                            static_cast<const float*>(v), out, lse, visit_log,
                            log_stride, dev_status, s);
  return launch_attn_tc(g, q, k, v, out, lse, visit_log, log_stride, dev_status, s);
}

ra_status ring_attn_fwd(const void* q, const void* k, const void* v,
                        void* out, float* lse, int B, int H_q, int H_kv, int S,
                        int D, int P, int causal, float scale, void* stream) {
  return ring_attn_fwd_ex(q, k, v, out, lse, B, H_q, H_kv, S, D, P, causal,
                          scale, RA_BF16, RA_ORDER_CONTIGUOUS, -1, nullptr,
                          nullptr, stream);
}

ra_status ring_attn_expiry_test(const void* q, const void* k, const void* v, void* out,
                                float* lse, int S, int* dev_status, void* stream) {
  if (!dev_status) return RA_ERR_NULL;
  ra_status st = check_attn_args(q, k, v, out, lse, 1, 1, 1, S, 128, RA_BF16, -1, nullptr,
                                 dev_status);
  if (st != RA_OK) return st;
  if (S > 4096) return RA_ERR_RANGE;
  Geometry g;
  st = make_geometry(1, 1, 1, S, 128, 1, 0, 0.f, RA_ORDER_CONTIGUOUS, -1,
                     tile_rows_for(RA_BF16, 128), &g);
  if (st != RA_OK) return st;
  int sms = 0;
  st = check_device(&sms);
  if (st != RA_OK) return st;
  return launch_attn_tc_withheld(g, q, k, v, out, lse, dev_status,
                                 reinterpret_cast<cudaStream_t>(stream));
}

ra_status ring_attn_bwd_workspace(int B, int H_q, int S, int D, int P, int order,
                                  size_t* bytes) {
  if (!bytes) return RA_ERR_NULL;
  if (D != 64 && D != 128) return RA_ERR_HEADDIM;
  Geometry g;
  ra_status st = make_geometry(B, H_q, 1, S, D, P, 0, 0.f, order, -1,
                               tile_rows_for(RA_BF16, D), &g);
  if (st != RA_OK) return st;
  const long long n = bwd_workspace_floats(g);
  if (n / 2 > kMaxElems) return RA_ERR_RANGE;
  *bytes = (size_t)n * sizeof(float);
  return RA_OK;
}

ra_status ring_attn_bwd_ex(const void* q, const void* k, const void* v, const void* out,
                           const float* lse, const void* dout, void* dq, void* dk, void* dv,
                           int B, int H_q, int H_kv, int S, int D, int P, int causal,
                           float scale, int dtype, int order, void* workspace,
                           size_t workspace_bytes, int phases, int* dev_status,
                           void* stream) {
  if (!lse || !dout || !dq || !dk || !dv || !workspace) return RA_ERR_NULL;
  if (phases <= 0 || phases > RA_BWD_ALL) return RA_ERR_RANGE;
  ra_status st = check_attn_args(q, k, v, out, lse, B, H_q, H_kv, S, D, dtype, -1,
                                 nullptr, dev_status);
  if (st != RA_OK) return st;
  if (dtype != RA_BF16) return RA_ERR_DTYPE;
  if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(workspace, 16))
    return RA_ERR_ALIGN;
  Geometry g;
  st = make_geometry(B, H_q, H_kv, S, D, P, causal, scale, order, -1,
                     tile_rows_for(dtype, D), &g);
  if (st != RA_OK) return st;
  size_t need = 0;
  st = ring_attn_bwd_workspace(B, H_q, S, D, P, order, &need);
  if (st != RA_OK) return st;
  if (workspace_bytes < need) return RA_ERR_BUFFER;
  int sms = 0;
  st = check_device(&sms);
  if (st != RA_OK) return st;
  return launch_attn_bwd(g, q, k, v, out, lse, dout, dq, dk, dv,
                         static_cast<float*>(workspace), phases, dev_status,
                         reinterpret_cast<cudaStream_t>(stream));
}

ra_status ring_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv,
                        int B, int H_q, int H_kv, int S, int D, int P, int causal,
                        float scale, int dtype, int order, void* workspace,
                        size_t workspace_bytes, int* dev_status, void* stream) {
  return ring_attn_bwd_ex(q, k, v, out, lse, dout, dq, dk, dv, B, H_q, H_kv, S, D, P, causal,
                          scale, dtype, order, workspace, workspace_bytes, RA_BWD_ALL,
                          dev_status, stream);
}

ra_status ring_attn_fwd_ulysses(const void* q, const void* k, const void* v, void* out,
                                float* lse, int B, int H_q, int H_kv, int S, int D, int P,
                                int causal, float scale, int dtype, int* dev_status,
                                void* stream) {
  if (P <= 0) return RA_ERR_SHAPE;
  if (H_q % P != 0 || H_kv % P != 0) return RA_ERR_SHAPE;
  Geometry g;
  ra_status st = make_geometry(B, H_q, H_kv, S, D, P, causal, scale, RA_ORDER_CONTIGUOUS, -1,
                               tile_rows_for(dtype, D), &g);
  if (st != RA_OK) return st;
  // the padded shards: P * C rows per batch
  st = check_attn_args(q, k, v, out, lse, B, H_q, H_kv, P * g.seg_len, D, dtype, -1, nullptr,
                       dev_status);
  if (st != RA_OK) return st;
  g.shard_rows = g.seg_len;
  int sms = 0;
  st = check_device(&sms);
  if (st != RA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == RA_F32)
    return launch_attn_simt_sharded(g, static_cast<const float*>(q),
                                    static_cast<const float*>(k), static_cast<const float*>(v),
                                    static_cast<float*>(out), lse, dev_status, s);
  return launch_attn_tc_sharded(g, q, k, v, out, lse, dev_status, s);
}

ra_status ring_attn_bwd_ulysses(const void* q, const void* k, const void* v, const void* out,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                int B, int H_q, int H_kv, int S, int D, int P, int causal,
                                float scale, int dtype, void* workspace, size_t workspace_bytes,
                                int* dev_status, void* stream) {
  if (!lse || !dout || !dq || !dk || !dv || !workspace) return RA_ERR_NULL;
  if (P <= 0) return RA_ERR_SHAPE;
  if (H_q % P != 0 || H_kv % P != 0) return RA_ERR_SHAPE;
  if (dtype != RA_BF16) return RA_ERR_DTYPE;
  Geometry g;
  ra_status st = make_geometry(B, H_q, H_kv, S, D, P, causal, scale, RA_ORDER_CONTIGUOUS, -1,
                               tile_rows_for(dtype, D), &g);
  if (st != RA_OK) return st;
  st = check_attn_args(q, k, v, out, lse, B, H_q, H_kv, P * g.seg_len, D, dtype, -1, nullptr,
                       dev_status);
  if (st != RA_OK) return st;
  if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(workspace, 16))
    return RA_ERR_ALIGN;
  size_t need = 0;
  st = ring_attn_bwd_workspace(B, H_q, S, D, P, RA_ORDER_CONTIGUOUS, &need);
  if (st != RA_OK) return st;
  if (workspace_bytes < need) return RA_ERR_BUFFER;
  g.shard_rows = g.seg_len;
  int sms = 0;
  st = check_device(&sms);
  if (st != RA_OK) return st;
  return launch_attn_bwd(g, q, k, v, out, lse, dout, dq, dk, dv,
                         static_cast<float*>(workspace), RA_BWD_ALL, dev_status,
                         reinterpret_cast<cudaStream_t>(stream));
}

ra_status ring_attn_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                               float* lse, const int* cu_seqlens, int n_seq, int total,
                               int max_seqlen, int H_q, int H_kv, int D, int P, int causal,
                               float scale, int dtype, int order, int* dev_status,
                               void* stream) {
  if (!cu_seqlens) return RA_ERR_NULL;
  if (n_seq <= 0 || total <= 0 || max_seqlen <= 0) return RA_ERR_SHAPE;
  if (!aligned(cu_seqlens, 4)) return RA_ERR_ALIGN;
  ra_status st = check_attn_args(q, k, v, out, lse, 1, H_q, H_kv, total, D, dtype, -1,
                                 nullptr, dev_status);
  if (st != RA_OK) return st;
  if ((long long)n_seq * max_seqlen * H_q > kMaxElems) return RA_ERR_RANGE;
  Geometry g;
  st = make_geometry(n_seq, H_q, H_kv, max_seqlen, D, P, causal, scale, order, -1,
                     tile_rows_for(dtype, D), &g);
  if (st != RA_OK) return st;
  g.cu_seqlens = cu_seqlens;
  g.total = total;
  int sms = 0;
  st = check_device(&sms);
  if (st != RA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == RA_F32)
    return launch_attn_simt_varlen(g, static_cast<const float*>(q),
                                   static_cast<const float*>(k), static_cast<const float*>(v),
                                   static_cast<float*>(out), lse, dev_status, s);
  return launch_attn_tc_varlen(g, q, k, v, out, lse, dev_status, s);
}

ra_status ring_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* out,
                               const float* lse, const void* dout, void* dq, void* dk,
                               void* dv, const int* cu_seqlens, int n_seq, int total,
                               int max_seqlen, int H_q, int H_kv, int D, int P, int causal,
                               float scale, int dtype, int order, void* workspace,
                               size_t workspace_bytes, int* dev_status, void* stream) {
  if (!cu_seqlens || !lse || !dout || !dq || !dk || !dv || !workspace) return RA_ERR_NULL;
  if (n_seq <= 0 || total <= 0 || max_seqlen <= 0) return RA_ERR_SHAPE;
  if (!aligned(cu_seqlens, 4)) return RA_ERR_ALIGN;
  ra_status st = check_attn_args(q, k, v, out, lse, 1, H_q, H_kv, total, D, dtype, -1,
                                 nullptr, dev_status);
  if (st != RA_OK) return st;
  if (dtype != RA_BF16) return RA_ERR_DTYPE;
  if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(workspace, 16))
    return RA_ERR_ALIGN;
  if ((long long)n_seq * max_seqlen * H_q > kMaxElems) return RA_ERR_RANGE;
  Geometry g;
  st = make_geometry(n_seq, H_q, H_kv, max_seqlen, D, P, causal, scale, order, -1,
                     tile_rows_for(dtype, D), &g);
  if (st != RA_OK) return st;
  g.cu_seqlens = cu_seqlens;
  g.total = total;
  size_t need = 0;
  st = ring_attn_bwd_workspace(n_seq, H_q, max_seqlen, D, P, order, &need);
  if (st != RA_OK) return st;
  if (workspace_bytes < need) return RA_ERR_BUFFER;
  int sms = 0;
  st = check_device(&sms);
  if (st != RA_OK) return st;
  return launch_attn_bwd(g, q, k, v, out, lse, dout, dq, dk, dv,
                         static_cast<float*>(workspace), RA_BWD_ALL, dev_status,
                         reinterpret_cast<cudaStream_t>(stream));
}

ra_status attn_lse_merge_n(const void* const* o, const float* const* lse,
                           int n, void* out, float* out_lse, int B, int H,
                           int S, int D, int dtype, void* stream) {
  if (!o || !lse || !out || !out_lse) return RA_ERR_NULL;
  if (n < 1 || n > RA_MERGE_MAX_N) return RA_ERR_SHAPE;
  if (dtype != RA_BF16 && dtype != RA_F32) return RA_ERR_DTYPE;
  if (B <= 0 || H <= 0 || S <= 0) return RA_ERR_SHAPE;
  if (D != 32 && D != 64 && D != 128 && D != 256) return RA_ERR_HEADDIM;
  MergeArgs a = {};
  for (int i = 0; i < n; ++i) {
    if (!o[i] || !lse[i]) return RA_ERR_NULL;
    if (!aligned(o[i], 16) || !aligned(lse[i], 4)) return RA_ERR_ALIGN;
    a.o[i] = o[i];
    a.lse[i] = lse[i];
  }
  if (!aligned(out, 16) || !aligned(out_lse, 4)) return RA_ERR_ALIGN;
  if ((long long)B * S * H * D > kMaxElems) return RA_ERR_RANGE;
  a.n = n;
  a.out = out;
  a.out_lse = out_lse;
  a.B = B; a.H = H; a.S = S; a.D = D;
  int sms = 0;
  ra_status st = check_device(&sms);
  if (st != RA_OK) return st;
  return launch_merge(a, dtype, sms, reinterpret_cast<cudaStream_t>(stream));
}

ra_status attn_lse_merge(const void* o_a, const float* lse_a, const void* o_b,
                         const float* lse_b, void* out, float* lse, int B,
                         int H, int S, int D, int dtype, void* stream) {
  const void* o[2] = {o_a, o_b};
  const float* l[2] = {lse_a, lse_b};
  return attn_lse_merge_n(o, l, 2, out, lse, B, H, S, D, dtype, stream);
}

}  // extern "C"
