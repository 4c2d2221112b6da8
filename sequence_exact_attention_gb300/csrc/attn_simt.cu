// Exact float32 ring attention on the CUDA cores (FMA pipe).
//
// The float32 workload is held to 1e-4 against the float64 definition, which
// rules out TF32 tensor-core products; this kernel keeps every product and
// sum in IEEE float32 and uses the accurate exp2f/log2f.
//
// Ring structure (glossary "sequence parallelism transformers", §Ring
// Attention): a block owns one query tile of 64 rows of one (batch, head)
// inside the segment of virtual rank r, and walks the key tiles of steps
// t = 0..P-1 in ring order (source rank (r - t) mod P). Per key tile it
// computes the 64 scores of each row, folds them into the running row state
// (max m, sum l, unnormalised output acc) -- the log-sum-exp merge of the
// per-tile partial results, done in registers -- and at the end writes
// out = acc / l and lse = ln(2) * (m + log2 l).
//
// Mapping: 256 threads = 64 rows x 4 threads. The 4 threads of a row split D
// in interleaved 16-byte vectors (thread p owns vectors p, p+4, ...), so a
// key row read from shared memory is one contiguous 64-byte broadcast per
// row group; partial dot products are combined with two xor-shuffles.
#include <cmath>
#include <cstdint>

#include "checks.cuh"
#include "ra_internal.h"
#include "ring_iter.cuh"

namespace ra {
namespace {

constexpr int kRows = 64;        // query / key tile rows
constexpr int kThreads = 256;    // 4 threads per query row

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

template <int D, bool kVarlen>
__global__ void __launch_bounds__(kThreads)
attn_simt_kernel(const Geometry gp, const float* __restrict__ q,
                 const float* __restrict__ k, const float* __restrict__ v,
                 float* __restrict__ out, float* __restrict__ lse,
                 int* __restrict__ vlog, int log_stride, int* __restrict__ status) {
  constexpr int V4 = D / 4;          // float4 per row
  constexpr int NV = V4 / 4;         // float4 per thread
  extern __shared__ float4 smem[];
  float4* Ks = smem;                 // [kRows][V4]
  float4* Vs = smem + kRows * V4;    // [kRows][V4]

  // With packed variable-length sequences, b is the sequence and the grid is
  // sized by the longest one; `g` is then this sequence's own geometry.
  const int BH = gp.B * gp.H_q;
  const int bh = blockIdx.x % BH;
  const int n_qt = gp.n_seg * gp.nt;
  const int qid = n_qt - 1 - blockIdx.x / BH;    // later positions first
  const int seg = qid / gp.nt, ti = qid % gp.nt;
  const int b = bh / gp.H_q, h = bh % gp.H_q;
  Geometry gv;
  int row0 = 0;
  if constexpr (kVarlen) varlen_geometry(gp, b, gv, row0, threadIdx.x == 0 ? status : nullptr);
  const Geometry& g = kVarlen ? gv : gp;
  const int q_lo = seg * g.seg_len + ti * kRows;
  const int q_valid = tile_tokens(g, seg, ti);     // <= 0: a tile of padding only
  const int r = seg_owner(g, seg);
  const int hk = h / (g.H_q / g.H_kv);
  // first row of this sequence in q, k, v, out, and its first lse entry; in
  // the sequence-sharded layout [P, B, C, H, D] the rows of segment p of
  // batch b start at ((p * B + b) * C - p * C) + position
  const bool sharded = !kVarlen && gp.shard_rows > 0;
  const size_t C_rows = (size_t)gp.shard_rows;
  size_t srow = kVarlen ? (size_t)row0 : (size_t)b * gp.S;
  size_t lrow = kVarlen ? (size_t)h * gp.total + row0 : (size_t)bh * gp.S;
  size_t qrow0 = srow;
  if (sharded) {
    const size_t lb = (size_t)seg * gp.B + b;
    qrow0 = lb * C_rows - (size_t)seg * C_rows;
    lrow = (lb * gp.H_q + h) * C_rows - (size_t)seg * C_rows;
  }

  const int row = threadIdx.x >> 2, part = threadIdx.x & 3;
  const int q_pos = q_lo + row;
  const bool row_valid = row < q_valid;

  // the visit log of this query tile: [count, 4 ints per visit]
  const long long log_off = ((long long)bh * n_qt + qid) * log_stride;
  const long long log_len = (long long)gp.B * gp.H_q * n_qt * log_stride;
  if (q_valid <= 0) {            // a tile of padding only: nothing to compute or write
    if (vlog && threadIdx.x == 0 && in_range(log_off, 1, log_len, status)) vlog[log_off] = 0;
    return;
  }

  float4 qv[NV], acc[NV];
  const long long q_elem = ((long long)(qrow0 + (row_valid ? q_pos : q_lo)) * g.H_q + h) * D;
  const bool row_ok = row_valid && in_range(q_elem, D, extent_q(gp), status);
  const float4* qrow = reinterpret_cast<const float4*>(q + q_elem);
#pragma unroll
  for (int e = 0; e < NV; ++e) {
    qv[e] = row_ok ? qrow[part + 4 * e] : make_float4(0.f, 0.f, 0.f, 0.f);
    acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = -INFINITY, l = 0.f;

  int* log_base = vlog ? vlog + log_off : nullptr;
  int n_vis = 0;

  KvIter it;
  it.init(g, r, q_lo, q_valid);
  KvTile kv;
  while (it.next(g, kv)) {
    const int work = kv.work;
    if (log_base && threadIdx.x == 0 && in_range(log_off + 1 + 4 * n_vis, 4, log_len, status))
      log_visit(log_base, n_vis, kv, tile_class(g, q_lo, kv));
    ++n_vis;

    __syncthreads();    // the previous tile is no longer read
    const size_t krow0 =
        sharded ? ((size_t)kv.seg * gp.B + b) * C_rows - (size_t)kv.seg * C_rows : srow;
    for (int idx = threadIdx.x; idx < kRows * V4; idx += kThreads) {
      const int kr = idx / V4, c = idx % V4;
      float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
      const size_t off = ((krow0 + kv.lo + kr) * g.H_kv + hk) * V4 + c;
      if (kr < kv.valid && in_range((long long)off * 4, 4, extent_kv(gp), status)) {
        kk = reinterpret_cast<const float4*>(k)[off];
        vv = reinterpret_cast<const float4*>(v)[off];
      }
      Ks[idx] = kk;
      Vs[idx] = vv;
    }
    __syncthreads();

    float s[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      float p = 0.f;
#pragma unroll
      for (int e = 0; e < NV; ++e) p = dot4(qv[e], Ks[j * V4 + part + 4 * e], p);
      p += __shfl_xor_sync(0xffffffffu, p, 1);
      p += __shfl_xor_sync(0xffffffffu, p, 2);
      s[j] = p;
    }
    if (work == kMask) {
#pragma unroll
      for (int j = 0; j < kRows; ++j)
        if (j >= kv.valid || (g.causal && kv.lo + j > q_pos)) s[j] = -INFINITY;
    }
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kRows; ++j) mx = fmaxf(mx, s[j]);
    const float m_new = fmaxf(m, mx * g.scale_log2);
    const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    l *= alpha;
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      acc[e].x *= alpha; acc[e].y *= alpha; acc[e].z *= alpha; acc[e].w *= alpha;
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const float p = exp2f(fmaf(s[j], g.scale_log2, -m_use));
      l += p;
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const float4 vv = Vs[j * V4 + part + 4 * e];
        acc[e].x = fmaf(p, vv.x, acc[e].x);
        acc[e].y = fmaf(p, vv.y, acc[e].y);
        acc[e].z = fmaf(p, vv.z, acc[e].z);
        acc[e].w = fmaf(p, vv.w, acc[e].w);
      }
    }
    m = m_new;
  }

  if (row_ok) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float4* orow = reinterpret_cast<float4*>(
        out + ((qrow0 + q_pos) * g.H_q + h) * D);
#pragma unroll
    for (int e = 0; e < NV; ++e)
      orow[part + 4 * e] = make_float4(acc[e].x * inv, acc[e].y * inv,
                                       acc[e].z * inv, acc[e].w * inv);
    if (part == 0 && lse && in_range((long long)(lrow + q_pos), 1, extent_lse(gp), status))
      lse[lrow + q_pos] =
          l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
  if (log_base && threadIdx.x == 0 && in_range(log_off, 1, log_len, status)) log_base[0] = n_vis;
}

template <int D, bool kVarlen = false>
ra_status launch_d(const Geometry& g, const float* q, const float* k,
                   const float* v, float* out, float* lse, int* vlog,
                   int log_stride, int* status, cudaStream_t stream) {
  const int smem = 2 * kRows * D * (int)sizeof(float);
  if (cudaFuncSetAttribute(attn_simt_kernel<D, kVarlen>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return RA_ERR_LAUNCH;
  const long long grid = (long long)g.n_seg * g.nt * g.B * g.H_q;
  if (grid > 0x7fffffffLL) return RA_ERR_RANGE;
  attn_simt_kernel<D, kVarlen><<<(unsigned)grid, kThreads, smem, stream>>>(
      g, q, k, v, out, lse, vlog, log_stride, status);
  return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_LAUNCH;
}

}  // namespace

ra_status launch_attn_simt_varlen(const Geometry& g, const float* q, const float* k,
                                  const float* v, float* out, float* lse, int* dev_status,
                                  cudaStream_t stream) {
  if (g.D == 64) return launch_d<64, true>(g, q, k, v, out, lse, nullptr, 0, dev_status, stream);
  return launch_d<128, true>(g, q, k, v, out, lse, nullptr, 0, dev_status, stream);
}

ra_status launch_attn_simt_sharded(const Geometry& g, const float* q, const float* k,
                                   const float* v, float* out, float* lse, int* dev_status,
                                   cudaStream_t stream) {
  if (g.D == 64) return launch_d<64>(g, q, k, v, out, lse, nullptr, 0, dev_status, stream);
  return launch_d<128>(g, q, k, v, out, lse, nullptr, 0, dev_status, stream);
}

ra_status launch_attn_simt(const Geometry& g, const float* q, const float* k,
                           const float* v, void* out, float* lse,
                           int* visit_log, int log_stride, int* dev_status,
                           cudaStream_t stream) {
  float* o = static_cast<float*>(out);
  if (g.D == 64) return launch_d<64>(g, q, k, v, o, lse, visit_log, log_stride, dev_status, stream);
  return launch_d<128>(g, q, k, v, o, lse, visit_log, log_stride, dev_status, stream);
}

}  // namespace ra
