// Standalone log-sum-exp merge of n partial attention results.
//
// Glossary "sequence parallelism transformers", §Ring Attention (a rank
// accumulates the outputs of every received block) and §Implementation
// Considerations ("Numerical Stability"): partial results over disjoint key
// sets combine exactly as
//     lse = M + log sum_t exp(lse_t - M),   M = max_t lse_t
//     out = sum_t exp(lse_t - lse) * o_t
// This kernel is bound by HBM bandwidth: per row it reads n * (D*esz + 4)
// bytes and writes D*esz + 4 bytes, and does O(n*D) flops.
//
// Mapping: one warp owns a block of 32 consecutive sequence positions of one
// (batch, head). Lane i reads the n lse values of position s0+i (coalesced
// 128-byte reads of the [B, H, S] lse tensors), computes the n weights, then
// the warp walks the 32 rows; each row of D elements is split into 16-byte
// vectors spread over the lanes, with all n vector loads of a lane issued
// before they are combined. Outputs and partials are streamed (read once,
// written once), so loads and stores bypass L1 and are marked evict-first.
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4* p, float4 v) { __stcs(p, v); }

// 16 bytes of the row as 4 floats (f32) or 8 floats (bf16).
template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int kElems = 4;
  __device__ static void load(const void* p, float* f) {
    float4 v = ld_stream(reinterpret_cast<const float4*>(p));
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  __device__ static void store(void* p, const float* f) {
    st_stream(reinterpret_cast<float4*>(p), make_float4(f[0], f[1], f[2], f[3]));
  }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ static void load(const void* p, float* f) {
    float4 v = ld_stream(reinterpret_cast<const float4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ static void store(void* p, const float* f) {
    float4 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    st_stream(reinterpret_cast<float4*>(p), v);
  }
};

// VECS: 16-byte vectors per row (D * sizeof(T) / 16), a power of two.
template <typename T, int VECS, int MAXN>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
lse_merge_kernel(MergeArgs a) {
  constexpr int kLanesPerRow = VECS < 32 ? VECS : 32;
  constexpr int kRowsPerPass = 32 / kLanesPerRow;
  constexpr int kVecPerLane = VECS / kLanesPerRow;
  constexpr int E = Vec<T>::kElems;

  const int lane = threadIdx.x & 31;
  const int warp_global = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int n_warps = gridDim.x * kWarpsPerBlock;
  const int blocks_per_bh = (a.S + 31) / 32;
  const long long n_tasks = (long long)a.B * a.H * blocks_per_bh;
  const int n = a.n;

  for (long long task = warp_global; task < n_tasks; task += n_warps) {
    const int bh = (int)(task / blocks_per_bh);
    const int s0 = (int)(task % blocks_per_bh) * 32;
    const int b = bh / a.H, h = bh % a.H;
    const int s = s0 + lane;
    const bool valid = s < a.S;
    const long long lse_off = (long long)bh * a.S + s;

    // weights exp(lse_t - lse) of row s, computed by lane (s - s0)
    float w[MAXN];
    float m = -INFINITY;
#pragma unroll
    for (int t = 0; t < MAXN; ++t) {
      w[t] = (t < n && valid) ? __ldcs(a.lse[t] + lse_off) : -INFINITY;
      m = fmaxf(m, w[t]);
    }
    const float m_safe = (m == -INFINITY) ? 0.f : m;
    float z = 0.f;
#pragma unroll
    for (int t = 0; t < MAXN; ++t) {
      w[t] = expf(w[t] - m_safe);     // exp(-inf) = 0
      z += w[t];
    }
    const float inv_z = z > 0.f ? 1.f / z : 0.f;
#pragma unroll
    for (int t = 0; t < MAXN; ++t) w[t] *= inv_z;
    const float lse_out = z > 0.f ? m_safe + logf(z) : -INFINITY;

    // rows s0 .. s0+31, kRowsPerPass at a time
    const int rows = min(32, a.S - s0);
    const int sub = lane / kLanesPerRow;        // which row of the pass
    const int l_in = lane % kLanesPerRow;       // lane within the row
    for (int r0 = 0; r0 < 32; r0 += kRowsPerPass) {
      const int r = r0 + sub;
      float wr[MAXN];
#pragma unroll
      for (int t = 0; t < MAXN; ++t) wr[t] = __shfl_sync(0xffffffffu, w[t], r & 31);
      if (r >= rows) continue;
      const long long row_off = ((long long)b * a.S + (s0 + r)) * a.H + h;
      const size_t row_bytes = (size_t)a.D * sizeof(T);
#pragma unroll
      for (int vv = 0; vv < kVecPerLane; ++vv) {
        const size_t byte_off = row_off * row_bytes + (size_t)(vv * kLanesPerRow + l_in) * 16;
        float in[MAXN][E];
#pragma unroll
        for (int t = 0; t < MAXN; ++t)
          if (t < n)
            Vec<T>::load(static_cast<const char*>(a.o[t]) + byte_off, in[t]);
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
        for (int t = 0; t < MAXN; ++t)
          if (t < n) {
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(wr[t], in[t][e], acc[e]);
          }
        Vec<T>::store(static_cast<char*>(a.out) + byte_off, acc);
      }
    }
    if (valid) a.out_lse[lse_off] = lse_out;
  }
}

template <typename T, int VECS>
ra_status launch_typed(const MergeArgs& a, int sm_count, cudaStream_t stream) {
  const long long tasks = (long long)a.B * a.H * ((a.S + 31) / 32);
  long long blocks = (tasks + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const long long cap = (long long)sm_count * 8;    // 64 warps per SM resident
  if (blocks > cap) blocks = cap;
  if (a.n <= 2)
    lse_merge_kernel<T, VECS, 2><<<(int)blocks, kWarpsPerBlock * 32, 0, stream>>>(a);
  else if (a.n <= 4)
    lse_merge_kernel<T, VECS, 4><<<(int)blocks, kWarpsPerBlock * 32, 0, stream>>>(a);
  else if (a.n <= 8)
    lse_merge_kernel<T, VECS, 8><<<(int)blocks, kWarpsPerBlock * 32, 0, stream>>>(a);
  else
    lse_merge_kernel<T, VECS, 16><<<(int)blocks, kWarpsPerBlock * 32, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_LAUNCH;
}

template <typename T>
ra_status launch_d(const MergeArgs& a, int sm_count, cudaStream_t stream) {
  constexpr int per = 16 / sizeof(T);
  switch (a.D / per) {
    case 32 / per: return launch_typed<T, 32 / per>(a, sm_count, stream);
    case 64 / per: return launch_typed<T, 64 / per>(a, sm_count, stream);
    case 128 / per: return launch_typed<T, 128 / per>(a, sm_count, stream);
    case 256 / per: return launch_typed<T, 256 / per>(a, sm_count, stream);
    default: return RA_ERR_HEADDIM;
  }
}

}  // namespace

ra_status launch_merge(const MergeArgs& a, int dtype, int sm_count,
                       cudaStream_t stream) {
  if (dtype == RA_F32) return launch_d<float>(a, sm_count, stream);
  return launch_d<__nv_bfloat16>(a, sm_count, stream);
}

}  // namespace ra
