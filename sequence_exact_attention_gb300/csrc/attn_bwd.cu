// Backward pass of exact ring attention on the tensor cores: bf16 in and
// out, float32 accumulation in tensor memory.
//
// Glossary "sequence parallelism transformers", §Implementation
// Considerations: the backward pass runs over the same ring as the forward.
// For an upstream gradient dO and the forward's lse, with
// p_ij = exp(s_ij - lse_i) on the allowed pairs:
//   dV_j = sum_i p_ij dO_i            ds_ij = p_ij (<dO_i, v_j> - delta_i)
//   dQ_i = scale sum_j ds_ij k_j      dK_j = scale sum_i ds_ij q_i
//   delta_i = <dO_i, o_i>
// Three launches on the caller's stream:
//  1. bwd_prep_kernel: per query row, -lse in base 2 and -delta (negated, so
//     that the gradient kernels add them with packed FMAs), into the
//     caller's workspace, tile-padded (padding rows get -lse = -inf, which
//     makes their p exactly 0, and -delta = 0).
//  2. bwd_dkdv_kernel: one CTA per key tile of one kv head. It walks the
//     query tiles that see the tile in ring order -- the owner rank's own
//     queries first (step 0), then ranks src+1, src+2, ... (the block's trip
//     around the ring back to its owner) -- over every query head of the
//     group. Per visit:
//       S^T = K Q^T, dP^T = V dO^T      tensor cores, float32 in TMEM
//       P^T, dS^T in bf16               CUDA cores, one thread per key row
//       dV += P^T dO, dK += dS^T Q      tensor cores, A operand from TMEM
//  3. bwd_dq_kernel: one CTA per query tile, walking the key tiles in the
//     forward's ring order: S = Q K^T, dP = dO V^T, dS, dQ += dS K.
// The two gradient kernels both recompute S and dP; in exchange neither needs
// atomics, and each gradient is accumulated on chip and written once.
//
// Roles (320 threads): warps 0-7 compute (TMEM lane quarter = warp mod 4,
// column half = warp / 4), warp 8 TMA producer, warp 9 tensor-core issuer
// and TMEM owner. Every wait is
// bounded (two seconds, then the CTA gives up, drains what it issued, frees
// its TMEM and reports RA_ERR_TIMEOUT in the status word).
#include <cuda.h>
#include <cuda_bf16.h>

#include "checks.cuh"
#include "fastmath.cuh"
#include "q_iter.cuh"
#include "ra_internal.h"
#include "ring_iter.cuh"
#include "sm100.cuh"

namespace ra {
namespace {

using namespace sm100;
using namespace fastmath;

constexpr int kT = 128;                         // tile rows (queries or keys)
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                   // S or S^T, then P / dS in bf16
constexpr uint32_t kColDP = 128;                // dP or dP^T, then dS^T in bf16
constexpr uint32_t kColAcc = 256;               // accumulators: dV | dK, or dQ
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kBoxBytes = kT * 64 * 2;          // one TMA box: 128 rows x 64 bf16
constexpr float kLog2e = 1.4426950408889634f;

// dK/dV kernel: K and V stay resident; each visit's Q, dO and statistics
// arrive together in a two-stage ring.
template <int D>
struct Cfg {
  static constexpr int kTileBytes = kT * D * 2;
  static constexpr int kBoxes = D / 64;
  static constexpr int kFixA = 0;                          // K
  static constexpr int kFixB = kTileBytes;                 // V
  static constexpr int kStage0 = 2 * kTileBytes;
  static constexpr int kStatBytes = 2 * kT * 4;            // lse2 and delta of a query tile
  static constexpr int kStageBytes = 2 * kTileBytes + kStatBytes;
  static constexpr int kBarOff = kStage0 + 2 * kStageBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kUsed = kBarOff + kBarBytes + 1024;  // + alignment slack
  // More than half an SM's shared memory: one CTA per SM, so the 512-column
  // TMEM allocation never waits for another CTA.
  static constexpr int kSmemBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
  static constexpr int bFix = 0;
  static constexpr int bFull = 1;     // [2] stage's Q and lse2 loaded
  static constexpr int bFree = 3;     // [2] stage no longer read by the tensor cores
  static constexpr int bS = 5;        // S^T in TMEM
  static constexpr int bDP = 6;       // dP^T in TMEM
  static constexpr int bP = 7;        // 256 arrivals: pass 1 done (P^T stored)
  static constexpr int bDS = 8;       // 256 arrivals: pass 2 done (dS^T stored)
  static constexpr int bAccK = 10;    // the last visit's dV and dK done
  static constexpr int bFinal = 11;
  static constexpr int bFullDO = 12;  // [2] stage's dO and delta loaded
  static constexpr int kHolderOff = kBarBytes - 16;
  static constexpr int kNeverOff = kBarBytes - 12;
  static constexpr int kAbortOff = kBarBytes - 8;
  static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// dQ kernel: Q and dO stay resident; keys and values arrive in rings of
// their own, since K_j is read until dQ(j) (three slots) and V_j only by
// dP(j) (two slots), so each slot is refilled as soon as its last product
// is done and the next tile has landed before the issuer needs it.
template <int D>
struct CfgQ {
  static constexpr int kTileBytes = kT * D * 2;
  static constexpr int kBoxes = D / 64;
  static constexpr int kKBuf = 3;
  static constexpr int kVBuf = 2;
  static constexpr int kFixA = 0;                          // Q
  static constexpr int kFixB = kTileBytes;                 // dO
  static constexpr int kK0 = 2 * kTileBytes;
  static constexpr int kV0 = kK0 + kKBuf * kTileBytes;
  static constexpr int kBarOff = kV0 + kVBuf * kTileBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kUsed = kBarOff + kBarBytes + 1024;  // + alignment slack
  // one CTA per SM, as in the other kernels
  static constexpr int kSmemBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
  static constexpr int bFix = 0;
  static constexpr int bKFull = 1;                // [kKBuf]
  static constexpr int bKFree = bKFull + kKBuf;   // [kKBuf] dQ of the slot's tile done
  static constexpr int bVFull = bKFree + kKBuf;   // [kVBuf]
  static constexpr int bVFree = bVFull + kVBuf;   // [kVBuf] dP of the slot's tile done
  static constexpr int bS = bVFree + kVBuf;       // S in TMEM
  static constexpr int bDP = bS + 1;              // dP in TMEM
  static constexpr int bP = bDP + 1;              // 256 arrivals: pass 1 has read S
  static constexpr int bDS = bP + 1;              // 256 arrivals: pass 2 done (dS stored)
  static constexpr int bAccB = bDS + 1;           // [2] dQ MMA of a visit done, per dS buffer
  static constexpr int bFinal = bAccB + 2;
  static constexpr int kNumBars = bFinal + 1;
  static constexpr int kHolderOff = kBarBytes - 16;
  static constexpr int kNeverOff = kBarBytes - 12;
  static constexpr int kAbortOff = kBarBytes - 8;
  static_assert(kNumBars * 8 <= kHolderOff, "barrier area overflow");
  static_assert(kColAcc + D + 128 <= kTmemCols, "two dS buffers after dQ");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Offset (in floats) of the first row of query tile `ti` of segment `seg`,
// batch-head `bh`, in each half of the workspace.
__host__ __device__ __forceinline__ long long ws_tile(const Geometry& g, int bh, int seg,
                                                      int ti) {
  return (((long long)bh * g.n_seg + seg) * g.nt + ti) * kT;
}

// TMEM column (relative to the S or dP range) of the bf16 operand columns
// that K step kk (16 rows of the reduction) reads: the two 64-column halves
// keep their 32 packed columns at the start of their own range.
__device__ __forceinline__ uint32_t pcol(int kk) {
  return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8);
}

// dQ kernel: the two dS buffers (64 bf16-pair columns each) follow the dQ
// accumulator; within a buffer the key half hf keeps its 32 columns at
// hf * 32, so K step kk (16 keys) reads columns (kk / 4) * 32 + (kk % 4) * 8.
template <int D>
__host__ __device__ constexpr uint32_t kColDSq() { return kColAcc + D; }
__device__ __forceinline__ uint32_t dscol(int kk) {
  return (uint32_t)((kk >> 2) * 32 + (kk & 3) * 8);
}

template <class C, class BarFn>
__device__ __forceinline__ void init_barriers(BarFn bar, volatile int* abort_flag,
                                              volatile int* never) {
  if (threadIdx.x == 0) {
    mbar_init(bar(C::bFix), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::bFull + i), 1);
      mbar_init(bar(C::bFullDO + i), 1);
      mbar_init(bar(C::bFree + i), 1);
    }
    mbar_init(bar(C::bS), 1);
    mbar_init(bar(C::bDP), 1);
    mbar_init(bar(C::bP), 256);
    mbar_init(bar(C::bDS), 256);
    mbar_init(bar(C::bAccK), 1);
    mbar_init(bar(C::bFinal), 1);
    *abort_flag = 0;
    *never = 0;
    fence_mbar_init();
  }
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// ------------------------------------------------------------------ prep
// 8 threads per padded query row; each reads D/8 elements of out and dout.
template <int D, bool kVarlen>
__global__ void __launch_bounds__(256)
bwd_prep_kernel(const Geometry gp, const __nv_bfloat16* __restrict__ out,
                const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
                float* __restrict__ lse2, float* __restrict__ delta, long long rows,
                int* __restrict__ status) {
  const long long gid = (long long)blockIdx.x * 32 + (threadIdx.x >> 3);
  const int sub = threadIdx.x & 7;
  if (gid >= rows) return;               // rows is a multiple of 32: whole blocks
  // the workspace is laid out by the grid's geometry (longest sequence);
  // positions follow the row's own sequence
  const int row = (int)(gid % kT);
  long long rest = gid / kT;
  const int ti = (int)(rest % gp.nt);
  rest /= gp.nt;
  const int seg = (int)(rest % gp.n_seg);
  const int bh = (int)(rest / gp.n_seg);
  const int b = bh / gp.H_q, h = bh % gp.H_q;
  Geometry gv;
  int row0 = 0;
  if constexpr (kVarlen) varlen_geometry(gp, b, gv, row0, threadIdx.x == 0 ? status : nullptr);
  const Geometry& g = kVarlen ? gv : gp;
  const size_t srow = seg_rows(gp, b, seg, row0, kVarlen).grow;
  const size_t lrow = lse_base(gp, b, h, seg, row0, kVarlen);
  const int in_seg = ti * kT + row;
  const bool valid = in_seg < seg_tokens(g, seg);
  const int pos = seg * g.seg_len + in_seg;
  float acc = 0.f;
  constexpr int E = D / 8;
  const size_t off = ((srow + pos) * g.H_q + h) * D + (size_t)sub * E;
  if (valid && in_range((long long)off, E, extent_q(gp), status)) {
    const uint4* po = reinterpret_cast<const uint4*>(out + off);
    const uint4* pd = reinterpret_cast<const uint4*>(dout + off);
#pragma unroll
    for (int v = 0; v < E / 8; ++v) {
      const uint4 a = po[v], d = pd[v];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        acc = fmaf(bf_lo(aw[w]), bf_lo(dw[w]), acc);
        acc = fmaf(bf_hi(aw[w]), bf_hi(dw[w]), acc);
      }
    }
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  if (sub == 0) {
    const bool lse_ok = valid && in_range((long long)(lrow + pos), 1, extent_lse(gp), status);
    lse2[gid] = lse_ok ? -(lse[lrow + pos] * kLog2e) : -INFINITY;
    delta[gid] = valid ? -acc : 0.f;
  }
}

// ------------------------------------------------------------------ query walk
using QIter = QIterT<kT>;     // csrc/q_iter.cuh

// K-major SW128 descriptor offset of K step kk (16 elements) in a tile made
// of 64-column boxes.
__device__ __forceinline__ uint64_t kstep_off(int kk) {
  return (uint64_t)(((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4);
}

// Stores 32 float32 values of one row, times `mul`, as bf16 (64 bytes).
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&u)[32],
                                            float mul) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    w[i] = pack_bf16x2(__uint_as_float(u[2 * i]) * mul, __uint_as_float(u[2 * i + 1]) * mul);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// ------------------------------------------------------------------ dK, dV
// Per visit the tensor cores run S^T, dP^T, dV, dK in that order and the
// compute warps run two passes: P^T (from S^T) while dP^T is computed, then
// dS^T (from dP^T and the P^T kept in registers) while dV is accumulated.
// Warp w covers key rows 32 (w mod 4) .. +31 and query columns 64 (w / 4)
// .. +63; its bf16 P^T and dS^T go into the first 32 columns of its own
// S^T and dP^T column ranges, so no warp writes columns another one reads.
template <int D, bool kVarlen>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_do, const Geometry gp,
                const float* __restrict__ lse2, const float* __restrict__ delta,
                __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                int* __restrict__ status) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  auto bar = [&](int i) -> uint32_t { return base + C::kBarOff + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kBarOff + C::kAbortOff);
  volatile int* never = reinterpret_cast<volatile int*>(base_ptr + C::kBarOff + C::kNeverOff);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + C::kBarOff + C::kHolderOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work item: key tile kt of kv head hk; (batch, kv head) outermost so that
  // the CTAs resident together read the queries of one group from L2; key
  // tiles in position order (most causal work first).
  const int grp = gp.H_q / gp.H_kv;
  const int n_kt = gp.n_seg * gp.nt;
  const int kt = (int)(blockIdx.x % n_kt);
  const int bhk = (int)(blockIdx.x / n_kt);
  const int b = bhk / gp.H_kv, hk = bhk % gp.H_kv;
  const int kseg = kt / gp.nt, kti = kt % gp.nt;
  // packed variable-length sequences: b is the sequence, `g` its geometry
  Geometry gv;
  int row0 = 0;
  if constexpr (kVarlen) varlen_geometry(gp, b, gv, row0, threadIdx.x == 0 ? status : nullptr);
  const Geometry& g = kVarlen ? gv : gp;
  const SegRows kr = seg_rows(gp, b, kseg, row0, kVarlen);   // the key tile's rows
  const int src = seg_owner(g, kseg);
  const int kv_lo = kseg * g.seg_len + kti * kT;
  const int kv_valid = tile_tokens(g, kseg, kti);   // <= 0: padding only
  const int h0 = hk * grp;
  if (kv_valid <= 0) return;     // no key, no gradient row: the CTA leaves at once

  init_barriers<C>(bar, abort_flag, never);
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::bFix), 2 * C::kTileBytes);
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_4d(base + C::kFixA + bx * kBoxBytes, &tm_k, bar(C::bFix), bx * 64, hk,
                    kr.trow + kv_lo, kr.tbat);
        tma_load_4d(base + C::kFixB + bx * kBoxBytes, &tm_v, bar(C::bFix), bx * 64, hk,
                    kr.trow + kv_lo, kr.tbat);
      }
      QIter it;
      it.init(g, src, kv_lo, kv_valid, h0, h0 + grp);
      QTile qt;
      int j = 0;
      while (it.next(g, qt)) {
        const int st = j & 1;
        if (j >= 2 &&
            !mbar_wait(bar(C::bFree + st), (uint32_t)((j >> 1) - 1) & 1, abort_flag, kTimeoutNs))
          break;
        const uint32_t sb = base + C::kStage0 + st * C::kStageBytes;
        const SegRows qr = seg_rows(gp, b, qt.seg, row0, kVarlen);
        long long wi = ws_tile(gp, b * gp.H_q + qt.h, qt.seg, qt.ti);
        if (!in_range(wi, kT, ws_tile(gp, gp.B * gp.H_q, 0, 0), status)) wi = 0;
        // Q and lse2 first, on a barrier of their own: S^T needs only them;
        // dO and delta follow for dP^T and the second pass
        mbar_arrive_expect_tx(bar(C::bFull + st), C::kTileBytes + kT * 4);
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_4d(sb + bx * kBoxBytes, &tm_q, bar(C::bFull + st), bx * 64, qt.h,
                      qr.trow + qt.lo, qr.tbat);
        bulk_load(sb + 2 * C::kTileBytes, lse2 + wi, kT * 4, bar(C::bFull + st));
        mbar_arrive_expect_tx(bar(C::bFullDO + st), C::kTileBytes + kT * 4);
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_4d(sb + C::kTileBytes + bx * kBoxBytes, &tm_do, bar(C::bFullDO + st), bx * 64,
                      qt.h, qr.trow + qt.lo, qr.tbat);
        bulk_load(sb + 2 * C::kTileBytes + kT * 4, delta + wi, kT * 4, bar(C::bFullDO + st));
        ++j;
      }
      // every issued copy lands before the CTA leaves
      for (int jj = (j > 2 ? j - 2 : 0); jj < j; ++jj) {
        mbar_wait(bar(C::bFull + (jj & 1)), (uint32_t)(jj >> 1) & 1, never, kTimeoutNs);
        mbar_wait(bar(C::bFullDO + (jj & 1)), (uint32_t)(jj >> 1) & 1, never, kTimeoutNs);
      }
      mbar_wait(bar(C::bFix), 0, never, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // The whole warp runs the issuer's loop, so its descriptor arithmetic is
    // warp-uniform; one elected lane issues every MMA and commit (a commit
    // tracks the MMAs of the thread that issues it).
    {
      const bool leader = elect_one_sync();
      constexpr uint32_t id_s = idesc_bf16_f32(128, kT, false);
      constexpr uint32_t id_acc = idesc_bf16_f32(128, D, true);
      const uint64_t k_kmaj = sw128_desc(base + C::kFixA, 16, 1024);
      const uint64_t v_kmaj = sw128_desc(base + C::kFixB, 16, 1024);
      const uint64_t q_kmaj = sw128_desc(base + C::kStage0, 16, 1024);
      const uint64_t do_kmaj = sw128_desc(base + C::kStage0 + C::kTileBytes, 16, 1024);
      const uint64_t q_mn = sw128_desc(base + C::kStage0, kBoxBytes, 1024);
      const uint64_t do_mn = sw128_desc(base + C::kStage0 + C::kTileBytes, kBoxBytes, 1024);
      bool ok = mbar_wait_warp(bar(C::bFix), 0, abort_flag, kTimeoutNs);
      QIter it;
      it.init(g, src, kv_lo, kv_valid, h0, h0 + grp);
      QTile qt;
      // S^T(j+1) is issued as soon as dV(j) has read P^T(j) (they share
      // columns), before dK(j): the next P^T pass then overlaps dK(j) and
      // dP^T(j+1).
      auto issue_s = [&](int jj) {
        const uint64_t qb = q_kmaj + (uint64_t)(((jj & 1) * C::kStageBytes) >> 4);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + kColS, k_kmaj + kstep_off(kk), qb + kstep_off(kk), id_s,
                    kk > 0 ? 1u : 0u);
          umma_commit(bar(C::bS));
        }
        __syncwarp();
      };
      bool have = ok && it.next(g, qt);
      if (have) {
        ok = mbar_wait_warp(bar(C::bFull + 0), 0, abort_flag, kTimeoutNs);
        if (ok) {
          tc_fence_after();
          issue_s(0);
        }
      }
      // dP^T(j) overwrites the dS^T(j-1) that dK(j-1) reads, and S^T(j+1)
      // the P^T(j) that dV(j) reads: one thread issues both pairs in that
      // order and the tensor core executes one thread's MMAs in issue order,
      // so neither waits for the other to complete (a wait would drain the
      // tensor core: it holds only the few MMAs queued behind the last issue).
      int j = 0;
      while (ok && have) {
        const int st = j & 1;
        const uint64_t so = (uint64_t)((st * C::kStageBytes) >> 4);
        const uint64_t dob = do_kmaj + so, domn = do_mn + so, qmn = q_mn + so;
        ok = mbar_wait_warp(bar(C::bFullDO + st), (uint32_t)(j >> 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + kColDP, v_kmaj + kstep_off(kk), dob + kstep_off(kk), id_s,
                    kk > 0 ? 1u : 0u);
          umma_commit(bar(C::bDP));
        }
        __syncwarp();
        ok = mbar_wait_warp(bar(C::bP), (uint32_t)j & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            umma_ts(tmem + kColAcc, tmem + kColS + pcol(kk), domn + (uint64_t)(kk * 2048 >> 4),
                    id_acc, (j > 0 || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
        have = it.next(g, qt);
        if (have) {
          ok = mbar_wait_warp(bar(C::bFull + ((j + 1) & 1)), (uint32_t)((j + 1) >> 1) & 1,
                              abort_flag, kTimeoutNs);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        ok = mbar_wait_warp(bar(C::bDS), (uint32_t)j & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            umma_ts(tmem + kColAcc + D, tmem + kColDP + pcol(kk), qmn + (uint64_t)(kk * 2048 >> 4),
                    id_acc, (j > 0 || kk > 0) ? 1u : 0u);
          if (!have) umma_commit(bar(C::bAccK));        // the accumulators are final
          umma_commit(bar(C::bFree + st));
        }
        __syncwarp();
        ++j;
      }
      if (leader) {
        umma_commit(bar(C::bFinal));
        mbar_wait(bar(C::bFinal), 0, never, kTimeoutNs);
      }
    }
    __syncwarp();
  } else {
    // ============ compute: key row = TMEM lane, 64 query columns per warp
    const int wq = warp & 3, hf = warp >> 2;
    const int row = wq * 32 + lane;
    const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
    const uint32_t c0 = (uint32_t)(hf * 64);          // this warp's first column
    const int kpos = kv_lo + row;
    const uint64_t sl2x2 = pack2(g.scale_log2, g.scale_log2);
    QIter it;
    it.init(g, src, kv_lo, kv_valid, h0, h0 + grp);
    QTile qt;
    int j = 0;
    bool ok = true;
    while (it.next(g, qt)) {
      const int st = j & 1;
      if (ok) ok = mbar_wait_warp(bar(C::bS), (uint32_t)j & 1, abort_flag, kTimeoutNs);
      if (!ok) { ++j; continue; }
      tc_fence_after();
      const float* stat =
          reinterpret_cast<const float*>(base_ptr + C::kStage0 + st * C::kStageBytes + 2 * C::kTileBytes);
      // the visit's per-column -lse2 and -delta, as packed pairs
      const uint64_t* nl2v = reinterpret_cast<const uint64_t*>(stat + c0);
      const uint64_t* ndlv = reinterpret_cast<const uint64_t*>(stat + kT + c0);
      // ---- pass 1: P^T = exp2(S^T * scale * log2 e - lse2), bf16 into TMEM
      float p[64];
      {
        uint32_t u0[32], u1[32];
        tmem_ld32(tmem + t_lane + kColS + c0, u0);
        tmem_ld32(tmem + t_lane + kColS + c0 + 32, u1);
        tmem_ld_wait();
        reg_fence(u0);
        reg_fence(u1);
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const uint32_t s0 = i < 32 ? u0[i] : u1[i - 32];
          const uint32_t s1 = i < 32 ? u0[i + 1] : u1[i - 31];
          float x0, x1;
          unpack2(ffma2(pack2(__uint_as_float(s0), __uint_as_float(s1)), sl2x2, nl2v[i >> 1]),
                  x0, x1);
          p[i] = ex2_approx(x0);
          p[i + 1] = ex2_approx(x1);
        }
        // visits the causal rule cuts: column c is masked iff c < lim
        if (qt.mask) {
          const int lim = kpos - qt.lo - (int)c0;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i < lim) p[i] = 0.f;
        }
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 64; i += 2) pk[i >> 1] = pack_bf16x2(p[i], p[i + 1]);
        tmem_st32(tmem + t_lane + kColS + c0, pk);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(C::bP));
      // ---- pass 2: dS^T = P^T * (dP^T - delta), bf16 into TMEM
      ok = mbar_wait_warp(bar(C::bDP), (uint32_t)j & 1, abort_flag, kTimeoutNs);
      if (!ok) { ++j; continue; }
      tc_fence_after();
      {
        uint32_t u0[32], u1[32];
        tmem_ld32(tmem + t_lane + kColDP + c0, u0);
        tmem_ld32(tmem + t_lane + kColDP + c0 + 32, u1);
        tmem_ld_wait();
        reg_fence(u0);
        reg_fence(u1);
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const uint32_t d0 = i < 32 ? u0[i] : u1[i - 32];
          const uint32_t d1 = i < 32 ? u0[i + 1] : u1[i - 31];
          const uint64_t t2 = fadd2(pack2(__uint_as_float(d0), __uint_as_float(d1)), ndlv[i >> 1]);
          float r0, r1;
          unpack2(ffma2(pack2(p[i], p[i + 1]), t2, 0ull), r0, r1);
          pk[i >> 1] = pack_bf16x2(r0, r1);
        }
        tmem_st32(tmem + t_lane + kColDP + c0, pk);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(C::bDS));
      ++j;
    }
    // ---- epilogue: this warp's half of the dV and dK columns, as bf16 rows
    // (the issuer commits bAccK once, after the last visit's dK)
    if (ok && j > 0) ok = mbar_wait_warp(bar(C::bAccK), 0, abort_flag, kTimeoutNs);
    if (ok) {
      tc_fence_after();
      const size_t off = ((kr.grow + kpos) * g.H_kv + hk) * D;
      const bool row_ok = row < kv_valid && in_range((long long)off, D, extent_kv(gp), status);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* dst = (which ? dk : dv) + off;
        const float mul = which ? g.scale : 1.f;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          const int col = hf * (D / 2) + c * 32;
          uint32_t u[32];
          tmem_ld32(tmem + t_lane + kColAcc + which * D + col, u);
          tmem_ld_wait(u);
          if (j == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = 0u;
          }
          if (row_ok) store_row32(dst + col, u, mul);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && (*abort_flag || *never) && status)
    atomicExch(status, (int)RA_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ dQ
// Per visit j the tensor cores run S(j), dP(j), dQ(j); the compute warps read
// S (pass 1, P kept in registers) and then dP (pass 2), writing bf16 dS into
// one of two TMEM buffers after the dQ accumulator. The issuer sends S(j+1)
// as soon as pass 1 has read S(j), and dP(j+1) right after pass 2, ahead of
// dQ(j), so both passes of the next visit find their product done. K_j stays
// in its slot until dQ(j), V_j only until dP(j).
template <int D, bool kVarlen>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
              const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_do, const Geometry gp,
              const float* __restrict__ lse2, const float* __restrict__ delta,
              __nv_bfloat16* __restrict__ dq, int* __restrict__ status) {
  using C = CfgQ<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  auto bar = [&](int i) -> uint32_t { return base + C::kBarOff + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kBarOff + C::kAbortOff);
  volatile int* never = reinterpret_cast<volatile int*>(base_ptr + C::kBarOff + C::kNeverOff);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + C::kBarOff + C::kHolderOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work item: one query tile, ordered as the forward's (kv head outermost,
  // query tiles by decreasing position, the group's heads innermost)
  const int grp = gp.H_q / gp.H_kv;
  const int n_qt = gp.n_seg * gp.nt;
  const int hg = (int)(blockIdx.x % grp);
  const int rest = (int)(blockIdx.x / grp);
  const int qt = n_qt - 1 - rest % n_qt;
  const int bhk = rest / n_qt;
  const int b = bhk / gp.H_kv, hk = bhk % gp.H_kv;
  const int h = hk * grp + hg;
  const int bh = b * gp.H_q + h;
  const int seg = qt / gp.nt;
  const int ti = qt % gp.nt;
  // packed variable-length sequences: b is the sequence, `g` its geometry
  Geometry gv;
  int row0 = 0;
  if constexpr (kVarlen) varlen_geometry(gp, b, gv, row0, threadIdx.x == 0 ? status : nullptr);
  const Geometry& g = kVarlen ? gv : gp;
  const SegRows qr = seg_rows(gp, b, seg, row0, kVarlen);    // the query tile's rows
  const int r = seg_owner(g, seg);
  const int q_lo = seg * g.seg_len + ti * kT;
  const int q_valid = tile_tokens(g, seg, ti);      // <= 0: padding only
  if (q_valid <= 0) return;      // no query, no gradient row: the CTA leaves at once

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bFix), 1);
    for (int i = 0; i < C::kKBuf; ++i) {
      mbar_init(bar(C::bKFull + i), 1);
      mbar_init(bar(C::bKFree + i), 1);
    }
    for (int i = 0; i < C::kVBuf; ++i) {
      mbar_init(bar(C::bVFull + i), 1);
      mbar_init(bar(C::bVFree + i), 1);
    }
    mbar_init(bar(C::bS), 1);
    mbar_init(bar(C::bDP), 1);
    mbar_init(bar(C::bP), 256);
    mbar_init(bar(C::bDS), 256);
    mbar_init(bar(C::bAccB + 0), 1);
    mbar_init(bar(C::bAccB + 1), 1);
    mbar_init(bar(C::bFinal), 1);
    *abort_flag = 0;
    *never = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::bFix), 2 * C::kTileBytes);
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_4d(base + C::kFixA + bx * kBoxBytes, &tm_q, bar(C::bFix), bx * 64, h,
                    qr.trow + q_lo, qr.tbat);
        tma_load_4d(base + C::kFixB + bx * kBoxBytes, &tm_do, bar(C::bFix), bx * 64, h,
                    qr.trow + q_lo, qr.tbat);
      }
      KvIter it;
      it.init(g, r, q_lo, q_valid);
      KvTile kv;
      int nk = 0, nv = 0;                  // K and V tiles loaded
      int ks = 0, kn = 0, vs = 0, vn = 0;  // next slot of each ring, and its use count
      while (it.next(g, kv)) {
        const SegRows kr = seg_rows(gp, b, kv.seg, row0, kVarlen);
        // K_j reuses the slot of K_{j-3}: free once dQ(j-3) is done
        if (kn > 0 &&
            !mbar_wait(bar(C::bKFree + ks), (uint32_t)(kn - 1) & 1, abort_flag, kTimeoutNs))
          break;
        mbar_arrive_expect_tx(bar(C::bKFull + ks), C::kTileBytes);
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_4d(base + C::kK0 + ks * C::kTileBytes + bx * kBoxBytes, &tm_k,
                      bar(C::bKFull + ks), bx * 64, hk, kr.trow + kv.lo, kr.tbat);
        ++nk;
        if (++ks == C::kKBuf) { ks = 0; ++kn; }
        // V_j reuses the slot of V_{j-2}: free once dP(j-2) is done
        if (vn > 0 &&
            !mbar_wait(bar(C::bVFree + vs), (uint32_t)(vn - 1) & 1, abort_flag, kTimeoutNs))
          break;
        mbar_arrive_expect_tx(bar(C::bVFull + vs), C::kTileBytes);
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_4d(base + C::kV0 + vs * C::kTileBytes + bx * kBoxBytes, &tm_v,
                      bar(C::bVFull + vs), bx * 64, hk, kr.trow + kv.lo, kr.tbat);
        ++nv;
        if (++vs == C::kVBuf) { vs = 0; ++vn; }
      }
      // every issued copy lands before the CTA leaves (the last use of each slot)
      for (int jj = (nk > C::kKBuf ? nk - C::kKBuf : 0); jj < nk; ++jj)
        mbar_wait(bar(C::bKFull + jj % C::kKBuf), (uint32_t)(jj / C::kKBuf) & 1, never,
                  kTimeoutNs);
      for (int jj = (nv > C::kVBuf ? nv - C::kVBuf : 0); jj < nv; ++jj)
        mbar_wait(bar(C::bVFull + jj % C::kVBuf), (uint32_t)(jj / C::kVBuf) & 1, never,
                  kTimeoutNs);
      mbar_wait(bar(C::bFix), 0, never, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // The whole warp runs the issuer's loop, so its descriptor arithmetic is
    // warp-uniform; one elected lane issues every MMA and commit (a commit
    // tracks the MMAs of the thread that issues it).
    {
      const bool leader = elect_one_sync();
      constexpr uint32_t id_s = idesc_bf16_f32(128, kT, false);
      constexpr uint32_t id_acc = idesc_bf16_f32(128, D, true);
      const uint64_t q_kmaj = sw128_desc(base + C::kFixA, 16, 1024);
      const uint64_t do_kmaj = sw128_desc(base + C::kFixB, 16, 1024);
      const uint64_t k_kmaj = sw128_desc(base + C::kK0, 16, 1024);
      const uint64_t v_kmaj = sw128_desc(base + C::kV0, 16, 1024);
      const uint64_t k_mn = sw128_desc(base + C::kK0, kBoxBytes, 1024);
      constexpr uint64_t kSlot = (uint64_t)(C::kTileBytes >> 4);   // one slot, in 16-byte units
      auto issue_s = [&](int slot) {
        const uint64_t kb = k_kmaj + slot * kSlot;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + kColS, q_kmaj + kstep_off(kk), kb + kstep_off(kk), id_s,
                    kk > 0 ? 1u : 0u);
          umma_commit(bar(C::bS));
        }
        __syncwarp();
      };
      auto issue_dp = [&](int slot) {
        const uint64_t vb = v_kmaj + slot * kSlot;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + kColDP, do_kmaj + kstep_off(kk), vb + kstep_off(kk), id_s,
                    kk > 0 ? 1u : 0u);
          umma_commit(bar(C::bDP));
          umma_commit(bar(C::bVFree + slot));       // V_j is read by dP(j) only
        }
        __syncwarp();
      };
      bool ok = mbar_wait_warp(bar(C::bFix), 0, abort_flag, kTimeoutNs);
      KvIter it;
      it.init(g, r, q_lo, q_valid);
      KvTile kv;
      bool have = ok && it.next(g, kv);
      // S(0), dP(0)
      if (have) {
        ok = mbar_wait_warp(bar(C::bKFull), 0, abort_flag, kTimeoutNs);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          ok = mbar_wait_warp(bar(C::bVFull), 0, abort_flag, kTimeoutNs);
          if (ok) {
            tc_fence_after();
            issue_dp(0);
          }
        }
      }
      // Per visit: S(j+1) once pass 1 has read S(j); then, once pass 2 has
      // read dP(j) and written dS(j) (into a buffer of its own, alternating),
      // dP(j+1) -- which pass 2 of the next visit waits for -- and dQ(j).
      // No product waits for another to finish.
      int ks = 0, kn = 0, vs = 0, vn = 0;   // slots of K(j) and V(j), and their use counts
      int j = 0;
      while (ok && have) {
        have = it.next(g, kv);
        int ks1 = ks + 1, kn1 = kn, vs1 = vs + 1, vn1 = vn;
        if (ks1 == C::kKBuf) { ks1 = 0; ++kn1; }
        if (vs1 == C::kVBuf) { vs1 = 0; ++vn1; }
        if (have) {
          ok = mbar_wait_warp(bar(C::bKFull + ks1), (uint32_t)kn1 & 1, abort_flag, kTimeoutNs) &&
               mbar_wait_warp(bar(C::bP), (uint32_t)j & 1, abort_flag, kTimeoutNs);
          if (!ok) break;
          tc_fence_after();
          issue_s(ks1);
        }
        ok = mbar_wait_warp(bar(C::bDS), (uint32_t)j & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        if (have) {
          ok = mbar_wait_warp(bar(C::bVFull + vs1), (uint32_t)vn1 & 1, abort_flag, kTimeoutNs);
          if (!ok) break;
          tc_fence_after();
          issue_dp(vs1);
        }
        tc_fence_after();
        const uint32_t ds_col = kColDSq<D>() + (uint32_t)((j & 1) * 64);
        const uint64_t kb = k_mn + ks * kSlot;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            umma_ts(tmem + kColAcc, tmem + ds_col + dscol(kk), kb + (uint64_t)(kk * 2048 >> 4),
                    id_acc, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(bar(C::bAccB + (j & 1)));
          umma_commit(bar(C::bKFree + ks));        // K_j's last reader is dQ(j)
        }
        __syncwarp();
        ks = ks1; kn = kn1; vs = vs1; vn = vn1;
        ++j;
      }
      if (leader) {
        umma_commit(bar(C::bFinal));
        mbar_wait(bar(C::bFinal), 0, never, kTimeoutNs);
      }
    }
    __syncwarp();
  } else {
    // ============ compute: query row = TMEM lane, 64 key columns per warp
    const int wq = warp & 3, hf = warp >> 2;
    const int row = wq * 32 + lane;
    const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
    const uint32_t c0 = (uint32_t)(hf * 64);
    const int q_pos = q_lo + row;
    const uint64_t sl2x2 = pack2(g.scale_log2, g.scale_log2);
    const long long wi = ws_tile(gp, bh, seg, ti) + row;
    const bool wi_ok = in_range(wi, 1, ws_tile(gp, gp.B * gp.H_q, 0, 0), status);
    // the row's -lse2 (-inf on padding rows: p = 0) and -delta, as pairs
    const float nl2_row = wi_ok ? lse2[wi] : -INFINITY;
    const float ndl_row = wi_ok ? delta[wi] : 0.f;
    const uint64_t nl2x2 = pack2(nl2_row, nl2_row), ndlx2 = pack2(ndl_row, ndl_row);
    KvIter it;
    it.init(g, r, q_lo, q_valid);
    KvTile kv;
    int j = 0;
    bool ok = true;
    while (it.next(g, kv)) {
      if (ok) ok = mbar_wait_warp(bar(C::bS), (uint32_t)j & 1, abort_flag, kTimeoutNs);
      if (!ok) { ++j; continue; }
      tc_fence_after();
      // ---- pass 1: P = exp2(S * scale * log2 e - lse2), kept in registers
      float p[64];
      {
        uint32_t u0[32], u1[32];
        tmem_ld32(tmem + t_lane + kColS + c0, u0);
        tmem_ld32(tmem + t_lane + kColS + c0 + 32, u1);
        tmem_ld_wait();
        reg_fence(u0);
        reg_fence(u1);
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const uint32_t s0 = i < 32 ? u0[i] : u1[i - 32];
          const uint32_t s1 = i < 32 ? u0[i + 1] : u1[i - 31];
          float x0, x1;
          unpack2(ffma2(pack2(__uint_as_float(s0), __uint_as_float(s1)), sl2x2, nl2x2), x0, x1);
          p[i] = ex2_approx(x0);
          p[i + 1] = ex2_approx(x1);
        }
        // key tiles the causal rule cuts, and ragged tails: key column c of
        // this warp is allowed iff c < lim
        if (kv.work == kMask) {
          const int lim = (g.causal ? min(kv.valid, q_pos - kv.lo + 1) : kv.valid) - (int)c0;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i >= lim) p[i] = 0.f;
        }
      }
      tc_fence_before();
      mbar_arrive(bar(C::bP));          // S may be overwritten
      // ---- pass 2: dS = P * (dP - delta), bf16 into TMEM
      ok = mbar_wait_warp(bar(C::bDP), (uint32_t)j & 1, abort_flag, kTimeoutNs);
      if (!ok) { ++j; continue; }
      tc_fence_after();
      {
        uint32_t u0[32], u1[32];
        tmem_ld32(tmem + t_lane + kColDP + c0, u0);
        tmem_ld32(tmem + t_lane + kColDP + c0 + 32, u1);
        tmem_ld_wait();
        reg_fence(u0);
        reg_fence(u1);
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const uint32_t d0 = i < 32 ? u0[i] : u1[i - 32];
          const uint32_t d1 = i < 32 ? u0[i + 1] : u1[i - 31];
          const uint64_t t2 = fadd2(pack2(__uint_as_float(d0), __uint_as_float(d1)), ndlx2);
          float r0, r1;
          unpack2(ffma2(pack2(p[i], p[i + 1]), t2, 0ull), r0, r1);
          pk[i >> 1] = pack_bf16x2(r0, r1);
        }
        // dS buffer j mod 2 was last read by dQ(j-2)
        if (j >= 2) {
          ok = mbar_wait_warp(bar(C::bAccB + (j & 1)), (uint32_t)((j >> 1) - 1) & 1,
                              abort_flag, kTimeoutNs);
          if (!ok) { ++j; continue; }
          tc_fence_after();
        }
        tmem_st32(tmem + t_lane + kColDSq<D>() + (uint32_t)((j & 1) * 64) + (uint32_t)(hf * 32), pk);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(C::bDS));
      ++j;
    }
    if (ok && j > 0)
      ok = mbar_wait_warp(bar(C::bAccB + ((j - 1) & 1)), (uint32_t)((j - 1) >> 1) & 1,
                          abort_flag, kTimeoutNs);
    if (ok) {
      tc_fence_after();
      const size_t off = ((qr.grow + q_pos) * g.H_q + h) * D;
      const bool row_ok = row < q_valid && in_range((long long)off, D, extent_q(gp), status);
      __nv_bfloat16* dst = dq + off;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = hf * (D / 2) + c * 32;
        uint32_t u[32];
        tmem_ld32(tmem + t_lane + kColAcc + col, u);
        tmem_ld_wait(u);
        if (j == 0) {
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = 0u;
        }
        if (row_ok) store_row32(dst + col, u, g.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && (*abort_flag || *never) && status)
    atomicExch(status, (int)RA_ERR_TIMEOUT);
}

template <int D, bool kVarlen>
ra_status launch_d(const Geometry& g, const CUtensorMap& mq, const CUtensorMap& mk,
                   const CUtensorMap& mv, const CUtensorMap& mdo, const void* out,
                   const float* lse, const void* dout, void* dq, void* dk, void* dv,
                   float* ws, int phases, int* status, cudaStream_t stream) {
  using C = Cfg<D>;
  const long long rows = bwd_workspace_floats(g) / 2;
  float* lse2 = ws;
  float* delta = ws + rows;
  const long long prep_blocks = rows / 32;
  const long long n_tiles = (long long)g.n_seg * g.nt;
  const long long grid_kv = n_tiles * g.B * g.H_kv;
  const long long grid_q = n_tiles * g.B * g.H_q;
  if (prep_blocks > 0x7fffffffLL || grid_q > 0x7fffffffLL) return RA_ERR_RANGE;
  if (phases & RA_BWD_PREP) {
    bwd_prep_kernel<D, kVarlen><<<(unsigned)prep_blocks, 256, 0, stream>>>(
        g, static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout),
        lse, lse2, delta, rows, status);
    if (cudaGetLastError() != cudaSuccess) return RA_ERR_LAUNCH;
  }
  if (phases & RA_BWD_DKDV) {
    if (cudaFuncSetAttribute(bwd_dkdv_kernel<D, kVarlen>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return RA_ERR_LAUNCH;
    bwd_dkdv_kernel<D, kVarlen><<<(unsigned)grid_kv, kThreads, C::kSmemBytes, stream>>>(
        mq, mk, mv, mdo, g, lse2, delta, static_cast<__nv_bfloat16*>(dk),
        static_cast<__nv_bfloat16*>(dv), status);
    if (cudaGetLastError() != cudaSuccess) return RA_ERR_LAUNCH;
  }
  if (phases & RA_BWD_DQ) {
    using CQ = CfgQ<D>;
    if (cudaFuncSetAttribute(bwd_dq_kernel<D, kVarlen>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             CQ::kSmemBytes) != cudaSuccess)
      return RA_ERR_LAUNCH;
    bwd_dq_kernel<D, kVarlen><<<(unsigned)grid_q, kThreads, CQ::kSmemBytes, stream>>>(
        mq, mk, mv, mdo, g, lse2, delta, static_cast<__nv_bfloat16*>(dq), status);
    if (cudaGetLastError() != cudaSuccess) return RA_ERR_LAUNCH;
  }
  return RA_OK;
}

}  // namespace

long long bwd_workspace_floats(const Geometry& g) {
  return 2 * ws_tile(g, g.B * g.H_q, 0, 0);
}

ra_status launch_attn_bwd(const Geometry& g, const void* q, const void* k, const void* v,
                          const void* out, const float* lse, const void* dout, void* dq,
                          void* dk, void* dv, float* workspace, int phases,
                          int* dev_status, cudaStream_t stream) {
  // packed variable-length tensors are mapped as one batch of `total` rows,
  // sequence-sharded ones [P, B, C, H, D] as P*B batches of C rows
  const bool varlen = g.cu_seqlens != nullptr;
  const int mb = varlen ? 1 : (g.shard_rows > 0 ? g.P * g.B : g.B);
  const int ms = varlen ? g.total : (g.shard_rows > 0 ? g.shard_rows : g.S);
  CUtensorMap mq, mk, mv, mdo;
  if (!make_bshd_map(&mq, q, mb, ms, g.H_q, g.D, kT) ||
      !make_bshd_map(&mk, k, mb, ms, g.H_kv, g.D, kT) ||
      !make_bshd_map(&mv, v, mb, ms, g.H_kv, g.D, kT) ||
      !make_bshd_map(&mdo, dout, mb, ms, g.H_q, g.D, kT))
    return RA_ERR_LAUNCH;
  if (varlen) {
    if (g.D == 64)
      return launch_d<64, true>(g, mq, mk, mv, mdo, out, lse, dout, dq, dk, dv, workspace,
                                phases, dev_status, stream);
    return launch_d<128, true>(g, mq, mk, mv, mdo, out, lse, dout, dq, dk, dv, workspace,
                               phases, dev_status, stream);
  }
  if (g.D == 64)
    return launch_d<64, false>(g, mq, mk, mv, mdo, out, lse, dout, dq, dk, dv, workspace,
                               phases, dev_status, stream);
  return launch_d<128, false>(g, mq, mk, mv, mdo, out, lse, dout, dq, dk, dv, workspace,
                              phases, dev_status, stream);
}

}  // namespace ra
