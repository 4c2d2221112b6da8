// Exact ring attention on the tcgen05 tensor cores (bf16 in, f32 accumulate).
//
// Glossary "sequence parallelism transformers":
//  - §Ring Attention: each virtual rank keeps its query block; at step t it
//    attends to the key/value block of rank (r - t) mod P ("receive from
//    i-1"), and accumulates outputs; only the local block and the received
//    blocks in flight need to be resident ("Memory Efficiency").
//  - §Flash Attention with Sequence Parallelism: attention is computed tile
//    by tile (prior art; the tiling below is laid out for sm_103a).
//  - §Implementation Considerations: the softmax normalisation across blocks
//    is kept exact with a running maximum and sum (log-sum-exp merge).
//
// One CTA owns one 128-row query tile of one (batch, head) inside one
// segment of virtual rank r and walks the key tiles of the ring in order,
// j = 0, 1, ... (tiles wholly after the query tile under a causal mask are
// left out). "Receiving" a block is a TMA load of its tiles from this GPU's
// HBM/L2 into shared memory. Warp roles (352 threads with kSplit = 2):
//   warps 0-7  softmax: kSplit = 2 threads per query row (row = TMEM lane),
//              each taking 64 of the 128 key columns and half of O's columns
//   warp  8    TMA producer: Q once, then K_j (3 slots) and V_j (2 slots)
//   warp  9    TMEM allocator; one thread issues the S = Q K^T MMAs
//   warp 10    one thread issues the O += P V MMAs
// The same kernel serves the fixed-length [B, S, H, D] layout, packed
// variable-length sequences (kVarlen) and the sequence-sharded layout
// (shard_rows > 0); only the rows its loads and stores address differ.
// Tensor memory (512 columns): three S buffers of 128 f32 columns at 0, 128,
// 256 (key tile j uses buffer j mod 3; softmax writes P as bf16 over the
// first 64 columns of that buffer) and the O accumulator at 384.
// With three buffers, S(j+3) only has to wait for PV(j), which the tensor
// core finished long before: the S issuer runs up to three tiles ahead, the
// softmax never waits for the tensor core in steady state, and the tensor
// core always has the next S or PV queued.
//
// Synchronisation (b = j mod 3, u = j / 3 is the use count of buffer b):
//   kfull[b]            TMA of K_j landed                  (phase u)
//   vfull[j mod 2]      TMA of V_j landed                  (phase j / 2)
//   sfull[b]            S(j) done (S issuer's commit)      (phase u)
//   pfull[b]            P(j) written, O rescaled (one arrival per softmax thread)
//   odone[b]            PV(j) done (PV issuer's commit)    (phase u)
// The producer reuses K_j's slot when sfull[b] completes phase u-1 and V_j's
// (two V slots) once PV(j-2) is done: the completion barriers double as
// "slot free". Every
// barrier's next phase depends on the waiter's own progress, so no waiter can
// fall two phases behind (parity waits are unambiguous).
//
// The running (max, sum, O) carried across key tiles -- across ring-step
// boundaries too -- is the in-register form of the log-sum-exp merge of the
// per-step partials.
//
// Every wait is bounded: after kTimeoutNs a thread raises a CTA-wide abort
// flag, every role falls through to the common teardown (which still waits,
// bounded, for the loads and tensor-core work it issued, then frees TMEM),
// and the kernel reports RA_ERR_TIMEOUT through the status word.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "checks.cuh"
#include "fastmath.cuh"
#include "ra_internal.h"
#include "ring_iter.cuh"
#include "sm100.cuh"

namespace ra {
namespace {

using namespace sm100;
using namespace fastmath;

constexpr int kTile = 128;
// Softmax warps per TMEM lane quarter: each row's 128 scores are split over
// this many warps (kSCols columns each), so 4 * kSplit softmax warps share
// the SM with the producer and the two issuers. Measured on GB300 (headline
// workload, 2070 MHz): 2 -> 1456-1464 TFLOP/s, 4 -> 1380 (the four-warp
// barrier per key tile costs more than the extra warps hide).
constexpr int kSplit = 2;
constexpr int kSCols = kTile / kSplit;
constexpr int kSoftmaxWarps = 4 * kSplit;
constexpr int kThreads = 32 * (kSoftmaxWarps + 3);
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kSIssuerWarp = kSoftmaxWarps + 1;   // also allocates / frees TMEM
constexpr int kPVIssuerWarp = kSoftmaxWarps + 2;
constexpr int kBuf = 3;               // S/P buffers in TMEM = K slots in smem
constexpr int kVBuf = 2;              // V slots in smem
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 384;
constexpr float kRescaleLog2 = 8.0f;          // lazy rescale threshold (x256)
// Of every 8 column pairs of a softmax row half, this many get their
// exponentials from exp2_poly2 on the FMA pipe, the rest from ex2.approx.
// Measured on GB300 (headline workload): 0 -> 1493, 2 -> 1416, 3 -> 1384,
// 4 -> 1334 TFLOP/s; the softmax is issue-bound, not bound by the special
// function unit, so every exponential stays on ex2.approx.
constexpr int kPolyPairsPer8 = 0;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kBoxBytes = kTile * 64 * 2;      // one TMA box: 128 rows x 64 bf16

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kBoxes = D / 64;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTileBytes;           // K_j in slot j mod 3
  static constexpr int kVOff = kKOff + kBuf * kTileBytes;    // V_j in slot j mod 2
  static constexpr int kBarOff = kVOff + kVBuf * kTileBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kFlagsOff = kBarBytes;          // 16 x u32: key-tile flags ring
  static constexpr int kFlagsBytes = 64;
  static constexpr int kRedOff = kBarOff + kBarBytes + kFlagsBytes;   // softmax exchange
  static constexpr int kRedBytes = 3 * kSplit * 128 * 4;   // maxima [2][kSplit][128], sums [kSplit][128]
  static constexpr int kUsed = kRedOff + kRedBytes + 1024;   // + alignment slack
  // Request more than half an SM's shared memory so that one CTA owns the SM
  // and its 512 TMEM columns (the D=64 layout alone would fit two).
  static constexpr int kSmemBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
  // barrier indices (8 bytes each)
  static constexpr int bQFull = 0;
  static constexpr int bKFull = 1;                     // [3]
  static constexpr int bVFull = bKFull + kBuf;         // [2]
  static constexpr int bSFull = bVFull + kVBuf;        // [3]
  static constexpr int bPFull = bSFull + kBuf;         // [3], 128 arrivals
  static constexpr int bODone = bPFull + kBuf;         // [3]
  static constexpr int bFinalS = bODone + kBuf;
  static constexpr int bFinalPV = bFinalS + 1;
  static constexpr int kNumBars = bFinalPV + 1;
  static constexpr int kHolderOff = kBarBytes - 16;    // TMEM base address
  static constexpr int kNeverOff = kBarBytes - 12;     // stays 0: waits that ignore aborts
  static constexpr int kAbortOff = kBarBytes - 8;      // abort flag
  static_assert(kNumBars * 8 <= kHolderOff, "barrier area overflow");
  static_assert(kSmemBytes > 116 * 1024, "must not fit two CTAs per SM");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ uint32_t s_col(int b) { return (uint32_t)(b * 128); }

// Barrier among `count` threads of the CTA (ids 1-15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// P columns of one softmax warp: 32 (two-way split) or 16 (four-way split).
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N == 32 || N == 16, "32 or 16 columns");
  if constexpr (N == 32) tmem_st32(taddr, r);
  else tmem_st16(taddr, r);
}

// Columns [tO, tO + N) of this thread's O row times alpha.
template <int N>
__device__ __forceinline__ void scale_cols(uint32_t tO, float alpha) {
  if constexpr (N >= 32) {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) {
      uint32_t uo[32];
      tmem_ld32(tO + c * 32, uo);
      tmem_ld_wait(uo);
#pragma unroll
      for (int i = 0; i < 32; ++i) uo[i] = __float_as_uint(__uint_as_float(uo[i]) * alpha);
      tmem_st32(tO + c * 32, uo);
    }
  } else {
    uint32_t uo[16];
    tmem_ld16(tO, uo);
    tmem_ld_wait(uo);
#pragma unroll
    for (int i = 0; i < 16; ++i) uo[i] = __float_as_uint(__uint_as_float(uo[i]) * alpha);
    tmem_st16(tO, uo);
  }
}

template <int CH>
__device__ __forceinline__ void ld_cols(uint32_t taddr, uint32_t (&r)[CH]) {
  if constexpr (CH == 32) tmem_ld32(taddr, r);
  else tmem_ld16(taddr, r);
  tmem_ld_wait(r);
}

// Epilogue of one softmax warp: its N columns of the O row, times 1/l, to
// `out` at element offset row_off (bf16, or float32 for single-step
// partials). Every thread loads (the TMEM load is warp-wide); valid rows store.
template <int N, bool kOutF32>
__device__ __forceinline__ void store_out_cols(uint32_t tO, bool have_o, bool row_valid,
                                               void* out, size_t row_off, float inv_l) {
  constexpr int CH = N >= 32 ? 32 : 16;
#pragma unroll
  for (int c = 0; c < N / CH; ++c) {
    uint32_t uo[CH];
    if (have_o) {
      ld_cols<CH>(tO + c * CH, uo);
    } else {
#pragma unroll
      for (int i = 0; i < CH; ++i) uo[i] = 0u;
    }
    if (!row_valid) continue;
    if constexpr (kOutF32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + row_off + c * CH);
#pragma unroll
      for (int i = 0; i < CH / 4; ++i)
        dst[i] = make_float4(__uint_as_float(uo[4 * i]) * inv_l,
                             __uint_as_float(uo[4 * i + 1]) * inv_l,
                             __uint_as_float(uo[4 * i + 2]) * inv_l,
                             __uint_as_float(uo[4 * i + 3]) * inv_l);
    } else {
      uint4* dst =
          reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + row_off + c * CH);
#pragma unroll
      for (int i = 0; i < CH / 8; ++i) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(uo[8 * i + 0]) * inv_l, __uint_as_float(uo[8 * i + 1]) * inv_l);
        w.y = pack_bf16x2(__uint_as_float(uo[8 * i + 2]) * inv_l, __uint_as_float(uo[8 * i + 3]) * inv_l);
        w.z = pack_bf16x2(__uint_as_float(uo[8 * i + 4]) * inv_l, __uint_as_float(uo[8 * i + 5]) * inv_l);
        w.w = pack_bf16x2(__uint_as_float(uo[8 * i + 6]) * inv_l, __uint_as_float(uo[8 * i + 7]) * inv_l);
        dst[i] = w;
      }
    }
  }
}

template <int D, bool kOutF32, bool kVarlen>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const Geometry gp,
               void* __restrict__ out, float* __restrict__ lse,
               int* __restrict__ vlog, int log_stride, int* __restrict__ status) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  auto bar = [&](int i) -> uint32_t { return base + C::kBarOff + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kBarOff + C::kAbortOff);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + C::kBarOff + C::kHolderOff);
  volatile int* never = reinterpret_cast<volatile int*>(base_ptr + C::kBarOff + C::kNeverOff);
  // Key-tile flags, written by the producer before it arms K_j's barrier and
  // read by the S issuer after that barrier completed: 1 = key tile j
  // exists, kFlagEnd = the sequence has j tiles.
  volatile uint32_t* tile_flags =
      reinterpret_cast<volatile uint32_t*>(base_ptr + C::kBarOff + C::kFlagsOff);
  constexpr uint32_t kFlagEnd = 4u;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: one query tile. Block order: (batch, kv head) outermost,
  // so the CTAs resident at one time read the keys/values of one or two kv
  // heads and find them in L2; then query tiles by decreasing position
  // (decreasing causal work, longest first); the query heads sharing the kv
  // head innermost, so they read the same key tiles at the same time.
  // With packed variable-length sequences, b is the sequence and the grid is
  // sized by the longest one; `g` is then this sequence's own geometry.
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
  Geometry gv;
  int row0 = 0;
  if constexpr (kVarlen) varlen_geometry(gp, b, gv, row0);
  const Geometry& g = kVarlen ? gv : gp;
  const int r = seg_owner(g, seg);
  const int q_lo = seg * g.seg_len + ti * kTile;
  const int q_valid = tile_tokens(g, seg, ti);     // <= 0: a tile of padding only
  // TMA row and batch coordinates, first output row, first lse entry. In the
  // sequence-sharded layout [P, B, C, H, D] (mapped as [P*B, C, H, D]) the
  // query tile's segment is its shard p: batch p*B + b, rows from p*C.
  const bool sharded = !kVarlen && gp.shard_rows > 0;
  int trow = kVarlen ? row0 : 0;
  int tbat = kVarlen ? 0 : b;
  size_t orow = kVarlen ? (size_t)row0 : (size_t)b * gp.S;
  size_t lrow = kVarlen ? (size_t)h * gp.total + row0 : (size_t)bh * gp.S;
  if (sharded) {
    const size_t lb = (size_t)seg * gp.B + b, rows = (size_t)gp.shard_rows;
    trow = -seg * gp.shard_rows;
    tbat = (int)lb;
    orow = lb * rows - (size_t)seg * rows;
    lrow = (lb * gp.H_q + h) * rows - (size_t)seg * rows;
  }

  // A tile of padding only (uneven or packed lengths) has nothing to compute
  // or write: the whole CTA leaves before it sets anything up.
  // the visit log of this query tile: [count, 4 ints per visit]
  const long long log_off = ((long long)bh * n_qt + qt) * log_stride;
  const long long log_len = (long long)gp.B * gp.H_q * n_qt * log_stride;
  if (q_valid <= 0) {
    if (vlog && threadIdx.x == 0 && in_range(log_off, 1, log_len, status)) vlog[log_off] = 0;
    return;
  }

  // ---- set-up: barriers, abort flag, TMEM
  if (threadIdx.x == 0) {
    mbar_init(bar(C::bQFull), 1);
    for (int i = 0; i < kVBuf; ++i) mbar_init(bar(C::bVFull + i), 1);
    for (int i = 0; i < kBuf; ++i) {
      mbar_init(bar(C::bKFull + i), 1);
      mbar_init(bar(C::bSFull + i), 1);
      mbar_init(bar(C::bPFull + i), 32 * kSoftmaxWarps);
      mbar_init(bar(C::bODone + i), 1);
    }
    mbar_init(bar(C::bFinalS), 1);
    mbar_init(bar(C::bFinalPV), 1);
    *abort_flag = 0;
    *never = 0;
    fence_mbar_init();
  }
  if (warp == kSIssuerWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == kProducerWarp) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      const uint32_t q_smem = base + C::kQOff;
      mbar_arrive_expect_tx(bar(C::bQFull), C::kTileBytes);
      for (int bx = 0; bx < C::kBoxes; ++bx)
        tma_load_4d(q_smem + bx * kBoxBytes, &tm_q, bar(C::bQFull), bx * 64, h, trow + q_lo,
                    tbat);
      KvIter it;
      it.init(g, r, q_lo, q_valid);
      KvTile kv;
      int j = 0;
      int nk = 0, nv = 0;   // key tiles whose K / V slot use has been armed
      bool ok = true;
      while (ok && it.next(g, kv)) {
        const int bb = j % kBuf;
        const uint32_t u = (uint32_t)(j / kBuf);
        const uint32_t k_smem = base + C::kKOff + bb * C::kTileBytes;
        // K_j reuses the slot of K_{j-3}: free once S(j-3) is done
        if (j >= kBuf && !mbar_wait(bar(C::bSFull + bb), (u - 1) & 1, abort_flag, kTimeoutNs)) {
          ok = false;
          break;
        }
        tile_flags[j & 15] = 1u;
        // the key tile's own shard in the sequence-sharded layout
        const int krow = sharded ? -kv.seg * gp.shard_rows : trow;
        const int kbat = sharded ? kv.seg * gp.B + b : tbat;
        mbar_arrive_expect_tx(bar(C::bKFull + bb), C::kTileBytes);
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_4d(k_smem + bx * kBoxBytes, &tm_k, bar(C::bKFull + bb), bx * 64, hk,
                      krow + kv.lo, kbat);
        nk = j + 1;
        // V_j reuses the slot of V_{j-2}: free once PV(j-2) is done
        // (odone of buffer (j-2) mod 3, phase (j-2) / 3)
        const int vb = j % kVBuf;
        if (j >= kVBuf &&
            !mbar_wait(bar(C::bODone + (j - 2) % kBuf), (uint32_t)((j - 2) / kBuf) & 1,
                       abort_flag, kTimeoutNs)) {
          ok = false;
          break;
        }
        if (!(g.withhold_v0 && j == 0)) {      // test of the expiry path only
          mbar_arrive_expect_tx(bar(C::bVFull + vb), C::kTileBytes);
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_4d(base + C::kVOff + vb * C::kTileBytes + bx * kBoxBytes, &tm_v,
                        bar(C::bVFull + vb), bx * 64, hk, krow + kv.lo, kbat);
        }
        nv = j + 1;
        ++j;
      }
      // Every issued load lands before the CTA leaves (already true unless
      // the CTA aborted). This comes before the end marker, which completes
      // one more phase of a K barrier.
      for (int jj = (nk > kBuf ? nk - kBuf : 0); jj < nk; ++jj)
        mbar_wait(bar(C::bKFull + jj % kBuf), (uint32_t)(jj / kBuf) & 1, never, kTimeoutNs);
      for (int jj = (nv > kVBuf ? nv - kVBuf : 0); jj < nv; ++jj)
        if (!(g.withhold_v0 && jj == 0))
          mbar_wait(bar(C::bVFull + jj % kVBuf), (uint32_t)(jj / kVBuf) & 1, never, kTimeoutNs);
      mbar_wait(bar(C::bQFull), 0, never, kTimeoutNs);
      // End marker: K barrier of tile j completes with no load, flag kFlagEnd.
      if (ok) {
        tile_flags[j & 15] = kFlagEnd;
        mbar_arrive(bar(C::bKFull + j % kBuf));
      }
    }
    __syncwarp();
  } else if (warp == kSIssuerWarp) {
    // ======================= S = Q K^T issuer =======================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kTile, false);
      // Descriptors differ only in the start-address field (bits 0-13, in
      // 16-byte units, no carry: shared addresses are < 256 KB), so they are
      // built once and offset per K step and slot.
      const uint64_t q_desc = sw128_desc(base + C::kQOff, 16, 1024);
      const uint64_t k_desc = sw128_desc(base + C::kKOff, 16, 1024);
      bool ok = mbar_wait(bar(C::bQFull), 0, abort_flag, kTimeoutNs);
      for (int j = 0; ok; ++j) {
        const int bb = j % kBuf;
        const uint32_t u = (uint32_t)(j / kBuf);
        ok = mbar_wait(bar(C::bKFull + bb), u & 1, abort_flag, kTimeoutNs);
        if (!ok || (tile_flags[j & 15] & kFlagEnd)) break;
        // buffer bb still holds P(j-3) until PV(j-3) is done
        if (j >= kBuf) ok = mbar_wait(bar(C::bODone + bb), (u - 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        const uint64_t kb_desc = k_desc + (uint64_t)((bb * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off16 = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
          umma_ss(tmem + s_col(bb), q_desc + off16, kb_desc + off16, idesc_s,
                  kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(C::bSFull + bb));
      }
      // all tensor-core work this thread issued has completed before teardown
      umma_commit(bar(C::bFinalS));
      mbar_wait(bar(C::bFinalS), 0, never, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp == kPVIssuerWarp) {
    // ======================= O += P V issuer =======================
    if (lane == 0) {
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, true);
      const uint64_t v_desc = sw128_desc(base + C::kVOff, kBoxBytes, 1024);
      KvIter it;
      it.init(g, r, q_lo, q_valid);
      KvTile kv;
      bool ok = true;
      int j = 0;
      while (ok && it.next(g, kv)) {
        const int bb = j % kBuf;
        const uint32_t u = (uint32_t)(j / kBuf);
        const int vb = j % kVBuf;
        ok = mbar_wait(bar(C::bVFull + vb), (uint32_t)(j / kVBuf) & 1, abort_flag, kTimeoutNs) &&
             mbar_wait(bar(C::bPFull + bb), u & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        const uint64_t vb_desc = v_desc + (uint64_t)((vb * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts(tmem + kOCol, tmem + s_col(bb) + kk * 8, vb_desc + (kk * 2048 >> 4), idesc_o,
                  (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(C::bODone + bb));
        ++j;
      }
      umma_commit(bar(C::bFinalPV));
      mbar_wait(bar(C::bFinalPV), 0, never, kTimeoutNs);
    }
    __syncwarp();
  } else {
    // ================= softmax: kSplit threads per row, kSCols columns each =================
    // Warps w, w+4, w+8, ... share TMEM lane quarter w % 4 (the same 32 rows);
    // warp part p = w / 4 handles key columns [p*kSCols, (p+1)*kSCols) and O
    // columns [p*kOC, (p+1)*kOC). The partial row maxima meet in shared memory
    // (one named barrier per row group and key tile); each part keeps its own
    // partial sum.
    constexpr int kOC = D / kSplit;          // O columns per softmax warp
    const int wq = warp & 3;                 // TMEM lane quarter
    const int part = warp >> 2;              // column part
    const int row = wq * 32 + lane;
    const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
    const uint32_t tO = tmem + t_lane + kOCol + part * kOC;
    const int q_pos = q_lo + row;
    const bool row_valid = row < q_valid;
    const float sl2 = g.scale_log2;
    const uint64_t sl2x2 = pack2(sl2, sl2);
    const uint32_t pair_bar = 1 + wq;        // named barrier of the row group
    constexpr uint32_t kGroup = 32 * kSplit; // threads meeting at that barrier
    // [2 tile parities][kSplit parts][128 rows] partial maxima, then
    // [kSplit][128] partial sums
    float* red = reinterpret_cast<float*>(base_ptr + C::kRedOff);

    int* log_base = (vlog && threadIdx.x == 0) ? vlog + log_off : nullptr;

    float m_run = -INFINITY, l_run = 0.f;    // l_run: this part's partial sum
    int j = 0;               // key tiles done (= P tiles published)
    bool ok = true;
    KvIter it;
    it.init(g, r, q_lo, q_valid);
    KvTile kv, nxt;
    // Every warp of a row group passes exactly one named barrier per key tile
    // (and one after the loop), also after an abort: a warp that gave up
    // keeps walking the tiles and only meets the barriers, so no partner is
    // left waiting at a barrier that would not complete.
    // The next key tile is looked up while this tile's scores load.
    bool have = it.next(g, kv);
    while (have) {
      const int work = kv.work;
      if (log_base && in_range(log_off + 1 + 4 * j, 4, log_len, status))
        log_visit(log_base, j, kv, tile_class(g, q_lo, kv));
      const int bb = j % kBuf;
      const uint32_t u = (uint32_t)(j / kBuf);
      const uint32_t tS = tmem + t_lane + s_col(bb) + part * kSCols;
      if (ok) ok = mbar_wait(bar(C::bSFull + bb), u & 1, abort_flag, kTimeoutNs);
      if (!ok) {
        named_bar_sync(pair_bar, kGroup);
        ++j;
        have = it.next(g, kv);
        continue;
      }
      tc_fence_after();

      float s[kSCols];
      bool have_next;
      {
        uint32_t uu[kSCols / 32][32];
#pragma unroll
        for (int c = 0; c < kSCols / 32; ++c) tmem_ld32(tS + c * 32, uu[c]);
        have_next = it.next(g, nxt);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < kSCols / 32; ++c) {
          reg_fence(uu[c]);
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(uu[c][i]);
        }
      }
      if (work == kMask) {
        const int lim =
            (g.causal ? min(kv.valid, q_pos - kv.lo + 1) : kv.valid) - part * kSCols;
#pragma unroll
        for (int c = 0; c < kSCols; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      // partial row max over kSCols columns: 8 chains of 3-input maxima
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = s[i];
      int c8 = 8;
#pragma unroll
      for (; c8 + 16 <= kSCols; c8 += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], s[c8 + i], s[c8 + 8 + i]);
      if (c8 < kSCols) {
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], s[c8 + i]);
      }
      const float mx_part = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                                  fmaxf(m8[6], m8[7]));
      // combine with the other parts of the row (the barrier also orders all
      // parts' S loads before any part writes P over the S columns)
      float* red_j = red + (j & 1) * (kSplit * 128);
      red_j[part * 128 + row] = mx_part;
      tc_fence_before();
      named_bar_sync(pair_bar, kGroup);
      tc_fence_after();
      float mx = red_j[row];
#pragma unroll
      for (int p2 = 1; p2 < kSplit; ++p2) mx = fmaxf(mx, red_j[p2 * 128 + row]);

      const float m_new = fmaxf(m_run, mx * sl2);
      const bool resc = m_new > m_run + kRescaleLog2;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m_run - m_new);     // 0 when m_run = -inf
        m_run = m_new;
        l_run *= alpha;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      const uint64_t neg_m2 = pack2(-m_use, -m_use);
      uint64_t sum2a = pack2(0.f, 0.f), sum2b = sum2a;
      uint32_t pk[kSCols / 2];
#pragma unroll
      for (int i = 0; i < kSCols / 2; ++i) {
        // (s0, s1) * scale*log2(e) - m in one packed FMA, then two exp2
        const uint64_t x2 = ffma2(pack2(s[2 * i], s[2 * i + 1]), sl2x2, neg_m2);
        float x0, x1;
        unpack2(x2, x0, x1);
        float p0, p1;
        if ((i & 7) < kPolyPairsPer8) {
          exp2_poly2(x0, x1, p0, p1);
        } else {
          p0 = ex2_approx(x0);
          p1 = ex2_approx(x1);
        }
        if (i & 1) sum2b = fadd2(sum2b, pack2(p0, p1));
        else sum2a = fadd2(sum2a, pack2(p0, p1));
        pk[i] = pack_bf16x2(p0, p1);
      }
      // P columns of this part (bf16 pairs)
      tmem_st_cols(tmem + t_lane + s_col(bb) + part * (kSCols / 2), pk);
      {
        float a0, a1;
        unpack2(fadd2(sum2a, sum2b), a0, a1);
        l_run += a0 + a1;
      }
      // O must be scaled by alpha before P(j) V_j is added to it, i.e. after
      // PV(j-1) is done (all parts take the same decision)
      if (__any_sync(0xffffffffu, resc) && j > 0) {
        const int pb = (j - 1) % kBuf;
        ok = mbar_wait(bar(C::bODone + pb), (uint32_t)((j - 1) / kBuf) & 1, abort_flag,
                       kTimeoutNs);
        if (!ok) {
          ++j;
          kv = nxt;
          have = have_next;
          continue;
        }
        tc_fence_after();
        scale_cols<kOC>(tO, alpha);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::bPFull + bb));
      ++j;
      kv = nxt;
      have = have_next;
    }
    if (log_base && in_range(log_off, 1, log_len, status)) log_base[0] = j;

    // ---- epilogue: out = O / l, lse = ln2 * (m + log2 l), l = sum of the parts
    float* red_l = red + 2 * kSplit * 128;
    red_l[part * 128 + row] = l_run;
    named_bar_sync(pair_bar, kGroup);
    float l_tot = 0.f;
#pragma unroll
    for (int p2 = 0; p2 < kSplit; ++p2) l_tot += red_l[p2 * 128 + row];
    if (ok && j > 0) {
      ok = mbar_wait(bar(C::bODone + (j - 1) % kBuf), (uint32_t)((j - 1) / kBuf) & 1,
                     abort_flag, kTimeoutNs);
      tc_fence_after();
    }
    if (ok) {
      const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
      const size_t row_off = ((orow + q_pos) * g.H_q + h) * D + part * kOC;
      const bool store = row_valid && in_range((long long)row_off, kOC, extent_q(gp), status);
      store_out_cols<kOC, kOutF32>(tO, j > 0, store, out, row_off, inv_l);
      if (row_valid && lse && part == 0 &&
          in_range((long long)(lrow + q_pos), 1, extent_lse(gp), status))
        lse[lrow + q_pos] =
            l_tot > 0.f ? (m_run + log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kSIssuerWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // a wait that expired anywhere, including the teardown drains, is reported
  if (threadIdx.x == 0 && (*abort_flag || *never) && status)
    atomicExch(status, (int)RA_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ host
using EncodeTiledFn = decltype(&cuTensorMapEncodeTiled);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// [B, S, H, D] bf16 tensor; box = 64 columns x 1 head x 128 rows x 1 batch,
// 128-byte swizzle (the layout tcgen05 reads with sw128 descriptors).
bool make_bshd_map(CUtensorMap* m, const void* ptr, int B, int S, int H, int D) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2,
                           (cuuint64_t)S * H * D * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)kTile, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool kOutF32, bool kVarlen = false>
ra_status launch_typed(const Geometry& g, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, void* out, float* lse, int* vlog,
                       int log_stride, int* status, cudaStream_t stream) {
  using C = Cfg<D>;
  auto kern = attn_tc_kernel<D, kOutF32, kVarlen>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes) != cudaSuccess)
    return RA_ERR_LAUNCH;
  const long long grid = (long long)g.n_seg * g.nt * g.B * g.H_q;   // one query tile per CTA
  if (grid > 0x7fffffffLL) return RA_ERR_RANGE;
  kern<<<(unsigned)grid, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, g, out, lse, vlog,
                                                            log_stride, status);
  return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_LAUNCH;
}

}  // namespace

ra_status launch_attn_tc_withheld(const Geometry& g0, const void* q, const void* k,
                                  const void* v, void* out, float* lse, int* dev_status,
                                  int sm_count, cudaStream_t stream) {
  Geometry g = g0;
  g.withhold_v0 = 1;
  return launch_attn_tc(g, q, k, v, out, lse, nullptr, 0, dev_status, sm_count, stream);
}

ra_status launch_attn_tc_varlen(const Geometry& g, const void* q, const void* k,
                                const void* v, void* out, float* lse, int* dev_status,
                                cudaStream_t stream) {
  // the packed tensors are mapped as one batch of `total` rows
  CUtensorMap mq, mk, mv;
  if (!make_bshd_map(&mq, q, 1, g.total, g.H_q, g.D) ||
      !make_bshd_map(&mk, k, 1, g.total, g.H_kv, g.D) ||
      !make_bshd_map(&mv, v, 1, g.total, g.H_kv, g.D))
    return RA_ERR_LAUNCH;
  if (g.D == 64)
    return launch_typed<64, false, true>(g, mq, mk, mv, out, lse, nullptr, 0, dev_status, stream);
  return launch_typed<128, false, true>(g, mq, mk, mv, out, lse, nullptr, 0, dev_status, stream);
}

ra_status launch_attn_tc_sharded(const Geometry& g, const void* q, const void* k,
                                 const void* v, void* out, float* lse, int* dev_status,
                                 cudaStream_t stream) {
  // [P, B, C, H, D] mapped as P*B batches of C rows
  const int nb = g.P * g.B, C = g.shard_rows;
  CUtensorMap mq, mk, mv;
  if (!make_bshd_map(&mq, q, nb, C, g.H_q, g.D) || !make_bshd_map(&mk, k, nb, C, g.H_kv, g.D) ||
      !make_bshd_map(&mv, v, nb, C, g.H_kv, g.D))
    return RA_ERR_LAUNCH;
  if (g.D == 64)
    return launch_typed<64, false>(g, mq, mk, mv, out, lse, nullptr, 0, dev_status, stream);
  return launch_typed<128, false>(g, mq, mk, mv, out, lse, nullptr, 0, dev_status, stream);
}

ra_status launch_attn_tc(const Geometry& g, const void* q, const void* k, const void* v,
                         void* out, float* lse, int* visit_log, int log_stride,
                         int* dev_status, int sm_count, cudaStream_t stream) {
  (void)sm_count;
  CUtensorMap mq, mk, mv;
  if (!make_bshd_map(&mq, q, g.B, g.S, g.H_q, g.D) ||
      !make_bshd_map(&mk, k, g.B, g.S, g.H_kv, g.D) ||
      !make_bshd_map(&mv, v, g.B, g.S, g.H_kv, g.D))
    return RA_ERR_LAUNCH;
  const bool f32_out = g.step >= 0;
  if (g.D == 64)
    return f32_out ? launch_typed<64, true>(g, mq, mk, mv, out, lse, visit_log, log_stride, dev_status, stream)
                   : launch_typed<64, false>(g, mq, mk, mv, out, lse, visit_log, log_stride, dev_status, stream);
  return f32_out ? launch_typed<128, true>(g, mq, mk, mv, out, lse, visit_log, log_stride, dev_status, stream)
                 : launch_typed<128, false>(g, mq, mk, mv, out, lse, visit_log, log_stride, dev_status, stream);
}

}  // namespace ra
