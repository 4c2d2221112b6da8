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
// One CTA owns a block of two adjacent 128-row query tiles (Q0 = rows 0-127,
// Q1 = rows 128-255 of the block) of one (batch, head) inside one segment of
// virtual rank r, and walks the key tiles of the ring in order, j = 0, 1, ...
// (tiles wholly after the block under a causal mask are left out). Both query
// tiles meet every key tile of that walk, so each K/V tile loaded from L2
// serves two query tiles; the one key tile of the walk that lies wholly after
// Q0 (the diagonal tile of Q1) reaches Q0 fully masked and adds nothing to it.
// "Receiving" a block is a TMA load of its tiles from this GPU's HBM/L2 into
// shared memory. Warp roles (320 threads at D = 128, 576 at D = 64):
//   softmax    two threads per query row (row = TMEM lane), 64 key columns
//              each (one warp holding a row's 128 scores loads them from TMEM
//              far more slowly than two warps holding 64 each). D = 128:
//              warps 0-7, for Q0 and then Q1 at every key tile. D = 64:
//              warps 0-7 for Q0 and 8-15 for Q1, side by side.
//   producer   (the next warp) TMA: Q0 and Q1 once, then K_j and V_j into
//              slot rings
//   issuer     (the last warp) TMEM allocator; one elected lane issues every
//              MMA
// Tensor memory (512 columns): S_i (128 f32 columns) at i * 128, softmax writes
// P_i as bf16 over the first 64 of them (D = 128) or over the first 32 of
// each part's 64 (D = 64); O_i (D columns) at 256 + i * D.
//
// The two query tiles give the SM two chains
//     S_i(j) -> softmax_i(j) -> PV_i(j) -> S_i(j+1) -> ...
// and the tensor core runs, per key tile j, PV0(j) S0(j+1) PV1(j) S1(j+1), so
// while the softmax works on one tile the tensor core runs the other tile's
// PV and S: with a softmax shorter than two products the tensor core never
// waits (at D = 64 the two tiles' softmax groups also run side by side, as
// the products there are short). S_i(j+1) overwrites P_i(j) right behind
// PV_i(j), which reads it:
// one thread issues both, and the tensor core executes the MMAs of a thread
// in issue order, so the read of P_i(j) precedes the write of S_i(j+1).
//
// Synchronisation (mbarriers in shared memory):
//   qfull[i]         TMA of Q_i landed
//   kfull/vfull[s]   TMA of K_j / V_j landed in slot s
//   done[j mod kKBuf] done(j): every MMA up to S1(j) is done, so K_j's slot
//                    and V_{j-1}'s slot may be refilled (one softmax thread
//                    arrives when it sees S1(j) complete)
//   sfull[i]         S_i(j) done (commit); it also covers PV_i(j-1), issued
//                    earlier by the same thread, so softmax may rescale O_i
//   pfull[i]         P_i(j) written and O_i rescaled (256 arrivals)
//   odone[i]         the last PV_i done (epilogue may read O_i)
//   staged[i]        bf16 output tile i staged in Q_i's buffer (D = 128, full
//                    tiles): the producer writes it out with TMA stores, one
//                    16 KB box of whole rows at a time, instead of every
//                    thread storing 16-byte pieces 8 KB apart
// Every barrier's next phase depends on its waiter's own progress, so parity
// waits are unambiguous.
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

#include "checks.cuh"
#include "fastmath.cuh"
#include "ra_internal.h"
#include "ring_iter.cuh"
#include "sm100.cuh"

namespace ra {
namespace {

using namespace sm100;
using namespace fastmath;

constexpr int kTile = 128;                 // rows of a query tile and of a key tile
constexpr int kBlockRows = 2 * kTile;      // query rows per CTA
// Warp roles by head size. D = 128: eight softmax warps run the softmax of
// Q0 and then of Q1 at every key tile (320 threads). D = 64, whose products
// take half as long: sixteen softmax warps, eight per query tile, run the two
// tiles' softmax side by side (576 threads; five warps share two of the
// sub-partitions, which caps a thread at 96 registers, so a softmax thread
// holds 32 scores at a time and reads each chunk from TMEM twice).
template <int D>
struct Roles {
  static constexpr bool kSplit = D == 64;
  static constexpr int kTileWarps = 8;                  // softmax warps on one tile at a time
  static constexpr int kSoftmaxWarps = kSplit ? 2 * kTileWarps : kTileWarps;
  static constexpr int kProducerWarp = kSoftmaxWarps;
  static constexpr int kMmaWarp = kSoftmaxWarps + 1;    // also allocates / frees TMEM
  static constexpr int kThreads = 32 * (kSoftmaxWarps + 2);
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;            // O_i at kOCol + i * D
constexpr float kRescaleLog2 = 8.0f;       // lazy rescale threshold (x256)
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kBoxBytes = kTile * 64 * 2;  // one TMA box: 128 rows x 64 bf16

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kBoxes = D / 64;
  static constexpr int kKBuf = D == 128 ? 2 : 3;   // K slots
  static constexpr int kVBuf = D == 128 ? 2 : 3;   // V slots
  static constexpr int kQOff = 0;                  // Q0, Q1
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKBuf * kTileBytes;
  static constexpr int kBarOff = kVOff + kVBuf * kTileBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kRedOff = kBarOff + kBarBytes;        // softmax exchange
  // maxima [2 parities][2 tiles][2 parts][128 rows], sums [2 tiles][2 parts][128 rows]
  static constexpr int kRedBytes = (1024 + 512) * 4;
  static constexpr int kUsed = kRedOff + kRedBytes + 1024;   // + alignment slack
  // More than half an SM's shared memory: one CTA per SM, so the 512-column
  // TMEM allocation never waits for another CTA.
  static constexpr int kSmemBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
  // barrier indices (8 bytes each)
  static constexpr int bQFull = 0;                  // [2]
  static constexpr int bKFull = 2;                  // [kKBuf]
  static constexpr int bVFull = bKFull + kKBuf;     // [kVBuf]
  static constexpr int bDone = bVFull + kVBuf;      // [kKBuf] ring: done(j) at j mod kKBuf
  static constexpr int bSFull = bDone + kKBuf;      // [2]
  static constexpr int bPFull = bSFull + 2;         // [2], 128 arrivals
  static constexpr int bODone = bPFull + 2;         // [2]
  static constexpr int bStaged = bODone + 2;        // [2] output tile i staged (8 warps, D = 128)
  static constexpr int bFinal = bStaged + 2;
  static constexpr int kNumBars = bFinal + 1;
  static constexpr int kHolderOff = kBarBytes - 16;   // TMEM base address
  static constexpr int kNeverOff = kBarBytes - 12;    // stays 0: waits that ignore aborts
  static constexpr int kAbortOff = kBarBytes - 8;     // abort flag
  static_assert(kNumBars * 8 <= kHolderOff, "barrier area overflow");
  static_assert(kSmemBytes > 116 * 1024, "must not fit two CTAs per SM");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kOCol + 2 * D <= kTmemCols, "tensor memory budget");
};

// Barrier among `count` threads of the CTA (ids 1-15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Three phase tests issued back to back (their shared-memory round trips
// overlap); true when all three phases have completed.
__device__ __forceinline__ bool mbar_test3(uint32_t b0, uint32_t p0, uint32_t b1, uint32_t p1,
                                           uint32_t b2, uint32_t p2) {
  const bool t0 = mbar_test_wait(b0, p0);
  const bool t1 = mbar_test_wait(b1, p1);
  const bool t2 = mbar_test_wait(b2, p2);
  return t0 && t1 && t2;
}

// The N columns of this thread's O row at tO, times alpha.
template <int N>
__device__ __forceinline__ void scale_cols(uint32_t tO, float alpha) {
#pragma unroll
  for (int c = 0; c < N / 32; ++c) {
    uint32_t uo[32];
    tmem_ld32(tO + c * 32, uo);
    tmem_ld_wait(uo);
#pragma unroll
    for (int i = 0; i < 32; ++i) uo[i] = __float_as_uint(__uint_as_float(uo[i]) * alpha);
    tmem_st32(tO + c * 32, uo);
  }
}

// Running 3-input maxima of 32 scores into 8 chains.
__device__ __forceinline__ void max_chunk(const uint32_t (&u)[32], float (&m8)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    m8[i] = fmax3(m8[i], __uint_as_float(u[i]), __uint_as_float(u[i + 8]));
#pragma unroll
  for (int i = 0; i < 8; ++i)
    m8[i] = fmax3(m8[i], __uint_as_float(u[16 + i]), __uint_as_float(u[24 + i]));
}

__device__ __forceinline__ float max8(const float (&m8)[8]) {
  return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

// p = 2^(s * scale * log2(e) - m) for 32 scores (packed FMA, two ex2 a pair),
// added to the two partial row sums and stored as 16 TMEM columns of bf16
// pairs at taddr.
__device__ __forceinline__ void exp_chunk(const uint32_t (&u)[32], uint64_t sl2x2,
                                          uint64_t neg_m2, uint64_t& sum2a, uint64_t& sum2b,
                                          uint32_t taddr) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t x2 =
        ffma2(pack2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1])), sl2x2, neg_m2);
    float x0, x1;
    unpack2(x2, x0, x1);
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    if (i & 1) sum2b = fadd2(sum2b, pack2(p0, p1));
    else sum2a = fadd2(sum2a, pack2(p0, p1));
    pk[i] = pack_bf16x2(p0, p1);
  }
  tmem_st16(taddr, pk);
}

// Epilogue of one softmax thread: its O row (N columns at tO), times 1/l, to
// `out` at element offset row_off (bf16, or float32 for single-step
// partials). Every thread loads (the TMEM load is warp-wide); valid rows store.
template <int N, bool kOutF32>
__device__ __forceinline__ void store_out_row(uint32_t tO, bool have_o, bool row_valid,
                                              void* out, size_t row_off, float inv_l) {
#pragma unroll
  for (int c = 0; c < N / 32; ++c) {
    uint32_t uo[32];
    if (have_o) {
      tmem_ld32(tO + c * 32, uo);
      tmem_ld_wait(uo);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) uo[i] = 0u;
    }
    if (!row_valid) continue;
    if constexpr (kOutF32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + row_off + c * 32);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(__uint_as_float(uo[4 * i]) * inv_l,
                             __uint_as_float(uo[4 * i + 1]) * inv_l,
                             __uint_as_float(uo[4 * i + 2]) * inv_l,
                             __uint_as_float(uo[4 * i + 3]) * inv_l);
    } else {
      uint4* dst =
          reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + row_off + c * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
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

// Epilogue of one softmax thread, staged for a TMA store: its N columns of
// O at tO (from column col0 of the row), times 1/l, as bf16 into the 128-row
// tile at smem_tile, laid out as the store's 64-column boxes with the
// 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r mod 8)).
template <int N>
__device__ __forceinline__ void stage_out_row(uint32_t tO, bool have_o, uint32_t smem_tile,
                                              int row, int col0, float inv_l) {
#pragma unroll
  for (int c = 0; c < N / 32; ++c) {
    uint32_t uo[32];
    if (have_o) {
      tmem_ld32(tO + c * 32, uo);
      tmem_ld_wait(uo);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) uo[i] = 0u;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int chunk = (col0 + c * 32) / 8 + i;          // 16-byte chunk of the row
      const uint32_t addr = smem_tile + (uint32_t)((chunk / 8) * kBoxBytes + row * 128 +
                                                   (((chunk % 8) ^ (row & 7)) * 16));
      const uint32_t w0 = pack_bf16x2(__uint_as_float(uo[8 * i + 0]) * inv_l, __uint_as_float(uo[8 * i + 1]) * inv_l);
      const uint32_t w1 = pack_bf16x2(__uint_as_float(uo[8 * i + 2]) * inv_l, __uint_as_float(uo[8 * i + 3]) * inv_l);
      const uint32_t w2 = pack_bf16x2(__uint_as_float(uo[8 * i + 4]) * inv_l, __uint_as_float(uo[8 * i + 5]) * inv_l);
      const uint32_t w3 = pack_bf16x2(__uint_as_float(uo[8 * i + 6]) * inv_l, __uint_as_float(uo[8 * i + 7]) * inv_l);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w0), "r"(w1),
                   "r"(w2), "r"(w3)
                   : "memory");
    }
  }
}

// S_i = Q_i K^T: M = 128 query rows, N = 128 keys, K = D in steps of 16.
template <int D>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, kTile, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    // 4 K steps of 16 columns per 64-column box; no carry into other fields
    const uint32_t off16 = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
    umma_ss(d_tmem, q_desc + off16, k_desc + off16, idesc, kk > 0 ? 1u : 0u);
  }
}

// O_i (+)= P_i V: A = P_i (bf16, TMEM), B = V (MN-major), M = 128, N = D,
// K = 128 keys in steps of 16 (8 TMEM columns of bf16 pairs each). P_i lies
// in the first 64 columns of S_i, or (kOwnCols) in the first 32 of each
// part's 64.
template <int D, bool kOwnCols>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, true);
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk)
    umma_ts(o_tmem, p_tmem + (kOwnCols ? (kk / 4) * 64 + (kk % 4) * 8 : kk * 8),
            v_desc + (uint64_t)((kk * 2048) >> 4), idesc, (accumulate || kk > 0) ? 1u : 0u);
}

template <int D, bool kOutF32, bool kVarlen, bool kWithholdV0>
__global__ void __launch_bounds__(Roles<D>::kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v,
               const __grid_constant__ CUtensorMap tm_o, const Geometry gp,
               void* __restrict__ out, float* __restrict__ lse,
               int* __restrict__ vlog, int log_stride, int* __restrict__ status,
               int tma_out) {
  using C = Cfg<D>;
  using R = Roles<D>;
  // Full bf16 output tiles go out through TMA stores at D = 128 (a row part
  // is 128 bytes); at D = 64 the per-row stores measured faster.
  constexpr bool kTmaOut = !kOutF32 && D == 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  auto bar = [&](int i) -> uint32_t { return base + C::kBarOff + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::kBarOff + C::kAbortOff);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + C::kBarOff + C::kHolderOff);
  volatile int* never = reinterpret_cast<volatile int*>(base_ptr + C::kBarOff + C::kNeverOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: one block of two query tiles. The query heads sharing a
  // kv head are innermost, so they read the same key tiles at the same time.
  // Blocks come by decreasing position (decreasing causal work, longest
  // first): within each (batch, kv head), which is outermost, so the CTAs
  // resident at one time read the keys/values of one or two kv heads and find
  // them in L2; or, when every head's keys and values fit in L2 (qb_major),
  // across all heads, so the grid ends with the shortest blocks of all.
  // With packed variable-length sequences, b is the sequence and the grid is
  // sized by the longest one; `g` is then this sequence's own geometry.
  const int grp = gp.H_q / gp.H_kv;
  const int nb = (gp.nt + 1) >> 1;                 // blocks per segment
  const int n_qb = gp.n_seg * nb;
  const int n_bhk = gp.B * gp.H_kv;
  const int hg = (int)(blockIdx.x % grp);
  const int rest = (int)(blockIdx.x / grp);
  const int qb = n_qb - 1 - (gp.qb_major ? rest / n_bhk : rest % n_qb);
  const int bhk = gp.qb_major ? rest % n_bhk : rest / n_qb;
  const int b = bhk / gp.H_kv, hk = bhk % gp.H_kv;
  const int h = hk * grp + hg;
  const int bh = b * gp.H_q + h;
  const int seg = qb / nb;
  const int blk = qb - seg * nb;
  Geometry gv;
  int row0 = 0;
  if constexpr (kVarlen) varlen_geometry(gp, b, gv, row0, threadIdx.x == 0 ? status : nullptr);
  const Geometry& g = kVarlen ? gv : gp;
  const int r = seg_owner(g, seg);
  const int q_lo = seg * g.seg_len + blk * kBlockRows;
  // rows of the block holding tokens (<= 0: padding only); Q1 takes part
  // only when it holds at least one
  const int q_valid = min(kBlockRows, seg_tokens(g, seg) - blk * kBlockRows);
  const bool two = q_valid > kTile;
  // TMA row and batch coordinates, first output row, first lse entry. In the
  // sequence-sharded layout [P, B, C, H, D] (mapped as [P*B, C, H, D]) the
  // block's segment is its shard p: batch p*B + b, rows from p*C.
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

  // The visit log holds one record per query tile: [count, 4 ints per
  // visit]; the block's tiles are tiles 2*blk and 2*blk + 1 of the segment
  // (the second exists only when the segment has that many tiles).
  const int n_qt = gp.n_seg * gp.nt;
  const int qt0 = seg * gp.nt + 2 * blk;
  const bool tile1_exists = 2 * blk + 1 < gp.nt;
  const long long log_len = (long long)gp.B * gp.H_q * n_qt * log_stride;
  auto log_off = [&](int i) -> long long {
    return ((long long)bh * n_qt + qt0 + i) * log_stride;
  };

  // A block of padding only (uneven or packed lengths) has nothing to compute
  // or write: the whole CTA leaves before it sets anything up.
  if (q_valid <= 0) {
    if (vlog && threadIdx.x == 0) {
      if (in_range(log_off(0), 1, log_len, status)) vlog[log_off(0)] = 0;
      if (tile1_exists && in_range(log_off(1), 1, log_len, status)) vlog[log_off(1)] = 0;
    }
    return;
  }

  // ---- set-up: barriers, abort flag, TMEM
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::bQFull + i), 1);
      mbar_init(bar(C::bSFull + i), 1);
      mbar_init(bar(C::bPFull + i), 32 * R::kTileWarps);
      mbar_init(bar(C::bODone + i), 1);
      if (kTmaOut) mbar_init(bar(C::bStaged + i), R::kSoftmaxWarps);
    }
    for (int i = 0; i < C::kKBuf; ++i) {
      mbar_init(bar(C::bKFull + i), 1);
      mbar_init(bar(C::bDone + i), 1);
    }
    for (int i = 0; i < C::kVBuf; ++i) mbar_init(bar(C::bVFull + i), 1);
    mbar_init(bar(C::bFinal), 1);
    *abort_flag = 0;
    *never = 0;
    fence_mbar_init();
  }
  if (warp == R::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  if (warp == R::kProducerWarp) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      for (int i = 0; i < (two ? 2 : 1); ++i) {
        const uint32_t q_smem = base + C::kQOff + i * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::bQFull + i), C::kTileBytes);
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_4d(q_smem + bx * kBoxBytes, &tm_q, bar(C::bQFull + i), bx * 64, h,
                      trow + q_lo + i * kTile, tbat);
      }
      // done(x) is phase x / kKBuf of ring barrier x mod kKBuf. The producer
      // waits for done(x) only while it has not loaded K_{x + kKBuf}, which
      // done(x + kKBuf) needs, so the barrier is never two phases ahead.
      auto wait_done = [&](int x) -> bool {
        return mbar_wait(bar(C::bDone + x % C::kKBuf), (uint32_t)(x / C::kKBuf) & 1, abort_flag,
                         kTimeoutNs);
      };
      KvIter it;
      it.init(g, r, q_lo, q_valid);
      KvTile kv;
      int j = 0;
      int ks = 0, kn = 0;      // K slot of tile j, and its use count
      int vs = 0, vn = 0;      // V slot of tile j, and its use count
      bool ok = true;
      while (ok && it.next(g, kv)) {
        // the key tile's own shard in the sequence-sharded layout
        const int krow = sharded ? -kv.seg * gp.shard_rows : trow;
        const int kbat = sharded ? kv.seg * gp.B + b : tbat;
        // K_j reuses the slot of K_{j-kKBuf}: free at done(j - kKBuf)
        if (kn > 0 && !wait_done(j - C::kKBuf)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(C::bKFull + ks), C::kTileBytes);
        for (int bx = 0; bx < C::kBoxes; ++bx)
          tma_load_4d(base + C::kKOff + ks * C::kTileBytes + bx * kBoxBytes, &tm_k,
                      bar(C::bKFull + ks), bx * 64, hk, krow + kv.lo, kbat);
        // V_j reuses the slot of V_{j-kVBuf}: free at done(j - kVBuf + 1)
        if (vn > 0 && !wait_done(j - C::kVBuf + 1)) {
          ok = false;
          break;
        }
        if (!(kWithholdV0 && j == 0)) {      // test of the expiry path only
          mbar_arrive_expect_tx(bar(C::bVFull + vs), C::kTileBytes);
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_4d(base + C::kVOff + vs * C::kTileBytes + bx * kBoxBytes, &tm_v,
                        bar(C::bVFull + vs), bx * 64, hk, krow + kv.lo, kbat);
        }
        ++j;
        if (++ks == C::kKBuf) { ks = 0; ++kn; }
        if (++vs == C::kVBuf) { vs = 0; ++vn; }
      }
      // Every issued load lands before the CTA leaves (already true unless
      // the CTA aborted): the last use of each slot.
      const int nk = j;
      for (int jj = (nk > C::kKBuf ? nk - C::kKBuf : 0); jj < nk; ++jj)
        mbar_wait(bar(C::bKFull + jj % C::kKBuf), (uint32_t)(jj / C::kKBuf) & 1, never,
                  kTimeoutNs);
      for (int jj = (nk > C::kVBuf ? nk - C::kVBuf : 0); jj < nk; ++jj)
        if (!(kWithholdV0 && jj == 0))
          mbar_wait(bar(C::bVFull + jj % C::kVBuf), (uint32_t)(jj / C::kVBuf) & 1, never,
                    kTimeoutNs);
      for (int i = 0; i < (two ? 2 : 1); ++i) mbar_wait(bar(C::bQFull + i), 0, never, kTimeoutNs);
      // full output tiles, once the softmax warps have staged them in Q_i's
      // buffer: one TMA store of whole rows each; their shared memory is read
      // before the CTA leaves
      if (kTmaOut && tma_out && ok) {
        for (int i = 0; i < (two ? 2 : 1); ++i) {
          if (q_valid - i * kTile < kTile) continue;
          if (!mbar_wait(bar(C::bStaged + i), 0, abort_flag, kTimeoutNs)) break;
          const uint32_t tile_smem = base + C::kQOff + (uint32_t)(i * C::kTileBytes);
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_store_4d(&tm_o, tile_smem + bx * kBoxBytes, bx * 64, h, trow + q_lo + i * kTile,
                         tbat);
          bulk_commit_group();
        }
        bulk_wait_read_all();
      }
    }
    __syncwarp();
  } else if (warp == R::kMmaWarp) {
    // ======================= MMA issuer =======================
    // One thread issues every MMA, so each product runs on the tensor core
    // as one uninterrupted group into its accumulator (MMAs of two threads
    // interleaved measured much slower). Per key tile j: PV0(j) S0(j+1)
    // PV1(j) S1(j+1). Between groups the warp only tests barriers: the
    // tensor core runs just the few MMAs queued behind the last issue, so any
    // longer stop here would leave it idle. The whole warp runs the loop, so
    // its descriptor arithmetic is warp-uniform; one elected lane issues the
    // MMAs and commits (a commit tracks the MMAs of the thread that issues
    // it).
    {
      const bool leader = elect_one_sync();
      // Descriptors differ only in the start-address field (bits 0-13, in
      // 16-byte units, no carry: shared addresses are < 256 KB), so they are
      // built once and offset per K step and slot.
      const uint64_t q_desc = sw128_desc(base + C::kQOff, 16, 1024);
      const uint64_t k_desc = sw128_desc(base + C::kKOff, 16, 1024);
      const uint64_t v_desc = sw128_desc(base + C::kVOff, kBoxBytes, 1024);
      const uint64_t q1_off = (uint64_t)(C::kTileBytes >> 4);
      const uint32_t tS0 = tmem, tS1 = tmem + kTile;
      const uint32_t tO0 = tmem + kOCol, tO1 = tmem + kOCol + D;
      // the walk's length, counted while Q lands
      const int n = kv_walk_length(g, r, q_lo, q_valid);
      bool ok = mbar_wait_warp(bar(C::bQFull), 0, abort_flag, kTimeoutNs) &&
                (!two || mbar_wait_warp(bar(C::bQFull + 1), 0, abort_flag, kTimeoutNs));
      if (ok && n > 0) {
        ok = mbar_wait_warp(bar(C::bKFull), 0, abort_flag, kTimeoutNs);
        if (ok) {
          tc_fence_after();
          if (leader) {
            issue_s<D>(tS0, q_desc, k_desc);
            umma_commit(bar(C::bSFull));
            if (two) {
              issue_s<D>(tS1, q_desc + q1_off, k_desc);
              umma_commit(bar(C::bSFull + 1));
            }
          }
          __syncwarp();
        }
      }
      int ks = 0, kn = 0, vs = 0, vn = 0;
      for (int j = 0; ok && j < n; ++j) {
        const bool last = j + 1 == n;
        int nks = ks + 1, nkn = kn;
        if (nks == C::kKBuf) { nks = 0; ++nkn; }
        const uint64_t vd = v_desc + (uint64_t)((vs * C::kTileBytes) >> 4);
        const uint64_t kd = k_desc + (uint64_t)((nks * C::kTileBytes) >> 4);
        // V_j and K_{j+1} have almost always landed long before P0(j): test
        // all three at once and wait one by one only when one is missing
        const uint32_t kb = bar(C::bKFull + (last ? ks : nks));
        const uint32_t kp = last ? (uint32_t)kn & 1 : (uint32_t)nkn & 1;
        if (!__all_sync(0xffffffffu, mbar_test3(bar(C::bVFull + vs), (uint32_t)vn & 1, kb, kp,
                                                bar(C::bPFull), (uint32_t)j & 1)))
          ok = mbar_wait_warp(bar(C::bVFull + vs), (uint32_t)vn & 1, abort_flag, kTimeoutNs) &&
               mbar_wait_warp(kb, kp, abort_flag, kTimeoutNs) &&
               mbar_wait_warp(bar(C::bPFull), (uint32_t)j & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        // PV0(j), then S0(j+1) over the same columns
        if (leader) {
          issue_pv<D, R::kSplit>(tO0, tS0, vd, j > 0);
          if (last) {
            umma_commit(bar(C::bODone));
          } else {
            issue_s<D>(tS0, q_desc, kd);
            umma_commit(bar(C::bSFull));
          }
        }
        __syncwarp();
        // PV1(j), then S1(j+1)
        if (two) {
          ok = mbar_wait_warp(bar(C::bPFull + 1), (uint32_t)j & 1, abort_flag, kTimeoutNs);
          if (!ok) break;
          tc_fence_after();
          if (leader) {
            issue_pv<D, R::kSplit>(tO1, tS1, vd, j > 0);
            if (last) {
              umma_commit(bar(C::bODone + 1));
            } else {
              issue_s<D>(tS1, q_desc + q1_off, kd);
              umma_commit(bar(C::bSFull + 1));
            }
          }
          __syncwarp();
        }
        ks = nks;
        kn = nkn;
        if (++vs == C::kVBuf) { vs = 0; ++vn; }
      }
      // all tensor-core work this warp issued has completed before teardown
      if (leader) {
        umma_commit(bar(C::bFinal));
        mbar_wait(bar(C::bFinal), 0, never, kTimeoutNs);
      }
    }
    __syncwarp();
  } else if (warp < R::kSoftmaxWarps) {
    if constexpr (R::kSplit) {
      // ============ softmax: warps 0-7 serve Q0, warps 8-15 serve Q1 ============
      // Two threads per query row: warps w and w+4 of a tile share TMEM lane
      // quarter w % 4 (the same 32 rows); part p takes key columns [64p, 64p+64)
      // of S_i and O columns [pD/2, (p+1)D/2). The two tiles' softmax warps run
      // side by side, so one tile's softmax overlaps the other's and the tensor
      // core's PV and S of the other tile. A row's two partial maxima meet in
      // shared memory at one named barrier of the pair; each part writes its P
      // into its own 64 columns and keeps its own partial sums, added in the
      // epilogue.
      const int qi = warp / R::kTileWarps;          // query tile served
      const int wq = warp & 3;                   // TMEM lane quarter
      const int part = (warp >> 2) & 1;          // column part
      const int row = wq * 32 + lane;
      const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
      const float sl2 = g.scale_log2;
      const uint64_t sl2x2 = pack2(sl2, sl2);
      const uint32_t pair_bar = 1 + qi * 4 + wq; // named barrier of the row's two warps
      const uint32_t tS = tmem + t_lane + (uint32_t)(qi * kTile);
      const uint32_t tOp = tmem + t_lane + kOCol + (uint32_t)(qi * D + part * (D / 2));
      const int qt_lo = q_lo + qi * kTile;
      const int q_pos = qt_lo + row;
      // [2 exchange parities][2 tiles][2 parts][128 rows] partial maxima, then
      // [2 tiles][2 parts][128 rows] partial sums
      float* red = reinterpret_cast<float*>(base_ptr + C::kRedOff);
      int ex = 0;                                // exchanges so far (buffer parity)
      float m_run = -INFINITY, l_run = 0.f;
      int j = 0;                                 // key tiles done
      bool ok = true;
      if (qi == 0 || two) {
        // one visit record per query tile, written by the tile's first thread
        int* log = (vlog && warp == qi * R::kTileWarps && lane == 0) ? vlog + log_off(qi) : nullptr;
        int n_log = 0;
        const int q_last = q_lo + min(kTile * (qi + 1), q_valid) - 1;
        KvIter it;
        it.init(g, r, q_lo, q_valid);
        KvTile kv;
        bool have = it.next(g, kv);
        // One thread arrives on done(j) once S(j) of the last tile is done: the
        // producer's signal that K_j's and V_{j-1}'s slots may be refilled.
        const bool relay = lane == 0 && warp == (two ? R::kTileWarps : 0);
        int rd = 0;
        while (have) {
          // a key tile wholly after the query tile is not part of its own walk
          // (it reaches the tile fully masked)
          if (log && !(g.causal && kv.lo > q_last) &&
              in_range(log_off(qi) + 1 + 4 * n_log, 4, log_len, status))
            log_visit(log, n_log++, kv, tile_class(g, qt_lo, kv));
          float* red_e = red + (ex & 1) * 512 + qi * 256;
          ++ex;
          if (ok) ok = mbar_wait_warp(bar(C::bSFull + qi), (uint32_t)j & 1, abort_flag, kTimeoutNs);
          if (!ok) {
            // keep meeting the partner at every exchange so it never waits alone
            named_bar_sync(pair_bar, 64);
            ++j;
            have = it.next(g, kv);
            continue;
          }
          tc_fence_after();
          // tiles the causal rule cuts for this query tile, and ragged tails:
          // columns from lim on (of this part's 64) are masked
          const bool all_allowed = !g.causal || kv.lo + kv.valid - 1 <= qt_lo;
          const bool cut = !(all_allowed && kv.valid == kTile);
          const int lim = (g.causal ? min(kv.valid, q_pos - kv.lo + 1) : kv.valid) - part * 64;
          float m8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t u[32];
            tmem_ld32(tS + part * 64 + c * 32, u);
            if (relay && c == 0) {
              mbar_arrive(bar(C::bDone + rd));
              if (++rd == C::kKBuf) rd = 0;
            }
            tmem_ld_wait();
            reg_fence(u);
            if (cut) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c * 32 + i >= lim) u[i] = __float_as_uint(-INFINITY);
            }
            max_chunk(u, m8);
          }
          red_e[part * 128 + row] = max8(m8);
          named_bar_sync(pair_bar, 64);
          const float mx = fmaxf(red_e[row], red_e[128 + row]);
          const float m_new = fmaxf(m_run, mx * sl2);
          const bool resc = m_new > m_run + kRescaleLog2;
          float alpha = 1.f;
          if (resc) {
            alpha = ex2_approx(m_run - m_new);         // 0 when m_run = -inf
            m_run = m_new;
            l_run *= alpha;
          }
          const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
          const uint64_t neg_m2 = pack2(-m_use, -m_use);
          uint64_t sum2a = pack2(0.f, 0.f), sum2b = sum2a;
          // the scores again, 32 at a time; P of chunk c (bf16 pairs) goes to
          // this part's own columns 64p + 16c .. 64p + 16c + 15, which hold
          // scores already read
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t u[32];
            tmem_ld32(tS + part * 64 + c * 32, u);
            tmem_ld_wait();
            reg_fence(u);
            if (cut) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c * 32 + i >= lim) u[i] = __float_as_uint(-INFINITY);
            }
            exp_chunk(u, sl2x2, neg_m2, sum2a, sum2b, tS + part * 64 + c * 16);
          }
          {
            float a0, a1;
            unpack2(fadd2(sum2a, sum2b), a0, a1);
            l_run += a0 + a1;
          }
          // O_i is scaled by alpha before P_i(j) V_j is added to it; PV_i(j-1)
          // is done (S_i(j)'s completion covers it). Both parts take the same
          // decision for a row.
          if (__any_sync(0xffffffffu, resc) && j > 0) scale_cols<D / 2>(tOp, alpha);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(C::bPFull + qi));
          ++j;
          have = it.next(g, kv);
        }
        if (log && in_range(log_off(qi), 1, log_len, status)) log[0] = n_log;

        // ---- epilogue: out = O / l, lse = ln2 * (m + log2 l), l = sum of both parts
        float* red_l = red + 1024 + qi * 256;
        red_l[part * 128 + row] = l_run;
        named_bar_sync(pair_bar, 64);
        const float l_tot = red_l[row] + red_l[128 + row];
        const bool row_valid = row < min(kTile, q_valid - qi * kTile);
        if (ok && j > 0) {
          ok = mbar_wait_warp(bar(C::bODone + qi), 0, abort_flag, kTimeoutNs);
          tc_fence_after();
        }
        if (ok) {
          const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
          const size_t row_off = ((orow + q_pos) * g.H_q + h) * D + part * (D / 2);
          const bool store = row_valid && in_range((long long)row_off, D / 2, extent_q(gp), status);
          store_out_row<D / 2, kOutF32>(tOp, j > 0, store, out, row_off, inv_l);
          if (row_valid && lse && part == 0 &&
              in_range((long long)(lrow + q_pos), 1, extent_lse(gp), status))
            lse[lrow + q_pos] =
                l_tot > 0.f ? (m_run + log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
        }
      } else if (vlog && warp == R::kTileWarps && lane == 0 && tile1_exists &&
                 in_range(log_off(1), 1, log_len, status)) {
        // a second query tile of padding only has an empty record
        vlog[log_off(1)] = 0;
      }
    } else {
      // ============ softmax: two threads per query row, Q0 and Q1 in turn ============
      // Warps w and w+4 share TMEM lane quarter w % 4 (the same 32 rows of each
      // query tile); part p = w / 4 takes key columns [64p, 64p+64) of S_i and
      // O columns [pD/2, (p+1)D/2). Per key tile the eight warps run softmax of
      // Q0, then of Q1. A row's two partial maxima meet in shared memory at one
      // named barrier of the pair (which also orders both parts' S loads before
      // either part writes P over the first 64 S columns); each part keeps its
      // own partial sums, added in the epilogue.
      const int wq = warp & 3;                   // TMEM lane quarter
      const int part = warp >> 2;                // column part
      const int row = wq * 32 + lane;
      const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
      const int ntile = two ? 2 : 1;
      const float sl2 = g.scale_log2;
      const uint64_t sl2x2 = pack2(sl2, sl2);
      const uint32_t pair_bar = 1 + wq;          // named barrier of the row's two warps
      // [2 exchange parities][2 parts][128 rows] partial maxima, then
      // [2 tiles][2 parts][128 rows] partial sums
      float* red = reinterpret_cast<float*>(base_ptr + C::kRedOff);
      int ex = 0;                                // exchanges so far (buffer parity)

      // one visit record per query tile, written by one thread
      int* log0 = (vlog && warp == 0 && lane == 0) ? vlog + log_off(0) : nullptr;
      int* log1 = (log0 && two) ? vlog + log_off(1) : nullptr;
      int n_log0 = 0, n_log1 = 0;

      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
      int j = 0;               // key tiles done
      bool ok = true;
      KvIter it;
      it.init(g, r, q_lo, q_valid);
      KvTile kv;
      bool have = it.next(g, kv);
      // One thread arrives on done(j) once S(j) of the last tile is done: the
      // producer's signal that K_j's and V_{j-1}'s slots may be refilled.
      const bool relay = warp == 0 && lane == 0;
      int rd = 0;
      while (have) {
        if (log0) {
          // a key tile wholly after query tile i is not part of its own walk
          // (it reaches the tile fully masked)
          if (!(g.causal && kv.lo > q_lo + min(kTile, q_valid) - 1) &&
              in_range(log_off(0) + 1 + 4 * n_log0, 4, log_len, status))
            log_visit(log0, n_log0++, kv, tile_class(g, q_lo, kv));
          if (log1 && !(g.causal && kv.lo > q_lo + q_valid - 1) &&
              in_range(log_off(1) + 1 + 4 * n_log1, 4, log_len, status))
            log_visit(log1, n_log1++, kv, tile_class(g, q_lo + kTile, kv));
        }
#pragma unroll
        for (int qi = 0; qi < 2; ++qi) {
          if (qi >= ntile) break;
          const uint32_t tS = tmem + t_lane + (uint32_t)(qi * kTile);
          const int qt_lo = q_lo + qi * kTile;
          const int q_pos = qt_lo + row;
          float* red_e = red + (ex & 1) * 256;
          ++ex;
          if (ok) ok = mbar_wait_warp(bar(C::bSFull + qi), (uint32_t)j & 1, abort_flag, kTimeoutNs);
          if (!ok) {
            // keep meeting the partner at every exchange so it never waits alone
            named_bar_sync(pair_bar, 64);
            continue;
          }
          tc_fence_after();
          uint32_t uu[2][32];
          tmem_ld32(tS + part * 64, uu[0]);
          tmem_ld32(tS + part * 64 + 32, uu[1]);
          if (relay && qi == ntile - 1) {
            mbar_arrive(bar(C::bDone + rd));
            if (++rd == C::kKBuf) rd = 0;
          }
          tmem_ld_wait();
          reg_fence(uu[0]);
          reg_fence(uu[1]);
          // tiles the causal rule cuts for this query tile, and ragged tails
          const bool all_allowed = !g.causal || kv.lo + kv.valid - 1 <= qt_lo;
          if (!(all_allowed && kv.valid == kTile)) {
            const int lim = (g.causal ? min(kv.valid, q_pos - kv.lo + 1) : kv.valid) - part * 64;
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c >= lim) uu[c / 32][c % 32] = __float_as_uint(-INFINITY);
          }
          float m8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
          max_chunk(uu[0], m8);
          max_chunk(uu[1], m8);
          red_e[part * 128 + row] = max8(m8);
          tc_fence_before();
          named_bar_sync(pair_bar, 64);
          tc_fence_after();
          const float mx = fmaxf(red_e[row], red_e[128 + row]);
          const float m_new = fmaxf(m_run[qi], mx * sl2);
          const bool resc = m_new > m_run[qi] + kRescaleLog2;
          float alpha = 1.f;
          if (resc) {
            alpha = ex2_approx(m_run[qi] - m_new);     // 0 when m_run = -inf
            m_run[qi] = m_new;
            l_run[qi] *= alpha;
          }
          const float m_use = (m_run[qi] == -INFINITY) ? 0.f : m_run[qi];
          const uint64_t neg_m2 = pack2(-m_use, -m_use);
          uint64_t sum2a = pack2(0.f, 0.f), sum2b = sum2a;
          // P of this part's 64 keys: TMEM columns 32p..32p+31 of S_i
          exp_chunk(uu[0], sl2x2, neg_m2, sum2a, sum2b, tS + part * 32);
          exp_chunk(uu[1], sl2x2, neg_m2, sum2a, sum2b, tS + part * 32 + 16);
          {
            float a0, a1;
            unpack2(fadd2(sum2a, sum2b), a0, a1);
            l_run[qi] += a0 + a1;
          }
          // O_i is scaled by alpha before P_i(j) V_j is added to it; PV_i(j-1)
          // is done (S_i(j)'s completion covers it). Both parts take the same
          // decision for a row.
          if (__any_sync(0xffffffffu, resc) && j > 0)
            scale_cols<D / 2>(tmem + t_lane + kOCol + (uint32_t)(qi * D + part * (D / 2)), alpha);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(C::bPFull + qi));
        }
        ++j;
        have = it.next(g, kv);
      }
      if (log0 && in_range(log_off(0), 1, log_len, status)) log0[0] = n_log0;
      if (log1 && in_range(log_off(1), 1, log_len, status)) log1[0] = n_log1;
      // a second query tile of padding only has an empty record
      if (log0 && !two && tile1_exists && in_range(log_off(1), 1, log_len, status))
        vlog[log_off(1)] = 0;

      // ---- epilogue: out = O / l, lse = ln2 * (m + log2 l), l = sum of both parts
      float* red_l = red + 512;
      for (int qi = 0; qi < ntile; ++qi) red_l[(qi * 2 + part) * 128 + row] = l_run[qi];
      named_bar_sync(pair_bar, 64);
      for (int qi = 0; qi < ntile; ++qi) {
        const float l_tot = red_l[qi * 256 + row] + red_l[qi * 256 + 128 + row];
        const int qt_lo = q_lo + qi * kTile;
        const int q_pos = qt_lo + row;
        const bool row_valid = row < min(kTile, q_valid - qi * kTile);
        if (ok && j > 0) {
          ok = mbar_wait_warp(bar(C::bODone + qi), 0, abort_flag, kTimeoutNs);
          tc_fence_after();
        }
        if (!ok) break;
        const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
        const uint32_t tO = tmem + t_lane + kOCol + (uint32_t)(qi * D + part * (D / 2));
        if (kTmaOut && tma_out && q_valid - qi * kTile >= kTile) {
          // a full tile: staged in Q_i's buffer (every MMA reading it is done)
          // and written by one TMA store of whole rows
          const uint32_t tile_smem = base + C::kQOff + (uint32_t)(qi * C::kTileBytes);
          stage_out_row<D / 2>(tO, j > 0, tile_smem, row, part * (D / 2), inv_l);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::bStaged + qi));   // the producer stores it
        } else {
          const size_t row_off = ((orow + q_pos) * g.H_q + h) * D + part * (D / 2);
          const bool store = row_valid && in_range((long long)row_off, D / 2, extent_q(gp), status);
          store_out_row<D / 2, kOutF32>(tO, j > 0, store, out, row_off, inv_l);
        }
        if (row_valid && lse && part == 0 &&
            in_range((long long)(lrow + q_pos), 1, extent_lse(gp), status))
          lse[lrow + q_pos] =
              l_tot > 0.f ? (m_run[qi] + log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // a wait that expired anywhere, including the teardown drains, is reported
  if (threadIdx.x == 0 && (*abort_flag || *never) && status)
    atomicExch(status, (int)RA_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ host
template <int D, bool kOutF32, bool kVarlen = false, bool kWithholdV0 = false>
ra_status launch_typed(const Geometry& g, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mo, bool tma_out, void* out,
                       float* lse, int* vlog, int log_stride, int* status, cudaStream_t stream) {
  using C = Cfg<D>;
  auto kern = attn_tc_kernel<D, kOutF32, kVarlen, kWithholdV0>;
  // keys and values of every head within half of the 126 MB L2: order the
  // grid longest block first across all heads
  Geometry gl = g;
  const long long kv_rows = g.cu_seqlens ? g.total
                            : (g.shard_rows > 0 ? (long long)g.P * g.B * g.shard_rows
                                                : (long long)g.B * g.S);
  gl.qb_major = kv_rows * g.H_kv * g.D * 2 * 2 <= (64ll << 20) ? 1 : 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes) != cudaSuccess)
    return RA_ERR_LAUNCH;
  // one block of two query tiles per CTA
  const long long grid = (long long)g.n_seg * ((g.nt + 1) / 2) * g.B * g.H_q;
  if (grid > 0x7fffffffLL) return RA_ERR_RANGE;
  kern<<<(unsigned)grid, Roles<D>::kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, mo, gl, out, lse, vlog,
                                                            log_stride, status, tma_out ? 1 : 0);
  return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_LAUNCH;
}

// q, k, v of [nb, rows, H, D] bf16 (natural, packed or sequence-sharded view)
bool make_maps(CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv, const Geometry& g,
               const void* q, const void* k, const void* v, int nb, int rows) {
  return make_bshd_map(mq, q, nb, rows, g.H_q, g.D, kTile) &&
         make_bshd_map(mk, k, nb, rows, g.H_kv, g.D, kTile) &&
         make_bshd_map(mv, v, nb, rows, g.H_kv, g.D, kTile);
}

// The bf16 output, laid out like q, as a TMA store target. False (the kernel
// then stores row by row) when the pointer does not suit a tensor map, and
// always in the checked build, whose per-row stores check every offset.
bool make_out_map(CUtensorMap* mo, const Geometry& g, const void* out, int nb, int rows) {
#ifdef RA_DEBUG_CHECKS
  (void)mo; (void)g; (void)out; (void)nb; (void)rows;
  return false;
#else
  if (reinterpret_cast<uintptr_t>(out) % 16 != 0) return false;
  return make_bshd_map(mo, out, nb, rows, g.H_q, g.D, kTile);
#endif
}

}  // namespace

ra_status launch_attn_tc_withheld(const Geometry& g, const void* q, const void* k,
                                  const void* v, void* out, float* lse, int* dev_status,
                                  cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mo;
  if (!make_maps(&mq, &mk, &mv, g, q, k, v, g.B, g.S)) return RA_ERR_LAUNCH;
  if (g.D != 128) return RA_ERR_HEADDIM;
  const bool tma_out = make_out_map(&mo, g, out, g.B, g.S);
  return launch_typed<128, false, false, true>(g, mq, mk, mv, mo, tma_out, out, lse, nullptr, 0,
                                               dev_status, stream);
}

ra_status launch_attn_tc_varlen(const Geometry& g, const void* q, const void* k,
                                const void* v, void* out, float* lse, int* dev_status,
                                cudaStream_t stream) {
  // the packed tensors are mapped as one batch of `total` rows
  CUtensorMap mq, mk, mv, mo;
  if (!make_maps(&mq, &mk, &mv, g, q, k, v, 1, g.total)) return RA_ERR_LAUNCH;
  const bool tma_out = make_out_map(&mo, g, out, 1, g.total);
  if (g.D == 64)
    return launch_typed<64, false, true>(g, mq, mk, mv, mo, tma_out, out, lse, nullptr, 0,
                                         dev_status, stream);
  return launch_typed<128, false, true>(g, mq, mk, mv, mo, tma_out, out, lse, nullptr, 0,
                                        dev_status, stream);
}

ra_status launch_attn_tc_sharded(const Geometry& g, const void* q, const void* k,
                                 const void* v, void* out, float* lse, int* dev_status,
                                 cudaStream_t stream) {
  // [P, B, C, H, D] mapped as P*B batches of C rows
  CUtensorMap mq, mk, mv, mo;
  if (!make_maps(&mq, &mk, &mv, g, q, k, v, g.P * g.B, g.shard_rows)) return RA_ERR_LAUNCH;
  const bool tma_out = make_out_map(&mo, g, out, g.P * g.B, g.shard_rows);
  if (g.D == 64)
    return launch_typed<64, false>(g, mq, mk, mv, mo, tma_out, out, lse, nullptr, 0, dev_status,
                                   stream);
  return launch_typed<128, false>(g, mq, mk, mv, mo, tma_out, out, lse, nullptr, 0, dev_status,
                                  stream);
}

ra_status launch_attn_tc(const Geometry& g, const void* q, const void* k, const void* v,
                         void* out, float* lse, int* visit_log, int log_stride,
                         int* dev_status, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mo;
  if (!make_maps(&mq, &mk, &mv, g, q, k, v, g.B, g.S)) return RA_ERR_LAUNCH;
  const bool f32_out = g.step >= 0;
  // single-step partials are float32: stored row by row
  const bool tma_out = !f32_out && make_out_map(&mo, g, out, g.B, g.S);
  if (g.D == 64)
    return f32_out ? launch_typed<64, true>(g, mq, mk, mv, mo, false, out, lse, visit_log, log_stride, dev_status, stream)
                   : launch_typed<64, false>(g, mq, mk, mv, mo, tma_out, out, lse, visit_log, log_stride, dev_status, stream);
  return f32_out ? launch_typed<128, true>(g, mq, mk, mv, mo, false, out, lse, visit_log, log_stride, dev_status, stream)
                 : launch_typed<128, false>(g, mq, mk, mv, mo, tma_out, out, lse, visit_log, log_stride, dev_status, stream);
}

}  // namespace ra
