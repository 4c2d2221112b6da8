// Exact ring attention on the tcgen05 tensor cores (bf16 in, f32 accumulate).
//
// Glossary "sequence parallelism transformers":
//  - §Ring Attention: each virtual rank keeps its query block; at step t it
//    attends to the key/value block of rank (r - t) mod P ("receive from
//    i-1"), and accumulates outputs; only the local block and the received
//    block need to be resident ("Memory Efficiency").
//  - §Flash Attention with Sequence Parallelism: attention is computed tile
//    by tile (prior art; the tiling below is laid out for sm_103a).
//  - §Implementation Considerations: the softmax normalisation across blocks
//    is kept exact with a running maximum and sum (log-sum-exp merge).
//
// One CTA owns a pair of 128-row query tiles of one (batch, head) inside one
// segment of virtual rank r, and walks the key tiles of the ring in order.
// "Receiving" a block is a TMA load of its tile from this GPU's HBM/L2 into a
// shared-memory ring of slots (K_0, V_0, K_1, V_1, ... in load order, so a
// load can start as soon as the slot of the load kSlots earlier is free).
// Warp roles (352 threads):
//   warps 0-3  softmax for query tile 0 (one thread per row = TMEM lane)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q once, then K/V tiles into the slot ring
//   warp  9    TMEM allocator and single-thread tcgen05.mma issuer
//   warps 10-11 spare (complete the third warpgroup for register re-allocation)
// The third warpgroup gives registers to the softmax warpgroups
// (setmaxnreg: 168 at launch; 56 for warps 8-11, 224 for warps 0-7;
// 128*56 + 256*224 = 384*168, the block's launch allocation).
// Tensor memory (512 columns): tile k uses columns [256k, 256k+128) for the
// f32 scores S = Q K^T, reused in place for P (bf16, packed two per column,
// 64 columns) and [256k+128, 256k+128+D) for the f32 output accumulator O.
// Per key tile j: S_k = Q_k K_j^T (SS MMA) -> softmax reads S_k, writes P_k,
// rescales O_k if its running max moved by more than 2^8 -> O_k += P_k V_j
// (TS MMA, P from TMEM). The running (max, sum, O) carried across ring steps
// is the in-register form of the log-sum-exp merge of per-step partials.
//
// Every wait is bounded: after kTimeoutNs a thread raises a CTA-wide abort
// flag, every role falls through to the common teardown (which still waits,
// bounded, for the tensor-core work it issued, then frees TMEM), and the
// kernel reports RA_ERR_TIMEOUT through the status word.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "ra_internal.h"
#include "ring_iter.cuh"
#include "sm100.cuh"

namespace ra {
namespace {

using namespace sm100;

constexpr int kTile = 128;
constexpr int kThreads = 384;         // 3 warpgroups; warps 10-11 only take part in set-up
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;           // also allocates / frees TMEM
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;          // lazy rescale threshold (x256)
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kBoxBytes = kTile * 64 * 2;      // one TMA box: 128 rows x 64 bf16

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kBoxes = D / 64;
  static constexpr int kSlots = D == 128 ? 5 : 8;     // K/V slot ring
  static constexpr int kQOff = 0;
  static constexpr int kSlotOff = kQOff + 2 * kTileBytes;
  static constexpr int kBarOff = kSlotOff + kSlots * kTileBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kFlagsOff = kBarBytes;          // 16 x u32: key-tile flags ring
  static constexpr int kFlagsBytes = 64;
  static constexpr int kSmemBytes = kBarOff + kBarBytes + kFlagsBytes + 1024;   // + alignment slack
  // barrier indices (8 bytes each)
  static constexpr int bQFull = 0;
  static constexpr int bFull = 1;                      // [kSlots]
  static constexpr int bEmpty = bFull + kSlots;        // [kSlots]
  static constexpr int bSFull = bEmpty + kSlots;       // [2]
  static constexpr int bPFull = bSFull + 2;            // [2]
  static constexpr int bODone = bPFull + 2;            // [2]
  static constexpr int bFinal = bODone + 2;
  static constexpr int kNumBars = bFinal + 1;
  static constexpr int kHolderOff = kBarBytes - 16;    // TMEM base address
  static constexpr int kNeverOff = kBarBytes - 12;     // stays 0: waits that ignore aborts
  static constexpr int kAbortOff = kBarBytes - 8;      // abort flag
  static_assert(kNumBars * 8 <= kHolderOff, "barrier area overflow");
  // one CTA per SM: the kernel owns all 512 TMEM columns
  static_assert(kSmemBytes > 116 * 1024, "must not fit two CTAs per SM");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ uint32_t s_col(int k) { return (uint32_t)(k * 256); }
__device__ __forceinline__ uint32_t o_col(int k) { return (uint32_t)(k * 256 + 128); }

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
static_assert(128 * 64 + 256 * 216 <= 384 * 168, "register split exceeds the launch allocation");

// Three-input maximum (sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two float32 lanes packed in one 64-bit register: d = a * b + c, d = a + b.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

template <int D, bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const Geometry g,
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
  // Key-tile flags, written by the producer before it arms K_j's slot and
  // read by the MMA thread after that slot's load completed: bit 0/1 = query
  // tile 0/1 uses key tile j, bit 2 = no key tile j (end of the sequence).
  volatile uint32_t* tile_flags =
      reinterpret_cast<volatile uint32_t*>(base_ptr + C::kBarOff + C::kFlagsOff);
  constexpr uint32_t kFlagEnd = 4u;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: a pair of query tiles. Block order: (batch, kv head)
  // outermost, so the CTAs resident at one time read the keys/values of one
  // or two kv heads and find them in L2; then pairs by decreasing position
  // (decreasing causal work, longest first); the query heads sharing the kv
  // head innermost, so they read the same key tiles at the same time.
  const int grp = g.H_q / g.H_kv;
  const int pairs_per_seg = (g.nt + 1) / 2;
  const int n_pairs = g.n_seg * pairs_per_seg;
  const int hg = (int)(blockIdx.x % grp);
  const int rest = (int)(blockIdx.x / grp);
  const int pair = n_pairs - 1 - rest % n_pairs;
  const int bhk = rest / n_pairs;
  const int b = bhk / g.H_kv, hk = bhk % g.H_kv;
  const int h = hk * grp + hg;
  const int bh = b * g.H_q + h;
  const int seg = pair / pairs_per_seg;
  const int ti0 = (pair % pairs_per_seg) * 2;
  const int r = seg_owner(g, seg);
  // the two query tiles (scalars: runtime-indexed arrays go to local memory)
  const int q_lo0 = seg * g.seg_len + ti0 * kTile;
  const int q_lo1 = q_lo0 + kTile;
  const int q_valid0 = min(kTile, g.seg_len - ti0 * kTile);
  const int q_valid1 = ti0 + 1 < g.nt ? min(kTile, g.seg_len - (ti0 + 1) * kTile) : 0;

  // ---- set-up: barriers, abort flag, TMEM
  if (threadIdx.x == 0) {
    mbar_init(bar(C::bQFull), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(C::bFull + s), 1);
      mbar_init(bar(C::bEmpty + s), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(C::bSFull + k), 1);
      mbar_init(bar(C::bPFull + k), 128);
      mbar_init(bar(C::bODone + k), 1);
    }
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

  if (warp >= 8) {
  setmaxnreg_dec<64>();
  if (warp == kProducerWarp) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      const uint32_t q_smem = base + C::kQOff;
      mbar_arrive_expect_tx(bar(C::bQFull), 2 * C::kTileBytes);
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_4d(q_smem + bx * kBoxBytes, &tm_q, bar(C::bQFull), bx * 64, h, q_lo0, b);
        tma_load_4d(q_smem + C::kTileBytes + bx * kBoxBytes, &tm_q, bar(C::bQFull), bx * 64,
                    h, q_lo1, b);
      }
      KvIter it;
      it.init(g);
      KvTile kv;
      int n = 0;            // loads issued: K_j is load 2j, V_j is load 2j+1
      bool ok = true;
      while (ok && it.next(g, r, kv)) {
        const bool act0 = tile_work(g, q_lo0, q_valid0, kv) != kSkip;
        const bool act1 = tile_work(g, q_lo1, q_valid1, kv) != kSkip;
        if (!act0 && !act1) continue;
#pragma unroll
        for (int which = 0; which < 2; ++which) {      // 0: K, 1: V
          const int slot = n % C::kSlots;
          const uint32_t use = (uint32_t)(n / C::kSlots);
          if (n >= C::kSlots &&
              !mbar_wait(bar(C::bEmpty + slot), (use - 1) & 1, abort_flag, kTimeoutNs)) {
            ok = false;
            break;
          }
          if (which == 0) tile_flags[(n >> 1) & 15] = (act0 ? 1u : 0u) | (act1 ? 2u : 0u);
          mbar_arrive_expect_tx(bar(C::bFull + slot), C::kTileBytes);
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_4d(base + C::kSlotOff + slot * C::kTileBytes + bx * kBoxBytes,
                        which ? (const void*)&tm_v : (const void*)&tm_k, bar(C::bFull + slot),
                        bx * 64, hk, kv.lo, b);
          ++n;
        }
      }
      // Every issued load lands before the CTA leaves (already true unless
      // the CTA aborted): wait, bounded, on the last use of each slot. This
      // comes before the end marker, which completes one more phase of a slot.
      for (int nn = (n > C::kSlots ? n - C::kSlots : 0); nn < n; ++nn)
        mbar_wait(bar(C::bFull + nn % C::kSlots), (uint32_t)(nn / C::kSlots) & 1, never,
                  kTimeoutNs);
      mbar_wait(bar(C::bQFull), 0, never, kTimeoutNs);
      // End marker: K's slot of the key tile after the last one completes
      // with no load and the flag kFlagEnd.
      if (ok) {
        const int slot = n % C::kSlots;
        const uint32_t use = (uint32_t)(n / C::kSlots);
        if (n < C::kSlots ||
            mbar_wait(bar(C::bEmpty + slot), (use - 1) & 1, abort_flag, kTimeoutNs)) {
          tile_flags[(n >> 1) & 15] = kFlagEnd;
          mbar_arrive(bar(C::bFull + slot));
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ======================= MMA issuer (one thread) =======================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kTile, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, true);
      // PV groups issued per query tile (scalars, not an array: a
      // runtime-indexed array would live in local memory)
      uint32_t npv0 = 0, npv1 = 0;
      bool ok = mbar_wait(bar(C::bQFull), 0, abort_flag, kTimeoutNs);
      tc_fence_after();
      // load n of the slot ring: K_j is load 2j, V_j is load 2j+1
      auto wait_load = [&](int n) {
        ok = ok && mbar_wait(bar(C::bFull + n % C::kSlots), (uint32_t)(n / C::kSlots) & 1,
                             abort_flag, kTimeoutNs);
        tc_fence_after();
      };
      // S_k = Q_k K_j^T. P_k of the previous key tile aliases S_k, so the
      // previous PV of tile k must have completed first.
      auto issue_s = [&](int k, uint32_t npv, int j) {
        if (ok && npv > 0) {
          ok = mbar_wait(bar(C::bODone + k), (npv - 1) & 1, abort_flag, kTimeoutNs);
          tc_fence_after();
        }
        if (!ok) return;
        const uint32_t q_smem = base + C::kQOff + k * C::kTileBytes;
        const uint32_t k_smem = base + C::kSlotOff + ((2 * j) % C::kSlots) * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * kBoxBytes + (kk % 4) * 32;
          umma_ss(tmem + s_col(k), sw128_desc(q_smem + off, 16, 1024),
                  sw128_desc(k_smem + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(C::bSFull + k));
      };
      // O_k += P_k V_j once softmax k has published P_k (and rescaled O_k).
      auto issue_pv = [&](int k, uint32_t npv, int j) {
        ok = ok && mbar_wait(bar(C::bPFull + k), npv & 1, abort_flag, kTimeoutNs);
        if (!ok) return;
        tc_fence_after();
        const uint32_t v_smem = base + C::kSlotOff + ((2 * j + 1) % C::kSlots) * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts(tmem + o_col(k), tmem + s_col(k) + kk * 8,
                  sw128_desc(v_smem + kk * 2048, kBoxBytes, 1024), idesc_o,
                  (npv > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(C::bODone + k));
      };

      // Software pipeline over the active key tiles j = 0, 1, ...:
      //   prologue  S_0(0) S_1(0)
      //   round j   PV_0(j) S_0(j+1) PV_1(j) S_1(j+1)
      // S_k(j+1) follows PV_k(j) so that softmax 0 works while the tensor
      // core runs tile 1's pair of MMAs and the other way round (the two
      // softmax warpgroups stay half a round apart).
      // The key-tile sequence comes from the producer's flags (read after
      // the K load of that tile completed), so this thread does no index
      // arithmetic between the MMAs it issues.
      // Waits and slot releases sit where the tensor core still has queued
      // work: V_j is waited for before S_1 is issued (not before PV_0), and
      // the release of K_j's slot is committed after PV_0(j).
      wait_load(0);
      uint32_t f = ok ? tile_flags[0] : kFlagEnd;
      bool have = !(f & kFlagEnd);
      bool a0c = f & 1u, a1c = f & 2u;
      int j = 0;
      if (have) {
        if (a0c) issue_s(0, npv0, 0);
        wait_load(1);
        if (a1c) issue_s(1, npv1, 0);
      }
      while (have && ok) {
        if (a0c) {
          issue_pv(0, npv0, j);
          ++npv0;
        }
        if (ok) umma_commit(bar(C::bEmpty + (2 * j) % C::kSlots));         // K_j
        wait_load(2 * j + 2);
        f = ok ? tile_flags[(j + 1) & 15] : kFlagEnd;
        const bool have_n = !(f & kFlagEnd);
        const bool a0n = have_n && (f & 1u), a1n = have_n && (f & 2u);
        if (a0n) issue_s(0, npv0, j + 1);
        if (a1c) {
          issue_pv(1, npv1, j);
          ++npv1;
        }
        if (ok) umma_commit(bar(C::bEmpty + (2 * j + 1) % C::kSlots));     // V_j
        if (have_n) {
          wait_load(2 * j + 3);
          if (a1n) issue_s(1, npv1, j + 1);
        }
        a0c = a0n;
        a1c = a1n;
        have = have_n;
        ++j;
      }
      // all tensor-core work of this CTA has completed before teardown
      umma_commit(bar(C::bFinal));
      mbar_wait(bar(C::bFinal), 0, never, kTimeoutNs);
    }
    __syncwarp();
  }
  } else {
    // ======================= softmax, one thread per row =======================
    setmaxnreg_inc<216>();
    const int k = warp >> 2;                 // query tile of this warpgroup
    const int wq = warp & 3;                 // TMEM lane quarter
    const int row = wq * 32 + lane;
    const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + t_lane + s_col(k);
    const uint32_t tO = tmem + t_lane + o_col(k);
    // (selects, not indexing: a runtime index would put the arrays in local memory)
    const int my_q_lo = k ? q_lo1 : q_lo0;
    const int my_q_valid = k ? q_valid1 : q_valid0;
    const int q_pos = my_q_lo + row;
    const bool row_valid = row < my_q_valid;
    const float sl2 = g.scale_log2;
    const uint64_t sl2x2 = pack2(sl2, sl2);

    const int n_qt = g.n_seg * g.nt;
    int* log_base = (vlog && my_q_valid > 0 && (threadIdx.x & 127) == 0)
                        ? vlog + ((size_t)bh * n_qt + seg * g.nt + ti0 + k) * log_stride
                        : nullptr;
    int n_vis = 0;

    float m_run = -INFINITY, l_run = 0.f;
    uint32_t n_pv = 0;       // P tiles published (= S tiles consumed)
    bool ok = true;
    KvIter it;
    it.init(g);
    KvTile kv;
    while (it.next(g, r, kv)) {
      const int work = tile_work(g, my_q_lo, my_q_valid, kv);
      if (work == kSkip) continue;
      if (log_base) log_visit(log_base, n_vis, kv, tile_class(g, my_q_lo, kv));
      ++n_vis;
      ok = mbar_wait(bar(C::bSFull + k), n_pv & 1, abort_flag, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();

      float s[kTile];
      {
        uint32_t u0[32], u1[32], u2[32], u3[32];
        tmem_ld32(tS + 0, u0);
        tmem_ld32(tS + 32, u1);
        tmem_ld32(tS + 64, u2);
        tmem_ld32(tS + 96, u3);
        tmem_ld_wait();
        reg_fence(u0); reg_fence(u1); reg_fence(u2); reg_fence(u3);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(u0[i]);
          s[32 + i] = __uint_as_float(u1[i]);
          s[64 + i] = __uint_as_float(u2[i]);
          s[96 + i] = __uint_as_float(u3[i]);
        }
      }
      if (work == kMask) {
        const int lim = g.causal ? min(kv.valid, q_pos - kv.lo + 1) : kv.valid;
#pragma unroll
        for (int c = 0; c < kTile; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      // row max: 8 independent chains of 3-input maxima, then a tree
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = fmax3(s[i], s[8 + i], s[16 + i]);
#pragma unroll
      for (int c = 24; c < kTile - 8; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], s[c + i], s[c + 8 + i]);
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], s[kTile - 8 + i]);
      const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                             fmaxf(m8[6], m8[7]));
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
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          // (s0, s1) * scale*log2(e) - m in one packed FMA, then two exp2
          const uint64_t x2 = ffma2(pack2(s[half * 64 + 2 * i], s[half * 64 + 2 * i + 1]),
                                    sl2x2, neg_m2);
          float x0, x1;
          unpack2(x2, x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          if (i & 1) sum2b = fadd2(sum2b, pack2(p0, p1));
          else sum2a = fadd2(sum2a, pack2(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tS + half * 32, pk);
      }
      {
        float a0, a1;
        unpack2(fadd2(sum2a, sum2b), a0, a1);
        l_run += a0 + a1;
      }
      // O_k must be scaled by alpha before P_k V_j is added to it
      if (__any_sync(0xffffffffu, resc) && n_pv > 0) {
        ok = mbar_wait(bar(C::bODone + k), (n_pv - 1) & 1, abort_flag, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t u[32];
          tmem_ld32(tO + c * 32, u);
          tmem_ld_wait(u);
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
          tmem_st32(tO + c * 32, u);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::bPFull + k));
      ++n_pv;
    }
    if (log_base) log_base[0] = n_vis;

    // ---- epilogue: out = O / l, lse = ln2 * (m + log2 l)
    if (ok && n_pv > 0) {
      ok = mbar_wait(bar(C::bODone + k), (n_pv - 1) & 1, abort_flag, kTimeoutNs);
      tc_fence_after();
    }
    if (ok) {
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      const size_t row_off = (((size_t)b * g.S + q_pos) * g.H_q + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        if (n_pv > 0) {
          tmem_ld32(tO + c * 32, u);
          tmem_ld_wait(u);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = 0u;
        }
        if (row_valid) {
          if (kOutF32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + row_off + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(u[4 * i]) * inv_l,
                                   __uint_as_float(u[4 * i + 1]) * inv_l,
                                   __uint_as_float(u[4 * i + 2]) * inv_l,
                                   __uint_as_float(u[4 * i + 3]) * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + row_off + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(u[8 * i + 0]) * inv_l, __uint_as_float(u[8 * i + 1]) * inv_l);
              w.y = pack_bf16x2(__uint_as_float(u[8 * i + 2]) * inv_l, __uint_as_float(u[8 * i + 3]) * inv_l);
              w.z = pack_bf16x2(__uint_as_float(u[8 * i + 4]) * inv_l, __uint_as_float(u[8 * i + 5]) * inv_l);
              w.w = pack_bf16x2(__uint_as_float(u[8 * i + 6]) * inv_l, __uint_as_float(u[8 * i + 7]) * inv_l);
              dst[i] = w;
            }
          }
        }
      }
      if (row_valid && lse)
        lse[(size_t)bh * g.S + q_pos] =
            l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
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

template <int D, bool kOutF32>
ra_status launch_typed(const Geometry& g, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, void* out, float* lse, int* vlog,
                       int log_stride, int* status, cudaStream_t stream) {
  using C = Cfg<D>;
  auto kern = attn_tc_kernel<D, kOutF32>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes) != cudaSuccess)
    return RA_ERR_LAUNCH;
  const long long pairs = (long long)g.n_seg * ((g.nt + 1) / 2);
  const long long grid = pairs * g.B * g.H_q;
  if (grid > 0x7fffffffLL) return RA_ERR_RANGE;
  kern<<<(unsigned)grid, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, g, out, lse, vlog,
                                                            log_stride, status);
  return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_LAUNCH;
}

}  // namespace

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
