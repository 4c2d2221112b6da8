/*
 * ring_attn.h - C ABI of the GB300 (sm_103a) exact ring-attention library.
 *
 * What it computes. Glossary "sequence parallelism transformers":
 *  - §Sequence Parallelism Fundamentals ("Sequence Dimension Splitting"): the
 *    length-S sequence is cut into P chunks, one per rank. Here the ranks are
 *    virtual: all P live on the one GPU running the call.
 *  - §Ring Attention: each rank keeps its query block; at step t it attends
 *    to the key/value block that started on rank (r - t) mod P (blocks move
 *    from rank i to i+1 each step) and accumulates the outputs; after P
 *    steps the result equals full softmax attention.
 *  - §Implementation Considerations ("Numerical Stability", "Load
 *    Balancing"): partial results are combined with an exact log-sum-exp
 *    merge; the zig-zag chunk order (2P halves, rank r owns halves r and
 *    2P-1-r) balances causal work across ranks.
 * Uneven lengths follow the mvp-engine "sequence-parallel" skill (seq_len
 * divisible by the split, else pad explicitly and mask): the sequence counts
 * as padded to the next multiple of P (contiguous) or 2P (zig-zag), every
 * chunk (half) spans L = ceil(S/P) (ceil(S/2P)) positions starting at a
 * multiple of L, and the padding positions (S and beyond) hold no token:
 * they are never read, never written and never attended to. A trailing
 * chunk can therefore be short or empty. The padding is virtual; tensors
 * keep exactly S rows.
 *
 * For each batch b, query head h and query position i, with key/value head
 * hk = h / (H_q / H_kv) and allowed keys A(i) = {0..S-1} (non-causal) or
 * {0..i} (causal, global positions):
 *     lse[b,h,i] = log sum_{j in A(i)} exp(scale * <q_i, k_j>)      (natural log)
 *     out[b,i,h] = sum_{j in A(i)} exp(scale * <q_i, k_j> - lse) * v_j
 *
 * Layouts (all row-major, contiguous, "BSHD": sequence is dimension 1):
 *     q, out      [B, S, H_q,  D]
 *     k, v        [B, S, H_kv, D]
 *     lse         [B, H_q, S]            float32
 * Element types: RA_BF16 (bfloat16 in and out, float32 accumulation) or
 * RA_F32 (float32 throughout).
 *
 * Conventions shared by every entry point:
 *  - Every data pointer is a DEVICE pointer on the current CUDA device, owned
 *    by the caller. Tensor pointers (q, k, v, out, o_*) are 16-byte aligned;
 *    lse, visit logs and status words 4-byte aligned (else RA_ERR_ALIGN).
 *    The library allocates no device memory and keeps no state between calls
 *    except read-only per-device facts and the one scratch array that
 *    ring_attn_bwd_noalloc uses (module memory, held until exit).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Calls enqueue work and return; they never synchronise.
 *  - Arguments are checked on the host before anything is enqueued; on error
 *    nothing is launched and the status says why. A failed launch returns
 *    RA_ERR_LAUNCH. A device-side bounded wait that expired is reported in
 *    `dev_status` (where the call takes one) as RA_ERR_TIMEOUT, after the
 *    stream has run the kernel.
 *  - Two builds export this same ABI: libringattn.so and the bounds-checked
 *    libringattn_debug.so. In the checked build every global-memory access
 *    a kernel computes from indices is tested against its tensor's extent.
 *    A violation skips the access and sets RA_ERR_RANGE in `dev_status`;
 *    there is no trap. In the release build the checks compile away.
 *  - `scale <= 0` means 1/sqrt(D).
 *  - Tensors stay in natural token order in every chunk order: the order only
 *    decides which virtual rank owns which tokens and the sequence of steps.
 */
#ifndef RING_ATTN_H
#define RING_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_NULL = 1,     /* a required pointer is NULL                              */
  RA_ERR_SHAPE = 2,    /* a size <= 0, H_q % H_kv != 0, merge n out of range       */
  RA_ERR_HEADDIM = 3,  /* D is not 64 or 128 (attention), not 32-256 (merge)     */
  RA_ERR_ALIGN = 4,    /* a data pointer is not 16-byte aligned                    */
  RA_ERR_DTYPE = 5,    /* unknown dtype or order value                             */
  RA_ERR_DEVICE = 6,   /* current device is not compute capability 10.3            */
  RA_ERR_LAUNCH = 7,   /* CUDA runtime error while preparing or launching          */
  RA_ERR_TIMEOUT = 8,  /* a device-side bounded wait expired (dev_status only)     */
  RA_ERR_BUFFER = 9,   /* a caller buffer is too small                             */
  RA_ERR_RANGE = 10,   /* a size overflows 32-bit indexing, or step out of range;
                          in dev_status (checked build only): a device index out
                          of its tensor's range                                   */
  RA_ERR_SCRATCH = 11  /* the problem needs more scratch than the library's
                          built-in array holds (ring_attn_bwd_noalloc)           */
} ra_status;

typedef enum { RA_BF16 = 0, RA_F32 = 1 } ra_dtype;
typedef enum { RA_ORDER_CONTIGUOUS = 0, RA_ORDER_ZIGZAG = 1 } ra_order;

/* Classes of a (query set, key set) pair under the causal rule j <= i. */
enum { RA_CLASS_SKIP = 0, RA_CLASS_FULL = 1, RA_CLASS_PARTIAL = 2 };

/* Largest n accepted by attn_lse_merge_n. */
#define RA_MERGE_MAX_N 16

/*
 * ring_attn_fwd - exact attention computed as a ring of P virtual ranks,
 * bfloat16 inputs and output, contiguous chunk order. Defined by glossary
 * "sequence parallelism transformers", §Ring Attention ("Block-Wise
 * Attention", "Ring Communication", "Computation": each rank keeps its query
 * block, attends to every key/value block as it passes, and accumulates
 * exactly the full-attention result).
 *
 * All P ring steps run inside one kernel launch: every query tile keeps its
 * running (max, sum, unnormalised output) on chip across steps, which is the
 * log-sum-exp merge of the per-step partials done in registers. Under a
 * causal mask, key tiles that lie entirely after the query tile are skipped.
 * `lse` may be NULL (not written). Errors: RA_ERR_NULL (q, k, v or out NULL),
 * RA_ERR_SHAPE, RA_ERR_HEADDIM, RA_ERR_ALIGN, RA_ERR_RANGE (B*S*H*D beyond
 * 2^31 elements per tensor), RA_ERR_DEVICE, RA_ERR_LAUNCH.
 */
ra_status ring_attn_fwd(const void* q, const void* k, const void* v,
                        void* out, float* lse,
                        int B, int H_q, int H_kv, int S, int D, int P,
                        int causal, float scale, void* stream);

/*
 * ring_attn_fwd_ex - ring_attn_fwd with every option. Defined by the same
 * glossary, §Ring Attention (the per-step partial results of `step`), and
 * §Implementation Considerations ("Load Balancing": the zig-zag `order`).
 *
 * dtype   RA_BF16 (tensor-core path) or RA_F32 (exact float32 CUDA-core path).
 * order   RA_ORDER_CONTIGUOUS (rank r owns [rS/P, (r+1)S/P)) or
 *         RA_ORDER_ZIGZAG (rank r owns halves r and 2P-1-r of length S/2P).
 * step    -1: all P steps, folded on chip (same result as ring_attn_fwd).
 *         t in [0, P): ring step t only. Every rank r attends to the chunk of
 *         rank (r - t) mod P and the call writes that step's PARTIAL result:
 *         `out` is then float32 [B, S, H_q, D] whatever `dtype` is, and `lse`
 *         (required) is the partial lse; rows with no allowed key in that
 *         chunk get out = 0 and lse = -inf. Folding the P partials with
 *         attn_lse_merge / attn_lse_merge_n gives the full result.
 * visit_log  NULL, or a device int32 buffer of ring_attn_visit_log_len(...)
 *         elements: for every (b, h, query tile) the key tiles the kernel
 *         visited, in visit order (layout at ring_attn_visit_log_len).
 * dev_status NULL, or a device int the kernel sets to RA_ERR_TIMEOUT if one of
 *         its bounded waits expired (it is never cleared by the library; the
 *         caller zeroes it).
 */
ra_status ring_attn_fwd_ex(const void* q, const void* k, const void* v,
                           void* out, float* lse,
                           int B, int H_q, int H_kv, int S, int D, int P,
                           int causal, float scale,
                           int dtype, int order, int step,
                           int* visit_log, int* dev_status, void* stream);

/*
 * ring_attn_fwd_varlen - ring attention over a batch of packed sequences of
 * different lengths.
 *
 * Sequence b occupies rows [cu_seqlens[b], cu_seqlens[b+1]) of the packed
 * tensors and is its own ring problem: its S_b tokens are cut into P chunks
 * (or 2P halves) of ceil(S_b / P) (ceil(S_b / 2P)) positions, padded like an
 * uneven S (see above), and its queries attend only to its own keys. Layouts:
 *     q, out   [total, H_q,  D]      k, v   [total, H_kv, D]
 *     lse      [H_q, total]          float32 (may be NULL)
 * cu_seqlens: DEVICE int32 array of n_seq + 1 nondecreasing offsets with
 * cu_seqlens[0] = 0 and cu_seqlens[n_seq] = total. max_seqlen >= every S_b
 * (it sizes the launch). The kernels clamp offsets into [0, total] and
 * lengths into [0, max_seqlen], so a malformed array never moves an access
 * outside the tensors (its sequences are then simply wrong). A sequence of
 * length 0 writes nothing. dtype RA_BF16 or RA_F32; all steps; no visit log.
 * Errors: RA_ERR_NULL, RA_ERR_SHAPE (n_seq, total or max_seqlen <= 0,
 * H_q % H_kv), RA_ERR_HEADDIM, RA_ERR_ALIGN (cu_seqlens 4-byte), RA_ERR_DTYPE,
 * RA_ERR_RANGE, RA_ERR_DEVICE, RA_ERR_LAUNCH.
 */
ra_status ring_attn_fwd_varlen(const void* q, const void* k, const void* v,
                               void* out, float* lse, const int* cu_seqlens,
                               int n_seq, int total, int max_seqlen,
                               int H_q, int H_kv, int D, int P, int causal,
                               float scale, int dtype, int order,
                               int* dev_status, void* stream);

/*
 * ring_attn_fwd_ulysses - exact attention in the sequence-parallel layout of
 * Ulysses-style sequence parallelism (glossary "sequence parallelism
 * transformers", §Ulysses Sequence Parallelism: an all-to-all turns the
 * sequence-parallel layout into a head-parallel one, each rank computes full
 * attention for its subset of heads, and a second all-to-all restores the
 * sequence-parallel layout).
 *
 * Virtual rank p holds the contiguous shard of C = ceil(S/P) positions
 * [p*C, min((p+1)*C, S)) of every batch and head, and the tensors are the P
 * ranks' local tensors stacked:
 *     q, out  [P, B, C, H_q,  D]      k, v  [P, B, C, H_kv, D]
 *     lse     [P, B, H_q, C]          float32 (may be NULL)
 * (rows of a last, partly filled shard past S are neither read nor written).
 * Rank r's head-parallel work is heads [r*H_q/P, (r+1)*H_q/P) (and the kv
 * heads they read) over all S positions. On one GPU both all-to-alls are an
 * index map inside the kernel's loads and stores: nothing is copied. The
 * result is full attention, as for every other entry point. H_q and H_kv
 * must be multiples of P (else RA_ERR_SHAPE). dtype RA_BF16 or RA_F32; all
 * steps; no visit log. Errors as ring_attn_fwd_ex.
 */
ra_status ring_attn_fwd_ulysses(const void* q, const void* k, const void* v,
                                void* out, float* lse,
                                int B, int H_q, int H_kv, int S, int D, int P,
                                int causal, float scale, int dtype,
                                int* dev_status, void* stream);

/*
 * ring_attn_visit_log_len - size of the visit log of ring_attn_fwd_ex.
 *
 * The kernel for `dtype` cuts every chunk (contiguous) or half (zig-zag) of
 * length L into query and key tiles of `*tile_rows` rows (the last one shorter
 * when L is not a multiple). Tiles are numbered globally: the segment's index
 * in position order times `*tiles_per_segment` plus the tile's index in it.
 * The log holds, for each (b, h, query tile id), `*stride` ints: the number
 * of visits n, then n entries of 4 ints (step, source rank, key tile id,
 * class). Total length = B * H_q * n_query_tiles * stride, returned in *len.
 * Host-only; never touches the GPU.
 */
ra_status ring_attn_visit_log_len(int B, int H_q, int S, int D, int P,
                                  int dtype, int order,
                                  int* tile_rows, int* tiles_per_segment,
                                  int* n_query_tiles, int* stride,
                                  long long* len);

/*
 * ring_attn_bwd_workspace - bytes of device workspace ring_attn_bwd needs
 * for this shape (written to *bytes). Host only; never touches the GPU.
 * The workspace holds two float32 statistics per query row of the forward
 * result, negated (-lse in base 2 and -delta_i, delta_i = <dout_i, out_i>),
 * stored per (b, h, query tile) with every tile padded to the kernels' tile
 * height; its contents are the library's own and only its phases read them.
 * Errors: RA_ERR_NULL (bytes NULL), RA_ERR_SHAPE, RA_ERR_HEADDIM,
 * RA_ERR_DTYPE (order), RA_ERR_RANGE.
 */
ra_status ring_attn_bwd_workspace(int B, int H_q, int S, int D, int P,
                                  int order, size_t* bytes);

/*
 * ring_attn_bwd - gradients of ring attention with respect to q, k and v,
 * bfloat16 (glossary "sequence parallelism transformers", §Implementation
 * Considerations: the backward pass runs over the same ring as the forward).
 *
 * For an upstream gradient dout = dL/d(out), with p_ij = exp(s_ij - lse_i)
 * on the allowed pairs of the forward definition above:
 *     dV_j = sum_i p_ij dout_i
 *     ds_ij = p_ij (<dout_i, v_j> - delta_i),   delta_i = <dout_i, out_i>
 *     dQ_i = scale * sum_j ds_ij k_j,   dK_j = scale * sum_i ds_ij q_i
 * A key/value head's dk and dv sum over the query heads of its group.
 * Ring structure: the dq of a query tile is accumulated on chip over the key
 * tiles in the forward's ring order; the dk, dv of a key tile over the query
 * tiles of ranks src, src+1, ..., src+P-1 (mod P) in step order, which is
 * the order in which the block, travelling the ring, meets them on its way
 * back to its owner. All P steps run; there is no single-step mode.
 *
 * q [B,S,H_q,D], k and v [B,S,H_kv,D], out and dout [B,S,H_q,D]: bfloat16
 *   device tensors; out and lse are the forward's results for the same
 *   arguments (lse float32 [B,H_q,S], natural log, as ring_attn_fwd_ex
 *   writes it).
 * dq [B,S,H_q,D], dk and dv [B,S,H_kv,D]: bfloat16, overwritten (not
 *   accumulated into). They must not overlap any input.
 * dtype RA_BF16 only (RA_ERR_DTYPE otherwise); order as in ring_attn_fwd_ex.
 * workspace / workspace_bytes: a device buffer of at least
 *   ring_attn_bwd_workspace(...) bytes (else RA_ERR_BUFFER), 16-byte aligned,
 *   owned by the caller; its contents on entry are ignored and on return
 *   undefined. The call allocates no memory of its own.
 * dev_status as in ring_attn_fwd_ex.
 * Errors: as ring_attn_fwd_ex, plus RA_ERR_BUFFER.
 */
ra_status ring_attn_bwd(const void* q, const void* k, const void* v,
                        const void* out, const float* lse, const void* dout,
                        void* dq, void* dk, void* dv,
                        int B, int H_q, int H_kv, int S, int D, int P,
                        int causal, float scale, int dtype, int order,
                        void* workspace, size_t workspace_bytes,
                        int* dev_status, void* stream);

/* Size of the scratch array built into the library for ring_attn_bwd_noalloc. */
#define RA_BWD_NOALLOC_MAX_BYTES (8u << 20)

/*
 * ring_attn_bwd_noalloc - ring_attn_bwd without a caller workspace; the call
 * allocates no memory at all. The pages have no counterpart to this entry
 * point: it exists for callers that cannot call cudaMalloc, such as a plugin
 * whose host framework owns the device memory through its own pool and hands
 * it no workspace, or a latency-critical path on which cudaMalloc / cudaFree
 * may synchronise the device.
 *
 * Arguments and results are those of ring_attn_bwd without `workspace` and
 * `workspace_bytes`: the caller still passes every input and output. The
 * workspace lives instead in a file-scope device array of
 * RA_BWD_NOALLOC_MAX_BYTES (8 MiB) that every GPU which loads the library
 * holds until the process exits. It fits ring_attn_bwd_workspace(...) <=
 * 8 MiB, i.e. up to 2^20 tile-padded query rows (B * H_q * S rounded up per
 * 128-row tile of each chunk or half); the S = 32768, H_q = 32 causal
 * zig-zag problem fits exactly. A larger problem returns RA_ERR_SCRATCH
 * before anything is launched.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture begins.
 *  - Every call shares the one array and it keeps the last call's contents.
 *    Nothing in it has to start at zero: the prep phase overwrites every
 *    entry a call reads. Calls whose work overlaps on the GPU (two streams,
 *    or two host threads on one device) race on the array: serialise them.
 *  - dev_status and every other convention as ring_attn_bwd.
 * Errors: as ring_attn_bwd, with RA_ERR_SCRATCH in place of RA_ERR_BUFFER.
 */
ra_status ring_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                const void* out, const float* lse, const void* dout,
                                void* dq, void* dk, void* dv,
                                int B, int H_q, int H_kv, int S, int D, int P,
                                int causal, float scale, int dtype, int order,
                                int* dev_status, void* stream);

/* Phases of the backward pass (bit flags) for ring_attn_bwd_ex. */
enum { RA_BWD_PREP = 1, RA_BWD_DKDV = 2, RA_BWD_DQ = 4, RA_BWD_ALL = 7 };

/*
 * ring_attn_bwd_ex - ring_attn_bwd restricted to the phases in `phases` (a
 * nonzero OR of RA_BWD_*, else RA_ERR_RANGE), enqueued in the order prep,
 * dK/dV, dQ; one kernel launch per phase. The prep phase writes the
 * workspace (-lse in base 2 and -delta per query row); the dK/dV phase
 * (writes dk, dv) and the dQ phase (writes dq) read it and are independent
 * of each other, so after the prep phase they may run on two streams at
 * once. A phase needs the prep phase of the same arguments to have run
 * before it on the device. ring_attn_bwd is phases = RA_BWD_ALL.
 */
ra_status ring_attn_bwd_ex(const void* q, const void* k, const void* v,
                           const void* out, const float* lse, const void* dout,
                           void* dq, void* dk, void* dv,
                           int B, int H_q, int H_kv, int S, int D, int P,
                           int causal, float scale, int dtype, int order,
                           void* workspace, size_t workspace_bytes, int phases,
                           int* dev_status, void* stream);

/*
 * ring_attn_bwd_varlen - ring_attn_bwd for packed sequences, with the
 * layouts and cu_seqlens / max_seqlen conventions of ring_attn_fwd_varlen
 * (dout, dq like q; dk, dv like k; lse [H_q, total]). The workspace size is
 * ring_attn_bwd_workspace(n_seq, H_q, max_seqlen, D, P, order, ...).
 * bf16 only. Errors: as ring_attn_fwd_varlen, plus RA_ERR_BUFFER.
 */
ra_status ring_attn_bwd_varlen(const void* q, const void* k, const void* v,
                               const void* out, const float* lse, const void* dout,
                               void* dq, void* dk, void* dv, const int* cu_seqlens,
                               int n_seq, int total, int max_seqlen,
                               int H_q, int H_kv, int D, int P, int causal,
                               float scale, int dtype, int order,
                               void* workspace, size_t workspace_bytes,
                               int* dev_status, void* stream);

/*
 * ring_attn_bwd_ulysses - ring_attn_bwd for tensors in the sequence-parallel
 * layout of ring_attn_fwd_ulysses (q, out, dout, dq [P, B, C, H_q, D]; k, v,
 * dk, dv [P, B, C, H_kv, D]; lse [P, B, H_q, C]; C = ceil(S/P)). The
 * all-to-alls are again index maps in the loads and stores. H_q and H_kv must
 * be multiples of P. The workspace size is ring_attn_bwd_workspace(B, H_q, S,
 * D, P, RA_ORDER_CONTIGUOUS, ...). bf16 only. Errors: as ring_attn_bwd.
 */
ra_status ring_attn_bwd_ulysses(const void* q, const void* k, const void* v,
                                const void* out, const float* lse, const void* dout,
                                void* dq, void* dk, void* dv,
                                int B, int H_q, int H_kv, int S, int D, int P,
                                int causal, float scale, int dtype,
                                void* workspace, size_t workspace_bytes,
                                int* dev_status, void* stream);

/*
 * attn_lse_merge - exact merge of two partial attention results over
 * disjoint key sets (glossary "sequence parallelism transformers",
 * §Ring Attention and §Implementation Considerations):
 *     lse = log(exp(lse_a) + exp(lse_b))
 *     out = exp(lse_a - lse) * o_a + exp(lse_b - lse) * o_b
 * evaluated with the larger lse factored out. A side with lse = -inf
 * contributes nothing; both -inf gives out = 0, lse = -inf.
 * o_a, o_b, out: [B, S, H, D] of `dtype`; lse_a, lse_b, lse: float32
 * [B, H, S]. `out` may alias o_a or o_b and `lse` may alias lse_a or lse_b
 * (each element is read before it is written, by the same thread).
 */
ra_status attn_lse_merge(const void* o_a, const float* lse_a,
                         const void* o_b, const float* lse_b,
                         void* out, float* lse,
                         int B, int H, int S, int D, int dtype, void* stream);

/*
 * attn_lse_merge_n - the same merge over n partials in one pass
 * (1 <= n <= RA_MERGE_MAX_N):
 *     lse = M + log sum_t exp(lse_t - M),  M = max_t lse_t
 *     out = sum_t exp(lse_t - lse) * o_t
 * `o` and `lse` are HOST arrays of n device pointers. Aliasing as for
 * attn_lse_merge. D is 32, 64, 128 or 256 here.
 */
ra_status attn_lse_merge_n(const void* const* o, const float* const* lse,
                           int n, void* out, float* out_lse,
                           int B, int H, int S, int D, int dtype, void* stream);

/*
 * ring_attn_plan - the ring schedule as an int32 table, host only. Defined
 * by glossary "sequence parallelism transformers", §Sequence Parallelism
 * Fundamentals (P chunks of S/P tokens) and §Ring Attention ("Ring
 * Communication": at step t rank r holds the block of rank (r - t) mod P).
 * One row of RA_PLAN_COLS ints per (rank, step), rank-major then step:
 *   rank, step, src = (rank - step) mod P, class of the whole (query chunk,
 *   key chunk) pair, segment length L (padded, see above), first and second
 *   query segment starts,
 *   first and second key segment starts (-1 where a rank owns one segment).
 * `table_len` is the capacity in ints (>= P*P*RA_PLAN_COLS, else
 * RA_ERR_BUFFER). Never touches the GPU.
 */
#define RA_PLAN_COLS 9
ra_status ring_attn_plan(int S, int P, int causal, int order,
                         int* table, size_t table_len);

/*
 * ring_attn_expiry_test - exercises the failure path of the tensor-core
 * kernel's bounded waits; for tests, never needed in normal use.
 * Runs the bf16 kernel on B = H_q = H_kv = 1, D = 128, P = 1, non-causal,
 * 1 <= S <= 4096 (q, k, v, out [1, S, 1, 128] bf16; lse [1, 1, S]) with the
 * load of the first value tile withheld, so the wait for it expires after
 * about two seconds. The kernel then gives up in every role, waits (bounded)
 * for the copies and tensor-core work it issued, frees its tensor memory,
 * returns, and sets *dev_status (device int, required) to RA_ERR_TIMEOUT.
 * `out` and `lse` are left partly unwritten. The CUDA context stays usable.
 * Returns RA_OK when the kernel was launched (the expiry shows in dev_status
 * after the stream has run it), else an argument or launch error.
 */
ra_status ring_attn_expiry_test(const void* q, const void* k, const void* v,
                                void* out, float* lse, int S, int* dev_status,
                                void* stream);

/* Human-readable text of a status; never NULL. */
const char* ring_attn_strerror(int status);

/* Library ABI version (major * 100 + minor); 103 adds the backward, the
 * packed variable-length and the Ulysses-layout entry points. */
int ring_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RING_ATTN_H */
