/*
 * moda.h -- C ABI of the Mixture-of-Depths Attention (MoDA) forward for
 * NVIDIA GB300 (sm_103a).
 *
 * MoDA (arXiv 2603.15619, Sec. 2.2 "Mixture-of-Depths Attention", Fig. 1):
 * every grouped-query attention head at token t attends, under ONE softmax,
 * to the causal sequence keys/values of its own layer (positions <= t) and to
 * the L depth key/value slots that earlier layers (attention layers and the
 * FFN-input KV projections) wrote for the SAME position t.
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE memory owned by the caller, dense,
 *     row-major, bf16 unless stated, 16-byte aligned. The library never
 *     allocates memory per call and never frees caller memory.
 *   - Calls enqueue work on `stream` (0 = the legacy default stream) and
 *     return after the launch; results are ready when the stream is.
 *   - Argument errors are reported synchronously by the return value and
 *     nothing is launched. A failure inside a running kernel (a bounded wait
 *     that gave up) is latched in a per-device error word and reported by
 *     moda_get_device_error().
 *   - Batch is 1; callers loop over sequences.
 *   - Thread safety: calls may be made from several host threads.
 *   - moda_fwd, moda_fwd_layer_major and moda_fwd_depth_cc hand out their
 *     tiles through a small per-device queue; each call takes the next of 64 queues
 *     in turn and leaves it zeroed when it completes. Up to 64 such calls may
 *     run on one device at the same time (on different streams); more are not
 *     supported. Calls may be captured in a CUDA graph: a captured call keeps
 *     the queue it took at capture for every replay, so replays of one graph
 *     must not overlap one another.
 */
#ifndef MODA_H_
#define MODA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MODA_API __attribute__((visibility("default")))
#else
#define MODA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moda_stream_t; /* identical to cudaStream_t */

typedef enum {
  MODA_OK = 0,
  MODA_ERR_INVALID_ARG = 1, /* NULL pointer, T < 1, L < 0, Hq % Hk != 0, aliasing */
  MODA_ERR_UNSUPPORTED = 2, /* d not in {64, 128}; G = Hq/Hk not in {1,2,4,8,16}; sizes too large */
  MODA_ERR_MISALIGNED = 3,  /* a tensor pointer not 16-byte aligned */
  MODA_ERR_CUDA = 4,        /* the CUDA runtime reported an error at launch */
  MODA_ERR_TIMEOUT = 5,     /* a kernel's bounded wait gave up (device-side) */
  MODA_ERR_NO_DEVICE = 6    /* no CUDA device of compute capability 10.3 is current */
} moda_status;

/*
 * moda_pack_depth -- relayout the depth stream into the flash-compatible,
 * chunk-aware order (Sec. 3.2 "Flash-compatible depth KV layout" and
 * "Chunk-aware depth KV layout", Fig. 4): the L slots of each position become
 * contiguous, so a query tile covering positions [t0, t1) of KV head hk reads
 * one contiguous block dst[hk][t0..t1)[0..L)[:].
 *
 *   dst[hk][t][l][c] = src[l][t][hk][c]      (bit-exact copy)
 *
 *   src  [L, T, Hk, d] bf16 -- slot l is what the l-th earlier layer appended;
 *        device memory, or page-locked host memory mapped into the device
 *        address space (cudaHostAlloc / cudaHostRegister): the kernel then
 *        reads it over the host link, so the host-to-device transfer and the
 *        relayout are one pass
 *   dst  [Hk, T, L, d] bf16 device memory -- must not overlap src
 *   d    64 or 128
 * Call once for the depth keys and once for the depth values. L == 0 is a
 * no-op (src and dst may then be NULL).
 * Errors: INVALID_ARG (NULL with L > 0, T < 1, Hk < 1, L < 0, src == dst,
 * pageable host memory or an address the device cannot reach), UNSUPPORTED (d),
 * MISALIGNED, CUDA.
 */
MODA_API moda_status moda_pack_depth(const void* src, void* dst, int L, int T, int Hk,
                            int d, moda_stream_t stream);

/*
 * moda_depth_write -- write one layer's keys (or values) into slot `slot` of
 * the packed depth stream as the layer runs (Sec. 2.2, "write": attention
 * layers append their K, V; FFN layers the KV projection of their input):
 *
 *   dst[hk][t][slot][c] = src[t][hk][c]      (bit-exact copy)
 *
 *   src  [T, Hk, d] bf16, one layer's K or V
 *   dst  [Hk, T, L, d] bf16, the packed stream moda_fwd reads; only slot
 *        `slot` is written, 0 <= slot < L
 * Writing every layer this way makes moda_pack_depth unnecessary.
 * Bounded depth cache, sliding window (Sec. 6.2's fixed budget S << L): give
 * the stream L = S slots and write layer l into slot l % S; moda_fwd with
 * L = min(layers written, S) then attends to the most recent S slots (slot
 * order does not matter to the joint softmax).
 * Errors: INVALID_ARG, UNSUPPORTED (d, L > 1024), MISALIGNED, CUDA.
 */
MODA_API moda_status moda_depth_write(const void* src, void* dst, int T, int Hk, int d, int L,
                                      int slot, moda_stream_t stream);

/*
 * Bounded depth KV cache (summary, Sec. 6.2 "bounded depth KV slot cache"):
 * the packed streams hold a fixed budget of S slots (S much smaller than the
 * number of depth entries a deep model writes), and a policy decides which
 * entries stay. The pages name three policies without defining them further:
 * keep the top S entries by utility, keep a sliding window of the most recent
 * entries, or a hybrid that reserves part of the slots for recent entries and
 * gives the rest to high-scoring ones. Readings taken here:
 *   - an entry is one layer's depth K/V (one slot index for all heads and
 *     positions); its age is its write order;
 *   - its utility is the depth probability mass it received in the latest
 *     read of the cache (moda_depth_mass, summed over KV heads); a new entry
 *     has not been read, so it is always admitted and a cached one leaves;
 *   - `recent` = R slots are reserved for the R most recent entries, the new
 *     one included (R >= S: sliding window; R <= 1: top-S by utility); of
 *     the other entries the one with the least utility leaves (equal
 *     utilities: the older, then the lower slot).
 * A layer loop runs entirely on the stream, with no host round trip:
 *   moda_fwd(q, k, v, kd, vd, ..., L = slots filled, o, lse)
 *   moda_depth_mass(q, kd, lse, ..., mass)         (when all S are filled)
 *   moda_depth_cache_admit(slot_age, mass, Hk, S, R, layer, slot)
 *   moda_depth_write_at(k_layer, kd, ..., slot); moda_depth_write_at(v_layer, vd, ..., slot)
 * Slots fill in order 0, 1, ... while any is empty, so the first L filled
 * slots are always slots 0..L-1.
 */

/*
 * moda_depth_mass -- how much the queries of one layer read each depth slot:
 *   mass[hk][l] = sum over t < T and the G heads h of group hk of
 *                 exp(scale * q[t,h,:].kd[hk,t,l,:] - lse[t,h])
 * i.e. the probability the joint softmax of moda_fwd gives slot l, summed
 * over the rows of KV head hk.
 *   q, kd, scale  as passed to moda_fwd (kd packed [Hk, T, L, d])
 *   lse           [T, Hq] fp32, the lse moda_fwd returned for them
 *   mass          [Hk, L] fp32 output
 *   workspace     caller-owned device scratch of at least
 *                 moda_depth_mass_workspace_bytes(T, Hk, L) bytes
 * Deterministic: per-block partial sums are added in a fixed order.
 * Supported: as moda_fwd, with 1 <= L. Errors: INVALID_ARG, UNSUPPORTED,
 * MISALIGNED, CUDA.
 */
MODA_API size_t moda_depth_mass_workspace_bytes(int T, int Hk, int L);
MODA_API moda_status moda_depth_mass(const void* q, const void* kd, const float* lse, int T,
                                     int Hq, int Hk, int d, int L, float scale, float* mass,
                                     float* workspace, size_t workspace_bytes,
                                     moda_stream_t stream);

/*
 * moda_depth_cache_admit -- chooses the slot that the entry of age `new_age`
 * goes into, by the policy above, and records it: slot_age[*slot] = new_age.
 *   slot_age  [S] int32 device memory, the age of the entry in each slot, -1
 *             for an empty slot (initialise to -1); updated in place
 *   mass      [Hk, S] fp32 device memory from moda_depth_mass over the S
 *             slots; read only when no slot is empty. Utility of slot s:
 *             the fp32 sum of mass[0][s], mass[1][s], ... in head order;
 *             NaN orders as the largest
 *   recent    R >= 0; new_age >= 0, larger than every age in the cache
 *   slot      one int32 of device memory, receives the chosen slot
 * One small kernel; the result is ready when the stream is. S <= 1024.
 * Errors: INVALID_ARG, UNSUPPORTED (S), MISALIGNED, CUDA.
 */
MODA_API moda_status moda_depth_cache_admit(int* slot_age, const float* mass, int Hk, int S,
                                            int recent, int new_age, int* slot,
                                            moda_stream_t stream);

/*
 * moda_depth_write_at -- moda_depth_write with the slot index read from
 * device memory when the kernel runs (as moda_depth_cache_admit leaves it),
 * so the write needs no host round trip. A slot outside [0, L) writes
 * nothing and latches MODA_ERR_INVALID_ARG in the device error word
 * (moda_get_device_error). Other arguments and errors as moda_depth_write.
 */
MODA_API moda_status moda_depth_write_at(const void* src, void* dst, int T, int Hk, int d,
                                         int L, const int* slot, moda_stream_t stream);

/*
 * moda_kv_proj_write -- an FFN layer's depth keys and values, projected from
 * the FFN's input and written straight into slot `slot` of the packed depth
 * streams (reading notes Sec. 二.3: the FFN branch adds a KV projection of its
 * INPUT X; summary Sec. 2.2, "write" step: FFN layers get their pair from a
 * light KV projection; MoDA keeps only the grouped depth K/V projections):
 *
 *   kd[hk][t][slot][j] = bf16( sum_c x[t][c] * wk[hk*d + j][c] )
 *   vd[hk][t][slot][j] = bf16( sum_c x[t][c] * wv[hk*d + j][c] )
 *
 *   x       [T, Dm] bf16, the FFN's input rows
 *   wk, wv  [Hk*d, Dm] bf16, one row per output feature (the layout of a
 *           linear layer's weight); feature hk*d + j is element j of KV head hk
 *   kd, vd  [Hk, T, L, d] bf16, the packed streams moda_fwd reads; only slot
 *           `slot` (0 <= slot < L) is written, every other slot is left as is
 * Arithmetic: bf16 products, fp32 accumulation over Dm, one rounding to bf16
 * (nearest even). No bias: the pages name a projection and no more.
 * Outputs must not overlap the inputs or each other. Supported: d in {64, 128},
 * Dm a multiple of 64, 1 <= T <= 2^24, 1 <= L <= 1024.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, CUDA (synchronous); TIMEOUT
 * via moda_get_device_error.
 */
MODA_API moda_status moda_kv_proj_write(const void* x, const void* wk, const void* wv, int T,
                                        int Dm, int Hk, int d, int L, int slot, void* kd,
                                        void* vd, moda_stream_t stream);

/*
 * moda_fwd -- the MoDA forward (Sec. 2.2 joint softmax; Sec. 3.3 fused
 * kernel: group-aware query tiles, grouped causal mask, block-diagonal depth
 * mask, one online-softmax state).
 *
 * For every position t < T and query head h < Hq, with G = Hq / Hk and
 * hk = floor(h / G) (contiguous groups of G query heads share KV head hk,
 * Sec. 2.1 Eq. (2) phi(h) read 0-based):
 *   z = [ scale * q[t,h,:].k[j,hk,:]   for j = 0..t          (causal, self included)
 *       | scale * q[t,h,:].kd[hk,t,l,:] for l = 0..L-1 ]      (depth slots of position t)
 *   o[t,h,:] = sum softmax(z) * [ v[j,hk,:] | vd[hk,t,l,:] ]   (one shared denominator)
 *   lse[t,h] = ln(sum exp(z))   (natural log, scaled-score domain)
 *
 *   q       [T, Hq, d] bf16
 *   k, v    [T, Hk, d] bf16
 *   kd, vd  [Hk, T, L, d] bf16, the PACKED depth stream (moda_pack_depth);
 *           may be NULL when L == 0, which makes the call plain causal GQA
 *   scale   the logit scale, > 0 and finite, usually 1/sqrt(d); used for
 *           sequence and depth logits alike
 *   o       [T, Hq, d] bf16 output, rounded to nearest even
 *   lse     [T, Hq] fp32 output (may be NULL if not wanted)
 * Arithmetic: bf16 products, fp32 accumulation, softmax in fp32 through exp2
 * with log2(e) folded into the scale, probabilities rounded to bf16 before
 * the P.V product.
 * Outputs must not overlap inputs. Supported: d in {64, 128},
 * G in {1, 2, 4, 8, 16}, 1 <= T <= 2^24, 0 <= L <= 1024.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, CUDA (synchronous);
 * TIMEOUT via moda_get_device_error.
 */
MODA_API moda_status moda_fwd(const void* q, const void* k, const void* v,
                     const void* kd, const void* vd, int T, int Hq, int Hk,
                     int d, int L, float scale, void* o, float* lse,
                     moda_stream_t stream);

/*
 * moda_fwd_layer_major -- moda_fwd on the depth K/V in the order the layers
 * write them, with no relayout pass: the chunk-aware grouping of Sec. 3.2
 * (Fig. 4: a query tile's depth rows side by side) happens inside the
 * forward's tensor-memory-accelerator copies, which gather each depth block
 * from the layer-major tensors straight into shared memory. Same result as
 * moda_pack_depth(kd) + moda_pack_depth(vd) + moda_fwd, to rounding order.
 *
 *   kd, vd  [L, T, Hk, d] bf16: slot l of position t for KV head hk at
 *           [l][t][hk][:] (the layout moda_pack_depth takes as its source);
 *           may be NULL when L == 0
 *   every other argument, the arithmetic, the supported shapes and the
 *   errors as moda_fwd.
 */
MODA_API moda_status moda_fwd_layer_major(const void* q, const void* k, const void* v,
                                          const void* kd, const void* vd, int T, int Hq,
                                          int Hk, int d, int L, float scale, void* o,
                                          float* lse, moda_stream_t stream);

/*
 * moda_fwd_layer_major_host -- moda_fwd_layer_major from and to HOST memory,
 * for a caller whose tensors live on the host: the inputs are copied into the
 * caller's device workspace, the forward runs there and o and lse are copied
 * back, all enqueued on `stream` in that order (one cudaMemcpyAsync per
 * tensor; the library allocates nothing).
 *
 *   q, k, v, kd, vd  host buffers with the shapes and layouts of
 *                    moda_fwd_layer_major (kd, vd [L, T, Hk, d]; may be NULL
 *                    when L == 0). Page-locked memory (cudaHostAlloc,
 *                    cudaHostRegister) makes the copies asynchronous; pageable
 *                    memory is accepted, its copies then go through the
 *                    driver's staging buffers and the call may block until
 *                    they are done
 *   o, lse           host outputs ([T, Hq, d] bf16, [T, Hq] fp32; lse may be
 *                    NULL), valid once the stream has passed the call
 *   workspace        device memory owned by the caller, 256-byte aligned, at
 *                    least moda_fwd_host_workspace_bytes(T, Hq, Hk, d, L)
 *                    bytes: the device copies of every input and output
 * The host inputs must stay unchanged, and the outputs unread, until the
 * stream has passed the call; o and lse must not overlap each other or the
 * workspace. Two calls on two streams with two workspaces overlap one call's
 * copies with the other's forward.
 * Errors: as moda_fwd; INVALID_ARG also for a NULL or too small workspace,
 * MISALIGNED for a workspace that is not 256-byte aligned.
 */
MODA_API size_t moda_fwd_host_workspace_bytes(int T, int Hq, int Hk, int d, int L);
MODA_API moda_status moda_fwd_layer_major_host(const void* q, const void* k, const void* v,
                                               const void* kd, const void* vd, int T, int Hq,
                                               int Hk, int d, int L, float scale, void* o,
                                               float* lse, void* workspace,
                                               size_t workspace_bytes, moda_stream_t stream);

/*
 * moda_fwd_depth_cc -- the same result as moda_fwd, with the depth slots on
 * CUDA cores instead of tensor cores: the sequence part runs as moda_fwd with
 * L = 0, then one warp per (KV head, position) reads that position's L slots
 * (16-byte loads of the packed rows), scores them for the G heads of the group
 * and merges its softmax state exactly into o and lse (the joint softmax of
 * Sec. 2.2 split into its sequence and depth halves, lse = log(e^lse_seq +
 * e^lse_depth)). It is the measured alternative to moda_fwd's depth blocks
 * under the block-diagonal mask of Sec. 3.3; moda_fwd is the faster of the two
 * on the measured shapes.
 * Arguments, layouts and errors as moda_fwd, except that lse is required
 * (it carries the sequence part's state into the merge). Probabilities of
 * depth slots stay fp32 here (moda_fwd rounds P to bf16 for the MMA).
 */
MODA_API moda_status moda_fwd_depth_cc(const void* q, const void* k, const void* v,
                                       const void* kd, const void* vd, int T, int Hq, int Hk,
                                       int d, int L, float scale, void* o, float* lse,
                                       moda_stream_t stream);

/*
 * moda_decode -- one decoding step: the new token at position t = Tctx - 1
 * attends, under one softmax, to the sequence KV cache (positions 0..t, its
 * own K/V included) and to the L depth slots of position t (Sec. 2.2; the
 * decode-time depth cache of Table 1 is these L slots of the current token).
 * It is row t of moda_fwd for all Hq heads.
 *
 *   q            [Hq, d] bf16, the new token's queries
 *   k_cache, v_cache  [Tctx, Hk, d] bf16
 *   kd_tok, vd_tok    the L depth slots of position t: KV head hk's slots
 *                form the [L, d] bf16 block at kd_tok + hk*depth_hk_stride
 *                (elements). A standalone [Hk, L, d] tensor has stride L*d;
 *                position t of the packed stream [Hk, T, L, d] has stride
 *                T*L*d (pass &kd[0][t][0][0]). Stride >= L*d, multiple of 8.
 *   o            [Hq, d] bf16 output; lse [Hq] fp32 (natural log) or NULL
 *   workspace    caller-owned device scratch of at least
 *                moda_decode_workspace_bytes(Tctx, Hq, d) bytes
 * Memory-bound: every cache row is read once for the G heads of its KV head.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, CUDA.
 */
MODA_API size_t moda_decode_workspace_bytes(int Tctx, int Hq, int d);
MODA_API moda_status moda_decode(const void* q, const void* k_cache, const void* v_cache,
                                 const void* kd_tok, const void* vd_tok,
                                 long long depth_hk_stride, int Tctx, int Hq, int Hk, int d,
                                 int L, float scale, void* o, float* lse, float* workspace,
                                 size_t workspace_bytes, moda_stream_t stream);

/*
 * moda_decode_strided -- moda_decode with the token's depth slots at any
 * spacing: slot l of KV head hk is the d values at
 * kd_tok + l*depth_slot_stride + hk*depth_hk_stride (elements; the same for
 * vd_tok). For the layer-major depth tensors of moda_fwd_layer_major,
 * [L, T, Hk, d], position t's slots are kd + t*Hk*d with
 * depth_slot_stride = T*Hk*d and depth_hk_stride = d. Both strides >= d and
 * multiples of 8 (depth_hk_stride is not used when Hk == 1); every other
 * argument, the arithmetic and the errors as moda_decode.
 */
MODA_API moda_status moda_decode_strided(const void* q, const void* k_cache, const void* v_cache,
                                         const void* kd_tok, const void* vd_tok,
                                         long long depth_slot_stride, long long depth_hk_stride,
                                         int Tctx, int Hq, int Hk, int d, int L, float scale,
                                         void* o, float* lse, float* workspace,
                                         size_t workspace_bytes, moda_stream_t stream);

/*
 * moda_bwd -- gradients of moda_fwd with respect to all of its inputs. The
 * pages time the fused operator forward + backward (Table 2, Table 7) without
 * writing the backward out; this is the chain rule through the joint softmax
 * of Sec. 2.2. For row (t, h) with probabilities p_c over its candidates c
 * (keys j <= t, then the L depth slots of position t):
 *   D = <dO[t,h], o[t,h]>,  dp_c = <dO[t,h], val_c>,  ds_c = p_c (dp_c - D)
 *   dq[t,h]  = scale * sum_c ds_c key_c
 *   dk[j,hk] = scale * sum of ds_j q[t,h] over the rows that see key j
 *   dv[j,hk] = sum of p_j dO[t,h] over those rows
 *   dkd[hk,t,l], dvd[hk,t,l]: the same for slot l, from the G rows of position t
 *
 *   q, k, v, kd, vd, scale  exactly as passed to moda_fwd (kd/vd packed)
 *   o       [T, Hq, d] bf16   the forward output
 *   lse     [T, Hq] fp32      the forward log-sum-exp (natural log)
 *   dO      [T, Hq, d] bf16   gradient of the loss with respect to o
 *   dq      [T, Hq, d] fp32   outputs, overwritten
 *   dk, dv  [T, Hk, d] fp32
 *   dkd, dvd [Hk, T, L, d] fp32 (packed, like kd/vd); may be NULL when L == 0
 *   delta   [T, Hq] fp32      workspace owned by the caller; holds D on return
 * Arithmetic: bf16 operands, fp32 accumulation; P and dS are rounded to bf16
 * as tensor-core operands. No atomics: results are deterministic.
 * Outputs and the workspace must not overlap the inputs or each other.
 * Same supported shapes as moda_fwd. Errors: INVALID_ARG, UNSUPPORTED,
 * MISALIGNED, CUDA.
 */
MODA_API moda_status moda_bwd(const void* q, const void* k, const void* v, const void* kd,
                              const void* vd, const void* o, const float* lse, const void* dO,
                              int T, int Hq, int Hk, int d, int L, float scale, float* dq,
                              float* dk, float* dv, float* dkd, float* dvd, float* delta,
                              moda_stream_t stream);

/*
 * moda_bwd_layer_major -- moda_bwd for moda_fwd_layer_major: kd, vd and the
 * outputs dkd, dvd are [L, T, Hk, d] (slot l of position t for KV head hk at
 * [l][t][hk][:]), every other argument as moda_bwd. The same values as
 * moda_bwd on the packed streams, element for element (only the depth rows'
 * addresses differ). Errors as moda_bwd.
 */
MODA_API moda_status moda_bwd_layer_major(const void* q, const void* k, const void* v,
                                          const void* kd, const void* vd, const void* o,
                                          const float* lse, const void* dO, int T, int Hq, int Hk,
                                          int d, int L, float scale, float* dq, float* dk,
                                          float* dv, float* dkd, float* dvd, float* delta,
                                          moda_stream_t stream);

/*
 * moda_bwd_noalloc -- moda_bwd without the caller's workspace; the paper has
 * no counterpart. It is meant for callers that cannot give the library device
 * memory for scratch: code whose device memory is owned by another allocator
 * (a framework's caching allocator, a fixed pool sized up front) and code
 * that must not risk cudaMalloc's implicit synchronisation. It allocates
 * nothing: its scratch is a 4 MiB array compiled into the library, held by
 * every GPU that loads it until the process exits.
 *   Arguments and results as moda_bwd, minus `delta`.
 *   Limit: T * Hq <= 1048576 (2^20) rows; larger calls return
 *   MODA_ERR_UNSUPPORTED and launch nothing.
 *   The first call on each device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture. The address belongs to the device's current context:
 *   after cudaDeviceReset the next call looks it up again (that call, too,
 *   should come before any capture). A device that is not an sm_103 part
 *   gives MODA_ERR_NO_DEVICE before any lookup.
 *   All calls share the one array, which keeps the last call's contents;
 *   each call writes every element it reads, so nothing is cleared between
 *   calls. Calls that overlap on the GPU (other streams, other host threads)
 *   race on the array: serialise them.
 */
MODA_API moda_status moda_bwd_noalloc(const void* q, const void* k, const void* v,
                                      const void* kd, const void* vd, const void* o,
                                      const float* lse, const void* dO, int T, int Hq, int Hk,
                                      int d, int L, float scale, float* dq, float* dk, float* dv,
                                      float* dkd, float* dvd, moda_stream_t stream);

/*
 * moda_get_device_error -- synchronises `stream`, then returns and clears
 * the current device's latched kernel error word (MODA_OK if none).
 */
MODA_API moda_status moda_get_device_error(moda_stream_t stream);

/*
 * moda_selftest_wait_timeout -- diagnostic of the failure path; the paper has
 * no counterpart. Launches one thread that waits, through the same bounded
 * shared-memory-barrier wait the forward kernel uses, on a barrier nothing
 * ever arrives on. After timeout_ms (1..5000) the wait gives up and latches
 * MODA_ERR_TIMEOUT in the device error word, as a stalled forward pipeline
 * would; the kernel returns normally and the context stays usable. Read the
 * result with moda_get_device_error. Errors: INVALID_ARG (timeout_ms), CUDA.
 */
MODA_API moda_status moda_selftest_wait_timeout(int timeout_ms, moda_stream_t stream);

/* Static, human-readable name of a status code. */
MODA_API const char* moda_status_string(moda_status s);

/* Detail of the last non-OK status returned on the calling host thread
 * (which argument, which CUDA error). Never NULL. */
MODA_API const char* moda_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* MODA_H_ */
