/*
 * moda.h — C ABI of the MoDA (Mixture-of-Depths Attention) library for one
 * NVIDIA GB300 (sm_103a).
 *
 * Operation (paper "Mixture-of-Depths Attention", arXiv:2603.15619; slides frame
 * "One denominator allocates probability across both memories", teaching form of
 * Sec. 2.2 and Algorithm 1): for batch b, query head h, position t, with
 * kv head g = h / G and G = H / Hkv (consecutive query heads share a kv head,
 * G = H_q / H_k as in the slides' Table 1 frame):
 *
 *     a_j = scale * q[b,h,t,:] . k[b,g,j,:]            j = 0 .. t     (causal)
 *     b_i = scale * q[b,h,t,:] . kd[b,g,t,i,:]         i = 0 .. S-1   (same position)
 *     o[b,h,t,:] = (sum_j e^{a_j} v[b,g,j,:] + sum_i e^{b_i} vd[b,g,t,i,:])
 *                  / (sum_j e^{a_j} + sum_i e^{b_i})
 *     lse[b,h,t] = ln(sum_j e^{a_j} + sum_i e^{b_i})
 *
 * Both memories share ONE softmax denominator; the depth slots are never
 * normalised separately (same frame, and "Shared online-softmax states
 * preserve the joint operator", Algorithm 1).  S = 0 is plain causal attention.
 *
 * Layouts: every tensor is dense, contiguous and row-major exactly as shaped:
 *     q, o, dout, dq        [B, H,   T, d]
 *     k, v, dk, dv          [B, Hkv, T, d]
 *     kd, vd, dkd, dvd      [B, Hkv, T, S, d]   (the [S, d] slab of one position is contiguous;
 *                                               [B, Hkv, T, C, d] with a slot capacity C, below)
 *     lse                   [B, H,   T]         float32, natural log
 * Element type: all of q..vd, o, dout and the gradients share desc->dtype;
 * lse is always float32.  Arithmetic accumulates in float32.
 *
 * Ownership: the caller owns every buffer (device memory unless a function says
 * otherwise); the library keeps no pointer after a call returns and allocates no
 * device memory.  Every device pointer must be 16-byte aligned.
 *
 * Streams: work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and the call returns without waiting, unless MODA_SYNC=1 is set in the
 * environment, in which case each call waits for its stream and reports device-side
 * errors (see moda_device_status).
 *
 * Errors: invalid or unsupported arguments are reported synchronously and
 * nothing is launched.  A failed launch returns MODA_ERR_CUDA.  Kernels never
 * trap: a bounded wait that runs out records MODA_ERR_TIMEOUT in a device status
 * word and the kernel returns early (its outputs are then undefined).
 */
#ifndef MODA_H_
#define MODA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MODA_OK = 0,
  MODA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer, H % Hkv != 0 */
  MODA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head dim, dtype) */
  MODA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  MODA_ERR_TIMEOUT = 4,      /* a device-side bounded wait ran out */
  MODA_ERR_WORKSPACE = 5     /* workspace missing or smaller than moda_bwd_workspace_bytes */
} moda_status;

typedef enum { MODA_DTYPE_F32 = 0, MODA_DTYPE_BF16 = 1 } moda_dtype;

/* Problem description.  B >= 1, H >= 1, Hkv >= 1 with H % Hkv == 0, T >= 1,
 * S >= 0 (S = 0: the depth history H_l is empty), d in {64, 128}.
 * scale <= 0 selects 1/sqrt(d) (the slides' a_j, b_i use 1/sqrt(d)).
 *
 * slot_capacity (bounded slot buffer; "Mixture-of-Depths Attention", the closing
 * frame's S << L slot buffer with a sliding window): 0 means kd/vd hold exactly S
 * slots per position.  Otherwise kd/vd (and dkd/dvd) are [B, Hkv, T, C, d] with
 * C = slot_capacity >= S, and only slots 0 .. S-1 of each position are read; the
 * layer's depth memory is those S slots, in any order (the softmax does not depend on
 * the order of its keys).  A sliding window of the last C slots written is a ring:
 * the w-th write goes to slot w mod C (moda_depth_store_kv / moda_depth_project_kv),
 * and a reader passes S = min(writes so far, C).  The unread slots S .. C-1 are never
 * read (they may hold anything, NaN included, e.g. a ring's unwritten slots), so a
 * half-full ring costs half the depth traffic; moda_bwd sets dkd/dvd of the unread
 * slots to zero. */
typedef struct {
  int32_t B, H, Hkv, T, S, d;
  int32_t dtype; /* moda_dtype */
  float scale;
  int32_t slot_capacity;
} moda_desc;

/* Forward (the operation above).
 * In:  q, k, v, kd, vd (device, desc->dtype; kd/vd may be NULL when S == 0).
 * Out: o (device, desc->dtype), lse (device, float32, may be NULL to skip it).
 * bf16 with d in {64, 128} runs on the tensor cores: tcgen05 MMAs with float32
 * accumulation for both memories (the depth slots read by each query's position enter
 * the same online softmax as one extra key step per 128 slots read, their products
 * masked to the rows of each position's queries; slots not read are never loaded), P
 * rounded to bf16 for the PV products.  float32 runs on the CUDA cores in float32. */
moda_status moda_fwd(const moda_desc* desc, const void* q, const void* k, const void* v, const void* kd,
                     const void* vd, void* o, float* lse, void* stream);

/* Bytes of device workspace moda_bwd needs for `desc` (float32 row statistics
 * and the float32 dq accumulator).  0 on invalid desc. */
size_t moda_bwd_workspace_bytes(const moda_desc* desc);

/* Backward: gradients of L = sum(dout * o) for the forward above (the pages give
 * no backward; this is the analytic gradient of the operation).  With
 * P = exp(score - lse), D_t = sum(dout_t * o_t), dS = P * (dout . value - D_t):
 *     dq  = scale * sum dS * key            (sequence keys and depth slots)
 *     dk  = scale * sum dS * q,  dv  = sum P * dout   (summed over the G heads and rows t >= j)
 *     dkd = scale * sum dS * q,  dvd = sum P * dout   (summed over the G heads of position t)
 * In:  q, k, v, kd, vd, o, lse (as written by moda_fwd), dout (device).
 * Out: dq, dk, dv, dkd, dvd (device, desc->dtype; dkd/dvd may be NULL when S == 0).
 * workspace: device scratch of at least moda_bwd_workspace_bytes(desc) bytes,
 * 256-byte aligned; its contents on entry do not matter.  Calls that share a
 * workspace must not overlap on the GPU.
 * bf16 with d in {64, 128} and G = H / Hkv <= 8 runs on the tensor cores (the depth
 * slots on the CUDA cores); G > 8 (and float32) runs every part on the CUDA cores,
 * which is correct but several times slower. */
moda_status moda_bwd(const moda_desc* desc, const void* q, const void* k, const void* v, const void* kd,
                     const void* vd, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                     void* dv, void* dkd, void* dvd, void* workspace, size_t workspace_bytes, void* stream);

/* moda_bwd with timing marks for profilers and benchmarks: same arguments, kernels and
 * results, plus `events`, an array of n_events cudaEvent_t handles (created by the
 * caller; entries may be NULL).  Stage k is bracketed by events[2k] (start) and
 * events[2k+1] (end), recorded on the stream that runs it: 0 = row statistics (Delta),
 * 1 = depth-slot gradients, 2 = dK/dV, 3 = dQ.  Events beyond n_events are not recorded.
 */
moda_status moda_bwd_profiled(const moda_desc* desc, const void* q, const void* k, const void* v, const void* kd,
                              const void* vd, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                              void* dv, void* dkd, void* dvd, void* workspace, size_t workspace_bytes, void* stream,
                              void** events, int32_t n_events);

/* Decode step (one new token per sequence; "Mixture-of-Depths Attention", the decode
 * cache of the Table 1 frame "Depth compute still accumulates quadratically in depth",
 * with the operation above): for every (b, h) the query of the newest position t = T-1
 * attends to the sequence keys 0 .. T-1 of the cache (itself included) and to the S
 * depth slots of its own position, under one softmax:
 *     a_j = scale * q[b,h,:] . k_cache[b,g,j,:]     j = 0 .. T-1
 *     b_i = scale * q[b,h,:] . kd[b,g,i,:]          i = 0 .. S-1
 *     o[b,h,:] = (sum_j e^{a_j} v_cache[b,g,j,:] + sum_i e^{b_i} vd[b,g,i,:]) / (sum of the weights)
 *     lse[b,h] = ln(sum of the weights)
 * This is row T-1 of moda_fwd for the same inputs.
 * desc: B, H, Hkv, S, d as for moda_fwd; T = number of cached positions (>= 1);
 *       dtype must be MODA_DTYPE_BF16 (else MODA_ERR_UNSUPPORTED); G = H/Hkv <= 8.
 * Layouts (device, bf16, dense row-major):
 *     q, o                   [B, H, d]
 *     k_cache, v_cache       [B, Hkv, kv_capacity, d]   (positions 0 .. T-1 are read)
 *     kd, vd                 [B, Hkv, S, d]            (may be NULL when S == 0;
 *                                                      [B, Hkv, C, d] with a slot capacity C)
 *     lse                    [B, H] float32, natural log (may be NULL)
 * kv_capacity: positions allocated per (b, kv head) in the cache; 0 means T; it must
 * be >= T, and B*Hkv*kv_capacity and B*Hkv*S must be below 2^31.
 * workspace: device scratch of at least moda_decode_workspace_bytes(desc) bytes,
 * 256-byte aligned (per-split partial softmax states); calls sharing it must not
 * overlap on the GPU.  Errors as for moda_fwd; MODA_ERR_WORKSPACE when the workspace
 * is missing or too small.
 * Runs two kernels: a key-split pass (TMA-staged K/V sub-tiles of 128 keys; the scores
 * and P V of each sub-tile as tensor-core products with float32 accumulation, P rounded to
 * bf16; the online softmax in float32 on the CUDA cores; the depth slots as one more
 * split) and a merge. */
size_t moda_decode_workspace_bytes(const moda_desc* desc);
moda_status moda_decode(const moda_desc* desc, int64_t kv_capacity, const void* q, const void* k_cache,
                        const void* v_cache, const void* kd, const void* vd, void* o, float* lse, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Depth-KV write path ("Mixture-of-Depths Attention", frame "Reuse attention KV; add a
 * projection for FFN inputs", Sec. 2.2, and Table 3's KV-projection variants): a layer
 * writes its contributions to the depth cache that later layers' moda_fwd reads as
 * kd, vd [B, Hkv, T, S, d], one slot at a time.  Only slot `slot` is written; every
 * other slot, and every other byte of kd/vd, is left as it was.
 * desc: B, Hkv, T, S, d as for moda_fwd (H and scale are not used; H must still be a
 * positive multiple of Hkv); dtype must be MODA_DTYPE_BF16 (else MODA_ERR_UNSUPPORTED);
 * 0 <= slot < C, the slots per position in memory (slot_capacity, or S when that is 0;
 * else MODA_ERR_INVALID_ARG).  Pointers are device memory, 16-byte
 * aligned, dense row-major; the caller owns them all.  Launch errors return
 * MODA_ERR_CUDA; nothing is allocated.
 *
 * moda_depth_store_kv: the attention KV reused as a slot:
 *     kd[b,g,t,slot,:] = k[b,g,t,:],  vd[b,g,t,slot,:] = v[b,g,t,:]
 * with k, v [B, Hkv, T, d].  One strided-copy kernel (exact). */
moda_status moda_depth_store_kv(const moda_desc* desc, int32_t slot, const void* k, const void* v, void* kd,
                                void* vd, void* stream);

/* moda_depth_project_kv: the FFN input projected into a slot:
 *     kd[b,g,t,slot,c] = sum_m x[b,t,m] * wk[m, g*d + c]
 *     vd[b,g,t,slot,c] = sum_m x[b,t,m] * wv[m, g*d + c]
 * with x [B, T, d_model] and wk, wv [d_model, Hkv*d] (bf16).  Products are summed in
 * float32 on the tensor cores and rounded to bf16 once.  d_model must be a positive
 * multiple of 8 and Hkv*d a multiple of 64 (else MODA_ERR_INVALID_ARG /
 * MODA_ERR_UNSUPPORTED).  One GEMM kernel whose epilogue stores straight into the slot. */
moda_status moda_depth_project_kv(const moda_desc* desc, int32_t slot, int32_t d_model, const void* x,
                                  const void* wk, const void* wv, void* kd, void* vd, void* stream);

/* moda_bwd for callers that cannot allocate device memory (allocator hooks, runtimes
 * with a device-memory budget fixed at start-up, plain-C callers without an
 * allocator).  The paper has no counterpart: this is a library convenience.
 * Same arguments and results as moda_bwd minus the workspace, which is taken from a
 * fixed array of moda_bwd_noalloc_max_workspace_bytes() (32 MiB) inside the
 * library's device image; nothing is allocated.  Problems whose
 * moda_bwd_workspace_bytes exceeds that size return MODA_ERR_WORKSPACE without
 * launching.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it, so that first call should precede any stream
 * capture on that device; after a cudaDeviceReset of a device the cached address is no
 * longer valid and this entry point must not be called on that device again.  Every
 * call shares the array: calls that overlap on the GPU race and must be serialised by
 * the caller. */
moda_status moda_bwd_noalloc(const moda_desc* desc, const void* q, const void* k, const void* v, const void* kd,
                             const void* vd, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                             void* dv, void* dkd, void* dvd, void* stream);

/* Size in bytes of the fixed scratch array moda_bwd_noalloc uses. */
size_t moda_bwd_noalloc_max_workspace_bytes(void);

/* ---------------------------------------------------------------- context parallelism
 * The pieces of a split of the positions 0 .. T-1 into chunks that live on different GPUs
 * ("Mixture-of-Depths Attention", the future work of frame "The main open cost is
 * retaining and reading depth history").  A query chunk's output is the joint softmax over
 * the sequence keys of the chunks it sees and the depth slots of its own positions; the
 * depth slots are read only by their own position (frame "Depth retrieval is restricted to
 * the same token position"), so they never leave the GPU that holds the position.  Each
 * (query chunk, key chunk) pair gives a partial state (O, lse) over that key chunk alone;
 * moda_merge_partial combines the states by the online rule of frame "Shared
 * online-softmax states preserve the joint operator".  Moving K/V between GPUs is the
 * caller's (e.g. NCCL send/recv into its own device buffers); these calls read only local
 * device memory.
 *
 * Chunk geometry (both moda_fwd_partial and moda_bwd_partial):
 *   desc->T  query positions of the query chunk: q, o, dout, dq [B,H,T,d], lse [B,H,T];
 *   desc->S  depth slots read with this key chunk: S > 0 in exactly one call per query
 *            chunk (normally the pair of the chunk with itself), kd/vd/dkd/dvd
 *            [B,Hkv,T,C,d] of the query chunk's own positions; S = 0 otherwise (kd, vd,
 *            dkd, dvd may be NULL);
 *   Tk       positions of the key chunk: k, v, dk_acc, dv_acc [B,Hkv,Tk,d];
 *   delta    first query position minus first key position: key j of the chunk is visible
 *            to query t of the chunk iff j <= t + delta.  0 <= delta and 1 <= Tk <= T + delta
 *            (every query sees key 0, the last query sees every key), else
 *            MODA_ERR_INVALID_ARG.  A chunk with itself: Tk = T, delta = 0 (moda_fwd's causal
 *            mask).  A key chunk that ends before the query chunk starts: delta >= Tk - 1,
 *            every key visible.  Pairs whose key chunk starts after the query chunk's
 *            first position are not called (their keys are causally invisible).
 * Errors, alignment, streams and ownership as for moda_fwd / moda_bwd. */

/* Partial forward: o (desc->dtype) and lse (float32, required) of the query chunk over
 * the visible keys of this key chunk (and the depth slots when S > 0) alone, normalised
 * over those keys. */
moda_status moda_fwd_partial(const moda_desc* desc, int32_t Tk, int32_t delta, const void* q, const void* k,
                             const void* v, const void* kd, const void* vd, void* o, float* lse, void* stream);

/* Merge of one partial state into a running state, rows = B*H*T of desc (d, dtype from desc):
 *     m = max(lse_acc, lse_part),  w_a = e^{lse_acc - m},  w_b = e^{lse_part - m}
 *     o_acc = (w_a o_acc + w_b o_part) / (w_a + w_b),   lse_acc = m + ln(w_a + w_b)
 * o_acc [B,H,T,d] and lse_acc [B,H,T] are float32 and updated in place; o_part
 * (desc->dtype) and lse_part (float32) are one moda_fwd_partial output.  first != 0 sets
 * the running state to the partial one (o_acc, lse_acc are not read).  o_out (desc->dtype,
 * may be NULL) receives the merged o_acc.  Once every visible key chunk is merged, o_acc
 * and lse_acc are moda_fwd's o and lse of the query chunk (in float32, up to rounding; the
 * order of the merges does not matter).  One elementwise kernel. */
moda_status moda_merge_partial(const moda_desc* desc, float* o_acc, float* lse_acc, const void* o_part,
                               const float* lse_part, int32_t first, void* o_out, void* stream);

/* Partial backward of one (query chunk, key chunk) pair, with the Tk, delta and S of its
 * moda_fwd_partial call.  o and lse are the query chunk's MERGED output and lse (over
 * every key chunk), dout the gradient of o.  Adds this pair's share of the gradients, in
 * float32:
 *     dq_acc [B,H,T,d]          += dq of the query chunk through this key chunk (and the
 *                                  depth slots when S > 0)
 *     dk_acc, dv_acc [B,Hkv,Tk,d] += dk, dv of the key chunk from this query chunk's rows
 * and, when S > 0, writes dkd, dvd (desc->dtype) of the query chunk's depth slots whole
 * (only their own position's rows see them).  Summed over every pair, dq_acc, dk_acc and
 * dv_acc are moda_bwd's dq, dk, dv in float32 (moda_convert_f32 rounds them).  workspace:
 * at least moda_bwd_workspace_bytes(desc), as for moda_bwd. */
moda_status moda_bwd_partial(const moda_desc* desc, int32_t Tk, int32_t delta, const void* q, const void* k,
                             const void* v, const void* kd, const void* vd, const void* o, const float* lse,
                             const void* dout, float* dq_acc, float* dk_acc, float* dv_acc, void* dkd, void* dvd,
                             void* workspace, size_t workspace_bytes, void* stream);

/* dst[i] = src[i] rounded to dtype (MODA_DTYPE_BF16: round to nearest even; MODA_DTYPE_F32:
 * a copy) for i < n; src float32, both device, 16-byte aligned.  One elementwise kernel
 * (none when n = 0). */
moda_status moda_convert_f32(int64_t n, const float* src, int32_t dtype, void* dst, void* stream);

/* Reads the device status word that bounded waits write (MODA_OK when clean) and,
 * when `clear` is non-zero, resets it.  Waits for `stream` first. */
moda_status moda_device_status(int clear, void* stream);

/* Human-readable name of a status code (static storage). */
const char* moda_status_str(moda_status status);

/* Self-test of the device-side failure path (no counterpart in the paper: it exists
 * so the timeout handling can be tested without hanging or faulting a GPU).
 * Launches one CTA whose first warp waits on an mbarrier that no thread arrives at
 * for at most limit_ns nanoseconds (clamped to [1e6, 2e9]) and then raises the CTA's
 * abort flag; its second warp waits on the same barrier and must leave on that flag,
 * long before the 2 s cap every kernel wait has.  Waits for `stream`, then returns
 * the status word and clears it: MODA_ERR_TIMEOUT when both waits gave up the
 * designed way, MODA_ERR_CUDA if either did not or a CUDA call failed.  A status
 * left by an earlier call is cleared first.  The context stays usable. */
moda_status moda_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Library version as major*10000 + minor*100 + patch. */
int32_t moda_version(void);

/* Number of CUDA kernels this library has launched since it was loaded (all
 * devices and streams; host-side count, no synchronisation). */
int64_t moda_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MODA_H_ */
