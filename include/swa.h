/*
 * swa.h -- C ABI of the GB300 (sm_103a) library for sliding-window softmax
 * attention with attention sinks, SWA(w,s).
 *
 * The operation.  Query position t attends to the attended set
 *
 *     A(t) = { i : 0 <= i < min(s, t+1) }  U  { i : max(0, t-(w-s)+1) <= i <= t }
 *
 * (0-based positions: the first s tokens plus the latest w-s tokens, each
 * counted once, so |A(t)| = min(t+1, w)), and
 *
 *     o_t = sum_{i in A(t)} exp(c q_t.k_i) v_i / sum_{i in A(t)} exp(c q_t.k_i),
 *     c = 1/sqrt(d).
 *
 * Source: "Sliding-window beats linear attention" (paper summary page),
 * section "Prerequisites / Sliding-window attention SWA(w, s)" -- the window
 * equation for x_t and the SWA(w,s) notation; section "Method steps", step two
 * (w includes the s sinks; s = 4).  w = SWA_W_INF gives full causal attention,
 * the "FA" baseline of the same page's "Research motivation".  Grouped-query
 * heads: query head h reads key/value head h / (Hq/Hkv).
 *
 * Conventions for every call:
 *   - tensors are bf16 -- or fp16 where a call takes an element type
 *     (swa_prefill_ex; the cache's dtype field for the calls on a cache) --,
 *     dense (contiguous) in the stated layout, in device
 *     memory of the current device, 16-byte aligned; the caller owns them and
 *     keeps them alive until the stream work completes;
 *   - calls are asynchronous on `stream` (NULL = the legacy default stream);
 *     the library never allocates device memory and never synchronises, except
 *     swa_get_device_error, which synchronises `stream`;
 *   - per device, the first launch of each kernel sets its attributes and
 *     the library keeps that state for the life of the process: do not reset
 *     a device (cudaDeviceReset) between calls;
 *   - errors are return codes; nothing aborts the process.  Argument errors
 *     are detected on the host before anything is enqueued.  Kernels that hit
 *     an internal wait limit record an error code on the device, read with
 *     swa_get_device_error;
 *   - Q and K arrive already position-encoded: the method changes only the
 *     mask and the cache eviction rule ("Microsoft SWA paper overturns linear
 *     attention", blog page, section "What they tested").
 */
#ifndef SWA_H
#define SWA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st *swa_stream_t;

typedef enum {
    SWA_OK = 0,
    SWA_ERR_INVALID_ARG = -1,  /* shape, window or pointer argument out of range      */
    SWA_ERR_UNSUPPORTED = -2,  /* valid but not built: head size, group size, device   */
    SWA_ERR_ALIGNMENT = -3,    /* a pointer is not 16-byte aligned                     */
    SWA_ERR_WORKSPACE = -4,    /* workspace missing or smaller than required           */
    SWA_ERR_CUDA = -5,         /* a CUDA runtime/driver call or a launch failed        */
    SWA_ERR_TIMEOUT = -6,      /* a kernel gave up waiting (device error word)         */
    SWA_ERR_BOUNDS = -7        /* a kernel skipped an out-of-range access (device word)*/
} swa_status;

/*
 * Element type of the 16-bit tensors.  bf16 is the default; fp16 is the
 * precision of the pages' own system measurements ("Sliding-window beats
 * linear attention", paper summary page, section "Method steps", step five).
 * Either way the kernels compute scores, the softmax and the output
 * accumulator in fp32; the attention weights P enter the P.V product rounded
 * to the element type, and the output is rounded to it (nearest even).
 */
typedef enum {
    SWA_BF16 = 0,
    SWA_F16 = 1
} swa_dtype;

/* Infinite window: full causal attention (A(t) = [0, t]); s is then ignored. */
#define SWA_W_INF (-1)

/* Largest number of sink tokens s this build supports. */
#define SWA_MAX_SINKS 64

/*
 * swa_prefill -- attention of every position of a prompt to its attended set.
 *
 *   q   [B, L, Hq,  d] bf16   queries (position-encoded)
 *   k   [B, L, Hkv, d] bf16   keys (position-encoded)
 *   v   [B, L, Hkv, d] bf16   values
 *   o   [B, L, Hq,  d] bf16   output, written; o_t as defined above, fp32
 *                             accumulation, rounded to bf16 (nearest even)
 *   lse [B, Hq, L]     fp32   optional (NULL to skip): natural-log
 *                             log-sum-exp of c q_t.k_i over A(t)
 *
 * Requires B >= 0, L >= 0 (B*L == 0 is a no-op returning SWA_OK), Hkv >= 1,
 * Hq a multiple of Hkv with G = Hq/Hkv a power of two <= 128, d in {64, 128};
 * w == SWA_W_INF or 0 <= s < w with s <= SWA_MAX_SINKS.  o and lse must not
 * overlap the inputs.  The band of keys a query tile needs is the sink block
 * plus the latest w-s keys before the tile ("Sliding-window beats linear
 * attention", section "Core method": the method adds no operator and
 * changes only the mask).
 */
swa_status swa_prefill(const void *q, const void *k, const void *v, void *o, float *lse,
                       int B, int L, int Hq, int Hkv, int d, int w, int s,
                       swa_stream_t stream);

/*
 * swa_prefill_ex -- swa_prefill with the element type of q, k, v and o given
 * by `dtype` (SWA_BF16 or SWA_F16; any other value returns
 * SWA_ERR_INVALID_ARG).  swa_prefill is swa_prefill_ex with SWA_BF16.
 */
swa_status swa_prefill_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                          int B, int L, int Hq, int Hkv, int d, int w, int s, swa_dtype dtype,
                          swa_stream_t stream);

/*
 * The fixed-size cache of one layer.  k and v are [B, Hkv, cap, d] of element
 * type `dtype` (SWA_BF16 -- the value of a zero-initialised struct -- or
 * SWA_F16) in device memory owned by the caller.  Position p lives in slot
 *     slot(p) = p                      if w == SWA_W_INF or p < s,
 *     slot(p) = s + (p - s) mod (w-s)  otherwise,
 * so cap == w for a finite window (s sink slots + a (w-s)-slot ring: the
 * cache stops growing once it holds the window -- news page "No
 * post-training, just 4 more tokens: sliding window attention overtakes linear
 * attention", section "Research method"), and cap is the longest sequence
 * for w == SWA_W_INF.  While fewer than w positions have been written, they
 * occupy slots [0, pos+1).
 */
typedef struct {
    void *k;
    void *v;
    int32_t B, Hkv, d, cap, w, s;
    int32_t dtype; /* swa_dtype of k, v, and of q and o in the calls on this cache */
} swa_cache;

/*
 * swa_cache_append -- write the keys/values of positions pos0 .. pos0+n-1.
 *
 *   k_new, v_new [B, n, Hkv, d] of the cache's element type (device)
 *
 * Each position is copied bit for bit to slot(p).  When n > w - s several
 * positions share a ring slot; only the latest one is written, so the result
 * equals appending the positions one at a time (the eviction rule of the blog
 * page above).  Requires pos0 >= 0, n >= 0 (0 is a no-op), and for
 * w == SWA_W_INF pos0 + n <= cap.  The cache fields must be consistent
 * (cap == w for finite w, 0 <= s < w, d in {64, 128}).
 */
swa_status swa_cache_append(const swa_cache *cache, const void *k_new, const void *v_new,
                            int n, int64_t pos0, swa_stream_t stream);

/*
 * swa_decode_workspace_bytes -- device workspace swa_decode needs for this
 * shape (0 if none).  Depends only on the arguments and the device's SM count;
 * call it with the same device current as swa_decode.
 */
size_t swa_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int cap, int w);

/*
 * swa_decode -- one new token per sequence attends to the cache.
 *
 *   q   [B, Hq, d]        the query of position pos[b] for each sequence b
 *                          (the cache's element type, as are k, v and o)
 *   pos [B] int32 (device) position of that query; the cache must already
 *                          hold positions 0..pos[b] (append before decode, so
 *                          the token attends to itself: the window equation's
 *                          sum ends at i = t)
 *   o   [B, Hq, d]        output, written
 *   workspace              device memory of at least
 *                          swa_decode_workspace_bytes(...) bytes (may be NULL
 *                          when that is 0); contents need no initialisation
 *
 * Supported group sizes G = Hq/Hkv: 1, 2, 4, 8 (others return
 * SWA_ERR_UNSUPPORTED), and B*Hkv*cap below 2^31.
 * w and s must equal the cache's.  Reads the filled slots
 * [0, min(pos[b]+1, w)) (or [0, pos[b]+1) for SWA_W_INF); the softmax over a
 * set does not depend on slot order.  pos is read on the device and is not
 * advanced, so a captured CUDA graph can be replayed with new positions.
 * A pos[b] outside [0, cap) (infinite window) is recorded as SWA_ERR_BOUNDS in
 * the device error word and that sequence's output is left untouched.
 */
swa_status swa_decode(const void *q, const swa_cache *cache, const int32_t *pos, int Hq,
                      int w, int s, void *o, void *workspace, size_t workspace_bytes,
                      swa_stream_t stream);

/*
 * swa_append_decode -- the decode step of one new token per sequence in one
 * kernel: swa_cache_append of that token at position pos[b], then
 * swa_decode at pos[b] (the operation is the same as the two calls; the
 * window equation of "Sliding-window beats linear attention", paper summary
 * page, section "Prerequisites / Sliding-window attention SWA(w, s)", with
 * the cache's sink + ring slots).
 *
 *   q            [B, Hq, d]   queries of position pos[b]
 *   k_new, v_new [B, Hkv, d]  the token's key and value (a [B, 1, Hkv, d]
 *                             append input is the same memory); written to
 *                             slot(pos[b]) of the cache
 *   pos          [B] int32 (device); the cache must hold positions
 *                0..pos[b]-1 (those still in the window)
 *   o, workspace as for swa_decode (same workspace size)
 *
 * Results, the cache afterwards and the errors are those of the two calls
 * (a pos[b] outside [0, cap) for SWA_W_INF records SWA_ERR_BOUNDS and that
 * sequence's slot and output are left untouched).  pos is read on the
 * device, so a captured graph can be replayed with new positions.  k_new and
 * v_new must be 16-byte aligned and overlap neither the cache nor o.
 */
swa_status swa_append_decode(const void *q, const void *k_new, const void *v_new,
                             const swa_cache *cache, const int32_t *pos, int Hq, int w, int s,
                             void *o, void *workspace, size_t workspace_bytes, swa_stream_t stream);

/* Size of the device scratch built into the library for swa_decode_noalloc. */
#define SWA_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * swa_decode_noalloc -- swa_decode for callers that cannot allocate device
 * memory.  The paper has no counterpart; this is a convenience of the library.
 *
 * Who needs it: code that may not call cudaMalloc or any allocator -- for
 * instance a plugin whose host framework owns all device memory and hands it
 * only the input and output buffers, or a latency-critical serving loop that
 * must not risk the device-wide synchronisation or failure an allocation can
 * bring.  Such callers cannot provide the workspace swa_decode asks for.
 *
 * Same arguments and result as swa_decode, minus the workspace: the split
 * partials go to a device array of SWA_NOALLOC_SCRATCH_BYTES that the library
 * defines at file scope, so every GPU that loads the library holds those 4 MiB
 * until the process exits.  Nothing is allocated and no allocating routine is
 * called.  The first call on each device looks up the array's device address
 * (once, with that device current); make that first call before any stream
 * capture.  The address is kept for the life of the process, so a device
 * reset (cudaDeviceReset) between calls is not supported: the kept address
 * would point into the released context.  If the decode plan for the shape needs more scratch than
 * SWA_NOALLOC_SCRATCH_BYTES, returns SWA_ERR_WORKSPACE before launching
 * anything (on a 152-SM GB300 every supported shape fits).
 *
 * All calls share the one array and it keeps whatever the last call wrote;
 * nothing in it needs to start at zero (each call writes every partial it
 * reads).  Calls whose work overlaps on the GPU -- on different streams, or
 * on different host threads without ordering -- race on the array: keep them
 * ordered, e.g. on one stream.
 */
swa_status swa_decode_noalloc(const void *q, const swa_cache *cache, const int32_t *pos, int Hq,
                              int w, int s, void *o, swa_stream_t stream);

/*
 * Bounds-checked debug build.  The library compiled with SWA_CHECK_BOUNDS=1
 * (the package's build step with that flag) tests, in every kernel, each
 * global access whose index the kernel computes against the extent of its
 * buffer.  An index outside the buffer is not accessed: the kernel records
 * SWA_ERR_BOUNDS (read with swa_get_device_error) and the first such index,
 * and carries on; nothing traps.  Accesses made by the tensor-copy engine
 * are clipped to their tensor maps by the hardware and need no test.  In
 * the normal build the tests are compiled out.  The pages define no such
 * thing; these calls are a debugging aid of the library.
 *
 * swa_debug_bounds_checked -- 1 in the bounds-checked build, else 0.
 *
 * swa_debug_bounds_index -- the first index (in elements, or in 16-byte
 * vectors for vector accesses) a kernel refused since the last call, or -1
 * if none (always -1 in the normal build); -2 if reading it failed.  Reads
 * and clears the record; synchronises `stream`.
 *
 * swa_debug_set_extent_margin -- bounds-checked build only: from now on the
 * kernels are told that every buffer they write (outputs, caches, linear
 * states, workspaces) is `elements` elements shorter than it is, so that
 * they refuse their last writes -- a way to see the checks work without
 * any access outside a real buffer.  0 restores the true extents.  Returns
 * SWA_ERR_UNSUPPORTED in the normal build, SWA_ERR_INVALID_ARG if negative.
 * Process-wide; not for use while other threads launch work.
 */
int swa_debug_bounds_checked(void);
int64_t swa_debug_bounds_index(swa_stream_t stream);
swa_status swa_debug_set_extent_margin(int64_t elements);

/*
 * swa_last_cuda_error -- name and description of the CUDA error behind the
 * most recent SWA_ERR_CUDA returned to the calling thread ("" if none).
 * Diagnostic only; static or thread-local storage owned by the library.
 */
const char *swa_last_cuda_error(void);

/* Human-readable name of a status code (static storage). */
const char *swa_status_string(swa_status status);

/*
 * swa_get_device_error -- synchronise `stream`, then read and clear the device
 * error word of the current device.  Returns SWA_OK if no kernel recorded an
 * error since the last call, else the recorded code (SWA_ERR_TIMEOUT,
 * SWA_ERR_BOUNDS); SWA_ERR_CUDA if the synchronisation itself failed.
 */
swa_status swa_get_device_error(swa_stream_t stream);

/*
 * swa_prefill_chunk -- prefill one chunk of a prompt that continues from a
 * cache, then append the chunk to it.  Positions pos0 .. pos0+n-1 attend to
 * what the cache holds of positions < pos0 (the s sinks and the latest w-s,
 * or every position for w = SWA_W_INF) and to the chunk itself, which is
 * exactly their attended set A(t): prefilling a prompt chunk by chunk with
 * this call gives the outputs of one swa_prefill of the whole prompt, with
 * memory bounded by the cache for a finite window.  The cache then also
 * holds the chunk (as swa_cache_append would leave it).
 *
 *   q        [B, n, Hq, d], positions pos0 .. pos0+n-1
 *   k_new, v_new  [B, n, Hkv, d], the same positions (position-encoded)
 *   o        [B, n, Hq, d] output; lse optional fp32 [B, Hq, n]
 *            (q, k_new, v_new and o of the cache's element type)
 *   cache    holds positions 0 .. pos0-1 exactly as appends left them; its
 *            w and s are the window's (w = SWA_W_INF: pos0 + n <= cap)
 *   workspace  device scratch of swa_prefill_chunk_workspace_bytes(...)
 *            bytes, 16-byte aligned, caller-owned, contents undefined
 *            between calls; 0 bytes (may be NULL) for w = SWA_W_INF, which
 *            reads K and V from the cache in place
 *
 * Enqueues on `stream`, in order, a gather of the attended keys into the
 * workspace (finite window only), the prefill, and the append; the cache must
 * not be used by other work until they complete.  Returns the swa_prefill /
 * swa_cache_append codes; SWA_ERR_WORKSPACE when the workspace is missing or
 * short.
 *
 * Source: the window equation of "Sliding-window beats linear attention"
 * (paper summary page), section "Prerequisites / Sliding-window attention
 * SWA(w, s)"; the fixed cache and its eviction rule: blog page "Microsoft SWA
 * paper overturns linear attention", section "What they tested".
 */
size_t swa_prefill_chunk_workspace_bytes(int B, int n, int Hkv, int d, int w, int64_t pos0);
swa_status swa_prefill_chunk(const void *q, const void *k_new, const void *v_new, void *o,
                             float *lse, const swa_cache *cache, int n, int64_t pos0, int Hq,
                             void *workspace, size_t workspace_bytes, swa_stream_t stream);

/*
 * swa_prefill_varlen -- swa_prefill of B sequences of different lengths in
 * one call (a ragged batch, as a serving system packs it).  The sequences are
 * packed one after the other:
 *
 *   q          [total, Hq,  d]  queries; sequence b is rows
 *                               cu_seqlens[b] .. cu_seqlens[b+1]-1
 *   k, v       [total, Hkv, d]  keys and values, packed the same way
 *   o          [total, Hq,  d]  output; lse optional fp32 [Hq, total]
 *   cu_seqlens [B+1] int32, DEVICE memory: 0 = cu_seqlens[0] <= ... <=
 *              cu_seqlens[B] = total (empty sequences allowed)
 *   max_len    an upper bound of the sequence lengths (host); it only picks
 *              the key tile width for w = SWA_W_INF
 *   workspace  device scratch of swa_prefill_varlen_workspace_bytes(B, total,
 *              Hq, Hkv) bytes, 16-byte aligned, contents undefined between
 *              calls
 *
 * Each position attends to its attended set A(t) within its own sequence
 * (positions counted from the sequence's first row; the sinks are its first
 * s tokens), exactly as swa_prefill of that sequence alone.  cu_seqlens is
 * read on the device: a cu_seqlens that is not such a partition of
 * [0, total) makes the call compute nothing and record SWA_ERR_BOUNDS in the
 * device error word.  Other requirements and codes as swa_prefill_ex.
 *
 * Source: the same window equation ("Sliding-window beats linear
 * attention", paper summary page, section "Prerequisites / Sliding-window
 * attention SWA(w, s)"); the pages' own system measurements run batch 1
 * (same page, section "Method steps", step five).
 */
size_t swa_prefill_varlen_workspace_bytes(int B, int total, int Hq, int Hkv);
swa_status swa_prefill_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                              const int32_t *cu_seqlens, int B, int total, int max_len, int Hq,
                              int Hkv, int d, int w, int s, swa_dtype dtype, void *workspace,
                              size_t workspace_bytes, swa_stream_t stream);
swa_status swa_check_prefill_varlen(const void *q, const void *k, const void *v, const void *o,
                                    const float *lse, const int32_t *cu_seqlens, int B, int total,
                                    int max_len, int Hq, int Hkv, int d, int w, int s,
                                    swa_dtype dtype, const void *workspace,
                                    size_t workspace_bytes);

/*
 * Hybrid window + linear attention (the LoLCATs-style mixture the pages
 * compare SWA(w,s) against: "Sliding-window beats linear attention", paper
 * summary page, sections "Prerequisites / Linear attention" and
 * "Post-training linearisation and LoLCATs").  The cache keeps the attended
 * set A(t) as for SWA(w,s); every token the cache evicts is folded into a
 * linear-attention state instead of being dropped, and decode mixes both:
 *
 *   y_t = ( sum_{i in A(t)} exp(c q.k_i) v_i + phi(q) S ) / ( sum_{i in A(t)} exp(c q.k_i) + phi(q).z )
 *
 * with S = sum of phi(k_i)^T v_i and z = sum of phi(k_i) over the evicted
 * positions (i <= t, i not in A(t)), and the Hedgehog feature map
 * phi(x) = (exp(x W), exp(-x W)) of 2 df features, W a d x df matrix per
 * key/value head (an input: the pages train it, this library takes it as
 * given).  The linear state of one layer:
 */
typedef struct {
    float *S;        /* [B, Hkv, 2*df, d] fp32, device, caller-owned; zero before the first token */
    float *z;        /* [B, Hkv, 2*df] fp32, device, caller-owned; zero before the first token */
    const float *W;  /* [Hkv, d, df] fp32, device: f(x) = x W */
    int32_t B, Hkv, d, df;  /* df in {32, 64}; B, Hkv, d equal to the cache's */
} swa_linear_state;

/*
 * swa_hybrid_append -- swa_cache_append that first folds the positions the
 * append evicts from the ring (from the cache, or from k_new/v_new when a
 * bulk append evicts its own early tokens) into the state.  Appending a
 * prompt of P tokens leaves S, z = the sums over positions s .. P-1-(w-s).
 * Same arguments and codes as swa_cache_append; the state must match the
 * cache (B, Hkv, d) and be 16-byte aligned.  Nothing is evicted for
 * w = SWA_W_INF.
 */
swa_status swa_hybrid_append(const swa_cache *cache, const swa_linear_state *state,
                             const void *k_new, const void *v_new, int n, int64_t pos0,
                             swa_stream_t stream);

/*
 * swa_hybrid_decode -- swa_decode with the linear part of the evicted
 * positions mixed in (the formula above).  Workspace:
 * swa_hybrid_decode_workspace_bytes(...) bytes (never 0).  Same arguments and
 * codes as swa_decode otherwise.
 */
size_t swa_hybrid_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int cap, int w);
swa_status swa_hybrid_decode(const void *q, const swa_cache *cache, const swa_linear_state *state,
                             const int32_t *pos, int Hq, int w, int s, void *o, void *workspace,
                             size_t workspace_bytes, swa_stream_t stream);

/*
 * swa_selftest_wait_timeout -- enqueue a one-CTA kernel whose bounded wait
 * runs out on purpose: it waits on an mbarrier that nothing arrives on,
 * through the same bounded wait as every kernel of the library, holding a
 * TMEM allocation.  After the wait limit (0.2 s) it records SWA_ERR_TIMEOUT,
 * frees the TMEM and returns, so the context stays usable.  Returns SWA_OK
 * when the kernel was enqueued; swa_get_device_error then reports
 * SWA_ERR_TIMEOUT.  For tests of the failure path; no GPU fault is involved.
 */
swa_status swa_selftest_wait_timeout(swa_stream_t stream);

/*
 * Host-only argument checks: the validation the calls above run before
 * enqueuing anything, without touching the GPU.  Same return codes.
 */
swa_status swa_check_prefill(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, int B, int L, int Hq, int Hkv, int d, int w,
                             int s);
swa_status swa_check_append(const swa_cache *cache, const void *k_new, const void *v_new, int n,
                            int64_t pos0);
swa_status swa_check_decode(const void *q, const swa_cache *cache, const int32_t *pos, int Hq,
                            int w, int s, const void *o, const void *workspace,
                            size_t workspace_bytes, size_t required_bytes);

swa_status swa_check_prefill_chunk(const void *q, const void *k_new, const void *v_new,
                                   const void *o, const float *lse, const swa_cache *cache, int n,
                                   int64_t pos0, int Hq, const void *workspace,
                                   size_t workspace_bytes);

/* Slot of position p in a cache of window w with s sinks (host helper; -1 if invalid). */
int64_t swa_cache_slot(int64_t p, int w, int s);

/* Library version, e.g. "0.1.0". */
const char *swa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SWA_H */
