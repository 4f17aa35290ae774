// swa_api.cu -- the C ABI (include/swa.h): argument validation, planning,
// launches on the caller's stream, status strings and the device error word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "swa_internal.h"

namespace swa {

cuTensorMapEncodeTiled_fn tensor_map_encoder() {
    static cuTensorMapEncodeTiled_fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<cuTensorMapEncodeTiled_fn>(ptr);
    });
    return fn;
}

namespace {
thread_local char g_last_cuda[256] = "";
}

swa_status cuda_fail(cudaError_t e, const char *where) {
    std::snprintf(g_last_cuda, sizeof(g_last_cuda), "%s: %s (%s)", where, cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return SWA_ERR_CUDA;
}

const char *last_cuda_error() { return g_last_cuda; }

#ifndef SWA_CHECK_BOUNDS
#define SWA_CHECK_BOUNDS 0
#endif

namespace {
// Test margin of the bounds-checked build (swa_debug_set_extent_margin).
std::atomic<long long> g_extent_margin{0};
}  // namespace

long long output_extent(long long n) {
    const long long m = n - g_extent_margin.load(std::memory_order_relaxed);
    return m > 0 ? m : 0;
}

int device_sm_count() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev < 64) cached[dev] = n;
    return n;
}

}  // namespace swa

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Byte ranges [a, a+na) and [b, b+nb) overlap?
bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

swa_status check_window(int w, int s) {
    if (w == SWA_W_INF) return SWA_OK;
    if (w < 1 || s < 0 || s >= w) return SWA_ERR_INVALID_ARG;
    if (s > SWA_MAX_SINKS) return SWA_ERR_UNSUPPORTED;
    return SWA_OK;
}

bool valid_dtype(int dtype) { return dtype == SWA_BF16 || dtype == SWA_F16; }

swa_status check_cache(const swa_cache *c) {
    if (c == nullptr) return SWA_ERR_INVALID_ARG;
    if (!valid_dtype(c->dtype)) return SWA_ERR_INVALID_ARG;
    if (c->B < 0 || c->Hkv < 1 || c->cap < 1) return SWA_ERR_INVALID_ARG;
    if (c->d != 64 && c->d != 128) return c->d < 1 ? SWA_ERR_INVALID_ARG : SWA_ERR_UNSUPPORTED;
    const swa_status ws = check_window(c->w, c->s);
    if (ws != SWA_OK) return ws;
    if (c->w != SWA_W_INF && c->cap != c->w) return SWA_ERR_INVALID_ARG;
    if (c->B > 0) {
        if (c->k == nullptr || c->v == nullptr) return SWA_ERR_INVALID_ARG;
        if (!aligned16(c->k) || !aligned16(c->v)) return SWA_ERR_ALIGNMENT;
        const size_t bytes = static_cast<size_t>(c->B) * c->Hkv * c->cap * c->d * 2;
        if (overlap(c->k, bytes, c->v, bytes)) return SWA_ERR_INVALID_ARG;
    }
    return SWA_OK;
}

bool decode_group_supported(int d, int G) {
    (void)d;
    return G == 1 || G == 2 || G == 4 || G == 8;
}

cudaStream_t as_cuda(swa_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Chunked prefill: the chunk's queries sit at key position q_off + i of the
// attended key sequence -- pos0 itself when the cache has not wrapped (and
// always for an infinite window), else w (s sinks + w-s ring slots).
int64_t chunk_q_off(int w, int64_t pos0) {
    if (w == SWA_W_INF) return pos0;
    return pos0 < w ? pos0 : w;
}

}  // namespace

extern "C" {

const char *swa_version(void) { return "0.1.0"; }

const char *swa_last_cuda_error(void) { return swa::last_cuda_error(); }

const char *swa_status_string(swa_status st) {
    switch (st) {
        case SWA_OK: return "SWA_OK";
        case SWA_ERR_INVALID_ARG: return "SWA_ERR_INVALID_ARG";
        case SWA_ERR_UNSUPPORTED: return "SWA_ERR_UNSUPPORTED";
        case SWA_ERR_ALIGNMENT: return "SWA_ERR_ALIGNMENT";
        case SWA_ERR_WORKSPACE: return "SWA_ERR_WORKSPACE";
        case SWA_ERR_CUDA: return "SWA_ERR_CUDA";
        case SWA_ERR_TIMEOUT: return "SWA_ERR_TIMEOUT";
        case SWA_ERR_BOUNDS: return "SWA_ERR_BOUNDS";
    }
    return "SWA_ERR_UNKNOWN";
}

int64_t swa_cache_slot(int64_t p, int w, int s) {
    if (p < 0 || check_window(w, s) != SWA_OK) return -1;
    if (w == SWA_W_INF || p < s) return p;
    return s + (p - s) % (w - s);
}

swa_status swa_check_prefill(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, int B, int L, int Hq, int Hkv, int d, int w,
                             int s) {
    if (B < 0 || L < 0 || Hkv < 1 || Hq < 1 || d < 1) return SWA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return SWA_ERR_INVALID_ARG;
    const swa_status ws = check_window(w, s);
    if (ws != SWA_OK) return ws;
    if (d != 64 && d != 128) return SWA_ERR_UNSUPPORTED;
    const int G = Hq / Hkv;
    if (!pow2(G) || G > 128) return SWA_ERR_UNSUPPORTED;
    if (B == 0 || L == 0) return SWA_OK;
    if (!q || !k || !v || !o) return SWA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return SWA_ERR_ALIGNMENT;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SWA_ERR_ALIGNMENT;
    // tensor-map limit: strides below 2^40 bytes
    if (static_cast<uint64_t>(L) * Hq * d * 2 >= (1ull << 40)) return SWA_ERR_UNSUPPORTED;
    const uint64_t qbytes = static_cast<uint64_t>(B) * L * Hq * d * 2;
    const uint64_t kbytes = static_cast<uint64_t>(B) * L * Hkv * d * 2;
    if (overlap(o, qbytes, q, qbytes) || overlap(o, qbytes, k, kbytes) ||
        overlap(o, qbytes, v, kbytes))
        return SWA_ERR_INVALID_ARG;
    if (lse) {
        const uint64_t lbytes = static_cast<uint64_t>(B) * Hq * L * 4;
        if (overlap(lse, lbytes, o, qbytes) || overlap(lse, lbytes, q, qbytes) ||
            overlap(lse, lbytes, k, kbytes) || overlap(lse, lbytes, v, kbytes))
            return SWA_ERR_INVALID_ARG;
    }
    return SWA_OK;
}

swa_status swa_check_append(const swa_cache *cache, const void *k_new, const void *v_new, int n,
                            int64_t pos0) {
    const swa_status cs = check_cache(cache);
    if (cs != SWA_OK) return cs;
    if (n < 0 || pos0 < 0) return SWA_ERR_INVALID_ARG;
    if (cache->w == SWA_W_INF && pos0 + n > cache->cap) return SWA_ERR_INVALID_ARG;
    if (n == 0 || cache->B == 0) return SWA_OK;
    if (!k_new || !v_new) return SWA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return SWA_ERR_ALIGNMENT;
    const size_t nb = static_cast<size_t>(cache->B) * n * cache->Hkv * cache->d * 2;
    const size_t cb = static_cast<size_t>(cache->B) * cache->Hkv * cache->cap * cache->d * 2;
    if (overlap(k_new, nb, cache->k, cb) || overlap(k_new, nb, cache->v, cb) ||
        overlap(v_new, nb, cache->k, cb) || overlap(v_new, nb, cache->v, cb))
        return SWA_ERR_INVALID_ARG;
    return SWA_OK;
}

swa_status swa_check_decode(const void *q, const swa_cache *cache, const int32_t *pos, int Hq,
                            int w, int s, const void *o, const void *workspace,
                            size_t workspace_bytes, size_t required_bytes) {
    const swa_status cs = check_cache(cache);
    if (cs != SWA_OK) return cs;
    if (Hq < 1 || Hq % cache->Hkv != 0) return SWA_ERR_INVALID_ARG;
    if (w != cache->w) return SWA_ERR_INVALID_ARG;
    if (w != SWA_W_INF && s != cache->s) return SWA_ERR_INVALID_ARG;
    if (!decode_group_supported(cache->d, Hq / cache->Hkv)) return SWA_ERR_UNSUPPORTED;
    // the cache is addressed as B*Hkv*cap rows with 32-bit row coordinates
    if (static_cast<int64_t>(cache->B) * cache->Hkv * cache->cap >= (int64_t(1) << 31))
        return SWA_ERR_UNSUPPORTED;
    if (cache->B == 0) return SWA_OK;
    if (!q || !o || !pos) return SWA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(o)) return SWA_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(pos) & 3u) return SWA_ERR_ALIGNMENT;
    if (required_bytes > 0) {
        if (!workspace || workspace_bytes < required_bytes) return SWA_ERR_WORKSPACE;
        if (!aligned16(workspace)) return SWA_ERR_ALIGNMENT;
    }
    const size_t qb = static_cast<size_t>(cache->B) * Hq * cache->d * 2;
    const size_t cb = static_cast<size_t>(cache->B) * cache->Hkv * cache->cap * cache->d * 2;
    if (overlap(o, qb, q, qb) || overlap(o, qb, cache->k, cb) || overlap(o, qb, cache->v, cb))
        return SWA_ERR_INVALID_ARG;
    if (required_bytes > 0 && (overlap(workspace, required_bytes, o, qb) ||
                               overlap(workspace, required_bytes, cache->k, cb) ||
                               overlap(workspace, required_bytes, cache->v, cb)))
        return SWA_ERR_INVALID_ARG;
    return SWA_OK;
}

size_t swa_prefill_chunk_workspace_bytes(int B, int n, int Hkv, int d, int w, int64_t pos0) {
    if (B <= 0 || n <= 0 || Hkv < 1 || (d != 64 && d != 128) || pos0 < 0) return 0;
    if (w == SWA_W_INF) return 0;
    const int64_t Lk = chunk_q_off(w, pos0) + n;
    return static_cast<size_t>(2) * B * Lk * Hkv * d * 2;
}

swa_status swa_check_prefill_chunk(const void *q, const void *k_new, const void *v_new,
                                   const void *o, const float *lse, const swa_cache *cache, int n,
                                   int64_t pos0, int Hq, const void *workspace,
                                   size_t workspace_bytes) {
    const swa_status cs = check_cache(cache);
    if (cs != SWA_OK) return cs;
    if (n < 0 || pos0 < 0 || Hq < 1 || Hq % cache->Hkv != 0) return SWA_ERR_INVALID_ARG;
    const int G = Hq / cache->Hkv;
    if (!pow2(G) || G > 128) return SWA_ERR_UNSUPPORTED;
    if (cache->w == SWA_W_INF && pos0 + n > cache->cap) return SWA_ERR_INVALID_ARG;
    const int64_t Lk = chunk_q_off(cache->w, pos0) + n;
    if (Lk >= (int64_t(1) << 31)) return SWA_ERR_UNSUPPORTED;
    if (n == 0 || cache->B == 0) return SWA_OK;
    const int B = cache->B, Hkv = cache->Hkv, d = cache->d;
    // tensor-map limit: strides below 2^40 bytes
    if (static_cast<uint64_t>(n) * Hq * d * 2 >= (1ull << 40) ||
        static_cast<uint64_t>(Lk) * Hkv * d * 2 >= (1ull << 40) ||
        static_cast<uint64_t>(cache->cap) * Hkv * d * 2 >= (1ull << 40))
        return SWA_ERR_UNSUPPORTED;
    if (!q || !k_new || !v_new || !o) return SWA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(o))
        return SWA_ERR_ALIGNMENT;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SWA_ERR_ALIGNMENT;
    const size_t need = swa_prefill_chunk_workspace_bytes(B, n, Hkv, d, cache->w, pos0);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return SWA_ERR_WORKSPACE;
        if (!aligned16(workspace)) return SWA_ERR_ALIGNMENT;
    }
    const size_t qb = static_cast<size_t>(B) * n * Hq * d * 2;
    const size_t kb = static_cast<size_t>(B) * n * Hkv * d * 2;
    const size_t cb = static_cast<size_t>(B) * Hkv * cache->cap * d * 2;
    const size_t lb = lse ? static_cast<size_t>(B) * Hq * n * 4 : 0;
    const void *outs[2] = {o, lse};
    const size_t outb[2] = {qb, lb};
    for (int i = 0; i < 2; ++i) {
        if (overlap(outs[i], outb[i], q, qb) || overlap(outs[i], outb[i], k_new, kb) ||
            overlap(outs[i], outb[i], v_new, kb) || overlap(outs[i], outb[i], cache->k, cb) ||
            overlap(outs[i], outb[i], cache->v, cb) || overlap(outs[i], outb[i], workspace, need))
            return SWA_ERR_INVALID_ARG;
    }
    if (overlap(o, qb, lse, lb)) return SWA_ERR_INVALID_ARG;
    if (overlap(k_new, kb, cache->k, cb) || overlap(k_new, kb, cache->v, cb) ||
        overlap(v_new, kb, cache->k, cb) || overlap(v_new, kb, cache->v, cb))
        return SWA_ERR_INVALID_ARG;
    if (need > 0 && (overlap(workspace, need, q, qb) || overlap(workspace, need, k_new, kb) ||
                     overlap(workspace, need, v_new, kb) || overlap(workspace, need, cache->k, cb) ||
                     overlap(workspace, need, cache->v, cb)))
        return SWA_ERR_INVALID_ARG;
    return SWA_OK;
}

swa_status swa_prefill_chunk(const void *q, const void *k_new, const void *v_new, void *o,
                             float *lse, const swa_cache *cache, int n, int64_t pos0, int Hq,
                             void *workspace, size_t workspace_bytes, swa_stream_t stream) {
    SWA_NVTX_RANGE("swa_prefill_chunk");
    const swa_status st = swa_check_prefill_chunk(q, k_new, v_new, o, lse, cache, n, pos0, Hq,
                                                  workspace, workspace_bytes);
    if (st != SWA_OK || n == 0 || cache->B == 0) return st;
    const swa_cache &c = *cache;
    const cudaStream_t cs = as_cuda(stream);
    const int q_off = static_cast<int>(chunk_q_off(c.w, pos0));
    if (c.w == SWA_W_INF) {
        // nothing is evicted: append first, then read K and V in place
        swa_status r = swa::append_launch(c, k_new, v_new, n, pos0, cs);
        if (r != SWA_OK) return r;
        return swa::prefill_launch_offset(q, c.k, c.v, o, lse, c.B, n, Hq, c.Hkv, c.d, c.w, 0,
                                          q_off, q_off + n, c.cap, c.dtype, cs);
    }
    void *wk = workspace;
    void *wv = static_cast<char *>(workspace) + static_cast<size_t>(c.B) * (q_off + n) * c.Hkv * c.d * 2;
    swa_status r = swa::chunk_gather_launch(c, k_new, v_new, n, pos0, q_off, wk, wv, cs);
    if (r != SWA_OK) return r;
    r = swa::prefill_launch_offset(q, wk, wv, o, lse, c.B, n, Hq, c.Hkv, c.d, c.w, c.s, q_off,
                                   q_off + n, 0, c.dtype, cs);
    if (r != SWA_OK) return r;
    return swa::append_launch(c, k_new, v_new, n, pos0, cs);
}

swa_status swa_prefill_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                          int B, int L, int Hq, int Hkv, int d, int w, int s, swa_dtype dtype,
                          swa_stream_t stream) {
    SWA_NVTX_RANGE("swa_prefill_ex");
    if (!valid_dtype(dtype)) return SWA_ERR_INVALID_ARG;
    const swa_status st = swa_check_prefill(q, k, v, o, lse, B, L, Hq, Hkv, d, w, s);
    if (st != SWA_OK || B == 0 || L == 0) return st;
    return swa::prefill_launch(q, k, v, o, lse, B, L, Hq, Hkv, d, w, s, dtype, as_cuda(stream));
}

swa_status swa_prefill(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                       int L, int Hq, int Hkv, int d, int w, int s, swa_stream_t stream) {
    return swa_prefill_ex(q, k, v, o, lse, B, L, Hq, Hkv, d, w, s, SWA_BF16, stream);
}

size_t swa_prefill_varlen_workspace_bytes(int B, int total, int Hq, int Hkv) {
    if (B < 1 || total < 0 || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0) return 0;
    return swa::varlen_workspace_bytes(B, total, Hq, Hkv);
}

swa_status swa_check_prefill_varlen(const void *q, const void *k, const void *v, const void *o,
                                    const float *lse, const int32_t *cu_seqlens, int B, int total,
                                    int max_len, int Hq, int Hkv, int d, int w, int s,
                                    swa_dtype dtype, const void *workspace,
                                    size_t workspace_bytes) {
    if (!valid_dtype(dtype)) return SWA_ERR_INVALID_ARG;
    if (B < 1 || total < 0 || max_len < 0) return SWA_ERR_INVALID_ARG;
    // the packed tensors as one sequence of `total` rows (shapes, window,
    // alignment, overlaps)
    const swa_status st = swa_check_prefill(q, k, v, o, lse, 1, total, Hq, Hkv, d, w, s);
    if (st != SWA_OK) return st;
    if (!cu_seqlens) return SWA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) return SWA_ERR_ALIGNMENT;
    const size_t need = swa::varlen_workspace_bytes(B, total, Hq, Hkv);
    if (!workspace || workspace_bytes < need) return SWA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SWA_ERR_ALIGNMENT;
    const size_t qb = static_cast<size_t>(total) * Hq * d * 2;
    const size_t kb = static_cast<size_t>(total) * Hkv * d * 2;
    const size_t lb = lse ? static_cast<size_t>(total) * Hq * 4 : 0;
    const size_t cb = (static_cast<size_t>(B) + 1) * 4;
    if (overlap(workspace, need, q, qb) || overlap(workspace, need, k, kb) ||
        overlap(workspace, need, v, kb) || overlap(workspace, need, o, qb) ||
        overlap(workspace, need, lse, lb) || overlap(workspace, need, cu_seqlens, cb) ||
        overlap(o, qb, cu_seqlens, cb) || overlap(lse, lb, cu_seqlens, cb))
        return SWA_ERR_INVALID_ARG;
    return SWA_OK;
}

swa_status swa_prefill_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                              const int32_t *cu_seqlens, int B, int total, int max_len, int Hq,
                              int Hkv, int d, int w, int s, swa_dtype dtype, void *workspace,
                              size_t workspace_bytes, swa_stream_t stream) {
    SWA_NVTX_RANGE("swa_prefill_varlen");
    const swa_status st = swa_check_prefill_varlen(q, k, v, o, lse, cu_seqlens, B, total, max_len,
                                                   Hq, Hkv, d, w, s, dtype, workspace,
                                                   workspace_bytes);
    if (st != SWA_OK || total == 0) return st;
    return swa::prefill_varlen_launch(q, k, v, o, lse, cu_seqlens, B, total, max_len, Hq, Hkv, d, w,
                                      w == SWA_W_INF ? 0 : s, dtype, workspace, as_cuda(stream));
}

swa_status swa_cache_append(const swa_cache *cache, const void *k_new, const void *v_new, int n,
                            int64_t pos0, swa_stream_t stream) {
    SWA_NVTX_RANGE("swa_cache_append");
    const swa_status st = swa_check_append(cache, k_new, v_new, n, pos0);
    if (st != SWA_OK) return st;
    return swa::append_launch(*cache, k_new, v_new, n, pos0, as_cuda(stream));
}

size_t swa_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int cap, int w) {
    if (B <= 0 || Hq < 1 || Hkv < 1 || cap < 1 || (d != 64 && d != 128)) return 0;
    return swa::decode_plan(B, Hq, Hkv, d, cap, w, swa::device_sm_count()).workspace;
}

swa_status swa_decode(const void *q, const swa_cache *cache, const int32_t *pos, int Hq, int w,
                      int s, void *o, void *workspace, size_t workspace_bytes,
                      swa_stream_t stream) {
    SWA_NVTX_RANGE("swa_decode");
    if (cache == nullptr) return SWA_ERR_INVALID_ARG;
    const int sms = swa::device_sm_count();
    if (sms <= 0) return swa::cuda_fail(cudaErrorInvalidDevice, "device_sm_count");
    const swa::DecodePlan plan =
        swa::decode_plan(cache->B, Hq, cache->Hkv, cache->d, cache->cap, cache->w, sms);
    const swa_status st =
        swa_check_decode(q, cache, pos, Hq, w, s, o, workspace, workspace_bytes, plan.workspace);
    if (st != SWA_OK || cache->B == 0) return st;
    return swa::decode_launch(q, *cache, pos, Hq, o, workspace, plan, as_cuda(stream));
}

swa_status swa_append_decode(const void *q, const void *k_new, const void *v_new,
                             const swa_cache *cache, const int32_t *pos, int Hq, int w, int s,
                             void *o, void *workspace, size_t workspace_bytes,
                             swa_stream_t stream) {
    SWA_NVTX_RANGE("swa_append_decode");
    if (cache == nullptr) return SWA_ERR_INVALID_ARG;
    const int sms = swa::device_sm_count();
    if (sms <= 0) return swa::cuda_fail(cudaErrorInvalidDevice, "device_sm_count");
    const swa::DecodePlan plan =
        swa::decode_plan(cache->B, Hq, cache->Hkv, cache->d, cache->cap, cache->w, sms);
    const swa_status st =
        swa_check_decode(q, cache, pos, Hq, w, s, o, workspace, workspace_bytes, plan.workspace);
    if (st != SWA_OK || cache->B == 0) return st;
    if (!k_new || !v_new) return SWA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return SWA_ERR_ALIGNMENT;
    const size_t nb = static_cast<size_t>(cache->B) * cache->Hkv * cache->d * 2;
    const size_t qb = static_cast<size_t>(cache->B) * Hq * cache->d * 2;
    const size_t cb = static_cast<size_t>(cache->B) * cache->Hkv * cache->cap * cache->d * 2;
    for (const void *t : {k_new, v_new})
        if (overlap(t, nb, cache->k, cb) || overlap(t, nb, cache->v, cb) || overlap(t, nb, o, qb))
            return SWA_ERR_INVALID_ARG;
    return swa::decode_launch(q, *cache, pos, Hq, o, workspace, plan, as_cuda(stream), nullptr,
                              k_new, v_new);
}

namespace {

// The linear state belongs to the cache: same B, Hkv, d; df in {32, 64};
// 16-byte aligned buffers that overlap neither each other nor the cache.
swa_status check_linear_state(const swa_linear_state *st, const swa_cache *c) {
    if (st == nullptr) return SWA_ERR_INVALID_ARG;
    if (st->B != c->B || st->Hkv != c->Hkv || st->d != c->d) return SWA_ERR_INVALID_ARG;
    if (st->df != 32 && st->df != 64) return st->df < 1 ? SWA_ERR_INVALID_ARG : SWA_ERR_UNSUPPORTED;
    if (c->B == 0) return SWA_OK;
    if (!st->S || !st->z || !st->W) return SWA_ERR_INVALID_ARG;
    if (!aligned16(st->S) || !aligned16(st->z) || !aligned16(st->W)) return SWA_ERR_ALIGNMENT;
    const size_t F = 2 * static_cast<size_t>(st->df);
    const size_t sb = static_cast<size_t>(c->B) * c->Hkv * F * c->d * 4;
    const size_t zb = static_cast<size_t>(c->B) * c->Hkv * F * 4;
    const size_t wb = static_cast<size_t>(c->Hkv) * c->d * st->df * 4;
    const size_t cb = static_cast<size_t>(c->B) * c->Hkv * c->cap * c->d * 2;
    if (overlap(st->S, sb, st->z, zb) || overlap(st->S, sb, st->W, wb) ||
        overlap(st->z, zb, st->W, wb) || overlap(st->S, sb, c->k, cb) ||
        overlap(st->S, sb, c->v, cb) || overlap(st->z, zb, c->k, cb) || overlap(st->z, zb, c->v, cb))
        return SWA_ERR_INVALID_ARG;
    return SWA_OK;
}

}  // namespace

swa_status swa_hybrid_append(const swa_cache *cache, const swa_linear_state *state,
                             const void *k_new, const void *v_new, int n, int64_t pos0,
                             swa_stream_t stream) {
    SWA_NVTX_RANGE("swa_hybrid_append");
    swa_status st = swa_check_append(cache, k_new, v_new, n, pos0);
    if (st != SWA_OK) return st;
    st = check_linear_state(state, cache);
    if (st != SWA_OK || n == 0 || cache->B == 0) return st;
    bool appended = false;
    st = swa::hybrid_fold_launch(*cache, *state, k_new, v_new, n, pos0, as_cuda(stream), &appended);
    if (st != SWA_OK || appended) return st;
    return swa::append_launch(*cache, k_new, v_new, n, pos0, as_cuda(stream));
}

size_t swa_hybrid_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int cap, int w) {
    if (B <= 0 || Hq < 1 || Hkv < 1 || cap < 1 || (d != 64 && d != 128)) return 0;
    const swa::DecodePlan plan = swa::decode_plan(B, Hq, Hkv, d, cap, w, swa::device_sm_count());
    return static_cast<size_t>(B) * Hq * plan.splits * (d + 2) * sizeof(float);
}

swa_status swa_hybrid_decode(const void *q, const swa_cache *cache, const swa_linear_state *state,
                             const int32_t *pos, int Hq, int w, int s, void *o, void *workspace,
                             size_t workspace_bytes, swa_stream_t stream) {
    SWA_NVTX_RANGE("swa_hybrid_decode");
    if (cache == nullptr) return SWA_ERR_INVALID_ARG;
    const int sms = swa::device_sm_count();
    if (sms <= 0) return swa::cuda_fail(cudaErrorInvalidDevice, "device_sm_count");
    const swa::DecodePlan plan =
        swa::decode_plan(cache->B, Hq, cache->Hkv, cache->d, cache->cap, cache->w, sms);
    const size_t need = static_cast<size_t>(cache->B) * Hq * plan.splits * (cache->d + 2) * 4;
    swa_status st =
        swa_check_decode(q, cache, pos, Hq, w, s, o, workspace, workspace_bytes, need);
    if (st != SWA_OK) return st;
    st = check_linear_state(state, cache);
    if (st != SWA_OK || cache->B == 0) return st;
    return swa::decode_launch(q, *cache, pos, Hq, o, workspace, plan, as_cuda(stream), state);
}

swa_status swa_selftest_wait_timeout(swa_stream_t stream) {
    SWA_NVTX_RANGE("swa_selftest_wait_timeout");
    return swa::selftest_wait_launch(as_cuda(stream));
}

swa_status swa_get_device_error(swa_stream_t stream) {
    SWA_NVTX_RANGE("swa_get_device_error");
    const cudaStream_t cs = as_cuda(stream);
    const int e[4] = {swa::prefill_read_clear_error(cs), swa::decode_read_clear_error(cs),
                      swa::append_read_clear_error(cs), swa::hybrid_read_clear_error(cs)};
    for (int v : e)
        if (v == SWA_ERR_CUDA) return SWA_ERR_CUDA;
    for (int v : e)
        if (v != 0) return static_cast<swa_status>(v);
    return SWA_OK;
}

int swa_debug_bounds_checked(void) { return SWA_CHECK_BOUNDS ? 1 : 0; }

int64_t swa_debug_bounds_index(swa_stream_t stream) {
    const cudaStream_t cs = as_cuda(stream);
    const long long w[4] = {swa::prefill_read_clear_where(cs), swa::decode_read_clear_where(cs),
                            swa::append_read_clear_where(cs), swa::hybrid_read_clear_where(cs)};
    for (long long v : w)
        if (v == -2) return -2;
    for (long long v : w)
        if (v != -1) return v;
    return -1;
}

swa_status swa_debug_set_extent_margin(int64_t elements) {
    if (!SWA_CHECK_BOUNDS) return SWA_ERR_UNSUPPORTED;
    if (elements < 0) return SWA_ERR_INVALID_ARG;
    swa::g_extent_margin.store(elements, std::memory_order_relaxed);
    return SWA_OK;
}

}  // extern "C"
