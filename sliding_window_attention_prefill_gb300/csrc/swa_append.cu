// swa_append.cu -- write new keys/values into the fixed SWA(w,s) cache.
//
// Position p goes to slot p (sinks, or any position when w is infinite) or
// to ring slot s + (p - s) mod (w - s).  The cache thereby holds the first s
// tokens plus the latest w-s tokens and stops growing at w ("Microsoft SWA
// paper overturns linear attention", blog page, section "What they tested":
// only the mask and the KV-cache eviction rule change; news page "No
// post-training, just 4 more tokens", section "Research method").
//
// A bulk append of n > w-s positions maps several of them to one ring slot;
// only the survivors are written -- the sinks among the new positions and
// the latest w-s of them -- so the result is the same as appending one
// position at a time, no two threads write the same slot, and a long prompt
// costs O(w) rather than O(n).  Pure copy: 16-byte vectors, one per
// thread, coalesced on both sides.
#include <cuda_runtime.h>

#include <cstdint>

#include "swa_internal.h"
#include "swa_ptx.cuh"

namespace swa {

__device__ int g_append_error;
__device__ unsigned long long g_append_where;

struct AppendParams {
    const uint4 *k_new;  // [B, n, Hkv, d] as 16-byte vectors
    const uint4 *v_new;
    uint4 *ck;           // [B, Hkv, cap, d]
    uint4 *cv;
    int64_t pos0;
    int B, n, Hkv, vpr, vpr_log2, cap, w, s;  // vpr: 16-byte vectors per row (d / 8)
    int a, b0;  // surviving new positions: j in [0, a) and j in [b0, n)
    long long n_new, n_cache;  // extents in 16-byte vectors (bounds-checked build)
};

// Grid (vector blocks, surviving positions, sequences): the threads of the x
// dimension cover the Hkv * d / 8 vectors of one position; y and z walk the
// surviving positions and the sequences (grid-stride, so any count fits the
// 65535 limit of those grid dimensions).  The only integer work per vector is
// one slot computation.
constexpr int kAppendThreads = 128;

__global__ void __launch_bounds__(kAppendThreads) swa_append_kernel(const AppendParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const int per_pos = p.Hkv * p.vpr;  // vectors of one position (all kv heads)
    const int t = blockIdx.x * kAppendThreads + threadIdx.x;
    if (t >= per_pos) return;
    const int h = t >> p.vpr_log2;
    const int vec = t & (p.vpr - 1);
    const int m = p.a + (p.n - p.b0);  // surviving positions per sequence
    for (int b = blockIdx.z; b < p.B; b += gridDim.z) {
        for (int jj = blockIdx.y; jj < m; jj += gridDim.y) {
            const int j = jj < p.a ? jj : p.b0 + (jj - p.a);
            const int64_t pos = p.pos0 + j;
            const int64_t slot =
                (p.w < 0 || pos < p.s) ? pos : p.s + (pos - p.s) % static_cast<int64_t>(p.w - p.s);
            const int64_t src = (static_cast<int64_t>(b) * p.n + j) * per_pos + t;
            const int64_t dst = ((static_cast<int64_t>(b) * p.Hkv + h) * p.cap + slot) * p.vpr + vec;
            if (!in_bounds(src, p.n_new, &g_append_error, &g_append_where) ||
                !in_bounds(dst, p.n_cache, &g_append_error, &g_append_where))
                continue;
            const uint4 kv = p.k_new[src];
            const uint4 vv = p.v_new[src];
            p.ck[dst] = kv;
            p.cv[dst] = vv;
        }
    }
}

swa_status append_launch(const swa_cache &c, const void *k_new, const void *v_new, int n,
                         int64_t pos0, cudaStream_t stream) {
    if (n == 0 || c.B == 0) return SWA_OK;
    AppendParams p{};
    p.k_new = static_cast<const uint4 *>(k_new);
    p.v_new = static_cast<const uint4 *>(v_new);
    p.ck = static_cast<uint4 *>(c.k);
    p.cv = static_cast<uint4 *>(c.v);
    p.pos0 = pos0;
    p.B = c.B;
    p.n = n;
    p.Hkv = c.Hkv;
    p.vpr = c.d / 8;
    p.vpr_log2 = p.vpr == 16 ? 4 : 3;  // d is 128 or 64
    p.cap = c.cap;
    p.w = c.w < 0 ? -1 : c.w;
    p.s = c.w < 0 ? 0 : c.s;
    p.n_new = static_cast<long long>(c.B) * n * c.Hkv * c.d / 8;
    p.n_cache = output_extent(static_cast<long long>(c.B) * c.Hkv * c.cap * c.d) / 8;
    if (p.w < 0) {
        p.a = n;  // every position keeps its own slot
        p.b0 = n;
    } else {
        // sinks among the new positions, then the latest w-s of them
        const int64_t a = p.s - pos0;
        p.a = static_cast<int>(a < 0 ? 0 : (a > n ? n : a));
        const int64_t b0 = static_cast<int64_t>(n) - (p.w - p.s);
        p.b0 = static_cast<int>(b0 < p.a ? p.a : b0);
    }
    const int m = p.a + (n - p.b0);  // surviving positions per sequence
    if (m == 0) return SWA_OK;
    const int per_pos = p.Hkv * p.vpr;
    const dim3 grid((per_pos + kAppendThreads - 1) / kAppendThreads,
                    static_cast<unsigned>(m < 65535 ? m : 65535),
                    static_cast<unsigned>(c.B < 65535 ? c.B : 65535));
    const cudaError_t e = launch_pdl(swa_append_kernel, grid, dim3(kAppendThreads), 0, stream, p);
    return e == cudaSuccess ? SWA_OK : cuda_fail(e, "launch swa_append_kernel");
}

// ---------------------------------------------------------------------------
// chunked prefill: the keys a chunk of queries attends to, in one sequence
// ---------------------------------------------------------------------------
// A chunk of positions pos0 .. pos0+n-1 of a finite window attends to the
// sinks and the latest w-s positions before it (what the cache holds) and to
// itself.  Row j < q_off of the gathered sequence is cache position
//   j                              if the cache has not wrapped (pos0 <= w)
//   j (sink) or pos0-(w-s)+(j-s)   otherwise (q_off = w)
// read from its slot; row q_off + i is chunk row i.  In these coordinates a
// query at chunk row i sits at position q_off + i and attends to exactly the
// SWA(w,s) set of that position, so the ordinary prefill runs on them.
struct GatherParams {
    const uint4 *ck, *cv;        // cache [B, Hkv, cap, d]
    const uint4 *k_new, *v_new;  // chunk [B, n, Hkv, d]
    uint4 *wk, *wv;              // gathered [B, q_off + n, Hkv, d]
    int64_t pos0;
    int B, n, Hkv, vpr, vpr_log2, cap, w, s, q_off;
    long long n_cache, n_new, n_ws;  // extents in 16-byte vectors (bounds-checked build)
};

__global__ void __launch_bounds__(kAppendThreads) swa_chunk_gather_kernel(const GatherParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const int per_pos = p.Hkv * p.vpr;  // vectors of one row (all kv heads)
    const int t = blockIdx.x * kAppendThreads + threadIdx.x;
    if (t >= per_pos) return;
    const int h = t >> p.vpr_log2;
    const int vec = t & (p.vpr - 1);
    const int Lk = p.q_off + p.n;
    for (int b = blockIdx.z; b < p.B; b += gridDim.z) {
        for (int j = blockIdx.y; j < Lk; j += gridDim.y) {
            uint4 kv, vv;
            if (j < p.q_off) {
                int64_t pos = j;
                if (p.pos0 > p.w && j >= p.s) pos = p.pos0 - (p.w - p.s) + (j - p.s);
                const int64_t slot = pos < p.s ? pos : p.s + (pos - p.s) % (p.w - p.s);
                const int64_t src = ((static_cast<int64_t>(b) * p.Hkv + h) * p.cap + slot) * p.vpr + vec;
                if (!in_bounds(src, p.n_cache, &g_append_error, &g_append_where)) continue;
                kv = p.ck[src];
                vv = p.cv[src];
            } else {
                const int64_t src = (static_cast<int64_t>(b) * p.n + (j - p.q_off)) * per_pos + t;
                if (!in_bounds(src, p.n_new, &g_append_error, &g_append_where)) continue;
                kv = p.k_new[src];
                vv = p.v_new[src];
            }
            const int64_t dst = (static_cast<int64_t>(b) * Lk + j) * per_pos + t;
            if (!in_bounds(dst, p.n_ws, &g_append_error, &g_append_where)) continue;
            p.wk[dst] = kv;
            p.wv[dst] = vv;
        }
    }
}

swa_status chunk_gather_launch(const swa_cache &c, const void *k_new, const void *v_new, int n,
                               int64_t pos0, int q_off, void *wk, void *wv, cudaStream_t stream) {
    GatherParams p{};
    p.ck = static_cast<const uint4 *>(c.k);
    p.cv = static_cast<const uint4 *>(c.v);
    p.k_new = static_cast<const uint4 *>(k_new);
    p.v_new = static_cast<const uint4 *>(v_new);
    p.wk = static_cast<uint4 *>(wk);
    p.wv = static_cast<uint4 *>(wv);
    p.pos0 = pos0;
    p.B = c.B;
    p.n = n;
    p.Hkv = c.Hkv;
    p.vpr = c.d / 8;
    p.vpr_log2 = p.vpr == 16 ? 4 : 3;
    p.cap = c.cap;
    p.w = c.w;
    p.s = c.s;
    p.q_off = q_off;
    const int Lk = q_off + n;
    p.n_cache = static_cast<long long>(c.B) * c.Hkv * c.cap * c.d / 8;
    p.n_new = static_cast<long long>(c.B) * n * c.Hkv * c.d / 8;
    p.n_ws = output_extent(static_cast<long long>(c.B) * Lk * c.Hkv * c.d) / 8;
    if (Lk == 0 || c.B == 0) return SWA_OK;
    const int per_pos = p.Hkv * p.vpr;
    const dim3 grid((per_pos + kAppendThreads - 1) / kAppendThreads,
                    static_cast<unsigned>(Lk < 65535 ? Lk : 65535),
                    static_cast<unsigned>(c.B < 65535 ? c.B : 65535));
    const cudaError_t e =
        launch_pdl(swa_chunk_gather_kernel, grid, dim3(kAppendThreads), 0, stream, p);
    return e == cudaSuccess ? SWA_OK : cuda_fail(e, "launch swa_chunk_gather_kernel");
}

int append_read_clear_error(cudaStream_t stream) {
    int v = 0;
    return read_clear_symbol(g_append_error, &v, stream) ? v : SWA_ERR_CUDA;
}

long long append_read_clear_where(cudaStream_t stream) {
    unsigned long long w = 0;
    return read_clear_symbol(g_append_where, &w, stream) ? where_index(w) : -2;
}

}  // namespace swa
