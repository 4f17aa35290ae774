// swa_hybrid.cu -- the linear-attention state of the hybrid window + linear
// mode: the tokens an append evicts from the fixed SWA(w,s) cache are folded
// into S += phi(k)^T v and z += phi(k), with the Hedgehog feature map
// phi(x) = (exp(x W), exp(-x W)) ("Sliding-window beats linear attention",
// paper summary page, sections "Prerequisites / Linear attention" and
// "Post-training linearisation and LoLCATs").  The decode that mixes the
// state with the window is the hybrid merge in swa_decode.cu.
//
// One CTA per (sequence, key/value head) owns its S [2 df, d] and z [2 df],
// so the update is a plain read-modify-write in a fixed order (no atomics):
// thread t holds feature t/2 and half of the d columns in registers while
// the evicted tokens stream through shared memory in batches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "swa_internal.h"
#include "swa_ptx.cuh"

namespace swa {

__device__ int g_hybrid_error;
__device__ unsigned long long g_hybrid_where;

namespace {

constexpr int kFoldTB = 8;  // evicted tokens per shared-memory batch

struct FoldParams {
    uint16_t *kc, *vc;        // cache [B, Hkv, cap, d] (written only through write_slot)
    const uint16_t *kn, *vn;  // appended tokens [B, n, Hkv, d]
    float *S, *z;             // state [B*Hkv, 2 df, d], [B*Hkv, 2 df]
    const float *W;           // [Hkv, d, df]
    int Hkv, cap, w, s, n;
    int64_t pos0, e_lo, e_hi;  // evicted positions e_lo .. e_hi
    // >= 0: a one-token append evicting one token; once it is read, the new
    // token is written to this slot (the evicted one's) by the same CTA
    int write_slot;
    long long n_cache, n_new, n_S, n_z;  // extents in elements (bounds-checked build)
};

template <int D, int DF, int DT>
__global__ void __launch_bounds__(4 * DF) swa_hybrid_fold_kernel(const FoldParams p) {
    constexpr int F = 2 * DF, NT = 4 * DF, HALF = D / 2;
    static_assert((D * DF / 4) % NT == 0 && (kFoldTB * D) % NT == 0, "whole loads per thread");
    __shared__ __align__(16) float sW[D * DF];
    __shared__ float sk[kFoldTB][D];
    __shared__ float sv[kFoldTB][D];
    __shared__ float sphi[kFoldTB][F];
    pdl_launch_dependents();
    pdl_wait();  // the cache and the state are the previous kernels'
    const int bh = blockIdx.x;
    const int b = bh / p.Hkv, kvh = bh - b * p.Hkv;
    const int tid = threadIdx.x;
    const int f = tid >> 1, half = tid & 1;
    // The state rows this thread updates, read first (their latency overlaps
    // the staging below), then W of this kv head into shared memory.
    const int64_t s0 = (static_cast<int64_t>(bh) * F + f) * D + half * HALF;
    const int64_t zi = static_cast<int64_t>(bh) * F + f;
    const bool s_ok = in_bounds(s0 + HALF - 1, p.n_S, &g_hybrid_error, &g_hybrid_where);
    const bool z_ok = half == 0 && in_bounds(zi, p.n_z, &g_hybrid_error, &g_hybrid_where);
    float *Srow = p.S + s0;
    float acc[HALF];
#pragma unroll
    for (int i = 0; i < HALF; ++i) acc[i] = s_ok ? Srow[i] : 0.f;
    float zacc = z_ok ? p.z[zi] : 0.f;
    const float4 *Wh4 = reinterpret_cast<const float4 *>(p.W + static_cast<int64_t>(kvh) * D * DF);
#pragma unroll
    for (int i = 0; i < D * DF / 4 / NT; ++i)
        reinterpret_cast<float4 *>(sW)[tid + i * NT] = __ldg(Wh4 + tid + i * NT);
    for (int64_t e0 = p.e_lo; e0 <= p.e_hi; e0 += kFoldTB) {
        if (e0 != p.e_lo) __syncthreads();  // the previous batch is consumed
#pragma unroll
        for (int it = 0; it < kFoldTB * D / NT; ++it) {
            const int idx = tid + it * NT;
            const int t = idx / D, c = idx - t * D;
            const int64_t e = e0 + t;
            float kx = 0.f, vx = 0.f;
            if (e <= p.e_hi) {
                int64_t off;
                if (e < p.pos0) {  // still in the ring: its slot
                    const int64_t slot = e < p.s ? e : p.s + (e - p.s) % (p.w - p.s);
                    off = (static_cast<int64_t>(bh) * p.cap + slot) * D + c;
                    if (in_bounds(off, p.n_cache, &g_hybrid_error, &g_hybrid_where)) {
                        kx = widen16<DT>(p.kc[off]);
                        vx = widen16<DT>(p.vc[off]);
                    }
                } else {  // appended by this call and evicted by it too
                    off = ((static_cast<int64_t>(b) * p.n + (e - p.pos0)) * p.Hkv + kvh) * D + c;
                    if (in_bounds(off, p.n_new, &g_hybrid_error, &g_hybrid_where)) {
                        kx = widen16<DT>(p.kn[off]);
                        vx = widen16<DT>(p.vn[off]);
                    }
                }
            }
            sk[t][c] = kx;
            sv[t][c] = vx;
        }
        __syncthreads();  // the batch (and, the first time, W) is in shared memory
        if (p.write_slot >= 0) {  // the evicted token is in shared memory: overwrite its slot
            const int64_t dst = (static_cast<int64_t>(bh) * p.cap + p.write_slot) * D;
            const int64_t src = (static_cast<int64_t>(b) * p.Hkv + kvh) * D;
            for (int c = tid; c < D; c += NT) {
                if (in_bounds(dst + c, p.n_cache, &g_hybrid_error, &g_hybrid_where) &&
                    in_bounds(src + c, p.n_new, &g_hybrid_error, &g_hybrid_where)) {
                    p.kc[dst + c] = p.kn[src + c];
                    p.vc[dst + c] = p.vn[src + c];
                }
            }
        }
        for (int idx = tid; idx < kFoldTB * DF; idx += NT) {
            const int t = idx / DF, j = idx - t * DF;
            float fx = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) fx = fmaf(sk[t][c], sW[c * DF + j], fx);
            const bool live = e0 + t <= p.e_hi;
            sphi[t][j] = live ? expf(fx) : 0.f;
            sphi[t][DF + j] = live ? expf(-fx) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < kFoldTB; ++t) {
            const float ph = sphi[t][f];
#pragma unroll
            for (int i = 0; i < HALF; ++i) acc[i] = fmaf(ph, sv[t][half * HALF + i], acc[i]);
            zacc += ph;
        }
    }
    if (s_ok) {
#pragma unroll
        for (int i = 0; i < HALF; ++i) Srow[i] = acc[i];
    }
    if (z_ok) p.z[zi] = zacc;
}

template <int D, int DF, int DT>
swa_status launch_fold(const FoldParams &fp, int grid, cudaStream_t stream) {
    const cudaError_t e = launch_pdl(swa_hybrid_fold_kernel<D, DF, DT>, dim3(grid), dim3(4 * DF), 0,
                                     stream, fp);
    return e == cudaSuccess ? SWA_OK : cuda_fail(e, "launch swa_hybrid_fold_kernel");
}

template <int DT>
swa_status launch_fold_dt(const FoldParams &fp, int grid, int d, int df, cudaStream_t stream) {
    if (d == 128)
        return df == 32 ? launch_fold<128, 32, DT>(fp, grid, stream)
                        : launch_fold<128, 64, DT>(fp, grid, stream);
    return df == 32 ? launch_fold<64, 32, DT>(fp, grid, stream)
                    : launch_fold<64, 64, DT>(fp, grid, stream);
}

}  // namespace

swa_status hybrid_fold_launch(const swa_cache &c, const swa_linear_state &lin, const void *k_new,
                              const void *v_new, int n, int64_t pos0, cudaStream_t stream,
                              bool *appended) {
    *appended = false;
    if (c.w == SWA_W_INF || c.B == 0 || n == 0) return SWA_OK;  // nothing is evicted
    // The cache holds positions up to pos0-1: its oldest ring entry is
    // pos0-(w-s) (or the first non-sink position); appending up to
    // pos0+n-1 evicts every non-sink position up to pos0+n-1-(w-s).
    FoldParams fp{};
    fp.e_lo = pos0 - (c.w - c.s) > c.s ? pos0 - (c.w - c.s) : c.s;
    fp.e_hi = pos0 + n - 1 - (c.w - c.s);
    if (fp.e_hi < fp.e_lo) return SWA_OK;
    fp.kc = static_cast<uint16_t *>(c.k);
    fp.vc = static_cast<uint16_t *>(c.v);
    fp.kn = static_cast<const uint16_t *>(k_new);
    fp.vn = static_cast<const uint16_t *>(v_new);
    fp.S = lin.S;
    fp.z = lin.z;
    fp.W = lin.W;
    fp.Hkv = c.Hkv;
    fp.cap = c.cap;
    fp.w = c.w;
    fp.s = c.s;
    fp.n = n;
    fp.pos0 = pos0;
    fp.n_cache = output_extent(static_cast<long long>(c.B) * c.Hkv * c.cap * c.d);
    fp.n_new = static_cast<long long>(c.B) * n * c.Hkv * c.d;
    fp.n_S = output_extent(static_cast<long long>(c.B) * c.Hkv * 2 * lin.df * c.d);
    fp.n_z = output_extent(static_cast<long long>(c.B) * c.Hkv * 2 * lin.df);
    // a decode step (one token, evicting one): the fold writes the new token
    fp.write_slot = -1;
    if (n == 1 && fp.e_lo == fp.e_hi) {
        fp.write_slot = static_cast<int>(pos0 < c.s ? pos0 : c.s + (pos0 - c.s) % (c.w - c.s));
        *appended = true;
    }
    const int grid = c.B * c.Hkv;
    return c.dtype == SWA_F16 ? launch_fold_dt<kF16>(fp, grid, c.d, lin.df, stream)
                              : launch_fold_dt<kBf16>(fp, grid, c.d, lin.df, stream);
}

int hybrid_read_clear_error(cudaStream_t stream) {
    int v = 0;
    return read_clear_symbol(g_hybrid_error, &v, stream) ? v : SWA_ERR_CUDA;
}

long long hybrid_read_clear_where(cudaStream_t stream) {
    unsigned long long w = 0;
    return read_clear_symbol(g_hybrid_where, &w, stream) ? where_index(w) : -2;
}

}  // namespace swa
