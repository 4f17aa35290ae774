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
// only the latest of them (p + (w-s) >= pos0 + n) is written, so the result is
// the same as appending one position at a time and no two threads write the
// same slot.  Pure copy: 16-byte vectors, one per thread-iteration,
// coalesced on both sides.
#include <cuda_runtime.h>

#include <cstdint>

#include "swa_internal.h"

namespace swa {

struct AppendParams {
    const uint4 *k_new;  // [B, n, Hkv, d] as 16-byte vectors
    const uint4 *v_new;
    uint4 *ck;           // [B, Hkv, cap, d]
    uint4 *cv;
    int64_t pos0;
    int B, n, Hkv, vpr, cap, w, s;  // vpr: 16-byte vectors per row (d / 8)
};

__global__ void __launch_bounds__(256) swa_append_kernel(const AppendParams p) {
    const int64_t total = static_cast<int64_t>(p.B) * p.n * p.Hkv * p.vpr;
    const int64_t last = p.pos0 + p.n;  // one past the last position written
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = idx / p.vpr;           // (b * n + j) * Hkv + h
        const int vec = static_cast<int>(idx - r * p.vpr);
        const int h = static_cast<int>(r % p.Hkv);
        const int64_t bj = r / p.Hkv;
        const int j = static_cast<int>(bj % p.n);
        const int b = static_cast<int>(bj / p.n);
        const int64_t pos = p.pos0 + j;
        int64_t slot;
        if (p.w < 0 || pos < p.s) {
            slot = pos;
        } else {
            const int64_t ring = p.w - p.s;
            if (pos + ring < last) continue;  // overwritten later in this same append
            slot = p.s + (pos - p.s) % ring;
        }
        const int64_t dst = ((static_cast<int64_t>(b) * p.Hkv + h) * p.cap + slot) * p.vpr + vec;
        p.ck[dst] = p.k_new[idx];
        p.cv[dst] = p.v_new[idx];
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
    p.cap = c.cap;
    p.w = c.w < 0 ? -1 : c.w;
    p.s = c.w < 0 ? 0 : c.s;
    const int64_t total = static_cast<int64_t>(p.B) * n * p.Hkv * p.vpr;
    const int sms = device_sm_count();
    int64_t blocks = (total + 255) / 256;
    const int64_t max_blocks = static_cast<int64_t>(sms > 0 ? sms : 148) * 8;
    if (blocks > max_blocks) blocks = max_blocks;
    swa_append_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

}  // namespace swa
