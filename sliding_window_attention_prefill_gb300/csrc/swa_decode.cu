// swa_decode.cu -- one new token per sequence attends to the fixed SWA cache.
//
// Operation: o = softmax over the filled cache slots of c q.k_slot, applied
// to v_slot.  The filled slots of an SWA(w,s) cache hold exactly the attended
// set A(pos) (first s tokens + latest w-s), in ring order rather than position
// order; a softmax over a set does not depend on the order.  Window equation
// and notation: "Sliding-window beats linear attention" (paper summary page),
// "Prerequisites / Sliding-window attention SWA(w, s)".  The cache stops
// growing at w tokens: news page "No post-training, just 4 more tokens",
// section "Research method".
//
// The path is bound by HBM bandwidth (each K/V byte is used by the G query
// heads of its group and nothing else), so it runs on the CUDA cores:
//   grid (split, kv head, sequence); each CTA streams its share of the slots
//   in 32-slot chunks.  One producer warp moves chunks of K and V into shared
//   memory with 1-D bulk copies (TMA engine, 4 stages, mbarrier completion);
//   four consumer warps take 8 slots of each chunk.  Scores: 8 lanes per slot
//   row, 16-byte shared loads, fp32 dot products for all G heads, then a
//   reduce-scatter over the 8 lanes (each lane ends with whole dot products).
//   Each warp keeps an online softmax (running max, sum, fp32 accumulators);
//   warps are merged through shared memory at the end.  With several splits
//   per (sequence, kv head) the CTAs write fp32 partials (max, sum, weighted
//   values) and a second kernel merges them: m = max m_j,
//   l = sum l_j 2^(m_j - m), o = sum acc_j 2^(m_j - m) / l.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "swa_internal.h"
#include "swa_ptx.cuh"

namespace swa {

__device__ int g_decode_error;

constexpr int kDecCH = 32;              // slots per chunk
constexpr int kDecStages = 4;           // chunk ring depth
constexpr int kDecWarps = 4;            // consumer warps
constexpr int kDecThreads = 32 * (kDecWarps + 1);

struct DecodeParams {
    const uint16_t *q;   // [B, Hq, D] bf16
    const uint16_t *ck;  // [B, Hkv, cap, D]
    const uint16_t *cv;
    const int32_t *pos;  // [B]
    uint16_t *o;         // [B, Hq, D]
    float *ws_acc;       // [B*Hq, splits, D]
    float *ws_ml;        // [B*Hq, splits, 2]
    int B, Hq, Hkv, cap, w, splits;
    float scale_log2;
};

template <int D, int G>
struct DecSmem {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kChunkBytes = kDecCH * kRowBytes;
    static constexpr int kK = 0;
    static constexpr int kV = kK + kDecStages * kChunkBytes;
    static constexpr int kScore = kV + kDecStages * kChunkBytes;      // [warp][8*G] f32
    static constexpr int kProb = kScore + kDecWarps * 8 * G * 4;       // [warp][8*G] f32
    static constexpr int kAcc = kProb + kDecWarps * 8 * G * 4;         // [warp][G][D] f32
    static constexpr int kML = kAcc + kDecWarps * G * D * 4;           // [warp][G][2] f32
    static constexpr int kBar = kML + kDecWarps * G * 2 * 4;           // full[st], empty[st]
    static constexpr int kAbort = kBar + 2 * kDecStages * 8;
    static constexpr int kBytes = kAbort + 16;
};

// Slot range of one split: [begin, end); `used` = number of non-empty splits.
__device__ __forceinline__ void split_range(int n_valid, int splits, int split, int &begin,
                                            int &end, int &used) {
    const int n_chunks = (n_valid + kDecCH - 1) / kDecCH;
    const int per = (n_chunks + splits - 1) / splits;
    used = (n_chunks + per - 1) / per;
    begin = split * per * kDecCH;
    end = min(begin + per * kDecCH, n_valid);
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    f[0] = bf16lo_to_f32(u.x);
    f[1] = bf16hi_to_f32(u.x);
    f[2] = bf16lo_to_f32(u.y);
    f[3] = bf16hi_to_f32(u.y);
    f[4] = bf16lo_to_f32(u.z);
    f[5] = bf16hi_to_f32(u.z);
    f[6] = bf16lo_to_f32(u.w);
    f[7] = bf16hi_to_f32(u.w);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads) swa_decode_kernel(const DecodeParams p) {
    using SL = DecSmem<D, G>;
    constexpr int SEG = D / 64;        // 16-byte pieces per lane per row
    constexpr int EPL = SEG * 8;       // elements per lane per row
    constexpr int NV = 2 * G;          // dot products per lane before the reduction
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t sbase = smem_u32(sm);
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SL::kAbort);
    auto full = [&](int st) { return sbase + SL::kBar + 8u * st; };
    auto empty = [&](int st) { return sbase + SL::kBar + 8u * (kDecStages + st); };

    const int pos = p.pos[b];
    if (pos < 0 || (p.w < 0 && pos >= p.cap)) {
        if (threadIdx.x == 0 && split == 0 && kvh == 0) atomicCAS(&g_decode_error, 0, kErrBounds);
        return;
    }
    const int cap_eff = p.w < 0 ? p.cap : p.w;
    const int n_valid = min(pos + 1, cap_eff);
    int begin, end, used;
    split_range(n_valid, p.splits, split, begin, end, used);
    if (begin >= end) return;  // uniform over the block
    const int n_chunks = (end - begin + kDecCH - 1) / kDecCH;

    if (threadIdx.x == 0) {
        for (int st = 0; st < kDecStages; ++st) {
            mbar_init(full(st), 1);
            mbar_init(empty(st), kDecWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int64_t row_base = (static_cast<int64_t>(b) * p.Hkv + kvh) * p.cap;  // slot 0

    if (warp == kDecWarps) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < n_chunks; ++c) {
                const int st = c % kDecStages;
                if (!mbar_wait(empty(st), ((c / kDecStages) & 1) ^ 1, &g_decode_error, abort_flag))
                    break;
                const int row0 = begin + c * kDecCH;
                const int rows = min(kDecCH, end - row0);
                const uint32_t bytes = static_cast<uint32_t>(rows) * SL::kRowBytes;
                mbar_arrive_expect_tx(full(st), 2 * bytes);
                bulk_load_1d(sbase + SL::kK + st * SL::kChunkBytes, p.ck + (row_base + row0) * D,
                             bytes, full(st));
                bulk_load_1d(sbase + SL::kV + st * SL::kChunkBytes, p.cv + (row_base + row0) * D,
                             bytes, full(st));
                issued = c + 1;
            }
            int no_abort = 0;  // drain the copies this thread started
            for (int i = 0; i < kDecStages && i < issued; ++i) {
                const int c = issued - 1 - i;
                mbar_wait(full(c % kDecStages), (c / kDecStages) & 1, &g_decode_error, &no_abort);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int rg = lane >> 3;  // row group: slot row within a 4-row step
    const int gi = lane & 7;   // lane within the row group
    float qf[G][EPL];          // q * log2(e)/sqrt(d), this lane's elements
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint16_t *qrow = p.q + (static_cast<int64_t>(b) * p.Hq + kvh * G + h) * D;
#pragma unroll
        for (int sg = 0; sg < SEG; ++sg) {
            const uint4 u = *reinterpret_cast<const uint4 *>(qrow + sg * 64 + gi * 8);
            float f[8];
            unpack8(u, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[h][sg * 8 + e] = f[e] * p.scale_log2;
        }
    }
    float acc[G][EPL];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[h][e] = 0.f;
    // per-head running max / sum, held by the lanes whose (lane % G) is the head
    float m_h = -INFINITY, l_h = 0.f;
    float *score = reinterpret_cast<float *>(sm + SL::kScore) + warp * 8 * G;
    float *prob = reinterpret_cast<float *>(sm + SL::kProb) + warp * 8 * G;
    constexpr int KC = (8 * G + 31) / 32;  // score entries per lane in the softmax step

    for (int c = 0; c < n_chunks; ++c) {
        const int st = c % kDecStages;
        mbar_wait(full(st), (c / kDecStages) & 1, &g_decode_error, abort_flag);
        const int row0 = begin + c * kDecCH;
        const int rows = min(kDecCH, end - row0);
        const int wrow0 = warp * 8;
        if (wrow0 < rows) {
            const uint32_t kst = sbase + SL::kK + st * SL::kChunkBytes;
            const uint32_t vst = sbase + SL::kV + st * SL::kChunkBytes;
            // ---- scores: lane (rg, gi) covers 8 elements per segment of rows
            //      wrow0 + sub*4 + rg, sub = 0, 1
            float dots[NV];
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
                const int r = wrow0 + sub * 4 + rg;
                float kf[EPL];
#pragma unroll
                for (int sg = 0; sg < SEG; ++sg) {
                    float f[8];
                    unpack8(lds128(kst + r * SL::kRowBytes + sg * 128 + gi * 16), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) kf[sg * 8 + e] = f[e];
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) a = fmaf(qf[h][e], kf[e], a);
                    dots[sub * G + h] = a;
                }
            }
            // ---- reduce over the 8 lanes of the row group (scatter while it
            //      halves the values, plain butterfly after that)
            int n = NV, idx0 = 0;
#pragma unroll
            for (int step = 4; step >= 1; step >>= 1) {
                if (n >= 2) {
                    const int half = n / 2;
                    const bool hi = (gi & step) != 0;
#pragma unroll
                    for (int i = 0; i < NV / 2; ++i) {
                        if (i < half) {
                            const float send = hi ? dots[i] : dots[half + i];
                            const float keep = hi ? dots[half + i] : dots[i];
                            dots[i] = keep + __shfl_xor_sync(0xffffffffu, send, step);
                        }
                    }
                    if (hi) idx0 += half;
                    n = half;
                } else {
                    dots[0] += __shfl_xor_sync(0xffffffffu, dots[0], step);
                }
            }
            // lane holds combos idx0 .. idx0+n-1, combo = sub*G + h
#pragma unroll
            for (int i = 0; i < (NV >= 8 ? NV / 8 : 1); ++i) {
                const int ci = idx0 + i;
                const int sub = ci / G, h = ci - sub * G;
                const int rw = sub * 4 + rg;  // row within this warp's 8
                score[rw * G + h] = (wrow0 + rw < rows) ? dots[i] : -INFINITY;
            }
            __syncwarp();
            // ---- online softmax per head (lane's head = lane % G)
            float sv[KC];
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < KC; ++k) {
                const int cj = lane + 32 * k;
                sv[k] = cj < 8 * G ? score[cj] : -INFINITY;
                mx = fmaxf(mx, sv[k]);
            }
#pragma unroll
            for (int msk = G; msk < 32; msk <<= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
            const float m_new = fmaxf(m_h, mx);
            const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(m_h - m_new);
            float psum = 0.f;
#pragma unroll
            for (int k = 0; k < KC; ++k) {
                const int cj = lane + 32 * k;
                const float pv = (sv[k] == -INFINITY) ? 0.f : ex2_approx(sv[k] - m_new);
                psum += pv;
                if (cj < 8 * G) prob[cj] = pv;
            }
#pragma unroll
            for (int msk = G; msk < 32; msk <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, msk);
            l_h = l_h * alpha + psum;
            m_h = m_new;
            __syncwarp();
            // ---- values: rescale, then accumulate this lane's rows
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float ah = __shfl_sync(0xffffffffu, alpha, h);
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[h][e] *= ah;
            }
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
                const int rw = sub * 4 + rg;
                if (wrow0 + rw < rows) {
                    float vf[EPL];
#pragma unroll
                    for (int sg = 0; sg < SEG; ++sg) {
                        float f[8];
                        unpack8(lds128(vst + (wrow0 + rw) * SL::kRowBytes + sg * 128 + gi * 16), f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) vf[sg * 8 + e] = f[e];
                    }
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float ph = prob[rw * G + h];
#pragma unroll
                        for (int e = 0; e < EPL; ++e) acc[h][e] = fmaf(ph, vf[e], acc[h][e]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(st));
    }

    // -------------------------------------------------------------------- merge
    // over the four row groups of the warp (lanes with equal gi)
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], 8);
            acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], 16);
        }
    float *wacc = reinterpret_cast<float *>(sm + SL::kAcc);
    float *wml = reinterpret_cast<float *>(sm + SL::kML);
    if (rg == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int sg = 0; sg < SEG; ++sg)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    wacc[(warp * G + h) * D + sg * 64 + gi * 8 + e] = acc[h][sg * 8 + e];
    }
    if (lane < G) {
        wml[(warp * G + lane) * 2 + 0] = m_h;
        wml[(warp * G + lane) * 2 + 1] = l_h;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
    // over the warps; thread t handles outputs t, t+128, ...
    for (int idx = threadIdx.x; idx < G * D; idx += kDecWarps * 32) {
        const int h = idx / D, e = idx - h * D;
        float m = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) m = fmaxf(m, wml[(w * G + h) * 2]);
        float l = 0.f, a = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
            const float wm = wml[(w * G + h) * 2];
            const float f = (wm == -INFINITY) ? 0.f : ex2_approx(wm - m);
            l = fmaf(wml[(w * G + h) * 2 + 1], f, l);
            a = fmaf(wacc[(w * G + h) * D + e], f, a);
        }
        const int64_t orow = static_cast<int64_t>(b) * p.Hq + kvh * G + h;
        if (p.splits == 1) {
            const float ov = l > 0.f ? a / l : 0.f;
            p.o[orow * D + e] = __bfloat16_as_ushort(__float2bfloat16_rn(ov));
        } else {
            p.ws_acc[(orow * p.splits + split) * D + e] = a;
            if (e == 0) {
                p.ws_ml[(orow * p.splits + split) * 2 + 0] = m;
                p.ws_ml[(orow * p.splits + split) * 2 + 1] = l;
            }
        }
    }
}

// One warp per (sequence, query head): merge the non-empty splits.
template <int D>
__global__ void __launch_bounds__(128) swa_decode_merge_kernel(const DecodeParams p) {
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.B * p.Hq) return;
    const int b = row / p.Hq;
    const int pos = p.pos[b];
    if (pos < 0 || (p.w < 0 && pos >= p.cap)) return;  // recorded by the split kernel
    const int cap_eff = p.w < 0 ? p.cap : p.w;
    const int n_valid = min(pos + 1, cap_eff);
    int begin, end, used;
    split_range(n_valid, p.splits, 0, begin, end, used);
    constexpr int E = D / 32;
    float m = -INFINITY;
    for (int j = 0; j < used; ++j)
        m = fmaxf(m, p.ws_ml[(static_cast<int64_t>(row) * p.splits + j) * 2]);
    float l = 0.f, a[E];
#pragma unroll
    for (int e = 0; e < E; ++e) a[e] = 0.f;
    for (int j = 0; j < used; ++j) {
        const int64_t base = static_cast<int64_t>(row) * p.splits + j;
        const float mj = p.ws_ml[base * 2];
        const float f = (mj == -INFINITY) ? 0.f : ex2_approx(mj - m);
        l = fmaf(p.ws_ml[base * 2 + 1], f, l);
#pragma unroll
        for (int e = 0; e < E; ++e) a[e] = fmaf(p.ws_acc[base * D + lane * E + e], f, a[e]);
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e)
        p.o[static_cast<int64_t>(row) * D + lane * E + e] =
            __bfloat16_as_ushort(__float2bfloat16_rn(a[e] * inv));
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
DecodePlan decode_plan(int B, int Hq, int Hkv, int d, int cap, int w, int sm_count) {
    DecodePlan plan{1, 0};
    const int cap_eff = w < 0 ? cap : w;
    const int chunks = (cap_eff + kDecCH - 1) / kDecCH;
    const int max_splits = (chunks + 3) / 4;  // at least 4 chunks (128 slots) per split
    const long long pairs = static_cast<long long>(B) * Hkv;
    const long long target = 6LL * (sm_count > 0 ? sm_count : 148);  // ~2 waves of 3 CTAs/SM
    if (pairs > 0 && pairs < target) {
        long long s = (target + pairs - 1) / pairs;
        if (s > max_splits) s = max_splits;
        if (s < 1) s = 1;
        plan.splits = static_cast<int>(s);
    }
    if (plan.splits > 1)
        plan.workspace = static_cast<size_t>(B) * Hq * plan.splits * (d + 2) * sizeof(float);
    return plan;
}

namespace {

template <int D, int G>
swa_status launch_decode(const DecodeParams &p, cudaStream_t stream) {
    using SL = DecSmem<D, G>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    static bool configured[64] = {};
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(swa_decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SL::kBytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode)");
        configured[dev] = true;
    }
    dim3 grid(p.splits, p.Hkv, p.B);
    swa_decode_kernel<D, G><<<grid, kDecThreads, SL::kBytes, stream>>>(p);
    e = cudaPeekAtLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch swa_decode_kernel");
    if (p.splits > 1) {
        const int rows = p.B * p.Hq;
        swa_decode_merge_kernel<D><<<(rows + 3) / 4, 128, 0, stream>>>(p);
        e = cudaPeekAtLastError();
        if (e != cudaSuccess) return cuda_fail(e, "launch swa_decode_merge_kernel");
    }
    return SWA_OK;
}

}  // namespace

swa_status decode_launch(const void *q, const swa_cache &c, const int32_t *pos, int Hq, void *o,
                         void *workspace, const DecodePlan &plan, cudaStream_t stream) {
    if (c.B == 0) return SWA_OK;
    DecodeParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.ck = static_cast<const uint16_t *>(c.k);
    p.cv = static_cast<const uint16_t *>(c.v);
    p.pos = pos;
    p.o = static_cast<uint16_t *>(o);
    p.B = c.B;
    p.Hq = Hq;
    p.Hkv = c.Hkv;
    p.cap = c.cap;
    p.w = c.w < 0 ? -1 : c.w;
    p.splits = plan.splits;
    if (plan.splits > 1) {
        p.ws_acc = static_cast<float *>(workspace);
        p.ws_ml = p.ws_acc + static_cast<size_t>(c.B) * Hq * plan.splits * c.d;
    }
    p.scale_log2 = 1.4426950408889634f / std::sqrt(static_cast<float>(c.d));
    const int G = Hq / c.Hkv;
    if (c.d == 128) {
        switch (G) {
            case 1: return launch_decode<128, 1>(p, stream);
            case 2: return launch_decode<128, 2>(p, stream);
            case 4: return launch_decode<128, 4>(p, stream);
            default: return SWA_ERR_UNSUPPORTED;
        }
    }
    switch (G) {
        case 1: return launch_decode<64, 1>(p, stream);
        case 2: return launch_decode<64, 2>(p, stream);
        case 4: return launch_decode<64, 4>(p, stream);
        case 8: return launch_decode<64, 8>(p, stream);
        default: return SWA_ERR_UNSUPPORTED;
    }
}

int decode_read_clear_error(cudaStream_t stream) {
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_decode_error, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess)
        return SWA_ERR_CUDA;
    if (cudaMemcpyToSymbolAsync(g_decode_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                stream) != cudaSuccess)
        return SWA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SWA_ERR_CUDA;
    return v;
}

// ---------------------------------------------------------------------------
// decode without a caller-provided workspace (swa_decode_noalloc)
// ---------------------------------------------------------------------------
// Split partials for callers that cannot allocate: a fixed device array owned
// by the library.  Host code must not use the symbol itself as an address;
// noalloc_scratch() looks the device address up once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SWA_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of g_noalloc_scratch on the current device (looked up once
// per device, with that device current); nullptr if the lookup fails.
void *noalloc_scratch() {
    static void *addr[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

}  // namespace swa

extern "C" swa_status swa_decode_noalloc(const void *q, const swa_cache *cache, const int32_t *pos,
                                         int Hq, int w, int s, void *o, swa_stream_t stream) {
    if (cache == nullptr) return SWA_ERR_INVALID_ARG;
    const int sms = swa::device_sm_count();
    if (sms <= 0) return SWA_ERR_CUDA;
    const swa::DecodePlan plan =
        swa::decode_plan(cache->B, Hq, cache->Hkv, cache->d, cache->cap, cache->w, sms);
    if (plan.workspace > SWA_NOALLOC_SCRATCH_BYTES) return SWA_ERR_WORKSPACE;
    void *ws = nullptr;
    if (plan.workspace > 0) {
        ws = swa::noalloc_scratch();
        if (ws == nullptr) return SWA_ERR_CUDA;
    }
    const swa_status st = swa_check_decode(q, cache, pos, Hq, w, s, o, ws,
                                           SWA_NOALLOC_SCRATCH_BYTES, plan.workspace);
    if (st != SWA_OK || cache->B == 0) return st;
    return swa::decode_launch(q, *cache, pos, Hq, o, ws, plan, reinterpret_cast<cudaStream_t>(stream));
}
