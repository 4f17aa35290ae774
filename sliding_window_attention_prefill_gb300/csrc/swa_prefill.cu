// swa_prefill.cu -- banded SWA(w,s) prefill on sm_103a: TMA-staged tiles,
// tcgen05 MMAs with fp32 accumulators in tensor memory, online softmax.
//
// Operation (o_t = softmax over A(t) of c q_t.k_i, applied to v_i): the window
// equation and SWA(w,s) notation of "Sliding-window beats linear attention"
// (paper summary page), section "Prerequisites / Sliding-window attention
// SWA(w, s)"; w = infinity is the full causal "FA" case of the same page.
//
// Work decomposition.  A work unit is (sequence b, key/value head kvh, query
// tile).  Its 128 MMA rows pack the G = Hq/Hkv query heads that share kvh for
// P = 128/G consecutive positions: row r is position t0 + r/G, head
// kvh*G + r%G, which is exactly a box of the [B, L, Hq, d] query tensor, so
// one TMA box loads it and one TMA box stores the output.  The unit needs the
// sink keys [0, s) and the band [lo, t1] with lo = max(s, t0-(w-s)+1): the
// key columns are laid out as [s_pad sink rows | band ...] in 128-column key
// tiles, the sink block (s rounded up to 8 rows) sharing the first tile.
//
// Roles (192 threads, one persistent CTA per SM):
//   warp 0      TMA producer: Q (double-buffered), K/V key tiles (NS stages)
//   warp 1      tcgen05 issuer; owns the 512-column TMEM allocation
//               S0 | S1 (double-buffered scores) | O (output accumulator)
//   warps 2..5  softmax + epilogue, one thread per MMA row (TMEM lane)
// Per key tile g the MMA warp issues S_g = Q K_g^T, then O += P_{g-1} V_{g-1},
// so the scores of the next tile are computed while the softmax of the
// current one runs.  P is written to shared memory in the 128-byte-swizzled
// K-major layout the MMA reads.  The running max is only raised when it grows
// by more than 2^8 (exact: numerator and denominator share the same stale
// max), so the O rescale through TMEM is rare.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "swa_internal.h"
#include "swa_ptx.cuh"

namespace swa {

__device__ int g_prefill_error;

struct PrefillMaps {
    CUtensorMap q, o;                 // box {64, G, P, 1} over [B, L, Hq, d]
    CUtensorMap k_band, v_band;       // box {64, 1, 128, 1} over [B, L, Hkv, d]
    CUtensorMap k_sink, v_sink;       // box {64, 1, s_pad, 1}
    CUtensorMap k_band0, v_band0;     // box {64, 1, 128 - s_pad, 1}
};

struct PrefillParams {
    int B, L, Hq, Hkv, G, P;  // P: positions per query tile (128 / G)
    int w, s;                 // w < 0: infinite window (s is then 0)
    int s_pad;                // sink rows loaded: s rounded up to 8 (0 if s == 0)
    int n_qtiles, n_units;
    float scale_log2;         // log2(e) / sqrt(d)
    float scale;              // 1 / sqrt(d)
    float *lse;               // optional [B, Hq, L]
};

struct Unit {
    int b, kvh, t0, t1, lo, n_cols, n_tiles;
};

// Geometry of work unit u.  Units run heaviest query tiles first (only
// matters for the infinite window, where cost grows with the position).
__device__ __forceinline__ Unit unit_geom(int u, const PrefillParams &p) {
    const int bh = p.B * p.Hkv;
    const int qt_rev = u / bh;
    const int r = u - qt_rev * bh;
    Unit x;
    x.b = r / p.Hkv;
    x.kvh = r - x.b * p.Hkv;
    const int qt = p.n_qtiles - 1 - qt_rev;
    x.t0 = qt * p.P;
    x.t1 = min(x.t0 + p.P, p.L) - 1;
    x.lo = p.w < 0 ? 0 : max(p.s, x.t0 - (p.w - p.s) + 1);
    const int nb = max(0, x.t1 - x.lo + 1);
    x.n_cols = p.s_pad + nb;
    x.n_tiles = (x.n_cols + 127) / 128;
    return x;
}

// Key columns of tile j, rounded up to the MMA's N granularity of 16.
__device__ __forceinline__ int tile_width(const Unit &x, int j) {
    const int n = min(128, x.n_cols - 128 * j);
    return (n + 15) & ~15;
}

template <int D, int NS>
struct PrefillSmem {
    static constexpr int kRegion = 128 * 128;           // one 64-column slab of 128 rows
    static constexpr int kQBytes = 128 * D * 2;         // Q / K / V tile bytes
    static constexpr int kQ = 0;                        // 2 Q buffers
    static constexpr int kK = kQ + 2 * kQBytes;         // NS K stages
    static constexpr int kV = kK + NS * kQBytes;        // NS V stages
    static constexpr int kP = kV + NS * kQBytes;        // P (2 slabs), also O staging
    static constexpr int kBar = kP + 2 * kRegion;       // mbarriers
    // barrier slots (8 bytes each)
    static constexpr int kQFull = 0, kQEmpty = 2, kKFull = 4, kVFull = 4 + NS,
                         kKVEmpty = 4 + 2 * NS, kSFull = 4 + 3 * NS, kSEmpty = 6 + 3 * NS,
                         kPFull = 8 + 3 * NS, kPVDone = 9 + 3 * NS, kNumBars = 10 + 3 * NS;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    static constexpr int kAbort = kTmemSlot + 8;
    static constexpr int kBytes = kAbort + 8;
    static constexpr int kAlloc = kBytes + 1024;        // room to align the base to 1024
};

constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;

template <int D, int NS>
__global__ void __launch_bounds__(kThreads, 1)
    swa_prefill_kernel(const __grid_constant__ PrefillMaps maps, const PrefillParams p) {
    using SL = PrefillSmem<D, NS>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + SL::kAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + SL::kTmemSlot);
    auto bar = [&](int i) { return base + SL::kBar + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < SL::kNumBars; ++i) {
            uint32_t cnt = 1;
            if (i == SL::kSEmpty || i == SL::kSEmpty + 1 || i == SL::kPFull) cnt = 4;
            mbar_init(bar(i), cnt);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(base + SL::kTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&maps.q);
            tma_prefetch_desc(&maps.k_band);
            tma_prefetch_desc(&maps.v_band);
            constexpr uint32_t kTileBytes = SL::kQBytes;
            uint32_t g = 0, uc = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++uc) {
                const Unit x = unit_geom(u, p);
                const uint32_t qb = uc & 1;
                ok = mbar_wait(bar(SL::kQEmpty + qb), ((uc >> 1) & 1) ^ 1, &g_prefill_error,
                               abort_flag);
                if (!ok) break;
                const uint32_t qdst = base + SL::kQ + qb * SL::kQBytes;
                mbar_arrive_expect_tx(bar(SL::kQFull + qb), kTileBytes);
#pragma unroll
                for (int db = 0; db < D / 64; ++db)
                    tma_load_4d(qdst + db * SL::kRegion, &maps.q, bar(SL::kQFull + qb), db * 64,
                                x.kvh * p.G, x.t0, x.b);
                for (int j = 0; j < x.n_tiles; ++j, ++g) {
                    const uint32_t st = g % NS;
                    ok = mbar_wait(bar(SL::kKVEmpty + st), ((g / NS) & 1) ^ 1, &g_prefill_error,
                                   abort_flag);
                    if (!ok) break;
                    const uint32_t kdst = base + SL::kK + st * SL::kQBytes;
                    const uint32_t vdst = base + SL::kV + st * SL::kQBytes;
                    const int key0 = x.lo + 128 * j - p.s_pad;  // key of column 0 (band)
                    mbar_arrive_expect_tx(bar(SL::kKFull + st), kTileBytes);
                    mbar_arrive_expect_tx(bar(SL::kVFull + st), kTileBytes);
#pragma unroll
                    for (int db = 0; db < D / 64; ++db) {
                        const uint32_t ko = kdst + db * SL::kRegion, vo = vdst + db * SL::kRegion;
                        if (j == 0 && p.s_pad > 0) {
                            const uint32_t off = p.s_pad * 128;
                            tma_load_4d(ko, &maps.k_sink, bar(SL::kKFull + st), db * 64, x.kvh, 0, x.b);
                            tma_load_4d(ko + off, &maps.k_band0, bar(SL::kKFull + st), db * 64,
                                        x.kvh, x.lo, x.b);
                            tma_load_4d(vo, &maps.v_sink, bar(SL::kVFull + st), db * 64, x.kvh, 0, x.b);
                            tma_load_4d(vo + off, &maps.v_band0, bar(SL::kVFull + st), db * 64,
                                        x.kvh, x.lo, x.b);
                        } else {
                            tma_load_4d(ko, &maps.k_band, bar(SL::kKFull + st), db * 64, x.kvh,
                                        key0, x.b);
                            tma_load_4d(vo, &maps.v_band, bar(SL::kVFull + st), db * 64, x.kvh,
                                        key0, x.b);
                        }
                    }
                }
            }
            // Drain: every copy this thread started has landed before exit.
            // (Bounded waits that ignore the abort flag; in the normal path the
            // consumers already saw these phases complete.)
            int no_abort = 0;
            for (uint32_t i = 0; i < NS && i < g; ++i) {
                const uint32_t gl = g - 1 - i;  // the last fill of stage gl % NS
                const uint32_t st = gl % NS, par = (gl / NS) & 1;
                mbar_wait(bar(SL::kKFull + st), par, &g_prefill_error, &no_abort);
                mbar_wait(bar(SL::kVFull + st), par, &g_prefill_error, &no_abort);
            }
            for (uint32_t i = 0; i < 2 && i < uc; ++i) {
                const uint32_t ul = uc - 1 - i;
                mbar_wait(bar(SL::kQFull + (ul & 1)), (ul >> 1) & 1, &g_prefill_error, &no_abort);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16_f32(128, 0, false);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, true);
            uint32_t g = 0, uc = 0;
            bool ok = true;
            bool have_prev = false;
            uint32_t prev_g = 0;
            int prev_n = 0;
            bool prev_first = false;
            uint32_t last_commit_g = 0;
            bool any_commit = false;

            auto issue_pv = [&](uint32_t pg, int pn, bool first) -> bool {
                const uint32_t st = pg % NS;
                if (!mbar_wait(bar(SL::kPFull), pg & 1, &g_prefill_error, abort_flag)) return false;
                if (!mbar_wait(bar(SL::kVFull + st), (pg / NS) & 1, &g_prefill_error, abort_flag))
                    return false;
                tc_fence_after_sync();
                const uint32_t pbase = base + SL::kP;
                const uint32_t vbase = base + SL::kV + st * SL::kQBytes;
                for (int ks = 0; ks < pn / 16; ++ks) {
                    // A = P (K-major, keys contiguous), B = V (MN-major: d contiguous,
                    // 64-column slabs LBO apart, 8-key groups SBO apart)
                    const uint64_t a = smem_desc_sw128(
                        pbase + (ks >> 2) * SL::kRegion + (ks & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc_sw128(vbase + ks * 16 * 128, SL::kRegion, 1024);
                    mma_bf16_ss(tmem + kTmemO, a, b, kIdescPV, (!first || ks > 0) ? 1u : 0u);
                }
                mma_commit(bar(SL::kPVDone));
                mma_commit(bar(SL::kKVEmpty + st));
                last_commit_g = pg;
                any_commit = true;
                return true;
            };

            for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++uc) {
                const Unit x = unit_geom(u, p);
                const uint32_t qb = uc & 1;
                ok = mbar_wait(bar(SL::kQFull + qb), (uc >> 1) & 1, &g_prefill_error, abort_flag);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t qbase = base + SL::kQ + qb * SL::kQBytes;
                for (int j = 0; j < x.n_tiles; ++j, ++g) {
                    const uint32_t st = g % NS;
                    const uint32_t sb = g & 1;
                    ok = mbar_wait(bar(SL::kKFull + st), (g / NS) & 1, &g_prefill_error, abort_flag) &&
                         mbar_wait(bar(SL::kSEmpty + sb), ((g >> 1) & 1) ^ 1, &g_prefill_error,
                                   abort_flag);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const int n = tile_width(x, j);
                    const uint32_t idesc = kIdescS | (static_cast<uint32_t>(n >> 3) << 17);
                    const uint32_t kbase = base + SL::kK + st * SL::kQBytes;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * SL::kRegion + (ks & 3) * 32;
                        const uint64_t a = smem_desc_sw128(qbase + off, 16, 1024);
                        const uint64_t b = smem_desc_sw128(kbase + off, 16, 1024);
                        mma_bf16_ss(tmem + sb * 128, a, b, idesc, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(SL::kSFull + sb));
                    if (j == x.n_tiles - 1) mma_commit(bar(SL::kQEmpty + qb));
                    if (have_prev) {
                        ok = issue_pv(prev_g, prev_n, prev_first);
                        if (!ok) break;
                    }
                    have_prev = true;
                    prev_g = g;
                    prev_n = n;
                    prev_first = (j == 0);
                }
            }
            if (ok && have_prev) issue_pv(prev_g, prev_n, prev_first);
            // Drain: all issued MMAs complete before TMEM is released.
            if (any_commit) {
                int no_abort = 0;
                mbar_wait(bar(SL::kPVDone), last_commit_g & 1, &g_prefill_error, &no_abort);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int quarter = warp & 3;             // TMEM lanes this warp may access
        const int row = quarter * 32 + lane;      // MMA row == TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const int prow = row / p.G;               // position offset within the tile
        const int hrow = row - prow * p.G;        // head offset within the group
        const bool leader = (threadIdx.x == 64);  // first softmax thread issues stores
        const uint32_t pbase = base + SL::kP;
        uint32_t g = 0;

        for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
            const Unit x = unit_geom(u, p);
            const int t = x.t0 + prow;
            const bool row_valid = (t <= x.t1);
            const int lo_t = p.w < 0 ? 0 : max(p.s, t - (p.w - p.s) + 1);
            float m_run = -INFINITY;
            float l_run = 0.f;

            for (int j = 0; j < x.n_tiles; ++j, ++g) {
                const uint32_t sb = g & 1;
                mbar_wait(bar(SL::kSFull + sb), (g >> 1) & 1, &g_prefill_error, abort_flag);
                tc_fence_after_sync();
                float sv[128];
                {
                    uint32_t r[32];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        tmem_ld32(tmem + lane_addr + sb * 128 + c4 * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) sv[c4 * 32 + i] = __uint_as_float(r[i]);
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SL::kSEmpty + sb));

                // mask: band columns [c_lo, c_hi], sink columns [0, sink_hi)
                const int key0 = x.lo + 128 * j - p.s_pad;
                int c_lo = max(j == 0 ? p.s_pad : 0, lo_t - key0);
                int c_hi = t - key0;
                int sink_hi = (j == 0) ? min(p.s, t + 1) : 0;
                if (!row_valid) {
                    c_lo = 1;
                    c_hi = 0;
                    sink_hi = 0;
                }
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const bool ok = (c >= c_lo && c <= c_hi) || (c < sink_hi);
                    sv[c] = ok ? sv[c] : -INFINITY;
                    mx = fmaxf(mx, sv[c]);
                }
                const float m_new = fmaxf(m_run, mx);
                float alpha = 1.f;
                if (m_new > m_run &&
                    (m_run == -INFINITY || (m_new - m_run) * p.scale_log2 > 8.f)) {
                    alpha = ex2_approx((m_run - m_new) * p.scale_log2);
                    m_run = m_new;
                }
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run * p.scale_log2;
                uint32_t pk[64];
                float lsum = 0.f;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const float p0 = ex2_approx(fmaf(sv[2 * i], p.scale_log2, neg_m));
                    const float p1 = ex2_approx(fmaf(sv[2 * i + 1], p.scale_log2, neg_m));
                    pk[i] = pack_bf16x2(p0, p1);
                    lsum += bf16lo_to_f32(pk[i]) + bf16hi_to_f32(pk[i]);
                }
                l_run = l_run * alpha + lsum;

                // P may be overwritten once the previous P*V has completed.
                if (g > 0)
                    mbar_wait(bar(SL::kPVDone), (g - 1) & 1, &g_prefill_error, abort_flag);
                tc_fence_after_sync();
#pragma unroll
                for (int cc = 0; cc < 16; ++cc) {
                    const uint32_t addr = pbase + (cc >> 3) * SL::kRegion + row * 128 +
                                          ((((cc & 7) ^ (row & 7))) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                 "r"(pk[4 * cc]), "r"(pk[4 * cc + 1]), "r"(pk[4 * cc + 2]),
                                 "r"(pk[4 * cc + 3])
                                 : "memory");
                }
                fence_proxy_async_smem();
                // Rescale O when this warp raised any running max (not on the
                // first tile: its P*V overwrites O).
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    uint32_t r[32];
#pragma unroll
                    for (int c4 = 0; c4 < D / 32; ++c4) {
                        const uint32_t ta = tmem + lane_addr + kTmemO + c4 * 32;
                        tmem_ld32(ta, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(ta, r);
                    }
                    tmem_wait_st();
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SL::kPFull));
            }

            // ---------------------------------------------------- epilogue
            const uint32_t glast = g - 1;
            mbar_wait(bar(SL::kPVDone), glast & 1, &g_prefill_error, abort_flag);
            tc_fence_after_sync();
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_addr + kTmemO + c4 * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 4; ++q) {  // four 16-byte chunks of 8 columns
                    const int cc = c4 * 4 + q;
                    const uint32_t v0 = pack_bf16x2(__uint_as_float(r[8 * q + 0]) * inv_l,
                                                    __uint_as_float(r[8 * q + 1]) * inv_l);
                    const uint32_t v1 = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * inv_l,
                                                    __uint_as_float(r[8 * q + 3]) * inv_l);
                    const uint32_t v2 = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * inv_l,
                                                    __uint_as_float(r[8 * q + 5]) * inv_l);
                    const uint32_t v3 = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * inv_l,
                                                    __uint_as_float(r[8 * q + 7]) * inv_l);
                    const uint32_t addr = pbase + (cc >> 3) * SL::kRegion + row * 128 +
                                          ((((cc & 7) ^ (row & 7))) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v0),
                                 "r"(v1), "r"(v2), "r"(v3)
                                 : "memory");
                }
            }
            fence_proxy_async_smem();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (leader && !*abort_flag) {
#pragma unroll
                for (int db = 0; db < D / 64; ++db)
                    tma_store_4d(&maps.o, pbase + db * SL::kRegion, db * 64, x.kvh * p.G, x.t0, x.b);
                tma_store_commit();
                tma_store_wait_read_all();
            }
            if (p.lse != nullptr && row_valid && !*abort_flag) {
                const int h = x.kvh * p.G + hrow;
                p.lse[(static_cast<int64_t>(x.b) * p.Hq + h) * p.L + t] =
                    m_run * p.scale + logf(l_run);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
        }
        if (leader) tma_store_wait_all();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

bool encode_map(CUtensorMap *m, const void *ptr, int d, int heads, int L, int B, int box_heads,
                int box_rows) {
    const cuTensorMapEncodeTiled_fn enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2,
                             (cuuint64_t)L * heads * d * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, int NS>
swa_status launch_prefill(const PrefillMaps &maps, const PrefillParams &p, cudaStream_t stream) {
    using SL = PrefillSmem<D, NS>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SWA_ERR_CUDA;
    static bool configured[64] = {};
    if (dev < 64 && !configured[dev]) {
        if (cudaFuncSetAttribute(swa_prefill_kernel<D, NS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SL::kAlloc) != cudaSuccess)
            return SWA_ERR_CUDA;
        configured[dev] = true;
    }
    const int sms = device_sm_count();
    if (sms <= 0) return SWA_ERR_CUDA;
    const int grid = p.n_units < sms ? p.n_units : sms;
    swa_prefill_kernel<D, NS><<<grid, kThreads, SL::kAlloc, stream>>>(maps, p);
    return cudaPeekAtLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

}  // namespace

swa_status prefill_launch(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                          int L, int Hq, int Hkv, int d, int w, int s, cudaStream_t stream) {
    PrefillParams p{};
    p.B = B;
    p.L = L;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.P = 128 / p.G;
    p.w = w < 0 ? -1 : w;
    p.s = w < 0 ? 0 : s;
    p.s_pad = (p.s + 7) & ~7;
    p.n_qtiles = (L + p.P - 1) / p.P;
    p.n_units = B * Hkv * p.n_qtiles;
    p.scale = 1.0f / std::sqrt(static_cast<float>(d));
    p.scale_log2 = p.scale * 1.4426950408889634f;
    p.lse = lse;

    PrefillMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    bool ok = encode_map(&maps.q, q, d, Hq, L, B, p.G, p.P) &&
              encode_map(&maps.o, o, d, Hq, L, B, p.G, p.P) &&
              encode_map(&maps.k_band, k, d, Hkv, L, B, 1, 128) &&
              encode_map(&maps.v_band, v, d, Hkv, L, B, 1, 128);
    if (ok && p.s_pad > 0)
        ok = encode_map(&maps.k_sink, k, d, Hkv, L, B, 1, p.s_pad) &&
             encode_map(&maps.v_sink, v, d, Hkv, L, B, 1, p.s_pad) &&
             encode_map(&maps.k_band0, k, d, Hkv, L, B, 1, 128 - p.s_pad) &&
             encode_map(&maps.v_band0, v, d, Hkv, L, B, 1, 128 - p.s_pad);
    if (!ok) return SWA_ERR_CUDA;
    if (d == 128) return launch_prefill<128, 2>(maps, p, stream);
    return launch_prefill<64, 4>(maps, p, stream);
}

int prefill_read_clear_error(cudaStream_t stream) {
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_prefill_error, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess)
        return SWA_ERR_CUDA;
    if (cudaMemcpyToSymbolAsync(g_prefill_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                stream) != cudaSuccess)
        return SWA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SWA_ERR_CUDA;
    return v;
}

}  // namespace swa
