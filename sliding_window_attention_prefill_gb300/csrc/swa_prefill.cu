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
// one TMA box loads it.  The unit needs the sink keys [0, s) and the band
// [lo, t1] with lo = max(s, t0-(w-s)+1): the key columns are laid out as
// [s_pad sink rows | band ...] in 128-column key tiles, the sink block (s
// rounded up to 8 rows) sharing the first tile.
//
// Roles (320 threads, one persistent CTA per SM):
//   warp 0       TMA producer: Q (one buffer per softmax warpgroup), K tiles
//                (NSK-slot ring), V tiles (NSV-slot ring)
//   warp 1       tcgen05 issuer; owns the 512-column TMEM allocation
//                S_A | S_B | O_A | O_B
//   warps 2..5   softmax warpgroup A, warps 6..9 softmax warpgroup B: each
//                takes every other work unit of the CTA, one thread per MMA
//                row (TMEM lane)
// The two warpgroups ping-pong on the tensor cores: while A runs the softmax
// of its tile, the MMA warp computes B's O += P V and next S = Q K^T, and
// vice versa.  A warpgroup writes P (bf16) over the first 64 columns of its
// own S and the P V product reads it from tensor memory (tcgen05.mma with the
// A operand in TMEM); the next S of that warpgroup is issued after that P V
// by the same thread, and tcgen05 MMAs of one thread execute in issue order.
// The running max is only raised when it grows by more than 2^8 (exact:
// numerator and denominator share the same stale max), so the O rescale
// through TMEM is rare.
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
    CUtensorMap q;                    // box {64, G, P, 1} over [B, L, Hq, d]
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
    uint16_t *o;              // [B, L, Hq, d] bf16
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

// The sequence of key tiles one softmax warpgroup works through: the CTA's
// units u = blockIdx.x + (2k + wg) * gridDim.x, k = 0, 1, ..., each split
// into its key tiles.
struct TileStream {
    int k, u, j;
    bool valid;
    Unit x;
    __device__ __forceinline__ void init(int wg, const PrefillParams &p) {
        k = 0;
        j = 0;
        u = blockIdx.x + wg * gridDim.x;
        valid = u < p.n_units;
        if (valid) x = unit_geom(u, p);
    }
    __device__ __forceinline__ void next(const PrefillParams &p) {
        if (++j >= x.n_tiles) {
            j = 0;
            ++k;
            u += 2 * gridDim.x;
            valid = u < p.n_units;
            if (valid) x = unit_geom(u, p);
        }
    }
};

template <int D, int NSK, int NSV>
struct PrefillSmem {
    static constexpr int kRegion = 128 * 128;           // one 64-column slab of 128 rows
    static constexpr int kTile = 128 * D * 2;           // Q / K / V tile bytes
    static constexpr int kQ = 0;                        // Q buffer per warpgroup
    static constexpr int kK = kQ + 2 * kTile;           // K ring
    static constexpr int kV = kK + NSK * kTile;         // V ring
    static constexpr int kBar = kV + NSV * kTile;       // mbarriers
    // barrier slots (8 bytes each)
    static constexpr int kQFull = 0, kQEmpty = 2, kKFull = 4, kKEmpty = 4 + NSK,
                         kVFull = 4 + 2 * NSK, kVEmpty = 4 + 2 * NSK + NSV,
                         kSFull = 4 + 2 * NSK + 2 * NSV, kPFull = kSFull + 2, kODone = kPFull + 2,
                         kNumBars = kODone + 2;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    static constexpr int kAbort = kTmemSlot + 8;
    static constexpr int kBytes = kAbort + 8;
    static constexpr int kAlloc = kBytes + 1024;        // room to align the base to 1024
};

constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;

template <int D, int NSK, int NSV>
__global__ void __launch_bounds__(kThreads, 1)
    swa_prefill_kernel(const __grid_constant__ PrefillMaps maps, const PrefillParams p) {
    using SL = PrefillSmem<D, NSK, NSV>;
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
            const bool four = (i == SL::kPFull || i == SL::kPFull + 1);
            mbar_init(bar(i), four ? 4u : 1u);
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
            constexpr uint32_t kBytes = SL::kTile;
            TileStream st[2];
            st[0].init(0, p);
            st[1].init(1, p);
            uint32_t gi = 0;  // global tile index, in the order the MMA warp issues S
            uint32_t nq[2] = {0, 0};
            bool ok = true;
            while (ok && (st[0].valid || st[1].valid)) {
                for (int wg = 0; wg < 2 && ok; ++wg) {
                    if (!st[wg].valid) continue;
                    const Unit &x = st[wg].x;
                    const int j = st[wg].j;
                    if (j == 0) {  // Q of a new unit of this warpgroup
                        ok = mbar_wait(bar(SL::kQEmpty + wg), (nq[wg] & 1) ^ 1, &g_prefill_error,
                                       abort_flag);
                        if (!ok) break;
                        const uint32_t qdst = base + SL::kQ + wg * SL::kTile;
                        mbar_arrive_expect_tx(bar(SL::kQFull + wg), kBytes);
#pragma unroll
                        for (int db = 0; db < D / 64; ++db)
                            tma_load_4d(qdst + db * SL::kRegion, &maps.q, bar(SL::kQFull + wg),
                                        db * 64, x.kvh * p.G, x.t0, x.b);
                        ++nq[wg];
                    }
                    const uint32_t ks = gi % NSK, vs = gi % NSV;
                    ok = mbar_wait(bar(SL::kKEmpty + ks), ((gi / NSK) & 1) ^ 1, &g_prefill_error,
                                   abort_flag);
                    if (!ok) break;
                    const uint32_t kdst = base + SL::kK + ks * SL::kTile;
                    const int key0 = x.lo + 128 * j - p.s_pad;  // key of column 0 (band)
                    const bool sink_tile = (j == 0 && p.s_pad > 0);
                    const uint32_t off = p.s_pad * 128;
                    mbar_arrive_expect_tx(bar(SL::kKFull + ks), kBytes);
#pragma unroll
                    for (int db = 0; db < D / 64; ++db) {
                        const uint32_t dst = kdst + db * SL::kRegion;
                        if (sink_tile) {
                            tma_load_4d(dst, &maps.k_sink, bar(SL::kKFull + ks), db * 64, x.kvh, 0, x.b);
                            tma_load_4d(dst + off, &maps.k_band0, bar(SL::kKFull + ks), db * 64,
                                        x.kvh, x.lo, x.b);
                        } else {
                            tma_load_4d(dst, &maps.k_band, bar(SL::kKFull + ks), db * 64, x.kvh,
                                        key0, x.b);
                        }
                    }
                    ok = mbar_wait(bar(SL::kVEmpty + vs), ((gi / NSV) & 1) ^ 1, &g_prefill_error,
                                   abort_flag);
                    if (!ok) break;
                    const uint32_t vdst = base + SL::kV + vs * SL::kTile;
                    mbar_arrive_expect_tx(bar(SL::kVFull + vs), kBytes);
#pragma unroll
                    for (int db = 0; db < D / 64; ++db) {
                        const uint32_t dst = vdst + db * SL::kRegion;
                        if (sink_tile) {
                            tma_load_4d(dst, &maps.v_sink, bar(SL::kVFull + vs), db * 64, x.kvh, 0, x.b);
                            tma_load_4d(dst + off, &maps.v_band0, bar(SL::kVFull + vs), db * 64,
                                        x.kvh, x.lo, x.b);
                        } else {
                            tma_load_4d(dst, &maps.v_band, bar(SL::kVFull + vs), db * 64, x.kvh,
                                        key0, x.b);
                        }
                    }
                    ++gi;
                    st[wg].next(p);
                }
            }
            // Drain: every copy this thread started has landed before exit
            // (bounded waits that ignore the abort flag; in the normal path the
            // consumers already saw these phases complete).
            int no_abort = 0;
            for (uint32_t i = 0; i < NSK && i < gi; ++i) {
                const uint32_t g = gi - 1 - i;
                mbar_wait(bar(SL::kKFull + g % NSK), (g / NSK) & 1, &g_prefill_error, &no_abort);
            }
            for (uint32_t i = 0; i < NSV && i < gi; ++i) {
                const uint32_t g = gi - 1 - i;
                mbar_wait(bar(SL::kVFull + g % NSV), (g / NSV) & 1, &g_prefill_error, &no_abort);
            }
            for (int wg = 0; wg < 2; ++wg)
                if (nq[wg] > 0)
                    mbar_wait(bar(SL::kQFull + wg), (nq[wg] - 1) & 1, &g_prefill_error, &no_abort);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16_f32(128, 0, false);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, true);
            TileStream st[2];
            st[0].init(0, p);
            st[1].init(1, p);
            uint32_t gi = 0;
            uint32_t nq[2] = {0, 0}, npv[2] = {0, 0};
            bool pend[2] = {false, false}, pend_first[2] = {false, false};
            uint32_t pend_gi[2] = {0, 0};
            int pend_n[2] = {0, 0};
            bool ok = true, any_pv = false;

            // S = Q K^T for the next tile of warpgroup wg (into S_wg).
            auto issue_s = [&](int wg) -> bool {
                const Unit &x = st[wg].x;
                const int j = st[wg].j;
                if (j == 0) {
                    if (!mbar_wait(bar(SL::kQFull + wg), nq[wg] & 1, &g_prefill_error, abort_flag))
                        return false;
                }
                const uint32_t ks = gi % NSK;
                if (!mbar_wait(bar(SL::kKFull + ks), (gi / NSK) & 1, &g_prefill_error, abort_flag))
                    return false;
                tc_fence_after_sync();
                const int n = tile_width(x, j);
                const uint32_t idesc = kIdescS | (static_cast<uint32_t>(n >> 3) << 17);
                const uint32_t qbase = base + SL::kQ + wg * SL::kTile;
                const uint32_t kbase = base + SL::kK + ks * SL::kTile;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * SL::kRegion + (kk & 3) * 32;
                    mma_bf16_ss(tmem + wg * 128, smem_desc_sw128(qbase + off, 16, 1024),
                                smem_desc_sw128(kbase + off, 16, 1024), idesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(SL::kSFull + wg));
                mma_commit(bar(SL::kKEmpty + ks));
                const bool last = (j == x.n_tiles - 1);
                if (last) {
                    mma_commit(bar(SL::kQEmpty + wg));
                    ++nq[wg];
                }
                pend[wg] = true;
                pend_gi[wg] = gi;
                pend_n[wg] = n;
                pend_first[wg] = (j == 0);
                ++gi;
                st[wg].next(p);
                return true;
            };
            // O += P V for warpgroup wg's pending tile (P from TMEM over S_wg).
            auto issue_pv = [&](int wg) -> bool {
                const uint32_t g = pend_gi[wg];
                const uint32_t vs = g % NSV;
                if (!mbar_wait(bar(SL::kPFull + wg), npv[wg] & 1, &g_prefill_error, abort_flag))
                    return false;
                if (!mbar_wait(bar(SL::kVFull + vs), (g / NSV) & 1, &g_prefill_error, abort_flag))
                    return false;
                tc_fence_after_sync();
                const uint32_t vbase = base + SL::kV + vs * SL::kTile;
                const uint32_t o_tmem = tmem + 256 + wg * 128;
                for (int kk = 0; kk < pend_n[wg] / 16; ++kk) {
                    const uint64_t b = smem_desc_sw128(vbase + kk * 16 * 128, SL::kRegion, 1024);
                    mma_bf16_ts(o_tmem, tmem + wg * 128 + kk * 8, b, kIdescPV,
                                (!pend_first[wg] || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(SL::kODone + wg));
                mma_commit(bar(SL::kVEmpty + vs));
                ++npv[wg];
                pend[wg] = false;
                any_pv = true;
                return true;
            };

            for (int wg = 0; wg < 2 && ok; ++wg)
                if (st[wg].valid) ok = issue_s(wg);
            while (ok && (pend[0] || pend[1])) {
                for (int wg = 0; wg < 2 && ok; ++wg) {
                    if (!pend[wg]) continue;
                    ok = issue_pv(wg);
                    if (ok && st[wg].valid) ok = issue_s(wg);
                }
            }
            // Drain: all issued MMAs complete before TMEM is released.
            if (any_pv) {
                int no_abort = 0;
                for (int wg = 0; wg < 2; ++wg)
                    if (npv[wg] > 0)
                        mbar_wait(bar(SL::kODone + wg), (npv[wg] - 1) & 1, &g_prefill_error,
                                  &no_abort);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int wg = (warp - 2) >> 2;           // warpgroup 0 (warps 2..5) or 1 (6..9)
        const int quarter = warp & 3;             // TMEM lanes this warp may access
        const int row = quarter * 32 + lane;      // MMA row == TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t s_tmem = tmem + lane_addr + wg * 128;
        const uint32_t o_tmem = tmem + lane_addr + 256 + wg * 128;
        const int prow = row / p.G;               // position offset within the tile
        const int hrow = row - prow * p.G;        // head offset within the group
        uint32_t nt = 0;                          // tiles this warpgroup has finished

        for (int u = blockIdx.x + wg * gridDim.x; u < p.n_units; u += 2 * gridDim.x) {
            const Unit x = unit_geom(u, p);
            const int t = x.t0 + prow;
            const bool row_valid = (t <= x.t1);
            const int lo_t = p.w < 0 ? 0 : max(p.s, t - (p.w - p.s) + 1);
            float m_run = -INFINITY;
            float l_run = 0.f;

            for (int j = 0; j < x.n_tiles; ++j, ++nt) {
                mbar_wait(bar(SL::kSFull + wg), nt & 1, &g_prefill_error, abort_flag);
                tc_fence_after_sync();
                // mask: band columns [c_lo, c_hi], sink columns [0, sink_hi)
                const int key0 = x.lo + 128 * j - p.s_pad;
                int c_lo = max(j == 0 ? p.s_pad : 0, lo_t - key0);
                int c_hi = min(t - key0, 127);
                int sink_hi = (j == 0) ? min(p.s, t + 1) : 0;
                if (!row_valid) {
                    c_lo = 128;
                    c_hi = -1;
                    sink_hi = 0;
                }
                // Column c of this tile is attended by the row when c is in the
                // band [c_lo, c_hi] or among the sinks [0, sink_hi).  Per
                // 32-column chunk the warp checks whether every row has the
                // whole chunk in its band ("full": no mask) or none of it
                // ("empty": no load, P = 0).
                const bool band_ok = c_lo <= c_hi;
                const unsigned span = band_ok ? static_cast<unsigned>(c_hi - c_lo) : 0u;
                const int band_from = band_ok ? c_lo : 1 << 20;
                auto flags = [&](int q, bool &full, bool &empty) {
                    const bool f = band_ok && c_lo <= 32 * q && c_hi >= 32 * q + 31;
                    const bool e = (!band_ok || c_hi < 32 * q || c_lo > 32 * q + 31) &&
                                   sink_hi <= 32 * q;
                    full = __all_sync(0xffffffffu, f);
                    empty = __all_sync(0xffffffffu, e);
                };
                // pass 1: masked row max, S read from TMEM two chunks per wait
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
                for (int q = 0; q < 4; q += 2) {
                    bool f0, e0, f1, e1;
                    flags(q, f0, e0);
                    flags(q + 1, f1, e1);
                    if (e0 && e1) continue;
                    uint32_t r0[32], r1[32];
                    tmem_ld32(s_tmem + 32 * q, r0);
                    tmem_ld32(s_tmem + 32 * q + 32, r1);
                    tmem_wait_ld();
                    const int x0 = 32 * q - band_from, sh = sink_hi - 32 * q;
                    if (f0 && f1) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            m4[i & 3] = fmaxf(m4[i & 3], __uint_as_float(r0[i]));
                            m4[i & 3] = fmaxf(m4[i & 3], __uint_as_float(r1[i]));
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const bool ok0 = static_cast<unsigned>(x0 + i) <= span || i < sh;
                            const bool ok1 = static_cast<unsigned>(x0 + 32 + i) <= span || i + 32 < sh;
                            m4[i & 3] = fmaxf(m4[i & 3], ok0 ? __uint_as_float(r0[i]) : -INFINITY);
                            m4[i & 3] = fmaxf(m4[i & 3], ok1 ? __uint_as_float(r1[i]) : -INFINITY);
                        }
                    }
                }
                const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                const float m_new = fmaxf(m_run, mx);
                float alpha = 1.f;
                if (m_new > m_run &&
                    (m_run == -INFINITY || (m_new - m_run) * p.scale_log2 > 8.f)) {
                    alpha = ex2_approx((m_run - m_new) * p.scale_log2);
                    m_run = m_new;
                }
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run * p.scale_log2;
                // pass 2: P = exp2(S*scale - m) in bf16, written over the first
                // 64 columns of S (the P of chunks q, q+1 lands on columns
                // 16q .. 16q+31, which this pass has already read)
                float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                for (int q = 0; q < 4; q += 2) {
                    bool f0, e0, f1, e1;
                    flags(q, f0, e0);
                    flags(q + 1, f1, e1);
                    uint32_t pk[32];
                    if (e0 && e1) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) pk[i] = 0u;
                    } else {
                        uint32_t r0[32], r1[32];
                        tmem_ld32(s_tmem + 32 * q, r0);
                        tmem_ld32(s_tmem + 32 * q + 32, r1);
                        tmem_wait_ld();
                        if (!(f0 && f1)) {
                            const int x0 = 32 * q - band_from, sh = sink_hi - 32 * q;
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                if (!(static_cast<unsigned>(x0 + i) <= span || i < sh))
                                    r0[i] = __float_as_uint(-INFINITY);
                                if (!(static_cast<unsigned>(x0 + 32 + i) <= span || i + 32 < sh))
                                    r1[i] = __float_as_uint(-INFINITY);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float a0 = ex2_approx(fmaf(__uint_as_float(r0[2 * i]), p.scale_log2, neg_m));
                            const float a1 = ex2_approx(fmaf(__uint_as_float(r0[2 * i + 1]), p.scale_log2, neg_m));
                            const float b0 = ex2_approx(fmaf(__uint_as_float(r1[2 * i]), p.scale_log2, neg_m));
                            const float b1 = ex2_approx(fmaf(__uint_as_float(r1[2 * i + 1]), p.scale_log2, neg_m));
                            pk[i] = pack_bf16x2(a0, a1);
                            pk[16 + i] = pack_bf16x2(b0, b1);
                            l4[i & 3] += (a0 + a1) + (b0 + b1);
                        }
                    }
                    uint32_t lo16[16], hi16[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        lo16[i] = pk[i];
                        hi16[i] = pk[16 + i];
                    }
                    tmem_st16(s_tmem + 16 * q, lo16);
                    tmem_st16(s_tmem + 16 * q + 16, hi16);
                }
                const float lsum = (l4[0] + l4[1]) + (l4[2] + l4[3]);
                l_run = l_run * alpha + lsum;
                // Rescale O when this warp raised any running max (not on the
                // first tile: its P V overwrites O).  The previous P V of this
                // warpgroup completed before this tile's S (same issuing thread).
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int c4 = 0; c4 < D / 32; ++c4) {
                        uint32_t r[32];
                        tmem_ld32(o_tmem + c4 * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(o_tmem + c4 * 32, r);
                    }
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SL::kPFull + wg));
            }

            // ---------------------------------------------------- epilogue
            mbar_wait(bar(SL::kODone + wg), (nt - 1) & 1, &g_prefill_error, abort_flag);
            tc_fence_after_sync();
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
            const bool store = row_valid && !*abort_flag;
            uint16_t *orow =
                p.o + ((static_cast<int64_t>(x.b) * p.L + t) * p.Hq + x.kvh * p.G + hrow) * D;
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
                uint32_t r[32];
                tmem_ld32(o_tmem + c4 * 32, r);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l,
                                        __uint_as_float(r[2 * i + 1]) * inv_l);
                if (store) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c4 * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            if (p.lse != nullptr && store) {
                const int h = x.kvh * p.G + hrow;
                p.lse[(static_cast<int64_t>(x.b) * p.Hq + h) * p.L + t] =
                    m_run * p.scale + logf(l_run);
            }
            tc_fence_before_sync();
        }
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

template <int D, int NSK, int NSV>
swa_status launch_prefill(const PrefillMaps &maps, const PrefillParams &p, cudaStream_t stream) {
    using SL = PrefillSmem<D, NSK, NSV>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    static bool configured[64] = {};
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(swa_prefill_kernel<D, NSK, NSV>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SL::kAlloc);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill)");
        configured[dev] = true;
    }
    const int sms = device_sm_count();
    if (sms <= 0) return cuda_fail(cudaErrorInvalidDevice, "device_sm_count");
    // two warpgroups per CTA: half as many CTAs as units keeps both busy
    const int want = (p.n_units + 1) / 2;
    const int grid = want < sms ? want : sms;
    swa_prefill_kernel<D, NSK, NSV><<<grid, kThreads, SL::kAlloc, stream>>>(maps, p);
    e = cudaPeekAtLastError();
    return e == cudaSuccess ? SWA_OK : cuda_fail(e, "launch swa_prefill_kernel");
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
    p.o = static_cast<uint16_t *>(o);
    p.lse = lse;

    PrefillMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    bool ok = encode_map(&maps.q, q, d, Hq, L, B, p.G, p.P) &&
              encode_map(&maps.k_band, k, d, Hkv, L, B, 1, 128) &&
              encode_map(&maps.v_band, v, d, Hkv, L, B, 1, 128);
    if (ok && p.s_pad > 0)
        ok = encode_map(&maps.k_sink, k, d, Hkv, L, B, 1, p.s_pad) &&
             encode_map(&maps.v_sink, v, d, Hkv, L, B, 1, p.s_pad) &&
             encode_map(&maps.k_band0, k, d, Hkv, L, B, 1, 128 - p.s_pad) &&
             encode_map(&maps.v_band0, v, d, Hkv, L, B, 1, 128 - p.s_pad);
    if (!ok) return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
    if (d == 128) return launch_prefill<128, 2, 3>(maps, p, stream);
    return launch_prefill<64, 4, 6>(maps, p, stream);
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
