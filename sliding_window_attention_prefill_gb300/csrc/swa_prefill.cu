// swa_prefill.cu -- banded SWA(w,s) prefill on sm_103a: TMA-staged tiles,
// tcgen05 MMAs with fp32 accumulators in tensor memory, online softmax.
//
// Operation (o_t = softmax over A(t) of c q_t.k_i, applied to v_i): the window
// equation and SWA(w,s) notation of "Sliding-window beats linear attention"
// (paper summary page), section "Prerequisites / Sliding-window attention
// SWA(w, s)"; w = infinity is the full causal "FA" case of the same page.
//
// Work decomposition (units of 128 query rows = G heads x 128/G positions;
// key columns [sink block | band]): swa_prefill_common.cuh.  This kernel cuts
// a unit's columns into key tiles of up to 256 and runs one unit at a time.
//
// Roles (384 threads = three warpgroups, one persistent CTA per SM; 512 with
// the epilogue warpgroup):
//   warp 0       TMA producer for Q (double-buffered), K and V tiles (V in
//                warp 3 for 256-column tiles)
//   warp 1       tcgen05 issuer of S = Q K^T; owns the 512-column TMEM
//                allocation S (256 columns) | P (128 columns, 16-bit pairs) |
//                O (d columns)
//   warp 2       tcgen05 issuer of O += P V (one issuing thread per product,
//                so that each one's waits and commits overlap the other's
//                MMAs: an issuing thread stays only a couple of MMAs ahead
//                of the tensor pipe)
//   warp 3       TMA stores of the staged output tile (narrow key tiles), or
//                the V producer (256-column tiles)
//   warps 4..11  softmax + epilogue: two threads per MMA row (TMEM lane), each
//                taking every other 32-column chunk of the key tile
//   warps 12..15 epilogue warpgroup (narrow tiles, chosen per call by
//                use_epilogue_wg): O / l of a finished unit out of TMEM into
//                the staging tile while the softmax warps go on
// Key tiles of 256 columns let S = Q K^T run as N = 256 MMAs (twice the work
// per instruction of N = 128 at a similar issue cost on this part), and P
// lives in its own TMEM columns, so S_{g+1} is issued as soon as the softmax
// has read S_g -- while the softmax of tile g is still running -- and
// O += P_g V_g once P_g is written.  The first warpgroup hands registers to the
// two softmax warpgroups (setmaxnreg) so a thread keeps its 128 scores in
// registers.  The running max is only raised when it grows by more than 2^8
// (exact: numerator and denominator share the same stale max), so the O
// rescale through TMEM is rare.
//
// Element type (template DT): bf16 or fp16 for Q, K, V, P and O alike (one
// kind::f16 MMA takes both operands of one type); scores, the softmax and the
// O accumulator are fp32 either way.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "swa_internal.h"
#include "swa_prefill_common.cuh"
#include "swa_ptx.cuh"

// 0: pick the key tile width per call (prefill_key_tile); 128 or 256: always
// that width (for measurements).
#ifndef SWA_PREFILL_FORCE_KT
#define SWA_PREFILL_FORCE_KT 0
#endif

// Epilogue warpgroup (narrow key tiles): 0 never, 1 for units of several key
// tiles or calls of at least 64 units per SM, 2 always (for measurements).
#ifndef SWA_PREFILL_EPI_WG
#define SWA_PREFILL_EPI_WG 1
#endif

namespace swa {

__device__ int g_prefill_error;
__device__ unsigned long long g_prefill_where;

// Key tile width KT: 256 columns (one K or V tile of 64 KB at d = 128, so one
// stage of each), or 128 columns for narrow bands (two stages of each in the
// same shared memory, so the next unit's K and V load during this one).
template <int D, int KT, int NSK, int NSV, bool EW>
struct PrefillSmem {
    static constexpr int kQRegion = 128 * 128;          // 64 columns x 128 query rows
    static constexpr int kKRegion = KT * 128;           // 64 columns x KT key rows
    static constexpr int kQTile = 128 * D * 2;
    static constexpr int kKTile = KT * D * 2;
    static constexpr int kQ = 0;                        // 2 Q buffers
    static constexpr int kK = kQ + 2 * kQTile;          // K ring
    static constexpr int kV = kK + NSK * kKTile;        // V ring
    // O tile staged for one TMA store (128-column tiles only: 128 x d 16-bit,
    // d/64 slabs of 128 rows x 128 bytes, 128-byte swizzle)
    static constexpr int kStageO = kV + NSV * kKTile;
    static constexpr int kStageBytes = (KT <= 128) ? 128 * D * 2 : 0;
    // unit row max for the epilogue warpgroup [2 unit parity][128]
    static constexpr int kEpiM = kStageO + kStageBytes;
    static constexpr int kRed = kEpiM + (EW ? 2 * 128 * 4 : 0);  // row max [2 parity][2 half][128]
    static constexpr int kRedL = kRed + 2 * 2 * 128 * 4;  // row sum [2 parity][2 half][128]
    static constexpr int kBar = kRedL + 2 * 2 * 128 * 4;
    static constexpr int kQFull = 0, kQEmpty = 2, kKFull = 4, kKEmpty = 4 + NSK,
                         kVFull = 4 + 2 * NSK, kVEmpty = 4 + 2 * NSK + NSV,
                         kSFull = 4 + 2 * NSK + 2 * NSV, kSEmpty = kSFull + 1,
                         kPFull = kSFull + 2, kPVDone = kSFull + 3,
                         // staged epilogue: O written (one arrive per softmax
                         // warp), staging buffer read by its stores
                         kOStaged = kSFull + 5, kOFree = kSFull + 6,
                         // P written, for odd tiles (kPFull: even tiles)
                         kPFull1 = kSFull + 7,
                         // epilogue warpgroup, by unit parity: the unit's row
                         // max and sums written, its O complete, its O read
                         kEpiReady = kSFull + 8, kOFull = kSFull + 10, kORead = kSFull + 12,
                         kNumBars = kSFull + (EW ? 14 : 8);
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    static constexpr int kAbort = kTmemSlot + 8;
    static constexpr int kBytes = kAbort + 8;
    static constexpr int kAlloc = kBytes + 1024;        // room to align the base to 1024
};

// 384 threads; 512 with the epilogue warpgroup (warps 12..15).
__host__ __device__ constexpr int prefill_threads(bool ew) { return ew ? 512 : 384; }
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;

template <int D, int KT, int NSK, int NSV, int DT, bool VL, bool EW>
__global__ void __launch_bounds__(prefill_threads(EW), 1)
    swa_prefill_kernel(const __grid_constant__ PrefillMaps maps, const PrefillParams p) {
    using SL = PrefillSmem<D, KT, NSK, NSV, EW>;
    constexpr int NC = (KT + 63) / 64;  // 32-column chunks of a tile per softmax thread
    // A 112-column tile ends in a 16-column chunk (columns 96..111, taken by
    // the second half): that chunk's other 16 columns are not computed.
    constexpr bool kShortTail = (KT % 64 == 48);
    // TMEM columns.  256-column tiles: S [0,256) | P [256,384) | O [384,384+d).
    // 128-column tiles leave room to double-buffer P (by tile) and O (by
    // unit): S [0,128) | P0, P1 [128,256) | O0, O1 [256,256+2d); then the
    // softmax of a tile need not wait for the previous P V to write its P,
    // and a unit's epilogue runs while the next unit's P V goes on.
    constexpr bool DB = (KT <= 128);
    constexpr bool kStageOut = (KT <= 128);  // epilogue through shared memory + TMA store
    // Epilogue warpgroup (warps 12..15): reads each unit's O out of TMEM,
    // normalises and stages it while the softmax warps go on with the next
    // unit (O is double-buffered by unit).
    static_assert(!EW || kStageOut, "the epilogue warpgroup stages the output");
    constexpr uint32_t kTP = DB ? 128u : 256u;
    constexpr uint32_t kTO = DB ? 256u : 384u;
    static_assert(kTO + (DB ? 2 : 1) * D <= kTmemCols, "TMEM columns");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + SL::kAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + SL::kTmemSlot);
    auto bar = [&](int i) { return base + SL::kBar + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int i = 0; i < SL::kNumBars; ++i) {
            const bool eight = (i == SL::kSEmpty || i == SL::kPFull || i == SL::kPFull1 ||
                                i == SL::kEpiReady || i == SL::kEpiReady + 1 ||
                                (i == SL::kOStaged && !EW));
            const bool four = (i == SL::kORead || i == SL::kORead + 1 || (i == SL::kOStaged && EW));
            mbar_init(bar(i), eight ? 8u : (four ? 4u : 1u));
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
    pdl_wait();  // inputs and outputs are the previous kernels' from here on
    const int n_units = prefill_units<VL>(p);

    // Register split.  Without the epilogue warpgroup: 3 x 128 threads
    // launched at 168 registers each (64512); the first warpgroup drops to 80
    // and the softmax warpgroups rise to 208: 80*128 + 2*208*128 = 63488 <=
    // 64512.  With it: 4 x 128 threads at 128 (65536); the softmax
    // warpgroups rise to 192, the first drops to 72 and the epilogue one to
    // 56 (88 and 40 for ragged batches): (72 + 2*192 + 56) * 128 =
    // (88 + 2*192 + 40) * 128 = 65536.
    if (warp < 4) {
        if constexpr (EW && VL)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
        else if constexpr (EW)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory");
        else
            asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
        if ((warp == 0 || (!kStageOut && warp == 3)) && lane == 0) {
            // -------------------------------------------------------- producers
            // Narrow tiles: one thread loads Q, K and V, K one tile ahead of
            // V (K_{g+1} then V_g, the order in which their slots come free:
            // S_{g-1} = Q K^T completes before P V_{g-2}), so neither waits
            // behind the other.  256-column tiles (one stage of each, where V
            // is the latency-critical load): warp 0 loads Q and K, and warp
            // 3, which has no output to store, loads V.
            const bool do_k = (warp == 0);
            const bool do_v = kStageOut || warp == 3;
            if (do_k) {
                tma_prefetch_desc(&maps.q);
                tma_prefetch_desc(&maps.k_band);
            }
            if (do_v) tma_prefetch_desc(&maps.v_band);
            uint32_t gk = 0, gv = 0, uc = 0;
            bool ok = true;
            // one K (kq) or V tile: tile j of unit x, ring position g
            auto load_tile = [&](bool kq, const Unit &x, int j, uint32_t g) -> bool {
                const uint32_t ns = kq ? NSK : NSV;
                const uint32_t slot = g % ns;
                if (!mbar_wait(bar((kq ? SL::kKEmpty : SL::kVEmpty) + slot), ((g / ns) & 1) ^ 1,
                               &g_prefill_error, abort_flag))
                    return false;
                const uint32_t dst0 = base + (kq ? SL::kK : SL::kV) + slot * SL::kKTile;
                const int key0 = x.lo + KT * j - p.s_pad;  // key of column 0 (band)
                const uint32_t fb = bar((kq ? SL::kKFull : SL::kVFull) + slot);
                mbar_arrive_expect_tx(fb, SL::kKTile);
#pragma unroll
                for (int db = 0; db < D / 64; ++db) {
                    const uint32_t dst = dst0 + db * SL::kKRegion;
                    if (j == 0 && p.s_pad > 0) {
                        tma_load_4d(dst, kq ? &maps.k_sink : &maps.v_sink, fb, db * 64, x.kvh,
                                    x.r0, x.b);
                        tma_load_4d(dst + p.s_pad * 128, kq ? &maps.k_band0 : &maps.v_band0, fb,
                                    db * 64, x.kvh, x.r0 + x.lo, x.b);
                    } else {
                        tma_load_4d(dst, kq ? &maps.k_band : &maps.v_band, fb, db * 64, x.kvh,
                                    x.r0 + key0, x.b);
                    }
                }
                return true;
            };
            Unit xv{};   // the unit of the next V tile
            int jv = 0;  // and its tile
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
                const Unit x = unit_geom<KT, VL>(u, p, n_units);
                if (!do_k) {  // V alone, in tile order
                    for (int j = 0; j < x.n_tiles && ok; ++j) {
                        ok = load_tile(false, x, j, gv);
                        if (ok) ++gv;
                    }
                    continue;
                }
                const uint32_t qb = uc & 1;
                ok = mbar_wait(bar(SL::kQEmpty + qb), ((uc >> 1) & 1) ^ 1, &g_prefill_error,
                               abort_flag);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(SL::kQFull + qb), SL::kQTile);
#pragma unroll
                for (int db = 0; db < D / 64; ++db)
                    tma_load_4d(base + SL::kQ + qb * SL::kQTile + db * SL::kQRegion, &maps.q,
                                bar(SL::kQFull + qb), db * 64, x.kvh * p.G, x.r0 + x.t0 - p.q_off,
                                x.b);
                if (uc == 0) xv = x;
                for (int j = 0; j < x.n_tiles && ok; ++j) {
                    ok = load_tile(true, x, j, gk);
                    if (!ok) break;
                    ++gk;
                    if (do_v && gk >= 2) {  // V of the tile before this one
                        ok = load_tile(false, xv, jv, gv);
                        if (!ok) break;
                        ++gv;
                        if (++jv == xv.n_tiles) {
                            xv = x;
                            jv = 0;
                        }
                    }
                }
            }
            if (ok && do_k && do_v && gv < gk) {  // the last V
                if (load_tile(false, xv, jv, gv)) ++gv;
            }
            // Drain: every copy this thread started has landed before exit
            // (bounded waits that ignore the abort flag; in the normal path the
            // consumers already saw these phases complete).
            int no_abort = 0;
            for (uint32_t i = 0; i < NSK && i < gk; ++i) {
                const uint32_t gl = gk - 1 - i;
                mbar_wait(bar(SL::kKFull + gl % NSK), (gl / NSK) & 1, &g_prefill_error, &no_abort);
            }
            for (uint32_t i = 0; i < NSV && i < gv; ++i) {
                const uint32_t gl = gv - 1 - i;
                mbar_wait(bar(SL::kVFull + gl % NSV), (gl / NSV) & 1, &g_prefill_error, &no_abort);
            }
            for (uint32_t i = 0; do_k && i < 2 && i < uc; ++i) {
                const uint32_t ul = uc - 1 - i;
                mbar_wait(bar(SL::kQFull + (ul & 1)), (ul >> 1) & 1, &g_prefill_error, &no_abort);
            }
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------------- S = Q K^T issuer
            // S_{g+1} goes to the tensor core as soon as the softmax has read
            // S_g (and K_{g+1} has landed), independently of the P V issuer.
            constexpr uint32_t kIdescS = idesc_f16k<DT>(128, 0, false);
            uint32_t g = 0, uc = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
                const Unit x = unit_geom<KT, VL>(u, p, n_units);
                const uint32_t qb = uc & 1;
                ok = mbar_wait(bar(SL::kQFull + qb), (uc >> 1) & 1, &g_prefill_error, abort_flag);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t qbase = base + SL::kQ + qb * SL::kQTile;
                for (int j = 0; j < x.n_tiles; ++j, ++g) {
                    const uint32_t ks = g % NSK;
                    ok = mbar_wait(bar(SL::kKFull + ks), (g / NSK) & 1, &g_prefill_error,
                                   abort_flag) &&
                         mbar_wait(bar(SL::kSEmpty), (g & 1) ^ 1, &g_prefill_error, abort_flag);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const int n = tile_width<KT>(x, j);
                    const uint32_t idesc = kIdescS | (static_cast<uint32_t>(n >> 3) << 17);
                    // Descriptors built once per tile; k-step kk (16 columns of d)
                    // is 32 bytes into a 64-column slab, slab kk/4 a region on
                    // (offsets added to the start-address field, in 16 bytes).
                    const uint64_t a0 = smem_desc_sw128(qbase, 16, 1024);
                    const uint64_t b0 = smem_desc_sw128(base + SL::kK + ks * SL::kKTile, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_f16k_ss(tmem + kTmemS,
                                    a0 + static_cast<uint64_t>(((kk >> 2) * SL::kQRegion + (kk & 3) * 32) >> 4),
                                    b0 + static_cast<uint64_t>(((kk >> 2) * SL::kKRegion + (kk & 3) * 32) >> 4),
                                    idesc, kk > 0 ? 1u : 0u);
                    mma_commit(bar(SL::kSFull));
                    mma_commit(bar(SL::kKEmpty + ks));
                    if (j == x.n_tiles - 1) mma_commit(bar(SL::kQEmpty + qb));
                }
            }
            // Drain: the last S has landed before TMEM is released.
            if (g > 0) {
                int no_abort = 0;
                mbar_wait(bar(SL::kSFull), (g - 1) & 1, &g_prefill_error, &no_abort);
            }
        } else if (warp == 2 && lane == 0) {
            // -------------------------------------------------------- O += P V issuer
            constexpr uint32_t kIdescPV = idesc_f16k<DT>(128, D, true);
            uint32_t g = 0, uc = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++uc) {
                const Unit x = unit_geom<KT, VL>(u, p, n_units);
                const uint32_t ob = uc & 1;
                for (int j = 0; j < x.n_tiles; ++j, ++g) {
                    const uint32_t vs = g % NSV;
                    // One barrier per tile parity: the softmax may finish tile
                    // g+1 before this thread has waited for tile g, and a
                    // waiter must not fall two phases behind an mbarrier (its
                    // phase parity would read as not yet complete).
                    ok = mbar_wait(bar((g & 1) ? SL::kPFull1 : SL::kPFull), (g >> 1) & 1,
                                   &g_prefill_error, abort_flag) &&
                         mbar_wait(bar(SL::kVFull + vs), (g / NSV) & 1, &g_prefill_error,
                                   abort_flag);
                    // O buffer ob held unit uc-2 until the epilogue warpgroup read it
                    if (EW && ok && j == 0 && uc >= 2)
                        ok = mbar_wait(bar(SL::kORead + ob), ((uc >> 1) & 1) ^ 1, &g_prefill_error,
                                       abort_flag);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const int n = tile_width<KT>(x, j);
                    // A = P (TMEM, two 16-bit values per column), B = V (MN-major:
                    // 64-column slabs LBO apart, 8-key groups SBO apart).  The
                    // descriptor is built once per tile; a k-step of 16 keys
                    // (2048 bytes) adds 2048 >> 4 to its start-address field.
                    const uint64_t b0 =
                        smem_desc_sw128(base + SL::kV + vs * SL::kKTile, SL::kKRegion, 1024);
                    const uint32_t d_o = tmem + kTO + (DB ? ob * D : 0u);
                    const uint32_t a_p = tmem + kTP + (DB ? (g & 1) * 64 : 0u);
                    mma_f16k_ts(d_o, a_p, b0, kIdescPV, j == 0 ? 0u : 1u);
                    for (int kk = 1; kk < n / 16; ++kk)
                        mma_f16k_ts(d_o, a_p + kk * 8, b0 + static_cast<uint64_t>(kk * 128),
                                    kIdescPV, 1u);
                    mma_commit(bar(SL::kPVDone + (DB ? (g & 1) : 0)));
                    mma_commit(bar(SL::kVEmpty + vs));
                    if (EW && j == x.n_tiles - 1) mma_commit(bar(SL::kOFull + ob));  // O complete
                }
            }
            // Drain: all issued MMAs complete before TMEM is released.
            if (g > 0) {
                int no_abort = 0;
                const uint32_t gl = g - 1;
                if (DB)
                    mbar_wait(bar(SL::kPVDone + (gl & 1)), (gl >> 1) & 1, &g_prefill_error,
                              &no_abort);
                else
                    mbar_wait(bar(SL::kPVDone), gl & 1, &g_prefill_error, &no_abort);
            }
        } else if (kStageOut && warp == 3) {
            // -------------------------------------------------------- output stores
            // For each unit in the softmax warps' order: once they have staged
            // its O tile, store it with TMA, wait until the store has read the
            // buffer and hand the buffer back.  A varlen unit at the end of
            // its sequence is copied row by row instead (its box would reach
            // into the next sequence's rows).
            uint32_t e = 0;
            for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++e) {
                const Unit x = unit_geom<KT, VL>(u, p, n_units);
                bool staged = false;
                if (lane == 0)
                    staged = mbar_wait(bar(SL::kOStaged), e & 1, &g_prefill_error, abort_flag) &&
                             !*abort_flag;
                staged = __shfl_sync(0xffffffffu, staged ? 1 : 0, 0) != 0;
                const int nrows = (x.t1 - x.t0 + 1) << p.g_log2;  // valid MMA rows
                if (staged && (!VL || nrows >= 128)) {
                    if (lane == 0) {
#pragma unroll
                        for (int db = 0; db < D / 64; ++db)
                            tma_store_4d(&maps.o, base + SL::kStageO + db * (128 * 128), db * 64,
                                         x.kvh * p.G, x.r0 + x.t0 - p.q_off, x.b);
                        tma_store_commit();
                        tma_store_wait_read_all();
                    }
                } else if (VL && staged) {
                    constexpr int kChunks = D / 8;  // 16-byte chunks of a row
                    for (int c = lane; c < nrows * kChunks; c += 32) {
                        const int r = c / kChunks, col = (c % kChunks) * 8;
                        const int ci = (col & 63) >> 3;
                        const uint32_t src = base + SL::kStageO + (col >> 6) * (128 * 128) + r * 128 +
                                             ((ci ^ (r & 7)) << 4);
                        uint4 v4;
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(v4.x), "=r"(v4.y), "=r"(v4.z), "=r"(v4.w)
                                     : "r"(src));
                        const int64_t grow = x.r0 + x.t0 + (r >> p.g_log2) - p.q_off;
                        const int64_t oi = (grow * p.Hq + x.kvh * p.G + (r & (p.G - 1))) * D + col;
                        if (in_bounds(oi / 8, p.n_o / 8, &g_prefill_error, &g_prefill_where))
                            *reinterpret_cast<uint4 *>(p.o + oi) = v4;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SL::kOFree));
            }
            if (lane == 0) tma_store_wait_all();  // the stores are complete before the CTA exits
        }
    } else if (!EW || warp < 12) {
        if constexpr (EW)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
        else
            asm volatile("setmaxnreg.inc.sync.aligned.u32 208;" ::: "memory");
        // ------------------------------------------------------------ softmax + epilogue
        const int half = (warp - 4) >> 2;         // this thread's chunks: half, half+2, ...
        const int quarter = warp & 3;             // TMEM lanes this warp may access
        const int row = quarter * 32 + lane;      // MMA row == TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t t_lane = tmem + lane_addr;
        const int prow = row >> p.g_log2;         // position offset within the tile
        const int hrow = row & (p.G - 1);         // head offset within the group
        float *red = reinterpret_cast<float *>(gbase + SL::kRed);    // [2][2][128]
        float *redl = reinterpret_cast<float *>(gbase + SL::kRedL);  // [2][2][128]
        uint32_t g = 0, uc = 0;

        // The epilogue of a unit (O / l -> 16-bit -> global, LSE) is deferred
        // into the first tile of the next unit: that tile's scores and
        // weights are computed while the previous unit's last P V runs, and
        // O is read out just before the new P is written.
        bool pend = false, pend_valid = false;
        int pend_b = 0, pend_kvh = 0, pend_t = 0, pend_t0 = 0, pend_t1 = 0, pend_r0 = 0;
        float pend_m = 0.f, pend_l = 0.f;
        uint32_t ep = 0;  // staged epilogues so far
        auto epilogue = [&](float l_tot, uint32_t ob) {
            const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
            const bool ok = !*abort_flag;
            if constexpr (kStageOut) {
                // Stage O / l as 16-bit values in the 128-byte-swizzled layout of the
                // output box (row r = MMA row: position r/G, head r%G); warp 3
                // stores the whole unit with one TMA tensor store per 64-column
                // slab (rows past the sequence end fall outside the tensor and
                // are not written), so no softmax warp waits on the store.
                const uint32_t stage = base + SL::kStageO;
                // the previous unit's stores have read the buffer
                mbar_wait(bar(SL::kOFree), (ep & 1u) ^ 1u, &g_prefill_error, abort_flag);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t r[32];
                    tmem_ld32(t_lane + kTO + (DB ? ob * D : 0u) + half * (D / 2) + 32 * c, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w4[e] = pack2<DT>(__uint_as_float(r[8 * v + 2 * e]) * inv_l,
                                                __uint_as_float(r[8 * v + 2 * e + 1]) * inv_l);
                        const int col = half * (D / 2) + 32 * c + 8 * v;  // first column
                        const int ci = (col & 63) >> 3;                   // 16-byte chunk in the row
                        const uint32_t addr = stage + (col >> 6) * (128 * 128) + row * 128 +
                                              ((ci ^ (row & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                     "r"(w4[0]), "r"(w4[1]), "r"(w4[2]), "r"(w4[3])
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SL::kOStaged));  // warp 3 stores it
                ++ep;
                if (p.lse != nullptr && ok && pend_valid && half == 0) {
                    const int h = pend_kvh * p.G + hrow;
                    const int64_t li = (static_cast<int64_t>(pend_b) * p.Hq + h) * p.L + (pend_r0 + pend_t - p.q_off);
                    if (in_bounds(li, p.n_lse, &g_prefill_error, &g_prefill_where))
                        p.lse[li] = pend_m * p.scale + logf(l_tot);
                }
                return;
            }
            // This thread's half row of O / l as CH 16-byte chunks of 16-bit values.
            constexpr int CH = D / 16;
            uint4 ch[CH];
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t r[32];
                tmem_ld32(t_lane + kTO + (DB ? ob * D : 0u) + half * (D / 2) + 32 * c, r);
                tmem_wait_ld();
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w4[e] = pack2<DT>(__uint_as_float(r[8 * v + 2 * e]) * inv_l,
                                            __uint_as_float(r[8 * v + 2 * e + 1]) * inv_l);
                    ch[4 * c + v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            }
            // Transpose the CH x CH chunks within each group of CH lanes
            // (butterfly over lane bits): afterwards lane CH*k + c holds chunk c
            // of the warp's rows CH*k + v in ch[v].  Each store below then
            // writes CH consecutive chunks of one half row -- whole 128-byte
            // lines -- instead of one chunk in each of 32 lines.
#pragma unroll
            for (int dd = CH / 2; dd >= 1; dd >>= 1) {
                const bool upper = (lane & dd) != 0;
#pragma unroll
                for (int lo = 0; lo < CH; ++lo) {
                    if (lo & dd) continue;
                    const int hi = lo | dd;
                    const uint4 snd = upper ? ch[lo] : ch[hi];
                    uint4 rcv;
                    rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, dd);
                    rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, dd);
                    rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, dd);
                    rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, dd);
                    if (upper)
                        ch[lo] = rcv;
                    else
                        ch[hi] = rcv;
                }
            }
            const int kgrp = lane / CH, cpos = lane % CH;
#pragma unroll
            for (int v = 0; v < CH; ++v) {
                const int rr = quarter * 32 + kgrp * CH + v;  // MMA row of ch[v]
                const int tv = pend_t0 + (rr >> p.g_log2);
                const int64_t oi =
                    ((static_cast<int64_t>(pend_b) * p.L + (pend_r0 + tv - p.q_off)) * p.Hq + pend_kvh * p.G +
                     (rr & (p.G - 1))) * D + half * (D / 2) + cpos * 8;
                if (ok && tv <= pend_t1 && in_bounds(oi / 8, p.n_o / 8, &g_prefill_error, &g_prefill_where))
                    *reinterpret_cast<uint4 *>(p.o + oi) = ch[v];
            }
            if (p.lse != nullptr && ok && pend_valid && half == 0) {
                const int h = pend_kvh * p.G + hrow;
                const int64_t li = (static_cast<int64_t>(pend_b) * p.Hq + h) * p.L + (pend_r0 + pend_t - p.q_off);
                if (in_bounds(li, p.n_lse, &g_prefill_error, &g_prefill_where))
                    p.lse[li] = pend_m * p.scale + logf(l_tot);
            }
        };

        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++uc) {
            const Unit x = unit_geom<KT, VL>(u, p, n_units);
            const int t = x.t0 + prow;
            const bool row_valid = (t <= x.t1);
            const int lo_t = p.w < 0 ? 0 : max(p.s, t - (p.w - p.s) + 1);
            float m_run = -INFINITY;
            float l_half = 0.f;

            for (int j = 0; j < x.n_tiles; ++j, ++g) {
                mbar_wait(bar(SL::kSFull), g & 1, &g_prefill_error, abort_flag);
                tc_fence_after_sync();
                // this thread's chunks: columns 32*(half + 2i) .. +31, i = 0..3
                uint32_t sr[NC][32];
#pragma unroll
                for (int i = 0; i < NC; ++i) tmem_ld32(t_lane + kTmemS + 32 * (half + 2 * i), sr[i]);
                // column c of this tile is attended when c is in the band
                // [c_lo, c_hi] or among the sinks [0, sink_hi)
                const int key0 = x.lo + KT * j - p.s_pad;
                int c_lo = max(j == 0 ? p.s_pad : 0, lo_t - key0);
                int c_hi = min(t - key0, KT - 1);
                int sink_hi = (j == 0) ? min(p.s, t + 1) : 0;
                if (!row_valid) {
                    c_lo = KT;
                    c_hi = -1;
                    sink_hi = 0;
                }
                const bool band_ok = c_lo <= c_hi;
                bool full[NC], empty[NC];
                // this thread's last chunk has only 16 columns (warp-uniform)
                const bool short_tail = kShortTail && half == 1;
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    const int c0 = 32 * (half + 2 * i);
                    const int cw = (short_tail && i == NC - 1) ? 16 : 32;
                    const bool f = band_ok && c_lo <= c0 && c_hi >= c0 + cw - 1;
                    const bool e = (!band_ok || c_hi < c0 || c_lo > c0 + 31) && sink_hi <= c0;
                    full[i] = __all_sync(0xffffffffu, f);
                    empty[i] = __all_sync(0xffffffffu, e);
                }
                tmem_wait_ld();
                // S has been read: the S issuer may compute the next S now.
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SL::kSEmpty));

                float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    if (empty[i]) continue;
                    if (!full[i]) {
                        // attended columns of this chunk as a bit mask: the band
                        // [c_lo, c_hi] and the sinks [0, sink_hi), clipped to it
                        const int c0 = 32 * (half + 2 * i);
                        const int lo = max(c_lo - c0, 0), hi = min(c_hi - c0, 31);
                        uint32_t vb = (band_ok && lo <= hi) ? ((0xFFFFFFFFu >> (31 - (hi - lo))) << lo) : 0u;
                        const int ns = sink_hi - c0;
                        vb |= ns <= 0 ? 0u : (ns >= 32 ? 0xFFFFFFFFu : ((1u << ns) - 1u));
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (!(vb & (1u << e))) sr[i][e] = __float_as_uint(-INFINITY);
                    }
                    // elements 0..1, then 2..13 four at a time, then 14..15;
                    // the same for 16..31 unless the chunk has 16 columns
                    float a = __uint_as_float(sr[i][0]), b = __uint_as_float(sr[i][1]);
#pragma unroll
                    for (int e = 2; e < 14; e += 4) {
                        a = fmax3(a, __uint_as_float(sr[i][e]), __uint_as_float(sr[i][e + 1]));
                        b = fmax3(b, __uint_as_float(sr[i][e + 2]), __uint_as_float(sr[i][e + 3]));
                    }
                    a = fmax3(a, __uint_as_float(sr[i][14]), __uint_as_float(sr[i][15]));
                    if (!(short_tail && i == NC - 1)) {
#pragma unroll
                        for (int e = 16; e < 32; e += 4) {
                            a = fmax3(a, __uint_as_float(sr[i][e]), __uint_as_float(sr[i][e + 1]));
                            b = fmax3(b, __uint_as_float(sr[i][e + 2]), __uint_as_float(sr[i][e + 3]));
                        }
                    }
                    mx_a = fmaxf(mx_a, a);
                    mx_b = fmaxf(mx_b, b);
                }
                // Row max over both halves through shared memory, one barrier
                // per tile (buffers alternate with the tile parity); the first
                // tile of a unit also exchanges the previous unit's row sums.
                float *rm = red + (g & 1) * 256;
                float *rl = redl + ((uc - 1) & 1) * 256;
                rm[half * 128 + row] = fmaxf(mx_a, mx_b);
                const bool do_epi = !EW && j == 0 && pend;
                if (do_epi) rl[half * 128 + row] = pend_l;
                asm volatile("bar.sync 1, 256;" ::: "memory");
                const float mx = fmaxf(rm[row], rm[128 + row]);
                const float l_prev = do_epi ? rl[row] + rl[128 + row] : 0.f;
                const float m_new = fmaxf(m_run, mx);
                float alpha = 1.f;
                if (m_new > m_run &&
                    (m_run == -INFINITY || (m_new - m_run) * p.scale_log2 > 8.f)) {
                    alpha = ex2_approx((m_run - m_new) * p.scale_log2);
                    m_run = m_new;
                }
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run * p.scale_log2;
                const uint64_t sc2 = f32x2(p.scale_log2, p.scale_log2);
                const uint64_t nm2 = f32x2(neg_m, neg_m);
                uint64_t l2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
                uint32_t pk[NC][16];
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    if (empty[i]) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) pk[i][e] = 0u;
                        continue;
                    }
                    auto pair = [&](int e) {
                        float a0, a1;
                        f32x2_split(fma_f32x2(f32x2(__uint_as_float(sr[i][2 * e]),
                                                    __uint_as_float(sr[i][2 * e + 1])),
                                              sc2, nm2),
                                    a0, a1);
                        a0 = ex2_approx(a0);
                        a1 = ex2_approx(a1);
                        pk[i][e] = pack2<DT>(a0, a1);
                        l2[e & 1] = add_f32x2(l2[e & 1], f32x2(a0, a1));
                    };
#pragma unroll
                    for (int e = 0; e < 8; ++e) pair(e);
                    if (short_tail && i == NC - 1) {
#pragma unroll
                        for (int e = 8; e < 16; ++e) pk[i][e] = 0u;
                    } else {
#pragma unroll
                        for (int e = 8; e < 16; ++e) pair(e);
                    }
                }
                float lx, ly, lz, lw;
                f32x2_split(l2[0], lx, ly);
                f32x2_split(l2[1], lz, lw);
                l_half = l_half * alpha + ((lx + ly) + (lz + lw));
                // The P buffer may be written once the P V that last read it
                // (tile g-1, or g-2 with two buffers) has completed; with one
                // O buffer the previous unit's O is read out first.
                if (DB) {
                    if (g >= 2)
                        mbar_wait(bar(SL::kPVDone + (g & 1)), ((g - 2) >> 1) & 1, &g_prefill_error,
                                  abort_flag);
                } else if (g > 0) {
                    mbar_wait(bar(SL::kPVDone), (g - 1) & 1, &g_prefill_error, abort_flag);
                }
                tc_fence_after_sync();
                if (!DB && do_epi) {
                    epilogue(l_prev, 0);
                    pend = false;
                }
#pragma unroll
                for (int i = 0; i < NC; ++i)
                    tmem_st16(t_lane + kTP + (DB ? (g & 1) * 64 : 0u) + 16 * (half + 2 * i), pk[i]);
                // Rescale O when this warp raised any running max (not on the
                // first tile: its P V overwrites O), after the previous P V
                // into it completed.  Each half owns d/2 columns.
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    if (DB) {
                        mbar_wait(bar(SL::kPVDone + ((g - 1) & 1)), ((g - 1) >> 1) & 1,
                                  &g_prefill_error, abort_flag);
                        tc_fence_after_sync();
                    }
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        uint32_t r[32];
                        const uint32_t ta =
                            t_lane + kTO + (DB ? (uc & 1) * D : 0u) + half * (D / 2) + 32 * c;
                        tmem_ld32(ta, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                        tmem_st32(ta, r);
                    }
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar((g & 1) ? SL::kPFull1 : SL::kPFull));
                // With two O buffers the previous unit's epilogue runs here,
                // beside this tile's P V, once that unit's last P V is done.
                if (DB && do_epi) {
                    mbar_wait(bar(SL::kPVDone + ((g - 1) & 1)), ((g - 1) >> 1) & 1,
                              &g_prefill_error, abort_flag);
                    tc_fence_after_sync();
                    epilogue(l_prev, (uc - 1) & 1);
                    pend = false;
                }
            }
            if constexpr (EW) {
                // Hand the unit to the epilogue warpgroup: its row max and the
                // two halves' sums, in the buffers of this unit's parity (read
                // out for unit uc-2 by now, in all but the rarest case).
                if (uc >= 2)
                    mbar_wait(bar(SL::kORead + (uc & 1)), ((uc >> 1) & 1) ^ 1, &g_prefill_error,
                              abort_flag);
                float *epm = reinterpret_cast<float *>(gbase + SL::kEpiM);
                if (half == 0) epm[(uc & 1) * 128 + row] = m_run;
                redl[(uc & 1) * 256 + half * 128 + row] = l_half;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SL::kEpiReady + (uc & 1)));
                continue;
            }
            pend = true;
            pend_valid = row_valid;
            pend_b = x.b;
            pend_r0 = x.r0;
            pend_kvh = x.kvh;
            pend_t = t;
            pend_t0 = x.t0;
            pend_t1 = x.t1;
            pend_m = m_run;
            pend_l = l_half;
        }
        if (pend) {  // the last unit's epilogue
            float *rl = redl + ((uc - 1) & 1) * 256;
            rl[half * 128 + row] = pend_l;
            if (DB)
                mbar_wait(bar(SL::kPVDone + ((g - 1) & 1)), ((g - 1) >> 1) & 1, &g_prefill_error,
                          abort_flag);
            else
                mbar_wait(bar(SL::kPVDone), (g - 1) & 1, &g_prefill_error, abort_flag);
            tc_fence_after_sync();
            asm volatile("bar.sync 1, 256;" ::: "memory");
            epilogue(rl[row] + rl[128 + row], (uc - 1) & 1);
        }
    } else if constexpr (EW) {
        if constexpr (VL)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 40;" ::: "memory");
        else
            asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
        // ------------------------------------------------------------ epilogue warpgroup
        // One thread per MMA row (TMEM lane): for each unit, once the softmax
        // has handed over its row max and sums and its last P V is complete,
        // O / l goes to the staging buffer as 16-bit values in the
        // 128-byte-swizzled layout of the output box, and warp 3 stores it.
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const float *epm = reinterpret_cast<const float *>(gbase + SL::kEpiM);
        const float *epl = reinterpret_cast<const float *>(gbase + SL::kRedL);
        const uint32_t stage = base + SL::kStageO;
        uint32_t uc = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++uc) {
            const uint32_t ob = uc & 1, ph = (uc >> 1) & 1;
            mbar_wait(bar(SL::kEpiReady + ob), ph, &g_prefill_error, abort_flag);
            mbar_wait(bar(SL::kOFull + ob), ph, &g_prefill_error, abort_flag);
            // the previous unit's stores have read the staging buffer
            mbar_wait(bar(SL::kOFree), ob ^ 1u, &g_prefill_error, abort_flag);
            tc_fence_after_sync();
            const float m = epm[ob * 128 + row];
            const float l = epl[ob * 256 + row] + epl[ob * 256 + 128 + row];
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                uint32_t r[16];
                tmem_ld16(t_lane + kTO + ob * D + 16 * c, r);
                tmem_wait_ld();
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w4[e] = pack2<DT>(__uint_as_float(r[8 * v + 2 * e]) * inv_l,
                                          __uint_as_float(r[8 * v + 2 * e + 1]) * inv_l);
                    const int col = 16 * c + 8 * v;  // first column
                    const int ci = (col & 63) >> 3;  // 16-byte chunk in the row
                    const uint32_t addr =
                        stage + (col >> 6) * (128 * 128) + row * 128 + ((ci ^ (row & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w4[0]),
                                 "r"(w4[1]), "r"(w4[2]), "r"(w4[3])
                                 : "memory");
                }
            }
            // O, m and l are read: the P V issuer may start unit uc+2 in this
            // O buffer and the softmax may hand it over
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(SL::kORead + ob));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(SL::kOStaged));  // warp 3 stores it
            if (p.lse != nullptr && !*abort_flag) {
                const Unit x = unit_geom<KT, VL>(u, p, n_units);
                const int t = x.t0 + (row >> p.g_log2);
                if (t <= x.t1) {
                    const int h = x.kvh * p.G + (row & (p.G - 1));
                    const int64_t li = (static_cast<int64_t>(x.b) * p.Hq + h) * p.L + (x.r0 + t - p.q_off);
                    if (in_bounds(li, p.n_lse, &g_prefill_error, &g_prefill_where))
                        p.lse[li] = m * p.scale + logf(l);
                }
            }
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

template <int D, int KT, int NSK, int NSV, int DT, bool VL, bool EW>
swa_status launch_prefill(const PrefillMaps &maps, const PrefillParams &p, cudaStream_t stream) {
    using SL = PrefillSmem<D, KT, NSK, NSV, EW>;
    static_assert(SL::kAlloc <= 232448, "shared memory per CTA");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    static bool configured[64] = {};
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(swa_prefill_kernel<D, KT, NSK, NSV, DT, VL, EW>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SL::kAlloc);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill)");
        configured[dev] = true;
    }
    const int sms = device_sm_count();
    if (sms <= 0) return cuda_fail(cudaErrorInvalidDevice, "device_sm_count");
    const int grid = p.n_units < sms ? p.n_units : sms;
    e = launch_pdl(swa_prefill_kernel<D, KT, NSK, NSV, DT, VL, EW>, dim3(grid),
                   dim3(prefill_threads(EW)), SL::kAlloc,
                   stream, maps, p);
    return e == cudaSuccess ? SWA_OK : cuda_fail(e, "launch swa_prefill_kernel");
}

}  // namespace

// Key tile width for a call, from the widest unit's span of key columns:
//   narrow: tiles with double-buffered P and O and the output staged for TMA
//           stores; at d = 128 they are 112 columns, whose 28 KB K and V
//           tiles leave room for two stages of each beside the 32 KB staged
//           output tile; at d = 64, 128 columns with four stages of each;
//   else:   256 (one tile fills the MMA's N = 256).
// Narrow up to 1280 columns at d = 128 and 768 at d = 64.  Measured on GB300
// (TFLOP/s, narrow / 256-column tiles): d = 128, Hq 32, Hkv 8: SWA(512,4)
// 990 / 825, SWA(768,4) 1018 / 968, SWA(1024,4) 1097 / 1055, SWA(2048,4)
// 1196 / 1239, full causal 1219 / 1412; d = 64, 16 heads: SWA(1024,4)
// 529 / 581, full causal 703 / 781.
// At d = 64 the 256-column tiles also pay when they cover a unit in half as
// many tiles as 128-column ones, at least four of those (the same columns
// computed, half the per-tile work of the softmax chain).  Kernel alone, 16
// heads of 64, fp16, L = 32768, µs (128 / 256-column tiles): SWA(128,4)
// 78.0 / 91.6 (3 / 2 tiles), SWA(256,4) 101.3 / 95.1 (4 / 2), SWA(384,4)
// 124.4 / 132.5 (5 / 3), SWA(512,4) 147.7 / 135.3 (6 / 3); SWA(64,4)
// 57.5 / 62.0 (2 / 1).
int prefill_key_tile(const PrefillParams &p, int d) {
    if (SWA_PREFILL_FORCE_KT != 0) return SWA_PREFILL_FORCE_KT;
    const long long cols =
        p.w < 0 ? static_cast<long long>(p.Lk) : static_cast<long long>(p.s_pad) + (p.w - p.s) + p.P - 1;
    if (cols > (d == 128 ? 1280 : 768)) return 256;
    if (d == 64) {
        const long long n128 = (cols + 127) / 128, n256 = (cols + 255) / 256;
        if (n128 >= 4 && 2 * n256 == n128) return 256;
    }
    return d == 128 ? 112 : 128;
}

namespace {

template <int DT, bool VL>
swa_status launch_prefill_dt(const PrefillMaps &maps, const PrefillParams &p, int d, int kt,
                             bool ew, cudaStream_t stream) {
    if (d == 128) {
        if (kt == 256) return launch_prefill<128, 256, 1, 1, DT, VL, false>(maps, p, stream);
        return ew ? launch_prefill<128, 112, 2, 2, DT, VL, true>(maps, p, stream)
                  : launch_prefill<128, 112, 2, 2, DT, VL, false>(maps, p, stream);
    }
    if (kt == 256) return launch_prefill<64, 256, 2, 2, DT, VL, false>(maps, p, stream);
    return ew ? launch_prefill<64, 128, 4, 4, DT, VL, true>(maps, p, stream)
              : launch_prefill<64, 128, 4, 4, DT, VL, false>(maps, p, stream);
}

}  // namespace

namespace {

// The widths that have a kernel: 112 or 256 at d = 128, 128 or 256 at d = 64.
int kernel_key_tile(const PrefillParams &p, int d) {
    const int kt = prefill_key_tile(p, d);
    return kt == 256 ? 256 : (d == 128 ? 112 : 128);
}

// The epilogue warpgroup for narrow tiles: it takes the unit epilogue
// (about 0.3 µs per unit) off the softmax warps, which pays when units span
// several key tiles; with single-tile units its extra stage per unit costs
// more than it saves unless a CTA runs very many of them.  Measured on GB300
// (without / with; Hq=32 Hkv=8 d=128 unless noted):
//   SWA(512,4): L=6144 61.5 / 58.9 µs, L=12288 113.0 / 106.5 µs, B=2
//     L=32768 990 / 1061 TFLOP/s; 16 heads of 64, fp16: L=8192 49.2 / 45.4
//     µs, L=32768 161.8 / 151.6 µs;
//   SWA(64,4), one tile per unit: L=4096 20.5 / 22.5 µs, L=12288 43.0 /
//     45.1 µs, B=2 L=32768 (108 units per SM) 207.9 / 202.8 µs.
bool use_epilogue_wg(const PrefillParams &p, int kt) {
    if (kt == 256 || SWA_PREFILL_EPI_WG == 0) return false;
    if (SWA_PREFILL_EPI_WG == 2) return true;
    const long long cols =
        p.w < 0 ? static_cast<long long>(p.Lk) : static_cast<long long>(p.s_pad) + (p.w - p.s) + p.P - 1;
    if (cols > kt) return true;  // several key tiles per unit
    const int sms = device_sm_count();
    return sms > 0 && static_cast<long long>(p.n_units) >= 64ll * sms;
}

// ---------------------------------------------------------------------------
// varlen planning: one CTA checks cu_seqlens and writes the query-tile records
// ---------------------------------------------------------------------------
// tile_off[b] = query tiles of sequences 0..b-1 (tile_off[B]: all of them, or
// 0 when cu_seqlens is not a valid partition of [0, total) or the tiles
// exceed tiles_max, which also records SWA_ERR_BOUNDS); tile_rec[T] =
// {b, tile index in b, first row of b, length of b}.
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) swa_varlen_plan_kernel(
    const int *cu, int B, int total, int P, int tiles_max, int *tile_off, int4 *tile_rec) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int s_warp[kPlanThreads / 32];
    __shared__ int s_carry, s_bad;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        s_carry = 0;
        s_bad = (cu[0] != 0 || cu[B] != total) ? 1 : 0;
    }
    __syncthreads();
    for (int b0 = 0; b0 < B; b0 += kPlanThreads) {
        const int b = b0 + tid;
        int tiles = 0;
        if (b < B) {
            const int len = cu[b + 1] - cu[b];
            if (len < 0) s_bad = 1;
            tiles = len > 0 ? (len + P - 1) / P : 0;
        }
        // inclusive scan of tiles over the block: within warps, then of warp sums
        int incl = tiles;
#pragma unroll
        for (int dd = 1; dd < 32; dd <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, dd);
            if (lane >= dd) incl += y;
        }
        if (lane == 31) s_warp[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            int ws = s_warp[lane];
#pragma unroll
            for (int dd = 1; dd < 32; dd <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, ws, dd);
                if (lane >= dd) ws += y;
            }
            s_warp[lane] = ws;  // inclusive warp prefix
        }
        __syncthreads();
        const int before = s_carry + (wid > 0 ? s_warp[wid - 1] : 0) + incl - tiles;
        if (b < B) tile_off[b] = before;
        __syncthreads();
        if (tid == kPlanThreads - 1) s_carry = before + tiles;
        __syncthreads();
    }
    const bool ok = !s_bad && s_carry <= tiles_max;
    if (tid == 0) {
        tile_off[B] = ok ? s_carry : 0;
        if (!ok) atomicCAS(&g_prefill_error, 0, kErrBounds);
    }
    if (!ok) return;
    __syncthreads();  // tile_off is written (global memory, same CTA)
    // one warp per sequence writes its records
    for (int b = wid; b < B; b += kPlanThreads / 32) {
        const int off = tile_off[b], row0 = cu[b], len = cu[b + 1] - row0;
        const int tiles = len > 0 ? (len + P - 1) / P : 0;
        for (int qt = lane; qt < tiles; qt += 32) tile_rec[off + qt] = make_int4(b, qt, row0, len);
    }
}

}  // namespace

size_t varlen_workspace_bytes(int B, int total, int Hq, int Hkv) {
    if (B < 1 || total < 0 || Hkv < 1 || Hq < Hkv) return 0;
    const int P = 128 / (Hq / Hkv);
    const size_t off_bytes = (static_cast<size_t>(B) + 1) * 4;
    const size_t tiles_max = static_cast<size_t>(B) + (static_cast<size_t>(total) + P - 1) / P;
    return ((off_bytes + 15) & ~static_cast<size_t>(15)) + tiles_max * 16;
}

swa_status prefill_varlen_launch(const void *q, const void *k, const void *v, void *o, float *lse,
                                 const int32_t *cu_seqlens, int B, int total, int max_len, int Hq,
                                 int Hkv, int d, int w, int s, int dtype, void *workspace,
                                 cudaStream_t stream) {
    PrefillParams p = make_prefill_params(o, lse, 1, total, Hq, Hkv, d, w, s, 0, total);
    const size_t off_bytes = ((static_cast<size_t>(B) + 1) * 4 + 15) & ~static_cast<size_t>(15);
    int *tile_off = static_cast<int *>(workspace);
    int4 *tile_rec = reinterpret_cast<int4 *>(static_cast<char *>(workspace) + off_bytes);
    const int tiles_max = B + (total + p.P - 1) / p.P;
    p.varlen = 1;
    p.tile_count = tile_off + B;
    p.tile_rec = tile_rec;
    p.n_units = tiles_max * Hkv;  // an upper bound, for the grid
    p.n_qtiles = 0;
    cudaError_t e = launch_pdl(swa_varlen_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream,
                               reinterpret_cast<const int *>(cu_seqlens), B, total, p.P, tiles_max,
                               tile_off, tile_rec);
    if (e != cudaSuccess) return cuda_fail(e, "launch swa_varlen_plan_kernel");
    // key tile width from the widest unit (max_len bounds it for w = infinity)
    PrefillParams span = p;
    span.Lk = max_len;
    const int kt = kernel_key_tile(span, d);
    PrefillMaps maps;
    if (!encode_prefill_maps(&maps, q, k, v, p, d, kt, dtype, 0))
        return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
    const bool ew = use_epilogue_wg(span, kt);
    return dtype == SWA_F16 ? launch_prefill_dt<kF16, true>(maps, p, d, kt, ew, stream)
                            : launch_prefill_dt<kBf16, true>(maps, p, d, kt, ew, stream);
}

swa_status prefill_launch_offset(const void *q, const void *k, const void *v, void *o, float *lse,
                                 int B, int L, int Hq, int Hkv, int d, int w, int s, int q_off,
                                 int Lk, int kv_cap, int dtype, cudaStream_t stream) {
    const PrefillParams p = make_prefill_params(o, lse, B, L, Hq, Hkv, d, w, s, q_off, Lk);
    const int kt = kernel_key_tile(p, d);
    PrefillMaps maps;
    if (!encode_prefill_maps(&maps, q, k, v, p, d, kt, dtype, kv_cap))
        return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
    const bool ew = use_epilogue_wg(p, kt);
    return dtype == SWA_F16 ? launch_prefill_dt<kF16, false>(maps, p, d, kt, ew, stream)
                            : launch_prefill_dt<kBf16, false>(maps, p, d, kt, ew, stream);
}

swa_status prefill_launch(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                          int L, int Hq, int Hkv, int d, int w, int s, int dtype,
                          cudaStream_t stream) {
    return prefill_launch_offset(q, k, v, o, lse, B, L, Hq, Hkv, d, w, s, 0, L, 0, dtype, stream);
}

long long prefill_read_clear_where(cudaStream_t stream) {
    unsigned long long w = 0;
    return read_clear_symbol(g_prefill_where, &w, stream) ? where_index(w) : -2;
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
