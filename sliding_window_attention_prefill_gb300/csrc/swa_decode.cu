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
// The path is bound by HBM bandwidth: each K/V byte is used by the G query
// heads of its group and nothing else.  The work is a list of items
// (sequence, kv head, split of the filled slots); a persistent grid of CTAs
// walks it with a stride of gridDim.x.  In each CTA a producer warp streams
// the K and V rows of its items in 64-slot chunks, back to back across item
// boundaries, into shared memory with 2-D TMA copies (128-byte swizzle,
// mbarrier ring of 1, 2 or 3 stages); q of the item rides along with its
// first chunk.  Four consumer warps use the warp-level tensor-core MMA
// (mma.sync m16n8k16, bf16 or fp16 in, fp32 accumulate) for both products
// with the G <= 8 heads as the N = 8 dimension:
//   S^T [16 slots x 8 heads] = K [16 x d] . Q^T [d x 8]      (K via ldmatrix)
//   O^T [d/4 x 8 heads]     += V^T [d/4 x 64] . P^T [64 x 8] (V via ldmatrix.trans)
// Warp w computes the scores of slots 16w .. 16w+15 and puts them in shared
// memory; after one barrier per chunk every warp runs the online softmax over
// all 64 slots (running max raised only when it grows by more than 2^8, which
// keeps the rescale rare and is exact) and accumulates its quarter of d, so
// no merge across warps is needed at the end of an item.  With several
// splits per (sequence, kv head) the items write fp32 partials (max, sum,
// weighted values) and a second kernel merges them: m = max m_j,
// l = sum l_j 2^(m_j - m), o = sum acc_j 2^(m_j - m) / l.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "swa_internal.h"
#include "swa_ptx.cuh"

namespace swa {

__device__ int g_decode_error;
__device__ unsigned long long g_decode_where;

#ifndef SWA_DEC_ITEMS_PER_SM
#define SWA_DEC_ITEMS_PER_SM 4
#endif
#ifndef SWA_DEC_CTAS_PER_SM
#define SWA_DEC_CTAS_PER_SM 2
#endif
#ifndef SWA_DEC_CTAS_PER_SM_SINGLE
#define SWA_DEC_CTAS_PER_SM_SINGLE 4
#endif
#ifndef SWA_DEC_CTAS_PER_SM_WIDE
#define SWA_DEC_CTAS_PER_SM_WIDE 3
#endif

// Persistent CTAs per SM: the 1-stage chunk ring (items of one chunk), and
// the rings of several stages -- SWA_DEC_CTAS_PER_SM, or
// SWA_DEC_CTAS_PER_SM_WIDE with two stages when a call has at least two items
// per CTA at that count (more chunks in flight per SM) and its shared memory
// fits.
constexpr int kDecCtasPerSm[2] = {SWA_DEC_CTAS_PER_SM_SINGLE, SWA_DEC_CTAS_PER_SM};
constexpr int kDecCH = 64;              // slots per chunk
constexpr int kDecWarps = 4;            // consumer warps, 16 slots each
constexpr int kDecThreads = 32 * (kDecWarps + 1);

struct DecodeMaps {
    CUtensorMap k, v;  // 2-D: {d, B*Hkv*cap rows}, box {64, 64}, 128-byte swizzle
};

struct DecodeParams {
    const uint16_t *q;   // [B, Hq, D] bf16 or fp16
    const int32_t *pos;  // [B]
    uint16_t *o;         // [B, Hq, D]
    float *ws_acc;       // [B*Hq, splits, D]
    float *ws_ml;        // [B*Hq, splits, 2]
    int B, Hq, Hkv, cap, w, splits;
    float scale_log2;
    // hybrid window + linear decode: partials even with one split, and the
    // linear state the merge adds (S [B*Hkv, 2 df, D], z [B*Hkv, 2 df],
    // feature weights W [Hkv, D, df])
    int partials;
    const float *S, *z, *W;
    // append + decode: the new token of each sequence ([B, Hkv, D]) goes to
    // its slot of the cache (kc, vc) and into the staged chunk that holds it
    const uint16_t *k_new, *v_new;
    uint16_t *kc, *vc;
    int s;
    // extents in elements (bounds-checked build): o, the cache tensors, the
    // new tokens, the workspace's partials and (max, sum) pairs
    long long n_o, n_cache, n_new, n_ws_acc, n_ws_ml;
};

// ST: depth of the chunk ring (1 when every item is a single chunk, which
// leaves room for more CTAs per SM; 2 or 3 when items span several chunks).
template <int D, int G, int ST>
struct DecSmem {
    static constexpr int kRegion = kDecCH * 128;            // 64 rows x 64 columns (bf16)
    static constexpr int kChunkBytes = (D / 64) * kRegion;  // one of K or V
    static constexpr int kQBytes = G * D * 2;               // q of the G heads of the item
    static constexpr int kNewBytes = 2 * D * 2;             // the appended token's k and v rows
    // K | V | q | k_new v_new (q and the new rows with an item's first chunk)
    static constexpr int kStage = 2 * kChunkBytes + ((kQBytes + kNewBytes + 1023) & ~1023);
    static constexpr int kSxRow = kDecCH + 8;       // one head's scores of a chunk (padded)
    static constexpr int kSx = ST * kStage;         // [2 chunk parity][8 heads][kSxRow] f32
    static constexpr int kOst = kSx + 2 * 8 * kSxRow * 4;  // [warp][G][D / 4] 16-bit output
    // full_k[st], full_v[st], empty_k[st], empty_v[st]
    static constexpr int kBar = kOst + kDecWarps * G * (D / kDecWarps) * 2;
    static constexpr int kAbort = kBar + 4 * ST * 8;
    static constexpr int kBytes = kAbort + 16;
    static constexpr int kAlloc = kBytes + 1024;              // align the base to 1024
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

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, uint32_t bar, int c0,
                                            int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D (16x8 fp32) += A (16x16, row) * B (16x8, col); A and B bf16 or fp16 (DT).
template <int DT>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    if constexpr (DT == kBf16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Address of 16-byte chunk `cc` (of the row's d/8) of chunk row `row` in a
// stage laid out by the 128-byte-swizzled TMA box.
__device__ __forceinline__ uint32_t swz(uint32_t stage, int row, int cc) {
    return stage + (cc >> 3) * (kDecCH * 128) + row * 128 + ((((cc & 7) ^ (row & 7))) << 4);
}

// One work item: the slots [begin, end) of (sequence b, kv head kvh) that
// split `split` covers, of which those below n_valid = min(pos + 1, cap_eff)
// are filled.
//   Finite window: the splits partition [0, w) whatever the position, so an
//   item's first chunk is known before pos is read; the producer issues it
//   at once (spec) and reads pos while it is in flight.  Slots at or past
//   n_valid (a cache not yet full) are masked.
//   Infinite window: the splits partition [0, n_valid); only split 0's first
//   chunk (slots 0..63) is known in advance.
// n_chunks counts the chunks both sides walk: those holding filled slots,
// and at least the speculative one.  A position outside the cache (bad) is
// recorded as an error; its chunks are consumed and nothing is written.
struct DecItem {
    int b, kvh, split, begin, end, n_chunks, n_valid;
    int snew;  // append + decode: the new token's slot, else -1
    bool bad, spec;
};

__device__ __forceinline__ DecItem dec_item_head(int it, const DecodeParams &p) {
    DecItem x;
    const int pair = it / p.splits;
    x.split = it - pair * p.splits;
    x.b = pair / p.Hkv;
    x.kvh = pair - x.b * p.Hkv;
    x.begin = x.end = x.n_chunks = x.n_valid = 0;
    x.snew = -1;
    x.bad = false;
    if (p.w >= 0) {
        int used;
        split_range(p.w, p.splits, x.split, x.begin, x.end, used);
        x.spec = x.end > x.begin;
    } else {
        x.spec = (x.split == 0);
    }
    return x;
}

// The position of item it's sequence.  With items of one chunk (a short
// chain per item) each side loads it one item ahead -- for it + gridDim.x
// while it works on it -- so the load's latency overlaps an item's work
// instead of preceding the next one.
__device__ __forceinline__ int dec_item_load_pos(int it, const DecodeParams &p) {
    return p.pos[(it / p.splits) / p.Hkv];
}

__device__ __forceinline__ void dec_item_pos(DecItem &x, const DecodeParams &p, int pos) {
    x.bad = pos < 0 || (p.w < 0 && pos >= p.cap);
    const int cap_eff = p.w < 0 ? p.cap : p.w;
    x.n_valid = x.bad ? 0 : min(pos + 1, cap_eff);
    if (p.w < 0) {
        int used;
        if (x.bad)
            x.begin = x.end = 0;
        else
            split_range(x.n_valid, p.splits, x.split, x.begin, x.end, used);
    }
    const int hi = min(x.end, x.n_valid);
    const int need = hi > x.begin ? (hi - x.begin + kDecCH - 1) / kDecCH : 0;
    x.n_chunks = max(need, x.spec ? 1 : 0);
    if (p.k_new != nullptr && !x.bad) {
        // slot(pos): the position itself below s (or for an infinite window),
        // else s + (pos - s) mod (w - s); this item holds it if it is in range
        const int sl = (p.w < 0 || pos < p.s) ? pos : p.s + (pos - p.s) % (p.w - p.s);
        if (sl >= x.begin && sl < hi) x.snew = sl;
    }
}

// Persistent: each CTA takes items blockIdx.x, blockIdx.x + gridDim.x, ...;
// the producer streams their chunks back to back, so the latency of the
// first loads is paid once per CTA rather than once per item.
// The minimum CTAs per SM of the launch bounds keeps the registers within
// what that many CTAs can hold (the grid assumes they are all resident).
// Most CTAs per SM a kernel of this shape may run at (its launch bounds).
template <int D, int G, int ST>
constexpr int dec_max_ctas() {
    if (ST == 1) return kDecCtasPerSm[0];
    return (SWA_DEC_CTAS_PER_SM_WIDE > SWA_DEC_CTAS_PER_SM &&
            SWA_DEC_CTAS_PER_SM_WIDE * (DecSmem<D, G, ST>::kAlloc + 1024) <= 233472)
               ? SWA_DEC_CTAS_PER_SM_WIDE
               : SWA_DEC_CTAS_PER_SM;
}

template <int D, int G, int ST, int DT>
__global__ void __launch_bounds__(kDecThreads, dec_max_ctas<D, G, ST>())
    swa_decode_kernel(const __grid_constant__ DecodeMaps maps, const DecodeParams p) {
    using SL = DecSmem<D, G, ST>;
    constexpr int kDecStages = ST;
    constexpr int KS = D / 16;  // k-steps of S, d-tiles of O
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SL::kAbort);
    // K and V of a stage fill and drain on barriers of their own: a stage's K
    // is released once the scores are computed, so the next chunk's K (and
    // its scores and softmax) can go ahead while this chunk's P V runs and
    // the next V loads.
    auto full_k = [&](int st) { return sbase + SL::kBar + 8u * st; };
    auto full_v = [&](int st) { return sbase + SL::kBar + 8u * (kDecStages + st); };
    auto empty_k = [&](int st) { return sbase + SL::kBar + 8u * (2 * kDecStages + st); };
    auto empty_v = [&](int st) { return sbase + SL::kBar + 8u * (3 * kDecStages + st); };
    const int n_items = p.B * p.Hkv * p.splits;
    constexpr bool kPosAhead = (ST == 1);
    pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int st = 0; st < kDecStages; ++st) {
            mbar_init(full_k(st), 1);
            mbar_init(full_v(st), 1);
            mbar_init(empty_k(st), kDecWarps);
            mbar_init(empty_v(st), kDecWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();  // the cache, q and pos are the previous kernels' from here on

    if (warp == kDecWarps) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&maps.k);
            tma_prefetch_desc(&maps.v);
            int cg = 0;  // chunks issued by this CTA
            bool ok = true;
            int pos_next = (kPosAhead && blockIdx.x < n_items) ? dec_item_load_pos(blockIdx.x, p) : 0;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
                DecItem x = dec_item_head(it, p);
                int pos_it = pos_next;
                if (kPosAhead) {
                    if (it + static_cast<int>(gridDim.x) < n_items) pos_next = dec_item_load_pos(it + gridDim.x, p);
                } else {
                    pos_it = p.pos[x.b];
                }
                const int row_base = (x.b * p.Hkv + x.kvh) * p.cap;  // row of slot 0
                const uint16_t *qsrc = p.q + (static_cast<int64_t>(x.b) * p.Hq + x.kvh * G) * D;
                // append + decode: the new token's k and v rows of this (b, kv head)
                const int64_t nsrc = (static_cast<int64_t>(x.b) * p.Hkv + x.kvh) * D;
                const bool stage_new = p.k_new != nullptr &&
                                       in_bounds(nsrc / 8 + D / 8 - 1, p.n_new / 8, &g_decode_error, &g_decode_where);
                // chunk c of the item into the next stage; q (and the new
                // token's rows) ride along with chunk 0
                auto issue = [&](int c) -> bool {
                    const int st = cg % kDecStages;
                    const uint32_t ph = ((cg / kDecStages) & 1) ^ 1;
                    const uint32_t stage = sbase + st * SL::kStage;
                    const int row = row_base + x.begin + c * kDecCH;
                    if (!mbar_wait(empty_k(st), ph, &g_decode_error, abort_flag)) return false;
                    mbar_arrive_expect_tx(full_k(st), SL::kChunkBytes +
                                                          (c == 0 ? SL::kQBytes + (stage_new ? SL::kNewBytes : 0) : 0));
#pragma unroll
                    for (int r = 0; r < D / 64; ++r)
                        tma_load_2d(stage + r * SL::kRegion, &maps.k, full_k(st), r * 64, row);
                    if (c == 0) {
                        bulk_load_1d(stage + 2 * SL::kChunkBytes, qsrc, SL::kQBytes, full_k(st));
                        if (stage_new) {
                            const uint32_t nd = stage + 2 * SL::kChunkBytes + SL::kQBytes;
                            bulk_load_1d(nd, p.k_new + nsrc, D * 2, full_k(st));
                            bulk_load_1d(nd + D * 2, p.v_new + nsrc, D * 2, full_k(st));
                        }
                    }
                    if (!mbar_wait(empty_v(st), ph, &g_decode_error, abort_flag)) return false;
                    mbar_arrive_expect_tx(full_v(st), SL::kChunkBytes);
#pragma unroll
                    for (int r = 0; r < D / 64; ++r)
                        tma_load_2d(stage + SL::kChunkBytes + r * SL::kRegion, &maps.v, full_v(st), r * 64, row);
                    ++cg;
                    return true;
                };
                int c = 0;
                if (x.spec) {
                    ok = issue(0);
                    c = 1;
                }
                dec_item_pos(x, p, pos_it);
                if (x.bad && x.kvh == 0 && x.split == 0) atomicCAS(&g_decode_error, 0, kErrBounds);
                for (; c < x.n_chunks && ok; ++c) ok = issue(c);
            }
            int no_abort = 0;  // drain the copies this thread started
            for (int i = 0; i < kDecStages && i < cg; ++i) {
                const int c = cg - 1 - i;
                mbar_wait(full_k(c % kDecStages), (c / kDecStages) & 1, &g_decode_error, &no_abort);
                mbar_wait(full_v(c % kDecStages), (c / kDecStages) & 1, &g_decode_error, &no_abort);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    // Warp w computes the scores of slots 16w .. 16w+15 of each chunk (S^T =
    // K Q^T on the tensor cores) and puts them, scaled to base 2, in shared
    // memory.  After one barrier every warp runs the softmax over all 64 slots
    // of the chunk -- lane (g, t) for head g -- and accumulates the d rows
    // [D/4 w, D/4 (w+1)) of O^T over them, so that at the end of an item each
    // warp holds the finished rows of its quarter of d: no merge across warps.
    constexpr int MW = D / 64;          // m16 tiles of O^T per warp
    constexpr int DW = D / kDecWarps;   // d rows per warp
    constexpr int SXR = SL::kSxRow;
    const int gq = lane >> 2;  // mma group id: slot row g (and g+8); softmax head g
    const int tq = lane & 3;   // thread in group: heads 2t, 2t+1 of S^T and O^T; k pairs 2t
    float *sx = reinterpret_cast<float *>(sm + SL::kSx);
    uint16_t *ost = reinterpret_cast<uint16_t *>(sm + SL::kOst) + warp * G * DW;
    const int slot0 = warp * 16;  // this warp's slots within a chunk (scores)
    int cg = 0;                   // chunks consumed by this CTA

    int pos_next = (kPosAhead && blockIdx.x < n_items) ? dec_item_load_pos(blockIdx.x, p) : 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        DecItem x = dec_item_head(it, p);
        int pos_it = pos_next;
        if (kPosAhead) {
            if (it + static_cast<int>(gridDim.x) < n_items) pos_next = dec_item_load_pos(it + gridDim.x, p);
        } else {
            pos_it = p.pos[x.b];
        }
        dec_item_pos(x, p, pos_it);
        if (x.n_chunks == 0) continue;
        // append + decode: the new token's k and v rows arrive with the item's
        // first chunk; when its slot is in a later chunk, the warp whose 16
        // slots will hold it also prefetches them now, so that their load
        // overlaps the chunk copies instead of following them
        const int onew = x.snew - x.begin;  // the new slot's offset in the item
        if (x.snew >= 0 && onew >= kDecCH && onew < x.end - x.begin && ((onew % kDecCH) >> 4) == warp &&
            lane < D / 8) {
            const int64_t src = (static_cast<int64_t>(x.b) * p.Hkv + x.kvh) * D + lane * 8;
            if (in_bounds(src / 8, p.n_new / 8, &g_decode_error, &g_decode_where)) {
                prefetch_l1(p.k_new + src);
                prefetch_l1(p.v_new + src);
            }
        }
        float acc[MW][4];  // O^T: d = DW*warp + 16*mt + gq (+8), heads 2tq, 2tq+1
#pragma unroll
        for (int mt = 0; mt < MW; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[mt][i] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;  // running max and sum of head gq (base 2)
        uint32_t qb[KS][2];                    // Q^T fragments; heads gq >= G are zero columns

        for (int c = 0; c < x.n_chunks; ++c, ++cg) {
            const int st = cg % kDecStages;
            const uint32_t ph = (cg / kDecStages) & 1;
            mbar_wait(full_k(st), ph, &g_decode_error, abort_flag);
            // filled slots of this chunk (none past n_valid, e.g. a speculative chunk)
            const int rows = min(kDecCH, min(x.end, x.n_valid) - (x.begin + c * kDecCH));
            const int mine = rows - slot0;  // valid slots among this warp's 16
            if (c == 0) {
                const uint16_t *qrow = reinterpret_cast<const uint16_t *>(
                                           sm + st * SL::kStage + 2 * SL::kChunkBytes) +
                                       (gq < G ? gq : 0) * D;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    qb[ks][0] = gq < G ? *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 2 * tq) : 0u;
                    qb[ks][1] = gq < G ? *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 8 + 2 * tq) : 0u;
                }
            }
            // append + decode: the warp whose 16 slots hold the new token puts
            // its k into the staged chunk now and its v once V has landed
            // (over what the copies read), and both into the cache
            // (warp-uniform test).  The proxy fence orders the stage writes
            // before the stage's next TMA fill; the cache stores follow it,
            // so it does not wait for them.
            const int rnew = x.snew - (x.begin + c * kDecCH);
            const bool patch = x.snew >= 0 && rnew >= slot0 && rnew < slot0 + 16 && rnew < rows;
            uint4 vv = make_uint4(0u, 0u, 0u, 0u);  // the new v row's part of this lane
            bool vok = false;
            const int off_new = (lane >> 3) * SL::kRegion + rnew * 128 + (((lane & 7) ^ (rnew & 7)) << 4);
            if (patch) {
                const int64_t src = (static_cast<int64_t>(x.b) * p.Hkv + x.kvh) * D + lane * 8;
                const int64_t dst =
                    ((static_cast<int64_t>(x.b) * p.Hkv + x.kvh) * p.cap + x.snew) * D + lane * 8;
                const bool ok = lane < D / 8 && in_bounds(src / 8, p.n_new / 8, &g_decode_error, &g_decode_where) &&
                                in_bounds(dst / 8, p.n_cache / 8, &g_decode_error, &g_decode_where);
                uint4 kk = make_uint4(0u, 0u, 0u, 0u);
                vok = ok;
                if (ok) {
                    if (c == 0) {  // staged with this chunk
                        const uint8_t *nb = sm + st * SL::kStage + 2 * SL::kChunkBytes + SL::kQBytes;
                        kk = *reinterpret_cast<const uint4 *>(nb + lane * 16);
                        vv = *reinterpret_cast<const uint4 *>(nb + D * 2 + lane * 16);
                    } else {
                        kk = *reinterpret_cast<const uint4 *>(p.k_new + src);
                        vv = *reinterpret_cast<const uint4 *>(p.v_new + src);
                    }
                    *reinterpret_cast<uint4 *>(sm + st * SL::kStage + off_new) = kk;
                }
                fence_proxy_async_smem();
                if (ok) {
                    *reinterpret_cast<uint4 *>(p.kc + dst) = kk;
                    *reinterpret_cast<uint4 *>(p.vc + dst) = vv;
                }
                __syncwarp();
            }
            const uint32_t kst = sbase + st * SL::kStage;
            const uint32_t vst = kst + SL::kChunkBytes;
            // ---- S^T = K Q^T for this warp's 16 slots, into the exchange buffer
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            if (mine > 0) {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t a[4];
                    ldsm_x4(swz(kst, slot0 + (lane & 15), 2 * ks + (lane >> 4)), a);
                    mma_16816<DT>(s, a, qb[ks][0], qb[ks][1]);
                }
            }
            float *sxb = sx + (cg & 1) * 8 * SXR;
            {
                const bool va = gq < mine, vb_ = gq + 8 < mine;
                const int h0 = 2 * tq, h1 = 2 * tq + 1;
                if (h0 < G) {
                    sxb[h0 * SXR + slot0 + gq] = va ? s[0] * p.scale_log2 : -INFINITY;
                    sxb[h0 * SXR + slot0 + gq + 8] = vb_ ? s[2] * p.scale_log2 : -INFINITY;
                }
                if (h1 < G) {
                    sxb[h1 * SXR + slot0 + gq] = va ? s[1] * p.scale_log2 : -INFINITY;
                    sxb[h1 * SXR + slot0 + gq + 8] = vb_ ? s[3] * p.scale_log2 : -INFINITY;
                }
            }
            // this warp is done with the stage's K (and q and the staged rows)
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_k(st));
            // the scores of all four warps are in place
            asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
            // ---- online softmax of head gq over the chunk's 64 slots: this
            // lane takes slots 16kk + {2t, 2t+1, 2t+8, 2t+9}, kk = 0..3 (the
            // ones its P^T fragments need); lanes 4g .. 4g+3 share head g
            float v[16];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float2 lo = make_float2(-INFINITY, -INFINITY), hi = lo;
                if (gq < G) {
                    lo = *reinterpret_cast<const float2 *>(sxb + gq * SXR + 16 * kk + 2 * tq);
                    hi = *reinterpret_cast<const float2 *>(sxb + gq * SXR + 16 * kk + 2 * tq + 8);
                }
                v[4 * kk] = lo.x;
                v[4 * kk + 1] = lo.y;
                v[4 * kk + 2] = hi.x;
                v[4 * kk + 3] = hi.y;
            }
            float xm = fmax3(v[0], v[1], v[2]);
#pragma unroll
            for (int i = 3; i < 15; i += 2) xm = fmax3(xm, v[i], v[i + 1]);
            xm = fmaxf(xm, v[15]);
            xm = fmaxf(xm, __shfl_xor_sync(0xffffffffu, xm, 1));
            xm = fmaxf(xm, __shfl_xor_sync(0xffffffffu, xm, 2));
            float alpha = 1.f;
            if (xm > m_run && (m_run == -INFINITY || xm - m_run > 8.f)) {
                alpha = ex2_approx(m_run - xm);
                m_run = xm;
            }
            const float u = m_run == -INFINITY ? 0.f : m_run;
            float ls = 0.f;
            uint32_t pb[4][2];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float p0 = ex2_approx(v[4 * kk] - u), p1 = ex2_approx(v[4 * kk + 1] - u);
                const float p2 = ex2_approx(v[4 * kk + 2] - u), p3 = ex2_approx(v[4 * kk + 3] - u);
                ls += (p0 + p1) + (p2 + p3);
                pb[kk][0] = pack2<DT>(p0, p1);
                pb[kk][1] = pack2<DT>(p2, p3);
            }
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            l_run = l_run * alpha + ls;
            // the O^T columns of this lane are heads 2t and 2t+1: their factors
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
                const float a0 = __shfl_sync(0xffffffffu, alpha, (2 * tq) * 4);
                const float a1 = __shfl_sync(0xffffffffu, alpha, (2 * tq + 1) * 4);
#pragma unroll
                for (int mt = 0; mt < MW; ++mt) {
                    acc[mt][0] *= a0;
                    acc[mt][2] *= a0;
                    acc[mt][1] *= a1;
                    acc[mt][3] *= a1;
                }
            }
            // ---- V: wait for it, then put in the new token's row and zero the
            // rows past the filled slots (a CTA-uniform test), all before any
            // warp reads them
            mbar_wait(full_v(st), ph, &g_decode_error, abort_flag);
            if ((x.snew >= 0 && rnew >= 0 && rnew < rows) || rows < kDecCH) {
                if (vok) *reinterpret_cast<uint4 *>(sm + st * SL::kStage + SL::kChunkBytes + off_new) = vv;
                if (mine < 16) {
                    // Every warp reads the V rows of all 64 slots: the rows of this
                    // warp's slots past the filled ones hold whatever the cache has
                    // there, so zero them (0-weights never meet a non-finite value).
                    uint8_t *vb = sm + st * SL::kStage + SL::kChunkBytes;
                    const int first = mine > 0 ? mine : 0;
                    for (int i = lane; i < (16 - first) * (D / 8); i += 32) {
                        const int r = slot0 + first + i / (D / 8), cc = i % (D / 8);
                        *reinterpret_cast<uint4 *>(vb + (cc >> 3) * SL::kRegion + r * 128 +
                                                   ((cc & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                if (patch || mine < 16) fence_proxy_async_smem();
                asm volatile("bar.sync 2, %0;" ::"n"(kDecWarps * 32) : "memory");
            }
            // ---- O^T rows of this warp += V^T P^T over the 64 slots
            const int vrow = ((lane >> 4) << 3) + (lane & 7);
#pragma unroll
            for (int mt = 0; mt < MW; ++mt) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    uint32_t a[4];
                    ldsm_x4_t(swz(vst, 16 * kk + vrow, 2 * (warp * MW + mt) + ((lane >> 3) & 1)), a);
                    mma_16816<DT>(acc[mt], a, pb[kk][0], pb[kk][1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_v(st));
        }

        // ---------------------------------------------------------------- output
        // Heads 2t and 2t+1 of this lane's O^T columns: their sums and maxima
        // are held by lanes 8t and 8t+4.  Nothing is written for a position
        // outside the cache.
        const float l0 = __shfl_sync(0xffffffffu, l_run, (2 * tq) * 4);
        const float l1 = __shfl_sync(0xffffffffu, l_run, (2 * tq + 1) * 4);
        const int h0 = 2 * tq, h1 = 2 * tq + 1;
        const int64_t orow0 = static_cast<int64_t>(x.b) * p.Hq + x.kvh * G;  // first head's row
        if (x.bad) continue;
        if (p.splits == 1 && !p.partials) {
            const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
            for (int mt = 0; mt < MW; ++mt) {
                const int dl = 16 * mt + gq;  // d row within this warp's quarter
                if (h0 < G) {
                    ost[h0 * DW + dl] = round16<DT>(acc[mt][0] * i0);
                    ost[h0 * DW + dl + 8] = round16<DT>(acc[mt][2] * i0);
                }
                if (h1 < G) {
                    ost[h1 * DW + dl] = round16<DT>(acc[mt][1] * i1);
                    ost[h1 * DW + dl + 8] = round16<DT>(acc[mt][3] * i1);
                }
            }
            __syncwarp();
            // G heads x DW values of 16 bits as 16-byte vectors
            constexpr int kVec = G * DW / 8;
            if (lane < kVec) {
                const int h = lane / (DW / 8), j = lane % (DW / 8);
                const int64_t oi = (orow0 + h) * D + DW * warp + 8 * j;
                if (in_bounds(oi / 8, p.n_o / 8, &g_decode_error, &g_decode_where))
                    *reinterpret_cast<uint4 *>(p.o + oi) = *reinterpret_cast<const uint4 *>(ost + h * DW + 8 * j);
            }
            __syncwarp();
        } else {
            // split partials: unnormalised O^T rows, and (max, sum) per head
#pragma unroll
            for (int mt = 0; mt < MW; ++mt) {
                const int d0 = DW * warp + 16 * mt + gq;
                if (h0 < G) {
                    const int64_t i0 = ((orow0 + h0) * p.splits + x.split) * D + d0;
                    if (in_bounds(i0 + 8, p.n_ws_acc, &g_decode_error, &g_decode_where)) {
                        p.ws_acc[i0] = acc[mt][0];
                        p.ws_acc[i0 + 8] = acc[mt][2];
                    }
                }
                if (h1 < G) {
                    const int64_t i1 = ((orow0 + h1) * p.splits + x.split) * D + d0;
                    if (in_bounds(i1 + 8, p.n_ws_acc, &g_decode_error, &g_decode_where)) {
                        p.ws_acc[i1] = acc[mt][1];
                        p.ws_acc[i1 + 8] = acc[mt][3];
                    }
                }
            }
            if (warp == 0 && tq == 0 && gq < G) {
                const int64_t im = ((orow0 + gq) * p.splits + x.split) * 2;
                if (in_bounds(im + 1, p.n_ws_ml, &g_decode_error, &g_decode_where)) {
                    p.ws_ml[im] = m_run;
                    p.ws_ml[im + 1] = l_run;
                }
            }
        }
    }
}

// One warp per (sequence, query head): merge the non-empty splits.
template <int D, int DT>
__global__ void __launch_bounds__(128) swa_decode_merge_kernel(const DecodeParams p) {
    pdl_launch_dependents();
    pdl_wait();  // the split kernel's partials
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.B * p.Hq) return;
    const int b = row / p.Hq;
    const int pos = p.pos[b];
    if (pos < 0 || (p.w < 0 && pos >= p.cap)) return;  // recorded by the split kernel
    const int cap_eff = p.w < 0 ? p.cap : p.w;
    const int n_valid = min(pos + 1, cap_eff);
    // the splits that wrote partials: those of [0, w) for a finite window
    // (some may hold no filled slot: m = -inf, l = 0), of [0, n_valid) else
    int begin, end, used;
    split_range(p.w >= 0 ? p.w : n_valid, p.splits, 0, begin, end, used);
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
    for (int e = 0; e < E; ++e) {
        const int64_t oi = static_cast<int64_t>(row) * D + lane * E + e;
        if (in_bounds(oi, p.n_o, &g_decode_error, &g_decode_where)) p.o[oi] = round16<DT>(a[e] * inv);
    }
}

// Hybrid window + linear decode, one CTA per (sequence, query head): the
// softmax partials of the window splits merged with the linear part of the
// evicted positions, phi(q) S and phi(q).z with phi(x) = (exp(xW), exp(-xW)),
// over one normaliser.  In the merge the linear part is a partial with
// m = 0 (in the base-2 exponent of the scores):
//   M = max(m_1, .., m_n, 0), l = sum l_j 2^(m_j - M) + (phi(q).z) 2^-M,
//   o = (sum acc_j 2^(m_j - M) + phi(q) S 2^-M) / l.
// The state is read once with every load in flight at the same time: thread
// t sums rows f = t / D (mod NT / D) of column t % D of S, and the row groups
// are added in shared memory.
constexpr int kHybThreads = 256;

template <int D, int DF, int DT>
__global__ void __launch_bounds__(kHybThreads) swa_hybrid_merge_kernel(const DecodeParams p) {
    constexpr int F = 2 * DF, RG = kHybThreads / D, RPT = F / RG;  // row groups, rows per thread
    constexpr int kPre = 8;  // window partials read ahead (more are read in a loop)
    static_assert(F % RG == 0 && F <= kHybThreads, "row split");
    __shared__ float s_phi[F];
    __shared__ float s_b[RG][D];
    __shared__ float s_z[F];
    pdl_launch_dependents();
    pdl_wait();  // the split kernel's partials
    const int row = blockIdx.x;
    const int tid = threadIdx.x;
    const int b = row / p.Hq, h = row - b * p.Hq;
    const int kvh = h / (p.Hq / p.Hkv);
    const int pos = p.pos[b];
    if (pos < 0 || (p.w < 0 && pos >= p.cap)) return;  // recorded by the split kernel
    const int64_t sr = static_cast<int64_t>(b) * p.Hkv + kvh;
    const int c = tid % D, g = tid / D;
    // Every global read is issued before any of them is used: the state rows
    // of this thread, z, q . W for phi(q), and the window partials.
    const float *Sc = p.S + sr * F * D + c;
    float sreg[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) sreg[i] = __ldg(Sc + static_cast<int64_t>(g + RG * i) * D);
    float zv = tid < F ? __ldg(p.z + sr * F + tid) : 0.f;
    float fx = 0.f;
    if (tid < DF) {
        const uint16_t *qrow = p.q + static_cast<int64_t>(row) * D;
        const float *Wh = p.W + static_cast<int64_t>(kvh) * D * DF + tid;
#pragma unroll
        for (int cc = 0; cc < D; ++cc) fx = fmaf(widen16<DT>(__ldg(qrow + cc)), __ldg(Wh + cc * DF), fx);
    }
    const int cap_eff = p.w < 0 ? p.cap : p.w;
    const int n_valid = min(pos + 1, cap_eff);
    int begin, end, used;
    split_range(p.w >= 0 ? p.w : n_valid, p.splits, 0, begin, end, used);
    float pm[kPre], pl[kPre], pa[kPre];
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
        const int64_t base = static_cast<int64_t>(row) * p.splits + j;
        const bool have = j < used && tid < D;
        pm[j] = have ? p.ws_ml[base * 2] : -INFINITY;
        pl[j] = have ? p.ws_ml[base * 2 + 1] : 0.f;
        pa[j] = have ? p.ws_acc[base * D + c] : 0.f;
    }
    if (tid < DF) {
        s_phi[tid] = expf(fx);
        s_phi[DF + tid] = expf(-fx);
    }
    if (tid < F) s_z[tid] = zv;
    __syncthreads();
    float acc_b = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) acc_b = fmaf(s_phi[g + RG * i], sreg[i], acc_b);
    s_b[g][c] = acc_b;
    __syncthreads();
    if (tid >= D) return;
    float bl = 0.f;
#pragma unroll
    for (int gg = 0; gg < RG; ++gg) bl += s_b[gg][c];
    float a_lin = 0.f;
#pragma unroll 8
    for (int f = 0; f < F; ++f) a_lin = fmaf(s_phi[f], s_z[f], a_lin);
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < kPre; ++j) m = fmaxf(m, pm[j]);
    for (int j = kPre; j < used; ++j)
        m = fmaxf(m, p.ws_ml[(static_cast<int64_t>(row) * p.splits + j) * 2]);
    const float flin = ex2_approx(-m);
    float l = a_lin * flin, acc = bl * flin;
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
        const float f = (pm[j] == -INFINITY) ? 0.f : ex2_approx(pm[j] - m);
        l = fmaf(pl[j], f, l);
        acc = fmaf(pa[j], f, acc);
    }
    for (int j = kPre; j < used; ++j) {
        const int64_t base = static_cast<int64_t>(row) * p.splits + j;
        const float mj = p.ws_ml[base * 2];
        const float f = (mj == -INFINITY) ? 0.f : ex2_approx(mj - m);
        l = fmaf(p.ws_ml[base * 2 + 1], f, l);
        acc = fmaf(p.ws_acc[base * D + c], f, acc);
    }
    const int64_t oi = static_cast<int64_t>(row) * D + c;
    if (in_bounds(oi, p.n_o, &g_decode_error, &g_decode_where))
        p.o[oi] = round16<DT>(l > 0.f ? acc / l : 0.f);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
DecodePlan decode_plan(int B, int Hq, int Hkv, int d, int cap, int w, int sm_count) {
    // Split a (sequence, kv head) only to give the persistent CTAs enough
    // items to balance: about SWA_DEC_ITEMS_PER_SM items per SM in total, at
    // least one chunk per split.
    DecodePlan plan{1, 0};
    const int cap_eff = w < 0 ? cap : w;
    const long long chunks = (cap_eff + kDecCH - 1) / kDecCH;
    const long long pairs = static_cast<long long>(B) * Hkv;
    const long long target = static_cast<long long>(SWA_DEC_ITEMS_PER_SM) * (sm_count > 0 ? sm_count : 148);
    if (pairs > 0 && pairs < target) {
        long long s = target / pairs;
        if (s > chunks) s = chunks;
        if (s < 1) s = 1;
        plan.splits = static_cast<int>(s);
    }
    if (plan.splits > 1)
        plan.workspace = static_cast<size_t>(B) * Hq * plan.splits * (d + 2) * sizeof(float);
    return plan;
}

namespace {

bool encode_cache_map(CUtensorMap *m, const void *ptr, int d, uint64_t rows, int dtype) {
    const cuTensorMapEncodeTiled_fn enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kDecCH};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType ty =
        dtype == SWA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return enc(m, ty, 2, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G, int ST, int DT>
swa_status launch_decode(const DecodeMaps &maps, const DecodeParams &p, int df,
                         cudaStream_t stream) {
    using SL = DecSmem<D, G, ST>;
    constexpr int kMaxCtas = dec_max_ctas<D, G, ST>();
    static_assert(kMaxCtas * (SL::kAlloc + 1024) <= 233472, "CTAs per SM must fit");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    static bool configured[64] = {};
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(swa_decode_kernel<D, G, ST, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SL::kAlloc);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode)");
        configured[dev] = true;
    }
    const int sms = device_sm_count();
    if (sms <= 0) return cuda_fail(cudaErrorInvalidDevice, "device_sm_count");
    const long long items = static_cast<long long>(p.B) * p.Hkv * p.splits;
    // 2-stage ring: the wide count when every CTA gets at least two items
    const int cps = (ST >= 2 && items >= 2ll * kMaxCtas * sms) ? kMaxCtas : kDecCtasPerSm[ST >= 2 ? 1 : 0];
    const long long cap_ctas = static_cast<long long>(cps) * sms;
    const int grid = static_cast<int>(items < cap_ctas ? items : cap_ctas);
    e = launch_pdl(swa_decode_kernel<D, G, ST, DT>, dim3(grid), dim3(kDecThreads), SL::kAlloc, stream,
                   maps, p);
    if (e != cudaSuccess) return cuda_fail(e, "launch swa_decode_kernel");
    if (p.partials) {  // hybrid: merge with the linear part
        const int rows = p.B * p.Hq;
        e = df == 32 ? launch_pdl(swa_hybrid_merge_kernel<D, 32, DT>, dim3(rows),
                                  dim3(kHybThreads), 0, stream, p)
                     : launch_pdl(swa_hybrid_merge_kernel<D, 64, DT>, dim3(rows),
                                  dim3(kHybThreads), 0, stream, p);
        if (e != cudaSuccess) return cuda_fail(e, "launch swa_hybrid_merge_kernel");
    } else if (p.splits > 1) {
        const int rows = p.B * p.Hq;
        e = launch_pdl(swa_decode_merge_kernel<D, DT>, dim3((rows + 3) / 4), dim3(128), 0, stream, p);
        if (e != cudaSuccess) return cuda_fail(e, "launch swa_decode_merge_kernel");
    }
    return SWA_OK;
}

}  // namespace

namespace {

// Chunk ring of a launch.  Items of one chunk: one stage (more CTAs per SM).
// Items of several chunks: two stages on the wide grid when that grid still
// gives every CTA at least two items (more CTAs in flight per SM), else three
// stages at SWA_DEC_CTAS_PER_SM per SM -- more of each CTA's chunks in
// flight, which keeps HBM busy when the grid's last round has CTAs idle.
template <int D, int G, int DT>
swa_status launch_decode_gs(const DecodeMaps &maps, const DecodeParams &p, bool single, int df,
                            cudaStream_t stream) {
    const long long items = static_cast<long long>(p.B) * p.Hkv * p.splits;
    if (single) return launch_decode<D, G, 1, DT>(maps, p, df, stream);
    if (items >= 2ll * dec_max_ctas<D, G, 2>() * device_sm_count())
        return launch_decode<D, G, 2, DT>(maps, p, df, stream);
    return launch_decode<D, G, 3, DT>(maps, p, df, stream);
}

template <int D, int DT>
swa_status launch_decode_g(const DecodeMaps &maps, const DecodeParams &p, int G, bool single,
                           int df, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_decode_gs<D, 1, DT>(maps, p, single, df, stream);
        case 2: return launch_decode_gs<D, 2, DT>(maps, p, single, df, stream);
        case 4: return launch_decode_gs<D, 4, DT>(maps, p, single, df, stream);
        case 8: return launch_decode_gs<D, 8, DT>(maps, p, single, df, stream);
        default: return SWA_ERR_UNSUPPORTED;
    }
}

template <int DT>
swa_status launch_decode_dt(const DecodeMaps &maps, const DecodeParams &p, int d, int G,
                            bool single, int df, cudaStream_t stream) {
    return d == 128 ? launch_decode_g<128, DT>(maps, p, G, single, df, stream)
                    : launch_decode_g<64, DT>(maps, p, G, single, df, stream);
}

}  // namespace

swa_status decode_launch(const void *q, const swa_cache &c, const int32_t *pos, int Hq, void *o,
                         void *workspace, const DecodePlan &plan, cudaStream_t stream,
                         const swa_linear_state *lin, const void *k_new, const void *v_new) {
    if (c.B == 0) return SWA_OK;
    DecodeParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.pos = pos;
    p.o = static_cast<uint16_t *>(o);
    p.B = c.B;
    p.Hq = Hq;
    p.Hkv = c.Hkv;
    p.cap = c.cap;
    p.w = c.w < 0 ? -1 : c.w;
    p.splits = plan.splits;
    if (lin != nullptr) {  // hybrid: every split writes partials for the merge
        p.partials = 1;
        p.S = lin->S;
        p.z = lin->z;
        p.W = lin->W;
    }
    if (plan.splits > 1 || lin != nullptr) {
        p.ws_acc = static_cast<float *>(workspace);
        p.ws_ml = p.ws_acc + static_cast<size_t>(c.B) * Hq * plan.splits * c.d;
    }
    p.scale_log2 = 1.4426950408889634f / std::sqrt(static_cast<float>(c.d));
    p.n_o = output_extent(static_cast<long long>(c.B) * Hq * c.d);
    p.n_cache = output_extent(static_cast<long long>(c.B) * c.Hkv * c.cap * c.d);
    p.n_new = static_cast<long long>(c.B) * c.Hkv * c.d;
    p.n_ws_acc = output_extent(static_cast<long long>(c.B) * Hq * plan.splits * c.d);
    p.n_ws_ml = output_extent(static_cast<long long>(c.B) * Hq * plan.splits * 2);
    if (k_new != nullptr) {
        p.k_new = static_cast<const uint16_t *>(k_new);
        p.v_new = static_cast<const uint16_t *>(v_new);
        p.kc = static_cast<uint16_t *>(c.k);
        p.vc = static_cast<uint16_t *>(c.v);
        p.s = c.w < 0 ? 0 : c.s;
    }
    DecodeMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const uint64_t rows = static_cast<uint64_t>(c.B) * c.Hkv * c.cap;
    if (!encode_cache_map(&maps.k, c.k, c.d, rows, c.dtype) ||
        !encode_cache_map(&maps.v, c.v, c.d, rows, c.dtype))
        return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(cache)");
    const int G = Hq / c.Hkv;
    // items of one chunk (at most 64 slots per split): one ring stage
    const long long cap_eff = c.w < 0 ? c.cap : c.w;
    const long long chunks = (cap_eff + kDecCH - 1) / kDecCH;
    const bool single = (chunks + plan.splits - 1) / plan.splits <= 1;
    const int df = lin != nullptr ? lin->df : 0;
    return c.dtype == SWA_F16 ? launch_decode_dt<kF16>(maps, p, c.d, G, single, df, stream)
                              : launch_decode_dt<kBf16>(maps, p, c.d, G, single, df, stream);
}

long long decode_read_clear_where(cudaStream_t stream) {
    unsigned long long w = 0;
    return read_clear_symbol(g_decode_where, &w, stream) ? where_index(w) : -2;
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
// self-test of the wait limit (swa_selftest_wait_timeout)
// ---------------------------------------------------------------------------
// One warp holds 32 TMEM columns and waits on an mbarrier that nothing
// arrives on.  Each lane's bounded wait gives up after SWA_WAIT_LIMIT_NS
// (the first records SWA_ERR_TIMEOUT and sets the abort flag, the others
// then return at once); the warp frees the TMEM and the kernel ends.
__global__ void __launch_bounds__(32) swa_wait_selftest_kernel() {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    tmem_alloc(smem_u32(&tmem_slot), 32);
    tmem_relinquish();
    tc_fence_before_sync();
    __syncwarp();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const bool ok = mbar_wait(smem_u32(&bar), 0, &g_decode_error, &abort_flag);
    if (ok) atomicCAS(&g_decode_error, 0, kErrBounds);  // cannot happen: nothing arrives
    tc_fence_before_sync();
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, 32);
}

swa_status selftest_wait_launch(cudaStream_t stream) {
    swa_wait_selftest_kernel<<<1, 32, 0, stream>>>();
    const cudaError_t e = cudaPeekAtLastError();
    return e == cudaSuccess ? SWA_OK : cuda_fail(e, "launch swa_wait_selftest_kernel");
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
