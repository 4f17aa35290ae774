// swa_prefill_common.cuh -- work decomposition of the prefill kernel
// (swa_prefill.cu): work units, their key columns and key tiles, and the
// tensor maps.
//
// A work unit is (sequence b, key/value head kvh, query tile).  Its 128 MMA
// rows pack the G = Hq/Hkv query heads that share kvh for P = 128/G
// consecutive positions: row r is position t0 + r/G, head kvh*G + r%G, which
// is exactly a box of the [B, L, Hq, d] query tensor, so one TMA box loads it.
// The unit needs the sink keys [0, s) and the band [lo, t1] with
// lo = max(s, t0-(w-s)+1) (the window of "Sliding-window beats linear
// attention", section "Prerequisites / Sliding-window attention SWA(w, s)"):
// its key columns are laid out as [s_pad sink rows | band ...] and cut into
// key tiles of KT columns, the sink block (s rounded up to 8 rows, so that the
// band starts on a 1024-byte swizzle atom) sharing the first tile.
//
// Variable-length batches (varlen): the sequences are packed one after the
// other in [1, total, heads, d] tensors; sequence b holds rows
// cu_seqlens[b] .. cu_seqlens[b+1]-1.  A small planning kernel writes one
// record per query tile ({b, tile index, first row, length}); unit u is
// (tile record, kv head) and its TMA coordinates add the first row.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "swa_internal.h"

namespace swa {

struct PrefillMaps {
    CUtensorMap q;                    // box {64, G, P, 1} over [B, L, Hq, d]
    CUtensorMap k_band, v_band;       // box {64, 1, KT, 1} over [B, L, Hkv, d]
    CUtensorMap k_sink, v_sink;       // box {64, 1, s_pad, 1}
    CUtensorMap k_band0, v_band0;     // box {64, 1, KT - s_pad, 1}
    CUtensorMap o;                    // box {64, G, P, 1} over the [B, L, Hq, d] output
};

// Division by a divisor fixed for a call, as a multiply-high and a shift
// (round-up method): l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (mulhi(m, n) + n) >> l, exact for 0 <= n < 2^31, 1 <= d < 2^31.
struct FastDiv {
    uint32_t m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
    return FastDiv{static_cast<uint32_t>(m), l};
}

__device__ __forceinline__ int fast_div(int n, const FastDiv &f) {
    return static_cast<int>((__umulhi(f.m, static_cast<uint32_t>(n)) + static_cast<uint32_t>(n)) >> f.l);
}

struct PrefillParams {
    int B, L, Hq, Hkv, G, P;  // L: query rows; P: positions per query tile (128 / G)
    int q_off, Lk;            // query row i sits at key position q_off + i; Lk key rows
    int g_log2;               // G is a power of two (row r: position r >> g_log2)
    int w, s;                 // w < 0: infinite window (s is then 0)
    int s_pad;                // sink rows loaded: s rounded up to 8 (0 if s == 0)
    int n_qtiles, n_units;
    FastDiv div_bh, div_hkv;  // by B * Hkv and by Hkv (unit geometry)
    float scale_log2;         // log2(e) / sqrt(d)
    float scale;              // 1 / sqrt(d)
    uint16_t *o;              // [B, L, Hq, d] bf16 or fp16
    float *lse;               // optional [B, Hq, L]
    // varlen: B sequences packed in L rows; the planning kernel's output
    int varlen;
    const int *tile_count;    // number of query tiles (0 if cu_seqlens is invalid)
    const int4 *tile_rec;     // per query tile: {b, tile index, first row, length}
    long long n_o, n_lse;     // extents of o and lse in elements (bounds-checked build)
};

// A work unit.  b is the batch coordinate of the tensor maps and r0 the row
// of position 0 of the unit's sequence (0 unless varlen, where b is 0).
struct Unit {
    int b, kvh, t0, t1, lo, n_cols, n_tiles, r0;
};

// Work units of the call (read from the planning kernel's output for varlen).
template <bool VL>
__device__ __forceinline__ int prefill_units(const PrefillParams &p) {
    if constexpr (VL) return *p.tile_count * p.Hkv;
    return p.n_units;
}

// Geometry of work unit u of n_units.  Units run heaviest query tiles first
// (only matters for the infinite window, where cost grows with the position);
// varlen units run in reverse order of their tile records.
template <int KT, bool VL>
__device__ __forceinline__ Unit unit_geom(int u, const PrefillParams &p, int n_units) {
    Unit x;
    if constexpr (VL) {
        const int tr = fast_div(u, p.div_hkv);
        x.kvh = u - tr * p.Hkv;
        const int4 rec = p.tile_rec[fast_div(n_units, p.div_hkv) - 1 - tr];
        x.b = 0;
        x.r0 = rec.z;
        x.t0 = rec.y * p.P;
        x.t1 = min(x.t0 + p.P, rec.w) - 1;
        x.lo = p.w < 0 ? 0 : max(p.s, x.t0 - (p.w - p.s) + 1);
        const int nb = max(0, x.t1 - x.lo + 1);
        x.n_cols = p.s_pad + nb;
        x.n_tiles = (x.n_cols + KT - 1) / KT;
        return x;
    } else {
    const int bh = p.B * p.Hkv;
    const int qt_rev = fast_div(u, p.div_bh);
    const int r = u - qt_rev * bh;
    x.b = fast_div(r, p.div_hkv);
    x.kvh = r - x.b * p.Hkv;
    x.r0 = 0;
    const int qt = p.n_qtiles - 1 - qt_rev;
    x.t0 = p.q_off + qt * p.P;                      // key-space positions
    x.t1 = min(x.t0 + p.P, p.q_off + p.L) - 1;
    x.lo = p.w < 0 ? 0 : max(p.s, x.t0 - (p.w - p.s) + 1);
    const int nb = max(0, x.t1 - x.lo + 1);
    x.n_cols = p.s_pad + nb;
    x.n_tiles = (x.n_cols + KT - 1) / KT;
    return x;
    }
}

// Key columns of tile j, rounded up to the MMA's N granularity of 16.
template <int KT>
__device__ __forceinline__ int tile_width(const Unit &x, int j) {
    const int n = min(KT, x.n_cols - KT * j);
    return (n + 15) & ~15;
}

// ------------------------------------------------------------------ host side
// q_off / Lk: the queries are key positions q_off .. q_off+L-1 of a key
// sequence of Lk rows (a plain prefill: 0 and L).
inline PrefillParams make_prefill_params(void *o, float *lse, int B, int L, int Hq, int Hkv, int d,
                                         int w, int s, int q_off = 0, int Lk = -1) {
    PrefillParams p{};
    p.B = B;
    p.L = L;
    p.q_off = q_off;
    p.Lk = Lk < 0 ? L : Lk;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.P = 128 / p.G;
    p.g_log2 = 0;
    while ((1 << p.g_log2) < p.G) ++p.g_log2;
    p.w = w < 0 ? -1 : w;
    p.s = w < 0 ? 0 : s;
    p.s_pad = (p.s + 7) & ~7;
    p.n_qtiles = (L + p.P - 1) / p.P;
    p.n_units = B * Hkv * p.n_qtiles;
    p.div_bh = make_fastdiv(static_cast<uint32_t>(B * Hkv > 0 ? B * Hkv : 1));
    p.div_hkv = make_fastdiv(static_cast<uint32_t>(Hkv > 0 ? Hkv : 1));
    p.scale = 1.0f / std::sqrt(static_cast<float>(d));
    p.scale_log2 = p.scale * 1.4426950408889634f;
    p.o = static_cast<uint16_t *>(o);
    p.lse = lse;
    p.n_o = output_extent(static_cast<long long>(B) * L * Hq * d);
    p.n_lse = lse ? output_extent(static_cast<long long>(B) * Hq * L) : 0;
    return p;
}

// Tensor-map element type of a swa_dtype value.
static inline CUtensorMapDataType tensor_map_type(int dtype) {
    return dtype == SWA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

// 4-D map (coordinates d, head, position, batch) over a 16-bit tensor of type
// `dtype`, 64-column boxes, 128-byte swizzle.  Layout [B, L, heads, d] when
// bhsd_cap == 0, else [B, heads, bhsd_cap, d] (a cache: positions 0 .. L-1
// of cap slots).
static inline bool encode_prefill_map(CUtensorMap *m, const void *ptr, int d, int heads, int L,
                                      int B, int box_heads, int box_rows, int dtype,
                                      int bhsd_cap = 0) {
    const cuTensorMapEncodeTiled_fn enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2,
                             (cuuint64_t)L * heads * d * 2};
    if (bhsd_cap > 0) {
        strides[0] = (cuuint64_t)bhsd_cap * d * 2;           // head
        strides[1] = (cuuint64_t)d * 2;                      // position
        strides[2] = (cuuint64_t)heads * bhsd_cap * d * 2;   // batch
    }
    cuuint32_t box[4] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, tensor_map_type(dtype), 4, const_cast<void *>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The maps of one call with key tiles of `kt` columns; K and V in the
// [B, Lk, Hkv, d] layout, or [B, Hkv, kv_cap, d] when kv_cap > 0.
static inline bool encode_prefill_maps(PrefillMaps *maps, const void *q, const void *k,
                                       const void *v, const PrefillParams &p, int d, int kt,
                                       int dtype, int kv_cap = 0) {
    std::memset(maps, 0, sizeof(*maps));
    const int dt = dtype;
    bool ok = encode_prefill_map(&maps->q, q, d, p.Hq, p.L, p.B, p.G, p.P, dt) &&
              encode_prefill_map(&maps->o, p.o, d, p.Hq, p.L, p.B, p.G, p.P, dt) &&
              encode_prefill_map(&maps->k_band, k, d, p.Hkv, p.Lk, p.B, 1, kt, dt, kv_cap) &&
              encode_prefill_map(&maps->v_band, v, d, p.Hkv, p.Lk, p.B, 1, kt, dt, kv_cap);
    if (ok && p.s_pad > 0)
        ok = encode_prefill_map(&maps->k_sink, k, d, p.Hkv, p.Lk, p.B, 1, p.s_pad, dt, kv_cap) &&
             encode_prefill_map(&maps->v_sink, v, d, p.Hkv, p.Lk, p.B, 1, p.s_pad, dt, kv_cap) &&
             encode_prefill_map(&maps->k_band0, k, d, p.Hkv, p.Lk, p.B, 1, kt - p.s_pad, dt,
                                kv_cap) &&
             encode_prefill_map(&maps->v_band0, v, d, p.Hkv, p.Lk, p.B, 1, kt - p.s_pad, dt,
                                kv_cap);
    return ok;
}

}  // namespace swa
