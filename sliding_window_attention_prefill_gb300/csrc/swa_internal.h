// swa_internal.h -- declarations shared by the library's translation units
// (host side only; kernels stay private to their .cu file).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstddef>
#include <cstdint>
#include <utility>

#include "swa.h"

typedef CUresult (*cuTensorMapEncodeTiled_fn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                              void *, const cuuint64_t *, const cuuint64_t *,
                                              const cuuint32_t *, const cuuint32_t *,
                                              CUtensorMapInterleave, CUtensorMapSwizzle,
                                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

namespace swa {

// One NVTX range around each call of the C ABI that enqueues GPU work, named
// after the call, so a profiler timeline shows which call launched which
// kernels.  With no tool attached an NVTX call only tests a function pointer.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
#define SWA_NVTX_RANGE(name) const ::swa::NvtxRange swa_nvtx_range_(name)

// Driver entry point for tensor-map encoding (resolved once through the
// runtime, so the library needs no link-time dependency on libcuda).
cuTensorMapEncodeTiled_fn tensor_map_encoder();

// Number of SMs of the current device (cached per device); <= 0 on error.
int device_sm_count();

// Decode work plan: how many key splits each (sequence, kv head) gets.
struct DecodePlan {
    int splits;          // >= 1
    size_t workspace;    // bytes of fp32 partials (0 when splits == 1)
};
DecodePlan decode_plan(int B, int Hq, int Hkv, int d, int cap, int w, int sm_count);

// Launchers (arguments already validated).
// dtype: SWA_BF16 or SWA_F16, the type of q, k, v and o.
swa_status prefill_launch(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                          int L, int Hq, int Hkv, int d, int w, int s, int dtype,
                          cudaStream_t stream);
// Prefill of L query rows that sit at key positions q_off .. q_off+L-1 of a
// key sequence of Lk rows: K/V in [B, Lk, Hkv, d], or in a cache's
// [B, Hkv, kv_cap, d] layout when kv_cap > 0.
swa_status prefill_launch_offset(const void *q, const void *k, const void *v, void *o, float *lse,
                                 int B, int L, int Hq, int Hkv, int d, int w, int s, int q_off,
                                 int Lk, int kv_cap, int dtype, cudaStream_t stream);
// Variable-length prefill: B sequences packed in [total, heads, d] tensors,
// sequence b at rows cu_seqlens[b] .. cu_seqlens[b+1]-1 (device array);
// workspace of varlen_workspace_bytes(B, total, Hq, Hkv) bytes.
size_t varlen_workspace_bytes(int B, int total, int Hq, int Hkv);
swa_status prefill_varlen_launch(const void *q, const void *k, const void *v, void *o, float *lse,
                                 const int32_t *cu_seqlens, int B, int total, int max_len, int Hq,
                                 int Hkv, int d, int w, int s, int dtype, void *workspace,
                                 cudaStream_t stream);
// Chunked prefill of a finite window: the key rows the chunk's queries need,
// in one sequence [B, q_off + n, Hkv, d] per tensor -- the cache's sinks and
// ring in position order, then the chunk.
swa_status chunk_gather_launch(const swa_cache &c, const void *k_new, const void *v_new, int n,
                               int64_t pos0, int q_off, void *wk, void *wv, cudaStream_t stream);
swa_status append_launch(const swa_cache &c, const void *k_new, const void *v_new, int n,
                         int64_t pos0, cudaStream_t stream);
// lin != nullptr: hybrid window + linear decode (workspace of
// hybrid_workspace_bytes, partials written even with one split).
// k_new, v_new != nullptr ([B, Hkv, d]): append + decode -- each sequence's
// new token is written to its slot of position pos[b] and attended at once.
swa_status decode_launch(const void *q, const swa_cache &c, const int32_t *pos, int Hq, void *o,
                         void *workspace, const DecodePlan &plan, cudaStream_t stream,
                         const swa_linear_state *lin = nullptr, const void *k_new = nullptr,
                         const void *v_new = nullptr);
// Fold the positions an append of n tokens at pos0 evicts from the ring into
// the linear state (before the append overwrites them).  *appended: the
// kernel has also written the tokens (a one-token append), so no append
// kernel is needed.
swa_status hybrid_fold_launch(const swa_cache &c, const swa_linear_state &lin, const void *k_new,
                              const void *v_new, int n, int64_t pos0, cudaStream_t stream,
                              bool *appended);

// Launch with programmatic stream serialization: the kernel's CTAs may be
// placed while the previous kernel of the stream drains, so its prologue
// (barrier init, TMEM allocation, tensor-map prefetch) overlaps that tail.
// Every kernel of the library executes griddepcontrol.wait before it reads
// or writes global memory, so stream order is kept for the data.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Record the CUDA error behind an SWA_ERR_CUDA (per host thread) and return
// SWA_ERR_CUDA; `where` names the failing call.
swa_status cuda_fail(cudaError_t e, const char *where);
const char *last_cuda_error();

// The wait-limit self-test kernel (records SWA_ERR_TIMEOUT in the decode
// module's error word).
swa_status selftest_wait_launch(cudaStream_t stream);

// Read and clear each module's device error word (synchronises `stream`).
// Returns 0 or a negative swa_status value.
int prefill_read_clear_error(cudaStream_t stream);
int decode_read_clear_error(cudaStream_t stream);
int append_read_clear_error(cudaStream_t stream);
int hybrid_read_clear_error(cudaStream_t stream);

// Bounds-checked build: read and clear each module's record of the first
// refused index (-1 if none; -2 if a CUDA call failed).  Synchronises.
long long prefill_read_clear_where(cudaStream_t stream);
long long decode_read_clear_where(cudaStream_t stream);
long long append_read_clear_where(cudaStream_t stream);
long long hybrid_read_clear_where(cudaStream_t stream);

// The extent (in elements) the kernels are told an output buffer of n
// elements has: n, less the test margin of the bounds-checked build
// (swa_debug_set_extent_margin), never below 0.
long long output_extent(long long n);

#ifdef __CUDACC__
// Copy a module's __device__ word to the host and reset it to zero (in the
// module that defines it: the symbol is that translation unit's own).
template <typename T>
inline bool read_clear_symbol(T &symbol, T *out, cudaStream_t stream) {
    const T zero{};
    if (cudaMemcpyFromSymbolAsync(out, symbol, sizeof(T), 0, cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
        return false;
    if (cudaMemcpyToSymbolAsync(symbol, &zero, sizeof(T), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return false;
    return cudaStreamSynchronize(stream) == cudaSuccess;
}

// A module's `where` word as the refused index (or -1).
inline long long where_index(unsigned long long w) {
    return w == 0 ? -1 : static_cast<long long>(w) - (1ll << 50);
}
#endif

}  // namespace swa
