// Shared device helpers of the QK-Normed MLA decode library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/qkmla.h"

namespace qkmla {

// Record the first device-side error in the per-device status word `st`
// (read and cleared by qkmla_get_device_status()).
__device__ __forceinline__ void report(int* st, int code) {
    if (st) atomicCAS(st, 0, code);
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialization: it may start while the previous kernel on
// the stream is still running, so it first does only work that touches no
// global memory, then waits (pdl_wait) until the previous grid has completed and
// its writes are visible, and then lets the next kernel start its own launch
// (pdl_trigger).  Launched without the attribute, both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float* p) { return *p; }
    static __device__ __forceinline__ float cast(float x) { return x; }
    static __device__ __forceinline__ void store(float* p, float x) { *p = x; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ float cast(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Physical slot of token t of sequence b (see the cache convention in qkmla.h).
// Returns -1 (and records a bounds error) for a page id outside [0, num_pages).
__device__ __forceinline__ int64_t slot_of(const int32_t* page_table, int b, int t, int page_size,
                                           int max_pages, int64_t num_pages, int* st) {
    const int p = t / page_size;
    const int64_t page = page_table ? (int64_t)page_table[(int64_t)b * max_pages + p]
                                    : (int64_t)b * max_pages + p;
    if (page < 0 || page >= num_pages) {
        report(st, QKMLA_ERR_DEVICE_BOUNDS);
        return -1;
    }
    return page * page_size + (t % page_size);
}

// alpha^k entry `idx` of the A^k_cache, stored as fp32 or (f16) as its RNE half cast.
__device__ __forceinline__ void store_alpha(void* ak, int64_t idx, float v, bool f16) {
    if (f16) reinterpret_cast<__half*>(ak)[idx] = __float2half_rn(v);
    else reinterpret_cast<float*>(ak)[idx] = v;
}
template <bool F16>
__device__ __forceinline__ float load_alpha(const void* ak, int64_t idx) {
    if constexpr (F16) return __half2float(reinterpret_cast<const __half*>(ak)[idx]);
    else return reinterpret_cast<const float*>(ak)[idx];
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Host: launch `kernel` on `s` with programmatic stream serialization.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace qkmla

// Launch-side helpers (host).
namespace qkmla {
int launch_absorb(const float* q, const float* gq, const float* gk, const float* wk, int rows, int H,
                  int G, int d_h, int d_c, float eps, bool plain, void* qt, int qt_dtype, float* aq,
                  cudaStream_t s);
bool absorb_tc_supported(const float* q, const float* wk, int d_h, int d_c);
int launch_absorb_tc(const float* q, const float* gq, const float* gk, const float* wk, int rows, int H, int G,
                     int d_h, int d_c, float eps, bool plain, void* qt, int qt_dtype, float* aq, cudaStream_t s);
int launch_append(const float* c_new, const float* r_new, const float* wk, const float* grk,
                  const int64_t* slots, int N, int G, int d_c, int d_h, int d_r, float eps, bool plain,
                  void* kv, int cache_dtype, void* ak, bool ak_f16, int64_t num_slots, const int32_t* positions,
                  float rope_theta, cudaStream_t s);

struct DecodePlan {
    int kernel;            // 0 = simt, 1 = tcgen05
    int num_splits;        // simt: splits per sequence
    int parts;             // number of partial (o, lse) records in the workspace
    size_t ws_bytes;
};
int plan_decode(const qkmla_decode_args* a, DecodePlan* plan);
int launch_decode_simt(const qkmla_decode_args* a, const DecodePlan& plan, cudaStream_t s);
int launch_decode_tc(const qkmla_decode_args* a, const DecodePlan& plan, cudaStream_t s);
bool tc_supported(const qkmla_decode_args* a);
bool pair_shape(const qkmla_decode_args* a);        // served by the two-CTA cluster kernel
bool sched_in_kernel(const qkmla_decode_args* a);   // split plan computed by the decode kernels themselves
size_t tc_workspace(const qkmla_decode_args* a, int sms, int* max_items_out);
int launch_combine(const float* o_part, const float* lse_part, int rows, int nsplit, int d_c, void* o,
                   int o_dtype, float* lse, cudaStream_t s);
int device_sm_count();
int* device_status_ptr();   // this device's status word (lazily resolved), or nullptr
}  // namespace qkmla
