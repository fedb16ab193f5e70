// Split-KV combine: merge per-split (o_s, lse_s) of one output row.
//
// A split covering tokens T_s yields o_s = sum_{t in T_s} p^s_t c_t (normalised
// over T_s) and lse_s = log sum_{t in T_s} exp(l_t).  The softmax over all
// tokens is recovered exactly:  lse = log sum_s exp(lse_s),
// o = sum_s exp(lse_s - lse) o_s.  Empty splits carry lse_s = -inf.
#include "common.cuh"

namespace qkmla {

namespace {

constexpr int kThreads = 128;
constexpr int kMaxSplits = 1024;

__global__ void __launch_bounds__(kThreads)
combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int nsplit, int d_c,
               void* __restrict__ o, int o_dtype, float* __restrict__ lse) {
    __shared__ float wts[kMaxSplits];
    __shared__ float red[kThreads / 32];
    __shared__ float s_m, s_inv, s_lse;
    const int64_t rh = blockIdx.x;
    const int tid = threadIdx.x;
    const float* lp = lse_part + rh * nsplit;
    pdl_wait();
    pdl_trigger();

    float m = -INFINITY;
    for (int s = tid; s < nsplit; s += kThreads) m = fmaxf(m, lp[s]);
    m = warp_max(m);
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    if (tid == 0) {
        float mm = red[0];
        for (int w = 1; w < kThreads / 32; ++w) mm = fmaxf(mm, red[w]);
        s_m = mm;
    }
    __syncthreads();
    m = s_m;
    float sum = 0.f;
    for (int s = tid; s < nsplit; s += kThreads) {
        const float w = (m == -INFINITY) ? 0.f : expf(lp[s] - m);
        wts[s] = w;
        sum += w;
    }
    sum = warp_sum(sum);
    __syncthreads();
    if ((tid & 31) == 0) red[tid >> 5] = sum;
    __syncthreads();
    if (tid == 0) {
        float ss = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) ss += red[w];
        s_inv = (ss > 0.f) ? 1.f / ss : 0.f;
        s_lse = (ss > 0.f) ? m + logf(ss) : -INFINITY;
    }
    __syncthreads();
    const float inv = s_inv;
    for (int k = tid; k < d_c; k += kThreads) {
        float acc = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const float w = wts[s];
            if (w != 0.f) acc = fmaf(w, o_part[(rh * nsplit + s) * d_c + k], acc);
        }
        acc *= inv;
        if (o_dtype == QKMLA_F32)
            ((float*)o)[rh * d_c + k] = acc;
        else
            ((__nv_bfloat16*)o)[rh * d_c + k] = __float2bfloat16_rn(acc);
    }
    if (tid == 0 && lse) lse[rh] = s_lse;
}

}  // namespace

int launch_combine(const float* o_part, const float* lse_part, int rows, int nsplit, int d_c, void* o,
                   int o_dtype, float* lse, cudaStream_t s) {
    if (nsplit > kMaxSplits) return QKMLA_ERR_UNSUPPORTED;
    return launch_pdl(combine_kernel, dim3(rows), dim3(kThreads), 0, s, o_part, lse_part, nsplit, d_c, o, o_dtype,
                      lse) == cudaSuccess
               ? QKMLA_OK
               : QKMLA_ERR_CUDA;
}

}  // namespace qkmla
