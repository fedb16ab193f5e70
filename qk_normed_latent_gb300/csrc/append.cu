// qkmla_append kernel: write new tokens into the latent cache and A^k_cache.
//
// Source: "QK-Normed MLA: QK normalization without full key caching", Technical
// Summary, Methodology -- "Dynamic Scalar Caching" (one inverse-RMS scalar per
// token and KV group), "Cache Layout" (keep c_t, add A^k_cache, never store
// full keys) and "Blockwise Normalization" (the RoPE part is normalised on its
// own, as a materialised vector).
//
// Per KV group the key statistic needs k_{t,g} = c^_t W^K_g, a small GEMM
// [N, d_c] x [d_c, d_h]; the key itself is reduced to its sum of squares in
// registers and never leaves the CTA.  The grid is (token tiles of 32) x G; the
// g = 0 CTAs also store the cast latent and the normalised RoPE key.
#include "common.cuh"

namespace qkmla {

namespace {

constexpr int kTT = 32;        // tokens per CTA
constexpr int kKC = 64;        // d_c chunk staged per step
constexpr int kThreads = 256;
constexpr int kMaxJ = 8;       // d_h <= 256

template <typename CT>
__global__ void __launch_bounds__(kThreads)
append_kernel(const float* __restrict__ c_new, const float* __restrict__ r_new, const float* __restrict__ wk,
              const float* __restrict__ grk, const int64_t* __restrict__ slots, int N, int G, int d_c,
              int d_h, int d_r, float eps, int plain, CT* __restrict__ kv, float* __restrict__ ak,
              int64_t num_slots, int* status) {
    __shared__ float Cs[kTT][kKC + 1];
    extern __shared__ float Ws[];              // [kKC][d_h]
    const int g = blockIdx.y;
    const int n0 = blockIdx.x * kTT;
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;   // ty: 0..7
    const int row = d_c + d_r;
    const int nj = (d_h + 31) / 32;

    float acc[4][kMaxJ];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < kMaxJ; ++j) acc[i][j] = 0.f;

    const float* wg = wk + (int64_t)g * d_c * d_h;
    for (int k0 = 0; k0 < d_c; k0 += kKC) {
        __syncthreads();
        for (int e = tid; e < kTT * kKC; e += kThreads) {
            const int tl = e / kKC, k = e % kKC;
            const int n = n0 + tl;
            // the statistic is taken over the STORED latent (cache dtype)
            Cs[tl][k] = (n < N && k0 + k < d_c) ? Elem<CT>::cast(c_new[(int64_t)n * d_c + k0 + k]) : 0.f;
        }
        for (int e = tid; e < kKC * d_h; e += kThreads) {
            const int k = e / d_h, j = e % d_h;
            Ws[k * d_h + j] = (k0 + k < d_c) ? wg[(int64_t)(k0 + k) * d_h + j] : 0.f;
        }
        __syncthreads();
        for (int k = 0; k < kKC; ++k) {
            float a[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = Cs[ty + 8 * i][k];
#pragma unroll
            for (int j = 0; j < kMaxJ; ++j) {
                if (j < nj) {
                    const int jj = tx + 32 * j;
                    const float b = (jj < d_h) ? Ws[k * d_h + jj] : 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i][j] = fmaf(a[i], b, acc[i][j]);
                }
            }
        }
    }

    // alpha^k_{t,g} = 1 / sqrt(mean_j k_j^2 + eps): warp ty owns tokens ty + 8 i
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxJ; ++j) ss = fmaf(acc[i][j], acc[i][j], ss);
        ss = warp_sum(ss);
        const int n = n0 + ty + 8 * i;
        if (tx == 0 && n < N) {
            const int64_t s = slots[n];
            if (s >= num_slots) {
                report(status, QKMLA_ERR_DEVICE_BOUNDS);
            } else if (s >= 0) {
                ak[s * G + g] = plain ? 1.f : 1.f / sqrtf(ss / (float)d_h + eps);
            }
        }
    }

    if (g != 0) return;
    // latent (pure cast) and RoPE key (normalised separately), one warp per token
    for (int tl = ty; tl < kTT; tl += kThreads / 32) {
        const int n = n0 + tl;
        if (n >= N) break;
        const int64_t s = slots[n];
        if (s < 0 || s >= num_slots) continue;
        CT* dst = kv + s * row;
        const float* cs = c_new + (int64_t)n * d_c;
        for (int k = tx; k < d_c; k += 32) Elem<CT>::store(dst + k, cs[k]);
        const float* rs = r_new + (int64_t)n * d_r;
        float beta = 1.f;
        if (!plain) {
            float ss = 0.f;
            for (int j = tx; j < d_r; j += 32) ss = fmaf(rs[j], rs[j], ss);
            ss = warp_sum(ss);
            beta = 1.f / sqrtf(ss / (float)d_r + eps);
        }
        for (int j = tx; j < d_r; j += 32) {
            const float gmul = (plain || grk == nullptr) ? 1.f : grk[j];
            Elem<CT>::store(dst + d_c + j, plain ? rs[j] : rs[j] * gmul * beta);
        }
    }
}

}  // namespace

int launch_append(const float* c_new, const float* r_new, const float* wk, const float* grk,
                  const int64_t* slots, int N, int G, int d_c, int d_h, int d_r, float eps, bool plain,
                  void* kv, int cache_dtype, float* ak, int64_t num_slots, cudaStream_t s) {
    if (N == 0) return QKMLA_OK;
    dim3 grid((N + kTT - 1) / kTT, G);
    const size_t smem = (size_t)kKC * d_h * sizeof(float);
    if (cache_dtype == QKMLA_F32) {
        auto k = append_kernel<float>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return QKMLA_ERR_CUDA;
        k<<<grid, kThreads, smem, s>>>(c_new, r_new, wk, grk, slots, N, G, d_c, d_h, d_r, eps, plain,
                                       (float*)kv, ak, num_slots, device_status_ptr());
    } else {
        auto k = append_kernel<__nv_bfloat16>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return QKMLA_ERR_CUDA;
        k<<<grid, kThreads, smem, s>>>(c_new, r_new, wk, grk, slots, N, G, d_c, d_h, d_r, eps, plain,
                                       (__nv_bfloat16*)kv, ak, num_slots, device_status_ptr());
    }
    return cudaGetLastError() == cudaSuccess ? QKMLA_OK : QKMLA_ERR_CUDA;
}

}  // namespace qkmla
