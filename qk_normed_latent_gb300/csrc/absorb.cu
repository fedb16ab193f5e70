// qkmla_absorb_query kernel: q~ = W^K_{g(h)} (q * gamma_q * gamma_k) and alpha^q = 1/S(q).
//
// Source: "QK-Normed MLA: QK normalization without full key caching", Technical
// Summary, Methodology -- "Static Weight Absorption" (gamma_k and gamma_q
// pre-multiply the query before the latent dot product) and the decode-logit
// equation (alpha^q is the query's inverse RMS, applied as a row scale).
//
// Per KV group g this is a GEMM  Q'_g [rows*H/G, d_h] x W_g^T [d_h, d_c]
// (W^K_g is d_c x d_h, row n holds the d_h weights of latent coordinate n).
// A CTA computes a 64 x 64 output tile with the whole K = d_h reduction staged
// in shared memory; fp32 FMA throughout, one RNE cast on the way out.
#include "common.cuh"

namespace qkmla {

namespace {

constexpr int kTM = 64, kTN = 64, kThreads = 256;

template <typename OutT>
__global__ void __launch_bounds__(kThreads)
absorb_kernel(const float* __restrict__ q, const float* __restrict__ gq, const float* __restrict__ gk,
              const float* __restrict__ wk, int rows, int H, int G, int d_h, int d_c, float eps,
              int plain, OutT* __restrict__ qt, float* __restrict__ aq) {
    extern __shared__ float smem[];
    const int ld = d_h + 1;                    // padded row: conflict-free column reads
    float* Qs = smem;                          // [kTM][ld]  q' rows of this tile
    float* Ws = smem + kTM * ld;               // [kTN][ld]  W^K_g rows n0..n0+63
    const int hpg = H / G;
    const int g = blockIdx.z;
    const int M = rows * hpg;
    const int m0 = blockIdx.x * kTM, n0 = blockIdx.y * kTN;
    const int tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();

    for (int e = tid; e < kTM * d_h; e += kThreads) {
        const int ml = e / d_h, k = e % d_h;
        const int m = m0 + ml;
        float v = 0.f;
        if (m < M) {
            const int r = m / hpg, h = g * hpg + m % hpg;
            v = q[((int64_t)r * H + h) * d_h + k];
            if (!plain) v *= gq[k] * gk[k];
        }
        Qs[ml * ld + k] = v;
    }
    const float* wg = wk + (int64_t)g * d_c * d_h;
    for (int e = tid; e < kTN * d_h; e += kThreads) {
        const int nl = e / d_h, k = e % d_h;
        const int n = n0 + nl;
        Ws[nl * ld + k] = (n < d_c) ? wg[(int64_t)n * d_h + k] : 0.f;
    }
    __syncthreads();

    // thread (tx, ty) owns rows ty + 16 i and columns tx + 16 j
    const int tx = tid & 15, ty = tid >> 4;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int k = 0; k < d_h; ++k) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = Qs[(ty + 16 * i) * ld + k];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = Ws[(tx + 16 * j) * ld + k];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty + 16 * i;
        if (m >= M) continue;
        const int r = m / hpg, h = g * hpg + m % hpg;
        OutT* dst = qt + ((int64_t)r * H + h) * d_c;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx + 16 * j;
            if (n < d_c) Elem<OutT>::store(dst + n, acc[i][j]);
        }
    }

    // alpha^q from the raw query (one warp per row), written by the first column tile
    if (blockIdx.y == 0) {
        const int warp = tid >> 5, lane = tid & 31;
        for (int ml = warp; ml < kTM; ml += kThreads / 32) {
            const int m = m0 + ml;
            if (m >= M) break;
            const int r = m / hpg, h = g * hpg + m % hpg;
            const float* src = q + ((int64_t)r * H + h) * d_h;
            float ss = 0.f;
            for (int k = lane; k < d_h; k += 32) ss = fmaf(src[k], src[k], ss);
            ss = warp_sum(ss);
            if (lane == 0) aq[(int64_t)r * H + h] = plain ? 1.f : 1.f / sqrtf(ss / (float)d_h + eps);
        }
    }
}

}  // namespace

int launch_absorb(const float* q, const float* gq, const float* gk, const float* wk, int rows, int H,
                  int G, int d_h, int d_c, float eps, bool plain, void* qt, int qt_dtype, float* aq,
                  cudaStream_t s) {
    // bf16 q~ (the tensor-core decode operand): split-bf16 tensor-core GEMM
    if (qt_dtype == QKMLA_BF16 && absorb_tc_supported(q, wk, d_h, d_c))
        return launch_absorb_tc(q, gq, gk, wk, rows, H, G, d_h, d_c, eps, plain, qt, qt_dtype, aq, s);
    const int M = rows * (H / G);
    dim3 grid((M + kTM - 1) / kTM, (d_c + kTN - 1) / kTN, G);
    const size_t smem = (size_t)(kTM + kTN) * (d_h + 1) * sizeof(float);
    if (qt_dtype == QKMLA_F32) {
        auto k = absorb_kernel<float>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return QKMLA_ERR_CUDA;
        if (launch_pdl(k, grid, dim3(kThreads), smem, s, q, gq, gk, wk, rows, H, G, d_h, d_c, eps, (int)plain,
                       (float*)qt, aq) != cudaSuccess)
            return QKMLA_ERR_CUDA;
    } else {
        auto k = absorb_kernel<__nv_bfloat16>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return QKMLA_ERR_CUDA;
        if (launch_pdl(k, grid, dim3(kThreads), smem, s, q, gq, gk, wk, rows, H, G, d_h, d_c, eps, (int)plain,
                       (__nv_bfloat16*)qt, aq) != cudaSuccess)
            return QKMLA_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? QKMLA_OK : QKMLA_ERR_CUDA;
}

}  // namespace qkmla
