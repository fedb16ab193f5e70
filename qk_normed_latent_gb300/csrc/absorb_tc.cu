// qkmla_absorb_query on the tensor cores (tcgen05, kind::f16).
//
// Source: "QK-Normed MLA: QK normalization without full key caching", Technical
// Summary, Methodology -- "Static Weight Absorption": gamma_k and gamma_q
// pre-multiply the query before the latent dot product, i.e. the query side of
// the logit is q~ = W^K_g (q * gamma_q * gamma_k); alpha^q = 1/S(q) is the
// row scale of the decode-logit equation.
//
// Per KV group g this is the GEMM  q~_g = Q'_g W_g^T  with Q'_g [rows*H/G, d_h]
// and W_g [d_c, d_h] (both K-major, fp32).  To keep fp32-level accuracy on the
// bf16 tensor cores every operand is split into x = hi + lo (two bf16 values,
// lo = bf16(x - hi)) and three MMAs accumulate hi*hi + hi*lo + lo*hi in fp32
// (the dropped lo*lo term is ~2^-16 relative).  A CTA owns 128 rows of one
// group and all d_c outputs; the accumulator sits in TMEM (up to 512 columns).
#include "common.cuh"
#include "tc_ptx.cuh"

namespace qkmla {

namespace {

using namespace tc;

constexpr int kM = 128;          // rows per CTA (MMA M)
constexpr int kN = 256;          // MMA N per chunk
constexpr int kThreads = 128;

__device__ __forceinline__ void split_store(uint8_t* hi_base, uint8_t* lo_base, uint32_t off, const float (&x)[8]) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 hh = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        const float r0 = x[2 * i] - __low2float(hh);
        const float r1 = x[2 * i + 1] - __high2float(hh);
        const __nv_bfloat162 ll = __floats2bfloat162_rn(r0, r1);
        h[i] = *reinterpret_cast<const uint32_t*>(&hh);
        l[i] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    *reinterpret_cast<uint4*>(hi_base + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo_base + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// Shared memory: A_hi, A_lo [kM x DH] and B_hi, B_lo [kN x DH], bf16, K-major,
// 128-byte swizzle, in 64-column blocks.
template <int DH>
struct AbsLayout {
    static constexpr int kKBlocks = DH / 64;
    static constexpr int kA = kKBlocks * kM * 128;
    static constexpr int kB = kKBlocks * kN * 128;
    static constexpr int kOffAhi = 0, kOffAlo = kA, kOffBhi = 2 * kA, kOffBlo = 2 * kA + kB;
    static constexpr int kOffMisc = 2 * kA + 2 * kB;
    static constexpr int kBytes = kOffMisc + 64 + 1024;
};

template <int DH, typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
absorb_tc_kernel(const float* __restrict__ q, const float* __restrict__ gq, const float* __restrict__ gk,
                 const float* __restrict__ wk, int rows, int H, int G, int d_c, float eps, int plain,
                 OutT* __restrict__ qt, float* __restrict__ aq, int* status) {
    using LY = AbsLayout<DH>;
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    uint64_t* bar = (uint64_t*)(sm + LY::kOffMisc);
    uint32_t* tmem_slot = (uint32_t*)(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.y;
    const int hpg = H / G;
    const int M = rows * hpg;
    const int m0 = blockIdx.x * kM;
    const int n_chunks = d_c / kN;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    // ---- A = q * gamma_q * gamma_k (or q), split hi/lo ----
    for (int e = tid; e < kM * (DH / 8); e += kThreads) {
        const int ml = e / (DH / 8), k8 = e % (DH / 8);
        const int m = m0 + ml;
        float x[8];
        if (m < M) {
            const int r = m / hpg, h = g * hpg + m % hpg;
            const float4* src = reinterpret_cast<const float4*>(q + ((size_t)r * H + h) * DH + k8 * 8);
            const float4 v0 = src[0], v1 = src[1];
            x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w;
            x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
            if (!plain) {
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] *= gq[k8 * 8 + i] * gk[k8 * 8 + i];
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = 0.f;
        }
        const uint32_t off = (k8 >> 3) * (kM * 128) + sw128_offset(ml, (k8 & 7) * 8);
        split_store(sm + LY::kOffAhi, sm + LY::kOffAlo, off, x);
    }
    // alpha^q: one thread per row from the raw query
    {
        const int m = m0 + tid;
        if (tid < kM && m < M) {
            const int r = m / hpg, h = g * hpg + m % hpg;
            const float4* src = reinterpret_cast<const float4*>(q + ((size_t)r * H + h) * DH);
            float ss = 0.f;
#pragma unroll 4
            for (int k4 = 0; k4 < DH / 4; ++k4) {
                const float4 v = src[k4];
                ss = fmaf(v.x, v.x, ss);
                ss = fmaf(v.y, v.y, ss);
                ss = fmaf(v.z, v.z, ss);
                ss = fmaf(v.w, v.w, ss);
            }
            aq[(size_t)r * H + h] = plain ? 1.f : 1.f / sqrtf(ss / (float)DH + eps);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const float* wg = wk + (size_t)g * d_c * DH;
    bool ok = true;

    for (int nc = 0; nc < n_chunks; ++nc) {
        // ---- B = W_g rows nc*256 .. +255, split hi/lo ----
        for (int e = tid; e < kN * (DH / 8); e += kThreads) {
            const int nl = e / (DH / 8), k8 = e % (DH / 8);
            const float4* src = reinterpret_cast<const float4*>(wg + (size_t)(nc * kN + nl) * DH + k8 * 8);
            const float4 v0 = src[0], v1 = src[1];
            float x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            const uint32_t off = (k8 >> 3) * (kN * 128) + sw128_offset(nl, (k8 & 7) * 8);
            split_store(sm + LY::kOffBhi, sm + LY::kOffBlo, off, x);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t idesc = idesc_bf16(kM, kN, 0, 0);
            const uint32_t a_hi = smem_u32(sm + LY::kOffAhi), a_lo = smem_u32(sm + LY::kOffAlo);
            const uint32_t b_hi = smem_u32(sm + LY::kOffBhi), b_lo = smem_u32(sm + LY::kOffBlo);
            const uint32_t d = tmem + nc * kN;
#pragma unroll
            for (int kb = 0; kb < DH / 16; ++kb) {
                const uint32_t ao = (kb >> 2) * (kM * 128) + (kb & 3) * 32;
                const uint32_t bo = (kb >> 2) * (kN * 128) + (kb & 3) * 32;
                mma_bf16(d, smem_desc(a_hi + ao, 16, 1024, kSwizzle128B), smem_desc(b_hi + bo, 16, 1024, kSwizzle128B),
                         idesc, kb > 0 ? 1u : 0u);
                mma_bf16(d, smem_desc(a_hi + ao, 16, 1024, kSwizzle128B), smem_desc(b_lo + bo, 16, 1024, kSwizzle128B),
                         idesc, 1u);
                mma_bf16(d, smem_desc(a_lo + ao, 16, 1024, kSwizzle128B), smem_desc(b_hi + bo, 16, 1024, kSwizzle128B),
                         idesc, 1u);
            }
            mma_commit(bar);
        }
        __syncwarp();
        // every thread waits (bounded) before B is overwritten or TMEM is read
        uint32_t done = 0;
        for (uint32_t it = 0; it < (1u << 24) && !done; ++it) done = mbar_try_wait(bar, nc & 1) ? 1u : 0u;
        if (!done) {
            report(status, QKMLA_ERR_TIMEOUT);
            ok = false;
        }
        tc_fence_after();
        if (__syncthreads_or(!ok)) break;
    }

    // ---- epilogue: row m = lane 32*warp + lane; columns = latent coordinates ----
    if (ok) {
        const int m = m0 + 32 * warp + lane;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const bool valid = m < M;
        OutT* dst = nullptr;
        if (valid) {
            const int r = m / hpg, h = g * hpg + m % hpg;
            dst = qt + ((size_t)r * H + h) * d_c;
        }
        for (int c0 = 0; c0 < d_c; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + lane_base + c0, v);
            tmem_wait_ld();
            if (valid) {
                if constexpr (sizeof(OutT) == 2) {
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                        w[i] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
                    d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
                } else {
                    float4* d4 = reinterpret_cast<float4*>(dst + c0);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                            __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int DH, typename OutT>
int launch_t(const float* q, const float* gq, const float* gk, const float* wk, int rows, int H, int G, int d_c,
             float eps, bool plain, void* qt, float* aq, cudaStream_t s) {
    using LY = AbsLayout<DH>;
    static_assert(LY::kBytes <= 232448, "shared memory budget");
    auto k = absorb_tc_kernel<DH, OutT>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes) != cudaSuccess)
        return QKMLA_ERR_CUDA;
    const int M = rows * (H / G);
    dim3 grid((M + kM - 1) / kM, G);
    k<<<grid, kThreads, LY::kBytes, s>>>(q, gq, gk, wk, rows, H, G, d_c, eps, plain ? 1 : 0, (OutT*)qt, aq,
                                         device_status_ptr());
    return cudaGetLastError() == cudaSuccess ? QKMLA_OK : QKMLA_ERR_CUDA;
}

}  // namespace

// Shapes the tensor-core absorb handles: d_h in {64, 128}, d_c a multiple of 256
// up to 512, 16-byte aligned fp32 inputs.
bool absorb_tc_supported(const float* q, const float* wk, int d_h, int d_c) {
    if (d_h != 64 && d_h != 128) return false;
    if (d_c % kN || d_c > 512) return false;
    if (((uintptr_t)q % 16) || ((uintptr_t)wk % 16)) return false;
    return true;
}

int launch_absorb_tc(const float* q, const float* gq, const float* gk, const float* wk, int rows, int H, int G,
                     int d_h, int d_c, float eps, bool plain, void* qt, int qt_dtype, float* aq, cudaStream_t s) {
    if (d_h == 128)
        return qt_dtype == QKMLA_BF16
                   ? launch_t<128, __nv_bfloat16>(q, gq, gk, wk, rows, H, G, d_c, eps, plain, qt, aq, s)
                   : launch_t<128, float>(q, gq, gk, wk, rows, H, G, d_c, eps, plain, qt, aq, s);
    return qt_dtype == QKMLA_BF16 ? launch_t<64, __nv_bfloat16>(q, gq, gk, wk, rows, H, G, d_c, eps, plain, qt, aq, s)
                                  : launch_t<64, float>(q, gq, gk, wk, rows, H, G, d_c, eps, plain, qt, aq, s);
}

}  // namespace qkmla
