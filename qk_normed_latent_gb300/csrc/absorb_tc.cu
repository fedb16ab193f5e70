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
// (the dropped lo*lo term is ~2^-16 relative).
//
// A CTA owns a 128-row x NB-latent output tile of one group (NB = 256, or 64
// when the 256-wide grid would leave most SMs idle: small batches).  Its raw fp32
// operands land in shared memory by bulk copies (one per query row, eight for
// the W_g slice), all in flight at once; the 512 threads then split them into
// bf16 hi/lo in place (each thread reads its elements, a barrier, then writes
// the swizzled K-major tiles over the raw bytes: 4 bytes in, 2 x 2 bytes out).
// The output tile is staged in the drained operand region as 128-byte boxes
// (128-byte swizzle) of the tile's rows -- nr query rows x the group's hpg heads,
// one 3-D box {128 B of columns, hpg, nr} -- and written by TMA stores, whole
// lines instead of each thread's 16-byte pieces; shapes whose heads per group do
// not divide 128 store directly.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "decode_common.cuh"
#include "tc_ptx.cuh"

namespace qkmla {

namespace {

using namespace tc;

constexpr int kM = 128;          // rows per CTA (MMA M)
constexpr int kNMax = 256;       // latent columns per CTA (MMA N) for large grids
constexpr int kThreads = 512;

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

// Shared memory.  A region: raw fp32 [kM][DH], then A_hi, A_lo (bf16 [kM x DH],
// K-major, 128-byte swizzle, 64-column blocks) over the same bytes; B region
// likewise for [kN][DH].  Thread t handles the 8-element groups
// e = t + i * kThreads (row e / kG8, columns 8 (e % kG8) .. +7).
template <int DH, int kN>
struct AbsLayout {
    static constexpr int kA = kM * DH * 4;                    // raw A bytes = A_hi + A_lo bytes
    static constexpr int kB = kN * DH * 4;
    static constexpr int kOffA = 0, kOffB = kA;
    static constexpr int kOffAlo = kA / 2, kOffBlo = kOffB + kB / 2;
    static constexpr int kOffG = kA + kB;                     // gamma_q * gamma_k [DH]
    static constexpr int kOffMisc = kOffG + DH * 4;
    static constexpr int kBytes = kOffMisc + 64 + 1024;
    static constexpr int kG8 = DH / 8;
    static constexpr int kAIter = kM * kG8 / kThreads;
    static constexpr int kBIter = kN * kG8 / kThreads;
    static constexpr int kBCopies = 8;
};

template <int DH, int kN, typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
absorb_tc_kernel(const __grid_constant__ CUtensorMap tm_out, const float* __restrict__ q, const float* __restrict__ gq,
                 const float* __restrict__ gk, const float* __restrict__ wk, int rows, int H, int G, int d_c, float eps,
                 int plain, int tma_out, OutT* __restrict__ qt, float* __restrict__ aq, int* status) {
    using LY = AbsLayout<DH, kN>;
    static_assert(LY::kAIter * kThreads == kM * LY::kG8 && LY::kBIter * kThreads == kN * LY::kG8, "tiling");
    static_assert(32 % LY::kG8 == 0, "a row's groups sit in one warp");
    static_assert(LY::kB % (LY::kBCopies * 16) == 0, "bulk copy sizes");
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    float* rawA = reinterpret_cast<float*>(sm + LY::kOffA);
    float* rawB = reinterpret_cast<float*>(sm + LY::kOffB);
    float* gprod = reinterpret_cast<float*>(sm + LY::kOffG);
    uint64_t* bar = (uint64_t*)(sm + LY::kOffMisc);
    uint32_t* tmem_slot = (uint32_t*)(bar + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.z;
    const int n0 = blockIdx.y * kN;
    const int hpg = H / G;
    const int M = rows * hpg;
    const int m0 = blockIdx.x * kM;
    const int m_valid = min(kM, M - m0);

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kN);
        tmem_relinquish();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    // ---- every operand byte in flight at once ----
    if (tid == 0) mbar_arrive_expect_tx(&bar[0], (uint32_t)(m_valid * DH * 4 + LY::kB));
    if (tid < m_valid) {
        const int m = m0 + tid, r = m / hpg, h = g * hpg + m % hpg;
        bulk_load(rawA + tid * DH, q + ((size_t)r * H + h) * DH, DH * 4, &bar[0]);
    } else if (tid >= kM && tid < kM + LY::kBCopies) {
        const int c = tid - kM;
        constexpr int bytes = LY::kB / LY::kBCopies;
        bulk_load(reinterpret_cast<uint8_t*>(rawB) + c * bytes,
                  reinterpret_cast<const uint8_t*>(wk + ((size_t)g * d_c + n0) * DH) + c * bytes, bytes, &bar[0]);
    }
    if (tid < DH) gprod[tid] = plain ? 1.f : gq[tid] * gk[tid];
    bool ok = mbar_wait(&bar[0], 0, 1u << 24);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) report(status, QKMLA_ERR_TIMEOUT);
        // copies that never landed may still be in flight: do not release the CTA's memory early
        mbar_wait(&bar[0], 0, 1u << 24);
        __syncthreads();
        if (warp == 0) tmem_dealloc(*tmem_slot, kN);
        return;
    }

    // ---- A = q * gamma_q * gamma_k (or q), split hi/lo in place; alpha^q from the raw q ----
    {
        float x[LY::kAIter][8];
#pragma unroll
        for (int i = 0; i < LY::kAIter; ++i) {
            const int e = tid + i * kThreads;
            const int ml = e / LY::kG8, k8 = e % LY::kG8;
            if (ml < m_valid) {
                const float4 v0 = *reinterpret_cast<const float4*>(rawA + ml * DH + k8 * 8);
                const float4 v1 = *reinterpret_cast<const float4*>(rawA + ml * DH + k8 * 8 + 4);
                x[i][0] = v0.x; x[i][1] = v0.y; x[i][2] = v0.z; x[i][3] = v0.w;
                x[i][4] = v1.x; x[i][5] = v1.y; x[i][6] = v1.z; x[i][7] = v1.w;
            } else {
#pragma unroll
                for (int t = 0; t < 8; ++t) x[i][t] = 0.f;
            }
            if (blockIdx.y == 0) {
                // the kG8 groups of one row are held by kG8 consecutive lanes
                float ss = 0.f;
#pragma unroll
                for (int t = 0; t < 8; ++t) ss = fmaf(x[i][t], x[i][t], ss);
#pragma unroll
                for (int o = LY::kG8 / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                if (k8 == 0 && ml < m_valid) {
                    const int m = m0 + ml, r = m / hpg, h = g * hpg + m % hpg;
                    aq[(size_t)r * H + h] = plain ? 1.f : 1.f / sqrtf(ss / (float)DH + eps);
                }
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) x[i][t] *= gprod[k8 * 8 + t];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < LY::kAIter; ++i) {
            const int e = tid + i * kThreads;
            const int ml = e / LY::kG8, k8 = e % LY::kG8;
            const uint32_t off = (k8 >> 3) * (kM * 128) + sw128_offset(ml, (k8 & 7) * 8);
            split_store(sm + LY::kOffA, sm + LY::kOffAlo, off, x[i]);
        }
    }
    // ---- B = W_g rows n0 .. n0 + 255, split hi/lo in place ----
    {
        float x[LY::kBIter][8];
#pragma unroll
        for (int i = 0; i < LY::kBIter; ++i) {
            const int e = tid + i * kThreads;
            const int nl = e / LY::kG8, k8 = e % LY::kG8;
            const float4 v0 = *reinterpret_cast<const float4*>(rawB + nl * DH + k8 * 8);
            const float4 v1 = *reinterpret_cast<const float4*>(rawB + nl * DH + k8 * 8 + 4);
            x[i][0] = v0.x; x[i][1] = v0.y; x[i][2] = v0.z; x[i][3] = v0.w;
            x[i][4] = v1.x; x[i][5] = v1.y; x[i][6] = v1.z; x[i][7] = v1.w;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < LY::kBIter; ++i) {
            const int e = tid + i * kThreads;
            const int nl = e / LY::kG8, k8 = e % LY::kG8;
            const uint32_t off = (k8 >> 3) * (kN * 128) + sw128_offset(nl, (k8 & 7) * 8);
            split_store(sm + LY::kOffB, sm + LY::kOffBlo, off, x[i]);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0) {
        const uint32_t idesc = idesc_bf16(kM, kN, 0, 0);
        const uint32_t a_hi = smem_u32(sm + LY::kOffA), a_lo = smem_u32(sm + LY::kOffAlo);
        const uint32_t b_hi = smem_u32(sm + LY::kOffB), b_lo = smem_u32(sm + LY::kOffBlo);
#pragma unroll
        for (int kb = 0; kb < DH / 16; ++kb) {
            const uint32_t ao = (kb >> 2) * (kM * 128) + (kb & 3) * 32;
            const uint32_t bo = (kb >> 2) * (kN * 128) + (kb & 3) * 32;
            mma_bf16(tmem, smem_desc(a_hi + ao, 16, 1024, kSwizzle128B), smem_desc(b_hi + bo, 16, 1024, kSwizzle128B),
                     idesc, kb > 0 ? 1u : 0u);
            mma_bf16(tmem, smem_desc(a_hi + ao, 16, 1024, kSwizzle128B), smem_desc(b_lo + bo, 16, 1024, kSwizzle128B),
                     idesc, 1u);
            mma_bf16(tmem, smem_desc(a_lo + ao, 16, 1024, kSwizzle128B), smem_desc(b_hi + bo, 16, 1024, kSwizzle128B),
                     idesc, 1u);
        }
        mma_commit(&bar[1]);
    }
    __syncwarp();
    // every thread waits (bounded) before TMEM is read
    ok = mbar_wait(&bar[1], 0, 1u << 24);
    if (!ok) report(status, QKMLA_ERR_TIMEOUT);
    tc_fence_after();

    // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (output rows) and
    //      columns kN/4 (w / 4) .. (latent coordinates n0 + ...) ----
    constexpr int kC16 = kN / 64;                  // 16-column chunks per warp
    constexpr int kBoxCols = 128 / (int)sizeof(OutT);
    const bool all_ok = __syncthreads_and(ok) != 0;
    if (all_ok) {
        const int ml = 32 * (warp & 3) + lane;
        const int c_base = (kN / 4) * (warp >> 2);
        const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + c_base;
        uint32_t v[kC16][16];
#pragma unroll
        for (int c = 0; c < kC16; ++c) tmem_ld16(taddr + 16 * c, v[c]);
        tmem_wait_ld();
        // this thread's 64 columns as stored (bf16: 128 B, one box row; fp32: 256 B, two)
        uint32_t w[kC16 * 16 * (int)sizeof(OutT) / 4];
#pragma unroll
        for (int c = 0; c < kC16; ++c) {
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                if constexpr (sizeof(OutT) == 2) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[c][i]), __uint_as_float(v[c][i + 1]));
                    w[8 * c + i / 2] = *reinterpret_cast<const uint32_t*>(&b2);
                } else {
                    w[16 * c + i] = v[c][i];
                    w[16 * c + i + 1] = v[c][i + 1];
                }
            }
        }
        constexpr int kChunks = (int)(sizeof(w) / 16);           // 16-byte chunks of the 64 columns
        if (tma_out) {
            // the operand region is drained (every MMA has completed): box c_base / kBoxCols onward
#pragma unroll
            for (int q16 = 0; q16 < kChunks; ++q16) {
                const int col = c_base * (int)sizeof(OutT) / 16 + q16;          // 16-byte chunk of the row
                uint8_t* box = sm + (col / 8) * (kM * 128) + ml * 128;
                *reinterpret_cast<uint4*>(box + (((uint32_t)(col & 7) ^ (uint32_t)(ml & 7)) << 4)) =
                    make_uint4(w[4 * q16], w[4 * q16 + 1], w[4 * q16 + 2], w[4 * q16 + 3]);
            }
        } else if (ml < m_valid) {
            const int m = m0 + ml, r = m / hpg, h = g * hpg + m % hpg;
            uint4* d4 = reinterpret_cast<uint4*>(qt + ((size_t)r * H + h) * d_c + n0 + c_base);
#pragma unroll
            for (int q16 = 0; q16 < kChunks; ++q16) d4[q16] = make_uint4(w[4 * q16], w[4 * q16 + 1], w[4 * q16 + 2], w[4 * q16 + 3]);
        }
        if (tma_out) {
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                // rows past the group's rows fall outside the tensor's row range and are not written
                for (int bx = 0; bx < kN / kBoxCols; ++bx)
                    tma_store_3d(&tm_out, n0 + bx * kBoxCols, g * hpg, m0 / hpg, sm + bx * (kM * 128));
                dec::bulk_commit_group();
                dec::bulk_wait_all();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kN);
    }
}

// Many row tiles per (group, 256-latent half) -- large batches: a persistent CTA
// keeps its W_g half split in shared memory (bf16 hi + lo, loaded before the
// dependency wait: no kernel of this library writes W^K) and walks row tiles
// ci, ci + cpp, ...; per tile it loads the q rows, splits them, issues the 24
// MMAs and stages the bf16 output for TMA stores in the drained A region.  The
// W split, redone by every CTA of the one-tile kernel, is paid once per CTA.
template <int DH>
__global__ void __launch_bounds__(kThreads, 1)
absorb_tc_persistent(const __grid_constant__ CUtensorMap tm_out, const float* __restrict__ q,
                     const float* __restrict__ gq, const float* __restrict__ gk, const float* __restrict__ wk,
                     int rows, int H, int G, int d_c, float eps, int plain, int cpp,
                     __nv_bfloat16* __restrict__ qt, float* __restrict__ aq, int* status) {
    using LY = AbsLayout<DH, kNMax>;
    static_assert(LY::kA >= kNMax * 2 / 128 * kM * 128, "the bf16 output boxes fit the A region");
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    float* rawA = reinterpret_cast<float*>(sm + LY::kOffA);
    float* rawB = reinterpret_cast<float*>(sm + LY::kOffB);
    float* gprod = reinterpret_cast<float*>(sm + LY::kOffG);
    uint64_t* bar = (uint64_t*)(sm + LY::kOffMisc);                 // [0] W, [1] A of a tile, [2] MMAs of a tile
    uint32_t* tmem_slot = (uint32_t*)(bar + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NH = d_c / kNMax;
    const int pr = blockIdx.x % (G * NH), ci = blockIdx.x / (G * NH);
    const int g = pr / NH, nh = pr % NH, n0 = nh * kNMax;
    const int hpg = H / G;
    const int M = rows * hpg;
    const int n_tiles = (M + kM - 1) / kM;

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar[i], 1);
        fence_barrier_init();
        prefetch_tmap(&tm_out);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kNMax);
        tmem_relinquish();
    }
    __syncthreads();
    // ---- W_g rows n0 .. n0 + 255: before the dependency wait ----
    if (tid == 0) mbar_arrive_expect_tx(&bar[0], (uint32_t)LY::kB);
    if (tid < LY::kBCopies) {
        constexpr int bytes = LY::kB / LY::kBCopies;
        bulk_load(reinterpret_cast<uint8_t*>(rawB) + tid * bytes,
                  reinterpret_cast<const uint8_t*>(wk + ((size_t)g * d_c + n0) * DH) + tid * bytes, bytes, &bar[0]);
    }
    if (tid < DH) gprod[tid] = plain ? 1.f : gq[tid] * gk[tid];
    bool ok = mbar_wait(&bar[0], 0, 1u << 24);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) report(status, QKMLA_ERR_TIMEOUT);
        mbar_wait(&bar[0], 0, 1u << 24);       // copies still in flight land before the memory is released
        __syncthreads();
        if (warp == 0) tmem_dealloc(*tmem_slot, kNMax);
        return;
    }
    {
        float x[LY::kBIter][8];
#pragma unroll
        for (int i = 0; i < LY::kBIter; ++i) {
            const int e = tid + i * kThreads;
            const int nl = e / LY::kG8, k8 = e % LY::kG8;
            const float4 v0 = *reinterpret_cast<const float4*>(rawB + nl * DH + k8 * 8);
            const float4 v1 = *reinterpret_cast<const float4*>(rawB + nl * DH + k8 * 8 + 4);
            x[i][0] = v0.x; x[i][1] = v0.y; x[i][2] = v0.z; x[i][3] = v0.w;
            x[i][4] = v1.x; x[i][5] = v1.y; x[i][6] = v1.z; x[i][7] = v1.w;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < LY::kBIter; ++i) {
            const int e = tid + i * kThreads;
            const int nl = e / LY::kG8, k8 = e % LY::kG8;
            const uint32_t off = (k8 >> 3) * (kNMax * 128) + sw128_offset(nl, (k8 & 7) * 8);
            split_store(sm + LY::kOffB, sm + LY::kOffBlo, off, x[i]);
        }
    }
    pdl_wait();                // q comes from an earlier kernel; q~ is written below
    pdl_trigger();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int it = 0;
    for (int t = ci; t < n_tiles && ok; t += cpp, ++it) {
        const int m0 = t * kM, m_valid = min(kM, M - m0);
        // ---- this tile's q rows (the previous tile's output boxes have been read out) ----
        if (tid == 0) mbar_arrive_expect_tx(&bar[1], (uint32_t)(m_valid * DH * 4));
        __syncwarp();
        // a query token's hpg heads of group g are contiguous (the launcher requires
        // kM % hpg == 0, so a tile holds whole tokens): one copy per token
        if (tid < m_valid / hpg) {
            const int r = m0 / hpg + tid;
            bulk_load(rawA + tid * hpg * DH, q + ((size_t)r * H + g * hpg) * DH, (uint32_t)(hpg * DH * 4), &bar[1]);
        }
        ok = mbar_wait(&bar[1], it & 1, 1u << 24);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) report(status, QKMLA_ERR_TIMEOUT);
            mbar_wait(&bar[1], it & 1, 1u << 24);
            ok = false;
            break;
        }
        // ---- A = q * gamma_q * gamma_k, split hi/lo in place; alpha^q from the raw q (first half only) ----
        {
            float x[LY::kAIter][8];
#pragma unroll
            for (int i = 0; i < LY::kAIter; ++i) {
                const int e = tid + i * kThreads;
                const int ml = e / LY::kG8, k8 = e % LY::kG8;
                if (ml < m_valid) {
                    const float4 v0 = *reinterpret_cast<const float4*>(rawA + ml * DH + k8 * 8);
                    const float4 v1 = *reinterpret_cast<const float4*>(rawA + ml * DH + k8 * 8 + 4);
                    x[i][0] = v0.x; x[i][1] = v0.y; x[i][2] = v0.z; x[i][3] = v0.w;
                    x[i][4] = v1.x; x[i][5] = v1.y; x[i][6] = v1.z; x[i][7] = v1.w;
                } else {
#pragma unroll
                    for (int u = 0; u < 8; ++u) x[i][u] = 0.f;
                }
                if (nh == 0) {
                    float ss = 0.f;
#pragma unroll
                    for (int u = 0; u < 8; ++u) ss = fmaf(x[i][u], x[i][u], ss);
#pragma unroll
                    for (int o = LY::kG8 / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                    if (k8 == 0 && ml < m_valid) {
                        const int m = m0 + ml, r = m / hpg, h = g * hpg + m % hpg;
                        aq[(size_t)r * H + h] = plain ? 1.f : 1.f / sqrtf(ss / (float)DH + eps);
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) x[i][u] *= gprod[k8 * 8 + u];
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < LY::kAIter; ++i) {
                const int e = tid + i * kThreads;
                const int ml = e / LY::kG8, k8 = e % LY::kG8;
                const uint32_t off = (k8 >> 3) * (kM * 128) + sw128_offset(ml, (k8 & 7) * 8);
                split_store(sm + LY::kOffA, sm + LY::kOffAlo, off, x[i]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t idesc = idesc_bf16(kM, kNMax, 0, 0);
            const uint32_t a_hi = smem_u32(sm + LY::kOffA), a_lo = smem_u32(sm + LY::kOffAlo);
            const uint32_t b_hi = smem_u32(sm + LY::kOffB), b_lo = smem_u32(sm + LY::kOffBlo);
#pragma unroll
            for (int kb = 0; kb < DH / 16; ++kb) {
                const uint32_t ao = (kb >> 2) * (kM * 128) + (kb & 3) * 32;
                const uint32_t bo = (kb >> 2) * (kNMax * 128) + (kb & 3) * 32;
                mma_bf16(tmem, smem_desc(a_hi + ao, 16, 1024, kSwizzle128B), smem_desc(b_hi + bo, 16, 1024, kSwizzle128B),
                         idesc, kb > 0 ? 1u : 0u);
                mma_bf16(tmem, smem_desc(a_hi + ao, 16, 1024, kSwizzle128B), smem_desc(b_lo + bo, 16, 1024, kSwizzle128B),
                         idesc, 1u);
                mma_bf16(tmem, smem_desc(a_lo + ao, 16, 1024, kSwizzle128B), smem_desc(b_hi + bo, 16, 1024, kSwizzle128B),
                         idesc, 1u);
            }
            mma_commit(&bar[2]);
        }
        __syncwarp();
        ok = mbar_wait(&bar[2], it & 1, 1u << 24);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) report(status, QKMLA_ERR_TIMEOUT);
            mbar_wait(&bar[2], it & 1, 1u << 24);   // the MMAs finish before TMEM is released
            ok = false;
            break;
        }
        tc_fence_after();
        // ---- epilogue: TMEM -> bf16 boxes in the drained A region -> TMA stores ----
        {
            constexpr int kC16 = kNMax / 64;
            const int ml = 32 * (warp & 3) + lane;
            const int c_base = (kNMax / 4) * (warp >> 2);
            const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + c_base;
            uint32_t v[kC16][16];
#pragma unroll
            for (int c = 0; c < kC16; ++c) tmem_ld16(taddr + 16 * c, v[c]);
            tmem_wait_ld();
            uint32_t w[kC16 * 8];
#pragma unroll
            for (int c = 0; c < kC16; ++c)
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[c][i]), __uint_as_float(v[c][i + 1]));
                    w[8 * c + i / 2] = *reinterpret_cast<const uint32_t*>(&b2);
                }
            uint8_t* box = sm + (c_base / 64) * (kM * 128) + ml * 128;     // 64 bf16 columns = one box row
#pragma unroll
            for (int q16 = 0; q16 < 8; ++q16)
                *reinterpret_cast<uint4*>(box + (((uint32_t)q16 ^ (uint32_t)(ml & 7)) << 4)) =
                    make_uint4(w[4 * q16], w[4 * q16 + 1], w[4 * q16 + 2], w[4 * q16 + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            // rows past the group's rows fall outside the tensor's row range and are not written
            for (int bx = 0; bx < kNMax / 64; ++bx)
                tma_store_3d(&tm_out, n0 + bx * 64, g * hpg, m0 / hpg, sm + bx * (kM * 128));
            dec::bulk_commit_group();
            dec::bulk_wait_read_all();          // the boxes are read out before the next q rows land
        }
        __syncthreads();
    }
    if (tid == 0) dec::bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kNMax);
    }
}

// q~ as a 3-D tensor {d_c, H, rows}: boxes {128 B of columns, hpg heads, 128 / hpg rows}, 128-byte swizzle.
bool make_qt_map(CUtensorMap* m, const void* qt, int esz, int rows, int H, int d_c, int hpg) {
    auto fn = dec::encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d_c, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d_c * esz, (cuuint64_t)H * d_c * esz};
    cuuint32_t box[3] = {(cuuint32_t)(128 / esz), (cuuint32_t)hpg, (cuuint32_t)(kM / hpg)};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, esz == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qt),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DH, int kN, typename OutT>
int launch_n(const float* q, const float* gq, const float* gk, const float* wk, int rows, int H, int G, int d_c,
             float eps, bool plain, void* qt, float* aq, cudaStream_t s) {
    using LY = AbsLayout<DH, kN>;
    static_assert(LY::kBytes <= 232448, "shared memory budget");
    // the staged output boxes must fit the drained operand region
    constexpr bool kBoxesFit = kN * (int)sizeof(OutT) / 128 * kM * 128 <= LY::kOffG;
    auto k = absorb_tc_kernel<DH, kN, OutT>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes) != cudaSuccess)
        return QKMLA_ERR_CUDA;
    const int hpg = H / G;
    const int M = rows * hpg;
    // TMA stores when a 128-row tile is whole query rows of the group (hpg divides 128)
    const int tma_out = (kBoxesFit && kM % hpg == 0 && (uintptr_t)qt % 16 == 0) ? 1 : 0;
    CUtensorMap tq;
    memset(&tq, 0, sizeof(tq));
    if (tma_out && !make_qt_map(&tq, qt, (int)sizeof(OutT), rows, H, d_c, hpg)) return QKMLA_ERR_CUDA;
    dim3 grid((M + kM - 1) / kM, d_c / kN, G);
    return launch_pdl(k, grid, dim3(kThreads), LY::kBytes, s, tq, q, gq, gk, wk, rows, H, G, d_c, eps, plain ? 1 : 0,
                      tma_out, (OutT*)qt, aq, device_status_ptr()) == cudaSuccess
               ? QKMLA_OK
               : QKMLA_ERR_CUDA;
}

// Persistent CTAs keeping a W_g half resident (d_h = 128, bf16 q~, enough row tiles
// per (group, half) for the W split to pay off): cpp CTAs per (group, half).
int launch_persistent(const float* q, const float* gq, const float* gk, const float* wk, int rows, int H, int G,
                      int d_c, float eps, bool plain, void* qt, float* aq, int cpp, cudaStream_t s) {
    using LY = AbsLayout<128, kNMax>;
    auto k = absorb_tc_persistent<128>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes) != cudaSuccess)
        return QKMLA_ERR_CUDA;
    CUtensorMap tq;
    if (!make_qt_map(&tq, qt, 2, rows, H, d_c, H / G)) return QKMLA_ERR_CUDA;
    dim3 grid(cpp * G * (d_c / kNMax));
    return launch_pdl(k, grid, dim3(kThreads), LY::kBytes, s, tq, q, gq, gk, wk, rows, H, G, d_c, eps, plain ? 1 : 0,
                      cpp, (__nv_bfloat16*)qt, aq, device_status_ptr()) == cudaSuccess
               ? QKMLA_OK
               : QKMLA_ERR_CUDA;
}

// 256-latent tiles, or 64-latent ones when the 256-wide grid has fewer than 64 CTAs.
template <int DH, typename OutT>
int launch_t(const float* q, const float* gq, const float* gk, const float* wk, int rows, int H, int G, int d_c,
             float eps, bool plain, void* qt, float* aq, cudaStream_t s) {
    const int M = rows * (H / G);
    const int hpg = H / G;
    const int pairs = G * (d_c / kNMax);
    const int n_tiles = (M + kM - 1) / kM;
    if constexpr (DH == 128 && sizeof(OutT) == 2) {
        // at least two tiles per persistent CTA when every SM gets one
        const int cpp = std::max(1, device_sm_count() / pairs);
        if (kM % hpg == 0 && (uintptr_t)qt % 16 == 0 && pairs <= device_sm_count() && n_tiles >= 2 * cpp)
            return launch_persistent(q, gq, gk, wk, rows, H, G, d_c, eps, plain, qt, aq, cpp, s);
    }
    const int ctas_wide = n_tiles * (d_c / kNMax) * G;
    return ctas_wide < 64 ? launch_n<DH, 64, OutT>(q, gq, gk, wk, rows, H, G, d_c, eps, plain, qt, aq, s)
                          : launch_n<DH, kNMax, OutT>(q, gq, gk, wk, rows, H, G, d_c, eps, plain, qt, aq, s);
}

}  // namespace

// Shapes the tensor-core absorb handles: d_h in {64, 128}, d_c a multiple of
// 256, 16-byte aligned fp32 inputs.
bool absorb_tc_supported(const float* q, const float* wk, int d_h, int d_c) {
    if (d_h != 64 && d_h != 128) return false;
    if (d_c % kNMax) return false;
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
