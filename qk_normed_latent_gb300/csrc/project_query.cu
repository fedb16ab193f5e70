// qkmla_project_query: the query projection ahead of the absorption, with the
// RoPE rotation of its RoPE block fused into the epilogue.
//
// Source: "QK-Normed MLA: QK normalization without full key caching", abstract
// (thelatestinai.com): the static key weight is absorbed into the MLA
// query-side projection -- the query comes from the layer input x through W^Q,
// and qkmla_absorb_query then folds gamma_q * gamma_k and W^K_g into it;
// Technical Summary, Methodology, "Blockwise Normalization" (the RoPE block is a
// separate, materialised vector; it is rotated here and normalised in decode).
//
//   [q_h | r_h] = x W^Q_h^T     (W^Q_h: (d_h + d_r) x d_x, one per head)
//   q[r][h]      = q_h                               (fp32)
//   q_rope[r][h] = RoPE(r_h, positions[r])           (fp32, not normalised)
//
// One CTA owns 128 rows (query tokens) and one head: the GEMM is M = 128,
// N = d_h + d_r, K = d_x in 64-wide blocks through a four-stage TMA ring (x and
// W^Q both K-major with the 128-byte swizzle); bf16 operands, fp32 accumulation
// in TMEM.  The epilogue (thread = row) rotates the RoPE pairs -- angles from
// the row's position by an exact fp32 reduction (rope.cuh) -- and writes both
// parts.  All waits are bounded.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "rope.cuh"
#include "tc_ptx.cuh"

namespace qkmla {

namespace {

using namespace tc;

constexpr int kPM = 128;           // rows per CTA
constexpr int kPK = 64;            // K per stage
constexpr int kPNst = 4;
constexpr int kPThreads = 128;
constexpr int kMaxDr = 64;

template <int N>
struct ProjLayout {
    static constexpr int kA = kPM * kPK * 2;         // x tile, 16 KB
    static constexpr int kB = N * kPK * 2;           // W^Q_h tile
    static constexpr int kStage = ((kA + kB) + 1023) / 1024 * 1024;
    static constexpr int kOffMisc = kPNst * kStage;
    static constexpr int kBytes = kOffMisc + 2 * kPNst * 8 + 16 + kMaxDr / 2 * 8 + 1024;
    static_assert(N % 16 == 0 && N <= 256, "N = d_h + d_r");
};

template <int N>
__global__ void __launch_bounds__(kPThreads, 1)
project_query_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     const int32_t* __restrict__ positions, float theta, int rows, int d_x, int H, int d_h, int d_r,
                     float* __restrict__ q, float* __restrict__ q_rope, int* status) {
    using LY = ProjLayout<N>;
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + LY::kOffMisc);     // [4] tiles landed
    uint64_t* empty = full + kPNst;                                       // [4] MMAs done with a stage
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(empty + kPNst);
    int* fail = reinterpret_cast<int*>(tmem_slot + 1);
    RopeFreq* freq = reinterpret_cast<RopeFreq*>(tmem_slot + 4);          // [d_r / 2]
    const int tid = threadIdx.x, warp = tid >> 5;
    const int h = blockIdx.y;
    const int r0 = blockIdx.x * kPM;
    const int nkb = d_x / kPK;

    if (tid == 0) {
        for (int i = 0; i < 2 * kPNst; ++i) mbar_init(&full[i], 1);
        *fail = 0;
        fence_barrier_init();
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_w);
    }
    if (tid < d_r / 2) freq[tid] = rope_freq(theta, tid, d_r);
    if (warp == 0) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_trigger();

    if (tid == 0) {
        // ---- one thread: TMA ring and MMAs ----
        const uint32_t idesc = idesc_bf16(kPM, N, 0, 0);
        auto issue = [&](int kb) {
            const int s = kb % kPNst;
            uint8_t* stg = sm + s * LY::kStage;
            mbar_arrive_expect_tx(&full[s], (uint32_t)(LY::kA + LY::kB));
            tma_load_2d(stg, &tm_x, kb * kPK, r0, &full[s]);
            tma_load_2d(stg + LY::kA, &tm_w, kb * kPK, h * N, &full[s]);
        };
        int issued = 0;
        for (; issued < kPNst && issued < nkb; ++issued) issue(issued);
        bool ok = true;
        int kb = 0;
        for (; kb < nkb; ++kb) {
            const int s = kb % kPNst;
            if (!mbar_wait(&full[s], (kb / kPNst) & 1, 1u << 26)) { ok = false; break; }
            tc_fence_after();
            const uint32_t a = smem_u32(sm + s * LY::kStage), b = a + LY::kA;
#pragma unroll
            for (int kk = 0; kk < kPK / 16; ++kk)
                mma_bf16(tmem, smem_desc(a + kk * 32, 16, 1024, kSwizzle128B),
                         smem_desc(b + kk * 32, 16, 1024, kSwizzle128B), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&empty[s]);
            if (issued < nkb) {
                // the stage is refilled once its MMAs are done
                if (!mbar_wait(&empty[s], (kb / kPNst) & 1, 1u << 26)) { ok = false; ++kb; break; }
                issue(issued++);
            }
        }
        if (ok && nkb > 0) {
            // the last MMAs (each stage's last phase, in order) before TMEM is read
            for (int j = max(0, nkb - kPNst); j < nkb; ++j)
                if (!mbar_wait(&empty[j % kPNst], (j / kPNst) & 1, 1u << 26)) ok = false;
        }
        if (!ok) {
            report(status, QKMLA_ERR_TIMEOUT);
            // tiles issued and not yet waited for land before the CTA's memory is released
            for (int j = kb; j < issued; ++j) mbar_wait(&full[j % kPNst], (j / kPNst) & 1, 1u << 26);
            *(volatile int*)fail = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*(volatile int*)fail == 0) {
        // ---- epilogue: thread = row (TMEM lane), N columns ----
        const int r = r0 + tid;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const int pos = (d_r > 0 && r < rows) ? positions[r] : 0;
        float* qd = q + ((size_t)r * H + h) * d_h;
        float* rd = q_rope + ((size_t)r * H + h) * d_r;
#pragma unroll 1
        for (int c16 = 0; c16 < N; c16 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + lane_base + c16, v);
            tmem_wait_ld();
            if (r >= rows) continue;
#pragma unroll
            for (int jj = 0; jj < 16; jj += 2) {
                const int j = c16 + jj;
                const float x0 = __uint_as_float(v[jj]), x1 = __uint_as_float(v[jj + 1]);
                if (j < d_h) {
                    *reinterpret_cast<float2*>(qd + j) = make_float2(x0, x1);
                } else {
                    // d_h is even: a pair never straddles the two parts
                    float c, s;
                    rope_cos_sin(pos, freq[(j - d_h) >> 1], &c, &s);
                    *reinterpret_cast<float2*>(rd + (j - d_h)) =
                        make_float2(rope_apply(0, x0, x1, c, s), rope_apply(1, x1, x0, c, s));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

template <int N>
int launch_proj(const CUtensorMap& tx, const CUtensorMap& tw, const int32_t* pos, float theta, int rows, int d_x,
                int H, int d_h, int d_r, float* q, float* qr, cudaStream_t s) {
    using LY = ProjLayout<N>;
    auto k = project_query_kernel<N>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes) != cudaSuccess)
        return QKMLA_ERR_CUDA;
    dim3 grid((rows + kPM - 1) / kPM, H);
    return launch_pdl(k, grid, dim3(kPThreads), LY::kBytes, s, tx, tw, pos, theta, rows, d_x, H, d_h, d_r, q, qr,
                      device_status_ptr()) == cudaSuccess
               ? QKMLA_OK
               : QKMLA_ERR_CUDA;
}

}  // namespace
}  // namespace qkmla

using namespace qkmla;

extern "C" int qkmla_project_query(const void* x, const void* w_q, const int32_t* positions, float rope_theta,
                                   int rows, int d_x, int H, int d_h, int d_r, float* q, float* q_rope,
                                   void* stream) {
    if (rows < 1 || d_x < 1 || H < 1 || d_h < 1 || d_r < 0) return QKMLA_ERR_INVALID;
    if (!x || !w_q || !q || (d_r > 0 && (!positions || !q_rope))) return QKMLA_ERR_INVALID;
    if (d_r > 0 && !(rope_theta > 1.f)) return QKMLA_ERR_INVALID;
    if (d_x % 64 || d_h % 2 || d_r % 2 || d_r > kMaxDr) return QKMLA_ERR_UNSUPPORTED;
    if (((uintptr_t)x % 16) || ((uintptr_t)w_q % 16) || ((uintptr_t)q % 8) || (q_rope && (uintptr_t)q_rope % 8))
        return QKMLA_ERR_INVALID;
    const int N = d_h + d_r;
    if (N % 16 || N > 256) return QKMLA_ERR_UNSUPPORTED;
    // x [rows][d_x] and W^Q [H * N][d_x], bf16, K-major boxes of 64 x (128 | N) rows
    CUtensorMap tx, tw;
    if (!dec::make_map(&tx, x, rows, d_x, kPK, kPM, CU_TENSOR_MAP_SWIZZLE_128B)) return QKMLA_ERR_CUDA;
    if (!dec::make_map(&tw, w_q, (int64_t)H * N, d_x, kPK, N, CU_TENSOR_MAP_SWIZZLE_128B)) return QKMLA_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    switch (N) {
        case 96: return launch_proj<96>(tx, tw, positions, rope_theta, rows, d_x, H, d_h, d_r, q, q_rope, s);
        case 128: return launch_proj<128>(tx, tw, positions, rope_theta, rows, d_x, H, d_h, d_r, q, q_rope, s);
        case 160: return launch_proj<160>(tx, tw, positions, rope_theta, rows, d_x, H, d_h, d_r, q, q_rope, s);
        case 192: return launch_proj<192>(tx, tw, positions, rope_theta, rows, d_x, H, d_h, d_r, q, q_rope, s);
        case 256: return launch_proj<256>(tx, tw, positions, rope_theta, rows, d_x, H, d_h, d_r, q, q_rope, s);
    }
    return QKMLA_ERR_UNSUPPORTED;
}
