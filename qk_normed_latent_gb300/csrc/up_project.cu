// qkmla_up_project: per-head values from the latent-space decode output.
//
// Source: "QK-Normed MLA: QK normalization without full key caching", Technical
// Summary, Problem Statement -- MLA caches only the latent c_t and recovers
// per-head quantities through up-projections (W^K_g for the key).  Decode keeps
// the latent path (the abstract), so attention returns o_h = sum_t p_t c_t and
// the value of head h is recovered once per query row:
//     v_h = o_h W^V_{g(h)},   W^V_g: d_c x d_v,  g(h) = h / (H / G_v).
// (Softmax weights sum to one, so this equals attention over materialised values
// c_t W^V_g.)
//
// Per group g this is the GEMM  V_g = O_g W^V_g  with O_g the [rows*H/G_v, d_c]
// rows of the group's heads.  A CTA owns 128 of those rows and all d_v output
// columns: M = 128, N = d_v, K = d_c in blocks of 64 through two shared-memory
// stages.  W^V_g blocks arrive by TMA as an MN-major operand (64 K-rows of 64
// output columns per box); the o rows are loaded by the threads (thread = row)
// and written K-major with the 128-byte swizzle.  An fp32 o is split into
// bf16 hi + lo (two MMAs per K-step, the weights being exact in bf16), so the
// product keeps fp32-level accuracy; a bf16 o takes one MMA.  fp32 accumulation
// in TMEM; the epilogue writes fp32 or bf16.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "tc_ptx.cuh"

namespace qkmla {

namespace {

using namespace tc;

constexpr int kM = 128;            // rows per CTA (MMA M)
constexpr int kKB = 64;            // K (d_c) per stage
constexpr int kThreadsU = 128;

template <int DV>
struct UpLayout {
    static constexpr int kA = kM * kKB * 2;                 // one bf16 A tile (hi or lo), 16 KB
    static constexpr int kB = kKB * DV * 2;                 // W^V block: DV/64 boxes of 64 x 64 bf16
    static constexpr int kStage = 2 * kA + kB;
    static constexpr int kOffMisc = 2 * kStage;
    static constexpr int kBytes = kOffMisc + 64 + 1024;
    static constexpr uint32_t kTmemCols = DV <= 64 ? 64 : DV <= 128 ? 128 : 256;
    static_assert(DV % 64 == 0 && DV <= 256, "d_v is 64, 128, 192 or 256");
    static_assert(kStage % 1024 == 0, "stage alignment");
};

template <typename OT>
__device__ __forceinline__ void load8(const OT* src, float (&x)[8]);
template <>
__device__ __forceinline__ void load8<float>(const float* src, float (&x)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(src));
    const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* src, float (&x)[8]) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

template <typename OT, typename OutT, int DV>
__global__ void __launch_bounds__(kThreadsU)
up_project_kernel(const __grid_constant__ CUtensorMap tm_w, const OT* __restrict__ o, int rows, int H, int Gv,
                  int d_c, OutT* __restrict__ out, int* status) {
    using LY = UpLayout<DV>;
    constexpr bool kSplit = sizeof(OT) == 4;                // fp32 o: hi + lo
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t* bfull = reinterpret_cast<uint64_t*>(sm + LY::kOffMisc);   // [2] W^V block landed
    uint64_t* mdone = bfull + 2;                                        // [2] MMAs of a stage done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 2);
    int* fail = reinterpret_cast<int*>(tmem_slot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.y;
    const int hpg = H / Gv;
    const int M = rows * hpg;
    const int m = blockIdx.x * kM + tid;                    // this thread's row of the group
    const bool row_ok = m < M;
    const int r = row_ok ? m / hpg : 0;
    const int h = g * hpg + (row_ok ? m % hpg : 0);
    const OT* orow = o + ((size_t)r * H + h) * d_c;
    const int nkb = d_c / kKB;

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bfull[i], 1);
        *fail = 0;
        fence_barrier_init();
        prefetch_tmap(&tm_w);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, LY::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_trigger();

    const uint32_t idesc = idesc_bf16(kM, DV, 0, 1);
    auto issue_b = [&](int kb) {             // thread 0: W^V block kb into stage kb & 1
        uint8_t* stg = sm + (kb & 1) * LY::kStage;
        mbar_arrive_expect_tx(&bfull[kb & 1], (uint32_t)LY::kB);
#pragma unroll
        for (int bx = 0; bx < DV / 64; ++bx)
            tma_load_2d(stg + 2 * LY::kA + bx * (kKB * 128), &tm_w, bx * 64, g * d_c + kb * kKB, &bfull[kb & 1]);
    };
    auto load_a = [&](int kb, float (&x)[kKB]) {   // this thread's row, K-block kb
#pragma unroll
        for (int c8 = 0; c8 < kKB / 8; ++c8) {
            float y[8];
            if (row_ok) {
                load8<OT>(orow + kb * kKB + 8 * c8, y);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) y[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) x[8 * c8 + i] = y[i];
        }
    };
    int pending = -1;                        // thread 0: a W^V block issued and not yet waited for
    if (tid == 0) {
        issue_b(0);
        pending = 0;
    }
    bool ok = true;
    float xa[kKB];
    if (nkb > 0) load_a(0, xa);
    for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb & 1;
        uint8_t* stg = sm + s * LY::kStage;
        // stage s is free once the MMAs of block kb - 2 have read it
        if (kb >= 2 && !mbar_wait(&mdone[s], ((kb >> 1) - 1) & 1, 1u << 26)) ok = false;
        if (__syncthreads_or(!ok)) { ok = false; break; }
        // A: block kb as bf16 (hi, and lo for an fp32 o), K-major, 128-byte swizzle
#pragma unroll
        for (int c8 = 0; c8 < kKB / 8; ++c8) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float x0 = xa[8 * c8 + 2 * i], x1 = xa[8 * c8 + 2 * i + 1];
                const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
                hi[i] = *reinterpret_cast<const uint32_t*>(&hh);
                if (kSplit) {
                    const __nv_bfloat162 ll = __floats2bfloat162_rn(x0 - __low2float(hh), x1 - __high2float(hh));
                    lo[i] = *reinterpret_cast<const uint32_t*>(&ll);
                }
            }
            const uint32_t off = sw128_offset(tid, 8 * c8);
            *reinterpret_cast<uint4*>(stg + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            if (kSplit) *reinterpret_cast<uint4*>(stg + LY::kA + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            if (!mbar_wait(&bfull[s], (kb >> 1) & 1, 1u << 26)) {
                *(volatile int*)fail = 1;
            } else {
                pending = -1;
                tc_fence_after();
                const uint32_t a_hi = smem_u32(stg), a_lo = smem_u32(stg + LY::kA);
                const uint32_t b = smem_u32(stg + 2 * LY::kA);
#pragma unroll
                for (int kk = 0; kk < kKB / 16; ++kk) {
                    // B: W^V rows (K) kb*64 + 16 kk .. +15, all DV columns (boxes LBO apart), MN-major
                    const uint64_t bd = smem_desc(b + kk * 2048, kKB * 128, 1024, kSwizzle128B);
                    mma_bf16(tmem, smem_desc(a_hi + kk * 32, 16, 1024, kSwizzle128B), bd, idesc,
                             (kb > 0 || kk > 0) ? 1u : 0u);
                    if (kSplit) mma_bf16(tmem, smem_desc(a_lo + kk * 32, 16, 1024, kSwizzle128B), bd, idesc, 1u);
                }
                mma_commit(&mdone[s]);
                // W^V block kb + 1 into the other stage once the MMAs of block kb - 1 are done
                if (kb + 1 < nkb) {
                    if (kb >= 1 && !mbar_wait(&mdone[s ^ 1], ((kb - 1) >> 1) & 1, 1u << 26)) {
                        *(volatile int*)fail = 1;
                    } else {
                        issue_b(kb + 1);
                        pending = kb + 1;
                    }
                }
            }
        }
        // the next block's o rows load while the MMAs run
        if (kb + 1 < nkb) load_a(kb + 1, xa);
        __syncthreads();
        if (*(volatile int*)fail) { ok = false; break; }
    }
    // every MMA done before TMEM is read (the last two stages' barriers, in order)
    if (ok) {
        for (int kb = max(0, nkb - 2); kb < nkb; ++kb)
            if (!mbar_wait(&mdone[kb & 1], (kb >> 1) & 1, 1u << 26)) ok = false;
    }
    if (!ok) {
        if (tid == 0) report(status, QKMLA_ERR_TIMEOUT);
        // a W^V copy still in flight lands before the CTA's memory is released
        if (tid == 0 && pending >= 0) mbar_wait(&bfull[pending & 1], (pending >> 1) & 1, 1u << 26);
    }
    ok = __syncthreads_and(ok) != 0;
    tc_fence_after();
    if (ok) {
        // epilogue: thread = row (TMEM lane), DV columns
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        OutT* dst = out + ((size_t)r * H + h) * DV;
#pragma unroll 1
        for (int c16 = 0; c16 < DV; c16 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + lane_base + c16, v);
            tmem_wait_ld();
            if (!row_ok) continue;
            if constexpr (sizeof(OutT) == 4) {
                float4* d4 = reinterpret_cast<float4*>(dst + c16);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                        __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            } else {
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    w[i] = *reinterpret_cast<const uint32_t*>(&b2);
                }
                uint4* d4 = reinterpret_cast<uint4*>(dst + c16);
                d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
                d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, LY::kTmemCols);
    }
}

template <typename OT, typename OutT, int DV>
int launch_up(const CUtensorMap& tm, const void* o, int rows, int H, int Gv, int d_c, void* out, cudaStream_t s) {
    using LY = UpLayout<DV>;
    auto k = up_project_kernel<OT, OutT, DV>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes) != cudaSuccess)
        return QKMLA_ERR_CUDA;
    const int M = rows * (H / Gv);
    dim3 grid((M + kM - 1) / kM, Gv);
    return launch_pdl(k, grid, dim3(kThreadsU), LY::kBytes, s, tm, (const OT*)o, rows, H, Gv, d_c, (OutT*)out,
                      device_status_ptr()) == cudaSuccess
               ? QKMLA_OK
               : QKMLA_ERR_CUDA;
}

template <typename OT, typename OutT>
int launch_dv(const CUtensorMap& tm, const void* o, int rows, int H, int Gv, int d_c, int d_v, void* out,
              cudaStream_t s) {
    switch (d_v) {
        case 64: return launch_up<OT, OutT, 64>(tm, o, rows, H, Gv, d_c, out, s);
        case 128: return launch_up<OT, OutT, 128>(tm, o, rows, H, Gv, d_c, out, s);
        case 192: return launch_up<OT, OutT, 192>(tm, o, rows, H, Gv, d_c, out, s);
        case 256: return launch_up<OT, OutT, 256>(tm, o, rows, H, Gv, d_c, out, s);
    }
    return QKMLA_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace qkmla

using namespace qkmla;

extern "C" int qkmla_up_project(const void* o, int o_dtype, const void* w_v, int rows, int H, int G_v, int d_c,
                                int d_v, void* out, int out_dtype, void* stream) {
    if (rows < 1 || H < 1 || G_v < 1 || d_c < 1 || d_v < 1 || H % G_v) return QKMLA_ERR_INVALID;
    if (!o || !w_v || !out) return QKMLA_ERR_INVALID;
    if ((o_dtype != QKMLA_F32 && o_dtype != QKMLA_BF16) || (out_dtype != QKMLA_F32 && out_dtype != QKMLA_BF16))
        return QKMLA_ERR_UNSUPPORTED;
    if (d_c % 64 || d_v % 64 || d_v > 256) return QKMLA_ERR_UNSUPPORTED;
    if (((uintptr_t)o % 16) || ((uintptr_t)w_v % 16) || ((uintptr_t)out % 16)) return QKMLA_ERR_INVALID;
    // W^V as a 2-D bf16 tensor [G_v * d_c][d_v]: 64 x 64 boxes, 128-byte swizzle
    CUtensorMap tm;
    if (!dec::make_map(&tm, w_v, (int64_t)G_v * d_c, d_v, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return QKMLA_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (o_dtype == QKMLA_F32)
        return out_dtype == QKMLA_F32 ? launch_dv<float, float>(tm, o, rows, H, G_v, d_c, d_v, out, s)
                                      : launch_dv<float, __nv_bfloat16>(tm, o, rows, H, G_v, d_c, d_v, out, s);
    return out_dtype == QKMLA_F32 ? launch_dv<__nv_bfloat16, float>(tm, o, rows, H, G_v, d_c, d_v, out, s)
                                  : launch_dv<__nv_bfloat16, __nv_bfloat16>(tm, o, rows, H, G_v, d_c, d_v, out, s);
}
