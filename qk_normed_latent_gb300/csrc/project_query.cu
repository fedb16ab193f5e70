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
// At decode sizes W^Q and the fp32 outputs are the traffic (DeepSeek-V3 shape:
// 75 MB of weights and 25 MB of q / q_rope against 0.8 MB of x for 256 query
// rows), so each W^Q_h is streamed from HBM once: one CTA owns one head and up to
// 256 rows (two M = 128 accumulators, N = d_h + d_r each, in TMEM) and walks
// K = d_x in 64-wide blocks through a TMA ring (x and W^Q both K-major with the
// 128-byte swizzle; x stays in L2).
// Warp 0 issues the loads, warp 1 the MMAs (bf16 operands, fp32 accumulation);
// no thread waits for an MMA before issuing the next K-block.  Each CTA starts
// its K walk at a block of its own, so the CTAs spread their reads of the shared
// x over L2 instead of all requesting the same lines at once.  The epilogue
// (thread = row = TMEM lane, all four warps) rotates the RoPE pairs -- angles
// from the row's position by an exact fp32 reduction (rope.cuh) -- and stages
// 32-column boxes of q and q_rope (128-byte swizzle) in the drained ring, which
// TMA stores write out as whole 128-byte lines (a thread storing its own row
// would write every line in 8-byte pieces).  When d_h is not a multiple of 32
// the threads store their rows directly.  All waits are bounded; a CTA that gives up still waits for the
// loads it issued and the MMAs it started before it exits.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "rope.cuh"
#include "tc_ptx.cuh"

namespace qkmla {

namespace {

using namespace tc;

constexpr int kPM = 128;           // rows per accumulator (MMA M)
constexpr int kPAcc = 2;           // accumulators per CTA: up to 256 rows
constexpr int kPK = 64;            // K per stage
constexpr int kPThreads = 128;
constexpr int kMaxDr = 64;
constexpr int kSmemBudget = 232448;
constexpr int kBox = kPM * 128;    // one staged output box: 128 rows x 32 fp32

template <int N>
struct ProjLayout {
    static constexpr int kA = kPM * kPK * 2;                     // one x box: 128 rows x 64, 16 KB
    static constexpr int kB = N * kPK * 2;                       // W^Q_h box: N rows x 64
    static constexpr int kStage = kPAcc * kA + kB;               // multiple of 1024 (N % 8 == 0)
    static constexpr int kMisc = 1024;                           // barriers, flags, RoPE frequencies
    static constexpr int kFit = (kSmemBudget - kMisc - 1024) / kStage;
    static constexpr int kNst = kFit > 4 ? 4 : kFit;
    static constexpr int kOffMisc = kNst * kStage;
    static constexpr int kBytes = kOffMisc + kMisc + 1024;       // + alignment slack
    // output staging in the drained ring: one accumulator's N / 32 boxes, twice when both fit
    static constexpr int kPerAcc = N / 32 * kBox;
    static constexpr bool kBothFit = kPAcc * kPerAcc <= kNst * kStage;
    static constexpr uint32_t kTmemCols = kPAcc * N <= 256 ? 256 : 512;
    static_assert(N % 32 == 0 && N <= 256, "N = d_h + d_r: a multiple of 32");
    static_assert(kNst >= 2 && kPerAcc <= kNst * kStage, "ring");
    static_assert(kBytes <= kSmemBudget, "shared memory budget");
    static_assert((2 * kNst + 1) * 8 + 16 + kMaxDr / 2 * 8 <= kMisc, "misc region");
};

template <int N>
__global__ void __launch_bounds__(kPThreads, 1)
project_query_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_r,
                     const int32_t* __restrict__ positions, float theta, int rows, int d_x, int H, int d_h, int d_r,
                     int tma_out, float* __restrict__ q, float* __restrict__ q_rope, int* status) {
    using LY = ProjLayout<N>;
    constexpr int kNst = LY::kNst;
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + LY::kOffMisc);     // [kNst] tiles landed
    uint64_t* empty = full + kNst;                                        // [kNst] MMAs done with a stage
    uint64_t* done = empty + kNst;                                        // every MMA done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    int* fail = reinterpret_cast<int*>(tmem_slot + 1);
    int* issued_s = fail + 1;                                             // K-blocks whose loads were issued
    RopeFreq* freq = reinterpret_cast<RopeFreq*>(tmem_slot + 4);          // [d_r / 2]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    const int r0 = blockIdx.x * (kPAcc * kPM);
    const int n_acc = min(kPAcc, (rows - r0 + kPM - 1) / kPM);          // 1 or 2
    const int nkb = d_x / kPK;
    // every CTA reads the same x: each starts its K walk at its own block (the sum
    // order is free) so the CTAs do not all request the same x lines at once
    const int kb0 = (int)(((unsigned)h * 5u) % (unsigned)nkb);
    const uint32_t stage_tx = (uint32_t)(n_acc * LY::kA + LY::kB);

    if (tid == 0) {
        for (int i = 0; i < 2 * kNst + 1; ++i) mbar_init(&full[i], 1);
        *fail = 0;
        *issued_s = 0;
        fence_barrier_init();
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_w);
        if (tma_out) {
            prefetch_tmap(&tm_q);
            if (d_r > 0) prefetch_tmap(&tm_r);
        }
    }
    if (tid < d_r / 2) freq[tid] = rope_freq(theta, tid, d_r);
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

    if (warp == 0 && lane == 0) {
        // ---- TMA producer: x rows [r0, r0 + 128 n_acc) and W^Q_h, one 64-wide K-block a stage ----
        int kb = 0;
        for (; kb < nkb; ++kb) {
            const int s = kb % kNst;
            if (kb >= kNst && !dec::wait_bounded(&empty[s], ((kb / kNst) - 1) & 1, status)) break;
            if (*(volatile int*)fail) break;
            uint8_t* stg = sm + s * LY::kStage;
            mbar_arrive_expect_tx(&full[s], stage_tx);
            const int kx = ((kb + kb0) % nkb) * kPK;
            for (int m = 0; m < n_acc; ++m) tma_load_2d(stg + m * LY::kA, &tm_x, kx, r0 + m * kPM, &full[s]);
            tma_load_2d(stg + kPAcc * LY::kA, &tm_w, kx, h * N, &full[s]);
        }
        *(volatile int*)issued_s = kb;
        if (kb < nkb) *(volatile int*)fail = 1;
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        const uint32_t idesc = idesc_bf16(kPM, N, 0, 0);
        int kb = 0;
        for (; kb < nkb; ++kb) {
            const int s = kb % kNst;
            if (!dec::wait_bounded(&full[s], (kb / kNst) & 1, status)) break;
            tc_fence_after();
            const uint32_t a = smem_u32(sm + s * LY::kStage), b = a + kPAcc * LY::kA;
            for (int m = 0; m < n_acc; ++m) {
#pragma unroll
                for (int kk = 0; kk < kPK / 16; ++kk)
                    mma_bf16(tmem + m * N, smem_desc(a + m * LY::kA + kk * 32, 16, 1024, kSwizzle128B),
                             smem_desc(b + kk * 32, 16, 1024, kSwizzle128B), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&empty[s]);
        }
        if (kb < nkb) *(volatile int*)fail = 1;
        mma_commit(done);          // tracks every MMA this thread issued
    }
    __syncthreads();
    // every MMA has completed before TMEM is read (or released); a failed CTA also
    // waits for the loads it issued and the MMA thread did not consume
    const bool got = dec::wait_bounded(done, 0, status);
    const bool failed = __syncthreads_or(*(volatile int*)fail != 0 || !got) != 0;   // uniform: the epilogue syncs
    if (failed) {
        if (tid == 0) {
            const int issued = *(volatile int*)issued_s;
            for (int j = max(0, issued - kNst); j < issued; ++j)
                dec::wait_bounded(&full[j % kNst], (j / kNst) & 1, status);
        }
    } else {
        tc_fence_after();
        // ---- epilogue: thread = row (TMEM lane), N columns per accumulator ----
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const uint32_t mrow = (uint32_t)(32 * warp + lane);
        for (int m = 0; m < n_acc; ++m) {
            const int r = r0 + m * kPM + (int)mrow;
            const int pos = (d_r > 0 && r < rows) ? positions[r] : 0;
            float* qd = q + ((size_t)r * H + h) * d_h;
            float* rd = q_rope + ((size_t)r * H + h) * d_r;
            uint8_t* stage_out = sm + ((LY::kBothFit ? m : 0) * LY::kPerAcc);
            if (tma_out && !LY::kBothFit && m > 0) {
                // the previous accumulator's boxes are read out before they are overwritten
                if (tid == 0) dec::bulk_wait_read_all();
                __syncthreads();
            }
#pragma unroll 1
            for (int c32 = 0; c32 < N; c32 += 32) {
                uint32_t v[32];
                tmem_ld16(tmem + m * N + c32 + lane_base, *reinterpret_cast<uint32_t(*)[16]>(v));
                tmem_ld16(tmem + m * N + c32 + 16 + lane_base, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
                tmem_wait_ld();
                float o[32];
                if (c32 + 32 <= d_h) {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) o[jj] = __uint_as_float(v[jj]);
                } else if (c32 >= d_h) {
                    // a chunk of 16 RoPE pairs: their angles four at a time
#pragma unroll
                    for (int p4 = 0; p4 < 16; p4 += 4) {
                        float c[4], sn[4];
                        rope_cos_sin4(pos, &freq[(c32 - d_h) / 2 + p4], c, sn);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int jj = 2 * (p4 + i);
                            const float x0 = __uint_as_float(v[jj]), x1 = __uint_as_float(v[jj + 1]);
                            o[jj] = rope_apply(0, x0, x1, c[i], sn[i]);
                            o[jj + 1] = rope_apply(1, x1, x0, c[i], sn[i]);
                        }
                    }
                } else {
                    // the chunk straddles d_h (only when d_h is not a multiple of 32)
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 2) {
                        const int j = c32 + jj;
                        const float x0 = __uint_as_float(v[jj]), x1 = __uint_as_float(v[jj + 1]);
                        if (j < d_h) {
                            o[jj] = x0;
                            o[jj + 1] = x1;
                        } else {
                            float c, sn;
                            rope_cos_sin(pos, freq[(j - d_h) >> 1], &c, &sn);
                            o[jj] = rope_apply(0, x0, x1, c, sn);
                            o[jj + 1] = rope_apply(1, x1, x0, c, sn);
                        }
                    }
                }
                if (tma_out) {
                    // box c32 / 32: this row's 128 bytes, 16-byte chunks swizzled by row
                    uint8_t* box = stage_out + (c32 / 32) * kBox + mrow * 128;
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4)
                        *reinterpret_cast<float4*>(box + (((uint32_t)q4 ^ (mrow & 7u)) << 4)) =
                            make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
                } else if (r < rows) {
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 2) {
                        const int j = c32 + jj;
                        if (j < d_h) *reinterpret_cast<float2*>(qd + j) = make_float2(o[jj], o[jj + 1]);
                        else *reinterpret_cast<float2*>(rd + (j - d_h)) = make_float2(o[jj], o[jj + 1]);
                    }
                }
            }
            if (tma_out) {
                fence_proxy_async_smem();
                __syncthreads();
                if (tid == 0) {
                    // rows past `rows` fall outside the tensor and are not written
                    for (int c32 = 0; c32 < N; c32 += 32) {
                        const uint8_t* box = stage_out + (c32 / 32) * kBox;
                        if (c32 < d_h) tma_store_3d(&tm_q, c32, h, r0 + m * kPM, box);
                        else tma_store_3d(&tm_r, c32 - d_h, h, r0 + m * kPM, box);
                    }
                    dec::bulk_commit_group();
                }
            }
        }
        if (tma_out && tid == 0) dec::bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, LY::kTmemCols);
    }
}

// out as a 3-D fp32 tensor {cols, H, rows}: 32-column, one-head, 128-row boxes (128-byte swizzle)
bool make_out_map(CUtensorMap* m, const float* out, int rows, int H, int cols) {
    auto fn = dec::encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)H * cols * 4};
    cuuint32_t box[3] = {32, 1, (cuuint32_t)kPM};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(out), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
int launch_proj(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& tq, const CUtensorMap& tr,
                const int32_t* pos, float theta, int rows, int d_x, int H, int d_h, int d_r, int tma_out, float* q,
                float* qr, cudaStream_t s) {
    using LY = ProjLayout<N>;
    auto k = project_query_kernel<N>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes) != cudaSuccess)
        return QKMLA_ERR_CUDA;
    dim3 grid((rows + kPAcc * kPM - 1) / (kPAcc * kPM), H);
    return launch_pdl(k, grid, dim3(kPThreads), LY::kBytes, s, tx, tw, tq, tr, pos, theta, rows, d_x, H, d_h, d_r,
                      tma_out, q, qr, device_status_ptr()) == cudaSuccess
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
    if (N % 32 || N > 256) return QKMLA_ERR_UNSUPPORTED;
    // x [rows][d_x] and W^Q [H * N][d_x], bf16, K-major boxes of 64 x (128 | N) rows
    CUtensorMap tx, tw, tq, tr;
    if (!dec::make_map(&tx, x, rows, d_x, kPK, kPM, CU_TENSOR_MAP_SWIZZLE_128B)) return QKMLA_ERR_CUDA;
    if (!dec::make_map(&tw, w_q, (int64_t)H * N, d_x, kPK, N, CU_TENSOR_MAP_SWIZZLE_128B)) return QKMLA_ERR_CUDA;
    // outputs by TMA store when both parts tile into 32-column boxes on 16-byte aligned rows
    const int tma_out = (d_h % 32 == 0 && d_r % 32 == 0 && (uintptr_t)q % 16 == 0 &&
                         (d_r == 0 || (uintptr_t)q_rope % 16 == 0)) ? 1 : 0;
    memset(&tq, 0, sizeof(tq));
    memset(&tr, 0, sizeof(tr));
    if (tma_out && !make_out_map(&tq, q, rows, H, d_h)) return QKMLA_ERR_CUDA;
    if (tma_out && d_r > 0 && !make_out_map(&tr, q_rope, rows, H, d_r)) return QKMLA_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    switch (N) {
        case 96: return launch_proj<96>(tx, tw, tq, tr, positions, rope_theta, rows, d_x, H, d_h, d_r, tma_out, q, q_rope, s);
        case 128: return launch_proj<128>(tx, tw, tq, tr, positions, rope_theta, rows, d_x, H, d_h, d_r, tma_out, q, q_rope, s);
        case 160: return launch_proj<160>(tx, tw, tq, tr, positions, rope_theta, rows, d_x, H, d_h, d_r, tma_out, q, q_rope, s);
        case 192: return launch_proj<192>(tx, tw, tq, tr, positions, rope_theta, rows, d_x, H, d_h, d_r, tma_out, q, q_rope, s);
        case 256: return launch_proj<256>(tx, tw, tq, tr, positions, rope_theta, rows, d_x, H, d_h, d_r, tma_out, q, q_rope, s);
    }
    return QKMLA_ERR_UNSUPPORTED;
}
