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
// Per group g this is the GEMM  V_g = O_g W^V_g  with O_g the rows of the group's
// heads.  It is HBM-bound (o is the traffic: fp32 o is 4 d_c bytes a row against
// 2 d_c d_v weight bytes a group), so every operand arrives by TMA through a ring
// deep enough to keep ~100 KB of loads in flight per SM.  A CTA owns one tile of
// up to 128 rows -- nr query rows x bh heads of one group, one 3-D TMA box
// {64 columns, bh heads, nr rows} of o per K-block, so the tile's rows are
// contiguous in shared memory -- and all d_v output columns: M = 128, N = d_v,
// K = d_c in 64-wide blocks.  W^V_g blocks arrive as an MN-major operand (64
// K-rows of 64 output columns per box).
//   * bf16 o: the o box (128-byte swizzle) is the MMA's A operand as it lands.
//   * fp32 o: two 32-column boxes per K-block (128-byte swizzle); the four
//     converter warps (thread = row) split each value into bf16 hi + lo and
//     write them back in place -- row m's 256 bytes become its hi row (64 bf16,
//     K-major, 128-byte swizzle) in the first half and its lo row in the second,
//     so a thread only touches its own row -- and the MMA warp issues two MMAs
//     per K-step (the weights are exact in bf16), which keeps fp32-level accuracy.
// Two CTAs fit on an SM (two stages each), so the usual grid runs in one wave.
// Warps: 0 TMA producer, 1-4 converters and epilogue (thread = row = TMEM lane),
// 5 MMA issuer.  fp32 accumulation in TMEM; the epilogue stages the tile as
// 128-byte boxes of fp32 or bf16 values (the o box's shape, 128-byte swizzle) in
// the drained ring and writes them with TMA stores, whole lines at a time.
// All waits are bounded; a CTA that gives up waits for its loads and MMAs.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "tc_ptx.cuh"

namespace qkmla {

namespace {

using namespace tc;

constexpr int kM = 128;            // rows per CTA (MMA M)
constexpr int kKB = 64;            // K (d_c) per stage
constexpr int kThreadsU = 192;
constexpr int kSmemU = 232448;
constexpr int kSmemHalf = 115712;  // per CTA when two share an SM (228 KB less 1 KB reserved each)

template <typename OT, int DV>
struct UpLayout {
    static constexpr bool kSplit = sizeof(OT) == 4;
    static constexpr int kTile = kM * 128;                          // 128 rows x 128 B (one swizzled box)
    static constexpr int kO = kSplit ? 2 * kTile : kTile;           // the o K-block as it lands
    static constexpr int kW = DV * 128;                             // W^V block: DV/64 boxes of 64 x 64 bf16
    static constexpr int kStage = kO + kW;
    static constexpr int kMisc = 256;
    // two CTAs an SM when two (fp32 o) or three (bf16 o) stages fit in half of it
    static constexpr int kNstTwo = kSplit ? 2 : 3;
    static constexpr bool kTwoPerSm = kNstTwo * kStage + kMisc + 1024 <= kSmemHalf;
    static constexpr int kNst = kTwoPerSm ? kNstTwo : 3;
    static constexpr int kOffMisc = kNst * kStage;
    static constexpr int kBytes = kOffMisc + kMisc + 1024;
    static constexpr uint32_t kTmemCols = DV <= 64 ? 64 : DV <= 128 ? 128 : 256;
    static_assert(DV % 64 == 0 && DV <= 256, "d_v is 64, 128, 192 or 256");
    static_assert(kStage % 1024 == 0, "stage alignment");
    static_assert(kBytes <= kSmemU, "shared memory budget");
};

template <typename OT, typename OutT, int DV>
__global__ void __launch_bounds__(kThreadsU, 2)
up_project_kernel(const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_w,
                  const __grid_constant__ CUtensorMap tm_v, int rows, int H, int Gv, int d_c, int bh, int nr, int nhb,
                  int tma_out, OutT* __restrict__ out, int* status) {
    using LY = UpLayout<OT, DV>;
    constexpr bool kSplit = LY::kSplit;
    constexpr int kNst = LY::kNst;
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + LY::kOffMisc);   // [kNst] o + W^V block landed
    uint64_t* sfree = full + kNst;                                      // [kNst] MMAs done with the stage
    uint64_t* aready = sfree + kNst;                                    // [kNst] converters rewrote the stage's o
    uint64_t* done = aready + kNst;                                     // every MMA done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    int* fail = reinterpret_cast<int*>(tmem_slot + 1);
    int* issued_s = fail + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.y;
    const int hpg = H / Gv;
    const int rb = blockIdx.x / nhb, hb = blockIdx.x % nhb;
    const int r0 = rb * nr, i0 = hb * bh;
    const int m_t = nr * bh;                                            // rows of the tile (<= 128)
    const int nkb = d_c / kKB;
    // the CTAs of a group read the same W^V_g: each starts its K walk at its own block
    const int kb0 = (int)(((unsigned)blockIdx.x * 3u) % (unsigned)nkb);
    const uint32_t stage_tx = (uint32_t)((kSplit ? 2 : 1) * m_t * 128 + LY::kW);

    if (tid == 0) {
        for (int i = 0; i < 3 * kNst + 1; ++i) mbar_init(&full[i], (i >= 2 * kNst && i < 3 * kNst) ? 128u : 1u);
        *fail = 0;
        *issued_s = 0;
        fence_barrier_init();
        prefetch_tmap(&tm_o);
        prefetch_tmap(&tm_w);
        if (tma_out) prefetch_tmap(&tm_v);
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

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer ----
            int kb = 0;
            for (; kb < nkb; ++kb) {
                const int s = kb % kNst;
                if (kb >= kNst && !dec::wait_bounded(&sfree[s], ((kb / kNst) - 1) & 1, status)) break;
                if (*(volatile int*)fail) break;
                uint8_t* stg = sm + s * LY::kStage;
                mbar_arrive_expect_tx(&full[s], stage_tx);
                const int kx = ((kb + kb0) % nkb) * kKB;
                tma_load_3d(stg, &tm_o, kx, g * hpg + i0, r0, &full[s]);
                if (kSplit) tma_load_3d(stg + LY::kTile, &tm_o, kx + 32, g * hpg + i0, r0, &full[s]);
#pragma unroll
                for (int bx = 0; bx < DV / 64; ++bx)
                    tma_load_2d(stg + LY::kO + bx * (kKB * 128), &tm_w, bx * 64, g * d_c + kx, &full[s]);
            }
            *(volatile int*)issued_s = kb;
            if (kb < nkb) *(volatile int*)fail = 1;
        }
    } else if (warp == 5) {
        if (lane == 0) {
            // ---- MMA issuer ----
            const uint32_t idesc = idesc_bf16(kM, DV, 0, 1);
            int kb = 0;
            for (; kb < nkb; ++kb) {
                const int s = kb % kNst;
                if (!dec::wait_bounded(&full[s], (kb / kNst) & 1, status)) break;
                if (kSplit && !dec::wait_bounded(&aready[s], (kb / kNst) & 1, status)) break;
                tc_fence_after();
                const uint32_t stg = smem_u32(sm + s * LY::kStage);
                const uint32_t a_hi = stg, a_lo = stg + LY::kTile;
                const uint32_t b = stg + LY::kO;
#pragma unroll
                for (int kk = 0; kk < kKB / 16; ++kk) {
                    // B: W^V rows (K) kb*64 + 16 kk .. +15, all DV columns (boxes LBO apart), MN-major
                    const uint64_t bd = smem_desc(b + kk * 2048, kKB * 128, 1024, kSwizzle128B);
                    mma_bf16(tmem, smem_desc(a_hi + kk * 32, 16, 1024, kSwizzle128B), bd, idesc,
                             (kb > 0 || kk > 0) ? 1u : 0u);
                    if (kSplit) mma_bf16(tmem, smem_desc(a_lo + kk * 32, 16, 1024, kSwizzle128B), bd, idesc, 1u);
                }
                mma_commit(&sfree[s]);
            }
            if (kb < nkb) *(volatile int*)fail = 1;
            mma_commit(done);      // tracks every MMA this thread issued
        }
    } else if (kSplit) {
        // ---- converters: fp32 row -> bf16 hi + lo (thread = row = TMEM lane) ----
        const uint32_t mrow = (uint32_t)(32 * (warp & 3) + lane);
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % kNst;
            if (!dec::wait_bounded(&full[s], (kb / kNst) & 1, status) || *(volatile int*)fail) {
                *(volatile int*)fail = 1;
                break;
            }
            uint8_t* row = sm + s * LY::kStage + mrow * 128;
            float x[kKB];
#pragma unroll
            for (int q = 0; q < kKB / 4; ++q) {
                // 16-byte chunk q: half q / 8 of the K-block, chunk q % 8 of the row, swizzled
                const float4 f = *reinterpret_cast<const float4*>(row + (q >> 3) * LY::kTile +
                                                                 (((uint32_t)(q & 7) ^ (mrow & 7u)) << 4));
                x[4 * q] = f.x; x[4 * q + 1] = f.y; x[4 * q + 2] = f.z; x[4 * q + 3] = f.w;
            }
#pragma unroll
            for (int c8 = 0; c8 < kKB / 8; ++c8) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float x0 = x[8 * c8 + 2 * i], x1 = x[8 * c8 + 2 * i + 1];
                    const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
                    const __nv_bfloat162 ll = __floats2bfloat162_rn(x0 - __low2float(hh), x1 - __high2float(hh));
                    hi[i] = *reinterpret_cast<const uint32_t*>(&hh);
                    lo[i] = *reinterpret_cast<const uint32_t*>(&ll);
                }
                const uint32_t off = ((uint32_t)c8 ^ (mrow & 7u)) << 4;
                *reinterpret_cast<uint4*>(row + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(row + LY::kTile + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&aready[s]);
        }
    }
    __syncthreads();
    // every MMA has completed before TMEM is read (or released); a failed CTA also
    // waits for the loads it issued that no MMA consumed
    const bool got = dec::wait_bounded(done, 0, status);
    const bool failed = __syncthreads_or(*(volatile int*)fail != 0 || !got) != 0;   // uniform: the epilogue syncs
    constexpr int kCols = 128 / (int)sizeof(OutT);                     // output columns per 128-byte box
    if (failed) {
        if (tid == 0) {
            const int issued = *(volatile int*)issued_s;
            for (int j = max(0, issued - kNst); j < issued; ++j)
                dec::wait_bounded(&full[j % kNst], (j / kNst) & 1, status);
        }
    } else {
        if (warp >= 1 && warp <= 4) {
            tc_fence_after();
            // ---- epilogue: thread = row (TMEM lane), DV columns ----
            const uint32_t mrow = (uint32_t)(32 * (warp & 3) + lane);
            const int z = (int)mrow / bh, i = i0 + (int)mrow % bh;
            const int r = r0 + z;
            const bool row_ok = (int)mrow < m_t && r < rows && i < hpg;
            const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
            OutT* dst = out + ((size_t)r * H + g * hpg + i) * DV;
#pragma unroll 1
            for (int c32 = 0; c32 < DV; c32 += 32) {
                uint32_t v[32];
                tmem_ld16(tmem + lane_base + c32, *reinterpret_cast<uint32_t(*)[16]>(v));
                tmem_ld16(tmem + lane_base + c32 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
                tmem_wait_ld();
                uint32_t w[32];                                     // the 32 values as stored: 128 B or 64 B
                if constexpr (sizeof(OutT) == 4) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) w[q] = v[q];
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
                        w[q] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
                }
                constexpr int kChunks = 32 * (int)sizeof(OutT) / 16;   // 16-byte chunks of these 32 values
                if (tma_out) {
                    // box c32 / kCols, its 16-byte chunks from (c32 % kCols) * sizeof(OutT) / 16, swizzled by row
                    uint8_t* box = sm + (c32 / kCols) * LY::kTile + mrow * 128;
                    const uint32_t ch0 = (uint32_t)((c32 % kCols) * (int)sizeof(OutT) / 16);
#pragma unroll
                    for (int q = 0; q < kChunks; ++q)
                        *reinterpret_cast<uint4*>(box + (((ch0 + q) ^ (mrow & 7u)) << 4)) =
                            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                } else if (row_ok) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c32);
#pragma unroll
                    for (int q = 0; q < kChunks; ++q) d4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                }
            }
            if (tma_out) fence_proxy_async_smem();
        }
        if (tma_out) {
            __syncthreads();
            if (tid == 0) {
                // rows past `rows` fall outside the tensor and are not written
                for (int bx = 0; bx < DV / kCols; ++bx)
                    tma_store_3d(&tm_v, bx * kCols, g * hpg + i0, r0, sm + bx * LY::kTile);
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
        tmem_dealloc(tmem, LY::kTmemCols);
    }
}

// o (or the output) as a 3-D tensor {cols, H, rows} (fp32 or bf16), boxes {128 B of columns, bh heads, nr rows}.
bool make_o_map(CUtensorMap* m, const void* o, int esz, int rows, int H, int d_c, int bh, int nr) {
    auto fn = dec::encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d_c, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d_c * esz, (cuuint64_t)H * d_c * esz};
    cuuint32_t box[3] = {(cuuint32_t)(128 / esz), (cuuint32_t)bh, (cuuint32_t)nr};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, esz == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(o),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename OT, typename OutT, int DV>
int launch_up(const CUtensorMap& tw, const void* o, int rows, int H, int Gv, int d_c, void* out, cudaStream_t s) {
    static_assert(DV / (128 / (int)sizeof(OutT)) * UpLayout<OT, DV>::kTile <= UpLayout<OT, DV>::kOffMisc,
                  "the output boxes fit in the ring");
    using LY = UpLayout<OT, DV>;
    auto k = up_project_kernel<OT, OutT, DV>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes) != cudaSuccess)
        return QKMLA_ERR_CUDA;
    // a tile: nr query rows x bh heads of one group (nr bh <= 128)
    const int hpg = H / Gv;
    const int bh = hpg < kM ? hpg : kM;
    const int nr = hpg < kM ? kM / hpg : 1;
    const int nhb = (hpg + bh - 1) / bh;
    CUtensorMap to, tv;
    if (!make_o_map(&to, o, (int)sizeof(OT), rows, H, d_c, bh, nr)) return QKMLA_ERR_CUDA;
    // the output by TMA store when a tile's box never reaches into the next group's heads
    const int tma_out = (hpg <= kM || hpg % kM == 0) ? 1 : 0;
    memset(&tv, 0, sizeof(tv));
    if (tma_out && !make_o_map(&tv, out, (int)sizeof(OutT), rows, H, DV, bh, nr)) return QKMLA_ERR_CUDA;
    dim3 grid(((rows + nr - 1) / nr) * nhb, Gv);
    return launch_pdl(k, grid, dim3(kThreadsU), LY::kBytes, s, to, tw, tv, rows, H, Gv, d_c, bh, nr, nhb, tma_out,
                      (OutT*)out, device_status_ptr()) == cudaSuccess
               ? QKMLA_OK
               : QKMLA_ERR_CUDA;
}

template <typename OT, typename OutT>
int launch_dv(const CUtensorMap& tw, const void* o, int rows, int H, int Gv, int d_c, int d_v, void* out,
              cudaStream_t s) {
    switch (d_v) {
        case 64: return launch_up<OT, OutT, 64>(tw, o, rows, H, Gv, d_c, out, s);
        case 128: return launch_up<OT, OutT, 128>(tw, o, rows, H, Gv, d_c, out, s);
        case 192: return launch_up<OT, OutT, 192>(tw, o, rows, H, Gv, d_c, out, s);
        case 256: return launch_up<OT, OutT, 256>(tw, o, rows, H, Gv, d_c, out, s);
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
    CUtensorMap tw;
    if (!dec::make_map(&tw, w_v, (int64_t)G_v * d_c, d_v, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return QKMLA_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (o_dtype == QKMLA_F32)
        return out_dtype == QKMLA_F32 ? launch_dv<float, float>(tw, o, rows, H, G_v, d_c, d_v, out, s)
                                      : launch_dv<float, __nv_bfloat16>(tw, o, rows, H, G_v, d_c, d_v, out, s);
    return out_dtype == QKMLA_F32 ? launch_dv<__nv_bfloat16, float>(tw, o, rows, H, G_v, d_c, d_v, out, s)
                                  : launch_dv<__nv_bfloat16, __nv_bfloat16>(tw, o, rows, H, G_v, d_c, d_v, out, s);
}
