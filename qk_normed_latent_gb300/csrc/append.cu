// qkmla_append kernel: write new tokens into the latent cache and A^k_cache.
//
// Source: "QK-Normed MLA: QK normalization without full key caching", Technical
// Summary, Methodology -- "Dynamic Scalar Caching" (one inverse-RMS scalar per
// token and KV group), "Cache Layout" (keep c_t, add A^k_cache, never store
// full keys) and "Blockwise Normalization" (the RoPE part is normalised on its
// own, as a materialised vector).
//
// Per KV group the key statistic needs k_{t,g} = c^_t W^K_g, a small GEMM
// [N, d_c] x [d_c, d_h] in fp32; the key itself is reduced to its sum of
// squares in registers and never leaves the CTA.  The grid is (token tiles) x G;
// the g = 0 CTAs also store the cast latent and the normalised RoPE key.
//
// A decode step appends a handful of tokens, so the kernel's time is the
// latency of streaming W^K_g (d_c x d_h fp32) through each CTA.  The main
// kernel therefore moves its operands with bulk copies: the token tile in one
// copy per token and W^K_g through a ring of kNST stages that are all in
// flight at once.  Shapes or pointers the bulk copies cannot take (rows that
// are not multiples of 16 bytes, misaligned bases) go to a plain-load kernel
// that forms every key element with the same fmaf chain over ascending k (its
// sum of squares is reduced across lanes in another order).
#include "common.cuh"
#include "tc_ptx.cuh"

namespace qkmla {

namespace {

constexpr int kTT = 32;        // tokens per CTA (plain-load kernel)
constexpr int kKC = 64;        // d_c chunk staged per step (plain-load kernel)
constexpr int kThreads = 256;
constexpr int kMaxJ = 8;       // d_h <= 256

// Bulk-copy kernel: a CTA owns FT tokens of one group.  W^K_g streams through a
// ring of kNST stages of kRows rows; warp w multiplies rows 4w .. 4w+3 of every
// stage into partial keys for all FT tokens x 32 NJ columns (lane + 32 j), so one
// float4 of the token tile feeds 4 NJ FMAs.  The eight warps' partial keys are
// summed in warp order through the (by then idle) ring memory.
constexpr int kNST = 4;
constexpr int kRows = 32;      // W^K_g rows per stage, 4 per warp
static_assert(kRows == 4 * (kThreads / 32), "four rows per warp and stage");

__host__ __device__ constexpr int bulk_ft(int nj) { return nj <= 4 ? 16 : 8; }
inline int bulk_nj(int d_h) { return d_h <= 64 ? 2 : d_h <= 128 ? 4 : 8; }
inline int bulk_cs_bytes(int ft, int d_c) { return (ft * d_c * 4 + 127) & ~127; }
__host__ __device__ inline int bulk_ring_bytes(int d_h) { return kNST * kRows * d_h * 4; }
inline int bulk_smem_bytes(int ft, int d_c, int d_h) {
    return bulk_cs_bytes(ft, d_c) + bulk_ring_bytes(d_h) + 8 * (1 + kNST);
}

// Latent (pure cast) and RoPE key (normalised on its own) of token n into slot s.
template <typename CT>
__device__ __forceinline__ void store_token(const float* lat, const float* __restrict__ r_new,
                                            const float* __restrict__ grk, int64_t n, int64_t s, int d_c, int d_r,
                                            float eps, int plain, CT* __restrict__ kv, int lane) {
    CT* dst = kv + s * (int64_t)(d_c + d_r);
    for (int k = lane; k < d_c; k += 32) Elem<CT>::store(dst + k, lat[k]);
    const float* rs = r_new + n * d_r;
    float beta = 1.f;
    if (!plain) {
        float ss = 0.f;
        for (int j = lane; j < d_r; j += 32) ss = fmaf(rs[j], rs[j], ss);
        ss = warp_sum(ss);
        beta = 1.f / sqrtf(ss / (float)d_r + eps);
    }
    for (int j = lane; j < d_r; j += 32) {
        const float gmul = (plain || grk == nullptr) ? 1.f : grk[j];
        Elem<CT>::store(dst + d_c + j, plain ? rs[j] : rs[j] * gmul * beta);
    }
}

template <typename CT, int NJ>
__global__ void __launch_bounds__(kThreads)
append_bulk_kernel(const float* __restrict__ c_new, const float* __restrict__ r_new, const float* __restrict__ wk,
                   const float* __restrict__ grk, const int64_t* __restrict__ slots, int N, int G, int d_c,
                   int d_h, int d_r, float eps, int plain, CT* __restrict__ kv, float* __restrict__ ak,
                   int64_t num_slots, int* status) {
    using namespace tc;
    constexpr int FT = bulk_ft(NJ);
    constexpr int TPT = kThreads / FT;           // threads per token in the final reduction
    static_assert(TPT <= 32 && 32 % TPT == 0, "a token's reducers sit in one warp");
    extern __shared__ __align__(128) uint8_t sm[];
    const int cs_bytes = (FT * d_c * 4 + 127) & ~127;
    float* Cs = reinterpret_cast<float*>(sm);                     // [FT][d_c]
    float* Ws = reinterpret_cast<float*>(sm + cs_bytes);          // kNST x [kRows][d_h]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + cs_bytes + bulk_ring_bytes(d_h));  // [0] tokens, [1 + s]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.y;
    const int n0 = blockIdx.x * FT;
    const int nvalid = min(FT, N - n0);
    const int stage_f = kRows * d_h;
    const uint32_t stage_bytes = (uint32_t)(stage_f * 4);
    const int n_chunks = d_c / kRows;
    const float* wg = wk + (int64_t)g * d_c * d_h;

    if (tid == 0) {
        for (int i = 0; i < 1 + kNST; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bars[0], (uint32_t)(nvalid * d_c * 4));
        for (int t = 0; t < nvalid; ++t)
            bulk_load(Cs + t * d_c, c_new + (int64_t)(n0 + t) * d_c, (uint32_t)(d_c * 4), &bars[0]);
        for (int c = 0; c < kNST && c < n_chunks; ++c) {
            mbar_arrive_expect_tx(&bars[1 + c], stage_bytes);
            bulk_load(Ws + c * stage_f, wg + (int64_t)c * stage_f, stage_bytes, &bars[1 + c]);
        }
    }
    // the statistic is taken over the STORED latent: round the tile to the cache type in place
    bool ok = mbar_wait(&bars[0], 0, 1u << 24);
    if (ok) {
        for (int e = tid; e < FT * d_c; e += kThreads) Cs[e] = (e < nvalid * d_c) ? Elem<CT>::cast(Cs[e]) : 0.f;
    }
    if (__syncthreads_or(!ok)) {
        if (tid == 0) report(status, QKMLA_ERR_TIMEOUT);
        return;
    }

    float acc[FT][NJ];
#pragma unroll
    for (int t = 0; t < FT; ++t)
#pragma unroll
        for (int j = 0; j < NJ; ++j) acc[t][j] = 0.f;
    for (int c = 0; c < n_chunks; ++c) {
        const int s = c % kNST;
        ok = mbar_wait(&bars[1 + s], (uint32_t)((c / kNST) & 1), 1u << 24);
        if (ok) {
            const float* wr = Ws + s * stage_f + 4 * warp * d_h;
            float bw[4][NJ];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int col = lane + 32 * j;
                    bw[kk][j] = col < d_h ? wr[kk * d_h + col] : 0.f;
                }
            const float* ap = Cs + c * kRows + 4 * warp;
#pragma unroll
            for (int t = 0; t < FT; ++t) {
                const float4 a = *reinterpret_cast<const float4*>(ap + t * d_c);
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    acc[t][j] = fmaf(a.x, bw[0][j], acc[t][j]);
                    acc[t][j] = fmaf(a.y, bw[1][j], acc[t][j]);
                    acc[t][j] = fmaf(a.z, bw[2][j], acc[t][j]);
                    acc[t][j] = fmaf(a.w, bw[3][j], acc[t][j]);
                }
            }
        }
        // every thread is done with stage s before it is refilled
        if (__syncthreads_or(!ok)) {
            if (tid == 0) report(status, QKMLA_ERR_TIMEOUT);
            return;
        }
        if (tid == 0 && c + kNST < n_chunks) {
            mbar_arrive_expect_tx(&bars[1 + s], stage_bytes);
            bulk_load(Ws + s * stage_f, wg + (int64_t)(c + kNST) * stage_f, stage_bytes, &bars[1 + s]);
        }
    }

    // every stage has been consumed and no copy is in flight: the ring holds the
    // partial keys red[warp][t][col] (8 FT d_h floats <= the ring)
    float* red = Ws;
#pragma unroll
    for (int t = 0; t < FT; ++t)
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int col = lane + 32 * j;
            if (col < d_h) red[(warp * FT + t) * d_h + col] = acc[t][j];
        }
    __syncthreads();
    // alpha^k_{t,g} = 1 / sqrt(mean_j k_j^2 + eps): TPT threads per token
    {
        const int t = tid / TPT, q = tid % TPT;
        float ss = 0.f;
        for (int col = q; col < d_h; col += TPT) {
            float k = 0.f;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) k += red[(w * FT + t) * d_h + col];
            ss = fmaf(k, k, ss);
        }
#pragma unroll
        for (int o = TPT / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (q == 0 && t < nvalid) {
            const int64_t sl = slots[n0 + t];
            if (sl >= num_slots) {
                report(status, QKMLA_ERR_DEVICE_BOUNDS);
            } else if (sl >= 0) {
                ak[sl * G + g] = plain ? 1.f : 1.f / sqrtf(ss / (float)d_h + eps);
            }
        }
    }
    if (g != 0) return;
    for (int t = warp; t < nvalid; t += kThreads / 32) {
        const int64_t sl = slots[n0 + t];
        if (sl < 0 || sl >= num_slots) continue;
        store_token<CT>(Cs + t * d_c, r_new, grk, n0 + t, sl, d_c, d_r, eps, plain, kv, lane);
    }
}

template <typename CT>
__global__ void __launch_bounds__(kThreads)
append_plain_kernel(const float* __restrict__ c_new, const float* __restrict__ r_new, const float* __restrict__ wk,
              const float* __restrict__ grk, const int64_t* __restrict__ slots, int N, int G, int d_c,
              int d_h, int d_r, float eps, int plain, CT* __restrict__ kv, float* __restrict__ ak,
              int64_t num_slots, int* status) {
    __shared__ float Cs[kTT][kKC + 1];
    extern __shared__ float Ws[];              // [kKC][d_h]
    const int g = blockIdx.y;
    const int n0 = blockIdx.x * kTT;
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;   // ty: 0..7
    const int nj = (d_h + 31) / 32;
    pdl_wait();
    pdl_trigger();

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
        store_token<CT>(c_new + (int64_t)n * d_c, r_new, grk, n, s, d_c, d_r, eps, plain, kv, tx);
    }
}

template <typename CT>
int launch_t(const float* c_new, const float* r_new, const float* wk, const float* grk, const int64_t* slots, int N,
             int G, int d_c, int d_h, int d_r, float eps, bool plain, CT* kv, float* ak, int64_t num_slots,
             cudaStream_t s) {
    const int nj = bulk_nj(d_h), ft = bulk_ft(nj);
    const int smem_bulk = bulk_smem_bytes(ft, d_c, d_h);
    const bool bulk = d_c % kRows == 0 && ((uintptr_t)c_new % 16) == 0 && ((uintptr_t)wk % 16) == 0 &&
                      smem_bulk <= 232448;
    if (bulk) {
        auto k = nj == 2 ? append_bulk_kernel<CT, 2> : nj == 4 ? append_bulk_kernel<CT, 4> : append_bulk_kernel<CT, 8>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bulk) != cudaSuccess)
            return QKMLA_ERR_CUDA;
        dim3 grid((N + ft - 1) / ft, G);
        if (launch_pdl(k, grid, dim3(kThreads), smem_bulk, s, c_new, r_new, wk, grk, slots, N, G, d_c, d_h, d_r, eps,
                       (int)plain, kv, ak, num_slots, device_status_ptr()) != cudaSuccess)
            return QKMLA_ERR_CUDA;
    } else {
        auto k = append_plain_kernel<CT>;
        const size_t smem = (size_t)kKC * d_h * sizeof(float);
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return QKMLA_ERR_CUDA;
        dim3 grid((N + kTT - 1) / kTT, G);
        if (launch_pdl(k, grid, dim3(kThreads), smem, s, c_new, r_new, wk, grk, slots, N, G, d_c, d_h, d_r, eps,
                       (int)plain, kv, ak, num_slots, device_status_ptr()) != cudaSuccess)
            return QKMLA_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? QKMLA_OK : QKMLA_ERR_CUDA;
}

}  // namespace

int launch_append(const float* c_new, const float* r_new, const float* wk, const float* grk,
                  const int64_t* slots, int N, int G, int d_c, int d_h, int d_r, float eps, bool plain,
                  void* kv, int cache_dtype, float* ak, int64_t num_slots, cudaStream_t s) {
    if (N == 0) return QKMLA_OK;
    if (cache_dtype == QKMLA_F32)
        return launch_t<float>(c_new, r_new, wk, grk, slots, N, G, d_c, d_h, d_r, eps, plain, (float*)kv, ak,
                               num_slots, s);
    return launch_t<__nv_bfloat16>(c_new, r_new, wk, grk, slots, N, G, d_c, d_h, d_r, eps, plain,
                                   (__nv_bfloat16*)kv, ak, num_slots, s);
}

}  // namespace qkmla
