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
// squares and never leaves the cluster.
//
// A decode step appends a handful of tokens, so the kernel's time is the
// latency of bringing W^K_g (d_c x d_h fp32) on chip.  The main kernel splits
// the d_c rows of W^K_g -- contiguous in memory -- over a cluster of S CTAs:
// each CTA brings its token slice and its W slice with bulk copies, forms the
// partial keys of its 16 tokens over its 64 rows, and CTA 0 of the cluster adds
// the S partial keys (read from the others' shared memory, in rank order)
// before squaring.  The g = 0 cluster also stores the cast latent (each CTA its
// slice) and the normalised RoPE key.  Shapes or pointers the bulk copies cannot
// take (d_c not a multiple of 64, misaligned bases) go to a plain-load kernel that
// forms every key element with one fmaf chain over ascending k.
//
// With token positions (qkmla_append_rope) the RoPE key arrives unrotated: it is
// rotated first (interleaved pairs, rope.cuh) and then normalised.
#include "common.cuh"
#include "rope.cuh"
#include "tc_ptx.cuh"

namespace qkmla {

namespace {

constexpr int kTT = 32;        // tokens per CTA (plain-load kernel)
constexpr int kKC = 64;        // d_c chunk staged per step (plain-load kernel)
constexpr int kThreads = 256;
constexpr int kMaxJ = 8;       // d_h <= 256

// Cluster-split kernel: cluster (tile, g) of S CTAs owns kFT tokens of group g;
// CTA r holds rows [r KS, r KS + KS) of W^K_g (KS = d_c / S = 64) and the same
// columns of the token tile.
constexpr int kFT = 16;        // tokens per cluster
constexpr int kKS = 64;        // d_c rows per CTA
__host__ __device__ inline int split_smem_bytes(int d_h) {
    return kFT * kKS * 4 + kKS * d_h * 4 + kFT * d_h * 4 + 8 * kFT * 4 + 16;
}

// cluster-wide barrier (every thread of every CTA), DSMEM address of rank r, remote load
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t smem_addr, uint32_t r) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_addr), "r"(r));
    return d;
}
__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Latent (pure cast) and RoPE key (normalised on its own) of token n into slot s.
// (The whole warp calls it: the rotation pairs lanes j and j ^ 1.)
template <typename CT>
__device__ __forceinline__ void store_token(const float* lat, const float* __restrict__ r_new,
                                            const float* __restrict__ grk, int64_t n, int64_t s, int d_c, int d_r,
                                            float eps, int plain, CT* __restrict__ kv, int lane, int pos,
                                            const RopeFreq* freq) {
    CT* dst = kv + s * (int64_t)(d_c + d_r);
    for (int k = lane; k < d_c; k += 32) Elem<CT>::store(dst + k, lat[k]);
    const float* rs = r_new + n * d_r;
    float rv[2];                                  // d_r <= 64: elements lane and lane + 32
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int j = lane + 32 * u;
        rv[u] = j < d_r ? rs[j] : 0.f;
        if (freq) {                               // rotate first, then normalise
            const float w = __shfl_xor_sync(0xffffffffu, rv[u], 1);
            if (j < d_r) {
                float c, sn;
                rope_cos_sin(pos, freq[j >> 1], &c, &sn);
                rv[u] = rope_apply(j, rv[u], w, c, sn);
            }
        }
    }
    float beta = 1.f;
    if (!plain) {
        const float ss = warp_sum(fmaf(rv[0], rv[0], rv[1] * rv[1]));
        beta = 1.f / sqrtf(ss / (float)d_r + eps);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int j = lane + 32 * u;
        if (j >= d_r) continue;
        const float gmul = (plain || grk == nullptr) ? 1.f : grk[j];
        Elem<CT>::store(dst + d_c + j, plain ? rv[u] : rv[u] * gmul * beta);
    }
}

// U = d_h / 16 key columns per thread: thread (t, q) owns token t = tid / 16 and
// columns q + 16 u.
template <typename CT, int S, int U>
__global__ void __cluster_dims__(S, 1, 1) __launch_bounds__(kThreads)
append_split_kernel(const float* __restrict__ c_new, const float* __restrict__ r_new, const float* __restrict__ wk,
                    const float* __restrict__ grk, const int64_t* __restrict__ slots, int N, int G, int d_r,
                    float eps, int plain, CT* __restrict__ kv, void* __restrict__ ak, int ak_f16, int64_t num_slots,
                    const int32_t* __restrict__ positions, float theta, int* status) {
    using namespace tc;
    __shared__ RopeFreq freq[32];
    constexpr int kDc = S * kKS, kDh = 16 * U;
    extern __shared__ __align__(128) uint8_t sm[];
    float* Cs = reinterpret_cast<float*>(sm);                              // [kFT][kKS]
    float* Ws = Cs + kFT * kKS;                                            // [kKS][kDh]
    float* red = Ws + kKS * kDh;                                           // [kFT][kDh] partial keys
    float* ssp = red + kFT * kDh;                                          // [S][kFT] (CTA 0) sums of squares
    uint64_t* bar = reinterpret_cast<uint64_t*>(ssp + 8 * kFT);
    const int tid = threadIdx.x;
    const int rank = (int)(blockIdx.x % S);
    const int g = blockIdx.y;
    const int n0 = (int)(blockIdx.x / S) * kFT;
    const int nvalid = min(kFT, N - n0);
    const int k0 = rank * kKS;                                             // first d_c row of this CTA

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (positions && tid < d_r / 2) freq[tid] = rope_freq(theta, tid, d_r);
    __syncthreads();
    pdl_trigger();
    // Every input (the weights, the new tokens, their slots and positions) is one no
    // kernel of this library writes, so the loads and the partial keys run before the
    // dependency wait, overlapping the previous kernel; only the cache writes wait.
    if (tid == 0) {
        mbar_arrive_expect_tx(bar, (uint32_t)((nvalid * kKS + kKS * kDh) * 4));
        bulk_load(Ws, wk + ((int64_t)g * kDc + k0) * kDh, (uint32_t)(kKS * kDh * 4), bar);
        for (int t = 0; t < nvalid; ++t)
            bulk_load(Cs + t * kKS, c_new + (int64_t)(n0 + t) * kDc + k0, (uint32_t)(kKS * 4), bar);
    }
    // The tail's mapping: thread (t, q) owns token t = tid / 16 and columns / elements
    // q + 16 v.  What the tail needs from global memory is loaded now, while the bulk
    // copies are in flight.
    const int t = tid >> 4, q = tid & 15;
    const bool tok = t < nvalid;
    const int64_t slot = tok ? slots[n0 + t] : -1;
    const bool rope_here = g == 0 && rank == 0 && tok;
    float rv[4], gv[4];                                                    // d_r <= 64
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int j = q + 16 * v;
        rv[v] = (rope_here && j < d_r) ? r_new[(int64_t)(n0 + t) * d_r + j] : 0.f;
        gv[v] = (rope_here && j < d_r && !plain && grk != nullptr) ? grk[j] : 1.f;
    }
    // The statistic is taken over the STORED latent: the slice is rounded to the cache
    // type and transposed to CsT[k][t] (in the partial-key buffer, unused until the
    // reduction), so that one 16-byte load gives four tokens of row k.
    float* CsT = red;
    static_assert(kKS * kFT <= kFT * kDh, "the transposed slice fits the partial-key buffer");
    const bool ok = mbar_wait(bar, 0, 1u << 24);
    if (ok) {
        for (int e = tid; e < kFT * kKS; e += kThreads) {
            const int tt = e / kKS, k = e % kKS;
            CsT[k * kFT + tt] = (tt < nvalid) ? Elem<CT>::cast(Cs[e]) : 0.f;
        }
    } else {
        report(status, QKMLA_ERR_TIMEOUT);
        mbar_wait(bar, 0, 1u << 24);       // copies still in flight land before the CTA's memory is released
    }
    const bool all_ok = __syncthreads_and(ok) != 0;
    // Partial keys: thread (part, c) owns key column c for all kFT tokens over rows
    // [part kRP, part kRP + kRP) of this CTA's slice (a warp reads 32 consecutive W
    // columns and broadcasts the token values), one fmaf chain per part over
    // ascending k; the parts are then added in order.
    constexpr int kParts = kThreads / kDh, kRP = kKS / kParts;
    static_assert(kThreads % kDh == 0 && kKS % kParts == 0, "thread split of the slice");
    const int c = tid % kDh, part = tid / kDh;
    float acc[kFT];
#pragma unroll
    for (int i = 0; i < kFT; ++i) acc[i] = 0.f;
    if (all_ok) {
#pragma unroll 4
        for (int k = part * kRP; k < part * kRP + kRP; ++k) {
            const float wv = Ws[k * kDh + c];
            const float4* cp = reinterpret_cast<const float4*>(CsT + k * kFT);
#pragma unroll
            for (int i4 = 0; i4 < kFT / 4; ++i4) {
                const float4 cv = cp[i4];
                acc[4 * i4 + 0] = fmaf(cv.x, wv, acc[4 * i4 + 0]);
                acc[4 * i4 + 1] = fmaf(cv.y, wv, acc[4 * i4 + 1]);
                acc[4 * i4 + 2] = fmaf(cv.z, wv, acc[4 * i4 + 2]);
                acc[4 * i4 + 3] = fmaf(cv.w, wv, acc[4 * i4 + 3]);
            }
        }
    }
    pdl_wait();                            // the cache writes follow the previous kernel
    const bool slot_ok = tok && slot >= 0 && slot < num_slots;
    // g = 0: this CTA's slice of the token's latent (a pure cast)
    if (g == 0 && all_ok && slot_ok) {
        CT* dst = kv + slot * (int64_t)(kDc + d_r) + k0;
#pragma unroll
        for (int v = 0; v < kKS / 16; ++v) Elem<CT>::store(dst + q + 16 * v, CsT[(q + 16 * v) * kFT + t]);
    }
    __syncthreads();                       // Ws and CsT are read: parts 1.. park their sums in Ws
    float* parked = Ws;                    // [kParts - 1][kFT][kDh]
    static_assert((kParts - 1) * kFT <= kKS, "the parked sums fit the W slice");
    if (part > 0) {
#pragma unroll
        for (int i = 0; i < kFT; ++i) parked[((part - 1) * kFT + i) * kDh + c] = acc[i];
    }
    __syncthreads();
    if (part == 0) {
#pragma unroll
        for (int i = 0; i < kFT; ++i) {
            float k = acc[i];
            for (int pp = 1; pp < kParts; ++pp) k += parked[((pp - 1) * kFT + i) * kDh + c];
            red[i * kDh + c] = k;
        }
    }
    cluster_sync_all();                    // every CTA's partial keys are in its shared memory
    {
        // The reduction is spread over the cluster: CTA r owns key columns
        // [r kCpr, r kCpr + kCpr).  Each key element is the sum over the CTAs in rank
        // order; this CTA's squares are added per token (thread (t, q): columns
        // q + 16 i) and the token's sum of squares goes to CTA 0.
        constexpr int kCpr = kDh / S;
        float sq = 0.f;
#pragma unroll
        for (int i = 0; i < (kCpr + 15) / 16; ++i) {
            const int cc = q + 16 * i;
            if (cc < kCpr) {
                const uint32_t off = smem_u32(red + t * kDh + rank * kCpr + cc);
                float k = 0.f;
#pragma unroll
                for (int r = 0; r < S; ++r) k += ld_shared_cluster_f32(map_shared_rank(off, (uint32_t)r));
                sq = fmaf(k, k, sq);
            }
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if (q == 0) st_shared_cluster_f32(map_shared_rank(smem_u32(ssp + rank * kFT + t), 0u), sq);
    }
    cluster_sync_all();                    // CTA 0 holds every CTA's sums; no CTA reads another's memory after this
    if (rank == 0) {
        float ss = 0.f;
#pragma unroll
        for (int r = 0; r < S; ++r) ss += ssp[r * kFT + t];
        if (q == 0 && tok && all_ok) {
            if (slot >= num_slots) {
                report(status, QKMLA_ERR_DEVICE_BOUNDS);
            } else if (slot >= 0) {
                store_alpha(ak, slot * G + g, plain ? 1.f : 1.f / sqrtf(ss / (float)kDh + eps), ak_f16 != 0);
            }
        }
        // the RoPE key, normalised on its own: the token's 16 threads hold its d_r values
        if (g == 0) {
            if (positions) {                   // rotate first (pairs j, j ^ 1 in lanes q, q ^ 1)
                const int pos = tok ? positions[n0 + t] : 0;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int j = q + 16 * v;
                    const float w = __shfl_xor_sync(0xffffffffu, rv[v], 1);
                    if (j < d_r) {
                        float c, sn;
                        rope_cos_sin(pos, freq[j >> 1], &c, &sn);
                        rv[v] = rope_apply(j, rv[v], w, c, sn);
                    }
                }
            }
            float sr = 0.f;
#pragma unroll
            for (int v = 0; v < 4; ++v) sr = fmaf(rv[v], rv[v], sr);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) sr += __shfl_xor_sync(0xffffffffu, sr, o);
            const float beta = plain ? 1.f : 1.f / sqrtf(sr / (float)d_r + eps);
            if (all_ok && slot_ok) {
                CT* dst = kv + slot * (int64_t)(kDc + d_r) + kDc;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int j = q + 16 * v;
                    if (j < d_r) Elem<CT>::store(dst + j, plain ? rv[v] : rv[v] * gv[v] * beta);
                }
            }
        }
    }
}

template <typename CT>
__global__ void __launch_bounds__(kThreads)
append_plain_kernel(const float* __restrict__ c_new, const float* __restrict__ r_new, const float* __restrict__ wk,
              const float* __restrict__ grk, const int64_t* __restrict__ slots, int N, int G, int d_c,
              int d_h, int d_r, float eps, int plain, CT* __restrict__ kv, void* __restrict__ ak, int ak_f16,
              int64_t num_slots, const int32_t* __restrict__ positions, float theta, int* status) {
    __shared__ float Cs[kTT][kKC + 1];
    __shared__ RopeFreq freq[32];
    extern __shared__ float Ws[];              // [kKC][d_h]
    const int g = blockIdx.y;
    const int n0 = blockIdx.x * kTT;
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;   // ty: 0..7
    const int nj = (d_h + 31) / 32;
    if (positions && tid < d_r / 2) freq[tid] = rope_freq(theta, tid, d_r);
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
                store_alpha(ak, s * G + g, plain ? 1.f : 1.f / sqrtf(ss / (float)d_h + eps), ak_f16 != 0);
            }
        }
    }

    if (g != 0) return;
    __syncthreads();                              // freq (rotation) is written
    // latent (pure cast) and RoPE key (normalised separately), one warp per token
    for (int tl = ty; tl < kTT; tl += kThreads / 32) {
        const int n = n0 + tl;
        if (n >= N) break;
        const int64_t s = slots[n];
        if (s < 0 || s >= num_slots) continue;
        store_token<CT>(c_new + (int64_t)n * d_c, r_new, grk, n, s, d_c, d_r, eps, plain, kv, tx,
                        positions ? positions[n] : 0, positions ? freq : nullptr);
    }
}

template <typename CT, int S>
cudaError_t launch_split(int U, const float* c_new, const float* r_new, const float* wk, const float* grk,
                         const int64_t* slots, int N, int G, int d_r, float eps, bool plain, CT* kv, void* ak,
                         bool ak_f16, int64_t num_slots, const int32_t* pos, float theta, cudaStream_t s) {
    auto k = U == 4 ? append_split_kernel<CT, S, 4> : append_split_kernel<CT, S, 8>;
    const int smem = split_smem_bytes(16 * U);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(((N + kFT - 1) / kFT) * S, G);
    return launch_pdl(k, grid, dim3(kThreads), smem, s, c_new, r_new, wk, grk, slots, N, G, d_r, eps, (int)plain, kv,
                      ak, (int)ak_f16, num_slots, pos, theta, device_status_ptr());
}

template <typename CT>
int launch_t(const float* c_new, const float* r_new, const float* wk, const float* grk, const int64_t* slots, int N,
             int G, int d_c, int d_h, int d_r, float eps, bool plain, CT* kv, void* ak, bool ak_f16,
             int64_t num_slots, const int32_t* pos, float theta, cudaStream_t s) {
    const int S = d_c / kKS;
    const bool split = d_c % kKS == 0 && (S == 2 || S == 4 || S == 8) && (d_h == 64 || d_h == 128) && d_r <= 64 &&
                       ((uintptr_t)c_new % 16) == 0 && ((uintptr_t)wk % 16) == 0;
    if (split) {
        const int U = d_h / 16;
        const cudaError_t e =
            S == 2   ? launch_split<CT, 2>(U, c_new, r_new, wk, grk, slots, N, G, d_r, eps, plain, kv, ak, ak_f16, num_slots, pos, theta, s)
            : S == 4 ? launch_split<CT, 4>(U, c_new, r_new, wk, grk, slots, N, G, d_r, eps, plain, kv, ak, ak_f16, num_slots, pos, theta, s)
                     : launch_split<CT, 8>(U, c_new, r_new, wk, grk, slots, N, G, d_r, eps, plain, kv, ak, ak_f16, num_slots, pos, theta, s);
        if (e != cudaSuccess) return QKMLA_ERR_CUDA;
    } else {
        auto k = append_plain_kernel<CT>;
        const size_t smem = (size_t)kKC * d_h * sizeof(float);
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return QKMLA_ERR_CUDA;
        dim3 grid((N + kTT - 1) / kTT, G);
        if (launch_pdl(k, grid, dim3(kThreads), smem, s, c_new, r_new, wk, grk, slots, N, G, d_c, d_h, d_r, eps,
                       (int)plain, kv, ak, (int)ak_f16, num_slots, pos, theta, device_status_ptr()) != cudaSuccess)
            return QKMLA_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? QKMLA_OK : QKMLA_ERR_CUDA;
}

}  // namespace

int launch_append(const float* c_new, const float* r_new, const float* wk, const float* grk,
                  const int64_t* slots, int N, int G, int d_c, int d_h, int d_r, float eps, bool plain,
                  void* kv, int cache_dtype, void* ak, bool ak_f16, int64_t num_slots, const int32_t* positions,
                  float rope_theta, cudaStream_t s) {
    if (N == 0) return QKMLA_OK;
    if (cache_dtype == QKMLA_F32)
        return launch_t<float>(c_new, r_new, wk, grk, slots, N, G, d_c, d_h, d_r, eps, plain, (float*)kv, ak,
                               ak_f16, num_slots, positions, rope_theta, s);
    return launch_t<__nv_bfloat16>(c_new, r_new, wk, grk, slots, N, G, d_c, d_h, d_r, eps, plain,
                                   (__nv_bfloat16*)kv, ak, ak_f16, num_slots, positions, rope_theta, s);
}

}  // namespace qkmla
