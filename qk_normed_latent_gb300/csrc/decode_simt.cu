// CUDA-core decode kernel (any cache dtype; the only path for an fp32 cache).
//
// Source: "QK-Normed MLA: QK normalization without full key caching", Technical
// Summary, Methodology -- decode-logit equation l = (q~ . c_t) alpha^q alpha^k_{t,g(h)}
// with the scalars applied as a row/column scaling before the softmax, and
// "Blockwise Normalization" (the RoPE logit uses materialised, separately
// normalised vectors); abstract: the latent decode path is kept, so the values
// are the latents themselves.
//
// One CTA serves one (sequence b, query token i, KV group g, split) and all
// H/G heads of the group, so every cached row is read once per group.  Tokens
// are staged 32 at a time in shared memory (fp32); logits, an online softmax
// (running max / sum in the exp2 domain) and the latent accumulation follow.
// fp32 arithmetic throughout.
#include "common.cuh"

namespace qkmla {

namespace {

constexpr int kTC = 32;          // tokens per chunk (one per lane in the softmax step)
constexpr int kThreads = 256;

struct SimtParams {
    const void* qt;
    const float* aq;
    const float* qr;
    const float* grq;
    const void* kv;
    const void* ak;     // fp32, or fp16 when ak_f16
    const int32_t* seq_lens;
    const int32_t* page_table;
    int64_t num_pages;
    int page_size, max_pages;
    int B, s_q, H, G, d_c, d_r;
    float scale, eps;
    int plain;
    int ak_f16;
    int nsplit;
    float* o_part;      // [rows*H][nsplit][d_c] when nsplit > 1
    float* lse_part;    // [rows*H][nsplit]
    void* o;
    int o_dtype;
    float* lse;
    int* status;
};

template <typename CT, int HPG, int NJ>
__global__ void __launch_bounds__(kThreads)
decode_simt_kernel(SimtParams p) {
    extern __shared__ float sm[];
    const int row = p.d_c + p.d_r;
    const int ldk = row + 1;
    float* qs = sm;                         // [HPG][row]   q~ (fp32) | normalised q_rope
    float* kvs = qs + HPG * row;            // [kTC][ldk]   staged cache rows
    float* ps = kvs + kTC * ldk;            // [HPG][kTC]   logits, then probabilities
    float* aks = ps + HPG * kTC;            // [kTC]        alpha^k of group g
    float* coef = aks + kTC;                // [HPG]        scale*alpha^q*log2e
    float* mrun = coef + HPG;               // [HPG]        running max (log2 domain)
    float* lrun = mrun + HPG;               // [HPG]        running sum
    float* corr = lrun + HPG;               // [HPG]        rescale factor of this chunk
    const int nfl = (int)(corr + HPG - sm);
    int64_t* slot = (int64_t*)(sm + ((nfl + 1) & ~1));   // [kTC], 8-byte aligned

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = blockIdx.x % p.G;
    const int bi = blockIdx.x / p.G;        // b * s_q + i
    const int b = bi / p.s_q, i = bi % p.s_q;
    const int sp = blockIdx.y;
    const int h0 = g * HPG;
    const CT* qt = (const CT*)p.qt;
    const CT* kv = (const CT*)p.kv;
    const float l2e = kLog2e;

    pdl_wait();
    pdl_trigger();
    const int seq_len = p.seq_lens[b];
    const bool bad_len = seq_len < p.s_q || seq_len > p.max_pages * p.page_size;
    if (bad_len && tid == 0) report(p.status, QKMLA_ERR_DEVICE_BOUNDS);
    const int L = bad_len ? 0 : seq_len - p.s_q + i + 1;
    int chunk = (L + p.nsplit - 1) / p.nsplit;
    chunk = (chunk + kTC - 1) / kTC * kTC;
    const int t0 = sp * chunk, t1 = min(L, t0 + chunk);

    // stage the query rows: q~ in fp32, the RoPE query normalised per head
    for (int e = tid; e < HPG * p.d_c; e += kThreads) {
        const int hl = e / p.d_c, k = e % p.d_c;
        qs[hl * row + k] = Elem<CT>::load(qt + (((int64_t)bi * p.H) + h0 + hl) * p.d_c + k);
    }
    for (int hl = warp; hl < HPG; hl += kThreads / 32) {
        const float* src = p.qr + (((int64_t)bi * p.H) + h0 + hl) * p.d_r;
        float ss = 0.f;
        for (int j = lane; j < p.d_r; j += 32) ss = fmaf(src[j], src[j], ss);
        ss = warp_sum(ss);
        const float beta = p.plain ? 1.f : 1.f / sqrtf(ss / (float)p.d_r + p.eps);
        for (int j = lane; j < p.d_r; j += 32) {
            const float gm = (p.plain || p.grq == nullptr) ? 1.f : p.grq[j];
            qs[hl * row + p.d_c + j] = src[j] * gm * beta;
        }
        if (lane == 0) {
            const float a = p.plain ? 1.f : p.aq[(int64_t)bi * p.H + h0 + hl];
            coef[hl] = p.scale * a * l2e;
            mrun[hl] = -INFINITY;
            lrun[hl] = 0.f;
        }
    }

    float acc[HPG][NJ];
#pragma unroll
    for (int hl = 0; hl < HPG; ++hl)
#pragma unroll
        for (int j = 0; j < NJ; ++j) acc[hl][j] = 0.f;

    const float rs = p.scale * l2e;
    for (int tb = t0; tb < t1; tb += kTC) {
        __syncthreads();
        if (tid < kTC) {
            const int t = tb + tid;
            slot[tid] = (t < t1) ? slot_of(p.page_table, b, t, p.page_size, p.max_pages, p.num_pages, p.status) : -1;
        }
        __syncthreads();
        for (int e = tid; e < kTC * row; e += kThreads) {
            const int tl = e / row, k = e % row;
            const int64_t s = slot[tl];
            kvs[tl * ldk + k] = (s >= 0) ? Elem<CT>::load(kv + s * row + k) : 0.f;
        }
        if (tid < kTC) {
            const int64_t s = slot[tid];
            aks[tid] = (s >= 0) ? (p.plain ? 1.f
                                           : p.ak_f16 ? load_alpha<true>(p.ak, s * p.G + g) : load_alpha<false>(p.ak, s * p.G + g))
                                : 0.f;
        }
        __syncthreads();
        // logits (log2 domain)
        for (int e = tid; e < HPG * kTC; e += kThreads) {
            const int hl = e / kTC, tl = e % kTC;
            const float* qv = qs + hl * row;
            const float* kr = kvs + tl * ldk;
            float c = 0.f, r = 0.f;
            for (int k = 0; k < p.d_c; ++k) c = fmaf(qv[k], kr[k], c);
            for (int j = p.d_c; j < row; ++j) r = fmaf(qv[j], kr[j], r);
            float lg = p.plain ? rs * (c + r) : fmaf(coef[hl] * aks[tl], c, rs * r);
            if (slot[tl] < 0) lg = -INFINITY;
            ps[hl * kTC + tl] = lg;
        }
        __syncthreads();
        // online softmax: warp per head, lane per token
        for (int hl = warp; hl < HPG; hl += kThreads / 32) {
            const float lg = ps[hl * kTC + lane];
            const float mt = warp_max(lg);
            const float mo = mrun[hl];
            const float mn = fmaxf(mo, mt);
            const float pe = (lg == -INFINITY) ? 0.f : exp2f(lg - mn);
            const float st = warp_sum(pe);
            ps[hl * kTC + lane] = pe;
            __syncwarp();
            if (lane == 0) {
                const float c = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
                corr[hl] = c;
                lrun[hl] = lrun[hl] * c + st;
                mrun[hl] = mn;
            }
        }
        __syncthreads();
        // latent accumulation: thread owns latent columns tid + 256 j
#pragma unroll
        for (int hl = 0; hl < HPG; ++hl) {
            const float c = corr[hl];
#pragma unroll
            for (int j = 0; j < NJ; ++j) acc[hl][j] *= c;
        }
        for (int tl = 0; tl < kTC; ++tl) {
            float v[NJ];
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int k = tid + kThreads * j;
                v[j] = (k < p.d_c) ? kvs[tl * ldk + k] : 0.f;
            }
#pragma unroll
            for (int hl = 0; hl < HPG; ++hl) {
                const float pw = ps[hl * kTC + tl];
#pragma unroll
                for (int j = 0; j < NJ; ++j) acc[hl][j] = fmaf(pw, v[j], acc[hl][j]);
            }
        }
    }
    __syncthreads();

    // write the final row (one split) or this split's partial (o normalised, lse)
#pragma unroll
    for (int hl = 0; hl < HPG; ++hl) {
        const int64_t rh = (int64_t)bi * p.H + h0 + hl;
        const float l = lrun[hl];
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        const float lse = (l > 0.f) ? (mrun[hl] + log2f(l)) * kLn2 : -INFINITY;
        if (p.nsplit == 1) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int k = tid + kThreads * j;
                if (k >= p.d_c) continue;
                if (p.o_dtype == QKMLA_F32)
                    ((float*)p.o)[rh * p.d_c + k] = acc[hl][j] * inv;
                else
                    ((__nv_bfloat16*)p.o)[rh * p.d_c + k] = __float2bfloat16_rn(acc[hl][j] * inv);
            }
            if (tid == 0 && p.lse) p.lse[rh] = lse;
        } else {
            float* dst = p.o_part + (rh * p.nsplit + sp) * p.d_c;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int k = tid + kThreads * j;
                if (k < p.d_c) dst[k] = acc[hl][j] * inv;
            }
            if (tid == 0) p.lse_part[rh * p.nsplit + sp] = lse;
        }
    }
}

template <typename CT, int HPG, int NJ>
int launch_t(const SimtParams& p, cudaStream_t s) {
    const int row = p.d_c + p.d_r;
    const size_t nfl = (size_t)HPG * row + (size_t)kTC * (row + 1) + HPG * kTC + kTC + 4 * HPG;
    const size_t smem = sizeof(float) * ((nfl + 1) & ~(size_t)1) + sizeof(int64_t) * kTC;
    auto k = decode_simt_kernel<CT, HPG, NJ>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return QKMLA_ERR_CUDA;
    dim3 grid(p.B * p.s_q * p.G, p.nsplit);
    return launch_pdl(k, grid, dim3(kThreads), smem, s, p) == cudaSuccess ? QKMLA_OK : QKMLA_ERR_CUDA;
}

template <typename CT, int NJ>
int launch_h(const SimtParams& p, int hpg, cudaStream_t s) {
    switch (hpg) {
        case 1: return launch_t<CT, 1, NJ>(p, s);
        case 2: return launch_t<CT, 2, NJ>(p, s);
        case 4: return launch_t<CT, 4, NJ>(p, s);
        case 8: return launch_t<CT, 8, NJ>(p, s);
        case 16: return launch_t<CT, 16, NJ>(p, s);
    }
    return QKMLA_ERR_UNSUPPORTED;
}

template <typename CT>
int launch_c(const SimtParams& p, int hpg, cudaStream_t s) {
    if (p.d_c <= kThreads) return launch_h<CT, 1>(p, hpg, s);
    return launch_h<CT, 2>(p, hpg, s);
}

}  // namespace

int launch_decode_simt(const qkmla_decode_args* a, const DecodePlan& plan, cudaStream_t s) {
    SimtParams p;
    p.qt = a->q_tilde;
    p.aq = a->alpha_q;
    p.qr = a->q_rope;
    p.grq = a->gamma_rope_q;
    p.kv = a->kv_cache;
    p.ak = a->ak_cache;
    p.seq_lens = a->seq_lens;
    p.page_table = a->page_table;
    p.num_pages = a->num_slots / a->page_size;
    p.page_size = a->page_size;
    p.max_pages = a->max_pages;
    p.B = a->B; p.s_q = a->s_q; p.H = a->H; p.G = a->G; p.d_c = a->d_c; p.d_r = a->d_r;
    p.scale = a->softmax_scale;
    p.eps = a->eps;
    p.plain = (a->flags & QKMLA_FLAG_PLAIN_MLA) ? 1 : 0;
    p.ak_f16 = (!p.plain && (a->flags & QKMLA_FLAG_ALPHA_F16)) ? 1 : 0;
    p.nsplit = plan.num_splits;
    const int64_t rows_h = (int64_t)a->B * a->s_q * a->H;
    p.o_part = (float*)a->workspace;
    p.lse_part = p.o_part ? p.o_part + rows_h * plan.num_splits * a->d_c : nullptr;
    p.o = a->o;
    p.o_dtype = a->o_dtype;
    p.lse = a->lse;
    p.status = device_status_ptr();
    const int hpg = a->H / a->G;
    int rc = (a->cache_dtype == QKMLA_F32) ? launch_c<float>(p, hpg, s) : launch_c<__nv_bfloat16>(p, hpg, s);
    if (rc != QKMLA_OK || plan.num_splits == 1) return rc;
    return launch_combine(p.o_part, p.lse_part, (int)rows_h, plan.num_splits, a->d_c, a->o, a->o_dtype,
                          a->lse, s);
}

}  // namespace qkmla
