// Two-CTA cluster decode kernel for the DeepSeek-V3 decode shape
// (d_c = 512, d_r = 64, 128 query heads per query token, bf16 cache).
//
// Source: "QK-Normed MLA: QK normalization without full key caching", Technical
// Summary, Methodology -- decode-logit equation
//     l_{i,t,h} = (q~_{i,h} . c_t) alpha^q_{i,h} alpha^k_{t,g(h)}
// with the scalars applied as a row/column scaling before the softmax, plus the
// separately normalised RoPE logit ("Blockwise Normalization"); values are the
// latents (the abstract's latent decode path).
//
// Why a pair.  A tcgen05.mma costs about the same time for any N <= 128, so
// the logit MMA wants M = 128 query rows; but the fp32 output of 128 rows x 512
// latents fills all of one SM's TMEM.  The pair therefore splits the latent
// dimension: CTA r owns latent columns [256 r, 256 r + 256) and RoPE columns
// [32 r, 32 r + 32).  Per 64-token tile each CTA
//   * computes partial logits over its half of K (M=128 rows, N=64, K=288),
//     and applies the column scaling alpha^k to its content part (the scaling
//     is linear, so partial logits add); the row factor scale log2e alpha^q,
//     common to both parts, is divided out of the RoPE query and applied once
//     to the summed logit, in the exponent argument,
//   * exchanges partials with the other CTA: every softmax warp stages its 32
//     rows -- 64 fp16 values relative to the row's own maximum, plus that
//     maximum in fp32, so the values near the maximum (the ones that matter
//     after exp) keep ~11 bits -- and sends them with one bulk copy into the
//     other CTA's shared memory (completing on a per-warp mbarrier there); each
//     CTA adds the received rows to its own fp32 partials,
//   * writes P (bf16) into TMEM and accumulates O = P C over its 256 latents
//     (M=128 rows, N=256, K=64 tokens, A read from TMEM).
// Each CTA streams only its half of every tile from HBM, through three stages:
// a stage stays busy until its tile's output MMA, so the third one keeps a load
// in flight while the other two are being used.
//
// Warps: 0 TMA producer (+ TMEM owner), 1 MMA issuer, 2-5 softmax / exchange /
// epilogue (thread = query row = TMEM lane).  The MMA issuer polls its two
// inputs (a landed tile, a written P) and issues whichever is ready, so an
// output MMA -- and the stage it frees -- never waits behind the next tile's
// load.  All waits are bounded (2 s).
#include <cudaTypedefs.h>

#include <cuda_fp16.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "decode_sched.cuh"
#include "tc_ptx.cuh"

namespace qkmla {
namespace dec {
namespace {

constexpr int kT = 64;             // tokens per tile
constexpr int kR = 128;            // query rows per pair
constexpr int kDC = 512, kDR = 64;
constexpr int kHalfLat = kDC / 2;  // latent columns per CTA
constexpr int kHalfRope = kDR / 2; // RoPE columns per CTA
constexpr int kThreadsP = 320;    // 2 + 4 + 4 warps
constexpr int kNst = 3;            // TMA stages

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kQLat = 4 * kR * 128;                    // Q~ half: 4 blocks of 128 rows x 128 B
constexpr int kQRope = kR * 64;                        // RoPE half: 128 rows x 64 B (64-byte swizzle)
constexpr int kSLat = 4 * kT * 128;                    // tile half: 4 boxes of 64 tokens x 128 B
constexpr int kSRope = kT * 64;                        // 64 tokens x 64 B
constexpr int kSAk = kT * kMaxG * 4;
constexpr int kStageB = kSLat + kSRope + kSAk;         // 38 KB
// exchange slice of one row group: 32 rows x 64 fp16 partial logits minus the
// row's maximum (128-byte rows, 16-byte chunks XOR-swizzled by row), then the
// 32 maxima (fp32)
constexpr int kXRowB = kT * 2;
constexpr int kXSlice = 32 * kXRowB + 32 * 4;
constexpr int kXB = 4 * kXSlice;
constexpr int kOffQ = 0;
constexpr int kOffStage = kQLat + kQRope;
constexpr int kOffX = kOffStage + kNst * kStageB;      // received partials
constexpr int kOffY = kOffX + kXB;                     // own partials (sent)
constexpr int kOffMisc = kOffY + kXB;
constexpr int kNumBars = 23;
constexpr int kBytesP = kOffMisc + kNumBars * 8 + 16 + kR * 4 + 1024;
static_assert(kStageB % 1024 == 0 && kOffStage % 1024 == 0 && kOffX % 16 == 0 && kOffY % 16 == 0, "align");
static_assert(kXSlice % 16 == 0, "bulk copy size");
static_assert(kBytesP <= 232448, "shared memory budget");

// TMEM columns: S_c at 0, S_r at 64, P[2] (64 bf16 tokens = 32 columns each) at
// 128 / 160, this CTA's scaled partial logits (fp32, parked by group A for group
// B) at 192, O (128 rows x 256 latents) at 256
constexpr uint32_t kCSc = 0, kCSr = 64, kCP = 128, kCOwn = 192, kCO = 256;

// AKH: A^k_cache entries are fp16 (else fp32)
template <bool PLAIN, bool AKH>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsP, 1)
decode_pair_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope,
                   const __grid_constant__ CUtensorMap tm_q, const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    // 1024-byte aligned base, formed from smraw itself so accesses stay in the shared window
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint8_t* sQ = sm + kOffQ;
    uint8_t* sX = sm + kOffX;
    uint8_t* sY = sm + kOffY;
    uint64_t* bars = (uint64_t*)(sm + kOffMisc);
    uint64_t* full = bars;          // [3] TMA -> MMA
    uint64_t* empty = bars + 3;     // [3] output MMA done -> TMA
    uint64_t* sfull = bars + 6;     // logit MMA done -> softmax (one S buffer)
    uint64_t* sfree = bars + 7;     // softmax read S -> MMA
    uint64_t* pdone = bars + 8;     // [2] output MMA done with P buffer -> softmax
    uint64_t* pfull = bars + 10;    // [2] P written -> output MMA
    uint64_t* xfull = bars + 12;    // [4] per warp: the other CTA's partial rows landed in X
    uint64_t* xfree = bars + 16;    // [4] per warp: the other CTA's X rows may be overwritten
    uint64_t* ownfull = bars + 20;  // group A parked a tile's partials -> group B
    uint64_t* ownfree = bars + 21;  // group B read them -> group A
    uint64_t* qfull = bars + 22;    // this CTA's half of Q~ landed
    uint32_t* tmem_slot = (uint32_t*)(bars + kNumBars);
    int* abort_flag = (int*)(tmem_slot + 1);
    float* coef_s = (float*)(sm + kOffMisc + kNumBars * 8 + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    WorkItem it;
    int seq_len;
    // the in-kernel plan reads only seq_lens, which no kernel of the call writes: it
    // is made before the dependency wait, overlapping the previous kernel's tail
    if (p.sched_inline) {                                // both CTAs derive the same plan
        __shared__ SchedSmem S;
        compute_schedule(p.seq_lens, p.B, p.s_q, p.sa, S, p.status, blockIdx.x == 0 && blockIdx.y == 0);
        if ((int)blockIdx.y >= S.n_items) return;        // uniform over the cluster
        it = schedule_item(S, p.B, (int)blockIdx.y);
        seq_len = S.len[it.b];                           // the plan's copy
    } else {
        pdl_wait();                                      // the scheduler kernel's items
        if ((int)blockIdx.y >= *p.n_items) return;       // uniform over the cluster
        it = p.items[blockIdx.y];
        seq_len = p.seq_lens[it.b];
    }
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int qi = blockIdx.x >> 1;                       // query token of this pair
    const int b = it.b;
    const bool bad = seq_len < p.s_q || seq_len > p.max_pages * p.page_size;
    const int L = bad ? 0 : seq_len - p.s_q + qi + 1;
    const int tiles = (L + kT - 1) / kT;
    const int jt0 = it.tile_begin;
    const int n_t = max(0, min(it.tile_end, tiles) - jt0);
    const int hpg = p.H / p.G;

    if (tid == 0) {
        if (bad && rank == 0) report(p.status, QKMLA_ERR_DEVICE_BOUNDS);
        for (int i = 0; i < kNumBars; ++i) {
            const bool four = (i == 7 || i == 10 || i == 11 || i == 20 || i == 21);   // one per warp of a group
            mbar_init(&bars[i], four ? 4u : 1u);
        }
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tm_lat);
        prefetch_tmap(&tm_rope);
        prefetch_tmap(&tm_q);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    pdl_wait();                // q~, alpha^q, the RoPE query and the cache are written by earlier kernels
    pdl_trigger();
    // ---- prologue: this CTA's half of Q~ (TMA, four 64-column boxes) and of the
    //      normalised RoPE query ----
    const size_t qrow0 = ((size_t)b * p.s_q + qi) * p.H;
    if (warp >= 2) {
        const int st = tid - 64;
        if (st < kR) {   // one thread per row: RMS over all 64 RoPE dims, keep this CTA's 32
            const int r = st;
            // every global read of the prologue is issued before the first shared-memory
            // store (a load after a store through generic pointers waits for it)
            const float* src = p.qr + (qrow0 + r) * kDR;
            float v[kDR], gq[kHalfRope];
#pragma unroll
            for (int j = 0; j < kDR; ++j) v[j] = src[j];
#pragma unroll
            for (int j = 0; j < kHalfRope; ++j) gq[j] = (PLAIN || !p.grq) ? 1.f : p.grq[rank * kHalfRope + j];
            const float a = PLAIN ? 0.f : p.aq[qrow0 + r];
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < kDR; ++j) ss = fmaf(v[j], v[j], ss);
            // QK mode: the RoPE query carries 1 / (RMS alpha^q), so its MMA output is the
            // RoPE logit in the exp2 domain divided by this row's content scale
            // coef = scale log2e alpha^q: the softmax groups work in logit / coef units
            // and apply coef once, in the exponent argument
            const float beta = PLAIN ? 1.f : 1.f / (sqrtf(ss / (float)kDR + p.eps) * a);
            uint8_t* qrope = sQ + kQLat;
#pragma unroll
            for (int j = 0; j < kHalfRope; j += 2) {
                const float v0 = rank ? v[kHalfRope + j] : v[j];          // register indices stay static
                const float v1 = rank ? v[kHalfRope + j + 1] : v[j + 1];
                const __nv_bfloat162 w2 = __floats2bfloat162_rn(v0 * gq[j] * beta, v1 * gq[j + 1] * beta);
                *reinterpret_cast<__nv_bfloat162*>(qrope + sw64_offset(r, j)) = w2;
            }
            coef_s[r] = PLAIN ? p.scale * kLog2e : p.scale * a * kLog2e;
        }
        fence_proxy_async_smem();
    }
    // no barrier is touched before this point: thread 0's mbarrier.init must be
    // ordered before every arrive, local or remote
    tc_fence_before();
    cluster_sync();            // both CTAs' barriers exist before any remote access
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0) {
        mbar_arrive_expect_tx(qfull, (uint32_t)(4 * kR * 128));
#pragma unroll
        for (int blk = 0; blk < 4; ++blk)
            tma_load_2d(sQ + blk * (kR * 128), &tm_q, rank * kHalfLat + blk * 64, (int)qrow0, qfull);
    }

    if (warp == 0) {
        // ===================== TMA producer: this CTA's half of each tile =====================
        // lane l holds the slot of tile (j & ~31) + l: 32 page-table reads in parallel
        auto slot_of_tile = [&](int j) -> int {
            if (j >= n_t) return 0;
            const int t0 = (jt0 + j) * kT;
            const int pg = t0 / p.page_size;
            int64_t page = p.page_table ? (int64_t)p.page_table[(int64_t)b * p.max_pages + pg]
                                        : (int64_t)b * p.max_pages + pg;
            if (page < 0 || page >= p.num_pages) {
                report(p.status, QKMLA_ERR_DEVICE_BOUNDS);
                page = 0;
            }
            return (int)(page * p.page_size + (t0 % p.page_size));
        };
        const uint32_t ak_bytes = PLAIN ? 0u : (uint32_t)(kT * p.G * (AKH ? 2 : 4));
        const uint32_t tx = (uint32_t)(kSLat + kSRope) + ak_bytes;
        int slot_batch = slot_of_tile(lane);
        for (int j = 0; j < n_t; ++j) {
            if ((j & 31) == 0 && j > 0) slot_batch = slot_of_tile(j + lane);
            const int slot0 = __shfl_sync(0xffffffffu, slot_batch, j & 31);
            int go = 1;
            if (lane == 0) {
                const int s = j % kNst;
                if (j >= kNst && !wait_bounded(&empty[s], ((j / kNst) - 1) & 1, p.status)) {
                    *abort_flag = 1;
                    go = 0;
                } else if (*(volatile int*)abort_flag) {
                    go = 0;
                } else {
                    uint8_t* stg = sm + kOffStage + s * kStageB;
                    mbar_arrive_expect_tx(&full[s], tx);
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk)
                        tma_load_2d(stg + blk * (kT * 128), &tm_lat, rank * kHalfLat + blk * 64, slot0, &full[s]);
                    tma_load_2d(stg + kSLat, &tm_rope, kDC + rank * kHalfRope, slot0, &full[s]);
                    if (!PLAIN)
                        bulk_load(stg + kSLat + kSRope, (const uint8_t*)p.ak + (int64_t)slot0 * p.G * (AKH ? 2 : 4),
                                  ak_bytes, &full[s]);
                }
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
        }
    } else if (warp == 1) {
        // ===================== MMA issuer: S(j) and O(j) in readiness order =====================
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(kR, kT, 0, 0);
            const uint32_t id_o = idesc_bf16(kR, kHalfLat, 0, 1);
            const uint32_t q_addr = smem_u32(sQ);
            auto issue_s = [&](int j) {
                const int s = j % kNst;
                tc_fence_after();
                const uint32_t st_addr = smem_u32(sm + kOffStage + s * kStageB);
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = smem_desc(q_addr + blk * (kR * 128) + kk * 32, 16, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(st_addr + blk * (kT * 128) + kk * 32, 16, 1024, kSwizzle128B);
                        mma_bf16(tmem + kCSc, a, bd, id_s, (blk > 0 || kk > 0) ? 1u : 0u);
                    }
                }
#pragma unroll
                for (int kk = 0; kk < kHalfRope / 16; ++kk) {
                    const uint64_t a = smem_desc(q_addr + kQLat + kk * 32, 16, 512, kSwizzle64B);
                    const uint64_t bd = smem_desc(st_addr + kSLat + kk * 32, 16, 512, kSwizzle64B);
                    if (PLAIN)
                        mma_bf16(tmem + kCSc, a, bd, id_s, 1u);
                    else
                        mma_bf16(tmem + kCSr, a, bd, id_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(sfull);
            };
            auto issue_o = [&](int j) {
                const int s = j % kNst, pb = j & 1;
                tc_fence_after();
                const uint32_t st_addr = smem_u32(sm + kOffStage + s * kStageB);
#pragma unroll
                for (int kk = 0; kk < kT / 16; ++kk) {
                    // A = P from TMEM (16 tokens = 8 packed columns per step); B = C^T: this
                    // CTA's 256 latents (4 boxes, LBO = box stride) x 16 tokens (SBO = 8 tokens)
                    const uint64_t bd = smem_desc(st_addr + kk * 2048, kT * 128, 1024, kSwizzle128B);
                    mma_bf16_tmem_a(tmem + kCO, tmem + kCP + pb * (kT / 2) + kk * 8, bd, id_o,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
                mma_commit(&pdone[pb]);
            };
            // every barrier below completes once per tile and is tested for its tiles in
            // order, so each parity names exactly one phase.  Q~ is always waited for,
            // so no CTA exits with its copy in flight.
            int js = 0, jo = 0;
            bool ok = wait_bounded(qfull, 0, p.status);
            uint64_t t_last = globaltimer();
            uint32_t idle = 0;
            while (ok && jo < n_t) {
                bool did = false;
                // the logit MMA of tile js: the tile has landed and the softmax has read S(js-1)
                if (js < n_t && mbar_test_wait(&full[js % kNst], (js / kNst) & 1) &&
                    (js == 0 || mbar_test_wait(sfree, (js - 1) & 1))) {
                    issue_s(js);
                    ++js;
                    did = true;
                }
                // the output MMA of tile jo: its P is written
                if (jo < js && mbar_test_wait(&pfull[jo & 1], (jo >> 1) & 1)) {
                    issue_o(jo);
                    ++jo;
                    did = true;
                }
                if (did) {
                    idle = 0;
                    t_last = globaltimer();
                } else if ((++idle & 255u) == 0) {
                    if (*(volatile int*)abort_flag || globaltimer() - t_last > kWaitNs) {
                        report(p.status, QKMLA_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) *(volatile int*)abort_flag = 1;
        }
    } else {
        // ===================== softmax: two groups of four warps, thread = query row =====================
        // Group A (warps 2-5) turns S(j) into this CTA's scaled partial logits, parks
        // them in TMEM (scratch columns) and sends them (fp16) to the other CTA; group
        // B (warps 6-9) adds the other CTA's partials, runs the online softmax and
        // writes P.  A works on tile j+1 while B finishes tile j.
        const int sub = warp & 3;                        // TMEM sub-partition = exchange slice
        const bool grp_a = warp < 6;
        const uint32_t lane_base = (uint32_t)(32 * sub) << 16;
        const int r = 32 * sub + lane;                   // M=128 accumulator: row r in TMEM lane r
        const uint32_t my_slice = (uint32_t)sub * kXSlice;
        const uint32_t xrow = my_slice + lane * kXRowB;  // this row's 128 fp16 bytes in a slice
        float* const x_off = reinterpret_cast<float*>(sX + my_slice + 32 * kXRowB);   // 32 maxima
        float* const y_off = reinterpret_cast<float*>(sY + my_slice + 32 * kXRowB);
        if (grp_a) {
            const int g = (r % p.H) / hpg;
            const uint32_t peer_x = map_to_rank(smem_u32(sX) + my_slice, peer);
            const uint32_t peer_xfull = map_to_rank(smem_u32(&xfull[sub]), peer);
            float pv[kT];
            for (int j = 0; j < n_t; ++j) {
                const int s = j % kNst;
                const int valid = min(kT, L - (jt0 + j) * kT);
                const bool got_s = __all_sync(0xffffffffu, wait_bounded(sfull, j & 1, p.status));
                tc_fence_after();
                const void* ak_t = sm + kOffStage + s * kStageB + kSLat + kSRope;
                {
                    // both loads first (a whole row each), one wait: a single TMEM round trip per tile
                    uint32_t sc[kT], sr[kT];
                    tmem_ld64(tmem + kCSc + lane_base, sc);
                    if (!PLAIN) tmem_ld64(tmem + kCSr + lane_base, sr);
                    tmem_wait_ld();
                    // S is in registers: release it to the next logit MMA before scaling
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sfree);
                    if (PLAIN) {
#pragma unroll
                        for (int t = 0; t < kT; ++t) pv[t] = __uint_as_float(sc[t]);
                    } else {
                        // alpha^k_t S_c + S_r (logit / coef), two tokens per packed instruction
#pragma unroll
                        for (int t = 0; t < kT; t += 2) {
                            const uint64_t ak2 = f2(load_alpha<AKH>(ak_t, t * p.G + g), load_alpha<AKH>(ak_t, (t + 1) * p.G + g));
                            const float2 r2 = f2_unpack(f2_fma(ak2, f2(__uint_as_float(sc[t]), __uint_as_float(sc[t + 1])),
                                                               f2(__uint_as_float(sr[t]), __uint_as_float(sr[t + 1]))));
                            pv[t] = r2.x;
                            pv[t + 1] = r2.y;
                        }
                    }
                }
                if (valid < kT) {
#pragma unroll
                    for (int t = 0; t < kT; ++t)
                        if (t >= valid) pv[t] = -INFINITY;
                }
                // park the fp32 partials for group B once it has read the previous ones
                bool ok_a = got_s;
                if (j >= 1) ok_a = __all_sync(0xffffffffu, wait_bounded(ownfree, (j - 1) & 1, p.status)) && ok_a;
                tc_fence_after();
                {
                    uint32_t w64[kT];
#pragma unroll
                    for (int t = 0; t < kT; ++t) w64[t] = __float_as_uint(pv[t]);
                    tmem_st64(tmem + kCOwn + lane_base, w64);
                }
                tmem_wait_st();
                // stage fp16 relative to the row max, once the previous send has read Y
                float mo[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) mo[q] = fmaxf(fmaxf(pv[q], pv[q + 8]), fmaxf(pv[q + 16], pv[q + 24]));
#pragma unroll
                for (int q = 0; q < 8; ++q) mo[q] = fmaxf(mo[q], fmaxf(fmaxf(pv[q + 32], pv[q + 40]), fmaxf(pv[q + 48], pv[q + 56])));
                const float m_own = fmaxf(fmaxf(fmaxf(mo[0], mo[1]), fmaxf(mo[2], mo[3])),
                                          fmaxf(fmaxf(mo[4], mo[5]), fmaxf(mo[6], mo[7])));
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
                const uint64_t mo2 = f2(m_own, m_own);
#pragma unroll
                for (int c8 = 0; c8 < kT / 8; ++c8) {
                    uint32_t w[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 d = f2_unpack(f2_sub(f2(pv[8 * c8 + 2 * u], pv[8 * c8 + 2 * u + 1]), mo2));
                        const __half2 h2 = __floats2half2_rn(d.x, d.y);
                        w[u] = *reinterpret_cast<const uint32_t*>(&h2);
                    }
                    *reinterpret_cast<uint4*>(sY + xrow + ((c8 ^ (lane & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                y_off[lane] = m_own;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // the other CTA's group B has consumed the previous tile from these rows
                    if (ok_a && j >= 1) ok_a = wait_bounded_cluster(&xfree[sub], (j - 1) & 1, p.status);
                    if (ok_a) {
                        bulk_copy_to_cta(peer_x, sY + my_slice, kXSlice, peer_xfull);
                        bulk_commit_group();
                    }
                }
                ok_a = __shfl_sync(0xffffffffu, ok_a ? 1 : 0, 0) != 0;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ownfull);
                if (!ok_a) { *(volatile int*)abort_flag = 1; break; }
            }
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
        } else {
            const uint32_t peer_xfree = map_to_rank(smem_u32(&xfree[sub]), peer);
            const float coef = coef_s[r];      // exp2-domain logit = coef x (this group's working units)
            // arm for tile 0's rows; the other CTA's copy may complete its bytes first
            // (the transaction count goes negative), the phase still needs this arrive
            if (lane == 0 && n_t > 0) mbar_arrive_expect_tx(&xfull[sub], kXSlice);
            float m_run = -INFINITY, l_run = 0.f;
            bool ok = true;
            float lg[kT];
            for (int j = 0; j < n_t; ++j) {
                const int s = j % kNst, pb = j & 1;
                const int valid = min(kT, L - (jt0 + j) * kT);
                // ---- this CTA's fp32 partials from group A ----
                const bool got_own = __all_sync(0xffffffffu, wait_bounded(ownfull, j & 1, p.status));
                tc_fence_after();
                {
                    uint32_t v[kT];
                    tmem_ld64(tmem + kCOwn + lane_base, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int t = 0; t < kT; ++t) lg[t] = __uint_as_float(v[t]);
                }
                const float m_own = y_off[lane];          // group A's row maximum of these partials
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ownfree);
                // P (bf16) into TMEM buffer pb once the output MMA two tiles back released it
                if (j >= 2) {
                    const bool got_p = __all_sync(0xffffffffu, wait_bounded(&pdone[pb], ((j >> 1) - 1) & 1, p.status));
                    if (!got_p) { ok = false; *(volatile int*)abort_flag = 1; break; }
                    tc_fence_after();
                }
                // ---- + the other CTA's ----
                const bool got_x =
                    __all_sync(0xffffffffu, got_own && wait_bounded_cluster(&xfull[sub], j & 1, p.status));
                if (!got_x) { ok = false; *(volatile int*)abort_flag = 1; break; }
                const float off = x_off[lane];
                uint32_t xw[kT / 2];
#pragma unroll
                for (int c8 = 0; c8 < kT / 8; ++c8) {
                    const uint4 v = *reinterpret_cast<const uint4*>(sX + xrow + ((c8 ^ (lane & 7)) << 4));
                    xw[4 * c8] = v.x; xw[4 * c8 + 1] = v.y; xw[4 * c8 + 2] = v.z; xw[4 * c8 + 3] = v.w;
                }
                {
                    // every X value has been read: arm for the next tile and let the other CTA
                    // overwrite these rows
                    uint32_t xdep = __float_as_uint(off);
#pragma unroll
                    for (int u = 0; u < kT / 2; u += 4) xdep ^= xw[u];   // one word per 16-byte load
                    const uint32_t xdep_w = __reduce_xor_sync(0xffffffffu, xdep);
                    if (lane == 0 && j + 1 < n_t) {
                        mbar_arrive_expect_tx(&xfull[sub], kXSlice);
                        mbar_arrive_remote_after(peer_xfree, xdep_w, p.zero);
                    }
                }
                // own max + partner max bounds the tile max: when it cannot move the running
                // max (by > 8, log2) for any row of the warp and the tile is full, the sums go
                // straight into the exponentials
                const bool fast = __all_sync(0xffffffffu, valid == kT && coef * (m_own + off) <= m_run + 8.f);
                float ps4[4] = {0.f, 0.f, 0.f, 0.f};
                if (fast) {
                    // two tokens per packed instruction: (lg + (off + x)) - m_run, then
                    // two exponentials and the packed running sums
                    const uint64_t c2 = f2(coef, coef), nm2 = f2(-m_run, -m_run);
                    uint64_t ps2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t w16[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const int t = 32 * h + 2 * q;
                            const float2 a = half2_plus(xw[t >> 1], off);          // off + partner, exact as before
                            const float2 x2 = f2_unpack(f2_fma(c2, f2_add(f2(lg[t], lg[t + 1]), f2(a.x, a.y)), nm2));
                            const float e0 = fast_exp2(x2.x);
                            const float e1 = fast_exp2(x2.y);
                            ps2[q & 1] = f2_add(ps2[q & 1], f2(e0, e1));
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(e0, e1);
                            w16[q] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        tmem_st16(tmem + kCP + pb * (kT / 2) + 16 * h + lane_base, w16);
                    }
                    tmem_wait_st();
                    const float2 s0 = f2_unpack(ps2[0]), s1 = f2_unpack(ps2[1]);
                    l_run += (s0.x + s0.y) + (s1.x + s1.y);
                } else {
#pragma unroll
                    for (int t = 0; t < kT; t += 2) {
                        const float2 a = half2_plus(xw[t >> 1], off);
                        lg[t] += a.x;
                        lg[t + 1] += a.y;
                    }
                    if (valid < kT) {
#pragma unroll
                        for (int t = 0; t < kT; ++t)
                            if (t >= valid) lg[t] = -INFINITY;
                    }
                    float corr = 1.f;
                    bool need = false;
                    if (coef * (m_own + off) > m_run + 8.f) {
                        float mx[8];                           // tree max: short dependency chains
#pragma unroll
                        for (int q = 0; q < 8; ++q) mx[q] = fmaxf(fmaxf(lg[q], lg[q + 8]), fmaxf(lg[q + 16], lg[q + 24]));
#pragma unroll
                        for (int q = 0; q < 8; ++q) mx[q] = fmaxf(mx[q], fmaxf(fmaxf(lg[q + 32], lg[q + 40]), fmaxf(lg[q + 48], lg[q + 56])));
                        const float mt = coef * fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                                      fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                        need = mt > m_run + 8.f;
                        if (need) {
                            corr = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mt);
                            m_run = mt;
                        }
                    }
                    // TMEM loads/stores are warp-collective: the whole warp rescales when any
                    // of its rows needs it, each lane by its own factor (1 for the others)
                    if (j > 0 && __any_sync(0xffffffffu, need)) {
                        const bool got_o =
                            __all_sync(0xffffffffu, wait_bounded(&pdone[(j - 1) & 1], ((j - 1) >> 1) & 1, p.status));
                        if (!got_o) { ok = false; *(volatile int*)abort_flag = 1; break; }
                        tc_fence_after();
#pragma unroll 1
                        for (int c16 = 0; c16 < kHalfLat; c16 += 16) {
                            uint32_t v[16];
                            tmem_ld16(tmem + kCO + c16 + lane_base, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) v[jj] = __float_as_uint(__uint_as_float(v[jj]) * corr);
                            tmem_st16(tmem + kCO + c16 + lane_base, v);
                        }
                        tmem_wait_st();
                    }
                    l_run *= corr;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t w16[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const float e0 = fast_exp2(fmaf(coef, lg[32 * h + 2 * q], -m_run));
                            const float e1 = fast_exp2(fmaf(coef, lg[32 * h + 2 * q + 1], -m_run));
                            ps4[q & 3] += e0 + e1;
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(e0, e1);
                            w16[q] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        tmem_st16(tmem + kCP + pb * (kT / 2) + 16 * h + lane_base, w16);
                    }
                    tmem_wait_st();
                    l_run += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
                }
                if (valid < kT) {   // zero this CTA's latent rows past the sequence end (this warp's share)
                    uint8_t* stg = sm + kOffStage + s * kStageB;
                    const int nrow = kT - valid;
                    for (int e = lane + 32 * sub; e < nrow * 4 * 8; e += 128) {
                        const int rr = valid + e / 32, rem = e % 32;
                        *reinterpret_cast<uint4*>(stg + (rem >> 3) * (kT * 128) + rr * 128 + (rem & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pfull[pb]);
            }
            // ---- epilogue: thread = row, its 256 latents ----
            bool got_last =
                (ok && n_t > 0) ? wait_bounded(&pdone[(n_t - 1) & 1], ((n_t - 1) >> 1) & 1, p.status) : true;
            got_last = __all_sync(0xffffffffu, got_last);      // TMEM reads below are warp-collective
            tc_fence_after();
            if (!got_last) *(volatile int*)abort_flag = 1;
            const size_t orow = ((size_t)b * p.s_q + qi) * p.H + r;
            if (rank == 0) {
                const float lse = (l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
                if (it.part < 0) {
                    if (p.lse) p.lse[orow] = lse;
                } else {
                    p.lse_part[(size_t)it.part * p.s_q * p.H + (size_t)qi * p.H + r] = lse;
                }
            }
            const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
            float* dst_part = (it.part >= 0)
                                  ? p.o_part + ((size_t)it.part * p.s_q * p.H + (size_t)qi * p.H + r) * kDC + rank * kHalfLat
                                  : nullptr;
#pragma unroll 1
            for (int c64 = 0; c64 < kHalfLat; c64 += 64) {
                uint32_t v[64];
                if (n_t > 0 && got_last) {
                    tmem_ld64(tmem + kCO + c64 + lane_base, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int jj = 0; jj < 64; ++jj) v[jj] = 0u;
                }
#pragma unroll
                for (int c16 = 0; c16 < 64; c16 += 16) {
                    float o16[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) o16[jj] = __uint_as_float(v[c16 + jj]) * inv;
                    const int col = rank * kHalfLat + c64 + c16;
                    if (dst_part) {
                        float4* d4 = reinterpret_cast<float4*>(dst_part + c64 + c16);
#pragma unroll
                        for (int q = 0; q < 4; ++q) d4[q] = make_float4(o16[4 * q], o16[4 * q + 1], o16[4 * q + 2], o16[4 * q + 3]);
                    } else if (p.o_dtype == QKMLA_F32) {
                        float4* d4 = reinterpret_cast<float4*>((float*)p.o + orow * kDC + col);
#pragma unroll
                        for (int q = 0; q < 4; ++q) d4[q] = make_float4(o16[4 * q], o16[4 * q + 1], o16[4 * q + 2], o16[4 * q + 3]);
                    } else {
                        uint32_t w[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(o16[2 * q], o16[2 * q + 1]);
                            w[q] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        uint4* d4 = reinterpret_cast<uint4*>((__nv_bfloat16*)p.o + orow * kDC + col);
                        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync();            // no remote access to this CTA after this point
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

int launch_pair(const qkmla_decode_args* a, const TcParams& tp, int max_items, cudaStream_t s) {
    CUtensorMap lat, rope, qmap;
    const int row = a->d_c + a->d_r;
    if (!make_map(&lat, a->kv_cache, a->num_slots, row, 64, kT, CU_TENSOR_MAP_SWIZZLE_128B)) return QKMLA_ERR_CUDA;
    if (!make_map(&rope, a->kv_cache, a->num_slots, row, 32, kT, CU_TENSOR_MAP_SWIZZLE_64B)) return QKMLA_ERR_CUDA;
    if (!make_map(&qmap, a->q_tilde, (int64_t)a->B * a->s_q * a->H, kDC, 64, kR, CU_TENSOR_MAP_SWIZZLE_128B))
        return QKMLA_ERR_CUDA;
    const bool plain = (a->flags & QKMLA_FLAG_PLAIN_MLA) != 0;
    const bool akh = !plain && (a->flags & QKMLA_FLAG_ALPHA_F16) != 0;
    auto k = plain ? decode_pair_kernel<true, false> : akh ? decode_pair_kernel<false, true> : decode_pair_kernel<false, false>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kBytesP) != cudaSuccess)
        return QKMLA_ERR_CUDA;
    dim3 grid(2 * a->s_q, max_items);
    return launch_pdl(k, grid, dim3(kThreadsP), kBytesP, s, lat, rope, qmap, tp) == cudaSuccess ? QKMLA_OK
                                                                                       : QKMLA_ERR_CUDA;
}

}  // namespace dec
}  // namespace qkmla
