// Tensor-core decode kernel for a bf16 latent cache (tcgen05 + TMEM + TMA).
//
// Source: "QK-Normed MLA: QK normalization without full key caching", Technical
// Summary, Methodology -- decode-logit equation l = (q~ . c_t) alpha^q alpha^k_{t,g(h)}
// with the scalars applied as a row/column scaling of the logit tile before the
// softmax; "Blockwise Normalization" (separately normalised RoPE logit); the
// Significance section's note that speed depends on fusing the scalar factors
// into the attention path.  Values are the latents (latent decode path).
//
// Work decomposition.  A CTA owns up to 64 query rows (heads of one query
// token) of one sequence and a contiguous range of tiles (64 tokens for
// d_c = 256, 32 for d_c = 512).  Per tile:
//   S_c = Q~ C^T   (M=64 rows, N=tile tokens, K=d_c)   tcgen05, fp32 in TMEM
//   S_r = Q^r K^rT (M=64,      N=tile tokens, K=d_r)   tcgen05, fp32 in TMEM
//   l   = scale*(alpha^q_row * alpha^k_{t,g(row)} * S_c + S_r)      (fused, fp32)
//   P   = exp2(l*log2e - m_row), stored bf16 into the tile's RoPE slot
//   O^T += C^T P^T (M=128 latent coords per chunk, N=rows, K=tile tokens)
// O is kept transposed in TMEM (latent coordinate = lane, row = column): 64 rows
// x 512 latents take 256 of the 512 TMEM columns, leaving room for two S
// buffers.  The running max only moves when a tile's max exceeds it by more
// than 2^8 (normalised logits are bounded, so after the first tile this almost
// never happens); then O is rescaled in TMEM.
//
// Warp roles (192 threads): warp 0 issues TMA loads (and owns the TMEM
// allocation), warp 1 issues MMAs, warps 2-5 do the softmax, the rescale and
// the epilogue.  Every wait is bounded; on expiry QKMLA_ERR_TIMEOUT is recorded.
//
// The split plan (work items: sequence, tile range) comes from seq_lens on the
// device -- computed by every CTA itself for up to 128 sequences, by a
// scheduler kernel beyond; long sequences are split and merged afterwards by a
// combine kernel.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "decode_common.cuh"
#include "decode_sched.cuh"
#include "tc_ptx.cuh"

namespace qkmla {

namespace {

using namespace tc;
using namespace dec;

constexpr int kRowsMMA = 64;       // M of the logit MMA
constexpr int kThreads = 192;

// Tokens per tile: 64 for d_c = 256, 32 for d_c = 512.  The logit MMA costs the
// same issue time for any N up to 128, so wider tiles cut its cost per token; the
// width is bounded by the TMA ring, which needs about three stages in flight to
// cover DRAM latency (stage = one tile, one TMA box, one page-table lookup).
template <int DC>
constexpr int tile_of() { return DC == 256 ? 64 : 32; }

// ---------------------------------------------------------------------------
// shared-memory layout
// ---------------------------------------------------------------------------
template <int DC, int DR, int NST, int KT>
struct Layout {
    static constexpr int kLatBlocks = DC / 64;                      // 64-column TMA boxes
    static constexpr int kRopeRowBytes = DR * 2;                    // 128 (SW128) or 64 (SW64)
    static constexpr int kQLat = kLatBlocks * kRowsMMA * 128;
    static constexpr int kQRope = kRowsMMA * kRopeRowBytes;
    static constexpr int kSLat = kLatBlocks * KT * 128;
    static constexpr int kSRope = KT * kRopeRowBytes;
    static constexpr int kSAk = KT * kMaxG * 4;
    // P^T (up to 64 rows x KT tokens, bf16) reuses the tile's RoPE slot when it fits
    // there (d_c = 512); for d_c = 256 it has a slot of its own, so 64 rows fit
    static constexpr int kPBytes = kRowsMMA * KT * 2;
    static constexpr bool kPOwn = kPBytes > kSRope;
    static constexpr int kOffP = kPOwn ? (kSLat + kSRope + kSAk + 1023) / 1024 * 1024 : kSLat;
    static constexpr int kStage = ((kPOwn ? kOffP + kPBytes : kSLat + kSRope + kSAk) + 1023) / 1024 * 1024;
    static constexpr int kQ = ((kQLat + kQRope) + 1023) / 1024 * 1024;
    static constexpr int kOffQ = 0;
    static constexpr int kOffStage = kQ;
    static constexpr int kOffMisc = kQ + NST * kStage;
    // logit buffers in TMEM: two when they fit beside the widest O^T (4 x 64 columns)
    static constexpr int kChunks = DC / 128;
    static constexpr int kNSB = (4 * KT + kChunks * 64 <= 512) ? 2 : 1;
    static constexpr uint32_t kColSc = 0, kColSr = kNSB * KT, kColO = 2 * kNSB * KT;
    // misc: barriers then per-row arrays
    static constexpr int kNumBars = 3 * NST + 2 * kNSB + 2;
    static constexpr int kMisc = kNumBars * 8 + 16 + 4 * kRowsMMA * 4;
    static constexpr int kBytes = kOffMisc + kMisc + 1024;        // + alignment slack
    // bytes one tile brings: latent blocks + RoPE rows (alpha^k is added at run time)
    static constexpr uint32_t kTileTx = (uint32_t)(kLatBlocks * KT * 128 + KT * kRopeRowBytes);
    static_assert(kColO + kChunks * 64 <= 512, "TMEM budget");
    static_assert(KT == 32 || KT == 64, "a tile is one TMA box of a 32- or 64-token page piece");
};

constexpr uint32_t kTmemCols = 512;

// Byte offset of P^T element (row r, token t) in the tile's RoPE slot: K-major
// (K = tokens); 32-token tiles use 64-byte rows with the 64-byte swizzle, wider
// tiles 64-token atoms of 128-byte rows with the 128-byte swizzle.
template <int KT>
__device__ __forceinline__ uint32_t pt_offset(int r, int t, int rows_o) {
    if (KT == 32) return sw64_offset(r, t);
    return (uint32_t)(t >> 6) * (uint32_t)(rows_o * 128) + sw128_offset(r, t & 63);
}

// AKH: A^k_cache entries are fp16 (else fp32)
template <int DC, int DR, bool PLAIN, int NST, int KT, bool AKH>
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope,
                 const __grid_constant__ CUtensorMap tm_q, const TcParams p) {
    using LY = Layout<DC, DR, NST, KT>;
    constexpr int kChunks = LY::kChunks;
    constexpr int NSB = LY::kNSB;
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = sm + LY::kOffQ;
    uint64_t* bars = (uint64_t*)(sm + LY::kOffMisc);
    uint64_t* full = bars;                   // [NST] TMA -> MMA
    uint64_t* empty = bars + NST;            // [NST] output MMA done -> TMA
    uint64_t* pfull = bars + 2 * NST;        // [NST] P written -> output MMA
    uint64_t* sfull = bars + 3 * NST;        // [NSB] logit MMA done -> softmax
    uint64_t* sfree = sfull + NSB;           // [NSB] softmax read S -> MMA
    uint64_t* odone = sfree + NSB;           // output MMA of a tile done
    uint64_t* qfull = odone + 1;             // Q~ tile landed
    uint32_t* tmem_slot = (uint32_t*)(bars + LY::kNumBars);
    int* abort_flag = (int*)(tmem_slot + 1);
    float* coef_s = (float*)(sm + LY::kOffMisc + LY::kNumBars * 8 + 16);
    float* corr_s = coef_s + kRowsMMA;
    float* l_s = corr_s + kRowsMMA;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int item_idx = blockIdx.y;
    WorkItem it;
    int seq_len;
    // the in-kernel plan reads only seq_lens, which no kernel of the call writes: it
    // is made before the dependency wait, overlapping the previous kernel's tail
    if (p.sched_inline) {
        __shared__ SchedSmem S;
        compute_schedule(p.seq_lens, p.B, p.s_q, p.sa, S, p.status, item_idx == 0 && blockIdx.x == 0);
        if (item_idx >= S.n_items) return;
        it = schedule_item(S, p.B, item_idx);
        seq_len = S.len[it.b];                     // the plan's copy: no second trip to memory
    } else {
        pdl_wait();                                // the scheduler kernel's items
        if (item_idx >= *p.n_items) return;
        it = p.items[item_idx];
        seq_len = p.seq_lens[it.b];
    }
    const int rows_o = p.rows_o;
    const int row0 = blockIdx.x * rows_o;          // row index within the sequence's s_q*H rows
    const int qi = row0 / p.H, h0 = row0 % p.H;    // the first row's query token and head
    const int b = it.b;
    const bool bad = seq_len < p.s_q || seq_len > p.max_pages * p.page_size;
    // rows_o may cover several query tokens (rows_o > H): the tiles run to the last
    // row's causal length, and each row masks past its own
    const int L = bad ? 0 : seq_len - p.s_q + (row0 + rows_o - 1) / p.H + 1;
    const int tiles = (L + KT - 1) / KT;
    const int jt0 = it.tile_begin;
    const int jt1 = min(it.tile_end, tiles);
    const int n_t = max(0, jt1 - jt0);
    const int hpg = p.H / p.G;
    // tiles the producer issues: all of them, or (test hook) those before the
    // withheld one -- the consumers' waits for the next tile then run out
    const int n_issue = p.withhold_tile >= 0 ? min(n_t, p.withhold_tile) : n_t;

    if (tid == 0) {
        if (bad) report(p.status, QKMLA_ERR_DEVICE_BOUNDS);
        for (int s = 0; s < LY::kNumBars; ++s) {
            uint32_t cnt = 1;
            if (s >= 2 * NST && s < 3 * NST) cnt = 4;                  // pfull: one arrive per softmax warp
            if (s >= 3 * NST + NSB && s < 3 * NST + 2 * NSB) cnt = 4;  // sfree
            mbar_init(&bars[s], cnt);
        }
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tm_lat);
        if (DR != 64) prefetch_tmap(&tm_rope);
        prefetch_tmap(&tm_q);
    }
    __syncthreads();
    pdl_wait();                                    // q~, alpha^q and the cache are written by earlier kernels
    pdl_trigger();
    const size_t qrow0 = ((size_t)b * p.s_q + qi) * p.H + h0;

    // ---- TMA producer state (warp 0): the slot of tile j + lane, 32 tiles at a time ----
    auto slot_of_tile = [&](int j) -> int64_t {
        if (j >= n_t) return 0;
        const int t0 = (jt0 + j) * KT;
        const int pg = t0 / p.page_size;
        int64_t page = p.page_table ? (int64_t)p.page_table[(int64_t)b * p.max_pages + pg]
                                    : (int64_t)b * p.max_pages + pg;
        if (page < 0 || page >= p.num_pages) {
            report(p.status, QKMLA_ERR_DEVICE_BOUNDS);
            page = 0;
        }
        return page * p.page_size + (t0 % p.page_size);
    };
    const uint32_t ak_bytes = PLAIN ? 0u : (uint32_t)(KT * p.G * (AKH ? 2 : 4));
    auto issue_tile = [&](int j, int64_t slot0) {        // lane 0 of warp 0
        const int s = j % NST;
        uint8_t* stg = sm + LY::kOffStage + s * LY::kStage;
        mbar_arrive_expect_tx(&full[s], LY::kTileTx + ak_bytes);
#pragma unroll
        for (int blk = 0; blk < LY::kLatBlocks; ++blk)
            tma_load_2d(stg + blk * (KT * 128), &tm_lat, blk * 64, (int)slot0, &full[s]);
        if (DR == 64)
            tma_load_2d(stg + LY::kSLat, &tm_lat, DC, (int)slot0, &full[s]);
        else
            tma_load_2d(stg + LY::kSLat, &tm_rope, DC, (int)slot0, &full[s]);
        if (!PLAIN)
            bulk_load(stg + LY::kSLat + LY::kSRope, (const uint8_t*)p.ak + slot0 * p.G * (AKH ? 2 : 4), ak_bytes, &full[s]);
    };
    int64_t slot_batch = 0;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
        // the Q~ tile and the first NST tiles go out before the prologue barrier
        slot_batch = slot_of_tile(lane);
        if (lane == 0) {
            mbar_arrive_expect_tx(qfull, (uint32_t)(LY::kLatBlocks * rows_o * 128));
#pragma unroll
            for (int blk = 0; blk < LY::kLatBlocks; ++blk)
                tma_load_2d(sQ + blk * (kRowsMMA * 128), &tm_q, blk * 64, (int)qrow0, qfull);
        }
        for (int j = 0; j < NST && j < n_issue; ++j) {
            const int64_t slot0 = __shfl_sync(0xffffffffu, slot_batch, j);
            if (lane == 0) issue_tile(j, slot0);
        }
    } else if (warp >= 2) {
        // ---- prologue (softmax warps): the normalised RoPE query, alpha^q, and
        //      zero Q~ rows past rows_o (the TMA fills rows 0 .. rows_o-1) ----
        const int st = tid - 64;
        for (int e = st; e < (kRowsMMA - rows_o) * 8 * LY::kLatBlocks; e += 128) {
            const int r = rows_o + e / (8 * LY::kLatBlocks), rem = e % (8 * LY::kLatBlocks);
            *reinterpret_cast<uint4*>(sQ + (rem >> 3) * (kRowsMMA * 128) + r * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        // RoPE query: two threads per row
        {
            const int r = st >> 1, half = st & 1;
            // every global read of the prologue is issued before the first shared-memory
            // store: a load after a store through generic pointers waits for it, which
            // would put one memory round trip per store on this path
            float vals[DR / 2], gq[DR / 2];
            const float* src = p.qr + (qrow0 + r) * DR + half * (DR / 2);
#pragma unroll
            for (int j = 0; j < DR / 2; ++j) {
                vals[j] = (r < rows_o) ? src[j] : 0.f;
                gq[j] = (PLAIN || !p.grq) ? 1.f : p.grq[half * (DR / 2) + j];
            }
            const float a = (PLAIN || r >= rows_o || half) ? 1.f : p.aq[qrow0 + r];
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < DR / 2; ++j) ss = fmaf(vals[j], vals[j], ss);
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            // QK mode: the RoPE query carries scale*log2e, so the MMA delivers the RoPE
            // logit already in the exp2 domain
            const float beta = PLAIN ? 1.f : p.scale * kLog2e / sqrtf(ss / (float)DR + p.eps);
            uint8_t* qrope = sQ + LY::kQLat;
#pragma unroll
            for (int j = 0; j < DR / 2; j += 2) {
                const int c = half * (DR / 2) + j;
                __nv_bfloat162 v = __floats2bfloat162_rn(vals[j] * gq[j] * beta, vals[j + 1] * gq[j + 1] * beta);
                const uint32_t off = (DR == 64) ? sw128_offset(r, c) : sw64_offset(r, c);
                *reinterpret_cast<__nv_bfloat162*>(qrope + off) = v;
            }
            if (half == 0) coef_s[r] = p.scale * a * kLog2e;
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ===================== TMA producer (lane 0 issues; lanes hold page slots) =====================
        for (int j = NST; j < n_issue; ++j) {
            if ((j & 31) == 0) slot_batch = slot_of_tile(j + lane);
            const int64_t slot0 = __shfl_sync(0xffffffffu, slot_batch, j & 31);
            int go = 1;
            if (lane == 0) {
                const int s = j % NST;
                if (!wait_bounded(&empty[s], ((j / NST) - 1) & 1, p.status, p.wait_ns)) {
                    *abort_flag = 1;
                    go = 0;
                } else if (*(volatile int*)abort_flag) {
                    go = 0;
                } else {
                    issue_tile(j, slot0);
                }
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(kRowsMMA, KT, 0, 0);
            const uint32_t id_o = idesc_bf16(128, rows_o, 1, 0);
            const uint32_t q_addr = smem_u32(sQ);
            auto issue_o = [&](int jj) -> bool {
                const int s = jj % NST;
                if (!wait_bounded(&pfull[s], (jj / NST) & 1, p.status, p.wait_ns)) return false;
                tc_fence_after();
                const uint32_t st_addr = smem_u32(sm + LY::kOffStage + s * LY::kStage);
                const uint32_t p_addr = st_addr + LY::kOffP;       // P^T: the RoPE slot or its own
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
#pragma unroll
                    for (int kk = 0; kk < KT / 16; ++kk) {
                        // A = C^T chunk c: MN-major, two 64-column boxes (LBO = box stride),
                        // 8-token groups 1024 B apart (SBO); B = P^T rows, K-major.
                        const uint64_t a = smem_desc(st_addr + (2 * c) * (KT * 128) + kk * 2048, KT * 128, 1024,
                                                     kSwizzle128B);
                        const uint64_t bdesc =
                            KT == 32 ? smem_desc(p_addr + kk * 32, 16, 512, kSwizzle64B)
                                     : smem_desc(p_addr + (kk >> 2) * (rows_o * 128) + (kk & 3) * 32, 16, 1024,
                                                 kSwizzle128B);
                        mma_bf16(tmem + LY::kColO + c * rows_o, a, bdesc, id_o, (jj > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                mma_commit(&empty[s]);
                mma_commit(odone);
                return true;
            };
            // always waited, so no CTA exits with the Q~ copy in flight
            bool ok = wait_bounded(qfull, 0, p.status, p.wait_ns);
            for (int j = 0; j < n_t && ok; ++j) {
                const int s = j % NST, sb = j % NSB;
                if (!wait_bounded(&full[s], (j / NST) & 1, p.status, p.wait_ns)) { ok = false; break; }
                if (j >= NSB && !wait_bounded(&sfree[sb], ((j / NSB) - 1) & 1, p.status, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t st_addr = smem_u32(sm + LY::kOffStage + s * LY::kStage);
                const uint32_t d_c = tmem + LY::kColSc + sb * KT;
                const uint32_t d_r = tmem + LY::kColSr + sb * KT;
#pragma unroll
                for (int blk = 0; blk < LY::kLatBlocks; ++blk) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = smem_desc(q_addr + blk * (kRowsMMA * 128) + kk * 32, 16, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(st_addr + blk * (KT * 128) + kk * 32, 16, 1024, kSwizzle128B);
                        mma_bf16(d_c, a, bd, id_s, (blk > 0 || kk > 0) ? 1u : 0u);
                    }
                }
#pragma unroll
                for (int kk = 0; kk < DR / 16; ++kk) {
                    uint64_t a, bd;
                    if (DR == 64) {
                        a = smem_desc(q_addr + LY::kQLat + kk * 32, 16, 1024, kSwizzle128B);
                        bd = smem_desc(st_addr + LY::kSLat + kk * 32, 16, 1024, kSwizzle128B);
                    } else {
                        a = smem_desc(q_addr + LY::kQLat + kk * 32, 16, 512, kSwizzle64B);
                        bd = smem_desc(st_addr + LY::kSLat + kk * 32, 16, 512, kSwizzle64B);
                    }
                    if (!PLAIN) {
                        mma_bf16(d_r, a, bd, id_s, kk > 0 ? 1u : 0u);
                    } else {
                        mma_bf16(d_c, a, bd, id_s, 1u);      // plain MLA: one accumulation over K = d_c + d_r
                    }
                }
                mma_commit(&sfull[sb]);
                if (j >= 1) ok = issue_o(j - 1);
            }
            if (ok && n_t > 0) ok = issue_o(n_t - 1);
            if (!ok) *(volatile int*)abort_flag = 1;
        }
    } else {
        // ===================== softmax / rescale / epilogue =====================
        const int sub = warp & 3;                      // TMEM sub-partition of this warp
        const uint32_t lane_base = (uint32_t)(32 * sub) << 16;
        // M=64 accumulator layout: row r sits in lane r%16 of sub-partition r/16.  The
        // 16x32bx2 TMEM load gives lanes 0-15 columns c..c+15 and lanes 16-31 columns
        // c+16..c+31 of the same 16 rows: two threads per row, every lane busy.  A
        // thread holds tokens 32 q + 16 half + (0..15) for q < KT/32.
        constexpr int kQ4 = KT / 32;
        const int half = lane >> 4;
        const int r = 16 * sub + (lane & 15);
        const int tb = 16 * half;
        const bool row_ok = r < rows_o;
        const int g = row_ok ? ((h0 + r) % p.H) / hpg : 0;
        const int L_r = bad ? 0 : seq_len - p.s_q + (row0 + (row_ok ? r : 0)) / p.H + 1;   // this row's length
        const float coef = row_ok ? coef_s[r] : 0.f;
        const float rs = p.scale * kLog2e;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        bool late_fail = false;      // a timed-out wait at the end of the previous tile
        for (int j = 0; j < n_t; ++j) {
            const int s = j % NST, sb = j % NSB;
            const int tile = jt0 + j;
            // a timed-out wait is folded into the per-tile vote below, so every abort
            // decision is uniform across the four softmax warps (none is left at a
            // named barrier)
            const bool got_s = wait_bounded(&sfull[sb], (j / NSB) & 1, p.status, p.wait_ns);
            if (!got_s) *(volatile int*)abort_flag = 1;
            tc_fence_after();
            uint8_t* stg = sm + LY::kOffStage + s * LY::kStage;
            const void* ak_t = stg + LY::kSLat + LY::kSRope;
            const int valid = min(KT, L - tile * KT);          // the CTA's longest row
            const int valid_r = min(KT, L_r - tile * KT);      // this row (may be <= 0)
            // the column scales of this thread's tokens first (shared memory, landed with
            // the tile the completed logit MMA read), then every TMEM load of the tile and one
            // wait: the latencies overlap instead of adding up per 32-token chunk
            float ca[kQ4][16];
            if (!PLAIN) {
#pragma unroll
                for (int q = 0; q < kQ4; ++q)
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 2) {      // two tokens per packed multiply
                        const float2 c2 = f2_unpack(f2_mul(f2(coef, coef),
                                                           f2(load_alpha<AKH>(ak_t, (32 * q + tb + jj) * p.G + g),
                                                              load_alpha<AKH>(ak_t, (32 * q + tb + jj + 1) * p.G + g))));
                        ca[q][jj] = c2.x;
                        ca[q][jj + 1] = c2.y;
                    }
            }
            uint32_t sc[kQ4][16], sr[kQ4][16];
#pragma unroll
            for (int q = 0; q < kQ4; ++q) {
                tmem_ld16x2(tmem + LY::kColSc + sb * KT + 32 * q + lane_base, sc[q]);
                if (!PLAIN) tmem_ld16x2(tmem + LY::kColSr + sb * KT + 32 * q + lane_base, sr[q]);
            }
            tmem_wait_ld();
            // S is in registers: release the buffer to the logit MMA before scaling
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfree[sb]);
            float lg[kQ4][16];
#pragma unroll
            for (int q = 0; q < kQ4; ++q) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    if (PLAIN) {
                        lg[q][jj] = rs * __uint_as_float(sc[q][jj]);
                    } else if ((jj & 1) == 0) {
                        const float2 l2 = f2_unpack(f2_fma(f2(ca[q][jj], ca[q][jj + 1]),
                                                           f2(__uint_as_float(sc[q][jj]), __uint_as_float(sc[q][jj + 1])),
                                                           f2(__uint_as_float(sr[q][jj]), __uint_as_float(sr[q][jj + 1]))));
                        lg[q][jj] = l2.x;
                        lg[q][jj + 1] = l2.y;
                    }
                }
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    if (32 * q + tb + jj >= valid_r) lg[q][jj] = -INFINITY;
            }
            float mt = -INFINITY;
#pragma unroll
            for (int q = 0; q < kQ4; ++q) {
                float m5[6];
#pragma unroll
                for (int i = 0; i < 5; ++i) m5[i] = fmax3(lg[q][3 * i], lg[q][3 * i + 1], lg[q][3 * i + 2]);
                m5[5] = lg[q][15];
                mt = fmax3(mt, fmax3(m5[0], m5[1], m5[2]), fmax3(m5[3], m5[4], m5[5]));
            }
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
            // lazy running max: move it only when the tile max exceeds it by > 8 (log2)
            float corr = 1.f;
            int need = 0;
            if (row_ok && mt > m_run + 8.f) {
                corr = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mt);
                m_run = mt;
                need = (j > 0) ? 1 : 0;
            }
            if (half == 0) corr_s[r] = row_ok ? corr : 1.f;
            const bool any = named_bar_any(need || !got_s || late_fail);
            if (any && *(volatile int*)abort_flag) { ok = false; break; }
            // odone completes once per tile.  Its phase j-1 (output MMA of the previous
            // tile) is consumed on every tile, before P(j) is released: the barrier is
            // then never two phases ahead of this wait, so the parity names one phase.
            bool o_seen = (j == 0);
            if (any) {
                // rescale O^T columns (rows) in TMEM once the previous output MMA is done
                const bool got_o = wait_bounded(odone, (j - 1) & 1, p.status, p.wait_ns);
                if (named_bar_any(!got_o)) { ok = false; break; }
                o_seen = true;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < kChunks; ++c) {
                    for (int c16 = 0; c16 < rows_o; c16 += 16) {
                        uint32_t v[16];
                        const uint32_t ta = tmem + LY::kColO + c * rows_o + c16 + lane_base;
                        tmem_ld16(ta, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            v[jj] = __float_as_uint(__uint_as_float(v[jj]) * corr_s[c16 + jj]);
                        tmem_st16(ta, v);
                    }
                }
                tmem_wait_st();
                // corr_s is rewritten by the next tile: every thread must be done reading it
                named_bar_sync();
            }
            l_run *= corr;
            // a row with no token yet (m_run still -inf) gets P = 0, not exp2(NaN)
            const float m_e = (m_run == -INFINITY) ? 0.f : m_run;
            // P^T row r, this thread's tokens, into the RoPE slot (bf16)
            uint8_t* pT = stg + LY::kOffP;
            float psum = 0.f;
#pragma unroll
            for (int q = 0; q < kQ4; ++q) {
                uint32_t w8[8];
                uint64_t ps2 = f2(0.f, 0.f);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float2 x2 = f2_unpack(f2_sub(f2(lg[q][2 * u], lg[q][2 * u + 1]), f2(m_e, m_e)));
                    const float e0 = fast_exp2(x2.x);
                    const float e1 = fast_exp2(x2.y);
                    ps2 = f2_add(ps2, f2(e0, e1));
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(e0, e1);
                    w8[u] = *reinterpret_cast<const uint32_t*>(&b2);
                }
                const float2 s2 = f2_unpack(ps2);
                psum += s2.x + s2.y;
                if (row_ok) {
                    const int t = 32 * q + tb;
                    *reinterpret_cast<uint4*>(pT + pt_offset<KT>(r, t, rows_o)) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
                    *reinterpret_cast<uint4*>(pT + pt_offset<KT>(r, t + 8, rows_o)) =
                        make_uint4(w8[4], w8[5], w8[6], w8[7]);
                }
            }
            l_run += psum;
            // the last tile of the sequence: zero the latent rows past its end so that
            // stale slot contents (possibly NaN) cannot reach the output MMA
            if (valid < KT) {
                const int st = tid - 64;
                const int nrow = KT - valid;
                for (int e = st; e < nrow * LY::kLatBlocks * 8; e += 128) {
                    const int rr = valid + e / (LY::kLatBlocks * 8);
                    const int rem = e % (LY::kLatBlocks * 8);
                    *reinterpret_cast<uint4*>(stg + (rem >> 3) * (KT * 128) + rr * 128 + (rem & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            if (!o_seen && !wait_bounded(odone, (j - 1) & 1, p.status, p.wait_ns)) {
                *(volatile int*)abort_flag = 1;
                late_fail = true;           // acted on, uniformly, at the next tile's vote
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pfull[s]);
        }
        // the two halves of a row hold partial sums
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
        // ---- epilogue ----
        const bool got_last = (ok && n_t > 0) ? wait_bounded(odone, (n_t - 1) & 1, p.status, p.wait_ns) : true;
        if (named_bar_any(!got_last)) ok = false;
        tc_fence_after();
        if (!ok) *(volatile int*)abort_flag = 1;
        if (row_ok && half == 0) {
            l_s[r] = l_run;
            const float lse = (l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
            const size_t orow = ((size_t)b * p.s_q + qi) * p.H + h0 + r;
            if (it.part < 0) {
                if (p.lse) p.lse[orow] = lse;
            } else {
                p.lse_part[(size_t)it.part * p.s_q * p.H + (size_t)qi * p.H + h0 + r] = lse;
            }
        }
        named_bar_sync();
        const size_t orow0 = ((size_t)b * p.s_q + qi) * p.H + h0;
        float* dst_part = (it.part >= 0) ? p.o_part + ((size_t)it.part * p.s_q * p.H + (size_t)qi * p.H + h0) * DC
                                         : nullptr;
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
            const int dc = c * 128 + 32 * sub + lane;
            for (int c16 = 0; c16 < rows_o; c16 += 16) {
                uint32_t v[16];
                if (n_t > 0) {
                    tmem_ld16(tmem + LY::kColO + c * rows_o + c16 + lane_base, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) v[jj] = 0u;
                }
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int rr = c16 + jj;
                    const float l = l_s[rr];
                    const float val = (l > 0.f) ? __uint_as_float(v[jj]) / l : 0.f;
                    if (dst_part) {
                        dst_part[(size_t)rr * DC + dc] = val;
                    } else if (p.o_dtype == QKMLA_F32) {
                        ((float*)p.o)[(orow0 + rr) * DC + dc] = val;
                    } else {
                        ((__nv_bfloat16*)p.o)[(orow0 + rr) * DC + dc] = __float2bfloat16_rn(val);
                    }
                }
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// scheduler: seq_lens -> work items (one CTA)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
sched_kernel(const int32_t* __restrict__ seq_lens, int B, int s_q, int max_len, int n_rb, int sms, int min_tokens,
             int tile, int fixed_splits, WorkItem* __restrict__ items, int* __restrict__ n_items, int* __restrict__ seq_nsplit,
             int* __restrict__ seq_part0, int* __restrict__ split_list, int* status) {
    __shared__ int tiles_s[kMaxB];
    __shared__ int ns_by_rank[kMaxB];
    __shared__ int rank_s[kMaxB];
    __shared__ int red[32];
    __shared__ int s_total, s_tpi, s_nsplit;
    const int tid = threadIdx.x, nt = blockDim.x;
    pdl_wait();
    pdl_trigger();
    int tot = 0, mx = 0;
    for (int b = tid; b < B; b += nt) {
        const int L = seq_lens[b];
        int tl = 0;
        if (L < s_q || L > max_len) {
            report(status, QKMLA_ERR_DEVICE_BOUNDS);
        } else {
            tl = (L + tile - 1) / tile;
        }
        tiles_s[b] = tl;
        tot += tl;
        mx = max(mx, tl);
    }
    // block reductions (sum, max)
    for (int o = 16; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if ((tid & 31) == 0) red[tid >> 5] = tot;
    __syncthreads();
    if (tid == 0) {
        int t = 0;
        for (int w = 0; w < (nt + 31) / 32; ++w) t += red[w];
        s_total = t;
        s_nsplit = 0;
    }
    __syncthreads();
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    if (tid == 0) {
        int m = 0;
        for (int w = 0; w < (nt + 31) / 32; ++w) m = max(m, red[w]);
        // ideal tiles per CTA if the whole GPU shares the work evenly
        const float ideal = (float)s_total * n_rb / (float)sms;
        int tpi = (float)m <= 1.25f * ideal ? m : (int)ceilf(ideal);
        s_tpi = max(max(tpi, min_tokens / tile), 1);
    }
    __syncthreads();
    const int tpi = s_tpi;
    // rank sequences by descending tile count (longest first), ties by index
    for (int b = tid; b < B; b += nt) {
        const int tb = tiles_s[b];
        int rk = 0;
        for (int o = 0; o < B; ++o) {
            const int to = tiles_s[o];
            rk += (to > tb) || (to == tb && o < b);
        }
        rank_s[b] = rk;
        ns_by_rank[rk] = fixed_splits > 0 ? max(1, min(fixed_splits, tb)) : max(1, (tb + tpi - 1) / tpi);
    }
    __syncthreads();
    // exclusive prefix sum over ranks (single thread; B <= 4096)
    if (tid == 0) {
        int acc = 0;
        for (int k = 0; k < B; ++k) {
            const int v = ns_by_rank[k];
            ns_by_rank[k] = acc;
            acc += v;
        }
        *n_items = acc;
    }
    __syncthreads();
    for (int b = tid; b < B; b += nt) {
        const int tb = tiles_s[b];
        const int ns = fixed_splits > 0 ? max(1, min(fixed_splits, tb)) : max(1, (tb + tpi - 1) / tpi);
        const int per = (tb + ns - 1) / ns;
        const int off = ns_by_rank[rank_s[b]];
        seq_nsplit[b] = ns;
        seq_part0[b] = off;
        if (ns > 1) split_list[atomicAdd(&s_nsplit, 1)] = b;   // sequences the combine visits
        for (int k = 0; k < ns; ++k) {
            WorkItem w;
            w.b = b;
            w.tile_begin = k * per;
            w.tile_end = min(tb, (k + 1) * per);
            w.part = (ns > 1) ? off + k : -1;
            items[off + k] = w;
        }
    }
    __syncthreads();
    if (tid == 0) n_items[1] = s_nsplit;
}

// ---------------------------------------------------------------------------
// combine for variable split counts
// ---------------------------------------------------------------------------
// A fixed grid walks the rows of the split sequences: with none, every CTA exits
// after the dependency wait.  When the decode kernels planned the split
// themselves, the combine derives the same plan from seq_lens -- which the decode
// call does not write -- before its dependency wait, while the decode kernel
// still runs; otherwise it reads the scheduler kernel's compact list.
template <int VEC>
__global__ void __launch_bounds__(128)
combine_var_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                   const int* __restrict__ seq_nsplit, const int* __restrict__ seq_part0,
                   const int* __restrict__ split_list, const int* __restrict__ n_split,
                   const int32_t* __restrict__ seq_lens, int B, int s_q, SchedArgs sa, int sched_inline,
                   int rows_per_seq, void* __restrict__ o, int o_dtype, float* __restrict__ lse) {
    constexpr int kDc = 128 * VEC;              // thread t owns columns VEC t .. VEC t + VEC-1
    constexpr int kRegSplits = 16;              // partials held in registers per thread
    __shared__ float w_s[256];
    __shared__ float s_inv, s_lse;
    __shared__ SchedSmem S;
    if (sched_inline) compute_schedule(seq_lens, B, s_q, sa, S, nullptr, false);
    pdl_wait();
    pdl_trigger();
    const int tasks = (sched_inline ? S.n_split : *n_split) * rows_per_seq;
    const int tid = threadIdx.x;
    for (int task = blockIdx.x; task < tasks; task += gridDim.x) {
        const int sq = task / rows_per_seq, rr = task % rows_per_seq;
        const int b = sched_inline ? S.split[sq] : split_list[sq];
        const int row = b * rows_per_seq + rr;      // (b, i, h)
        const int ns = sched_inline ? S.ns[b] : seq_nsplit[b];
        const int p0 = sched_inline ? S.base[b] : seq_part0[b];
        __syncthreads();                            // w_s / s_inv of the previous task are read
        // every thread's loads of the first kRegSplits partials go out now, while
        // warp 0 turns the partial lse values into weights
        float v[kRegSplits][VEC];
#pragma unroll
        for (int u = 0; u < kRegSplits; ++u) {
            if (u < ns) {
                const float* src = o_part + ((size_t)(p0 + u) * rows_per_seq + rr) * kDc + VEC * tid;
                if constexpr (VEC == 4) {
                    const float4 x = __ldcg(reinterpret_cast<const float4*>(src));
                    v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
                } else {
                    const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
                    v[u][0] = x.x; v[u][1] = x.y;
                }
            }
        }
        if (tid < 32) {
            float m = -INFINITY;
            for (int s = tid; s < ns; s += 32) m = fmaxf(m, __ldcg(lse_part + (size_t)(p0 + s) * rows_per_seq + rr));
            m = warp_max(m);
            float sum = 0.f;
            for (int s = tid; s < ns; s += 32) {
                const float w =
                    (m == -INFINITY) ? 0.f : expf(__ldcg(lse_part + (size_t)(p0 + s) * rows_per_seq + rr) - m);
                w_s[s] = w;                         // ns <= 256
                sum += w;
            }
            sum = warp_sum(sum);
            if (tid == 0) {
                s_inv = sum > 0.f ? 1.f / sum : 0.f;
                s_lse = sum > 0.f ? m + logf(sum) : -INFINITY;
            }
        }
        __syncthreads();
        const float inv = s_inv;
        float acc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
        // a split with no tokens has weight 0 and contributes nothing
#pragma unroll
        for (int u = 0; u < kRegSplits; ++u) {
            const float w = u < ns ? w_s[u] : 0.f;
            if (w != 0.f) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
            }
        }
        for (int u = kRegSplits; u < ns; ++u) {
            const float w = w_s[u];
            if (w == 0.f) continue;
            const float* src = o_part + ((size_t)(p0 + u) * rows_per_seq + rr) * kDc + VEC * tid;
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[e] = fmaf(w, __ldcg(src + e), acc[e]);
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] *= inv;
        if (o_dtype == QKMLA_F32) {
            float* dst = (float*)o + (size_t)row * kDc + VEC * tid;
            if constexpr (VEC == 4) *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            else *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
        } else {
            __nv_bfloat16* dst = (__nv_bfloat16*)o + (size_t)row * kDc + VEC * tid;
            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0], acc[1]);
            if constexpr (VEC == 4) {
                const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2], acc[3]);
                uint2 pk;
                pk.x = *reinterpret_cast<const uint32_t*>(&lo);
                pk.y = *reinterpret_cast<const uint32_t*>(&hi);
                *reinterpret_cast<uint2*>(dst) = pk;
            } else {
                *reinterpret_cast<__nv_bfloat162*>(dst) = lo;
            }
        }
        if (tid == 0 && lse) lse[row] = s_lse;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int DC, int DR, bool PLAIN, int NST, bool AKH>
int launch_kernel(const CUtensorMap& lat, const CUtensorMap& rope, const CUtensorMap& qmap, const TcParams& tp,
                  int n_rb, int max_items, cudaStream_t s) {
    constexpr int KT = tile_of<DC>();
    using LY = Layout<DC, DR, NST, KT>;
    auto k = decode_tc_kernel<DC, DR, PLAIN, NST, KT, AKH>;
    static_assert(LY::kBytes <= 232448, "shared memory budget");
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes) != cudaSuccess)
        return QKMLA_ERR_CUDA;
    dim3 grid(n_rb, max_items);
    return launch_pdl(k, grid, dim3(kThreads), LY::kBytes, s, lat, rope, qmap, tp) == cudaSuccess ? QKMLA_OK
                                                                                         : QKMLA_ERR_CUDA;
}

}  // namespace

namespace dec {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    }
    return fn;
}

bool make_map(CUtensorMap* m, const void* base, int64_t rows, int row_elems, int box_cols, int box_rows,
              CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_elems * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dec

// The two-CTA cluster kernel: DeepSeek-V3 decode shape, 128 heads per query token.
bool pair_shape(const qkmla_decode_args* a) {
    return a->d_c == 512 && a->d_r == 64 && a->H == 128 && a->page_size % 64 == 0;
}

// Batches whose split plan every decode CTA computes itself (no scheduler launch).
bool sched_in_kernel(const qkmla_decode_args* a) { return a->B >= 1 && a->B <= dec::kMaxBSched; }

// Query rows per CTA of the 64-row kernel.  With fewer than 64 heads it packs k
// query tokens of a sequence (k dividing s_q), so that a CTA streams each tile
// once for all of them, while k H stays within the 64 MMA rows and, for d_c =
// 512, within the RoPE slot that P^T reuses there (k H <= d_r).
int tc_rows(const qkmla_decode_args* a) {
    if (a->H >= 64) return 64;
    const int cap = (a->d_c == 256 || a->d_r >= 64) ? 64 : a->d_r;
    int rows = a->H;
    for (int k = 2; k <= a->s_q; ++k)
        if (a->s_q % k == 0 && a->H * k <= cap && (a->H * k) % 16 == 0) rows = a->H * k;
    return rows;
}

// Shapes the tensor-core kernel is built for (bf16 cache).
bool tc_supported(const qkmla_decode_args* a) {
    if (a->cache_dtype != QKMLA_BF16) return false;
    if (!((a->d_c == 512 && a->d_r == 64) || (a->d_c == 256 && a->d_r == 32))) return false;
    if (a->G > kMaxG || a->B > kMaxB) return false;
    // a tile (64 tokens for d_c = 256, 32 for d_c = 512) never straddles a page
    if (a->page_size % (a->d_c == 256 ? 64 : 32)) return false;
    const int rows_o = a->H < 64 ? a->H : 64;
    if (rows_o % 16 || a->H % rows_o) return false;
    if (a->d_c != 256 && rows_o > a->d_r) return false;   // P^T (rows_o x tile tokens) reuses the RoPE slot
    if (((uintptr_t)a->kv_cache % 16) || ((uintptr_t)a->q_tilde % 16) || ((uintptr_t)a->o % 16)) return false;
    if (!(a->flags & QKMLA_FLAG_PLAIN_MLA) && ((uintptr_t)a->ak_cache % 16)) return false;
    return true;
}

size_t tc_workspace(const qkmla_decode_args* a, int sms, int* max_items_out) {
    const int rows_o = pair_shape(a) ? 64 : tc_rows(a);
    const int n_rb = a->s_q * a->H / rows_o;
    const int target = (sms + n_rb - 1) / n_rb;
    int max_items = a->B + target + 1;
    if (a->num_splits > 0) max_items = a->B * a->num_splits;
    if (max_items_out) *max_items_out = max_items;
    size_t off = 0;
    off += (size_t)max_items * sizeof(WorkItem);
    off += 16 + 3 * (size_t)a->B * sizeof(int);
    off = (off + 255) & ~(size_t)255;
    off += (size_t)max_items * a->s_q * a->H * a->d_c * sizeof(float);
    off += (size_t)max_items * a->s_q * a->H * sizeof(float);
    return off + 256;
}

int launch_decode_tc(const qkmla_decode_args* a, const DecodePlan& plan, cudaStream_t s) {
    const int sms = device_sm_count();
    int max_items = 0;
    tc_workspace(a, sms, &max_items);
    const int rows_o = pair_shape(a) ? 64 : tc_rows(a);
    const int n_rb = a->s_q * a->H / rows_o;
    uint8_t* ws = (uint8_t*)a->workspace;
    WorkItem* items = (WorkItem*)ws;
    size_t off = (size_t)max_items * sizeof(WorkItem);
    int* n_items = (int*)(ws + off);
    int* seq_nsplit = n_items + 4;
    int* seq_part0 = seq_nsplit + a->B;
    int* split_list = seq_part0 + a->B;
    off += 16 + 3 * (size_t)a->B * sizeof(int);
    off = (off + 255) & ~(size_t)255;
    float* o_part = (float*)(ws + off);
    float* lse_part = o_part + (size_t)max_items * a->s_q * a->H * a->d_c;
    int* status = device_status_ptr();
    const int max_len = a->max_pages * a->page_size;

    const int tile = pair_shape(a) ? 64 : a->d_c == 256 ? tile_of<256>() : tile_of<512>();
    const int box = tile;
    SchedArgs sa;
    sa.max_len = max_len;
    sa.n_rb = n_rb;
    sa.sms = sms;
    sa.min_tokens = 512;
    sa.tile = tile;
    sa.fixed_splits = a->num_splits;
    // small batches: the decode and combine kernels plan the split themselves
    const int sched_inline = sched_in_kernel(a) ? 1 : 0;
    if (!sched_inline &&
        launch_pdl(sched_kernel, dim3(1), dim3(1024), 0, s, a->seq_lens, a->B, a->s_q, max_len, n_rb, sms,
                   sa.min_tokens, tile, a->num_splits, items, n_items, seq_nsplit, seq_part0, split_list, status) !=
            cudaSuccess)
        return QKMLA_ERR_CUDA;

    CUtensorMap lat, rope;
    const int row = a->d_c + a->d_r;
    if (!make_map(&lat, a->kv_cache, a->num_slots, row, 64, box, CU_TENSOR_MAP_SWIZZLE_128B)) return QKMLA_ERR_CUDA;
    if (a->d_r == 64) {
        rope = lat;
    } else if (!make_map(&rope, a->kv_cache, a->num_slots, row, 32, box, CU_TENSOR_MAP_SWIZZLE_64B)) {
        return QKMLA_ERR_CUDA;
    }
    CUtensorMap qmap;
    if (!pair_shape(a) && !make_map(&qmap, a->q_tilde, (int64_t)a->B * a->s_q * a->H, a->d_c, 64, rows_o,
                                    CU_TENSOR_MAP_SWIZZLE_128B))
        return QKMLA_ERR_CUDA;
    TcParams tp;
    tp.qt = (const __nv_bfloat16*)a->q_tilde;
    tp.aq = a->alpha_q;
    tp.qr = a->q_rope;
    tp.grq = a->gamma_rope_q;
    tp.ak = a->ak_cache;
    tp.seq_lens = a->seq_lens;
    tp.page_table = a->page_table;
    tp.num_pages = a->num_slots / a->page_size;
    tp.page_size = a->page_size;
    tp.max_pages = a->max_pages;
    tp.B = a->B; tp.s_q = a->s_q; tp.H = a->H; tp.G = a->G;
    tp.rows_o = rows_o;
    tp.scale = a->softmax_scale;
    tp.eps = a->eps;
    tp.items = items;
    tp.n_items = n_items;
    tp.sa = sa;
    tp.sched_inline = sched_inline;
    tp.o_part = o_part;
    tp.lse_part = lse_part;
    tp.o = a->o;
    tp.o_dtype = a->o_dtype;
    tp.lse = a->lse;
    tp.status = status;
    // test hook: withhold the second tile and give up waiting after 1 ms (64-row kernel only;
    // plan_decode rejects the flag for the other kernels)
    const bool stall = (a->flags & QKMLA_FLAG_TEST_STALL) != 0;
    tp.wait_ns = stall ? 1000000ull : kWaitNs;
    tp.withhold_tile = stall ? 1 : -1;
    tp.zero = 0;
    const bool plain = (a->flags & QKMLA_FLAG_PLAIN_MLA) != 0;
    const bool akh = !plain && (a->flags & QKMLA_FLAG_ALPHA_F16) != 0;
    int rc;
    if (pair_shape(a)) {
        rc = launch_pair(a, tp, max_items, s);
    } else if (a->d_c == 512) {
        rc = plain ? launch_kernel<512, 64, true, 4, false>(lat, rope, qmap, tp, n_rb, max_items, s)
             : akh ? launch_kernel<512, 64, false, 4, true>(lat, rope, qmap, tp, n_rb, max_items, s)
                   : launch_kernel<512, 64, false, 4, false>(lat, rope, qmap, tp, n_rb, max_items, s);
    } else {
        rc = plain ? launch_kernel<256, 32, true, 4, false>(lat, rope, qmap, tp, n_rb, max_items, s)
             : akh ? launch_kernel<256, 32, false, 4, true>(lat, rope, qmap, tp, n_rb, max_items, s)
                   : launch_kernel<256, 32, false, 4, false>(lat, rope, qmap, tp, n_rb, max_items, s);
    }
    if (rc != QKMLA_OK) return rc;
    // one CTA per merged row where few sequences make few, long, split rows (every
    // CTA computes the plan, so many CTAs cost more than they give on large batches)
    const int combine_ctas = std::min(a->B * a->s_q * a->H, (a->B <= 32 ? 8 : 2) * sms);
    auto ck = a->d_c == 512 ? combine_var_kernel<4> : combine_var_kernel<2>;   // d_c = 128 x VEC
    return launch_pdl(ck, dim3(combine_ctas), dim3(128), 0, s, (const float*)o_part, (const float*)lse_part,
                      (const int*)seq_nsplit, (const int*)seq_part0, (const int*)split_list,
                      (const int*)(n_items + 1), a->seq_lens, a->B, a->s_q, sa, sched_inline, a->s_q * a->H, a->o,
                      a->o_dtype, a->lse) == cudaSuccess
               ? QKMLA_OK
               : QKMLA_ERR_CUDA;
}

}  // namespace qkmla
