// Split-KV schedule computed inside the kernels that need it (decode, combine).
//
// Every CTA derives the same plan from seq_lens, so no separate scheduler launch
// (and no kernel boundary) sits between the previous kernel and the decode:
//   * tiles per sequence tb_b = ceil(L_b / tile);
//   * tiles per work item tpi: the longest sequence when that is within 25 % of
//     an even share of the GPU (s_total * n_rb / sms), else that share rounded
//     up; at least min_tokens worth of tiles;
//   * a sequence splits into ns_b = ceil(tb_b / tpi) items (or the caller's
//     fixed split count), of per = ceil(tb_b / ns_b) tiles each;
//   * items are numbered by sequence, longest first (ties by index), so the
//     work that bounds the tail starts first; an item's index is also the index
//     of its partial output when its sequence is split.
// Ranking costs B^2 / threads comparisons, so this path serves batches of up to
// kMaxBSched sequences; larger batches use the scheduler kernel.
#pragma once

#include "decode_common.cuh"

namespace qkmla {
namespace dec {

constexpr int kMaxBSched = 128;

struct SchedSmem {
    int len[kMaxBSched];       // seq_lens[b] as read
    int tb[kMaxBSched];        // tiles of sequence b
    int ns[kMaxBSched];        // items of sequence b
    int base[kMaxBSched];      // first item of sequence b
    int by_rank[kMaxBSched];   // sequence at rank k
    int split[kMaxBSched];     // the split sequences (ns > 1), in rank order
    int red[32];
    int n_items, n_split, tpi;
};

// Block-wide: every thread of the CTA calls it; on return `S` holds the plan.
// Sequences with an invalid length get no tiles (and a status report when
// `report_errors`).
__device__ __forceinline__ void compute_schedule(const int32_t* __restrict__ seq_lens, int B, int s_q,
                                                 const SchedArgs& a, SchedSmem& S, int* status, bool report_errors) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = (nt + 31) >> 5;
    int tot = 0, mx = 0;
    for (int b = tid; b < B; b += nt) {
        const int L = __ldcg(seq_lens + b);   // through L2: the lengths may change between calls
        S.len[b] = L;
        int tl = 0;
        if (L < s_q || L > a.max_len) {
            if (report_errors) report(status, QKMLA_ERR_DEVICE_BOUNDS);
        } else {
            tl = (L + a.tile - 1) / a.tile;
        }
        S.tb[b] = tl;
        tot += tl;
        mx = max(mx, tl);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) S.red[warp] = tot;
    __syncthreads();
    if (tid == 0) {
        int t = 0;
        for (int w = 0; w < nw; ++w) t += S.red[w];
        S.n_items = t;                       // s_total for now
    }
    __syncthreads();
    if (lane == 0) S.red[warp] = mx;
    __syncthreads();
    if (tid == 0) {
        int m = 0;
        for (int w = 0; w < nw; ++w) m = max(m, S.red[w]);
        const float ideal = (float)S.n_items * a.n_rb / (float)a.sms;
        const int tpi = (float)m <= 1.25f * ideal ? m : (int)ceilf(ideal);
        S.tpi = max(max(tpi, a.min_tokens / a.tile), 1);
    }
    __syncthreads();
    const int tpi = S.tpi;
    for (int b = tid; b < B; b += nt) {
        const int tb = S.tb[b];
        int rk = 0;
        for (int o = 0; o < B; ++o) {
            const int to = S.tb[o];
            rk += (to > tb) || (to == tb && o < b);
        }
        S.by_rank[rk] = b;
        S.ns[b] = a.fixed_splits > 0 ? max(1, min(a.fixed_splits, tb)) : max(1, (tb + tpi - 1) / tpi);
    }
    __syncthreads();
    // exclusive prefix of the item counts in rank order (one warp, B <= 128: four ranks a lane)
    if (warp == 0) {
        int v[kMaxBSched / 32], sp[kMaxBSched / 32];
        int run = 0, nsp = 0;
#pragma unroll
        for (int i = 0; i < kMaxBSched / 32; ++i) {
            const int k = lane * (kMaxBSched / 32) + i;
            v[i] = k < B ? S.ns[S.by_rank[k]] : 0;
            sp[i] = (k < B && v[i] > 1) ? 1 : 0;
            run += v[i];
            nsp += sp[i];
        }
        int incl = run, incl_sp = nsp;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            const int y = __shfl_up_sync(0xffffffffu, incl_sp, o);
            if (lane >= o) { incl += x; incl_sp += y; }
        }
        int acc = incl - run, acc_sp = incl_sp - nsp;
#pragma unroll
        for (int i = 0; i < kMaxBSched / 32; ++i) {
            const int k = lane * (kMaxBSched / 32) + i;
            if (k < B) {
                const int b = S.by_rank[k];
                S.base[b] = acc;
                if (sp[i]) S.split[acc_sp] = b;
                acc += v[i];
            }
            acc_sp += sp[i];
        }
        if (lane == 31) {
            S.n_items = incl;
            S.n_split = incl_sp;
        }
    }
    __syncthreads();
}

// The work item `item` of the plan in `S` (item < S.n_items).
__device__ __forceinline__ WorkItem schedule_item(const SchedSmem& S, int B, int item) {
    // the rank whose items contain `item`: bases are increasing in rank order
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (S.base[S.by_rank[mid]] <= item) lo = mid; else hi = mid - 1;
    }
    const int b = S.by_rank[lo];
    const int ns = S.ns[b], tb = S.tb[b];
    const int k = item - S.base[b];
    const int per = (tb + ns - 1) / ns;
    WorkItem w;
    w.b = b;
    w.tile_begin = k * per;
    w.tile_end = min(tb, (k + 1) * per);
    w.part = ns > 1 ? item : -1;
    return w;
}

}  // namespace dec
}  // namespace qkmla
