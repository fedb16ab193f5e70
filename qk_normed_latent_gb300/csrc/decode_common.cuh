// Device helpers shared by the tensor-core decode kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace qkmla {
namespace dec {

using namespace tc;

constexpr int kMaxG = 8;
constexpr int kMaxB = 4096;
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s bound on any single wait

struct WorkItem {
    int b;
    int tile_begin;
    int tile_end;
    int part;          // -1: the item is the whole sequence, write the final row
};

// Parameters of the split-KV schedule (see decode_sched.cuh).
struct SchedArgs {
    int max_len, n_rb, sms, min_tokens, tile, fixed_splits;
};

struct TcParams {
    const __nv_bfloat16* qt;   // [B][s_q][H][d_c]
    const float* aq;           // [B][s_q][H]
    const float* qr;           // [B][s_q][H][d_r]
    const float* grq;          // [d_r] or null
    const void* ak;            // [num_slots][G] fp32 or fp16 (the kernels' AKH template flag)
    const int32_t* seq_lens;
    const int32_t* page_table;
    int64_t num_pages;
    int page_size, max_pages;
    int B, s_q, H, G;
    int rows_o;                // query rows per CTA (N of the output MMA)
    float scale, eps;
    const WorkItem* items;     // scheduler kernel's plan (when sched_inline == 0)
    const int* n_items;
    SchedArgs sa;
    int sched_inline;          // 1: every CTA computes the plan from seq_lens itself
    float* o_part;             // [max_items][s_q*H][d_c]
    float* lse_part;           // [max_items][s_q*H]
    void* o;
    int o_dtype;
    float* lse;
    int* status;
    uint64_t wait_ns;          // bound on any single wait (64-row kernel)
    int withhold_tile;         // test hook (64-row kernel): the producer issues no tile from this one on; -1 off
    uint32_t zero;             // always 0, unknown to the compiler: masks data dependencies into addresses
};

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Packed fp32 pairs (f32x2 arithmetic, sm_100 and later): one instruction does the
// work of two, each element rounded exactly as the scalar round-to-nearest
// operation would round it (no flush to zero, like the scalar code here).
__device__ __forceinline__ uint64_t f2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// c + (the two fp16 halves of w), each as one mixed-precision add (the half is
// converted exactly, the sum rounded once: the same bits as converting first).
__device__ __forceinline__ float2 half2_plus(uint32_t w, float c) {
    float2 r;
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.f16 %0, lo, %3;\n\tadd.rn.f32.f16 %1, hi, %3;\n\t}"
        : "=f"(r.x), "=f"(r.y) : "r"(w), "f"(c));
    return r;
}
// Three-input maximum (one instruction on sm_100 and later); exact, like fmaxf.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// Bounded wait: spins on try_wait, checks the wall clock every 256 polls and
// gives up (recording QKMLA_ERR_TIMEOUT) after limit_ns.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, int* status,
                                             uint64_t limit_ns = kWaitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && globaltimer() - t0 > limit_ns) {
            report(status, QKMLA_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ bool named_bar_any(int pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(pred)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void named_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// 2^x with the hardware approximation (ex2.approx.ftz); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16 lanes x 32 bit x 16 columns, two halves: lanes 0-15 of the warp read TMEM
// lanes base..base+15 at columns c..c+15, lanes 16-31 the same TMEM lanes at
// columns c+16..c+31.
__device__ __forceinline__ void tmem_ld16x2(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], 16;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}


// ---------------------------------------------------------------------------
// thread-block clusters: rank, distributed shared memory, remote signalling
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
// Bounded wait with cluster-scope acquire (data written by the other CTA).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool wait_bounded_cluster(uint64_t* bar, uint32_t parity, int* status) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((i & 255u) == 0 && globaltimer() - t0 > kWaitNs) {
            report(status, QKMLA_ERR_TIMEOUT);
            return false;
        }
    }
}
// Bulk copy from this CTA's shared memory into another CTA's (of the cluster),
// completing `bytes` on the mbarrier `remote_bar` there.
__device__ __forceinline__ void bulk_copy_to_cta(uint32_t remote_dst, const void* local_src, uint32_t bytes,
                                                 uint32_t remote_bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(remote_dst), "r"(smem_u32(local_src)), "r"(bytes), "r"(remote_bar)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk copy has finished READING its source.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until every committed bulk copy has completed (its writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Remote arrive ordered after this thread's earlier READS of the rows the other
// CTA will overwrite, without a release fence (a release at cluster scope costs
// ~10 % of the pair kernel).  `dep` is computed from every value those reads
// returned; masked with `zero` (a kernel argument that is always 0, so no
// compiler pass can drop it) and added to the barrier address, it makes the
// arrive's own operand depend on every read: the arrive cannot issue before
// they have returned their values, after which a remote write cannot change them.
// (An operand the arrive does not consume is dead code to the assembler, which
// then may issue the arrive ahead of the reads.)
__device__ __forceinline__ void mbar_arrive_remote_after(uint32_t remote_bar, uint32_t dep, uint32_t zero) {
    asm volatile("{\n\t.reg .b32 t, a;\n\t"
                 "and.b32 t, %1, %2;\n\t"
                 "add.u32 a, %0, t;\n\t"
                 "mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [a];\n\t}"
                 ::"r"(remote_bar), "r"(dep), "r"(zero) : "memory");
}
// Cluster-wide barrier (all threads of every CTA of the cluster).  The
// non-aligned form: callers may arrive from diverged code paths.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Host side, shared by the launchers.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();   // the driver's tensor-map encoder (nullptr if absent)
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int row_elems, int box_cols, int box_rows,
              CUtensorMapSwizzle sw);
int launch_pair(const qkmla_decode_args* a, const TcParams& tp, int max_items, cudaStream_t s);
}  // namespace dec
bool pair_shape(const qkmla_decode_args* a);
namespace dec {

}  // namespace dec
}  // namespace qkmla
