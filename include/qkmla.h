/*
 * qkmla.h -- C ABI of the QK-Normed MLA decode library (GB300, sm_103a).
 *
 * The method (arXiv 2606.16310, "QK-Normed MLA: QK normalization without full
 * key caching"; gist.science Technical Summary, Methodology) splits
 * post-projection RMSNorm(z) = z * gamma / S(z) into a static weight and a
 * dynamic scalar.  The static key weight gamma_k (with gamma_q) is absorbed
 * into the query; the dynamic key statistic is cached as one inverse-RMS
 * scalar alpha^k per token and KV group next to the MLA latent c_t; decode
 * computes the row/column-scaled logit
 *
 *     l_{i,t,h} = scale * ( alpha^q_{i,h} * alpha^k_{t,g(h)} * (q~_{i,h} . c_t)
 *                           + q^rope_{i,h} . k^rope_t )
 *
 * then a softmax over t and the latent-space output o = sum_t p_t c_t.
 *
 * Three calls form the decode path: qkmla_absorb_query, qkmla_append,
 * qkmla_decode.  Conventions shared by every call:
 *
 *  - All array pointers are DEVICE pointers owned by the caller; the library
 *    keeps no reference after the call returns.  `stream` is a cudaStream_t
 *    (NULL = legacy default stream).  Calls are asynchronous on that stream.
 *  - Host-side validation (null pointers, sizes, dtypes, alignment) returns an
 *    error code before anything is launched.  Launch failures return
 *    QKMLA_ERR_CUDA.  Problems that only the device can see (an out-of-range
 *    page id, a sequence length outside its bounds, an expired bounded wait)
 *    never trap: the kernel skips the offending work and records the first
 *    such error in a per-device status word read by qkmla_get_device_status().
 *  - Shapes: B sequences, s_q query tokens per sequence in this step
 *    (rows = B*s_q), H query heads, G KV groups with g(h) = h / (H/G),
 *    d_h head dim of the content (nope) part, d_c latent dim, d_r RoPE dim.
 *  - Cache: one flat array of slots.  kv_cache[slot] = [c_t (d_c) | k^rope_t
 *    (d_r)] in the cache dtype; ak_cache[slot] = [alpha^k_{t,0..G-1}] fp32
 *    (fp16 with QKMLA_FLAG_ALPHA_F16).
 *    Token t of sequence b lives in slot
 *        page_table[b*max_pages + t/page_size]*page_size + t%page_size,
 *    and with page_table == NULL in slot (b*max_pages + t/page_size)*page_size
 *    + t%page_size (a contiguous cache of max_pages*page_size slots per
 *    sequence).
 *  - The library is stateless apart from the status word and a small per-
 *    device table of launch limits; it is thread-safe.
 *  - Every kernel is launched with programmatic stream serialization and lets
 *    the next kernel of the stream launch early.  Its writes, and its reads of
 *    anything a kernel of this library produces (q~, alpha^q, the cache, q and
 *    q_rope of qkmla_project_query, o), wait for the previous kernel of the
 *    stream.  Reads of inputs no kernel of the library writes may start
 *    earlier: seq_lens in qkmla_decode; W^K, the new tokens, their slots and
 *    positions in qkmla_append / qkmla_append_rope.  A previous kernel that
 *    itself signals early dependent launch must therefore not be writing
 *    those inputs (kernels that do not signal it, and copies, are waited for
 *    in full as usual).
 */
#ifndef QKMLA_H
#define QKMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
enum {
    QKMLA_OK = 0,
    QKMLA_ERR_INVALID = -1,       /* bad argument: null pointer, size, alignment */
    QKMLA_ERR_UNSUPPORTED = -2,   /* valid but not built (dtype / dims combination) */
    QKMLA_ERR_CUDA = -3,          /* a CUDA runtime/driver call failed */
    QKMLA_ERR_WORKSPACE = -4,     /* workspace missing or smaller than required */
    QKMLA_ERR_DEVICE_BOUNDS = -5, /* device saw a page id / length out of range */
    QKMLA_ERR_TIMEOUT = -6        /* device bounded wait expired */
};

/* Element types. */
enum { QKMLA_F32 = 0, QKMLA_BF16 = 1 };

/* Flags. */
enum {
    /* Plain MLA (the comparator without QK normalisation): absorb writes
     * q~ = W^K_g q and alpha^q = 1; append stores the raw RoPE key and
     * alpha^k = 1; decode uses l = scale * (q~ . c_t + q_rope . k^rope_t). */
    QKMLA_FLAG_PLAIN_MLA = 1u,
    /* Decode: force the CUDA-core (SIMT) kernel even where the tensor-core
     * kernel applies.  Used to cross-check the two kernels. */
    QKMLA_FLAG_FORCE_SIMT = 2u,
    /* Decode, test hook for the failure path: the 64-row tensor-core kernel's
     * loader issues no tile from the second one on and every wait gives up
     * after 1 ms, so a call whose sequences span two or more tiles ends with
     * QKMLA_ERR_TIMEOUT in the status word (outputs undefined) and leaves the
     * context usable.  QKMLA_ERR_UNSUPPORTED for arguments that select another
     * kernel.  Never set outside tests. */
    QKMLA_FLAG_TEST_STALL = 4u,
    /* Append and decode: A^k_cache holds IEEE half-precision scalars
     * ([num_slots][G], 2 bytes each, round-to-nearest-even of the fp32
     * alpha^k) instead of fp32.  Halves the scalar cache, the method's only
     * storage overhead over MLA (Technical Summary, Key Contributions and
     * Results).  alpha^k = 1/sqrt(mean k^2 + eps) stays in fp16's normal range
     * (6.1e-5 .. 65504) for key RMS up to ~16000 and eps down to 2.3e-10; 11
     * significant bits keep each content logit within 2^-11 of its fp32 value.
     * Ignored with QKMLA_FLAG_PLAIN_MLA. */
    QKMLA_FLAG_ALPHA_F16 = 8u
};

/*
 * qkmla_absorb_query -- query side of the absorbed formulation.
 * Source: Technical Summary, Methodology, "Static Weight Absorption" (gamma_k
 * and gamma_q pre-multiply the query before the latent dot product) and the
 * decode-logit equation (alpha^q_{i,h} is the query's inverse RMS).
 *
 *   alpha_q[r][h]    = 1 / sqrt(mean_j q[r][h][j]^2 + eps)
 *   q_tilde[r][h][n] = sum_j W^K[g(h)][n][j] * q[r][h][j] * gamma_q[j] * gamma_k[j]
 *
 * q        [rows][H][d_h] fp32          gamma_q, gamma_k [d_h] fp32
 * w_k      [G][d_c][d_h]  fp32 (k_{t,g} = c_t W^K_g, i.e. W^K_g is d_c x d_h)
 * q_tilde  [rows][H][d_c] in qt_dtype (QKMLA_F32 or QKMLA_BF16, RNE cast)
 * alpha_q  [rows][H] fp32
 * PLAIN_MLA: gamma_* are ignored (may be NULL), alpha_q = 1.
 * Errors: INVALID for null pointers or non-positive sizes, H % G != 0,
 * d_h > 256 or d_c % 8 != 0; UNSUPPORTED for another qt_dtype.
 */
int qkmla_absorb_query(const float* q, const float* gamma_q, const float* gamma_k,
                       const float* w_k, int rows, int H, int G, int d_h, int d_c,
                       float eps, unsigned flags, void* q_tilde, int qt_dtype,
                       float* alpha_q, void* stream);

/*
 * qkmla_append -- write new tokens into the latent cache and A^k_cache.
 * Source: Technical Summary, Methodology, "Dynamic Scalar Caching" (one
 * inverse-RMS scalar per token and KV group), "Cache Layout" (keep c_t, add
 * the scalar cache, never store full keys) and "Blockwise Normalization"
 * (the RoPE part is normalised separately, as a materialised vector).
 *
 * For each new token n with slot s = slot_mapping[n] (s < 0: skipped):
 *   kv[s][0:d_c]   = cast(c_new[n])                       (bit-exact RNE cast)
 *   ak[s][g]       = 1 / sqrt(mean_j (c^ W^K_g)_j^2 + eps)  with c^ the stored latent
 *   kv[s][d_c:]    = cast(k_rope_new[n] * gamma_rope_k * beta_n),
 *                    beta_n = 1 / sqrt(mean_j k_rope_new[n][j]^2 + eps)
 * c_new [N][d_c] fp32, k_rope_new [N][d_r] fp32 (post-RoPE), w_k as above,
 * gamma_rope_k [d_r] fp32 or NULL (ones), slot_mapping [N] int64 device.
 * kv_cache [num_slots][d_c+d_r] in cache_dtype, ak_cache [num_slots][G] fp32
 * (fp16, the RNE cast of the fp32 value, with QKMLA_FLAG_ALPHA_F16).
 * PLAIN_MLA: the raw RoPE key is stored and ak = 1.
 * A slot >= num_slots is a device-side bounds error (skipped, status set).
 * N == 0 is a no-op.  Errors: INVALID / UNSUPPORTED as for absorb; d_h <= 256.
 */
int qkmla_append(const float* c_new, const float* k_rope_new, const float* w_k,
                 const float* gamma_rope_k, const int64_t* slot_mapping, int N, int G,
                 int d_c, int d_h, int d_r, float eps, unsigned flags, void* kv_cache,
                 int cache_dtype, void* ak_cache, int64_t num_slots, void* stream);

/*
 * qkmla_append_rope -- qkmla_append for RoPE keys that are not yet rotated:
 * each new token's RoPE key is first rotated by its position, then normalised
 * and stored exactly as qkmla_append stores a post-RoPE key.
 * Source: as qkmla_append, and Technical Summary, Methodology, "Blockwise
 * Normalization" (the RoPE part is a materialised vector normalised on its
 * own; the normalised vector is the rotated one).
 *
 * Rotation (the original rotary formulation; the pages name none): interleaved
 * pairs (x_2i, x_2i+1) of the d_r-vector turn by positions[n] * rope_theta^(-2i/d_r).
 * Angles are reduced exactly enough for positions up to 2^24 (fp64 frequency,
 * error-free fp32 product, two-part 2*pi reduction).
 * k_rope_raw [N][d_r] fp32 (before rotation); positions [N] int32 device.
 * Errors: as qkmla_append, and INVALID for a missing positions array, d_r odd
 * or rope_theta <= 1; UNSUPPORTED for d_r > 64.
 */
int qkmla_append_rope(const float* c_new, const float* k_rope_raw, const int32_t* positions, float rope_theta,
                      const float* w_k, const float* gamma_rope_k, const int64_t* slot_mapping, int N, int G,
                      int d_c, int d_h, int d_r, float eps, unsigned flags, void* kv_cache, int cache_dtype,
                      void* ak_cache, int64_t num_slots, void* stream);

/*
 * qkmla_project_query -- the query projection ahead of qkmla_absorb_query,
 * with the RoPE rotation of the RoPE block fused in.
 * Source: thelatestinai.com abstract (the static key weight is absorbed into
 * the MLA query-side projection: the query comes from the layer input through
 * W^Q, then qkmla_absorb_query folds gamma_q * gamma_k and W^K_g into it);
 * Technical Summary, Methodology, "Blockwise Normalization".
 *
 *   [q_h | r_h] = x W^Q_h^T,  q[r][h] = q_h,  q_rope[r][h] = RoPE(r_h, positions[r])
 *
 * x [rows][d_x] bf16; w_q [H][d_h + d_r][d_x] bf16 (row j of W^Q_h holds output
 * j's weights: the d_h content outputs, then the d_r RoPE outputs);
 * positions [rows] int32 device (RoPE position of each query row);
 * q [rows][H][d_h] fp32 (qkmla_absorb_query's input); q_rope [rows][H][d_r]
 * fp32, rotated as in qkmla_append_rope, not normalised (qkmla_decode's input).
 * Tensor cores, fp32 accumulation.  Errors: INVALID for null pointers, bad
 * sizes or alignment, rope_theta <= 1 with d_r > 0; UNSUPPORTED for d_x % 64,
 * odd d_h or d_r, d_r > 64, or d_h + d_r not in {96, 128, 160, 192, 256}.
 */
int qkmla_project_query(const void* x, const void* w_q, const int32_t* positions, float rope_theta, int rows,
                        int d_x, int H, int d_h, int d_r, float* q, float* q_rope, void* stream);

/* Arguments of qkmla_decode (plain pointers and sizes). */
typedef struct qkmla_decode_args {
    const void* q_tilde;        /* [B][s_q][H][d_c] in cache_dtype (from absorb) */
    const float* alpha_q;       /* [B][s_q][H] fp32 */
    const float* q_rope;        /* [B][s_q][H][d_r] fp32, post-RoPE, not normalised */
    const float* gamma_rope_q;  /* [d_r] fp32 or NULL (ones) */
    const void* kv_cache;       /* [num_slots][d_c+d_r] cache_dtype */
    const void* ak_cache;       /* [num_slots][G] fp32 (fp16 with QKMLA_FLAG_ALPHA_F16) */
    const int32_t* seq_lens;    /* [B] int32 device: tokens in the cache incl. this step's s_q */
    const int32_t* page_table;  /* [B][max_pages] int32 device, or NULL (contiguous) */
    int64_t num_slots;          /* slots in kv_cache / ak_cache (multiple of page_size) */
    int page_size;              /* tokens per page (> 0) */
    int max_pages;              /* page-table row length; max tokens = max_pages*page_size */
    int B, s_q, H, G, d_c, d_r;
    int cache_dtype;            /* QKMLA_F32 or QKMLA_BF16 */
    float softmax_scale;        /* multiplies the whole logit, e.g. 1/sqrt(d_h+d_r) */
    float eps;                  /* RMS epsilon of the RoPE query normalisation */
    unsigned flags;             /* QKMLA_FLAG_* */
    int num_splits;             /* 0: automatic; k >= 1: k equal token ranges per sequence */
    void* workspace;            /* device scratch, >= qkmla_decode_workspace_size(args) bytes */
    size_t workspace_bytes;
    void* o;                    /* [B][s_q][H][d_c] output in o_dtype */
    int o_dtype;                /* QKMLA_F32 or QKMLA_BF16 */
    float* lse;                 /* [B][s_q][H] fp32: natural log of sum_t exp(l_t); may be NULL */
} qkmla_decode_args;

/*
 * qkmla_decode_workspace_size -- bytes of device scratch qkmla_decode needs
 * for these arguments (split-KV partial outputs and scheduler metadata).  Only
 * the shape fields, flags, cache_dtype and num_splits are read.  Returns 0 for
 * arguments qkmla_decode would reject.  Depends on the current device.
 */
size_t qkmla_decode_workspace_size(const qkmla_decode_args* a);

/*
 * qkmla_decode -- QK-Normed MLA decode attention over the latent cache.
 * Source: Technical Summary, Methodology, decode-logit equation (row scaling
 * by alpha^q, column scaling by alpha^k, before the softmax) and "Blockwise
 * Normalization" (the RoPE logit uses materialised normalised vectors); the
 * abstract's "preserves MLA's latent decode path" (values are the latents).
 *
 * Query i of sequence b attends to tokens t < seq_lens[b] - s_q + i + 1.
 * q^rope = q_rope * gamma_rope_q / sqrt(mean(q_rope^2) + eps) per head.
 * o[b][i][h] = sum_t p_t c_t with p = softmax_t(l); lse = log sum_t exp(l_t).
 * Long contexts are split over CTAs (split-KV) and merged by a combine kernel.
 * Errors: INVALID (null pointer, bad dims, H % G, d_c % 64 for bf16, ...),
 * UNSUPPORTED (heads per group H / G other than 1, 2, 4, 8 or 16; d_c > 512
 * or d_r > 128; a cache or output dtype other than fp32 / bf16), WORKSPACE
 * (workspace smaller than required).  Device-side:
 * seq_len < s_q or > max_pages*page_size, or a page id outside
 * [0, num_slots/page_size), set QKMLA_ERR_DEVICE_BOUNDS; the sequence's
 * affected rows are then undefined.
 */
int qkmla_decode(const qkmla_decode_args* a, void* stream);

/*
 * qkmla_get_device_status -- synchronise `stream`, return and clear the
 * current device's status word (QKMLA_OK or the first device-side error since
 * the last call).  Returns QKMLA_ERR_CUDA if synchronisation fails.
 */
int qkmla_get_device_status(void* stream);

/* Human-readable name of a return code (static string). */
const char* qkmla_status_string(int status);

/* Library version: major*10000 + minor*100 + patch. */
int qkmla_version(void);

/*
 * qkmla_decode_kernel_name -- which decode kernel qkmla_decode would launch for
 * these arguments on the current device: "tcgen05" (tensor-core kernel),
 * "simt" (CUDA-core kernel) or "invalid".  Static string.
 */
const char* qkmla_decode_kernel_name(const qkmla_decode_args* a);

/*
 * qkmla_decode_launch_count -- number of kernels one qkmla_decode call with
 * these arguments launches on the stream (tensor-core path: decode and
 * combine, plus a split-scheduler kernel ahead of them for batches of more
 * than 128 sequences -- smaller batches are planned inside the decode and
 * combine kernels; CUDA-core path: decode, plus combine when it splits).
 * Returns 0 for arguments qkmla_decode would reject.
 */
int qkmla_decode_launch_count(const qkmla_decode_args* a);

/*
 * qkmla_decode_noalloc -- qkmla_decode for callers that cannot allocate
 * device memory when they decode: a runtime that hands out only pre-planned
 * buffers, a plugin whose host owns every allocation, or a thread that must
 * not enter the CUDA allocator.  The paper has no counterpart to this call.
 *
 * Same arguments and results as qkmla_decode, except that `workspace` and
 * `workspace_bytes` are ignored: the split-KV partials and scheduler data live
 * in a fixed array of qkmla_decode_noalloc_max_workspace() bytes (64 MiB)
 * inside the library.  The array is part of the library's device code, so it
 * is reserved on a GPU when that code is loaded there -- with CUDA's default
 * lazy loading, at the first launch of any of the library's kernels on that
 * device; with CUDA_MODULE_LOADING=EAGER, when a context is created -- and is
 * held until the process exits.  The call allocates nothing.  Arguments
 * needing more scratch than that return QKMLA_ERR_WORKSPACE before anything is
 * launched.
 * The first call on a device resolves the array's address on that device (it
 * must be current) and keeps it for the process; make that first call before
 * any stream capture, and do not use the library across a cudaDeviceReset
 * (the kept address would be stale).  All calls on a device share the array:
 * calls whose kernels can overlap on the GPU (different streams with no
 * ordering between them) race on it.  The array keeps the previous call's
 * contents; decode writes every scratch entry it reads, so nothing needs to
 * start at zero.
 */
int qkmla_decode_noalloc(const qkmla_decode_args* a, void* stream);

/*
 * qkmla_up_project -- per-head values from the latent-space decode output.
 * Source: Technical Summary, Problem Statement (MLA keeps the low-dimensional
 * latent and recovers per-head quantities through up-projections, as W^K_g
 * recovers the key); the abstract (decode keeps the latent path, so attention
 * returns o = sum_t p_t c_t).  The value of head h is recovered once per query
 * row instead of once per cached token:
 *
 *   out[r][h][j] = sum_n o[r][h][n] * W^V[g(h)][n][j],   g(h) = h / (H / G_v)
 *
 * which equals softmax attention over materialised values c_t W^V_{g(h)}
 * (the softmax weights sum to one).
 * o     [rows][H][d_c] in o_dtype (QKMLA_F32 or QKMLA_BF16): qkmla_decode's output
 * w_v   [G_v][d_c][d_v] bf16 (G_v = H: one matrix per head)
 * out   [rows][H][d_v] in out_dtype (QKMLA_F32 or QKMLA_BF16)
 * Tensor cores, fp32 accumulation; an fp32 o is split into two bf16 parts
 * (fp32-level accuracy).  Errors: INVALID for null pointers, non-positive
 * sizes, H % G_v != 0 or a base not 16-byte aligned; UNSUPPORTED for other
 * dtypes, d_c % 64 != 0, or d_v not in {64, 128, 192, 256}.
 */
int qkmla_up_project(const void* o, int o_dtype, const void* w_v, int rows, int H, int G_v, int d_c,
                     int d_v, void* out, int out_dtype, void* stream);

/* Bytes of scratch qkmla_decode_noalloc can use (its fixed array). */
size_t qkmla_decode_noalloc_max_workspace(void);

#ifdef __cplusplus
}
#endif

#endif /* QKMLA_H */
