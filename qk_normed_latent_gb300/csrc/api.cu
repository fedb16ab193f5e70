// C-ABI entry points: argument validation, planning and dispatch.
//
// Every call validates on the host before launching anything and returns a
// QKMLA_* code; nothing here allocates device memory except the per-device
// status word, a static __device__ variable.
#include <mutex>

#include "common.cuh"

namespace qkmla {

__device__ int g_status_word;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sm_count[kMaxDevices];
int* g_status_ptr[kMaxDevices];

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }
}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

int* device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_status_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = (int*)p;
    }
    return g_status_ptr[dev];
}

static int validate_decode(const qkmla_decode_args* a) {
    if (!a) return QKMLA_ERR_INVALID;
    const bool plain = (a->flags & QKMLA_FLAG_PLAIN_MLA) != 0;
    if (a->B < 1 || a->s_q < 1 || a->H < 1 || a->G < 1 || a->d_c < 1 || a->d_r < 0) return QKMLA_ERR_INVALID;
    if (a->H % a->G) return QKMLA_ERR_INVALID;
    if (a->page_size < 1 || a->max_pages < 1 || a->num_slots < 1 || a->num_slots % a->page_size)
        return QKMLA_ERR_INVALID;
    if (a->num_splits < 0 || a->num_splits > 1024) return QKMLA_ERR_INVALID;
    if (a->cache_dtype != QKMLA_F32 && a->cache_dtype != QKMLA_BF16) return QKMLA_ERR_UNSUPPORTED;
    if (a->o_dtype != QKMLA_F32 && a->o_dtype != QKMLA_BF16) return QKMLA_ERR_UNSUPPORTED;
    if (!a->q_tilde || !a->kv_cache || !a->seq_lens || !a->o) return QKMLA_ERR_INVALID;
    if (!plain && (!a->alpha_q || !a->ak_cache)) return QKMLA_ERR_INVALID;
    if (a->d_r > 0 && !a->q_rope) return QKMLA_ERR_INVALID;
    if (!(a->softmax_scale > 0.f) || !(a->eps >= 0.f)) return QKMLA_ERR_INVALID;
    const size_t esz = a->cache_dtype == QKMLA_F32 ? 4 : 2;
    if (!aligned(a->q_tilde, esz) || !aligned(a->kv_cache, esz) || !aligned(a->o, 4)) return QKMLA_ERR_INVALID;
    const int hpg = a->H / a->G;
    if (hpg != 1 && hpg != 2 && hpg != 4 && hpg != 8 && hpg != 16) return QKMLA_ERR_UNSUPPORTED;
    if (a->d_c > 512 || a->d_r > 128) return QKMLA_ERR_UNSUPPORTED;
    return QKMLA_OK;
}

int plan_decode(const qkmla_decode_args* a, DecodePlan* plan) {
    const int v = validate_decode(a);
    if (v != QKMLA_OK) return v;
    const int sms = device_sm_count();
    if (sms <= 0) return QKMLA_ERR_CUDA;
    const bool stall = (a->flags & QKMLA_FLAG_TEST_STALL) != 0;
    if (!(a->flags & QKMLA_FLAG_FORCE_SIMT) && tc_supported(a) && a->num_splits <= 256) {
        if (stall && pair_shape(a)) return QKMLA_ERR_UNSUPPORTED;   // the hook exists in the 64-row kernel only
        plan->kernel = 1;
        plan->num_splits = a->num_splits;
        plan->parts = 0;
        plan->ws_bytes = tc_workspace(a, sms, nullptr);
        return QKMLA_OK;
    }
    if (stall) return QKMLA_ERR_UNSUPPORTED;
    plan->kernel = 0;
    int ns = a->num_splits;
    if (ns == 0) {
        const int64_t base = (int64_t)a->B * a->s_q * a->G;
        const int64_t max_len = (int64_t)a->max_pages * a->page_size;
        int64_t want = (2LL * sms + base - 1) / base;
        const int64_t cap = (max_len + 255) / 256;
        if (want > cap) want = cap;
        if (want < 1) want = 1;
        if (want > 256) want = 256;
        ns = (int)want;
    }
    plan->num_splits = ns;
    plan->parts = ns;
    const int64_t rows_h = (int64_t)a->B * a->s_q * a->H;
    plan->ws_bytes = ns > 1 ? (size_t)rows_h * ns * (a->d_c + 1) * sizeof(float) : 0;
    return QKMLA_OK;
}

}  // namespace qkmla

using namespace qkmla;

extern "C" {

int qkmla_version(void) { return 100; }

const char* qkmla_status_string(int st) {
    switch (st) {
        case QKMLA_OK: return "ok";
        case QKMLA_ERR_INVALID: return "invalid argument";
        case QKMLA_ERR_UNSUPPORTED: return "unsupported configuration";
        case QKMLA_ERR_CUDA: return "CUDA error";
        case QKMLA_ERR_WORKSPACE: return "workspace missing or too small";
        case QKMLA_ERR_DEVICE_BOUNDS: return "device-side bounds error (page id or sequence length)";
        case QKMLA_ERR_TIMEOUT: return "device-side bounded wait expired";
    }
    return "unknown status";
}

int qkmla_absorb_query(const float* q, const float* gamma_q, const float* gamma_k, const float* w_k, int rows,
                       int H, int G, int d_h, int d_c, float eps, unsigned flags, void* q_tilde, int qt_dtype,
                       float* alpha_q, void* stream) {
    const bool plain = (flags & QKMLA_FLAG_PLAIN_MLA) != 0;
    if (rows < 1 || H < 1 || G < 1 || d_h < 1 || d_c < 1 || H % G) return QKMLA_ERR_INVALID;
    if (d_h > 256 || d_c % 8) return QKMLA_ERR_INVALID;
    if (!q || !w_k || !q_tilde || !alpha_q) return QKMLA_ERR_INVALID;
    if (!plain && (!gamma_q || !gamma_k)) return QKMLA_ERR_INVALID;
    if (!(eps >= 0.f)) return QKMLA_ERR_INVALID;
    if (qt_dtype != QKMLA_F32 && qt_dtype != QKMLA_BF16) return QKMLA_ERR_UNSUPPORTED;
    return launch_absorb(q, gamma_q, gamma_k, w_k, rows, H, G, d_h, d_c, eps, plain, q_tilde, qt_dtype, alpha_q,
                         (cudaStream_t)stream);
}

int qkmla_append(const float* c_new, const float* k_rope_new, const float* w_k, const float* gamma_rope_k,
                 const int64_t* slot_mapping, int N, int G, int d_c, int d_h, int d_r, float eps, unsigned flags,
                 void* kv_cache, int cache_dtype, void* ak_cache, int64_t num_slots, void* stream) {
    const bool plain = (flags & QKMLA_FLAG_PLAIN_MLA) != 0;
    if (N < 0 || G < 1 || d_c < 1 || d_h < 1 || d_r < 0 || num_slots < 1) return QKMLA_ERR_INVALID;
    if (d_h > 256) return QKMLA_ERR_INVALID;
    if (cache_dtype != QKMLA_F32 && cache_dtype != QKMLA_BF16) return QKMLA_ERR_UNSUPPORTED;
    if (N == 0) return QKMLA_OK;
    if (!c_new || !w_k || !slot_mapping || !kv_cache || !ak_cache) return QKMLA_ERR_INVALID;
    if (d_r > 0 && !k_rope_new) return QKMLA_ERR_INVALID;
    if (!(eps >= 0.f)) return QKMLA_ERR_INVALID;
    const bool ak_f16 = !plain && (flags & QKMLA_FLAG_ALPHA_F16) != 0;
    return launch_append(c_new, k_rope_new, w_k, gamma_rope_k, slot_mapping, N, G, d_c, d_h, d_r, eps, plain,
                         kv_cache, cache_dtype, ak_cache, ak_f16, num_slots, nullptr, 0.f, (cudaStream_t)stream);
}

int qkmla_append_rope(const float* c_new, const float* k_rope_raw, const int32_t* positions, float rope_theta,
                      const float* w_k, const float* gamma_rope_k, const int64_t* slot_mapping, int N, int G, int d_c,
                      int d_h, int d_r, float eps, unsigned flags, void* kv_cache, int cache_dtype, void* ak_cache,
                      int64_t num_slots, void* stream) {
    if (N > 0 && d_r > 0 && (!positions || !(rope_theta > 1.f) || d_r % 2)) return QKMLA_ERR_INVALID;
    if (d_r > 64) return QKMLA_ERR_UNSUPPORTED;
    const bool plain = (flags & QKMLA_FLAG_PLAIN_MLA) != 0;
    if (N < 0 || G < 1 || d_c < 1 || d_h < 1 || d_r < 0 || num_slots < 1) return QKMLA_ERR_INVALID;
    if (d_h > 256) return QKMLA_ERR_INVALID;
    if (cache_dtype != QKMLA_F32 && cache_dtype != QKMLA_BF16) return QKMLA_ERR_UNSUPPORTED;
    if (N == 0) return QKMLA_OK;
    if (!c_new || !w_k || !slot_mapping || !kv_cache || !ak_cache) return QKMLA_ERR_INVALID;
    if (d_r > 0 && !k_rope_raw) return QKMLA_ERR_INVALID;
    if (!(eps >= 0.f)) return QKMLA_ERR_INVALID;
    const bool ak_f16 = !plain && (flags & QKMLA_FLAG_ALPHA_F16) != 0;
    return launch_append(c_new, k_rope_raw, w_k, gamma_rope_k, slot_mapping, N, G, d_c, d_h, d_r, eps, plain,
                         kv_cache, cache_dtype, ak_cache, ak_f16, num_slots, d_r > 0 ? positions : nullptr,
                         rope_theta, (cudaStream_t)stream);
}

size_t qkmla_decode_workspace_size(const qkmla_decode_args* a) {
    DecodePlan plan;
    if (plan_decode(a, &plan) != QKMLA_OK) return 0;
    return plan.ws_bytes;
}

const char* qkmla_decode_kernel_name(const qkmla_decode_args* a) {
    DecodePlan plan;
    if (plan_decode(a, &plan) != QKMLA_OK) return "invalid";
    return plan.kernel == 1 ? "tcgen05" : "simt";
}

int qkmla_decode_launch_count(const qkmla_decode_args* a) {
    DecodePlan plan;
    if (plan_decode(a, &plan) != QKMLA_OK) return 0;
    if (plan.kernel == 1) return sched_in_kernel(a) ? 2 : 3;   // [scheduler,] decode, combine
    return plan.parts > 1 ? 2 : 1;
}

int qkmla_decode(const qkmla_decode_args* a, void* stream) {
    DecodePlan plan;
    const int rc = plan_decode(a, &plan);
    if (rc != QKMLA_OK) return rc;
    if (plan.ws_bytes > 0 && (!a->workspace || a->workspace_bytes < plan.ws_bytes)) return QKMLA_ERR_WORKSPACE;
    if (plan.ws_bytes > 0 && !aligned(a->workspace, 16)) return QKMLA_ERR_INVALID;
    if (plan.kernel == 1) return launch_decode_tc(a, plan, (cudaStream_t)stream);
    return launch_decode_simt(a, plan, (cudaStream_t)stream);
}

int qkmla_get_device_status(void* stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return QKMLA_ERR_CUDA;
    int* p = device_status_ptr();
    if (!p) return QKMLA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return QKMLA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return QKMLA_ERR_CUDA;
    return v;
}

}  // extern "C"
