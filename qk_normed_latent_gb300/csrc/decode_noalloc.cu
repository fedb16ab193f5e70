// qkmla_decode_noalloc: qkmla_decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they decode:
// code that runs inside an allocator-free runtime (a serving engine that
// hands out only pre-planned buffers, a plugin whose host owns every
// allocation, or a thread that must not touch the CUDA allocator because it
// would synchronise or fail under memory pressure).  This entry point takes
// the same arguments as qkmla_decode but ignores `workspace` /
// `workspace_bytes`: the split-KV partials and scheduler metadata live in a
// fixed, file-scope device array.  It belongs to the library's device code, so
// a GPU reserves it when that code is loaded there (CUDA's default lazy
// loading: at the first launch of any kernel of this library on the device;
// eager loading: at context creation) and holds it until the process exits.
//
// The first call on a device resolves the array's device address with
// cudaGetSymbolAddress (with that device current) and keeps it for the
// process; make that first call before any stream capture, and do not use the
// library across a cudaDeviceReset (the kept address would be stale).  All calls on a device share the one
// array, so calls whose kernels overlap on the GPU (different streams without
// ordering) race on it; calls serialised on one stream are fine.  The array
// keeps the previous call's contents; the decode path writes every scheduler
// and partial entry it later reads, so nothing has to start at zero.
#include <mutex>

#include "common.cuh"

namespace qkmla {
namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;   // 64 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDev];

// Device address of this device's scratch array (resolved once per device).
int scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return QKMLA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return QKMLA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return QKMLA_OK;
}

}  // namespace
}  // namespace qkmla

extern "C" {

size_t qkmla_decode_noalloc_max_workspace(void) { return qkmla::kNoAllocScratchBytes; }

int qkmla_decode_noalloc(const qkmla_decode_args* a, void* stream) {
    if (!a) return QKMLA_ERR_INVALID;
    const size_t need = qkmla_decode_workspace_size(a);
    qkmla_decode_args b = *a;
    if (need > qkmla::kNoAllocScratchBytes) return QKMLA_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int rc = qkmla::scratch_for_current_device(&scratch);
    if (rc != QKMLA_OK) return rc;
    b.workspace = scratch;
    b.workspace_bytes = qkmla::kNoAllocScratchBytes;
    return qkmla_decode(&b, stream);
}

}  // extern "C"
