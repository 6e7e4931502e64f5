// la_forward_causal_noalloc: the causal forward with its scratch in a fixed
// device array instead of a caller-provided workspace, for callers that may
// not allocate device memory on their hot path (budgeted serving loops,
// plug-ins inside frameworks that own all device memory).
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library reserves it until the process exits.  In host code its name only
// stands for the host-side shadow, never a device address: the device
// address is looked up once per device with cudaGetSymbolAddress while that
// device is current, cached, and passed to the kernels as the workspace.
// All calls on a device share the array; the planning phase of every call
// rewrites the header it later reads, so no clearing is needed, and calls
// whose GPU work overlaps race on it.
#include <mutex>

#include "internal.h"

namespace la {
namespace {

constexpr size_t kScratchBytes = LA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once).
la_status scratch_address(void** addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return LA_OK;
}

}  // namespace
}  // namespace la

extern "C" la_status la_noalloc_error(int* code, void* stream) {
    void* scratch = nullptr;
    const la_status st = la::scratch_address(&scratch);
    if (st != LA_OK) return st;
    return la_workspace_error(scratch, code, stream);
}

extern "C" la_status la_forward_causal_noalloc(const void* q, const void* k, const void* v, const float* omega,
                                               int map, int dtype, const int32_t* cu_seqlens, int nseq, int64_t T,
                                               int H, int d_k, int d_v, int r, float eps, void* out,
                                               void* stream) {
    void* scratch = nullptr;
    const la_status st = la::scratch_address(&scratch);
    if (st != LA_OK) return st;
    // forward_entry checks every argument and returns LA_ERR_WORKSPACE, with
    // nothing enqueued, when the plan needs more than kScratchBytes.
    return la::forward_entry(1, LA_PHASE_PLAN, LA_PHASE_OUTPUT, q, k, v, omega, map, dtype, cu_seqlens, nseq, T, H,
                             d_k, d_v, r, eps, out, scratch, la::kScratchBytes, stream, nullptr);
}
