// muon_ns5_batched_static: the Newton-Schulz entry point for callers that
// cannot allocate device memory.
//
// Some callers must not call cudaMalloc (or anything that allocates): code
// that runs while a framework's caching allocator owns the whole device
// budget and would be pushed out of memory by a stray allocation, code on a
// latency-critical path where cudaMalloc's implicit device synchronisation is
// not acceptable, and hosts that hand the library a fixed memory budget.  For
// them this entry point runs the same kernels as muon_ns5_batched, but its
// scratch (the per-tile norm partials, the per-matrix scales and the padded
// iterates X, A, B) lives in one file-scope device array of fixed size,
// reserved when the library is loaded and kept by every GPU that loads it
// until the process exits.  The caller still passes the matrices themselves.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "internal.h"
#include "muon.h"

namespace muon {
namespace {

constexpr size_t kStaticScratchBytes = MUON_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch array.  In host code this name is only a host-side stand-in:
// its device address comes from cudaGetSymbolAddress (below).
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.
int static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_last_error(MUON_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return set_last_error(MUON_ERR_UNSUPPORTED, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || p == nullptr) {
            char msg[256];
            std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch failed: %s",
                          cudaGetErrorString(e));
            return set_last_error(MUON_ERR_CUDA, msg);
        }
        g_static_addr[dev] = p;
    }
    *out = g_static_addr[dev];
    return MUON_OK;
}

}  // namespace
}  // namespace muon

using namespace muon;

extern "C" int muon_ns5_batched_static(void* const* ptrs, const int* rows, const int* cols, int count,
                                       int steps, const float* coeffs, cudaStream_t stream) {
    if (count < 0) return set_last_error(MUON_ERR_INVALID_ARG, "count is negative");
    if (count == 0) return MUON_OK;
    if (ptrs == nullptr || rows == nullptr || cols == nullptr)
        return set_last_error(MUON_ERR_INVALID_ARG, "a pointer array is NULL");
    const size_t need = muon_workspace_bytes(rows, cols, count);
    if (need == 0)
        return set_last_error(MUON_ERR_INVALID_ARG, "a matrix has a dimension outside [1, MUON_MAX_DIM]");
    if (need > kStaticScratchBytes) {
        char msg[256];
        std::snprintf(msg, sizeof msg,
                      "this batch needs %zu bytes of scratch; the static scratch of "
                      "muon_ns5_batched_static holds %zu bytes (MUON_STATIC_SCRATCH_BYTES)",
                      need, kStaticScratchBytes);
        return set_last_error(MUON_ERR_UNSUPPORTED, msg);
    }
    void* scratch = nullptr;
    const int rc = static_scratch(&scratch);
    if (rc != MUON_OK) return rc;
    return ns5_batched_on_workspace(ptrs, rows, cols, count, steps, coeffs, scratch, kStaticScratchBytes,
                                    stream);
}
