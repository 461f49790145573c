// Debug guard regions of the library workspace (MUON_DEBUG_GUARD=1).
//
// With guards on, the planner leaves kGuardBytes before the first and after
// every workspace region; each call fills them with kGuardWord before its
// first kernel and, after its last one, this kernel checks that they still
// hold it.  A changed guard means some kernel wrote outside its region; the
// check records MUON_ERR_CORRUPT (6) in its status word, which
// muon_device_status reports.  One CTA per guard region.
#include <cuda_runtime.h>

#include "internal.h"

namespace muon {

__device__ int g_muon_guard_error = 0;

namespace {

constexpr int kErrCorrupt = 6;

__global__ void __launch_bounds__(256) k_guard_check(const __grid_constant__ GuardParams p) {
    if (static_cast<int>(blockIdx.x) >= p.n) return;
    const uint4* q = reinterpret_cast<const uint4*>(p.base + p.off[blockIdx.x]);
    bool bad = false;
    for (int i = threadIdx.x; i < static_cast<int>(kGuardBytes / 16); i += blockDim.x) {
        const uint4 v = q[i];
        bad |= v.x != kGuardWord || v.y != kGuardWord || v.z != kGuardWord || v.w != kGuardWord;
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicCAS(&g_muon_guard_error, 0, kErrCorrupt);
}

}  // namespace

cudaError_t launch_guard_check(const GuardParams& p, cudaStream_t s) {
    if (p.n <= 0) return cudaSuccess;
    k_guard_check<<<p.n, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t read_and_clear_guard_error(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_muon_guard_error, sizeof(int));
    if (e != cudaSuccess) return e;
    *code = v;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_muon_guard_error, &zero, sizeof(int));
}

}  // namespace muon
