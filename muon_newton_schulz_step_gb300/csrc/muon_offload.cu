// muon_step_host: the Muon step on optimizer state kept in (pinned) host memory.
//
// "Domyn is training a 1T-parameter MoE on Europe's Jupiter supercomputer,
// and published the recipe", section "What moved the number" (Offloading
// bullet): optimizer state lives in Grace memory and moves over NVLink-C2C.
// Here W, G and M stay in host memory; the call streams them through the GPU
// in chunks of whole matrices with three device staging sets, so that the copy
// in of chunk c+1 and the copy out of chunk c-1 overlap the step on chunk c,
// and the copy in never waits for the copy out of the chunk before:
//
//   copy-in stream:   W,G,M(c) -> staging[c % 3]          (after staging[c % 3] is free)
//   caller's stream:  muon_step_ex on staging[c % 3]       (after its copy-in)
//   copy-out stream:  W,M(c) -> host                       (after its step)
//
// (With two sets the copy in of chunk c+1 waits for the copy out of chunk
// c-1, idling the host-to-device link for part of every other chunk.)
//
// The caller's stream waits for the last copy-out before the call returns, so
// the whole step is ordered on the caller's stream like every other call.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "muon.h"

namespace muon {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kChunkTargetBytes = size_t(1) << 30;  // ~1 GiB of W+G+M per chunk
constexpr size_t kEdgeChunkBytes = size_t(256) << 20;  // first and last chunk
constexpr int kStagingSets = 3;

struct Staging {
    void* buf = nullptr;
    size_t bytes = 0;
    cudaEvent_t copied_in = nullptr;   // chunk data on the device
    cudaEvent_t stepped = nullptr;     // step done, results ready to copy out
    cudaEvent_t free_ev = nullptr;     // copy-out done, buffer reusable
    bool used = false;
};

struct HostState {
    bool init = false;
    cudaStream_t in = nullptr, out = nullptr;
    Staging st[kStagingSets];
};

std::mutex g_host_mu;
HostState g_host[kMaxDevices];

int host_state(HostState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_last_error(MUON_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return set_last_error(MUON_ERR_UNSUPPORTED, "device ordinal out of range");
    HostState& h = g_host[dev];
    if (!h.init) {
        if (cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) != cudaSuccess)
            return set_last_error(MUON_ERR_CUDA, "creating the copy streams failed");
        for (Staging& s : h.st)
            if (cudaEventCreateWithFlags(&s.copied_in, cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&s.stepped, cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&s.free_ev, cudaEventDisableTiming) != cudaSuccess)
                return set_last_error(MUON_ERR_CUDA, "creating events failed");
        h.init = true;
    }
    *out = &h;
    return MUON_OK;
}

bool pinned(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Chunk boundaries (first matrix of every chunk, then count) for matrices of
// mb[i] bytes of state: a first and a last chunk of at most kEdgeChunkBytes,
// so that the pipeline fills and drains quickly (while the first chunk comes
// in and the last goes out the link carries one direction only), and greedy
// chunks of at most kChunkTargetBytes in between.  Every chunk holds at least
// one matrix.
std::vector<int> plan_chunks(const std::vector<size_t>& mb) {
    const int count = static_cast<int>(mb.size());
    int tail = count - 1;   // first matrix of the last chunk
    for (size_t tb = mb[count - 1]; tail > 1 && tb + mb[tail - 1] <= kEdgeChunkBytes; --tail) tb += mb[tail - 1];
    std::vector<int> b{0};
    int i = 0;
    for (size_t acc = 0; i < tail && (acc == 0 || acc + mb[i] <= kEdgeChunkBytes); ++i) acc += mb[i];
    while (i < tail) {
        b.push_back(i);
        for (size_t acc = 0; i < tail && (acc == 0 || acc + mb[i] <= kChunkTargetBytes); ++i) acc += mb[i];
    }
    if (tail > 0) b.push_back(tail);
    b.push_back(count);
    return b;
}

}  // namespace
}  // namespace muon

using namespace muon;

extern "C" int muon_step_host(void* const* W, const void* const* G, float* const* M, const int* rows,
                              const int* cols, int count, float lr, float mu, float wd,
                              const muon_step_opts* opts, cudaStream_t stream) {
    muon_step_opts o;
    muon_step_opts_init(&o);
    if (opts != nullptr) o = *opts;
    if (count < 0) return set_last_error(MUON_ERR_INVALID_ARG, "count is negative");
    if (count == 0) return MUON_OK;
    if (W == nullptr || G == nullptr || M == nullptr || rows == nullptr || cols == nullptr)
        return set_last_error(MUON_ERR_INVALID_ARG, "a pointer array is NULL");
    if (o.workspace != nullptr || o.o_out != nullptr)
        return set_last_error(MUON_ERR_INVALID_ARG, "muon_step_host takes no workspace and no o_out");
    if ((o.w_dtype != MUON_BF16 && o.w_dtype != MUON_F32) || (o.g_dtype != MUON_BF16 && o.g_dtype != MUON_F32))
        return set_last_error(MUON_ERR_INVALID_ARG, "unknown dtype");
    if (o.steps < 0 || o.steps > 64 || o.nesterov < 0 || o.nesterov > 1 || !(o.eps >= 0.0f) ||
        !std::isfinite(o.eps) || !std::isfinite(lr) || !std::isfinite(mu) || !std::isfinite(wd))
        return set_last_error(MUON_ERR_INVALID_ARG, "steps, nesterov, eps, lr, mu or wd out of range");
    if (o.coeffs_per_step != 0 && o.coeffs_per_step != 1)
        return set_last_error(MUON_ERR_INVALID_ARG, "coeffs_per_step must be 0 or 1");
    if (o.g_count < 1 || o.g_count > 64) return set_last_error(MUON_ERR_INVALID_ARG, "g_count must be in [1, 64]");
    if (o.ns_fp8_gram != 0 && o.ns_fp8_gram != 1)
        return set_last_error(MUON_ERR_INVALID_ARG, "ns_fp8_gram must be 0 or 1");
    if (o.coeffs != nullptr)
        for (int j = 0; j < (o.coeffs_per_step ? 3 * o.steps : 3); ++j)
            if (!std::isfinite(o.coeffs[j])) return set_last_error(MUON_ERR_INVALID_ARG, "coefficient not finite");
    const size_t wsz = o.w_dtype == MUON_F32 ? 4 : 2;
    const size_t gsz = (o.g_dtype == MUON_F32 ? 4 : 2) * static_cast<size_t>(o.g_count);  // all stacked gradients
    std::vector<std::pair<uintptr_t, std::pair<uintptr_t, int>>> iv;  // [lo, hi), writes
    for (int i = 0; i < count; ++i) {
        if (W[i] == nullptr || G[i] == nullptr || M[i] == nullptr)
            return set_last_error(MUON_ERR_INVALID_ARG, "a host pointer is NULL");
        const size_t n = static_cast<size_t>(std::max(rows[i], 0)) * static_cast<size_t>(std::max(cols[i], 0));
        const uintptr_t w = reinterpret_cast<uintptr_t>(W[i]), g = reinterpret_cast<uintptr_t>(G[i]),
                        m = reinterpret_cast<uintptr_t>(M[i]);
        iv.push_back({w, {w + n * wsz, 1}});
        iv.push_back({g, {g + n * gsz, 0}});
        iv.push_back({m, {m + n * 4, 1}});
    }
    std::sort(iv.begin(), iv.end());
    uintptr_t run_hi = 0;
    int run_w = 0;
    for (size_t i = 0; i < iv.size(); ++i) {
        if (i > 0 && iv[i].first < run_hi && (iv[i].second.second || run_w))
            return set_last_error(MUON_ERR_INVALID_ARG, "host buffers overlap");
        if (i == 0 || iv[i].second.first > run_hi) {
            run_hi = iv[i].second.first;
            run_w = iv[i].second.second;
        } else {
            run_w |= iv[i].second.second;
        }
    }
    for (int i = 0; i < count; ++i) {
        if (rows[i] < 1 || cols[i] < 1 || rows[i] > MUON_MAX_DIM || cols[i] > MUON_MAX_DIM)
            return set_last_error(MUON_ERR_INVALID_ARG, "a matrix has a dimension outside [1, MUON_MAX_DIM]");
        if (!pinned(W[i]) || !pinned(G[i]) || !pinned(M[i])) {
            char msg[160];
            std::snprintf(msg, sizeof msg, "host buffers of matrix %d are not pinned (page-locked) host memory", i);
            return set_last_error(MUON_ERR_INVALID_ARG, msg);
        }
    }

    std::vector<size_t> mb(count);
    for (int i = 0; i < count; ++i) {
        const size_t n = static_cast<size_t>(rows[i]) * cols[i];
        mb[i] = align256(n * wsz) + align256(n * gsz) + align256(n * 4);
    }
    const std::vector<int> first = plan_chunks(mb);
    size_t chunk_max = 0;
    for (size_t c = 0; c + 1 < first.size(); ++c) {
        size_t acc = 0;
        for (int i = first[c]; i < first[c + 1]; ++i) acc += mb[i];
        chunk_max = std::max(chunk_max, acc);
    }

    std::lock_guard<std::mutex> lock(g_host_mu);
    HostState* h = nullptr;
    int rc = host_state(&h);
    if (rc != MUON_OK) return rc;
    for (Staging& s : h->st) {
        if (s.bytes < chunk_max) {
            if (s.buf != nullptr) {
                if (s.used) cudaStreamWaitEvent(stream, s.free_ev, 0);
                cudaFreeAsync(s.buf, stream);
                s.buf = nullptr;
                s.bytes = 0;
            }
            if (cudaMallocAsync(&s.buf, chunk_max, stream) != cudaSuccess) {
                cudaGetLastError();
                return set_last_error(MUON_ERR_OOM, "staging allocation failed");
            }
            s.bytes = chunk_max;
            s.used = false;
        }
    }
    // copy-in may start only after the caller's prior work (and any staging allocation)
    cudaEvent_t ready = nullptr;
    if (cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) != cudaSuccess)
        return set_last_error(MUON_ERR_CUDA, "creating an event failed");
    cudaEventRecord(ready, stream);
    cudaStreamWaitEvent(h->in, ready, 0);
    cudaStreamWaitEvent(h->out, ready, 0);
    cudaEventDestroy(ready);  // destruction is deferred until the event completes

    // A failure after the first copy was enqueued: the copies already on the two
    // copy streams still read or write the caller's host buffers, so the
    // caller's stream is ordered after both streams' tails before returning.
    auto fail_in_flight = [&](int status, const char* msg) -> int {
        for (cudaStream_t cs : {h->in, h->out}) {
            cudaEvent_t tail = nullptr;
            if (cudaEventCreateWithFlags(&tail, cudaEventDisableTiming) == cudaSuccess) {
                cudaEventRecord(tail, cs);
                cudaStreamWaitEvent(stream, tail, 0);
                cudaEventDestroy(tail);
            }
        }
        return msg != nullptr ? set_last_error(status, msg) : status;
    };

    const int nchunks = static_cast<int>(first.size()) - 1;
    std::vector<void*> dW, dG, dM;
    for (int c = 0; c < nchunks; ++c) {
        Staging& s = h->st[c % kStagingSets];
        const int i0 = first[c], i1 = first[c + 1], n = i1 - i0;
        if (s.used) cudaStreamWaitEvent(h->in, s.free_ev, 0);
        dW.assign(n, nullptr);
        dG.assign(n, nullptr);
        dM.assign(n, nullptr);
        char* p = static_cast<char*>(s.buf);
        for (int j = 0; j < n; ++j) {
            const size_t e = static_cast<size_t>(rows[i0 + j]) * cols[i0 + j];
            dW[j] = p; p += align256(e * wsz);
            dG[j] = p; p += align256(e * gsz);
            dM[j] = p; p += align256(e * 4);
            if (cudaMemcpyAsync(dW[j], W[i0 + j], e * wsz, cudaMemcpyHostToDevice, h->in) != cudaSuccess ||
                cudaMemcpyAsync(dG[j], G[i0 + j], e * gsz, cudaMemcpyHostToDevice, h->in) != cudaSuccess ||
                cudaMemcpyAsync(dM[j], M[i0 + j], e * 4, cudaMemcpyHostToDevice, h->in) != cudaSuccess)
                return fail_in_flight(MUON_ERR_CUDA, "host-to-device copy failed to enqueue");
        }
        cudaEventRecord(s.copied_in, h->in);
        cudaStreamWaitEvent(stream, s.copied_in, 0);
        muon_step_opts od = o;
        rc = muon_step_ex(dW.data(), const_cast<const void* const*>(dG.data()),
                          reinterpret_cast<float* const*>(dM.data()), rows + i0, cols + i0, n, lr, mu, wd, &od,
                          stream);
        if (rc != MUON_OK) return fail_in_flight(rc, nullptr);   // muon_step_ex set the message
        cudaEventRecord(s.stepped, stream);
        cudaStreamWaitEvent(h->out, s.stepped, 0);
        for (int j = 0; j < n; ++j) {
            const size_t e = static_cast<size_t>(rows[i0 + j]) * cols[i0 + j];
            if (cudaMemcpyAsync(W[i0 + j], dW[j], e * wsz, cudaMemcpyDeviceToHost, h->out) != cudaSuccess ||
                cudaMemcpyAsync(M[i0 + j], dM[j], e * 4, cudaMemcpyDeviceToHost, h->out) != cudaSuccess)
                return fail_in_flight(MUON_ERR_CUDA, "device-to-host copy failed to enqueue");
        }
        cudaEventRecord(s.free_ev, h->out);
        s.used = true;
    }
    // the caller's stream completes only after every copy-out
    for (Staging& s : h->st)
        if (s.used) cudaStreamWaitEvent(stream, s.free_ev, 0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_last_error(MUON_ERR_CUDA, cudaGetErrorString(e));
    return MUON_OK;
}
