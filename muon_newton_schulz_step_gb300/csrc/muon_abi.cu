// C ABI of the Muon optimizer-step library (include/muon.h): validation,
// ragged-batch planning, workspace, TMA descriptors and the launch sequence.
//
// The step it runs is the per-matrix Muon step over whole matrices held on
// one rank ("How PyTorch Scaled a Near-1T MoE on Europe's Public
// Supercomputer", section "Three optimizations that changed the economics",
// FlexShard bullet: whole experts on one rank, so the Newton-Schulz
// orthogonalisation of each full matrix needs no communication).  Every
// matrix is independent; a call batches any number of them:
//
//   per chunk of <= kEwMaxMats matrices:  norm pass -> finalize -> pack
//   per Newton-Schulz iteration:          Gram -> Poly -> Update  (one launch
//                                          each over all shape buckets; the
//                                          last Update also writes W or O)
//   small matrices:                       every iteration in one launch
//                                          (clusters of CTAs, ns_small.cu)
//   per chunk:                            unpack of the matrices the last
//                                          Update did not write (small ones)
//
// Shape buckets: matrices are oriented so that r = min(m, n) <= k = max(m, n)
// and grouped by (r, k) rounded up to multiples of 256; each bucket owns
// contiguous, zero-padded iterate buffers X0, X1 (nmat x r_pad x k_pad) and
// A, B (nmat x r_pad x r_pad) in one workspace, addressed by 3-D TMA maps.
// A large batch runs as two parts on two streams (run_split); a batch whose
// workspace cannot be had in one piece runs as consecutive groups
// (make_groups / run_groups).
#include <cudaTypedefs.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "muon.h"

namespace muon {
namespace {

constexpr float kDefaultCoeffs[3] = {3.4445f, -4.7750f, 2.0315f};
constexpr int kMaxSteps = 64;
constexpr int kPad = 256;
constexpr int kMaxDevices = 64;

thread_local std::string t_last_error;
std::mutex g_mu;

int fail(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return status;
}

#define MUON_CUDA_TRY(expr, what)                                                         \
    do {                                                                                  \
        cudaError_t e_ = (expr);                                                          \
        if (e_ != cudaSuccess)                                                            \
            return fail(MUON_ERR_CUDA, "%s: %s", (what), cudaGetErrorString(e_));         \
    } while (0)

// ------------------------------------------------------------ device state --
struct DeviceState {
    bool init = false;
    int sms = 0;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    cudaEvent_t last_use = nullptr;
    cudaStream_t last_stream = nullptr;
    bool have_last = false;
    cudaStream_t aux = nullptr;        // second stream of a split call
    cudaEvent_t ev[4] = {};            // fork, front done, ns done, join
};
DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_state(DeviceState** out) {
    int dev = 0;
    MUON_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(MUON_ERR_UNSUPPORTED, "device ordinal %d", dev);
    DeviceState& d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0;
        MUON_CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "attr");
        MUON_CUDA_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "attr");
        if (major != 10 || minor != 3)
            return fail(MUON_ERR_UNSUPPORTED,
                        "device %d is sm_%d%d; this library is built for sm_103a only", dev, major, minor);
        MUON_CUDA_TRY(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev), "attr");
        MUON_CUDA_TRY(cudaEventCreateWithFlags(&d.last_use, cudaEventDisableTiming), "cudaEventCreate");
        MUON_CUDA_TRY(cudaStreamCreateWithFlags(&d.aux, cudaStreamNonBlocking), "cudaStreamCreate");
        for (cudaEvent_t& e : d.ev)
            MUON_CUDA_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "cudaEventCreate");
        d.init = true;
    }
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return fail(MUON_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = &d;
    return MUON_OK;
}

// --------------------------------------------------------------- profiling --
enum Kind : int {
    kKNorm = 0, kKFinalize, kKPack, kKGram, kKPoly, kKUpdate, kKSmall, kKUnpack, kKAdamW, kKFinal, kNumKinds
};
const char* const kKindNames[kNumKinds] = {"norm_pass",    "norm_finalize",  "pack",     "ns_gemm_gram",
                                           "ns_gemm_poly", "ns_gemm_update", "ns_small", "unpack",
                                           "adamw",        "ns_gemm_final"};
struct ProfRec {
    int kind;
    cudaEvent_t a, b;
    double flops, bytes;
};
struct ProfAgg {
    int launches = 0;
    double ms = 0, flops = 0, bytes = 0;
};
bool g_prof_on = false;
std::vector<ProfRec> g_prof_pending;
std::vector<cudaEvent_t> g_event_pool;
ProfAgg g_prof[kNumKinds];

cudaEvent_t pool_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

template <class F>
int launch(int kind, double flops, double bytes, cudaStream_t s, F&& f) {
    ProfRec r{kind, nullptr, nullptr, flops, bytes};
    if (g_prof_on) {
        r.a = pool_event();
        r.b = pool_event();
        if (r.a) cudaEventRecord(r.a, s);
    }
    cudaError_t e = f();
    if (g_prof_on) {
        if (r.b) cudaEventRecord(r.b, s);
        if (r.a && r.b) g_prof_pending.push_back(r);
    }
    if (e != cudaSuccess)
        return fail(MUON_ERR_CUDA, "%s launch failed: %s", kKindNames[kind], cudaGetErrorString(e));
    return MUON_OK;
}

// -------------------------------------------------------------------- plan --
struct MatPlan {
    int rows, cols, r, k, trans, bucket, slot;
    int small;                 // 1: iterates in shared memory (ns_small.cu), no bucket
    int r_pad64, k_pad64;      // padded iterate of a small matrix
    size_t xoff;               // its offset in the small-matrix region
    long long tiles1, part;
};
struct BucketPlan {
    int r_pad, k_pad, nmat = 0;
    size_t x0 = 0, x1 = 0, a = 0, b = 0;
    size_t x8 = 0;             // FP8 Gram: E4M3 copy of the current iterate (nmat x r_pad x k_pad bytes)
    double flops_gram = 0, flops_poly = 0, flops_update = 0;
};
struct Plan {
    std::vector<MatPlan> mats;
    std::vector<BucketPlan> buckets;
    size_t off_partials = 0, off_sigma = 0, off_small = 0, bytes = 0;
    int fp8 = 0;               // 1: the buckets carry the FP8 Gram's E4M3 iterate copies
    std::vector<size_t> guards;   // offsets of the debug guard regions (MUON_DEBUG_GUARD)
    long long total_tiles1 = 0;
    int nsmall = 0;
    size_t small_smem = 0;     // largest shared-memory need of the small matrices
    double small_flops = 0;
};

long long round_up(long long v, long long m) { return (v + m - 1) / m * m; }

bool env_flag(const char* name) {
    const char* v = std::getenv(name);
    return v != nullptr && v[0] != '\0' && v[0] != '0';
}

// MUON_DISABLE_SMALL_NS=1 sends every matrix through the tensor-core path
// (used by the tests to exercise that path on small shapes).
bool small_path_enabled() { return !env_flag("MUON_DISABLE_SMALL_NS"); }

// MUON_DEBUG_GUARD=1 (debugging): guard regions around the workspace regions,
// checked after every call; "poison" also overwrites one guard byte after
// filling them, to exercise the check.
bool guard_enabled() { return env_flag("MUON_DEBUG_GUARD"); }
bool guard_poison() {
    const char* v = std::getenv("MUON_DEBUG_GUARD");
    return v != nullptr && std::strcmp(v, "poison") == 0;
}

// fp8: also lay out the FP8 Gram's E4M3 copy of each bucket's iterate (1 byte
// per element of the padded iterate; one copy serves every iteration: the update
// that writes it for the next Gram runs after this Gram has read it)
void build_plan(const int* rows, const int* cols, int count, Plan& pl, bool fp8 = false) {
    const bool allow_small = small_path_enabled();
    pl.mats.resize(count);
    pl.buckets.clear();
    long long part = 0;
    for (int i = 0; i < count; ++i) {
        MatPlan& m = pl.mats[i];
        m.rows = rows[i];
        m.cols = cols[i];
        m.trans = m.rows > m.cols;
        m.r = std::min(m.rows, m.cols);
        m.k = std::max(m.rows, m.cols);
        m.tiles1 = round_up(m.rows, kEwTile) / kEwTile * (round_up(m.cols, kEwTile) / kEwTile);
        m.part = part;
        part += m.tiles1;
        m.small = allow_small && ns_small_smem_bytes(m.r, m.k) <= kSmallMaxSmem;
        if (m.small) {
            m.bucket = -1;
            m.slot = pl.nsmall++;
            m.r_pad64 = static_cast<int>(round_up(m.r, kEwTile));
            m.k_pad64 = static_cast<int>(round_up(m.k, kEwTile));
            pl.small_smem = std::max(pl.small_smem, ns_small_smem_bytes(m.r, m.k));
            pl.small_flops += 4.0 * m.r * m.r * m.k + 2.0 * m.r * m.r * m.r;
            continue;
        }
        const int rp = static_cast<int>(round_up(m.r, kPad));
        const int kp = static_cast<int>(round_up(m.k, kPad));
        int b = -1;
        for (size_t j = 0; j < pl.buckets.size(); ++j)
            if (pl.buckets[j].r_pad == rp && pl.buckets[j].k_pad == kp) b = static_cast<int>(j);
        if (b < 0) {
            BucketPlan bp;
            bp.r_pad = rp;
            bp.k_pad = kp;
            pl.buckets.push_back(bp);
            b = static_cast<int>(pl.buckets.size()) - 1;
        }
        BucketPlan& bp = pl.buckets[b];
        m.bucket = b;
        m.slot = bp.nmat++;
        const double r = m.r, k = m.k;
        bp.flops_gram += 2.0 * r * r * k;
        bp.flops_poly += 2.0 * r * r * r;
        bp.flops_update += 2.0 * r * r * k;
    }
    pl.total_tiles1 = part;
    size_t off = 0;
    // MUON_DEBUG_GUARD: a guard region before the first and after every region
    const bool guard = guard_enabled();
    pl.guards.clear();
    auto add_guard = [&]() {
        pl.guards.push_back(off);
        off = static_cast<size_t>(round_up(static_cast<long long>(off + kGuardBytes), 1024));
    };
    if (guard) add_guard();
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = static_cast<size_t>(round_up(static_cast<long long>(off + bytes), 1024));
        if (guard) add_guard();
        return o;
    };
    pl.off_partials = take(static_cast<size_t>(part) * sizeof(double));
    pl.off_sigma = take(static_cast<size_t>(count) * sizeof(float));
    size_t small_bytes = 0;
    for (MatPlan& m : pl.mats) {
        if (!m.small) continue;
        m.xoff = small_bytes;
        small_bytes += static_cast<size_t>(round_up(static_cast<long long>(m.r_pad64) * m.k_pad64 * 2, 256));
    }
    pl.off_small = take(small_bytes);
    pl.fp8 = fp8 && !pl.buckets.empty() ? 1 : 0;
    for (BucketPlan& bp : pl.buckets) {
        const size_t xb = static_cast<size_t>(bp.nmat) * bp.r_pad * bp.k_pad * 2;
        const size_t ab = static_cast<size_t>(bp.nmat) * bp.r_pad * bp.r_pad * 2;
        bp.x0 = take(xb);
        bp.x1 = take(xb);
        bp.a = take(ab);
        bp.b = take(ab);
        bp.x8 = pl.fp8 ? take(static_cast<size_t>(bp.nmat) * bp.r_pad * bp.k_pad) : 0;
    }
    pl.bytes = off;
}

// -------------------------------------------------------------- validation --
struct Interval {
    uintptr_t lo, hi;
    int writes;
    int mat;
};

int validate_dims(const int* rows, const int* cols, int count) {
    if (rows == nullptr || cols == nullptr) return fail(MUON_ERR_INVALID_ARG, "rows/cols is NULL");
    for (int i = 0; i < count; ++i) {
        if (rows[i] < 1 || cols[i] < 1 || rows[i] > MUON_MAX_DIM || cols[i] > MUON_MAX_DIM)
            return fail(MUON_ERR_INVALID_ARG, "matrix %d has shape %d x %d (each dim must be in [1, %d])",
                        i, rows[i], cols[i], MUON_MAX_DIM);
    }
    return MUON_OK;
}

int check_ptr(const void* p, const char* what, int i) {
    if (p == nullptr) return fail(MUON_ERR_INVALID_ARG, "%s[%d] is NULL", what, i);
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
        return fail(MUON_ERR_INVALID_ARG, "%s[%d] is not 16-byte aligned", what, i);
    return MUON_OK;
}

int check_overlaps(std::vector<Interval>& iv) {
    std::sort(iv.begin(), iv.end(), [](const Interval& x, const Interval& y) { return x.lo < y.lo; });
    // any overlap that involves a written range is an error
    uintptr_t run_hi = 0;
    int run_writes = 0, run_mat = -1;
    for (size_t i = 0; i < iv.size(); ++i) {
        if (i > 0 && iv[i].lo < run_hi && (iv[i].writes || run_writes))
            return fail(MUON_ERR_INVALID_ARG, "buffers of matrices %d and %d overlap", run_mat, iv[i].mat);
        if (i == 0 || iv[i].hi > run_hi) {
            run_hi = iv[i].hi;
            run_writes = iv[i].writes;
            run_mat = iv[i].mat;
        } else {
            run_writes |= iv[i].writes;
        }
    }
    return MUON_OK;
}

// -------------------------------------------------------------- workspace --
// MUON_FAULT_INJECT=alloc: every workspace allocation fails; alloc>N: those of
// more than N bytes fail (tests of the out-of-memory paths, made on the host).
bool fault_inject_alloc(size_t bytes) {
    const char* v = std::getenv("MUON_FAULT_INJECT");
    if (v == nullptr) return false;
    if (std::strcmp(v, "alloc") == 0) return true;
    if (std::strncmp(v, "alloc>", 6) == 0) return bytes > static_cast<size_t>(std::strtoull(v + 6, nullptr, 10));
    return false;
}

bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    return cudaStreamIsCapturing(s, &st) == cudaSuccess && st != cudaStreamCaptureStatusNone;
}

// During stream capture (a CUDA graph) the workspace must already exist (a
// first call outside the capture creates it), and ordering against work
// outside the graph is the caller's: the cross-stream event is neither waited
// on nor recorded.
int acquire_workspace(DeviceState& d, size_t need, cudaStream_t s, char** out) {
    const bool cap = capturing(s);
    if (cap && d.ws_bytes < need)
        return fail(MUON_ERR_UNSUPPORTED,
                    "the workspace (%zu bytes) must exist before stream capture: make one call with these "
                    "shapes outside the capture first", need);
    if (!cap && d.have_last && d.last_stream != s)
        MUON_CUDA_TRY(cudaStreamWaitEvent(s, d.last_use, 0), "cudaStreamWaitEvent");
    if (d.ws_bytes < need) {
        if (fault_inject_alloc(need))
            return fail(MUON_ERR_OOM, "workspace allocation of %zu bytes failed (injected)", need);
        if (d.ws != nullptr) {
            MUON_CUDA_TRY(cudaFreeAsync(d.ws, s), "cudaFreeAsync");
            d.ws = nullptr;
            d.ws_bytes = 0;
        }
        void* p = nullptr;
        cudaError_t e = cudaMallocAsync(&p, need, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(MUON_ERR_OOM, "workspace allocation of %zu bytes failed: %s", need,
                        cudaGetErrorString(e));
        }
        d.ws = p;
        d.ws_bytes = need;
    }
    *out = static_cast<char*>(d.ws);
    return MUON_OK;
}

void release_workspace_use(DeviceState& d, cudaStream_t s) {
    if (capturing(s)) return;
    cudaEventRecord(d.last_use, s);
    d.last_stream = s;
    d.have_last = true;
}

// ------------------------------------------------------------- TMA maps --
int encode_map(CUtensorMap* map, void* base, int cols, int rows, int nmat, int box_cols, int box_rows,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B, bool bytes = false) {
    const cuuint64_t esz = bytes ? 1 : 2;   // bf16, or one byte (the E4M3 copy)
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(nmat)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * esz,
                                   static_cast<cuuint64_t>(cols) * static_cast<cuuint64_t>(rows) * esz};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t es[3] = {1, 1, 1};
    const CUresult r = g_encode(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                                base, dims, strides, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MUON_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return MUON_OK;
}

// ---------------------------------------------------------------- run --
struct Call {
    bool step;                      // full Muon step (else ns-only)
    void* const* dst;               // W (step) or the matrices (ns)
    const void* const* src;         // G (step) or the matrices (ns)
    float* const* mom;              // M (step)
    void* const* oout;              // optional O copies (step)
    int count;
    int w_dtype, g_dtype, steps, nesterov;
    int g_count;                    // stacked gradients per matrix (1 for ns-only)
    std::vector<float> coef;        // (a, b, c) of every iteration, 3 * steps values
    float eps, lr, mu, wd;
    int fp8_gram = 0;               // tensor-core matrices: Gram product on E4M3 operands
};

enum Stage : int { kStageFront = 1, kStageNs = 2, kStageBack = 4, kStageAll = 7 };

// Weight-update scalars of one matrix, in double and rounded to fp32 once:
// dcy = 1 - lr*wd, s = lr * 0.2 * sqrt(max(m, n)).
void update_scalars(const Call& c, const MatPlan& m, float& dcy, float& s) {
    const double mx = std::max(m.rows, m.cols);
    dcy = static_cast<float>(1.0 - static_cast<double>(c.lr) * static_cast<double>(c.wd));
    s = static_cast<float>(static_cast<double>(c.lr) * 0.2 * std::sqrt(mx));
}

// Stages of one call: front = norm pass, finalize, pack; ns = the Newton-Schulz
// iterations (tensor-core GEMMs and the small-matrix kernel); back = unpack.
int run(const Call& c, const Plan& pl, DeviceState& d, char* ws, cudaStream_t s, int stages = kStageAll) {
    double* partials = reinterpret_cast<double*>(ws + pl.off_partials);
    float* sigma = reinterpret_cast<float*>(ws + pl.off_sigma);
    const int nb = static_cast<int>(pl.buckets.size());
    std::vector<__nv_bfloat16*> X0(nb), X1(nb), Am(nb), Bm(nb);
    for (int b = 0; b < nb; ++b) {
        X0[b] = reinterpret_cast<__nv_bfloat16*>(ws + pl.buckets[b].x0);
        X1[b] = reinterpret_cast<__nv_bfloat16*>(ws + pl.buckets[b].x1);
        Am[b] = reinterpret_cast<__nv_bfloat16*>(ws + pl.buckets[b].a);
        Bm[b] = reinterpret_cast<__nv_bfloat16*>(ws + pl.buckets[b].b);
    }
    __nv_bfloat16* small_base = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_small);
    // FP8 Gram: the E4M3 copy of each bucket's iterate (written with X0 by the pack and
    // with every later iterate by the update that writes it)
    const bool fp8 = c.fp8_gram != 0 && pl.fp8 != 0;
    std::vector<uint8_t*> X8(nb, nullptr);
    if (fp8)
        for (int b = 0; b < nb; ++b) X8[b] = reinterpret_cast<uint8_t*>(ws + pl.buckets[b].x8);
    if ((stages & kStageFront) && !pl.guards.empty()) {
        for (size_t g : pl.guards)
            if (cudaMemsetAsync(ws + g, 0xA5, kGuardBytes, s) != cudaSuccess)
                return fail(MUON_ERR_CUDA, "filling a guard region failed");
        if (guard_poison() && cudaMemsetAsync(ws + pl.guards[0], 0, 1, s) != cudaSuccess)
            return fail(MUON_ERR_CUDA, "poisoning a guard region failed");
    }
    const double gsz = (c.step && c.g_dtype == MUON_F32) ? 4.0 * c.g_count : 2.0 * (c.step ? c.g_count : 1);
    const double wsz = (c.step && c.w_dtype == MUON_F32) ? 4.0 : 2.0;

    std::unique_ptr<EwParams> ep(new EwParams());
    // matrices idx[0..n) (the front stage passes consecutive ones: sigma is indexed from idx[0])
    // with_x8: the pack of X0, which also writes the FP8 Gram's E4M3 copy
    auto fill_chunk = [&](const int* idx, int n, std::vector<__nv_bfloat16*>& xbuf, bool with_x8 = false) {
        EwParams& p = *ep;
        std::memset(&p, 0, sizeof(EwParams));
        p.nmats = n;
        p.src_dtype = (c.step && c.g_dtype == MUON_F32) ? kSrcF32 : kSrcBf16;
        p.dst_dtype = (c.step && c.w_dtype == MUON_F32) ? kSrcF32 : kSrcBf16;
        p.nesterov = c.nesterov;
        p.g_count = c.step ? c.g_count : 1;
        p.mu = c.mu;
        p.eps = c.eps;
        p.partials = partials;
        p.sigma = sigma;
        p.sigma_base = idx[0];
        for (int j = 0; j < n; ++j) {
            const int i = idx[j];
            const MatPlan& m = pl.mats[i];
            EwMat& e = p.m[j];
            e.src = c.src[i];
            e.mom = c.step ? c.mom[i] : nullptr;
            e.dst = c.dst[i];
            e.oout = (c.step && c.oout != nullptr) ? static_cast<__nv_bfloat16*>(c.oout[i]) : nullptr;
            if (m.small) {
                e.x = small_base + m.xoff / 2;
                e.ldx = m.k_pad64;
                e.xrows_pad = m.r_pad64;
            } else {
                const BucketPlan& bp = pl.buckets[m.bucket];
                e.x = xbuf[m.bucket] + static_cast<size_t>(m.slot) * bp.r_pad * bp.k_pad;
                e.ldx = bp.k_pad;
                e.xrows_pad = bp.r_pad;
            }
            e.part = m.part;
            e.rows = m.rows;
            e.cols = m.cols;
            e.trans = m.trans;
            e.vec = (m.cols % 8) == 0;
            // the pack writes X0's E4M3 copy for the FP8 Gram (tensor-core matrices only)
            e.x8 = (with_x8 && fp8 && !m.small)
                       ? X8[m.bucket] + static_cast<size_t>(m.slot) * pl.buckets[m.bucket].r_pad * pl.buckets[m.bucket].k_pad
                       : nullptr;
            if (c.step) update_scalars(c, m, e.dcy, e.s);
        }
        p.fp8 = fp8 ? 1 : 0;
    };
    // tiles in input space (norm pass, unpack) or in iterate space (pack)
    auto set_tiles = [&](const int* idx, bool iterate_space) {
        EwParams& p = *ep;
        int t = 0;
        for (int j = 0; j < p.nmats; ++j) {
            p.m[j].tile0 = t;
            const MatPlan& m = pl.mats[idx[j]];
            const int xr = m.small ? m.r_pad64 : pl.buckets[m.bucket].r_pad;
            const int xk = m.small ? m.k_pad64 : pl.buckets[m.bucket].k_pad;
            t += iterate_space ? (xr / kEwTile) * (xk / kEwTile) : static_cast<int>(m.tiles1);
        }
        p.total_tiles = t;
        return t;
    };

    std::vector<int> all(c.count);
    for (int i = 0; i < c.count; ++i) all[i] = i;

    // -- momentum / normalisation / pack, chunked (the pack also writes X0's E4M3 copy for the FP8 Gram)
    for (int start = 0; (stages & kStageFront) && start < c.count; start += kEwMaxMats) {
        const int n = std::min(kEwMaxMats, c.count - start);
        fill_chunk(&all[start], n, X0, true);
        double elems = 0, xelems = 0, x8elems = 0;
        for (int j = 0; j < n; ++j) {
            const MatPlan& m = pl.mats[start + j];
            elems += static_cast<double>(m.rows) * m.cols;
            xelems += static_cast<double>(m.r) * m.k;
            if (fp8 && !m.small) x8elems += static_cast<double>(m.r) * m.k;
        }
        int tiles = set_tiles(&all[start], false);
        int rc = launch(kKNorm, 0.0, elems * (c.step ? gsz + 8.0 : 2.0), s, [&] {
            return c.step ? launch_momentum_norm(*ep, d.sms, s) : launch_input_norm(*ep, d.sms, s);
        });
        if (rc != MUON_OK) return rc;
        rc = launch(kKFinalize, 0.0, 8.0 * tiles, s, [&] { return launch_norm_finalize(*ep, s); });
        if (rc != MUON_OK) return rc;
        tiles = set_tiles(&all[start], true);
        rc = launch(kKPack, 0.0, elems * (c.step ? gsz + 4.0 : 2.0) + 2.0 * xelems + x8elems, s,
                    [&] { return launch_pack(*ep, d.sms, c.step, s); });
        if (rc != MUON_OK) return rc;
    }

    // -- Newton-Schulz iterations: three tensor-core launches per iteration
    std::vector<int> order(nb);
    for (int b = 0; b < nb; ++b) order[b] = b;
    std::sort(order.begin(), order.end(), [&](int x, int y) {
        const BucketPlan &bx = pl.buckets[x], &by = pl.buckets[y];
        return static_cast<double>(bx.r_pad) * bx.k_pad > static_cast<double>(by.r_pad) * by.k_pad;
    });
    std::unique_ptr<GemmParams> gp(new GemmParams());
    // Pair-CTA tiles: 256 x 256 outputs on two SMs
    // the update product on clusters of two pairs sharing A by multicast
    const bool multicast = env_flag("MUON_GEMM_MULTICAST");
    // the symmetric products store only their upper tiles (their consumers read the
    // rest from the transpose); MUON_GEMM_MIRROR=1, or multicast, keeps full storage
    const bool upper_only = !multicast && !env_flag("MUON_GEMM_MIRROR");
    // the update's epilogue input and output moved by TMA
    const bool tma_epilogue = fp8 || !env_flag("MUON_GEMM_NO_TMA_EPI");
    const int tm_rows = 256;   // output rows per tile
    const int tn_cols = kBN;   // output columns per tile
    const int a_box = 128;     // rows of the A operand one CTA loads
    const int b_box = 128;     // rows (K-major) of the B operand one CTA loads
    // the last update writes W (or O) directly when every launch group's
    // matrices fit the kernel's table
    std::vector<std::vector<int>> bucket_mats(nb);
    for (int i = 0; i < c.count; ++i)
        if (!pl.mats[i].small) bucket_mats[pl.mats[i].bucket].push_back(i);
    bool fuse_final = c.steps > 0 && nb > 0 && !env_flag("MUON_NO_FUSED_UPDATE");
    for (int g0 = 0; fuse_final && g0 < nb; g0 += kMaxBuckets) {
        int n = 0;
        for (int gi = 0; gi < std::min(kMaxBuckets, nb - g0); ++gi) n += pl.buckets[order[g0 + gi]].nmat;
        if (n > kFinalMaxMats) fuse_final = false;
    }
    const int fin_kind = !c.step ? kFinStore : (c.w_dtype == MUON_F32 ? kFinWF32 : kFinWBf16);
    // MUON_TEST_STALL=1 (tests only): the first tensor-core launch of the call issues no
    // MMA and waits at most 50 ms, so its bounded waits expire and it reports
    // MUON_ERR_TIMEOUT through muon_device_status
    bool stall_next = env_flag("MUON_TEST_STALL");
    std::unique_ptr<FinalParams> fp(fuse_final ? new FinalParams() : nullptr);
    int cur = 0;
    for (int it = 0; (stages & kStageNs) && it < c.steps; ++it) {
        std::vector<__nv_bfloat16*>& Xc = cur ? X1 : X0;
        std::vector<__nv_bfloat16*>& Xn = cur ? X0 : X1;
        for (int mode = kGram; mode <= kUpdate; ++mode) {
            for (int g0 = 0; g0 < nb; g0 += kMaxBuckets) {
                const int ng = std::min(kMaxBuckets, nb - g0);
                // FP8 Gram: its operands are the E4M3 copy of this iterate, written with it
                const bool f8 = fp8 && mode == kGram;
                GemmParams& p = *gp;
                std::memset(&p, 0, sizeof(GemmParams));
                p.nbuckets = ng;
                p.mode = mode;
                p.upper_only = upper_only ? 1 : 0;
                p.fp8 = f8 ? 1 : 0;
                // the update before an FP8 Gram writes that Gram's operand too
                p.fp8_next = (fp8 && mode == kUpdate && it + 1 < c.steps) ? 1 : 0;
                if (stall_next) {
                    p.stall = 1;
                    p.wait_ns = 50000000ull;
                    stall_next = false;
                }
                p.a = c.coef[3 * it];
                p.bcoef = c.coef[3 * it + 1];
                p.c = c.coef[3 * it + 2];
                int tile = 0, items = 0;
                double flops = 0;
                for (int gi = 0; gi < ng; ++gi) {
                    const int b = order[g0 + gi];
                    const BucketPlan& bp = pl.buckets[b];
                    GemmBucket& B = p.b[gi];
                    const int rp = bp.r_pad, kp = bp.k_pad;
                    int rc = MUON_OK;
                    if (f8) {
                        // E4M3 copy of X: 128 elements (128 bytes) of K per stage
                        rc = encode_map(&B.tmA, X8[b], kp, rp, bp.nmat, 2 * kBK, a_box, CU_TENSOR_MAP_SWIZZLE_128B, true);
                        if (rc == MUON_OK)
                            rc = encode_map(&B.tmB, X8[b], kp, rp, bp.nmat, 2 * kBK, b_box, CU_TENSOR_MAP_SWIZZLE_128B, true);
                        B.out = Am[b];
                        B.epi = nullptr;
                        B.mat_stride = static_cast<long long>(rp) * rp;
                        B.ld = rp;
                        B.mt = rp / tm_rows;
                        B.nt = rp / tn_cols;
                        B.kblocks = kp / (2 * kBK);
                        B.tiles_per_mat = B.nt * (B.nt + 1) / 2;
                        flops += bp.flops_gram;
                    } else if (mode == kGram || mode == kPoly) {
                        __nv_bfloat16* src = mode == kGram ? Xc[b] : Am[b];
                        const int kdim = mode == kGram ? kp : rp;
                        rc = encode_map(&B.tmA, src, kdim, rp, bp.nmat, kBK, a_box);
                        if (rc == MUON_OK) rc = encode_map(&B.tmB, src, kdim, rp, bp.nmat, kBK, b_box);
                        // polynomial: A (upper tiles only) also as 64 x 64 blocks of its transpose
                        if (rc == MUON_OK && mode == kPoly && upper_only)
                            rc = encode_map(&B.tmT, Am[b], rp, rp, bp.nmat, 64, kBK);
                        B.out = mode == kGram ? Am[b] : Bm[b];
                        B.epi = mode == kGram ? nullptr : Am[b];
                        B.mat_stride = static_cast<long long>(rp) * rp;
                        B.ld = rp;
                        B.mt = rp / tm_rows;
                        B.nt = rp / tn_cols;
                        B.kblocks = kdim / kBK;
                        B.tiles_per_mat = B.nt * (B.nt + 1) / 2;
                        flops += mode == kGram ? bp.flops_gram : bp.flops_poly;
                    } else {
                        rc = encode_map(&B.tmA, Bm[b], rp, rp, bp.nmat, kBK, a_box);
                        if (rc == MUON_OK) rc = encode_map(&B.tmB, Xc[b], kp, rp, bp.nmat, 64, kBK);
                        // B (upper tiles only) also as 64 x 64 blocks of its transpose
                        if (rc == MUON_OK && upper_only) rc = encode_map(&B.tmT, Bm[b], rp, rp, bp.nmat, 64, kBK);
                        // epilogue input X and output X' in 32 x 32 blocks
                        if (rc == MUON_OK)
                            rc = encode_map(&B.tmE, Xc[b], kp, rp, bp.nmat, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
                        if (rc == MUON_OK)
                            rc = encode_map(&B.tmO, Xn[b], kp, rp, bp.nmat, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
                        // before an FP8 Gram: X' * 2^8 in E4M3, 32 x 32 byte blocks (rows of 32 bytes)
                        if (rc == MUON_OK && p.fp8_next)
                            rc = encode_map(&B.tmQ, X8[b], kp, rp, bp.nmat, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE, true);
                        B.out = Xn[b];
                        B.epi = Xc[b];
                        B.mat_stride = static_cast<long long>(rp) * kp;
                        B.ld = kp;
                        B.mt = rp / tm_rows;
                        B.nt = kp / tn_cols;
                        B.kblocks = rp / kBK;
                        B.tiles_per_mat = B.mt * B.nt;
                        B.nt2 = (B.nt + 1) / 2;
                        B.item0 = items;
                        items += B.mt * B.nt2 * bp.nmat;
                        flops += bp.flops_update;
                    }
                    if (rc != MUON_OK) return rc;
                    B.nmat = bp.nmat;
                    B.tile0 = tile;
                    tile += B.tiles_per_mat * bp.nmat;
                }
                p.total_tiles = tile;
                p.total_items = items;
                const bool final_launch = fuse_final && mode == kUpdate && it == c.steps - 1;
                if (final_launch) {
                    int nf = 0;
                    for (int gi = 0; gi < ng; ++gi) {
                        const int b = order[g0 + gi];
                        p.b[gi].fin0 = nf;
                        for (int i : bucket_mats[b]) {
                            const MatPlan& m = pl.mats[i];
                            FinalMat& f = fp->m[nf++];
                            f.w = c.dst[i];
                            f.oout = (c.step && c.oout != nullptr) ? static_cast<__nv_bfloat16*>(c.oout[i]) : nullptr;
                            f.dcy = f.s = 0.0f;
                            if (c.step) update_scalars(c, m, f.dcy, f.s);
                            f.rows = m.rows;
                            f.cols = m.cols;
                            f.trans = m.trans;
                            f.vec = (m.cols % 8) == 0;
                        }
                    }
                }
                const int kind = final_launch ? kKFinal : (mode == kGram ? kKGram : (mode == kPoly ? kKPoly : kKUpdate));
                int rc;
                if (final_launch) {
                    rc = launch(kind, flops, 0.0, s,
                                [&] { return launch_gemm_pair_final(*gp, *fp, fin_kind, d.sms, multicast, s); });
                } else {
                    rc = launch(kind, flops, 0.0, s,
                                [&] { return launch_gemm_pair(*gp, d.sms, multicast, tma_epilogue, s); });
                }
                if (rc != MUON_OK) return rc;
            }
        }
        cur ^= 1;
    }

    // -- small matrices: every iteration in one launch
    if ((stages & kStageNs) && pl.nsmall > 0 && c.steps > 0) {
        std::unique_ptr<SmallParams> sp(new SmallParams());
        int n = 0;
        auto flush = [&]() -> int {
            if (n == 0) return MUON_OK;
            sp->nmats = n;
            sp->steps = c.steps;
            for (int j = 0; j < 3 * c.steps; ++j) sp->coef[j] = c.coef[j];
            double flops = 0;
            for (int j = 0; j < n; ++j) {
                const double r = sp->m[j].r, k = sp->m[j].k;
                flops += c.steps * (4.0 * r * r * k + 2.0 * r * r * r);
            }
            const int rc = launch(kKSmall, flops, 0.0, s, [&] { return launch_ns_small(*sp, pl.small_smem, s); });
            n = 0;
            return rc;
        };
        for (const MatPlan& m : pl.mats) {
            if (!m.small) continue;
            SmallMat& sm = sp->m[n++];
            sm.x = small_base + m.xoff / 2;
            sm.r = m.r;
            sm.k = m.k;
            sm.ldx = m.k_pad64;
            sm.pad_ = 0;
            if (n == kSmallMaxMats) {
                const int rc = flush();
                if (rc != MUON_OK) return rc;
            }
        }
        const int rc = flush();
        if (rc != MUON_OK) return rc;
    }

    // -- weight update (or store of O), chunked, of the matrices the fused last
    // update did not cover: the final iterate is X1 after an odd number of
    // iterations (the ping-pong parity does not depend on stages)
    if (!(stages & kStageNs)) cur = c.steps & 1;
    std::vector<int> back;
    for (int i = 0; i < c.count; ++i)
        if (!fuse_final || pl.mats[i].small) back.push_back(i);
    const int nback = static_cast<int>(back.size());
    for (int start = 0; (stages & kStageBack) && start < nback; start += kEwMaxMats) {
        const int n = std::min(kEwMaxMats, nback - start);
        fill_chunk(&back[start], n, cur ? X1 : X0);
        double elems = 0;
        for (int j = 0; j < n; ++j) elems += static_cast<double>(pl.mats[back[start + j]].rows) * pl.mats[back[start + j]].cols;
        const int tiles = set_tiles(&back[start], false);
        const int rc = launch(kKUnpack, 0.0, elems * (c.step ? 2.0 + 2.0 * wsz : 4.0), s,
                              [&] { return launch_unpack(*ep, d.sms, c.step, s); });
        if (rc != MUON_OK) return rc;
    }
    // -- debug guard regions: still intact after every kernel of the call?
    if ((stages & kStageBack) && !pl.guards.empty()) {
        std::unique_ptr<GuardParams> gp(new GuardParams());
        for (size_t i0 = 0; i0 < pl.guards.size(); i0 += kMaxGuards) {
            const int n = static_cast<int>(std::min<size_t>(kMaxGuards, pl.guards.size() - i0));
            gp->base = ws;
            gp->n = n;
            for (int j = 0; j < n; ++j) gp->off[j] = pl.guards[i0 + j];
            if (launch_guard_check(*gp, s) != cudaSuccess) return fail(MUON_ERR_CUDA, "guard check launch failed");
        }
    }
    return MUON_OK;
}

// (a, b, c) of every iteration: `coeffs` is NULL (defaults), one triple used at
// every step, or (per_step) one triple per step.
void fill_coef(Call& c, const float* coeffs, int per_step) {
    c.coef.clear();
    if (c.steps < 0 || c.steps > kMaxSteps) return;   // rejected by validation
    for (int t = 0; t < c.steps; ++t)
        for (int j = 0; j < 3; ++j)
            c.coef.push_back(coeffs == nullptr ? kDefaultCoeffs[j] : coeffs[(per_step ? 3 * t : 0) + j]);
}

// A large batch runs as two parts (by nominal work) on two streams: the
// second part's norm/pack overlaps the first part's Newton-Schulz GEMMs and
// the first part's back stage (unpack) overlaps the second part's GEMMs.
// Returns the size of the first part, or 0 when the batch is too small to gain
// from it.  MUON_NO_SPLIT=1 keeps every call on the caller's stream.
constexpr double kSplitMinFlops = 2e12;
// Share of the work in the first part.  Only the first part's front (norm
// and pack) runs alone; the second part's front hides under the first part's
// GEMMs as long as it is shorter than them.  MUON_SPLIT_FRACTION overrides it
// (0.05 .. 0.95; tuning).
constexpr double kSplitFraction = 0.5;
double split_fraction() {
    const char* v = std::getenv("MUON_SPLIT_FRACTION");
    if (v == nullptr || v[0] == '\0') return kSplitFraction;
    const double f = std::atof(v);
    return (f >= 0.05 && f <= 0.95) ? f : kSplitFraction;
}

int split_point(const int* rows, const int* cols, int count) {
    if (count < 4 || env_flag("MUON_NO_SPLIT")) return 0;
    std::vector<double> w(count);
    double tot = 0;
    for (int i = 0; i < count; ++i) {
        const double r = std::min(rows[i], cols[i]), k = std::max(rows[i], cols[i]);
        w[i] = 4.0 * r * r * k + 2.0 * r * r * r;
        tot += w[i];
    }
    if (tot * 5 < kSplitMinFlops) return 0;
    const double frac = split_fraction();
    double acc = 0;
    for (int i = 0; i < count - 1; ++i) {
        acc += w[i];
        if (acc >= frac * tot) return i + 1;
    }
    return count - 1;
}

size_t plan_bytes(const int* rows, const int* cols, int count, int n1, bool fp8 = false) {
    Plan a;
    build_plan(rows, cols, n1 > 0 ? n1 : count, a, fp8);
    if (n1 <= 0) return a.bytes;
    Plan b;
    build_plan(rows + n1, cols + n1, count - n1, b, fp8);
    return static_cast<size_t>(round_up(static_cast<long long>(a.bytes), 1024)) + b.bytes;
}

Call sub_call(const Call& c, int i0, int n) {
    Call h = c;
    h.count = n;
    h.dst = c.dst + i0;
    h.src = c.src + i0;
    h.mom = c.mom ? c.mom + i0 : nullptr;
    h.oout = c.oout ? c.oout + i0 : nullptr;
    return h;
}

int run_split(const Call& c, const int* rows, const int* cols, int n1, DeviceState& d, char* ws, cudaStream_t s) {
    Plan p1, p2;
    build_plan(rows, cols, n1, p1, c.fp8_gram != 0);
    build_plan(rows + n1, cols + n1, c.count - n1, p2, c.fp8_gram != 0);
    char* ws2 = ws + round_up(static_cast<long long>(p1.bytes), 1024);
    const Call h1 = sub_call(c, 0, n1), h2 = sub_call(c, n1, c.count - n1);
    cudaStream_t a = d.aux;
    int rc;
    MUON_CUDA_TRY(cudaEventRecord(d.ev[0], s), "cudaEventRecord");              // fork
    if ((rc = run(h1, p1, d, ws, s, kStageFront)) != MUON_OK) return rc;
    MUON_CUDA_TRY(cudaEventRecord(d.ev[1], s), "cudaEventRecord");              // first half packed
    MUON_CUDA_TRY(cudaStreamWaitEvent(a, d.ev[1], 0), "cudaStreamWaitEvent");
    if ((rc = run(h2, p2, d, ws2, a, kStageFront)) != MUON_OK) return rc;      // overlaps GEMMs of half 1
    if ((rc = run(h1, p1, d, ws, s, kStageNs)) != MUON_OK) return rc;
    MUON_CUDA_TRY(cudaEventRecord(d.ev[2], s), "cudaEventRecord");              // GEMMs of half 1 done
    MUON_CUDA_TRY(cudaStreamWaitEvent(a, d.ev[2], 0), "cudaStreamWaitEvent");
    if ((rc = run(h2, p2, d, ws2, a, kStageNs | kStageBack)) != MUON_OK) return rc;
    if ((rc = run(h1, p1, d, ws, s, kStageBack)) != MUON_OK) return rc;       // overlaps GEMMs of half 2
    MUON_CUDA_TRY(cudaEventRecord(d.ev[3], a), "cudaEventRecord");              // join
    MUON_CUDA_TRY(cudaStreamWaitEvent(s, d.ev[3], 0), "cudaStreamWaitEvent");
    return MUON_OK;
}

// Consecutive groups of matrices, each the longest run whose plan fits
// `budget` bytes: group starts, then count.  False (and *big) if one matrix
// alone does not fit.
bool make_groups(const int* rows, const int* cols, int count, size_t budget, std::vector<int>& groups, int* big,
                 bool fp8) {
    groups.clear();
    for (int i0 = 0; i0 < count;) {
        if (plan_bytes(rows + i0, cols + i0, 1, 0, fp8) > budget) {
            *big = i0;
            return false;
        }
        int lo = 1, hi = count - i0;   // the longest fitting run is in [lo, hi]
        while (lo < hi) {
            const int mid = lo + (hi - lo + 1) / 2;
            if (plan_bytes(rows + i0, cols + i0, mid, 0, fp8) <= budget) lo = mid; else hi = mid - 1;
        }
        groups.push_back(i0);
        i0 += lo;
    }
    groups.push_back(count);
    return true;
}

// The groups one after the other on `s`, all on the workspace `ws`.
int run_groups(const Call& c, const int* rows, const int* cols, const std::vector<int>& groups, DeviceState& d,
               char* ws, cudaStream_t s) {
    for (size_t gi = 0; gi + 1 < groups.size(); ++gi) {
        const int i0 = groups[gi], n = groups[gi + 1] - i0;
        Plan pg;
        build_plan(rows + i0, cols + i0, n, pg, c.fp8_gram != 0);
        const int rc = run(sub_call(c, i0, n), pg, d, ws, s);
        if (rc != MUON_OK) return rc;
    }
    return MUON_OK;
}

int validate_and_run(Call& c, const int* rows, const int* cols, void* user_ws, size_t user_ws_bytes,
                     cudaStream_t s) {
    if (c.count < 0) return fail(MUON_ERR_INVALID_ARG, "count is negative");
    if (c.count == 0) return MUON_OK;
    if (c.dst == nullptr || c.src == nullptr || (c.step && c.mom == nullptr))
        return fail(MUON_ERR_INVALID_ARG, "a pointer array is NULL");
    int rc = validate_dims(rows, cols, c.count);
    if (rc != MUON_OK) return rc;
    if (c.steps < 0 || c.steps > kMaxSteps)
        return fail(MUON_ERR_INVALID_ARG, "steps = %d (must be in [0, %d])", c.steps, kMaxSteps);
    for (size_t j = 0; j < c.coef.size(); ++j)
        if (!std::isfinite(c.coef[j])) return fail(MUON_ERR_INVALID_ARG, "coefficient %d is not finite", static_cast<int>(j));
    if (!(c.eps >= 0.0f) || !std::isfinite(c.eps)) return fail(MUON_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (c.step) {
        if (!std::isfinite(c.lr) || !std::isfinite(c.mu) || !std::isfinite(c.wd))
            return fail(MUON_ERR_INVALID_ARG, "lr, mu and wd must be finite");
        if ((c.w_dtype != MUON_BF16 && c.w_dtype != MUON_F32) || (c.g_dtype != MUON_BF16 && c.g_dtype != MUON_F32))
            return fail(MUON_ERR_INVALID_ARG, "unknown dtype");
        if (c.nesterov != 0 && c.nesterov != 1) return fail(MUON_ERR_INVALID_ARG, "nesterov must be 0 or 1");
        if (c.g_count < 1 || c.g_count > 64) return fail(MUON_ERR_INVALID_ARG, "g_count = %d (must be in [1, 64])", c.g_count);
    }
    std::vector<Interval> iv;
    iv.reserve(static_cast<size_t>(c.count) * 3);
    for (int i = 0; i < c.count; ++i) {
        const uintptr_t n = static_cast<uintptr_t>(rows[i]) * static_cast<uintptr_t>(cols[i]);
        if (c.step) {
            if ((rc = check_ptr(c.dst[i], "W", i)) != MUON_OK) return rc;
            if ((rc = check_ptr(c.src[i], "G", i)) != MUON_OK) return rc;
            if ((rc = check_ptr(c.mom[i], "M", i)) != MUON_OK) return rc;
            const uintptr_t w = reinterpret_cast<uintptr_t>(c.dst[i]);
            const uintptr_t g = reinterpret_cast<uintptr_t>(c.src[i]);
            const uintptr_t m = reinterpret_cast<uintptr_t>(c.mom[i]);
            iv.push_back({w, w + n * (c.w_dtype == MUON_F32 ? 4 : 2), 1, i});
            iv.push_back({g, g + n * (c.g_dtype == MUON_F32 ? 4 : 2) * static_cast<uintptr_t>(c.g_count), 0, i});
            iv.push_back({m, m + n * 4, 1, i});
            if (c.oout != nullptr) {
                if ((rc = check_ptr(c.oout[i], "o_out", i)) != MUON_OK) return rc;
                const uintptr_t o = reinterpret_cast<uintptr_t>(c.oout[i]);
                iv.push_back({o, o + n * 2, 1, i});
            }
        } else {
            if (c.dst[i] != c.src[i]) return fail(MUON_ERR_INVALID_ARG, "internal: ns src != dst");
            if ((rc = check_ptr(c.dst[i], "ptrs", i)) != MUON_OK) return rc;
            const uintptr_t x = reinterpret_cast<uintptr_t>(c.dst[i]);
            iv.push_back({x, x + n * 2, 1, i});
        }
    }
    if ((rc = check_overlaps(iv)) != MUON_OK) return rc;
    if (user_ws != nullptr && reinterpret_cast<uintptr_t>(user_ws) % 256 != 0)
        return fail(MUON_ERR_INVALID_ARG, "workspace is not 256-byte aligned");

    const int n1 = split_point(rows, cols, c.count);
    const bool fp8 = c.fp8_gram != 0;
    const size_t need = plan_bytes(rows, cols, c.count, n1, fp8);

    // A caller workspace smaller than the batch needs: consecutive groups of
    // matrices that fit, one after the other on `s` (each matrix's result does
    // not depend on the rest of its batch).
    std::vector<int> groups;
    if (user_ws != nullptr && user_ws_bytes < need) {
        int big = -1;
        if (!make_groups(rows, cols, c.count, user_ws_bytes, groups, &big, fp8))
            return fail(MUON_ERR_OOM, "caller workspace has %zu bytes; matrix %d alone needs %zu", user_ws_bytes,
                        big, plan_bytes(rows + big, cols + big, 1, 0, fp8));
    }
    Plan pl;
    if (n1 == 0 && groups.empty()) build_plan(rows, cols, c.count, pl, fp8);

    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* d = nullptr;
    if ((rc = device_state(&d)) != MUON_OK) return rc;
    char* ws = nullptr;
    if (!groups.empty()) return run_groups(c, rows, cols, groups, *d, static_cast<char*>(user_ws), s);
    if (user_ws != nullptr) {
        ws = static_cast<char*>(user_ws);
    } else if ((rc = acquire_workspace(*d, need, s, &ws)) != MUON_OK) {
        // The workspace for the whole batch cannot be allocated: try groupings of
        // ever smaller largest group until one finds memory (not during a
        // capture, whose workspace must exist beforehand).  The largest group's
        // plan shrinks with every attempt, so this ends once a single matrix no
        // longer fits.
        if (rc != MUON_ERR_OOM || capturing(s) || c.count < 2) return rc;
        const std::string first = muon_last_error();
        for (size_t budget = need - 1; budget > 0;) {
            int big = -1;
            if (!make_groups(rows, cols, c.count, budget, groups, &big, fp8)) break;
            size_t gneed = 0;
            for (size_t gi = 0; gi + 1 < groups.size(); ++gi)
                gneed = std::max(gneed, plan_bytes(rows + groups[gi], cols + groups[gi], groups[gi + 1] - groups[gi], 0,
                                                   fp8));
            if (acquire_workspace(*d, gneed, s, &ws) != MUON_OK) {
                budget = gneed - 1;
                continue;
            }
            rc = run_groups(c, rows, cols, groups, *d, ws, s);
            release_workspace_use(*d, s);
            return rc;
        }
        return fail(MUON_ERR_OOM, "%s; no grouping of the batch found memory either", first.c_str());
    }
    rc = n1 > 0 ? run_split(c, rows, cols, n1, *d, ws, s) : run(c, pl, *d, ws, s);
    if (user_ws == nullptr) release_workspace_use(*d, s);
    return rc;
}

}  // namespace

// Newton-Schulz of a batch on a caller-supplied device workspace (nothing is
// allocated); used by the static-scratch entry point.
int ns5_batched_on_workspace(void* const* ptrs, const int* rows, const int* cols, int count, int steps,
                             const float* coeffs, void* ws, size_t ws_bytes, cudaStream_t stream) {
    Call c{};
    c.step = false;
    c.dst = ptrs;
    c.src = reinterpret_cast<const void* const*>(ptrs);
    c.mom = nullptr;
    c.count = count;
    c.steps = steps;
    c.nesterov = 1;
    fill_coef(c, coeffs, 0);
    c.eps = 1e-7f;
    return validate_and_run(c, rows, cols, ws, ws_bytes, stream);
}

int set_last_error(int status, const char* msg) { return fail(status, "%s", msg); }

}  // namespace muon

using namespace muon;

extern "C" {

void muon_step_opts_init(muon_step_opts* o) {
    if (o == nullptr) return;
    o->w_dtype = MUON_BF16;
    o->g_dtype = MUON_BF16;
    o->steps = 5;
    o->coeffs = nullptr;
    o->eps = 1e-7f;
    o->nesterov = 1;
    o->workspace = nullptr;
    o->workspace_bytes = 0;
    o->o_out = nullptr;
    o->coeffs_per_step = 0;
    o->g_count = 1;
    o->ns_fp8_gram = 0;
}

int muon_ns5_batched(void* const* ptrs, const int* rows, const int* cols, int count, int steps,
                     const float* coeffs, cudaStream_t stream) {
    Call c{};
    c.step = false;
    c.dst = ptrs;
    c.src = reinterpret_cast<const void* const*>(ptrs);
    c.mom = nullptr;
    c.count = count;
    c.steps = steps;
    c.nesterov = 1;
    fill_coef(c, coeffs, 0);
    c.eps = 1e-7f;
    return validate_and_run(c, rows, cols, nullptr, 0, stream);
}

int muon_ns_batched_ex(void* const* ptrs, const int* rows, const int* cols, int count, int steps,
                       const float* coeffs, int coeffs_per_step, cudaStream_t stream) {
    if (coeffs_per_step != 0 && coeffs_per_step != 1)
        return fail(MUON_ERR_INVALID_ARG, "coeffs_per_step must be 0 or 1");
    Call c{};
    c.step = false;
    c.dst = ptrs;
    c.src = reinterpret_cast<const void* const*>(ptrs);
    c.mom = nullptr;
    c.count = count;
    c.steps = steps;
    c.nesterov = 1;
    fill_coef(c, coeffs, coeffs_per_step);
    c.eps = 1e-7f;
    return validate_and_run(c, rows, cols, nullptr, 0, stream);
}

int muon_step_ex(void* const* W, const void* const* G, float* const* M, const int* rows, const int* cols,
                 int count, float lr, float mu, float wd, const muon_step_opts* opts, cudaStream_t stream) {
    muon_step_opts o;
    muon_step_opts_init(&o);
    if (opts != nullptr) o = *opts;
    Call c{};
    c.step = true;
    c.dst = W;
    c.src = G;
    c.mom = M;
    c.oout = o.o_out;
    c.count = count;
    c.w_dtype = o.w_dtype;
    c.g_dtype = o.g_dtype;
    c.steps = o.steps;
    c.nesterov = o.nesterov;
    c.g_count = o.g_count;
    if (o.ns_fp8_gram != 0 && o.ns_fp8_gram != 1)
        return set_last_error(MUON_ERR_INVALID_ARG, "ns_fp8_gram must be 0 or 1");
    c.fp8_gram = o.ns_fp8_gram;
    if (o.coeffs_per_step != 0 && o.coeffs_per_step != 1)
        return fail(MUON_ERR_INVALID_ARG, "coeffs_per_step must be 0 or 1");
    fill_coef(c, o.coeffs, o.coeffs_per_step);
    c.eps = o.eps;
    c.lr = lr;
    c.mu = mu;
    c.wd = wd;
    return validate_and_run(c, rows, cols, o.workspace, o.workspace_bytes, stream);
}

int muon_step(void* const* W, const void* const* G, float* const* M, const int* rows, const int* cols,
              int count, float lr, float mu, float wd, cudaStream_t stream) {
    return muon_step_ex(W, G, M, rows, cols, count, lr, mu, wd, nullptr, stream);
}

int muon_adamw_step(void* const* P, const void* const* G, float* const* M, float* const* V,
                    const long long* numel, int count, int p_dtype, int g_dtype, float lr, float beta1,
                    float beta2, float eps, float wd, int step, cudaStream_t stream) {
    if (count < 0) return fail(MUON_ERR_INVALID_ARG, "count is negative");
    if (count == 0) return MUON_OK;
    if (P == nullptr || G == nullptr || M == nullptr || V == nullptr || numel == nullptr)
        return fail(MUON_ERR_INVALID_ARG, "a pointer array is NULL");
    if ((p_dtype != MUON_BF16 && p_dtype != MUON_F32) || (g_dtype != MUON_BF16 && g_dtype != MUON_F32))
        return fail(MUON_ERR_INVALID_ARG, "unknown dtype");
    if (!std::isfinite(lr) || !std::isfinite(eps) || !std::isfinite(wd) || !(beta1 >= 0.0f && beta1 < 1.0f) ||
        !(beta2 >= 0.0f && beta2 < 1.0f) || !(eps >= 0.0f))
        return fail(MUON_ERR_INVALID_ARG, "lr, eps, wd must be finite, eps >= 0 and betas in [0, 1)");
    if (step < 1) return fail(MUON_ERR_INVALID_ARG, "step must be >= 1");
    const size_t psz = p_dtype == MUON_F32 ? 4 : 2, gsz = g_dtype == MUON_F32 ? 4 : 2;
    std::vector<Interval> iv;
    int rc;
    for (int i = 0; i < count; ++i) {
        if (numel[i] < 0) return fail(MUON_ERR_INVALID_ARG, "numel[%d] is negative", i);
        if (numel[i] == 0) continue;
        if ((rc = check_ptr(P[i], "P", i)) != MUON_OK) return rc;
        if ((rc = check_ptr(G[i], "G", i)) != MUON_OK) return rc;
        if ((rc = check_ptr(M[i], "M", i)) != MUON_OK) return rc;
        if ((rc = check_ptr(V[i], "V", i)) != MUON_OK) return rc;
        const uintptr_t n = static_cast<uintptr_t>(numel[i]);
        const uintptr_t p = reinterpret_cast<uintptr_t>(P[i]), g = reinterpret_cast<uintptr_t>(G[i]),
                        m = reinterpret_cast<uintptr_t>(M[i]), v = reinterpret_cast<uintptr_t>(V[i]);
        iv.push_back({p, p + n * psz, 1, i});
        iv.push_back({g, g + n * gsz, 0, i});
        iv.push_back({m, m + n * 4, 1, i});
        iv.push_back({v, v + n * 4, 1, i});
    }
    if ((rc = check_overlaps(iv)) != MUON_OK) return rc;

    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* d = nullptr;
    if ((rc = device_state(&d)) != MUON_OK) return rc;
    std::unique_ptr<AdamWParams> ap(new AdamWParams());
    const double t = step;
    const float b1c = static_cast<float>(1.0 - static_cast<double>(beta1));
    const float b2c = static_cast<float>(1.0 - static_cast<double>(beta2));
    const float dcy = static_cast<float>(1.0 - static_cast<double>(lr) * static_cast<double>(wd));
    const float step_size = static_cast<float>(static_cast<double>(lr) / (1.0 - std::pow(static_cast<double>(beta1), t)));
    const float inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(1.0 - std::pow(static_cast<double>(beta2), t)));
    const long long tile = adamw_tile_elems();
    int i = 0;
    while (i < count) {
        AdamWParams& p = *ap;
        std::memset(&p, 0, sizeof p);
        p.p_bf16 = p_dtype == MUON_BF16;
        p.g_bf16 = g_dtype == MUON_BF16;
        p.beta1 = beta1;
        p.beta2 = beta2;
        p.eps = eps;
        p.b1c = b1c;
        p.b2c = b2c;
        p.dcy = dcy;
        p.step_size = step_size;
        p.inv_sqrt_bc2 = inv_sqrt_bc2;
        long long tiles = 0;
        double bytes = 0;
        for (; i < count && p.ntensors < kAdamMaxTensors; ++i) {
            if (numel[i] == 0) continue;
            AdamWTensor& T = p.t[p.ntensors++];
            T.p = P[i];
            T.g = G[i];
            T.m = M[i];
            T.v = V[i];
            T.n = numel[i];
            T.tile0 = tiles;
            tiles += (numel[i] + tile - 1) / tile;
            bytes += static_cast<double>(numel[i]) * (2.0 * psz + gsz + 16.0);
        }
        if (p.ntensors == 0) break;
        p.total_tiles = tiles;
        rc = launch(kKAdamW, 0.0, bytes, stream, [&] { return launch_adamw(*ap, d->sms, stream); });
        if (rc != MUON_OK) return rc;
    }
    return MUON_OK;
}

size_t muon_workspace_bytes(const int* rows, const int* cols, int count) {
    if (count <= 0) return 0;
    if (validate_dims(rows, cols, count) != MUON_OK) return 0;
    return plan_bytes(rows, cols, count, split_point(rows, cols, count));
}

const char* muon_status_string(int status) {
    switch (status) {
        case MUON_OK: return "MUON_OK";
        case MUON_ERR_INVALID_ARG: return "MUON_ERR_INVALID_ARG: invalid argument";
        case MUON_ERR_UNSUPPORTED: return "MUON_ERR_UNSUPPORTED: unsupported device or shape";
        case MUON_ERR_CUDA: return "MUON_ERR_CUDA: a CUDA call failed";
        case MUON_ERR_OOM: return "MUON_ERR_OOM: workspace allocation failed";
        case MUON_ERR_TIMEOUT: return "MUON_ERR_TIMEOUT: a device-side wait ran out";
        case MUON_ERR_CORRUPT: return "MUON_ERR_CORRUPT: a workspace guard region was overwritten";
        default: return "unknown muon status";
    }
}

const char* muon_last_error(void) { return t_last_error.c_str(); }

int muon_device_status(cudaStream_t stream, int* device_status) {
    if (device_status == nullptr) return fail(MUON_ERR_INVALID_ARG, "device_status is NULL");
    std::lock_guard<std::mutex> lock(g_mu);
    MUON_CUDA_TRY(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
    int code = 0, code2 = 0;
    MUON_CUDA_TRY(read_and_clear_pair_error(&code), "reading the device status");
    MUON_CUDA_TRY(read_and_clear_guard_error(&code2), "reading the device status");
    *device_status = code != 0 ? code : code2;
    return MUON_OK;
}

void muon_release_workspace(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
    DeviceState& d = g_dev[dev];
    if (d.ws != nullptr) {
        cudaDeviceSynchronize();
        cudaFree(d.ws);
        d.ws = nullptr;
        d.ws_bytes = 0;
        d.have_last = false;
    }
}

int muon_profile_enable(int on) {
    std::lock_guard<std::mutex> lock(g_mu);
    for (ProfRec& r : g_prof_pending) {
        cudaEventSynchronize(r.b);
        g_event_pool.push_back(r.a);
        g_event_pool.push_back(r.b);
    }
    g_prof_pending.clear();
    for (auto& a : g_prof) a = ProfAgg();
    g_prof_on = on != 0;
    return MUON_OK;
}

int muon_profile_read(muon_kernel_stat* out, int max_entries, int* n_entries) {
    if (n_entries == nullptr || (out == nullptr && max_entries > 0))
        return fail(MUON_ERR_INVALID_ARG, "NULL output");
    std::lock_guard<std::mutex> lock(g_mu);
    for (ProfRec& r : g_prof_pending) {
        MUON_CUDA_TRY(cudaEventSynchronize(r.b), "cudaEventSynchronize");
        float ms = 0.0f;
        MUON_CUDA_TRY(cudaEventElapsedTime(&ms, r.a, r.b), "cudaEventElapsedTime");
        ProfAgg& a = g_prof[r.kind];
        a.launches += 1;
        a.ms += ms;
        a.flops += r.flops;
        a.bytes += r.bytes;
        g_event_pool.push_back(r.a);
        g_event_pool.push_back(r.b);
    }
    g_prof_pending.clear();
    int n = 0;
    for (int k = 0; k < kNumKinds; ++k) {
        if (n < max_entries) {
            muon_kernel_stat& s = out[n];
            std::memset(&s, 0, sizeof s);
            std::snprintf(s.name, sizeof s.name, "%s", kKindNames[k]);
            s.launches = g_prof[k].launches;
            s.total_ms = g_prof[k].ms;
            s.flops = g_prof[k].flops;
            s.bytes = g_prof[k].bytes;
        }
        ++n;
    }
    *n_entries = std::min(n, max_entries);
    return MUON_OK;
}

}  // extern "C"
