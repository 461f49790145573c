// Internal structures shared by the host code and the kernels of the Muon
// library.  Nothing here crosses the C ABI.
#pragma once

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime_api.h>

namespace muon {

// ------------------------------------------------------------ elementwise --
// The momentum / normalisation / packing / update kernels walk 64 x 64 tiles
// of one matrix at a time; a launch covers up to kEwMaxMats matrices whose
// descriptors travel as a kernel parameter (no host->device copy per call).
constexpr int kEwTile = 64;
constexpr int kEwThreads = 256;
constexpr int kEwMaxMats = 224;

enum EwSrc : int { kSrcBf16 = 0, kSrcF32 = 1 };

struct EwMat {
    const void* src;          // G (muon_step) or the input matrix (ns only)
    float* mom;               // fp32 momentum (muon_step) or nullptr
    void* dst;                // W (muon_step) or the input matrix (ns only, output)
    __nv_bfloat16* x;         // oriented, padded bf16 iterate X0 (pack) / O (unpack)
    __nv_bfloat16* oout;      // optional copy of O, rows x cols (unpack, weight update)
    long long part;           // first norm partial of this matrix
    int rows, cols;           // m, n as stored
    int ldx;                  // row length of the oriented, padded iterate
    int xrows_pad;            // rows of the oriented, padded iterate
    int trans;                // 1 when m > n (the iterate holds the transpose)
    int vec;                  // 1 when 8-element vector access is legal for this matrix
    int tile0;                // first tile of this matrix in this launch
    uint8_t* x8;              // pack with the FP8 Gram: E4M3 copy of X0 * 2^8, layout of x (or nullptr)
    float dcy, s;             // weight-update scalars (muon_step)
};

struct EwParams {
    int nmats;
    int total_tiles;
    int src_dtype;            // EwSrc of src
    int dst_dtype;            // EwSrc of dst (W)
    int nesterov;
    int g_count;              // stacked gradients per matrix, summed in fp32 in order
    float mu;
    double eps;               // normalisation epsilon
    double* partials;         // per-tile sums of squares (pass 1 writes, finalize reads)
    float* sigma;             // per-matrix 1/(|U|_F + eps), indexed by sigma_base + i
    int sigma_base;
    int fp8;                  // pack: some matrices also get the E4M3 copy of X0 (EwMat::x8)
    EwMat m[kEwMaxMats];
};

// ----------------------------------------------------------------- FP8 Gram --
// FP8 variant of the Gram product: its operands are X * 2^8 rounded to E4M3
// (an exact scaling; every iterate's elements stay below its largest singular
// value, which the quintic keeps under 1.21, and 1.21 * 2^8 < 448, E4M3's
// largest finite value); the product's fp32 sums are unscaled by 2^-16 before
// the bf16 rounding.  The E4M3 copy is written beside X by the kernel that
// writes X: the pack for X0, the update's epilogue for the later iterates.
constexpr int kFp8ScaleExp = 8;

// ------------------------------------------------------------------- GEMM --
// One persistent, warp-specialised tcgen05 kernel runs the three products of
// a Newton-Schulz iteration over every matrix of every shape bucket.
constexpr int kBN = 256;      // accumulator columns per tile
constexpr int kBK = 64;       // bf16 elements of K per stage (one 128-byte swizzle row)
constexpr int kMaxBuckets = 8;

enum GemmMode : int {
    kGram = 0,                // out = bf16(X X^T)                  (symmetric)
    kPoly = 1,                // out = bf16(b*A + c*A A)            (symmetric)
    kUpdate = 2               // out = bf16(a*X + B X)
};

struct GemmBucket {
    CUtensorMap tmA;          // A operand, box {64, 128, 1}, K-major
    CUtensorMap tmB;          // B operand: K-major box {64, 256, 1} or MN-major box {64, 64, 1}
    __nv_bfloat16* out;       // output, nmat x rows x ld
    const __nv_bfloat16* epi; // epilogue input with the same layout as out (Poly: A, Update: X)
    long long mat_stride;     // elements between matrices of out / epi
    int ld;                   // row length of out / epi
    int mt, nt;               // tiles along M and N of one matrix
    int kblocks;              // K / kBK
    int tiles_per_mat;
    int nmat;
    int tile0;                // first global tile of this bucket
    int fin0;                 // first entry of this bucket's matrices in FinalParams (final update)
    CUtensorMap tmE;          // update: the iterate X as epilogue input, box {32, 32, 1}, 64-byte swizzle
    CUtensorMap tmO;          // update: the output X', box {32, 32, 1}, 64-byte swizzle
    CUtensorMap tmT;          // upper-only symmetric operand (polynomial: A, update: B): box {64, 64, 1}
                              // over its rows, read as MN-major blocks of the transpose
    CUtensorMap tmQ;          // update before an FP8 Gram: E4M3 copy of X' * 2^8, bytes, box {32, 32, 1}
    int nt2;                  // update on clusters of two pairs: tile pairs along N, ceil(nt / 2)
    int item0;                // update on clusters of two pairs: first global tile pair of this bucket
};

struct GemmParams {
    GemmBucket b[kMaxBuckets];
    int nbuckets;
    int total_tiles;
    int mode;
    float a, bcoef, c;
    unsigned long long wait_ns;   // limit of every wait of the launch; 0: the default (2 s)
    int stall;                    // test hook (pair kernel): no MMA is issued, so the waits expire
    int total_items;              // update on clusters of two pairs: tile pairs of the launch
    int fp8;                      // Gram: E4M3 operands (tmA / tmB over the E4M3 copy, kblocks of 128)
    int fp8_next;                 // update (TMA epilogue): also writes the E4M3 copy of X' through tmQ
    // 1: the symmetric products (Gram, polynomial) store only their tiles with
    // tm <= tn (diagonal tiles in full), and their consumers (polynomial,
    // update) read the K blocks left of a row tile's diagonal as MN-major
    // blocks of the stored transpose (tmT); 0: full storage, K-major reads only
    int upper_only;
};

// Last update of the iteration fused with what follows it: the epilogue rounds
// O = bf16(a X + B X) and writes it straight to the caller's matrix in its
// stored orientation -- the weight update W <- dcy*W - s*O (muon_step) or the
// store of O into the input (Newton-Schulz only) -- so O never makes a round
// trip through HBM.  One table entry per matrix of the launch.
constexpr int kFinalMaxMats = 448;

enum FinalKind : int {
    kFinNone = 0,             // plain update: X' to the workspace
    kFinStore = 1,            // O (bf16) into the caller's bf16 matrix
    kFinWBf16 = 2,            // weight update of a bf16 W
    kFinWF32 = 3              // weight update of an fp32 W
};

struct FinalMat {
    void* w;                  // W (weight update) or the input matrix (store), rows x cols as stored
    __nv_bfloat16* oout;      // optional copy of O, rows x cols, or nullptr
    float dcy, s;             // weight-update scalars
    int rows, cols;           // as stored
    int trans;                // 1 when rows > cols (the iterate holds the transpose)
    int vec;                  // 1 when cols % 8 == 0 (16-byte vector access along a stored row)
};

struct FinalParams {
    FinalMat m[kFinalMaxMats];
};

// ------------------------------------------------------------ small path --
// Matrices whose iterate, A and B fit in shared memory run every
// Newton-Schulz iteration in one CTA (ns_small.cu).
constexpr int kSmallMaxMats = 512;
constexpr size_t kSmallMaxSmem = 200 * 1024;

struct SmallMat {
    __nv_bfloat16* x;         // oriented iterate (r x k, row stride ldx), updated in place
    int r, k, ldx, pad_;
};

constexpr int kMaxNsSteps = 64;

struct SmallParams {
    int nmats;
    int steps;
    float coef[3 * kMaxNsSteps];   // (a, b, c) of every iteration
    SmallMat m[kSmallMaxMats];
};

// ------------------------------------------------------------------ AdamW --
constexpr int kAdamMaxTensors = 256;

struct AdamWTensor {
    void* p;                  // parameter (bf16 or fp32), updated in place
    const void* g;            // gradient (bf16 or fp32)
    float* m;                 // first moment, fp32
    float* v;                 // second moment, fp32
    long long n;              // elements
    long long tile0;          // first tile of this tensor in this launch
};

struct AdamWParams {
    int ntensors;
    int p_bf16, g_bf16;
    long long total_tiles;
    float beta1, beta2, eps, b1c, b2c, dcy, step_size, inv_sqrt_bc2;
    AdamWTensor t[kAdamMaxTensors];
};

cudaError_t launch_adamw(const AdamWParams& p, int sms, cudaStream_t s);
long long adamw_tile_elems();

// Launch helpers implemented in the .cu files.
// `sms`: the grid is one CTA per resident slot on every SM (capped by the tiles).
cudaError_t launch_momentum_norm(const EwParams& p, int sms, cudaStream_t s);
cudaError_t launch_input_norm(const EwParams& p, int sms, cudaStream_t s);
cudaError_t launch_norm_finalize(const EwParams& p, cudaStream_t s);
cudaError_t launch_pack(const EwParams& p, int sms, bool from_momentum, cudaStream_t s);
cudaError_t launch_unpack(const EwParams& p, int sms, bool weight_update, cudaStream_t s);
// Pair-CTA variant (ns_gemm_pair.cu): 256 x 256 tiles on clusters of two CTAs.
// The update product (p.mode == kUpdate) runs on clusters of two pairs that
// share the A operand by multicast when `multicast` is set and such clusters
// fit on the device (p.total_items and the buckets' nt2 / item0 must be set);
// `sms` bounds the grid.
// `tma_epilogue`: the update moves its epilogue input and output by TMA
// (the buckets' tmE / tmO must be set).
cudaError_t launch_gemm_pair(const GemmParams& p, int sms, bool multicast, bool tma_epilogue, cudaStream_t s);
// The same kernel with the fused final epilogue (p.mode must be kUpdate).
cudaError_t launch_gemm_pair_final(const GemmParams& p, const FinalParams& f, int kind, int sms, bool multicast,
                                   cudaStream_t s);
size_t gemm_pair_smem_bytes();
cudaError_t read_and_clear_pair_error(int* code);

// ------------------------------------------------------------ debug guard --
// MUON_DEBUG_GUARD=1: guard regions around every workspace region (guard.cu).
constexpr size_t kGuardBytes = 4096;
constexpr unsigned kGuardWord = 0xA5A5A5A5u;   // every byte 0xA5
constexpr int kMaxGuards = 480;

struct GuardParams {
    const char* base;          // workspace base
    int n;                     // guard regions in this launch
    unsigned long long off[kMaxGuards];   // their offsets from base
};

cudaError_t launch_guard_check(const GuardParams& p, cudaStream_t s);
cudaError_t read_and_clear_guard_error(int* code);

// Host helpers of muon_abi.cu used by other entry points.
int ns5_batched_on_workspace(void* const* ptrs, const int* rows, const int* cols, int count, int steps,
                             const float* coeffs, void* ws, size_t ws_bytes, cudaStream_t stream);
int set_last_error(int status, const char* msg);
cudaError_t launch_ns_small(const SmallParams& p, size_t smem, cudaStream_t s);
size_t ns_small_smem_bytes(int r, int k);

}  // namespace muon
