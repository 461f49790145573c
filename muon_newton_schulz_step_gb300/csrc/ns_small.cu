// Newton-Schulz for small matrices: one CTA per matrix, every iteration in
// shared memory, one launch for all iterations and all small matrices.
//
// A matrix counts as small when its oriented iterate X (r x k), X', A and B
// (r x r) fit in shared memory together; for those the tensor-core path
// would spend its time on padding (tiles are 128 x 256) and on 3 launches per
// iteration.  Here each product is a plain fp32 FMA chain over p in
// ascending order: since the product of two bf16 values is exact in fp32,
// fma(x, y, acc) equals acc + x*y rounded once, so every A, B and X element
// is the correctly rounded fp32 running sum followed by one bf16 rounding --
// the same value as a sequential IEEE fp32 accumulation.
//
//   A  = bf16(X X^T)              (upper triangle computed, mirrored)
//   B  = bf16(b A + c A A)        (A A is symmetric: upper triangle, mirrored)
//   X' = bf16(a X + B X)
//
// The orthogonalisation on whole matrices is the step described in "How
// PyTorch Scaled a Near-1T MoE on Europe's Public Supercomputer", section
// "Three optimizations that changed the economics", FlexShard bullet.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace muon {
namespace {

constexpr int kSmallThreads = 256;
constexpr int kTM = 4;  // register tile of one thread
constexpr int kTN = 4;

__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// acc(i, j) = sum_{p < K} L[i*lsi + p*lsp] * R[p*rsp + j*rsj], p ascending,
// for 0 <= i < M, 0 <= j < N (only blocks reaching j >= i when upper), then
// epi(i, j, acc).
template <class Epi>
__device__ __forceinline__ void small_mm(const __nv_bfloat16* L, int lsi, int lsp, const __nv_bfloat16* R,
                                         int rsp, int rsj, int M, int N, int K, bool upper, Epi epi) {
    const int tm = (M + kTM - 1) / kTM;
    const int tn = (N + kTN - 1) / kTN;
    for (int t = threadIdx.x; t < tm * tn; t += blockDim.x) {
        const int i0 = (t / tn) * kTM;
        const int j0 = (t % tn) * kTN;
        if (upper && j0 + kTN - 1 < i0) continue;
        float acc[kTM][kTN];
#pragma unroll
        for (int a = 0; a < kTM; ++a)
#pragma unroll
            for (int b = 0; b < kTN; ++b) acc[a][b] = 0.0f;
        int ia[kTM], jb[kTN];
#pragma unroll
        for (int a = 0; a < kTM; ++a) ia[a] = min(i0 + a, M - 1);
#pragma unroll
        for (int b = 0; b < kTN; ++b) jb[b] = min(j0 + b, N - 1);
        for (int p = 0; p < K; ++p) {
            float l[kTM], r[kTN];
#pragma unroll
            for (int a = 0; a < kTM; ++a) l[a] = ld(L + ia[a] * lsi + p * lsp);
#pragma unroll
            for (int b = 0; b < kTN; ++b) r[b] = ld(R + p * rsp + jb[b] * rsj);
#pragma unroll
            for (int a = 0; a < kTM; ++a)
#pragma unroll
                for (int b = 0; b < kTN; ++b) acc[a][b] = __fmaf_rn(l[a], r[b], acc[a][b]);
        }
#pragma unroll
        for (int a = 0; a < kTM; ++a)
#pragma unroll
            for (int b = 0; b < kTN; ++b)
                if (i0 + a < M && j0 + b < N) epi(i0 + a, j0 + b, acc[a][b]);
    }
}

__global__ void __launch_bounds__(kSmallThreads) k_ns_small(const __grid_constant__ SmallParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const SmallMat& m = p.m[blockIdx.x];
    const int r = m.r, k = m.k;
    const int sx = k + 2;  // padded row strides: consecutive rows fall in different banks
    const int sa = r + 2;
    __nv_bfloat16* X = reinterpret_cast<__nv_bfloat16*>(smem_raw);
    __nv_bfloat16* Xn = X + r * sx;
    __nv_bfloat16* A = Xn + r * sx;
    __nv_bfloat16* B = A + r * sa;

    for (int e = threadIdx.x; e < r * k; e += blockDim.x) {
        const int i = e / k, j = e - (e / k) * k;
        X[i * sx + j] = m.x[static_cast<size_t>(i) * m.ldx + j];
    }
    __syncthreads();

    for (int it = 0; it < p.steps; ++it) {
        const float ca = p.coef[3 * it], cb = p.coef[3 * it + 1], cc = p.coef[3 * it + 2];
        // A = X X^T  (L = X rows, R(p, j) = X[j][p])
        small_mm(X, sx, 1, X, 1, sx, r, r, k, true, [&](int i, int j, float v) {
            if (j >= i) {
                const __nv_bfloat16 h = __float2bfloat16_rn(v);
                A[i * sa + j] = h;
                A[j * sa + i] = h;
            }
        });
        __syncthreads();
        // B = b A + c A A  (A symmetric: A A is symmetric with identical sums)
        small_mm(A, sa, 1, A, sa, 1, r, r, r, true, [&](int i, int j, float v) {
            if (j >= i) {
                const float lin = __fmul_rn(cb, ld(A + i * sa + j));
                const __nv_bfloat16 h = __float2bfloat16_rn(__fadd_rn(lin, __fmul_rn(cc, v)));
                B[i * sa + j] = h;
                B[j * sa + i] = h;
            }
        });
        __syncthreads();
        // X' = a X + B X
        small_mm(B, sa, 1, X, sx, 1, r, k, r, false, [&](int i, int j, float v) {
            const float lin = __fmul_rn(ca, ld(X + i * sx + j));
            Xn[i * sx + j] = __float2bfloat16_rn(__fadd_rn(lin, v));
        });
        __syncthreads();
        __nv_bfloat16* t = X;
        X = Xn;
        Xn = t;
    }

    for (int e = threadIdx.x; e < r * k; e += blockDim.x) {
        const int i = e / k, j = e - (e / k) * k;
        m.x[static_cast<size_t>(i) * m.ldx + j] = X[i * sx + j];
    }
}

}  // namespace

size_t ns_small_smem_bytes(int r, int k) {
    return static_cast<size_t>(2) * (2 * static_cast<size_t>(r) * (k + 2) + 2 * static_cast<size_t>(r) * (r + 2));
}

cudaError_t launch_ns_small(const SmallParams& p, size_t smem, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(k_ns_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    k_ns_small<<<p.nmats, kSmallThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace muon
