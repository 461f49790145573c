// Newton-Schulz for small matrices: one CTA per matrix, every iteration in
// shared memory, one launch for all iterations and all small matrices.
//
// A matrix counts as small when its oriented iterate X (r x k), X', A and B
// (r x r) fit in shared memory together; for those the tensor-core path
// would spend its time on padding (tiles are 128 x 256) and on 3 launches per
// iteration.  Here each product is a plain fp32 FMA chain over p in
// ascending order (operands staged 8 elements of p at a time in registers):
// since the product of two bf16 values is exact in fp32, fma(x, y, acc)
// equals acc + x*y rounded once, so every A, B and X element
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
#include <cstdlib>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace muon {
namespace {

constexpr int kSmallThreads = 512;
constexpr int kPadK = 8;     // sums run over 8-element chunks of p (16-byte loads); padding is zero

__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ void bf8(const __nv_bfloat16* p, float (&f)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 t = __bfloat1622float2(h[q]);
        f[2 * q] = t.x;
        f[2 * q + 1] = t.y;
    }
}

__device__ __forceinline__ void bf4(const __nv_bfloat16* p, float (&f)[4]) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const float2 t = __bfloat1622float2(h[q]);
        f[2 * q] = t.x;
        f[2 * q + 1] = t.y;
    }
}

// acc(i, j) = sum_{p < Kp} L[i*ls + p] * R[j*rs + p], p ascending (rows of
// both operands contiguous in p; Kp a multiple of 8 with zero padding), for
// 0 <= i < M, 0 <= j < N, then epi(i, j, acc).  A thread owns rows
// R0 + q + 8a and columns C0 + q' + 8b (a, b < 4) of a 32 x 32 block, so that
// neighbouring lanes read neighbouring rows (no bank conflicts with a row
// stride of 4 mod 32 words).  upper: blocks left of the diagonal are skipped.
template <class Epi>
__device__ __forceinline__ void small_mm_nt(const __nv_bfloat16* L, int ls, const __nv_bfloat16* R, int rs, int M,
                                            int N, int Kp, bool upper, Epi epi) {
    const int bm = (M + 31) / 32, bn = (N + 31) / 32;
    for (int t = threadIdx.x; t < bm * bn * 64; t += blockDim.x) {
        const int blk = t >> 6, qi = (t >> 3) & 7, qj = t & 7;
        const int r0 = (blk / bn) * 32, c0 = (blk % bn) * 32;
        if (upper && c0 < r0) continue;
        float acc[4][4];
        int ia[4], jb[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            ia[a] = min(r0 + qi + 8 * a, M - 1);
            jb[a] = min(c0 + qj + 8 * a, N - 1);
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;
        }
        for (int p = 0; p < Kp; p += kPadK) {
            float l[4][8], r[4][8];
#pragma unroll
            for (int a = 0; a < 4; ++a) bf8(L + ia[a] * ls + p, l[a]);
#pragma unroll
            for (int b = 0; b < 4; ++b) bf8(R + jb[b] * rs + p, r[b]);
#pragma unroll
            for (int q = 0; q < kPadK; ++q)
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = __fmaf_rn(l[a][q], r[b][q], acc[a][b]);
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int i = r0 + qi + 8 * a, j = c0 + qj + 8 * b;
                if (i < M && j < N) epi(i, j, acc[a][b]);
            }
    }
}

// acc(i, j) = sum_{p < Kp} L[i*ls + p] * R[p*rs + j], p ascending; a thread
// owns a 4 x 4 block (rows i0 .. i0+3, columns j0 .. j0+3: one 8-byte load of
// R per p).  R's rows must hold at least N rounded up to 4 columns.
template <class Epi>
__device__ __forceinline__ void small_mm_nn(const __nv_bfloat16* L, int ls, const __nv_bfloat16* R, int rs, int M,
                                            int N, int Kp, Epi epi) {
    const int tm = (M + 3) / 4, tn = (N + 3) / 4;
    for (int t = threadIdx.x; t < tm * tn; t += blockDim.x) {
        const int i0 = (t / tn) * 4, j0 = (t % tn) * 4;
        float acc[4][4];
        int ia[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            ia[a] = min(i0 + a, M - 1);
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;
        }
        for (int p = 0; p < Kp; p += kPadK) {
            float l[4][8];
#pragma unroll
            for (int a = 0; a < 4; ++a) bf8(L + ia[a] * ls + p, l[a]);
#pragma unroll
            for (int q = 0; q < kPadK; ++q) {
                float r[4];
                bf4(R + (p + q) * rs + j0, r);
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = __fmaf_rn(l[a][q], r[b], acc[a][b]);
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b)
                if (i0 + a < M && j0 + b < N) epi(i0 + a, j0 + b, acc[a][b]);
    }
}

// Shared-memory layout of one matrix: X and X' (rp x sx), A and B (rp x sa),
// rp = r and kp = k rounded up to 8, row strides sx = kp + 8 and sa = rp + 8
// (16-byte aligned rows, consecutive rows 4 banks apart).  Rows and columns
// past r and k hold zeros, so the padded sums equal the exact ones.
struct SmallLayout {
    int rp, kp, sx, sa;
    __device__ __host__ SmallLayout(int r, int k)
        : rp((r + kPadK - 1) / kPadK * kPadK), kp((k + kPadK - 1) / kPadK * kPadK), sx(kp + 8), sa(rp + 8) {}
    __device__ __host__ size_t bytes() const {
        return 2 * (2 * static_cast<size_t>(rp) * sx + 2 * static_cast<size_t>(rp) * sa);
    }
};

__global__ void __launch_bounds__(kSmallThreads) k_ns_small(const __grid_constant__ SmallParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const SmallMat& m = p.m[blockIdx.x];
    const int r = m.r, k = m.k;
    const SmallLayout g(r, k);
    const int sx = g.sx, sa = g.sa;
    __nv_bfloat16* X = reinterpret_cast<__nv_bfloat16*>(smem_raw);
    __nv_bfloat16* Xn = X + g.rp * sx;
    __nv_bfloat16* A = Xn + g.rp * sx;
    __nv_bfloat16* B = A + g.rp * sa;

    // zero everything (padding must read as zeros), then load the iterate
    {
        uint4* z = reinterpret_cast<uint4*>(smem_raw);
        const int n16 = static_cast<int>(g.bytes() / 16);
        for (int e = threadIdx.x; e < n16; e += blockDim.x) z[e] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < r * k; e += blockDim.x) {
        const int i = e / k, j = e - (e / k) * k;
        X[i * sx + j] = m.x[static_cast<size_t>(i) * m.ldx + j];
    }
    __syncthreads();

    for (int it = 0; it < p.steps; ++it) {
        const float ca = p.coef[3 * it], cb = p.coef[3 * it + 1], cc = p.coef[3 * it + 2];
        // A = X X^T  (both operands rows of X)
        small_mm_nt(X, sx, X, sx, r, r, g.kp, true, [&](int i, int j, float v) {
            if (j >= i) {
                const __nv_bfloat16 h = __float2bfloat16_rn(v);
                A[i * sa + j] = h;
                A[j * sa + i] = h;
            }
        });
        __syncthreads();
        // B = b A + c A A  (A symmetric: (A A)(i, j) = sum_p A[i][p] A[j][p], the
        // same terms in the same order as sum_p A[i][p] A[p][j])
        small_mm_nt(A, sa, A, sa, r, r, g.rp, true, [&](int i, int j, float v) {
            if (j >= i) {
                const float lin = __fmul_rn(cb, ld(A + i * sa + j));
                const __nv_bfloat16 h = __float2bfloat16_rn(__fadd_rn(lin, __fmul_rn(cc, v)));
                B[i * sa + j] = h;
                B[j * sa + i] = h;
            }
        });
        __syncthreads();
        // X' = a X + B X
        small_mm_nn(B, sa, X, sx, r, k, g.rp, [&](int i, int j, float v) {
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

// ---------------------------------------------------------------------------
// The same iterations on a cluster of kSmallCluster CTAs per matrix.  Every
// CTA keeps full copies of X and A in its shared memory (the layout above) and
// computes a slice of rows: full rows of A (no symmetric skip: A[i][j] and
// A[j][i] are the same sum of the same exact products in the same order),
// rows of B (only its own rows are ever needed: X'(i, :) uses B(i, :)) and
// rows of X'.  After the Gram and after the update the CTAs meet at a cluster
// barrier and each copies the other CTAs' rows from their shared memory
// (distributed shared memory, 16-byte loads).  Every output element is still
// one thread's fp32 FMA chain over p in ascending order: the results equal the
// one-CTA kernel's bit for bit.
constexpr int kSmallCluster = 8;
constexpr int kClusterThreads = 512;

__device__ __forceinline__ uint4 ld_dsmem16(uint32_t cluster_addr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

// acc(i, j) = sum_{p < Kp} L[i*ls + p] * R[j*rs + p], p ascending, for rows
// i0 <= i < i1 and 0 <= j < N: one output per thread and item.
template <class Epi>
__device__ __forceinline__ void rows_nt(const __nv_bfloat16* L, int ls, const __nv_bfloat16* R, int rs, int i0,
                                        int i1, int N, int Kp, Epi epi) {
    const int items = (i1 - i0) * N;
    for (int t = threadIdx.x; t < items; t += blockDim.x) {
        const int i = i0 + t / N, j = t - (t / N) * N;
        float acc = 0.0f;
        for (int p = 0; p < Kp; p += kPadK) {
            float l[8], r[8];
            bf8(L + i * ls + p, l);
            bf8(R + j * rs + p, r);
#pragma unroll
            for (int q = 0; q < kPadK; ++q) acc = __fmaf_rn(l[q], r[q], acc);
        }
        epi(i, j, acc);
    }
}

// acc(i, j) = sum_{p < Kp} L[i*ls + p] * R[p*rs + j], p ascending, for rows
// i0 <= i < i1, four consecutive columns per item (R rows hold at least N
// rounded up to 4 columns).
template <class Epi>
__device__ __forceinline__ void rows_nn(const __nv_bfloat16* L, int ls, const __nv_bfloat16* R, int rs, int i0,
                                        int i1, int N, int Kp, Epi epi) {
    const int n4 = (N + 3) / 4;
    const int items = (i1 - i0) * n4;
    for (int t = threadIdx.x; t < items; t += blockDim.x) {
        const int i = i0 + t / n4, j0 = (t - (t / n4) * n4) * 4;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int p = 0; p < Kp; p += kPadK) {
            float l[8];
            bf8(L + i * ls + p, l);
#pragma unroll
            for (int q = 0; q < kPadK; ++q) {
                float r[4];
                bf4(R + (p + q) * rs + j0, r);
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[b] = __fmaf_rn(l[q], r[b], acc[b]);
            }
        }
#pragma unroll
        for (int b = 0; b < 4; ++b)
            if (j0 + b < N) epi(i, j0 + b, acc[b]);
    }
}

// Copy the rows of every other CTA's slice of `buf` (rows x stride bf16, the
// first `cols` columns, a multiple of 8) from that CTA's shared memory.
__device__ __forceinline__ void pull_rows(__nv_bfloat16* buf, int stride, int rows, int cols, int slice,
                                          uint32_t rank) {
    const uint32_t local = ptx::smem_addr(buf);
    const int per_row = cols / 8;
    for (uint32_t c = 0; c < static_cast<uint32_t>(kSmallCluster); ++c) {
        if (c == rank) continue;
        const int r0 = static_cast<int>(c) * slice, r1 = min(rows, r0 + slice);
        if (r0 >= r1) continue;
        const uint32_t remote = ptx::mapa_shared(local, c);
        const int n = (r1 - r0) * per_row;
        for (int e = threadIdx.x; e < n; e += blockDim.x) {
            const int row = r0 + e / per_row, u = e - (e / per_row) * per_row;
            const uint32_t off = static_cast<uint32_t>((row * stride + u * 8) * 2);
            *reinterpret_cast<uint4*>(reinterpret_cast<char*>(buf) + off) = ld_dsmem16(remote + off);
        }
    }
}

__global__ void __launch_bounds__(kClusterThreads) k_ns_small_cluster(const __grid_constant__ SmallParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const uint32_t rank = ptx::cluster_ctarank();
    const SmallMat& m = p.m[blockIdx.x / kSmallCluster];
    const int r = m.r, k = m.k;
    const SmallLayout g(r, k);
    const int sx = g.sx, sa = g.sa;
    const int slice = (r + kSmallCluster - 1) / kSmallCluster;
    const int i0 = min(r, static_cast<int>(rank) * slice), i1 = min(r, i0 + slice);
    __nv_bfloat16* X = reinterpret_cast<__nv_bfloat16*>(smem_raw);
    __nv_bfloat16* Xn = X + g.rp * sx;
    __nv_bfloat16* A = Xn + g.rp * sx;
    __nv_bfloat16* B = A + g.rp * sa;

    {
        uint4* z = reinterpret_cast<uint4*>(smem_raw);
        const int n16 = static_cast<int>(g.bytes() / 16);
        for (int e = threadIdx.x; e < n16; e += blockDim.x) z[e] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    // the iterate in 16-byte vectors: its rows in the workspace hold ldx >= kp
    // elements (a multiple of 64), zero past k
    {
        const int per_row = g.kp / 8;
        for (int e = threadIdx.x; e < r * per_row; e += blockDim.x) {
            const int i = e / per_row, u = e - (e / per_row) * per_row;
            *reinterpret_cast<uint4*>(X + i * sx + u * 8) =
                *reinterpret_cast<const uint4*>(m.x + static_cast<size_t>(i) * m.ldx + u * 8);
        }
    }
    __syncthreads();

    for (int it = 0; it < p.steps; ++it) {
        const float ca = p.coef[3 * it], cb = p.coef[3 * it + 1], cc = p.coef[3 * it + 2];
        // A rows of this slice: A(i, j) = sum_p X[i][p] X[j][p]
        rows_nt(X, sx, X, sx, i0, i1, r, g.kp, [&](int i, int j, float v) { A[i * sa + j] = __float2bfloat16_rn(v); });
        ptx::cluster_sync();
        pull_rows(A, sa, r, g.rp, slice, rank);
        __syncthreads();
        // B rows of this slice: b A + c A A with (A A)(i, j) = sum_p A[i][p] A[j][p]
        rows_nt(A, sa, A, sa, i0, i1, r, g.rp, [&](int i, int j, float v) {
            const float lin = __fmul_rn(cb, ld(A + i * sa + j));
            B[i * sa + j] = __float2bfloat16_rn(__fadd_rn(lin, __fmul_rn(cc, v)));
        });
        __syncthreads();
        // X' rows of this slice: a X + B X
        rows_nn(B, sa, X, sx, i0, i1, k, g.rp, [&](int i, int j, float v) {
            const float lin = __fmul_rn(ca, ld(X + i * sx + j));
            Xn[i * sx + j] = __float2bfloat16_rn(__fadd_rn(lin, v));
        });
        ptx::cluster_sync();
        pull_rows(Xn, sx, r, g.kp, slice, rank);
        __syncthreads();
        __nv_bfloat16* t = X;
        X = Xn;
        Xn = t;
    }

    {
        const int per_row = g.kp / 8;   // columns k .. kp of X hold zeros
        for (int e = threadIdx.x; e < (i1 - i0) * per_row; e += blockDim.x) {
            const int i = i0 + e / per_row, u = e - (e / per_row) * per_row;
            *reinterpret_cast<uint4*>(m.x + static_cast<size_t>(i) * m.ldx + u * 8) =
                *reinterpret_cast<const uint4*>(X + i * sx + u * 8);
        }
    }
    // no CTA leaves while a peer may still read its shared memory
    ptx::cluster_sync();
}

}  // namespace

size_t ns_small_smem_bytes(int r, int k) { return SmallLayout(r, k).bytes(); }

namespace {

// Clusters of kSmallCluster CTAs with `smem` each, if the device can hold at
// least one (otherwise the one-CTA kernel runs).
bool cluster_fits(size_t smem) {
    if (cudaFuncSetAttribute(k_ns_small_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(k_ns_small_cluster, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kSmallCluster, 1, 1);
    cfg.blockDim = dim3(kClusterThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSmallCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_ns_small_cluster, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return n >= 1;
}

}  // namespace

// MUON_SMALL_NO_CLUSTER=1 keeps one CTA per matrix (comparison).
cudaError_t launch_ns_small(const SmallParams& p, size_t smem, cudaStream_t s) {
    const char* env = std::getenv("MUON_SMALL_NO_CLUSTER");
    const bool no_cluster = env != nullptr && env[0] != '\0' && env[0] != '0';
    if (!no_cluster && cluster_fits(smem)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(p.nmats * kSmallCluster, 1, 1);
        cfg.blockDim = dim3(kClusterThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kSmallCluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, k_ns_small_cluster, p);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    cudaError_t e = cudaFuncSetAttribute(k_ns_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    k_ns_small<<<p.nmats, kSmallThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace muon
