// HBM-bound parts of the Muon step on sm_103a:
//
//   norm pass   M <- fma(mu, M, G);  U = fma(mu, M, G) (Nesterov) or U = M;
//               per-tile sum of U^2.  (ns-only: sum of X^2 of the input.)
//               One optimizer state per matrix -- "Domyn is training a
//               1T-parameter MoE on Europe's Jupiter supercomputer, and
//               published the recipe", section "What moved the number".
//   finalize    sigma = fp32(1 / (sqrt(sum) + eps)), one CTA per matrix,
//               partials added in a fixed order (deterministic).
//   pack        X0 = bf16(U * sigma) written into the oriented (r <= k),
//               zero-padded iterate; U is recomputed from G and the new M
//               (bit-identical to the norm pass), tall matrices are
//               transposed through shared memory.
//   unpack      W <- round_W(fma(-s, O, dcy * W)) (or, ns-only, the matrix
//               <- O), reading O from the oriented iterate, transposing tall
//               matrices back through shared memory.
//
// All kernels walk 64 x 64 tiles; a thread handles 8 consecutive elements of
// a row (one 16-byte bf16 vector), so a warp touches 4 rows x 128 contiguous
// bytes.  Matrices whose row length is not a multiple of 8 take a scalar path.
// fp32 arithmetic uses explicit _rn intrinsics so that no contraction can
// change a rounding: the momentum is bit-exact by construction.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace muon {
namespace {

enum : int { kMomBf16 = 0, kMomF32 = 1, kInput = 2 };         // source kinds
enum : int { kWBf16 = 0, kWF32 = 1, kStoreBf16 = 2 };         // destination kinds

__device__ __forceinline__ int find_mat(const EwParams& p, int t) {
    int lo = 0, hi = p.nmats - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.m[mid].tile0 <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float (&f)[8]) {
    uint4 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
}

template <int KIND>
__device__ __forceinline__ void load_src8(const EwMat& m, size_t off, float (&g)[8]) {
    if (KIND == kMomF32) {
        const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(m.src) + off);
        const float4 a = s[0], b = s[1];
        g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
        g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
    } else {
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(m.src) + off), g);
    }
}

template <int KIND>
__device__ __forceinline__ float load_src1(const EwMat& m, size_t off) {
    if (KIND == kMomF32) return static_cast<const float*>(m.src)[off];
    return __bfloat162float(static_cast<const __nv_bfloat16*>(m.src)[off]);
}

// The gradient: K stacked matrices (stride rows * cols) summed in fp32 in
// order, g = G_0 + G_1 + ... (one rounding per add) -- bf16 gradients that
// arrive separately and are accumulated in fp32 locally.
template <int KIND, bool MULTI>
__device__ __forceinline__ void load_grad8(const EwParams& p, const EwMat& m, size_t off, float (&g)[8]) {
    load_src8<KIND>(m, off, g);
    if (KIND == kInput || !MULTI) return;
    const size_t stride = static_cast<size_t>(m.rows) * static_cast<size_t>(m.cols);
    for (int j = 1; j < p.g_count; ++j) {
        float t[8];
        load_src8<KIND>(m, off + j * stride, t);
#pragma unroll
        for (int e = 0; e < 8; ++e) g[e] = __fadd_rn(g[e], t[e]);
    }
}

template <int KIND, bool MULTI>
__device__ __forceinline__ float load_grad1(const EwParams& p, const EwMat& m, size_t off) {
    float g = load_src1<KIND>(m, off);
    if (KIND == kInput || !MULTI) return g;
    const size_t stride = static_cast<size_t>(m.rows) * static_cast<size_t>(m.cols);
    for (int j = 1; j < p.g_count; ++j) g = __fadd_rn(g, load_src1<KIND>(m, off + j * stride));
    return g;
}

// U from G and the already-updated momentum (pack pass).
template <int KIND, bool MULTI>
__device__ __forceinline__ void u_from_state8(const EwParams& p, const EwMat& m, size_t off,
                                              float (&u)[8]) {
    float g[8];
    load_grad8<KIND, MULTI>(p, m, off, g);
    if (KIND == kInput) {
#pragma unroll
        for (int j = 0; j < 8; ++j) u[j] = g[j];
    } else {
        const float4* mp = reinterpret_cast<const float4*>(m.mom + off);
        const float4 a = mp[0], b = mp[1];
        const float mo[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) u[j] = p.nesterov ? __fmaf_rn(p.mu, mo[j], g[j]) : mo[j];
    }
}

template <int KIND, bool MULTI>
__device__ __forceinline__ float u_from_state1(const EwParams& p, const EwMat& m, size_t off) {
    const float g = load_grad1<KIND, MULTI>(p, m, off);
    if (KIND == kInput) return g;
    const float mo = m.mom[off];
    return p.nesterov ? __fmaf_rn(p.mu, mo, g) : mo;
}

// ------------------------------------------------------------- norm pass --
template <int KIND, bool MULTI>
__global__ void __launch_bounds__(kEwThreads) k_norm_pass(const __grid_constant__ EwParams p) {
    __shared__ double red[kEwThreads / 32];
    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        const int mi = find_mat(p, t);
        const EwMat& m = p.m[mi];
        const int local = t - m.tile0;
        const int tcols = (m.cols + kEwTile - 1) / kEwTile;
        const int r0 = (local / tcols) * kEwTile;
        const int c0 = (local % tcols) * kEwTile;
        float ss = 0.0f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int v = threadIdx.x + h * kEwThreads;
            const int row = r0 + (v >> 3);
            const int col = c0 + (v & 7) * 8;
            if (row >= m.rows || col >= m.cols) continue;
            const size_t off = static_cast<size_t>(row) * m.cols + col;
            if (m.vec && col + 8 <= m.cols) {
                float g[8];
                load_grad8<KIND, MULTI>(p, m, off, g);
                if (KIND == kInput) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) ss = fmaf(g[j], g[j], ss);
                } else {
                    float4* mp = reinterpret_cast<float4*>(m.mom + off);
                    const float4 a = mp[0], b = mp[1];
                    float mo[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float mn = __fmaf_rn(p.mu, mo[j], g[j]);
                        mo[j] = mn;
                        const float u = p.nesterov ? __fmaf_rn(p.mu, mn, g[j]) : mn;
                        ss = fmaf(u, u, ss);
                    }
                    mp[0] = make_float4(mo[0], mo[1], mo[2], mo[3]);
                    mp[1] = make_float4(mo[4], mo[5], mo[6], mo[7]);
                }
            } else {
                const int n = min(8, m.cols - col);
                for (int j = 0; j < n; ++j) {
                    const float g = load_grad1<KIND, MULTI>(p, m, off + j);
                    if (KIND == kInput) {
                        ss = fmaf(g, g, ss);
                    } else {
                        const float mn = __fmaf_rn(p.mu, m.mom[off + j], g);
                        m.mom[off + j] = mn;
                        const float u = p.nesterov ? __fmaf_rn(p.mu, mn, g) : mn;
                        ss = fmaf(u, u, ss);
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = static_cast<double>(ss);
        __syncthreads();
        if (threadIdx.x == 0) {
            double tot = 0.0;
            for (int w = 0; w < kEwThreads / 32; ++w) tot += red[w];
            p.partials[m.part + local] = tot;
        }
        __syncthreads();
    }
}

// -------------------------------------------------------------- finalize --
__global__ void __launch_bounds__(kEwThreads) k_norm_finalize(const __grid_constant__ EwParams p) {
    __shared__ double red[kEwThreads];
    const EwMat& m = p.m[blockIdx.x];
    const int n1 = ((m.rows + kEwTile - 1) / kEwTile) * ((m.cols + kEwTile - 1) / kEwTile);
    double s = 0.0;
    for (int i = threadIdx.x; i < n1; i += kEwThreads) s += p.partials[m.part + i];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = kEwThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double d = sqrt(red[0]) + p.eps;
        p.sigma[p.sigma_base + blockIdx.x] = static_cast<float>(1.0 / d);
    }
}

// ------------------------------------------------------------------ pack --
// FP8 (the FP8 Gram): also write X0's E4M3 copy (X0 * 2^8) for matrices that have one
template <int KIND, bool MULTI, bool FP8>
__global__ void __launch_bounds__(kEwThreads) k_pack(const __grid_constant__ EwParams p) {
    __shared__ __align__(16) __nv_bfloat16 tile[kEwTile][kEwTile + 8];
    constexpr float kFp8Scale = static_cast<float>(1 << kFp8ScaleExp);
    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        const int mi = find_mat(p, t);
        const EwMat& m = p.m[mi];
        const int local = t - m.tile0;
        const int tcx = m.ldx / kEwTile;
        const int i0 = (local / tcx) * kEwTile;  // iterate row
        const int j0 = (local % tcx) * kEwTile;  // iterate column
        const float sg = p.sigma[p.sigma_base + mi];
        if (!m.trans) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int v = threadIdx.x + h * kEwThreads;
                const int i = i0 + (v >> 3);
                const int j = j0 + (v & 7) * 8;
                float u[8];
                if (i < m.rows && m.vec && j + 8 <= m.cols) {
                    u_from_state8<KIND, MULTI>(p, m, static_cast<size_t>(i) * m.cols + j, u);
                } else {
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        u[jj] = (i < m.rows && j + jj < m.cols)
                                    ? u_from_state1<KIND, MULTI>(p, m, static_cast<size_t>(i) * m.cols + j + jj)
                                    : 0.0f;
                }
                float x[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) x[jj] = __fmul_rn(u[jj], sg);
                const uint4 xb = f32x8_to_bf16(x);
                const size_t off = static_cast<size_t>(i) * m.ldx + j;
                *reinterpret_cast<uint4*>(m.x + off) = xb;
                if constexpr (FP8)
                    if (m.x8 != nullptr) *reinterpret_cast<uint2*>(m.x8 + off) = ptx::e4m3x8_from_bf16x8(xb, kFp8Scale);
            }
        } else {
            // iterate X[i][j] = U[j][i]: read input rows j0.., columns i0.. (coalesced)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int v = threadIdx.x + h * kEwThreads;
                const int jr = v >> 3;
                const int ic = (v & 7) * 8;
                const int row = j0 + jr;
                const int col = i0 + ic;
                float u[8];
                if (row < m.rows && m.vec && col + 8 <= m.cols) {
                    u_from_state8<KIND, MULTI>(p, m, static_cast<size_t>(row) * m.cols + col, u);
                } else {
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        u[jj] = (row < m.rows && col + jj < m.cols)
                                    ? u_from_state1<KIND, MULTI>(p, m, static_cast<size_t>(row) * m.cols + col + jj)
                                    : 0.0f;
                }
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) tile[jr][ic + jj] = __float2bfloat16_rn(__fmul_rn(u[jj], sg));
            }
            __syncthreads();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int v = threadIdx.x + h * kEwThreads;
                const int ir = v >> 3;
                const int jc = (v & 7) * 8;
                __align__(16) __nv_bfloat16 o[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) o[jj] = tile[jc + jj][ir];
                const uint4 xb = *reinterpret_cast<const uint4*>(o);
                const size_t off = static_cast<size_t>(i0 + ir) * m.ldx + j0 + jc;
                *reinterpret_cast<uint4*>(m.x + off) = xb;
                if constexpr (FP8)
                    if (m.x8 != nullptr) *reinterpret_cast<uint2*>(m.x8 + off) = ptx::e4m3x8_from_bf16x8(xb, kFp8Scale);
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------- unpack --
template <int KIND>
__device__ __forceinline__ void write_dst(const EwMat& m, size_t off, const float (&o)[8], int n,
                                          bool vec) {
    if (KIND == kStoreBf16) {
        __nv_bfloat16* d = static_cast<__nv_bfloat16*>(m.dst) + off;
        if (vec) {
            *reinterpret_cast<uint4*>(d) = f32x8_to_bf16(o);
        } else {
            for (int j = 0; j < n; ++j) d[j] = __float2bfloat16_rn(o[j]);
        }
    } else if (KIND == kWBf16) {
        if (m.oout != nullptr) {
            if (vec) *reinterpret_cast<uint4*>(m.oout + off) = f32x8_to_bf16(o);
            else for (int j = 0; j < n; ++j) m.oout[off + j] = __float2bfloat16_rn(o[j]);
        }
        __nv_bfloat16* d = static_cast<__nv_bfloat16*>(m.dst) + off;
        if (vec) {
            float w[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(d), w);
            float r[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) r[j] = __fmaf_rn(-m.s, o[j], __fmul_rn(m.dcy, w[j]));
            *reinterpret_cast<uint4*>(d) = f32x8_to_bf16(r);
        } else {
            for (int j = 0; j < n; ++j)
                d[j] = __float2bfloat16_rn(
                    __fmaf_rn(-m.s, o[j], __fmul_rn(m.dcy, __bfloat162float(d[j]))));
        }
    } else {
        if (m.oout != nullptr) {
            if (vec) *reinterpret_cast<uint4*>(m.oout + off) = f32x8_to_bf16(o);
            else for (int j = 0; j < n; ++j) m.oout[off + j] = __float2bfloat16_rn(o[j]);
        }
        float* d = static_cast<float*>(m.dst) + off;
        if (vec) {
            float4* d4 = reinterpret_cast<float4*>(d);
            const float4 a = d4[0], b = d4[1];
            const float w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            float r[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) r[j] = __fmaf_rn(-m.s, o[j], __fmul_rn(m.dcy, w[j]));
            d4[0] = make_float4(r[0], r[1], r[2], r[3]);
            d4[1] = make_float4(r[4], r[5], r[6], r[7]);
        } else {
            for (int j = 0; j < n; ++j) d[j] = __fmaf_rn(-m.s, o[j], __fmul_rn(m.dcy, d[j]));
        }
    }
}

template <int KIND>
__global__ void __launch_bounds__(kEwThreads) k_unpack(const __grid_constant__ EwParams p) {
    __shared__ __align__(16) __nv_bfloat16 tile[kEwTile][kEwTile + 8];
    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        const int mi = find_mat(p, t);
        const EwMat& m = p.m[mi];
        const int local = t - m.tile0;
        const int tcols = (m.cols + kEwTile - 1) / kEwTile;
        const int r0 = (local / tcols) * kEwTile;
        const int c0 = (local % tcols) * kEwTile;
        if (!m.trans) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int v = threadIdx.x + h * kEwThreads;
                const int row = r0 + (v >> 3);
                const int col = c0 + (v & 7) * 8;
                if (row >= m.rows || col >= m.cols) continue;
                float o[8];
                bf16x8_to_f32(*reinterpret_cast<const uint4*>(m.x + static_cast<size_t>(row) * m.ldx + col), o);
                const bool vec = m.vec && col + 8 <= m.cols;
                write_dst<KIND>(m, static_cast<size_t>(row) * m.cols + col, o, min(8, m.cols - col), vec);
            }
        } else {
            // O[i][j] = X[j][i]: iterate rows c0.., columns r0.. (inside the padded iterate)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int v = threadIdx.x + h * kEwThreads;
                const int xr = v >> 3;
                const int xc = (v & 7) * 8;
                *reinterpret_cast<uint4*>(&tile[xr][xc]) = *reinterpret_cast<const uint4*>(
                    m.x + static_cast<size_t>(c0 + xr) * m.ldx + r0 + xc);
            }
            __syncthreads();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int v = threadIdx.x + h * kEwThreads;
                const int wr = v >> 3;
                const int wc = (v & 7) * 8;
                const int row = r0 + wr;
                const int col = c0 + wc;
                if (row < m.rows && col < m.cols) {
                    float o[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) o[jj] = __bfloat162float(tile[wc + jj][wr]);
                    const bool vec = m.vec && col + 8 <= m.cols;
                    write_dst<KIND>(m, static_cast<size_t>(row) * m.cols + col, o, min(8, m.cols - col), vec);
                }
            }
            __syncthreads();
        }
    }
}

}  // namespace

// Grid of a persistent grid-stride kernel: every resident CTA slot once.
template <class K>
int resident_grid(K kernel, int sms, int tiles) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kEwThreads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    return tiles < sms * per_sm ? tiles : sms * per_sm;
}

template <int KIND, bool MULTI>
cudaError_t run_norm(const EwParams& p, int sms, cudaStream_t s) {
    const int grid = resident_grid(k_norm_pass<KIND, MULTI>, sms, p.total_tiles);
    k_norm_pass<KIND, MULTI><<<grid, kEwThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_momentum_norm(const EwParams& p, int sms, cudaStream_t s) {
    const bool multi = p.g_count > 1;
    if (p.src_dtype == kSrcF32) return multi ? run_norm<kMomF32, true>(p, sms, s) : run_norm<kMomF32, false>(p, sms, s);
    return multi ? run_norm<kMomBf16, true>(p, sms, s) : run_norm<kMomBf16, false>(p, sms, s);
}

cudaError_t launch_input_norm(const EwParams& p, int sms, cudaStream_t s) { return run_norm<kInput, false>(p, sms, s); }

cudaError_t launch_norm_finalize(const EwParams& p, cudaStream_t s) {
    k_norm_finalize<<<p.nmats, kEwThreads, 0, s>>>(p);
    return cudaGetLastError();
}

template <int KIND, bool MULTI>
cudaError_t run_pack(const EwParams& p, int sms, cudaStream_t s) {
    if (p.fp8) {
        const int grid = resident_grid(k_pack<KIND, MULTI, true>, sms, p.total_tiles);
        k_pack<KIND, MULTI, true><<<grid, kEwThreads, 0, s>>>(p);
        return cudaGetLastError();
    }
    const int grid = resident_grid(k_pack<KIND, MULTI, false>, sms, p.total_tiles);
    k_pack<KIND, MULTI, false><<<grid, kEwThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_pack(const EwParams& p, int sms, bool from_momentum, cudaStream_t s) {
    if (!from_momentum) return run_pack<kInput, false>(p, sms, s);
    const bool multi = p.g_count > 1;
    if (p.src_dtype == kSrcF32) return multi ? run_pack<kMomF32, true>(p, sms, s) : run_pack<kMomF32, false>(p, sms, s);
    return multi ? run_pack<kMomBf16, true>(p, sms, s) : run_pack<kMomBf16, false>(p, sms, s);
}

template <int KIND>
cudaError_t run_unpack(const EwParams& p, int sms, cudaStream_t s) {
    const int grid = resident_grid(k_unpack<KIND>, sms, p.total_tiles);
    k_unpack<KIND><<<grid, kEwThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const EwParams& p, int sms, bool weight_update, cudaStream_t s) {
    if (!weight_update) return run_unpack<kStoreBf16>(p, sms, s);
    if (p.dst_dtype == kSrcF32) return run_unpack<kWF32>(p, sms, s);
    return run_unpack<kWBf16>(p, sms, s);
}

}  // namespace muon
