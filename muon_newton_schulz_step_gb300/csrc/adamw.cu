// AdamW for the parameters Muon does not cover ("Domyn is training a
// 1T-parameter MoE on Europe's Jupiter supercomputer, and published the
// recipe", table "The model and the machine": Muon for about 99.5% of the
// parameters, AdamW for the rest -- vectors, norms, embeddings).
//
// One launch updates a ragged list of flat tensors.  Every operation is a
// single IEEE fp32 rounding (explicit _rn intrinsics, no contraction):
//   m' = fma(beta1, m, b1c*g)
//   v' = fma(beta2, v, b2c*(g*g))
//   p' = round_P( fma(-step_size, m' / (sqrt(v') * inv_sqrt_bc2 + eps), dcy*p) )
// with b1c = 1-beta1, b2c = 1-beta2, dcy = 1-lr*wd, step_size = lr/(1-beta1^t),
// inv_sqrt_bc2 = 1/sqrt(1-beta2^t) computed on the host in double and rounded
// once.  HBM-bound: 16 consecutive elements per thread in 8-element groups
// (16-byte bf16 vectors; 16 rather than 8 elements per thread keep twice the
// bytes in flight: 96 % instead of 88 % of the copy bandwidth), 4096-element
// tiles, grid-stride persistent grid.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace muon {
namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 16;
constexpr int kGroups = kPerThread / 8;
constexpr long long kTileElems = kThreads * kPerThread;

__device__ __forceinline__ int find_tensor(const AdamWParams& p, long long t) {
    int lo = 0, hi = p.ntensors - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.t[mid].tile0 <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void adam1(const AdamWParams& p, float g, float& m, float& v, float& w) {
    const float gm = __fmul_rn(p.b1c, g);
    m = __fmaf_rn(p.beta1, m, gm);
    const float gg = __fmul_rn(g, g);
    const float gv = __fmul_rn(p.b2c, gg);
    v = __fmaf_rn(p.beta2, v, gv);
    const float denom = __fadd_rn(__fmul_rn(__fsqrt_rn(v), p.inv_sqrt_bc2), p.eps);
    const float ratio = __fdiv_rn(m, denom);
    w = __fmaf_rn(-p.step_size, ratio, __fmul_rn(p.dcy, w));
}

// 8 consecutive elements (16-byte aligned) to and from fp32 registers
__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16* src, float* f) {
    const uint4 raw = *reinterpret_cast<const uint4*>(src);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ void load_f32x8(const float* src, float* f) {
    const float4 a = reinterpret_cast<const float4*>(src)[0], b = reinterpret_cast<const float4*>(src)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ void store_bf16x8(__nv_bfloat16* dst, const float* f) {
    uint4 raw;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<uint4*>(dst) = raw;
}

__device__ __forceinline__ void store_f32x8(float* dst, const float* f) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

template <int PBF16, int GBF16>
__global__ void __launch_bounds__(kThreads) k_adamw(const __grid_constant__ AdamWParams p) {
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        const int ti = find_tensor(p, t);
        const AdamWTensor& T = p.t[ti];
        const long long base = (t - T.tile0) * kTileElems + static_cast<long long>(threadIdx.x) * kPerThread;
        if (base >= T.n) continue;
        float g[kPerThread], m[kPerThread], v[kPerThread], w[kPerThread];
        const bool full = base + kPerThread <= T.n;
        if (full) {
#pragma unroll
            for (int c = 0; c < kGroups; ++c) {
                const long long e = base + 8 * c;
                float* gc = g + 8 * c;
                float* wc = w + 8 * c;
                if (GBF16) {
                    load_bf16x8(static_cast<const __nv_bfloat16*>(T.g) + e, gc);
                } else {
                    load_f32x8(static_cast<const float*>(T.g) + e, gc);
                }
                load_f32x8(T.m + e, m + 8 * c);
                load_f32x8(T.v + e, v + 8 * c);
                if (PBF16) {
                    load_bf16x8(static_cast<const __nv_bfloat16*>(T.p) + e, wc);
                } else {
                    load_f32x8(static_cast<const float*>(T.p) + e, wc);
                }
            }
#pragma unroll
            for (int i = 0; i < kPerThread; ++i) adam1(p, g[i], m[i], v[i], w[i]);
#pragma unroll
            for (int c = 0; c < kGroups; ++c) {
                const long long e = base + 8 * c;
                store_f32x8(T.m + e, m + 8 * c);
                store_f32x8(T.v + e, v + 8 * c);
                if (PBF16) {
                    store_bf16x8(static_cast<__nv_bfloat16*>(T.p) + e, w + 8 * c);
                } else {
                    store_f32x8(static_cast<float*>(T.p) + e, w + 8 * c);
                }
            }
        } else {
            const int n = static_cast<int>(T.n - base);
            for (int i = 0; i < n; ++i) {
                const long long e = base + i;
                const float gi = GBF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(T.g)[e])
                                       : static_cast<const float*>(T.g)[e];
                float mi = T.m[e], vi = T.v[e];
                float wi = PBF16 ? __bfloat162float(static_cast<__nv_bfloat16*>(T.p)[e]) : static_cast<float*>(T.p)[e];
                adam1(p, gi, mi, vi, wi);
                T.m[e] = mi;
                T.v[e] = vi;
                if (PBF16) static_cast<__nv_bfloat16*>(T.p)[e] = __float2bfloat16_rn(wi);
                else static_cast<float*>(T.p)[e] = wi;
            }
        }
    }
}

}  // namespace

long long adamw_tile_elems() { return kTileElems; }

template <int PBF16, int GBF16>
cudaError_t run_adamw(const AdamWParams& p, int sms, cudaStream_t s) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_adamw<PBF16, GBF16>, kThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const long long cap = static_cast<long long>(sms) * per_sm;
    const int grid = static_cast<int>(p.total_tiles < cap ? p.total_tiles : cap);
    k_adamw<PBF16, GBF16><<<grid, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_adamw(const AdamWParams& p, int sms, cudaStream_t s) {
    if (p.p_bf16 && p.g_bf16) return run_adamw<1, 1>(p, sms, s);
    if (p.p_bf16) return run_adamw<1, 0>(p, sms, s);
    if (p.g_bf16) return run_adamw<0, 1>(p, sms, s);
    return run_adamw<0, 0>(p, sms, s);
}

}  // namespace muon
