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
// once.  HBM-bound: 8 consecutive elements per thread (16-byte bf16 vectors),
// 2048-element tiles, grid-stride persistent grid.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace muon {
namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 8;
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
            if (GBF16) {
                const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(T.g) + base);
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(h[i]);
                    g[2 * i] = f.x;
                    g[2 * i + 1] = f.y;
                }
            } else {
                const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(T.g) + base);
                const float4 a = s[0], b = s[1];
                g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w; g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
            }
            const float4* ms = reinterpret_cast<const float4*>(T.m + base);
            const float4* vs = reinterpret_cast<const float4*>(T.v + base);
            const float4 m0 = ms[0], m1 = ms[1], v0 = vs[0], v1 = vs[1];
            m[0] = m0.x; m[1] = m0.y; m[2] = m0.z; m[3] = m0.w; m[4] = m1.x; m[5] = m1.y; m[6] = m1.z; m[7] = m1.w;
            v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w; v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
            if (PBF16) {
                const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(T.p) + base);
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(h[i]);
                    w[2 * i] = f.x;
                    w[2 * i + 1] = f.y;
                }
            } else {
                const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(T.p) + base);
                const float4 a = s[0], b = s[1];
                w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
            }
#pragma unroll
            for (int i = 0; i < kPerThread; ++i) adam1(p, g[i], m[i], v[i], w[i]);
            float4* md = reinterpret_cast<float4*>(T.m + base);
            float4* vd = reinterpret_cast<float4*>(T.v + base);
            md[0] = make_float4(m[0], m[1], m[2], m[3]);
            md[1] = make_float4(m[4], m[5], m[6], m[7]);
            vd[0] = make_float4(v[0], v[1], v[2], v[3]);
            vd[1] = make_float4(v[4], v[5], v[6], v[7]);
            if (PBF16) {
                uint4 raw;
                __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
                for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(w[2 * i], w[2 * i + 1]);
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(T.p) + base) = raw;
            } else {
                float4* d = reinterpret_cast<float4*>(static_cast<float*>(T.p) + base);
                d[0] = make_float4(w[0], w[1], w[2], w[3]);
                d[1] = make_float4(w[4], w[5], w[6], w[7]);
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
