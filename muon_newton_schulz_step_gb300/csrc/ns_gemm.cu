// Newton-Schulz products on the sm_103a tensor cores.
//
// One persistent kernel runs one of the three products of a Newton-Schulz
// iteration (the orthogonalisation step of Muon, which "operates on full
// matrices" -- "How PyTorch Scaled a Near-1T MoE on Europe's Public
// Supercomputer", section "Three optimizations that changed the economics",
// FlexShard bullet) over every matrix of every shape bucket in one launch:
//
//   kGram    A = bf16(X X^T)            M = N = r, K = k   symmetric: only tiles
//                                                          touching the upper triangle
//   kPoly    B = bf16(b A + c A A)      M = N = K = r       symmetric, A A = A A^T
//   kUpdate  X' = bf16(a X + B X)       M = r, N = k, K = r
//
// X is r x k row-major (r <= k), A and B are r x r; every buffer is padded
// with zeros to multiples of 256, which keeps the iteration exact and lets
// every tile be full.
//
// Per CTA (one per SM, 192 threads):
//   warp 0     TMA producer: 4-stage ring of {A tile 128x64, B tile 256x64}
//              bf16, 128-byte swizzled, completion on an mbarrier
//   warp 1     TMEM owner (512 columns = two 128x256 fp32 accumulators) and
//              single-thread issuer of tcgen05.mma (M=128, N=256, K=16)
//   warps 2-5  epilogue: tcgen05.ld the accumulator, apply the fused
//              polynomial term, round to bf16, store (mirrored for the
//              symmetric products); overlaps the next tile's main loop
//
// In kGram / kPoly both operands are K-major rows of the same r x K matrix
// (X rows for X X^T; A rows for A A, using A = A^T).  In kUpdate the B
// operand X[p][j] is read MN-major (j contiguous) straight from the row-major
// iterate, so no transposed copy of X is ever made.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace muon {

// Device-side status word: 0, or MUON_ERR_TIMEOUT (5) after a bounded wait ran out.
__device__ int g_muon_device_error = 0;

namespace {

constexpr int kGemmThreads = 192;
constexpr uint32_t kStageA = kBM * kBK * 2;           // 16 KB
constexpr uint32_t kStageB = kBN * kBK * 2;           // 32 KB
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr uint32_t kTmemCols = 2 * kBN;                // two fp32 accumulators
constexpr uint64_t kWaitLimitNs = 2000000000ull;       // 2 s per wait
constexpr uint64_t kDrainLimitNs = 20000000ull;        // 20 ms when unwinding
constexpr int kErrTimeout = 5;

struct TileCoord {
    int bucket, mat, tm, tn;
};

__device__ __forceinline__ TileCoord decode_tile(const GemmParams& p, int t) {
    int bi = 0;
    while (bi + 1 < p.nbuckets && t >= p.b[bi + 1].tile0) ++bi;
    const GemmBucket& B = p.b[bi];
    const int local = t - B.tile0;
    TileCoord c;
    c.bucket = bi;
    c.mat = local / B.tiles_per_mat;
    int r = local - c.mat * B.tiles_per_mat;
    if (p.mode == kUpdate) {
        c.tm = r / B.nt;
        c.tn = r - c.tm * B.nt;
    } else {
        // Tiles whose rows [128 tm, +128) and columns [256 tn, +256) reach the
        // upper triangle (col >= row) are those with tm < 2 tn + 2; they are
        // numbered column by column.
        int tn = 0;
        for (;;) {
            const int h = min(B.mt, 2 * tn + 2);
            if (r < h) break;
            r -= h;
            ++tn;
        }
        c.tm = r;
        c.tn = tn;
    }
    return c;
}

__device__ __forceinline__ void record_failure(volatile int* abort) {
    atomicCAS(&g_muon_device_error, 0, kErrTimeout);
    *abort = 1;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
    uint4 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
}

__global__ void __launch_bounds__(kGemmThreads, 1) ns_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment: the 128-byte swizzle pattern repeats every 8 rows.
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kStageA;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kStageB);
    uint64_t* full = bars;                   // [kStages] TMA -> MMA
    uint64_t* empty = bars + kStages;        // [kStages] MMA -> TMA
    uint64_t* tfull = bars + 2 * kStages;    // [2] MMA -> epilogue
    uint64_t* tempty = bars + 2 * kStages + 2;  // [2] epilogue -> MMA
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_addr(&tfull[a]), 1);
            ptx::mbar_init(ptx::smem_addr(&tempty[a]), 128);
        }
        *abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int b = 0; b < p.nbuckets; ++b) {
            ptx::prefetch_tmap(&p.b[b].tmA);
            ptx::prefetch_tmap(&p.b[b].tmB);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int armed[kStages];
            uint32_t armed_parity[kStages];
            for (int s = 0; s < kStages; ++s) armed[s] = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
                const TileCoord c = decode_tile(p, t);
                const GemmBucket& B = p.b[c.bucket];
                for (int kb = 0; kb < B.kblocks; ++kb) {
                    if (!ptx::wait_parity(ptx::smem_addr(&empty[stage]), phase ^ 1u, abort,
                                          kWaitLimitNs)) {
                        record_failure(abort);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = ptx::smem_addr(&full[stage]);
                    ptx::mbar_arrive_expect_tx(fb, kStageBytes);
                    armed[stage] = 1;
                    armed_parity[stage] = phase;
                    ptx::tma_load_3d(ptx::smem_addr(sA + stage * kStageA), &B.tmA, fb, kb * kBK,
                                     c.tm * kBM, c.mat);
                    const uint32_t sb = ptx::smem_addr(sB + stage * kStageB);
                    if (p.mode == kUpdate) {
                        // four 64-column MN-major blocks of X rows [64 kb, +64)
#pragma unroll
                        for (int q = 0; q < kBN / 64; ++q)
                            ptx::tma_load_3d(sb + q * (kBK * 128), &B.tmB, fb, c.tn * kBN + q * 64,
                                             kb * kBK, c.mat);
                    } else {
                        ptx::tma_load_3d(sb, &B.tmB, fb, kb * kBK, c.tn * kBN, c.mat);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok || *abort) {
                // unwinding: let the copies already issued land before the CTA exits
                for (int s = 0; s < kStages; ++s)
                    if (armed[s])
                        ptx::wait_parity(ptx::smem_addr(&full[s]), armed_parity[s], nullptr,
                                        kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA --
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(kBM, kBN, false, p.mode == kUpdate);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x, ++it) {
                const TileCoord c = decode_tile(p, t);
                const GemmBucket& B = p.b[c.bucket];
                const int acc = it & 1;
                const uint32_t aphase = static_cast<uint32_t>(it >> 1) & 1u;
                if (!ptx::wait_parity(ptx::smem_addr(&tempty[acc]), aphase ^ 1u, abort,
                                      kWaitLimitNs)) {
                    record_failure(abort);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kBN);
                for (int kb = 0; kb < B.kblocks; ++kb) {
                    if (!ptx::wait_parity(ptx::smem_addr(&full[stage]), phase, abort,
                                          kWaitLimitNs)) {
                        record_failure(abort);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a0 = ptx::smem_addr(sA + stage * kStageA);
                    const uint32_t b0 = ptx::smem_addr(sB + stage * kStageB);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // K-major, 128B swizzle: a K step of 16 bf16 is +32 bytes
                        const uint64_t ad = ptx::sdesc_sw128(a0 + kk * 32, 16, 1024);
                        // MN-major, 128B swizzle: a K step of 16 rows is +2048 bytes;
                        // 64-column blocks are kBK*128 bytes apart (LBO), 8-row groups 1024 (SBO)
                        const uint64_t bd =
                            (p.mode == kUpdate) ? ptx::sdesc_sw128(b0 + kk * 2048, kBK * 128, 1024)
                                                : ptx::sdesc_sw128(b0 + kk * 32, 16, 1024);
                        ptx::mma_bf16(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(ptx::smem_addr(&empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(ptx::smem_addr(&tfull[acc]));
            }
        }
    } else {
        // ------------------------------------------------------ epilogue --
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        int it = 0;
        for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
            const TileCoord c = decode_tile(p, t);
            const GemmBucket& B = p.b[c.bucket];
            const int acc = it & 1;
            const uint32_t aphase = static_cast<uint32_t>(it >> 1) & 1u;
            const int row = c.tm * kBM + q * 32 + lane;
            const size_t mat_off = static_cast<size_t>(c.mat) * static_cast<size_t>(B.mat_stride);
            __nv_bfloat16* out = B.out + mat_off;
            const size_t ld = static_cast<size_t>(B.ld);
            // The epilogue operand (A for the polynomial, X for the update) does not
            // depend on this tile's products: load this thread's 256-element row
            // segment before waiting, so its latency hides under the main loop.
            uint4 pre[kBN / 8];
            if (p.mode != kGram) {
                const uint4* src = reinterpret_cast<const uint4*>(B.epi + mat_off + row * ld + c.tn * kBN);
#pragma unroll
                for (int g = 0; g < kBN / 8; ++g) pre[g] = __ldg(src + g);
            }
            if (!ptx::wait_parity(ptx::smem_addr(&tfull[acc]), aphase, abort, kWaitLimitNs)) {
                record_failure(abort);
                break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int ch = 0; ch < kBN / 32; ++ch) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(
                    tmem_base + static_cast<uint32_t>(acc * kBN + ch * 32) +
                        (static_cast<uint32_t>(q * 32) << 16),
                    r);
                ptx::tmem_wait_ld();
                const int col0 = c.tn * kBN + ch * 32;
                float v[32];
                if (p.mode == kGram) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                } else {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float e[8];
                        unpack8(pre[ch * 4 + g], e);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float s = __uint_as_float(r[8 * g + j]);
                            v[8 * g + j] = (p.mode == kPoly)
                                               ? __fadd_rn(__fmul_rn(p.bcoef, e[j]), __fmul_rn(p.c, s))
                                               : __fadd_rn(__fmul_rn(p.a, e[j]), s);
                        }
                    }
                }
                if (p.mode == kUpdate || col0 >= row) {
                    // every element of the chunk is on or above the diagonal (or no symmetry)
                    uint4* dst = reinterpret_cast<uint4*>(out + row * ld + col0);
#pragma unroll
                    for (int g = 0; g < 4; ++g) dst[g] = pack8(&v[8 * g]);
                } else if (col0 + 31 >= row) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j >= row) out[row * ld + col0 + j] = __float2bfloat16_rn(v[j]);
                }
                if (p.mode != kUpdate && col0 + 31 > row) {
                    // mirror the strict upper part: lanes hold consecutive rows, so each
                    // of these stores writes 64 contiguous bytes across the warp
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j > row)
                            out[static_cast<size_t>(col0 + j) * ld + row] = __float2bfloat16_rn(v[j]);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_addr(&tempty[acc]));
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

size_t gemm_smem_bytes() {
    return 1024 + kStages * kStageBytes + (2 * kStages + 4) * sizeof(uint64_t) + 16;
}

cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t s) {
    // the attribute belongs to the current device's context: set it on every launch (cheap)
    cudaError_t e = cudaFuncSetAttribute(ns_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(gemm_smem_bytes()));
    if (e != cudaSuccess) return e;
    ns_gemm_kernel<<<grid, kGemmThreads, gemm_smem_bytes(), s>>>(p);
    return cudaGetLastError();
}

cudaError_t read_and_clear_device_error(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_muon_device_error, sizeof(int));
    if (e != cudaSuccess) return e;
    *code = v;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_muon_device_error, &zero, sizeof(int));
}

}  // namespace muon
