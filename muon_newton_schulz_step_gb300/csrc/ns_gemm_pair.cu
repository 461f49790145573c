// Newton-Schulz products on pairs of SMs (tcgen05 cta_group::2).
//
// Same three products as ns_gemm.cu -- the Gram X X^T, the polynomial
// b A + c A A and the update a X + B X of one Newton-Schulz iteration of Muon,
// the orthogonalisation that "operates on full matrices" ("How PyTorch Scaled
// a Near-1T MoE on Europe's Public Supercomputer", section "Three
// optimizations that changed the economics", FlexShard bullet) -- but each
// 256 x 256 output tile is computed by a cluster of two CTAs on two SMs:
//
//   * the even CTA ("leader") issues tcgen05.mma.cta_group::2 with M = 256:
//     rows 0-127 of the tile accumulate in the leader's TMEM, rows 128-255 in
//     the peer's;
//   * each CTA TMA-loads its own 128 rows of the A operand and its own half
//     (128 of the 256 columns) of the B operand, so per SM and per K step the
//     tensor core reads 8 KB of shared memory instead of 12 KB and TMA writes
//     32 KB per stage instead of 48 KB;
//   * both CTAs' loads complete on the leader's "full" barrier; the leader's
//     commits are multicast to both CTAs' "empty" and "accumulator full"
//     barriers; both CTAs' epilogue warps release an accumulator on the
//     leader's "accumulator empty" barrier.
//
// Per CTA: warp 0 TMA producer (6-stage ring, 32 KB per stage), warp 1 TMEM
// owner + MMA issuer (leader only), warps 2-5 epilogue on the CTA's own 128
// accumulator rows.  Symmetric products compute only tiles with tm <= tn and
// mirror their strict upper part.  Every wait is bounded (see ptx.cuh).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace muon {

// Device-side status word of this kernel: 0, or MUON_ERR_TIMEOUT (5).
__device__ int g_muon_pair_error = 0;

namespace {

constexpr int kThreads = 192;
constexpr int kTile = 256;                              // output tile edge (pair)
constexpr int kHalf = 128;                              // rows / B columns per CTA
constexpr int kPairStages = 6;
constexpr uint32_t kStageA = kHalf * kBK * 2;           // 16 KB
constexpr uint32_t kStageB = kHalf * kBK * 2;           // 16 KB
constexpr uint32_t kStageBytes = kStageA + kStageB;     // per CTA
constexpr uint32_t kTmemCols = 2 * kTile;               // two 128 x 256 fp32 accumulators per CTA
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 20000000ull;
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
        // upper-triangle 256 x 256 tiles (tm <= tn), numbered column by column
        int tn = 0;
        while (r > tn) {
            r -= tn + 1;
            ++tn;
        }
        c.tm = r;
        c.tn = tn;
    }
    return c;
}

__device__ __forceinline__ void record_failure(volatile int* abort) {
    atomicCAS(&g_muon_pair_error, 0, kErrTimeout);
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

__global__ void __launch_bounds__(kThreads, 1) ns_gemm_pair_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kPairStages * kStageA;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kPairStages * kStageB);
    uint64_t* full = bars;                          // [stages] loads of both CTAs -> MMA (leader's used)
    uint64_t* empty = bars + kPairStages;           // [stages] MMA -> this CTA's producer
    uint64_t* tfull = bars + 2 * kPairStages;       // [2] MMA -> this CTA's epilogue
    uint64_t* tempty = bars + 2 * kPairStages + 2;  // [2] both epilogues -> MMA (leader's used)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kPairStages + 4);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();   // 0 = leader, 1 = peer
    const bool leader = rank == 0;
    const int pair = static_cast<int>(ptx::cluster_id_x());
    const int npairs = static_cast<int>(ptx::num_clusters_x());

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_addr(&tfull[a]), 1);
            ptx::mbar_init(ptx::smem_addr(&tempty[a]), 8);  // 4 epilogue warps x 2 CTAs
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
        ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();   // barriers of both CTAs initialised and TMEM allocated before any use
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int armed[kPairStages];
            uint32_t armed_parity[kPairStages];
            for (int s = 0; s < kPairStages; ++s) armed[s] = 0;
            bool ok = true;
            for (int t = pair; ok && t < p.total_tiles; t += npairs) {
                const TileCoord c = decode_tile(p, t);
                const GemmBucket& B = p.b[c.bucket];
                const int arow = c.tm * kTile + static_cast<int>(rank) * kHalf;
                const int bcol = c.tn * kTile + static_cast<int>(rank) * kHalf;
                for (int kb = 0; kb < B.kblocks; ++kb) {
                    if (!ptx::wait_parity_cluster(ptx::smem_addr(&empty[stage]), phase ^ 1u, abort,
                                                  kWaitLimitNs)) {
                        record_failure(abort);
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = ptx::smem_addr(&full[stage]);
                    const uint32_t fb = ptx::mapa_shared(fb_local, 0);   // the leader's barrier
                    if (leader) {
                        ptx::mbar_arrive_expect_tx(fb_local, 2 * kStageBytes);
                        armed[stage] = 1;
                        armed_parity[stage] = phase;
                    }
                    ptx::tma_load_3d_pair(ptx::smem_addr(sA + stage * kStageA), &B.tmA, fb, kb * kBK, arow,
                                          c.mat);
                    const uint32_t sb = ptx::smem_addr(sB + stage * kStageB);
                    if (p.mode == kUpdate) {
                        // two 64-column MN-major blocks of X rows [64 kb, +64)
                        ptx::tma_load_3d_pair(sb, &B.tmB, fb, bcol, kb * kBK, c.mat);
                        ptx::tma_load_3d_pair(sb + kBK * 128, &B.tmB, fb, bcol + 64, kb * kBK, c.mat);
                    } else {
                        ptx::tma_load_3d_pair(sb, &B.tmB, fb, kb * kBK, bcol, c.mat);
                    }
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (leader && (!ok || *abort)) {
                for (int s = 0; s < kPairStages; ++s)
                    if (armed[s])
                        ptx::wait_parity_cluster(ptx::smem_addr(&full[s]), armed_parity[s], nullptr,
                                                 kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA --
        if (leader && lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(kTile, kTile, false, p.mode == kUpdate);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int t = pair; ok && t < p.total_tiles; t += npairs, ++it) {
                const TileCoord c = decode_tile(p, t);
                const GemmBucket& B = p.b[c.bucket];
                const int acc = it & 1;
                const uint32_t aphase = static_cast<uint32_t>(it >> 1) & 1u;
                if (!ptx::wait_parity_cluster(ptx::smem_addr(&tempty[acc]), aphase ^ 1u, abort,
                                              kWaitLimitNs)) {
                    record_failure(abort);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kTile);
                for (int kb = 0; kb < B.kblocks; ++kb) {
                    if (!ptx::wait_parity_cluster(ptx::smem_addr(&full[stage]), phase, abort,
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
                        const uint64_t ad = ptx::sdesc_sw128(a0 + kk * 32, 16, 1024);
                        const uint64_t bd =
                            (p.mode == kUpdate) ? ptx::sdesc_sw128(b0 + kk * 2048, kBK * 128, 1024)
                                                : ptx::sdesc_sw128(b0 + kk * 32, 16, 1024);
                        ptx::mma_bf16_pair(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    ptx::mma_commit_pair(ptx::smem_addr(&empty[stage]), 0x3);
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit_pair(ptx::smem_addr(&tfull[acc]), 0x3);
            }
        }
    } else {
        // ------------------------------------------------------ epilogue --
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t tempty_leader0 = ptx::mapa_shared(ptx::smem_addr(&tempty[0]), 0);
        const uint32_t tempty_leader1 = ptx::mapa_shared(ptx::smem_addr(&tempty[1]), 0);
        int it = 0;
        for (int t = pair; t < p.total_tiles; t += npairs, ++it) {
            const TileCoord c = decode_tile(p, t);
            const GemmBucket& B = p.b[c.bucket];
            const int acc = it & 1;
            const uint32_t aphase = static_cast<uint32_t>(it >> 1) & 1u;
            const int row = c.tm * kTile + static_cast<int>(rank) * kHalf + q * 32 + lane;
            const size_t mat_off = static_cast<size_t>(c.mat) * static_cast<size_t>(B.mat_stride);
            __nv_bfloat16* out = B.out + mat_off;
            const size_t ld = static_cast<size_t>(B.ld);
            // the epilogue operand does not depend on this tile's products: load it now
            uint4 pre[kTile / 8];
            if (p.mode != kGram) {
                const uint4* src = reinterpret_cast<const uint4*>(B.epi + mat_off + row * ld + c.tn * kTile);
#pragma unroll
                for (int g = 0; g < kTile / 8; ++g) pre[g] = __ldg(src + g);
            }
            if (!ptx::wait_parity_cluster_backoff(ptx::smem_addr(&tfull[acc]), aphase, abort, kWaitLimitNs, 256)) {
                record_failure(abort);
                break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int ch = 0; ch < kTile / 32; ++ch) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(
                    tmem_base + static_cast<uint32_t>(acc * kTile + ch * 32) +
                        (static_cast<uint32_t>(q * 32) << 16),
                    r);
                ptx::tmem_wait_ld();
                const int col0 = c.tn * kTile + ch * 32;
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
                    uint4* dst = reinterpret_cast<uint4*>(out + row * ld + col0);
#pragma unroll
                    for (int g = 0; g < 4; ++g) dst[g] = pack8(&v[8 * g]);
                } else if (col0 + 31 >= row) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j >= row) out[row * ld + col0 + j] = __float2bfloat16_rn(v[j]);
                }
                if (p.mode != kUpdate && col0 + 31 > row) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j > row)
                            out[static_cast<size_t>(col0 + j) * ld + row] = __float2bfloat16_rn(v[j]);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();   // no CTA leaves while its peer may still signal its barriers
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

}  // namespace

cudaError_t read_and_clear_pair_error(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_muon_pair_error, sizeof(int));
    if (e != cudaSuccess) return e;
    *code = v;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_muon_pair_error, &zero, sizeof(int));
}

size_t gemm_pair_smem_bytes() {
    return 1024 + kPairStages * kStageBytes + (2 * kPairStages + 4) * sizeof(uint64_t) + 16;
}

cudaError_t launch_gemm_pair(const GemmParams& p, int npairs, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(ns_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(gemm_pair_smem_bytes()));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * npairs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = gemm_pair_smem_bytes();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, ns_gemm_pair_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace muon
