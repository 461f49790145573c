// Newton-Schulz products on pairs of SMs (tcgen05 cta_group::2).
//
// The three products of one Newton-Schulz iteration of Muon -- the Gram
// X X^T, the polynomial b A + c A A and the update a X + B X -- the
// orthogonalisation that "operates on full matrices" ("How PyTorch Scaled
// a Near-1T MoE on Europe's Public Supercomputer", section "Three
// optimizations that changed the economics", FlexShard bullet).  Each
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
// Per CTA: warp 0 TMA producer (5- or 6-stage ring, 32 KB per stage), warp 1
// TMEM owner + MMA issuer (leader only), warps 2-9 epilogue on the CTA's own
// 128 accumulator rows (two warps per TMEM lane quadrant, each on half of the
// tile's columns; 4 warps for the plain update).  Symmetric products compute
// only tiles with tm <= tn.  By default they also store only those tiles (the
// diagonal ones in full, their strict upper part mirrored), and the products
// that read them (polynomial: A, update: B) take each K block left of the row
// tile's diagonal from the stored transpose, as MN-major 64 x 64 blocks: the
// same values, since the matrix is symmetric bit for bit.  Every wait is
// bounded (see ptx.cuh).
//
// The last update of the iteration can run with a fused epilogue (template
// argument FK, FinalKind): O = bf16(a X + B X) goes straight to the caller's
// matrix in its stored orientation -- W <- dcy*W - s*O, the decoupled weight
// decay and scaled step of Muon ("Domyn is training a 1T-parameter MoE on
// Europe's Jupiter supercomputer, and published the recipe", table "The model
// and the machine": Muon with weight decay), or the store of O for the
// Newton-Schulz-only call -- with the same roundings as the separate weight
// update kernel: O rounded to bf16, then one fma in fp32, then W's dtype.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace muon {

// Device-side status word of this kernel: 0, or MUON_ERR_TIMEOUT (5).
__device__ int g_muon_pair_error = 0;

namespace {

// Epilogue warps per CTA (a multiple of 4: each TMEM lane quadrant gets
// EW / 4 warps, which split the tile's columns between them).  The update
// product keeps one warp per quadrant; the symmetric products and the fused
// final update use two.
constexpr int kUpdateEpiWarps = 4;
constexpr int kEpiWarps = 8;
constexpr int kTile = 256;                              // output tile edge (pair)
constexpr int kHalf = 128;                              // rows / B columns per CTA
constexpr int kPairStages = 6;
constexpr uint32_t kStageA = kHalf * kBK * 2;           // 16 KB
constexpr uint32_t kStageB = kHalf * kBK * 2;           // 16 KB
constexpr uint32_t kStageBytes = kStageA + kStageB;     // per CTA
constexpr uint32_t kTmemCols = 2 * kTile;               // two 128 x 256 fp32 accumulators per CTA
constexpr uint32_t kBarBytes = 256;                     // mbarriers, TMEM address, abort flag
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

// Update product on clusters of two pairs: item w is a pair of horizontally
// adjacent tiles (tm, 2 j) and (tm, 2 j + 1) of one matrix; pair `pp` of the
// cluster takes the second one.  Both need the same rows of the A operand,
// which the two pairs load once between them and multicast.  With an odd
// number of tile columns the last item's second tile lies beyond the matrix
// (valid = false): its pair loads zeros for B, computes, and stores nothing.
struct ItemCoord {
    TileCoord c;
    bool valid;
};

template <int CS>
__device__ __forceinline__ ItemCoord decode_item(const GemmParams& p, int w, int pp) {
    ItemCoord r;
    if constexpr (CS == 2) {
        r.c = decode_tile(p, w);
        r.valid = true;
    } else {
        int bi = 0;
        while (bi + 1 < p.nbuckets && w >= p.b[bi + 1].item0) ++bi;
        const GemmBucket& B = p.b[bi];
        const int per_mat = B.mt * B.nt2;
        const int local = w - B.item0;
        r.c.bucket = bi;
        r.c.mat = local / per_mat;
        const int q = local - r.c.mat * per_mat;
        r.c.tm = q / B.nt2;
        r.c.tn = 2 * (q - r.c.tm * B.nt2) + pp;
        r.valid = r.c.tn < B.nt;
    }
    return r;
}

template <int CS>
__device__ __forceinline__ int total_items(const GemmParams& p) {
    return CS == 2 ? p.total_tiles : p.total_items;
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

struct NoFinal {
    int unused;
};

// ---- fused final update --------------------------------------------------
// Per 32-column chunk of the accumulator an epilogue thread owns one oriented
// row (TMEM lane = row).  Accessing W in that layout would make every warp
// instruction touch 32 rows, i.e. 32 cache lines.  So the warp first rounds O
// to bf16 and exchanges its 32 x 32 block through shared memory (2 KB per
// warp), after which four lanes cover one 64-byte stored row segment: lane l
// holds stored rows sr + l/4 + 8i (i < 4), stored columns sc + 8 (l % 4) ..
// + 7.  A warp instruction on W then touches 8 lines.  For a transposed
// matrix the same exchange performs the transpose: the stored rows are the
// oriented columns.
constexpr int kFinChunks = kTile / 32;

// TMA epilogue of the update product: per epilogue warp, the iterate's 32 x 32
// blocks (this warp's 32 rows, one 32-column chunk) arrive by TMA in a ring of
// kTeDepth 2 KB buffers, and the rounded output blocks leave by TMA store from
// two 2 KB staging buffers (64-byte swizzle: a lane reading or writing its row
// in 16-byte units meets no bank conflict).  Neither direction goes through
// the load/store unit, whose row-per-lane accesses (one cache line per lane)
// would otherwise take a large share of the SM's L1 cycles from the operand
// traffic of the main loop.  Before an FP8 Gram the same blocks also leave as
// E4M3 (X' * 2^8, 32 x 32 bytes) from two 1 KB staging buffers: the next
// Gram's operands, written where X' is written.
constexpr int kTeDepth = 3;
constexpr uint32_t kTeBlock = 32 * 32 * 2;
constexpr uint32_t kTe8Block = 32 * 32;
constexpr uint32_t kTeWarpBytes = (kTeDepth + 2) * kTeBlock + 2 * kTe8Block;
// fused final update: the same input ring plus one exchange block per warp
constexpr uint32_t kFinWarpBytes = (kTeDepth + 1) * kTeBlock;
constexpr int kTeBarIndex = 18;     // first TE mbarrier (uint64 index into the barrier block)
constexpr uint32_t kXchgBytes = 32 * 32 * 2;                    // one 32 x 32 bf16 block

template <int EW>
struct Epi {
    static_assert(EW % 4 == 0 && EW >= 4 && EW <= 8, "epilogue warps");
    static constexpr int threads = 64 + 32 * EW;
    static constexpr int chunks = kFinChunks * 4 / EW;                           // 32-column chunks per warp
    static constexpr uint32_t xchg_bytes() { return EW * kXchgBytes; }           // one block per warp
};

template <int FK>
struct FinTraits {
    static constexpr int depth = FK == kFinWF32 ? 2 : (FK == kFinWBf16 ? 3 : 1);   // W chunks loaded ahead
    static constexpr int wslots = FK == kFinWF32 ? 32 : (FK == kFinWBf16 ? 16 : 1);
};

// Where one thread's four 8-element runs of a chunk lie in the stored
// matrix: rows sr + 8i (i < 4), columns sc .. sc + 7.
struct FinSeg {
    int sr, sc;
};

__device__ __forceinline__ FinSeg fin_seg(const FinalMat& f, int rowbase, int lane, int col0) {
    FinSeg g;
    if (!f.trans) {
        g.sr = rowbase + (lane >> 2);
        g.sc = col0 + (lane & 3) * 8;
    } else {
        g.sr = col0 + (lane >> 2);
        g.sc = rowbase + (lane & 3) * 8;
    }
    return g;
}

__device__ __forceinline__ bool fin_vec(const FinalMat& f, const FinSeg& g) { return f.vec && g.sc + 8 <= f.cols; }

// One chunk of W loaded ahead of use, in the exchanged layout (bf16: one
// 16-byte run per i; fp32: two).  The iterate X arrives by TMA.
template <int FK>
struct FinChunk {
    uint32_t w[FinTraits<FK>::wslots];
};

template <int FK>
__device__ __forceinline__ void fin_issue(const FinalMat& f, const FinSeg& g, FinChunk<FK>& b) {
    if (FK == kFinStore) return;
    constexpr int per = FinTraits<FK>::wslots / 4;   // 32-bit slots per run
    const bool vec = fin_vec(f, g);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = g.sr + 8 * i;
#pragma unroll
        for (int j = 0; j < per; ++j) b.w[per * i + j] = 0;
        if (r >= f.rows) continue;
        const size_t base = static_cast<size_t>(r) * f.cols + g.sc;
        if (vec) {
            const uint4* src = FK == kFinWF32
                                   ? reinterpret_cast<const uint4*>(static_cast<const float*>(f.w) + base)
                                   : reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(f.w) + base);
#pragma unroll
            for (int v = 0; v < per / 4; ++v) {
                const uint4 t = src[v];
                b.w[per * i + 4 * v] = t.x;
                b.w[per * i + 4 * v + 1] = t.y;
                b.w[per * i + 4 * v + 2] = t.z;
                b.w[per * i + 4 * v + 3] = t.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (g.sc + e < f.cols) {
                    if (FK == kFinWF32) {
                        b.w[per * i + e] = __float_as_uint(static_cast<const float*>(f.w)[base + e]);
                    } else {
                        const uint32_t h = __bfloat16_as_ushort(static_cast<const __nv_bfloat16*>(f.w)[base + e]);
                        b.w[per * i + (e >> 1)] |= h << (16 * (e & 1));
                    }
                }
            }
        }
    }
}

// W' = fma(-s, O, dcy * W) in fp32 (O already rounded to bf16).
__device__ __forceinline__ float weight_update(const FinalMat& f, float o, float w) {
    return __fmaf_rn(-f.s, o, __fmul_rn(f.dcy, w));
}

// Element e of run i of a chunk's W as fp32 (bf16 slots hold two elements).
template <int FK>
__device__ __forceinline__ float fin_w(const FinChunk<FK>& b, int i, int e) {
    if (FK == kFinWF32) return __uint_as_float(b.w[8 * i + e]);
    return __uint_as_float(((b.w[4 * i + (e >> 1)] >> (16 * (e & 1))) & 0xffffu) << 16);
}

// Exchange the warp's 32 x 32 block of rounded O (o: this lane's oriented row)
// into the layout of FinSeg; ob[i] receives the 8 bf16 values of run i.
__device__ __forceinline__ void fin_exchange(bool trans, const float (&o)[32], uint8_t* blk, int lane, uint4 (&ob)[4]) {
    if (!trans) {
        // row `lane`, 16-byte unit u of the row stored at unit (u + lane / 2) % 4:
        // conflict-free for the row-per-lane writes and the 4-lanes-per-row reads
#pragma unroll
        for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(blk + lane * 64 + (((u + (lane >> 1)) & 3) << 4)) = pack8(&o[8 * u]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rr = (lane >> 2) + 8 * i;
            ob[i] = *reinterpret_cast<const uint4*>(blk + rr * 64 + ((((lane & 3) + (rr >> 1)) & 3) << 4));
        }
    } else {
        // element (oriented row lane, column j) to block row j: the block holds
        // the stored layout, read back one 16-byte unit per lane and run
        __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(blk);
#pragma unroll
        for (int j = 0; j < 32; ++j) h[j * 32 + lane] = __float2bfloat16_rn(o[j]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rr = (lane >> 2) + 8 * i;
            ob[i] = *reinterpret_cast<const uint4*>(blk + rr * 64 + ((lane & 3) << 4));
        }
    }
    __syncwarp();   // the block is rewritten by the next chunk
}

// Store O (kFinStore) or the updated W, and the optional copy of O, for one
// chunk in the exchanged layout.
template <int FK>
__device__ __forceinline__ void fin_store(const FinalMat& f, const FinSeg& g, const uint4 (&ob)[4],
                                          const FinChunk<FK>& b) {
    const bool vec = fin_vec(f, g);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = g.sr + 8 * i;
        if (r >= f.rows) continue;
        const size_t base = static_cast<size_t>(r) * f.cols + g.sc;
        float o8[8];
        unpack8(ob[i], o8);
        if (vec) {
            if (f.oout != nullptr) *reinterpret_cast<uint4*>(f.oout + base) = ob[i];
            if (FK == kFinStore) {
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(f.w) + base) = ob[i];
            } else if (FK == kFinWBf16) {
                float r8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) r8[e] = weight_update(f, o8[e], fin_w<FK>(b, i, e));
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(f.w) + base) = pack8(r8);
            } else {
                float4* d = reinterpret_cast<float4*>(static_cast<float*>(f.w) + base);
                d[0] = make_float4(weight_update(f, o8[0], fin_w<FK>(b, i, 0)), weight_update(f, o8[1], fin_w<FK>(b, i, 1)),
                                   weight_update(f, o8[2], fin_w<FK>(b, i, 2)), weight_update(f, o8[3], fin_w<FK>(b, i, 3)));
                d[1] = make_float4(weight_update(f, o8[4], fin_w<FK>(b, i, 4)), weight_update(f, o8[5], fin_w<FK>(b, i, 5)),
                                   weight_update(f, o8[6], fin_w<FK>(b, i, 6)), weight_update(f, o8[7], fin_w<FK>(b, i, 7)));
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (g.sc + e < f.cols) {
                    const __nv_bfloat16 oe = __float2bfloat16_rn(o8[e]);
                    if (f.oout != nullptr) f.oout[base + e] = oe;
                    if (FK == kFinStore) {
                        static_cast<__nv_bfloat16*>(f.w)[base + e] = oe;
                    } else if (FK == kFinWBf16) {
                        static_cast<__nv_bfloat16*>(f.w)[base + e] =
                            __float2bfloat16_rn(weight_update(f, o8[e], fin_w<FK>(b, i, e)));
                    } else {
                        static_cast<float*>(f.w)[base + e] = weight_update(f, o8[e], fin_w<FK>(b, i, e));
                    }
                }
            }
        }
    }
}

// L2 prefetch of the W lines one warp's part of a tile will read in the fused
// epilogue: columns cb .. cb + ncols - 1 of the thread's oriented row (a
// stored row segment) or, transposed, of the warp's 32 oriented rows (one
// stored row segment per column).  Addresses stay inside W.
template <int FK>
__device__ __forceinline__ void fin_prefetch_w(const FinalMat& f, int row, int rowbase, int lane, int cb, int ncols,
                                               int fr, int fk) {
    if (FK == kFinStore || cb >= fk) return;
    constexpr int esz = FK == kFinWF32 ? 4 : 2;
    const char* w = static_cast<const char*>(f.w);
    const int n = min(ncols, fk - cb);
    if (!f.trans) {
        if (row >= fr) return;
        const char* a = w + (static_cast<size_t>(row) * f.cols + cb) * esz;
        const int bytes = n * esz;
        for (int o = 0; o < bytes; o += 128) ptx::prefetch_l2(a + o);
        ptx::prefetch_l2(a + bytes - 1);
    } else {
        if (rowbase >= fr) return;
        for (int j = lane; j < n; j += 32)
            ptx::prefetch_l2(w + (static_cast<size_t>(cb + j) * f.cols + rowbase) * esz);
    }
}

// XS (symmetric products only): store the tile and its mirror through the
// per-warp exchange block, 8 cache lines per instruction, instead of one row
// per lane and 2-byte mirror stores.  ST: pipeline stages.
// CS: CTAs per cluster -- 2 (one pair) or 4 (two pairs sharing the A operand
// of the update product by multicast; p.mode must be kUpdate).
// TE: the update's epilogue moves X and X' by TMA (p.mode must be kUpdate, FK kFinNone).
// F8: the Gram product on E4M3 operands (p.mode must be kGram).
template <int FK, int EW, bool XS, int ST, int CS, bool TE, bool F8, class FP>
__global__ void __launch_bounds__(Epi<EW>::threads, 1) ns_gemm_pair_kernel(const __grid_constant__ GemmParams p,
                                                                     const __grid_constant__ FP fin) {
    static_assert(CS == 2 || CS == 4, "cluster size");
    static_assert(!TE || (FK == kFinNone && !XS && ST <= 6), "TMA epilogue: plain update only");
    static_assert(!F8 || (FK == kFinNone && !TE && !XS), "FP8 operands: Gram only");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + ST * kStageA;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + ST * kStageB);
    uint64_t* full = bars;                          // [stages] loads of both CTAs -> MMA (leader's used)
    uint64_t* empty = bars + ST;           // [stages] MMA -> this CTA's producer
    uint64_t* tfull = bars + 2 * ST;       // [2] MMA -> this CTA's epilogue
    uint64_t* tempty = bars + 2 * ST + 2;  // [2] both epilogues -> MMA (leader's used)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * ST + 4);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // fused final update only: one 32 x 32 bf16 exchange block per epilogue warp
    uint8_t* xchg = reinterpret_cast<uint8_t*>(bars) + kBarBytes +
                    (threadIdx.x / 32 >= 2 ? (threadIdx.x / 32 - 2) * kXchgBytes : 0);
    // TMA epilogue only: kTeDepth input buffers and two staging buffers per epilogue
    // warp (1024-byte aligned, after the barrier block), kTeDepth mbarriers per warp
    uint8_t* te_buf = reinterpret_cast<uint8_t*>(bars) + 1024 +
                      (threadIdx.x / 32 >= 2 ? (threadIdx.x / 32 - 2) * (FK != kFinNone ? kFinWarpBytes : kTeWarpBytes)
                                             : 0);
    uint64_t* te_bar = bars + kTeBarIndex + (threadIdx.x / 32 >= 2 ? (threadIdx.x / 32 - 2) * kTeDepth : 0);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = ptx::cluster_ctarank();
    const uint32_t rank = crank & 1u;               // in the pair: 0 = leader, 1 = peer
    const uint32_t lead = crank & ~1u;              // cluster rank of this pair's leader
    const int pp = static_cast<int>(crank >> 1);    // pair within the cluster (CS == 4)
    const bool leader = rank == 0;
    const int pair = static_cast<int>(ptx::cluster_id_x());
    const int npairs = static_cast<int>(ptx::num_clusters_x());
    const int nitems = total_items<CS>(p);
    const uint64_t wait_limit = p.wait_ns != 0 ? p.wait_ns : kWaitLimitNs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
            // a stage is free once every pair that reads it (CS / 2 of them) is done with it
            ptx::mbar_init(ptx::smem_addr(&empty[s]), CS / 2);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_addr(&tfull[a]), 1);
            ptx::mbar_init(ptx::smem_addr(&tempty[a]), 2 * EW);  // every epilogue warp of both CTAs
        }
        if constexpr (TE || FK != kFinNone)
            for (int j = 0; j < EW * kTeDepth; ++j) ptx::mbar_init(ptx::smem_addr(&bars[kTeBarIndex + j]), 1);
        *abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int b = 0; b < p.nbuckets; ++b) {
            ptx::prefetch_tmap(&p.b[b].tmA);
            ptx::prefetch_tmap(&p.b[b].tmB);
            if constexpr (TE || FK != kFinNone) ptx::prefetch_tmap(&p.b[b].tmE);
            if constexpr (TE) ptx::prefetch_tmap(&p.b[b].tmO);
            if constexpr (TE)
                if (p.fp8_next) ptx::prefetch_tmap(&p.b[b].tmQ);
            if (p.upper_only && p.mode != kGram) ptx::prefetch_tmap(&p.b[b].tmT);
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
            // stages whose full barrier this leader armed, and the phase it armed (bit per stage;
            // kept in registers: the loop below is on the path that feeds the tensor pipe)
            uint32_t armed = 0, armed_parity = 0;
            const bool upd = p.mode == kUpdate;
            // upper-only symmetric operands: K blocks left of the row tile's diagonal come
            // from the stored transpose (never with clusters of two pairs).  They are
            // loaded by a loop of their own ahead of the main loop, which stays free of any
            // per-K-block choice (the producer feeds the tensor pipe as directly as the MMA
            // issuer: a second TMA path inside that loop, even never taken, cost 12 %)
            const bool sym_a = CS == 2 && p.upper_only && p.mode != kGram;
            const bool sym_b = CS == 2 && p.upper_only && p.mode == kPoly;
            bool ok = true;
            for (int t = pair; ok && t < nitems; t += npairs) {
                const TileCoord c = decode_item<CS>(p, t, pp).c;
                const GemmBucket& B = p.b[c.bucket];
                const int arow = c.tm * kTile + static_cast<int>(rank) * kHalf;
                const int bcol = c.tn * kTile + static_cast<int>(rank) * kHalf;
                const int kstep = F8 ? 2 * kBK : kBK;   // K elements per stage (128-byte rows)
                int kb = 0;
                if constexpr (CS == 2 && !F8) {
                    const int a_lim = sym_a ? c.tm * (kTile / kBK) : 0;        // A from the transpose below
                    const int t_end = sym_b ? c.tn * (kTile / kBK) : a_lim;    // B from the transpose below (polynomial)
                    for (; kb < t_end; ++kb) {
                        if (!ptx::wait_parity_cluster(ptx::smem_addr(&empty[stage]), phase ^ 1u, abort,
                                                      wait_limit)) {
                            record_failure(abort);
                            ok = false;
                            break;
                        }
                        const uint32_t fb_local = ptx::smem_addr(&full[stage]);
                        const uint32_t fb = ptx::mapa_shared(fb_local, lead);
                        if (leader) {
                            ptx::mbar_arrive_expect_tx(fb_local, 2 * kStageBytes);
                            armed |= 1u << stage;
                            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        }
                        const uint32_t sa = ptx::smem_addr(sA + stage * kStageA);
                        if (kb < a_lim) {
                            // rows [arow, +128) of K block kb = columns of the stored rows
                            // [64 kb, +64): two MN-major 64 x 64 blocks
                            ptx::tma_load_3d_pair(sa, &B.tmT, fb, arow, kb * kBK, c.mat);
                            ptx::tma_load_3d_pair(sa + kBK * 128, &B.tmT, fb, arow + 64, kb * kBK, c.mat);
                        } else {
                            ptx::tma_load_3d_pair(sa, &B.tmA, fb, kb * kBK, arow, c.mat);
                        }
                        // B: the update's iterate (always MN-major) or the polynomial's
                        // transpose, both as two 64-column blocks
                        const uint32_t sb = ptx::smem_addr(sB + stage * kStageB);
                        const CUtensorMap* mb = upd ? &B.tmB : &B.tmT;
                        ptx::tma_load_3d_pair(sb, mb, fb, bcol, kb * kBK, c.mat);
                        ptx::tma_load_3d_pair(sb + kBK * 128, mb, fb, bcol + 64, kb * kBK, c.mat);
                        if (++stage == ST) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                }
                for (; kb < B.kblocks; ++kb) {
                    if (!ptx::wait_parity_cluster(ptx::smem_addr(&empty[stage]), phase ^ 1u, abort,
                                                  wait_limit)) {
                        record_failure(abort);
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = ptx::smem_addr(&full[stage]);
                    const uint32_t fb = ptx::mapa_shared(fb_local, lead);   // this pair's leader's barrier
                    if (leader) {
                        ptx::mbar_arrive_expect_tx(fb_local, 2 * kStageBytes);
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if constexpr (CS == 2) {
                        ptx::tma_load_3d_pair(ptx::smem_addr(sA + stage * kStageA), &B.tmA, fb, kb * kstep, arow,
                                              c.mat);
                    } else if ((kb & 1) == pp) {
                        // the A rows of this K block for this CTA and its counterpart in the
                        // other pair (same rank in its pair): the pairs take turns by K block
                        const uint16_t mask = static_cast<uint16_t>((1u << rank) | (1u << (2u + rank)));
                        ptx::tma_load_3d_pair_mc(ptx::smem_addr(sA + stage * kStageA), &B.tmA, fb, kb * kBK, arow,
                                                 c.mat, mask);
                    }
                    const uint32_t sb = ptx::smem_addr(sB + stage * kStageB);
                    if (upd) {
                        // two 64-column MN-major blocks of X rows [64 kb, +64)
                        ptx::tma_load_3d_pair(sb, &B.tmB, fb, bcol, kb * kBK, c.mat);
                        ptx::tma_load_3d_pair(sb + kBK * 128, &B.tmB, fb, bcol + 64, kb * kBK, c.mat);
                    } else {
                        ptx::tma_load_3d_pair(sb, &B.tmB, fb, kb * kstep, bcol, c.mat);
                    }
                    if (++stage == ST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (leader && (!ok || *abort)) {
                for (int s = 0; s < ST; ++s)
                    if ((armed >> s) & 1u)
                        ptx::wait_parity_cluster(ptx::smem_addr(&full[s]), (armed_parity >> s) & 1u, nullptr,
                                                 kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA --
        // p.stall (test hook): issue nothing, so that the other warps' bounded waits
        // expire and the launch reports MUON_ERR_TIMEOUT
        if (leader && lane == 0 && !p.stall) {
            // The issue loop is on the critical path (one thread feeds the tensor pipe):
            // everything that does not change per MMA is computed here.  Descriptors of
            // later stages and K steps differ from stage 0 / step 0 only in their start
            // address field (address >> 4, 14 bits; shared memory stays below 2^18 bytes).
            const bool upd = p.mode == kUpdate;
            const uint32_t idesc = F8 ? ptx::idesc_e4m3_f32(kTile, kTile, false, false)
                                      : ptx::idesc_bf16_f32(kTile, kTile, false, upd);
            const uint64_t ad0 = ptx::sdesc_sw128(ptx::smem_addr(sA), 16, 1024);
            const uint64_t bd0 = upd ? ptx::sdesc_sw128(ptx::smem_addr(sB), kBK * 128, 1024)
                                     : ptx::sdesc_sw128(ptx::smem_addr(sB), 16, 1024);
            constexpr uint64_t a_k = 32 >> 4;                  // next 32 bytes of K in a 128-byte row
            const uint64_t b_k = upd ? (2048 >> 4) : (32 >> 4);   // MN-major B: next 16 rows of K
            // upper-only symmetric operands: the K blocks left of the row tile's diagonal
            // come as MN-major 64 x 64 blocks of the stored transpose (8 KB between the
            // two 64-row halves, 1 KB between groups of 8 K rows); B is MN-major there
            // (the polynomial's B from the transpose, the update's iterate always).  They run
            // in a loop of their own ahead of the main loop, whose body stays as for full
            // storage (no per-K-block choice there)
            const bool sym_a = CS == 2 && p.upper_only && p.mode != kGram;
            const bool sym_b = CS == 2 && p.upper_only && p.mode == kPoly;
            const uint64_t ad_mn = ptx::sdesc_sw128(ptx::smem_addr(sA), kBK * 128, 1024);
            const uint64_t bd_mn = ptx::sdesc_sw128(ptx::smem_addr(sB), kBK * 128, 1024);
            constexpr uint32_t idesc_tt = ptx::idesc_bf16_f32(kTile, kTile, true, true);
            constexpr uint32_t idesc_kt = ptx::idesc_bf16_f32(kTile, kTile, false, true);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            // stage release reaches every CTA whose producer may refill the stage
            const uint16_t empty_mask = CS == 4 ? 0xFu : 0x3u;
            const uint16_t acc_mask = static_cast<uint16_t>(0x3u << lead);
            for (int t = pair; ok && t < nitems; t += npairs, ++it) {
                const TileCoord c = decode_item<CS>(p, t, pp).c;
                const GemmBucket& B = p.b[c.bucket];
                const int acc = it & 1;
                const uint32_t aphase = static_cast<uint32_t>(it >> 1) & 1u;
                if (!ptx::wait_parity_cluster(ptx::smem_addr(&tempty[acc]), aphase ^ 1u, abort,
                                              wait_limit)) {
                    record_failure(abort);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kTile);
                int kb = 0;
                if constexpr (!F8) {
                    const int a_lim = sym_a ? c.tm * (kTile / kBK) : 0;
                    const int t_end = sym_b ? c.tn * (kTile / kBK) : a_lim;   // end of the transposed blocks
                    for (; kb < t_end; ++kb) {
                        if (!ptx::wait_parity_cluster(ptx::smem_addr(&full[stage]), phase, abort,
                                                      wait_limit)) {
                            record_failure(abort);
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const bool at = kb < a_lim;
                        const uint64_t ad = (at ? ad_mn : ad0) + static_cast<uint64_t>(stage) * (kStageA >> 4);
                        const uint64_t ak = at ? (2048 >> 4) : (32 >> 4);
                        const uint64_t bd = bd_mn + static_cast<uint64_t>(stage) * (kStageB >> 4);
                        const uint32_t id = at ? idesc_tt : idesc_kt;
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            ptx::mma_bf16_pair(d, ad + kk * ak, bd + kk * (2048 >> 4), id,
                                               (kk != 0 || kb != 0) ? 1u : 0u);
                        ptx::mma_commit_pair(ptx::smem_addr(&empty[stage]), empty_mask);
                        if (++stage == ST) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                }
                for (; kb < B.kblocks; ++kb) {
                    if (!ptx::wait_parity_cluster(ptx::smem_addr(&full[stage]), phase, abort,
                                                  wait_limit)) {
                        record_failure(abort);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t ad = ad0 + static_cast<uint64_t>(stage) * (kStageA >> 4);
                    const uint64_t bd = bd0 + static_cast<uint64_t>(stage) * (kStageB >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint32_t accum = (kk != 0 || kb != 0) ? 1u : 0u;
                        if constexpr (F8)
                            ptx::mma_f8_pair(d, ad + kk * a_k, bd + kk * b_k, idesc, accum);
                        else
                            ptx::mma_bf16_pair(d, ad + kk * a_k, bd + kk * b_k, idesc, accum);
                    }
                    ptx::mma_commit_pair(ptx::smem_addr(&empty[stage]), empty_mask);
                    if (++stage == ST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit_pair(ptx::smem_addr(&tfull[acc]), acc_mask);
            }
        }
    } else {
        // ------------------------------------------------------ epilogue --
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        constexpr int kChunksPerWarp = Epi<EW>::chunks;
        const int ch0 = ((warp - 2) >> 2) * kChunksPerWarp;   // first 32-column chunk of this warp
        const uint32_t tempty_leader0 = ptx::mapa_shared(ptx::smem_addr(&tempty[0]), lead);
        const uint32_t tempty_leader1 = ptx::mapa_shared(ptx::smem_addr(&tempty[1]), lead);
        uint32_t te_phase = 0;      // TMA epilogue: phase bit of each input buffer's barrier
        uint32_t te_pending = 0;    // TMA epilogue: input buffers with a load in flight
        int te_stores = 0;          // TMA epilogue: output blocks stored so far (staging parity)
        int it = 0;
        for (int t = pair; t < nitems; t += npairs, ++it) {
            const ItemCoord ic = decode_item<CS>(p, t, pp);
            const TileCoord c = ic.c;
            const GemmBucket& B = p.b[c.bucket];
            const int acc = it & 1;
            const uint32_t aphase = static_cast<uint32_t>(it >> 1) & 1u;
            const int row = c.tm * kTile + static_cast<int>(rank) * kHalf + q * 32 + lane;
            const size_t mat_off = static_cast<size_t>(c.mat) * static_cast<size_t>(B.mat_stride);
            __nv_bfloat16* out = B.out + mat_off;
            const size_t ld = static_cast<size_t>(B.ld);
            if (!ic.valid) {
                // a tile beyond the matrix (odd tile columns, clusters of two pairs):
                // only release its accumulator
                if (!ptx::wait_parity_cluster_backoff(ptx::smem_addr(&tfull[acc]), aphase, abort, wait_limit, 256)) {
                    record_failure(abort);
                    break;
                }
                ptx::tc_fence_after();
            } else if constexpr (FK != kFinNone) {
                // ---- fused final update: X arrives by TMA as in the plain update; W
                // streams through a register ring in the exchanged layout
                constexpr int D = FinTraits<FK>::depth;
                const FinalMat& f = fin.m[B.fin0 + c.mat];
                const int fr = min(f.rows, f.cols), fk = max(f.rows, f.cols);
                const int rowbase = row - lane;
                const int colb = c.tn * kTile;
                uint8_t* const xch = te_buf + kTeDepth * kTeBlock;   // this warp's exchange block
                auto issue_x = [&](int u) {
                    const int b = u % kTeDepth;
                    const uint32_t bar = ptx::smem_addr(&te_bar[b]);
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive_expect_tx(bar, kTeBlock);
                    ptx::tma_load_3d(ptx::smem_addr(te_buf + b * kTeBlock), &B.tmE, bar, colb + 32 * (ch0 + u), rowbase,
                                     c.mat);
                };
                // W is not in L2: bring this tile's lines (first tile) and the next tile's in
                if (it == 0) fin_prefetch_w<FK>(f, row, rowbase, lane, colb + 32 * ch0, 32 * kChunksPerWarp, fr, fk);
                const ItemCoord n2 = t + npairs < nitems ? decode_item<CS>(p, t + npairs, pp) : ItemCoord{};
                if (t + npairs < nitems && n2.valid) {
                    const TileCoord c2 = n2.c;
                    const FinalMat& f2 = fin.m[p.b[c2.bucket].fin0 + c2.mat];
                    const int row2 = c2.tm * kTile + static_cast<int>(rank) * kHalf + q * 32 + lane;
                    fin_prefetch_w<FK>(f2, row2, row2 - lane, lane, c2.tn * kTile + 32 * ch0, 32 * kChunksPerWarp,
                                       min(f2.rows, f2.cols), max(f2.rows, f2.cols));
                }
                // the first blocks do not depend on this tile's products: request them now
                constexpr int XD = kTeDepth < kChunksPerWarp ? kTeDepth : kChunksPerWarp;
                if (lane == 0)
                    for (int u = 0; u < XD; ++u) issue_x(u);
                te_pending |= (1u << XD) - 1u;
                FinChunk<FK> buf[D];
#pragma unroll
                for (int u = 0; u < D; ++u) fin_issue<FK>(f, fin_seg(f, rowbase, lane, colb + 32 * (ch0 + u)), buf[u]);
                if (!ptx::wait_parity_cluster_backoff(ptx::smem_addr(&tfull[acc]), aphase, abort, wait_limit, 256)) {
                    record_failure(abort);
                    break;
                }
                ptx::tc_fence_after();
                bool ok = true;
                const int sw = (lane >> 1) & 3;
#pragma unroll
                for (int u = 0; u < kChunksPerWarp; ++u) {
                    const int ch = ch0 + u;
                    const int bx = u % kTeDepth;
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(
                        tmem_base + static_cast<uint32_t>(acc * kTile + ch * 32) + (static_cast<uint32_t>(q * 32) << 16), r);
                    ptx::tmem_wait_ld();
                    if (!ptx::wait_parity(ptx::smem_addr(&te_bar[bx]), (te_phase >> bx) & 1u, abort, wait_limit)) {
                        ok = false;
                        break;
                    }
                    te_phase ^= 1u << bx;
                    te_pending &= ~(1u << bx);
                    uint4 xv[4];
                    const uint8_t* xr = te_buf + bx * kTeBlock + lane * 64;
#pragma unroll
                    for (int k = 0; k < 4; ++k) xv[k] = *reinterpret_cast<const uint4*>(xr + ((k ^ sw) << 4));
                    __syncwarp();   // every lane has read X block bx
                    if (u + kTeDepth < kChunksPerWarp) {
                        if (lane == 0) issue_x(u + kTeDepth);
                        te_pending |= 1u << bx;
                    }
                    float o[32];
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float e[8];
                        unpack8(xv[g], e);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            o[8 * g + j] = __bfloat162float(__float2bfloat16_rn(
                                __fadd_rn(__fmul_rn(p.a, e[j]), __uint_as_float(r[8 * g + j]))));
                    }
                    uint4 ob[4];
                    fin_exchange(f.trans != 0, o, xch, lane, ob);   // f.trans is uniform across the warp
                    FinChunk<FK>& b = buf[u % D];
                    fin_store<FK>(f, fin_seg(f, rowbase, lane, colb + 32 * ch), ob, b);
                    if (u + D < kChunksPerWarp) fin_issue<FK>(f, fin_seg(f, rowbase, lane, colb + 32 * (ch + D)), b);
                }
                if (!ok) {
                    record_failure(abort);
                    break;
                }
            } else if constexpr (TE) {
                // ---- update, TMA epilogue: X' = bf16(a X + acc) in 32 x 32 blocks
                const int rowbase = row - lane;
                const int colb = c.tn * kTile;
                auto issue_x = [&](int u) {
                    const int b = u % kTeDepth;
                    const uint32_t bar = ptx::smem_addr(&te_bar[b]);
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive_expect_tx(bar, kTeBlock);
                    ptx::tma_load_3d(ptx::smem_addr(te_buf + b * kTeBlock), &B.tmE, bar, colb + 32 * (ch0 + u), rowbase,
                                     c.mat);
                };
                // the iterate's blocks do not depend on this tile's products: request them now
                if (lane == 0)
                    for (int u = 0; u < kTeDepth && u < kChunksPerWarp; ++u) issue_x(u);
                te_pending |= (1u << kTeDepth) - 1u;
                if (!ptx::wait_parity_cluster_backoff(ptx::smem_addr(&tfull[acc]), aphase, abort, wait_limit, 256)) {
                    record_failure(abort);
                    break;
                }
                ptx::tc_fence_after();
                bool ok = true;
                const bool q8 = p.fp8_next != 0;   // also the next FP8 Gram's E4M3 operand
#pragma unroll
                for (int u = 0; u < kChunksPerWarp; ++u) {
                    const int ch = ch0 + u;
                    const int b = u % kTeDepth;
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(
                        tmem_base + static_cast<uint32_t>(acc * kTile + ch * 32) + (static_cast<uint32_t>(q * 32) << 16), r);
                    ptx::tmem_wait_ld();
                    if (!ptx::wait_parity(ptx::smem_addr(&te_bar[b]), (te_phase >> b) & 1u, abort, wait_limit)) {
                        ok = false;
                        break;
                    }
                    te_phase ^= 1u << b;
                    te_pending &= ~(1u << b);
                    // this lane's row of the block, 16-byte unit k stored at unit k ^ ((row / 2) % 4)
                    const uint8_t* xrow = te_buf + b * kTeBlock + lane * 64;
                    const int sw = (lane >> 1) & 3;
                    uint4 xv[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) xv[k] = *reinterpret_cast<const uint4*>(xrow + ((k ^ sw) << 4));
                    __syncwarp();   // every lane has read buffer b
                    if (u + kTeDepth < kChunksPerWarp) {
                        if (lane == 0) issue_x(u + kTeDepth);
                        te_pending |= 1u << b;
                    }
                    float v[32];
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float e[8];
                        unpack8(xv[g], e);
#pragma unroll
                        for (int j = 0; j < 8; ++j) v[8 * g + j] = __fadd_rn(__fmul_rn(p.a, e[j]), __uint_as_float(r[8 * g + j]));
                    }
                    // staging buffers of this block (bf16, and E4M3 before an FP8 Gram): the
                    // stores issued two blocks ago must have read them
                    uint8_t* stg = te_buf + (kTeDepth + (te_stores & 1)) * kTeBlock;
                    uint8_t* stg8 = te_buf + (kTeDepth + 2) * kTeBlock + (te_stores & 1) * kTe8Block;
                    if (te_stores >= 2 && lane == 0) ptx::bulk_wait_group_read<1>();
                    __syncwarp();
                    uint8_t* srow = stg + lane * 64;
                    uint2 q[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 xb = pack8(&v[8 * k]);
                        *reinterpret_cast<uint4*>(srow + ((k ^ sw) << 4)) = xb;
                        if (q8) q[k] = ptx::e4m3x8_from_bf16x8(xb, static_cast<float>(1 << kFp8ScaleExp));
                    }
                    if (q8) {
                        // this lane's row of the E4M3 block: 32 bytes, rows one after the other
                        uint4* q8row = reinterpret_cast<uint4*>(stg8 + lane * 32);
                        q8row[0] = make_uint4(q[0].x, q[0].y, q[1].x, q[1].y);
                        q8row[1] = make_uint4(q[2].x, q[2].y, q[3].x, q[3].y);
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_3d(&B.tmO, ptx::smem_addr(stg), colb + 32 * ch, rowbase, c.mat);
                        if (q8) ptx::tma_store_3d(&B.tmQ, ptx::smem_addr(stg8), colb + 32 * ch, rowbase, c.mat);
                        ptx::bulk_commit_group();
                    }
                    ++te_stores;
                }
                if (!ok) {
                    record_failure(abort);
                    break;
                }
            } else {
            // the epilogue operand does not depend on this tile's products: load it now
            uint4 pre[kChunksPerWarp * 4];
            if (p.mode != kGram) {
                const uint4* src =
                    reinterpret_cast<const uint4*>(B.epi + mat_off + row * ld + c.tn * kTile + ch0 * 32);
#pragma unroll
                for (int g = 0; g < kChunksPerWarp * 4; ++g) pre[g] = __ldg(src + g);
            }
            if (!ptx::wait_parity_cluster_backoff(ptx::smem_addr(&tfull[acc]), aphase, abort, wait_limit, 256)) {
                record_failure(abort);
                break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int u = 0; u < kChunksPerWarp; ++u) {
                const int ch = ch0 + u;
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(
                    tmem_base + static_cast<uint32_t>(acc * kTile + ch * 32) +
                        (static_cast<uint32_t>(q * 32) << 16),
                    r);
                ptx::tmem_wait_ld();
                const int col0 = c.tn * kTile + ch * 32;
                float v[32];
                if (p.mode == kGram) {
                    // FP8 operands were scaled by 2^8: the sums carry 2^16 (an exact unscaling)
                    constexpr float unscale = F8 ? 1.0f / static_cast<float>(1 << (2 * kFp8ScaleExp)) : 1.0f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(__uint_as_float(r[j]), unscale);
                } else {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float e[8];
                        unpack8(pre[u * 4 + g], e);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float s = __uint_as_float(r[8 * g + j]);
                            v[8 * g + j] = (p.mode == kPoly)
                                               ? __fadd_rn(__fmul_rn(p.bcoef, e[j]), __fmul_rn(p.c, s))
                                               : __fadd_rn(__fmul_rn(p.a, e[j]), s);
                        }
                    }
                }
                if constexpr (XS) {
                    const int rowbase = row - lane;
                    if (c.tm < c.tn || col0 >= rowbase) {
                        // the warp's 32 x 32 block lies above the diagonal (or on it, col0 ==
                        // rowbase): store it and its mirror through the exchange block; on
                        // the diagonal block only the upper part goes in place and only the
                        // strict upper part is mirrored
                        const bool diag = c.tm == c.tn && col0 == rowbase;
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) v[jj] = __bfloat162float(__float2bfloat16_rn(v[jj]));
                        uint4 ob[4];
                        const int c8 = (lane & 3) * 8;
                        fin_exchange(false, v, xchg, lane, ob);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int rr = (lane >> 2) + 8 * i;   // row in the block; columns c8 .. c8 + 7
                            __nv_bfloat16* dst = out + static_cast<size_t>(rowbase + rr) * ld + col0 + c8;
                            if (!diag || c8 >= rr) {
                                *reinterpret_cast<uint4*>(dst) = ob[i];
                            } else if (c8 + 7 >= rr) {
                                const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&ob[i]);
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    if (c8 + e >= rr) dst[e] = h[e];
                            }
                        }
                        // upper-only storage: only the diagonal tiles hold their lower part
                        if (!p.upper_only || c.tm == c.tn) {
                            fin_exchange(true, v, xchg, lane, ob);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                // stored row col0 + rr, columns rowbase + c8 ..: the mirror of block
                                // element (c8 + e, rr), strictly upper when rr > c8 + e
                                const int rr = (lane >> 2) + 8 * i;
                                __nv_bfloat16* dst = out + static_cast<size_t>(col0 + rr) * ld + rowbase + c8;
                                if (!diag || rr > c8 + 7) {
                                    *reinterpret_cast<uint4*>(dst) = ob[i];
                                } else if (rr > c8) {
                                    const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&ob[i]);
#pragma unroll
                                    for (int e = 0; e < 8; ++e)
                                        if (rr > c8 + e) dst[e] = h[e];
                                }
                            }
                        }
                    }
                    // blocks below the diagonal are written as the mirror of their transposes
                    continue;
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
                // the mirror (upper-only storage: in the diagonal tiles only)
                if (p.mode != kUpdate && (!p.upper_only || c.tm == c.tn) && col0 + 31 > row) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j > row)
                            out[static_cast<size_t>(col0 + j) * ld + row] = __float2bfloat16_rn(v[j]);
                }
            }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
        }
        if constexpr (TE || FK != kFinNone) {
            if (lane == 0) {
                // loads still in flight after a failure land before the CTA exits
                for (int b = 0; b < kTeDepth; ++b)
                    if ((te_pending >> b) & 1u)
                        ptx::wait_parity(ptx::smem_addr(&te_bar[b]), (te_phase >> b) & 1u, nullptr, kDrainLimitNs);
                ptx::bulk_wait_group_all();   // every output block written
            }
            __syncwarp();
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

static_assert((2 * kPairStages + 4) * sizeof(uint64_t) + 8 <= kBarBytes, "barrier block too small");
static_assert(sizeof(GemmParams) + sizeof(FinalParams) <= 32764, "kernel parameters above the launch limit");
// (with the TMA epilogue or the fused final update the barrier block spans the 1024 bytes before the buffers)
static_assert((kTeBarIndex + kEpiWarps * kTeDepth) * 8 <= 1024, "final-update barriers do not fit");
static_assert(1024 + (kPairStages - 1) * kStageBytes + 1024 + kEpiWarps * kFinWarpBytes <= 232448,
              "final update's shared memory");

static_assert(kTeBarIndex * 8 >= (2 * kPairStages + 4) * 8 + 8 &&
                  (kTeBarIndex + kUpdateEpiWarps * kTeDepth) * 8 <= kBarBytes,
              "TMA-epilogue barriers overlap the barrier block's other contents");

// pipeline ring, barriers and (XCHG) one exchange block per epilogue warp or
// (TE) the TMA epilogue's buffers, 1024 bytes after the barrier block
template <int EW, bool XCHG, int ST, bool TE = false, int FK = kFinNone>
size_t pair_smem_bytes() {
    if (TE) return 1024 + ST * kStageBytes + 1024 + EW * kTeWarpBytes;
    if (FK != kFinNone) return 1024 + ST * kStageBytes + 1024 + EW * kFinWarpBytes;
    return 1024 + ST * kStageBytes + kBarBytes + (XCHG ? Epi<EW>::xchg_bytes() : 0);
}

size_t gemm_pair_smem_bytes() { return pair_smem_bytes<kEpiWarps, false, kPairStages>(); }

namespace {

// Clusters of CS CTAs that can be resident at once for this instantiation
// (0 if none), queried once per device.
template <int FK, int EW, bool XS, int ST, int CS, bool TE, class FP>
int max_clusters(size_t smem) {
    static int cached[64];
    static bool have[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!have[dev]) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(CS, 1, 1);
        cfg.blockDim = dim3(Epi<EW>::threads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CS;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, ns_gemm_pair_kernel<FK, EW, XS, ST, CS, TE, false, FP>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cached[dev] = n;
        have[dev] = true;
    }
    return cached[dev];
}

template <int FK, int EW, bool XS, int ST, int CS, bool TE, class FP, bool F8 = false>
cudaError_t launch_pair(const GemmParams& p, const FP& f, int nclusters, cudaStream_t s) {
    const size_t smem = pair_smem_bytes<EW, XS, ST, TE, FK>();
    cudaError_t e = cudaFuncSetAttribute(ns_gemm_pair_kernel<FK, EW, XS, ST, CS, TE, F8, FP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CS * nclusters, 1, 1);
    cfg.blockDim = dim3(Epi<EW>::threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, ns_gemm_pair_kernel<FK, EW, XS, ST, CS, TE, F8, FP>, p, f);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// The update product (plain or fused final): on clusters of two pairs sharing
// A by multicast when asked for and when such clusters fit, else on pairs.
template <int FK, int EW, int ST, bool TE, class FP>
cudaError_t launch_update(const GemmParams& p, const FP& f, int sms, bool multicast, cudaStream_t s) {
    // (the multicast loads read K-major blocks only: not with upper-only storage)
    if (multicast && p.total_items > 0 && !p.upper_only) {
        const size_t smem = pair_smem_bytes<EW, false, ST, TE, FK>();
        if (cudaFuncSetAttribute(ns_gemm_pair_kernel<FK, EW, false, ST, 4, TE, false, FP>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) == cudaSuccess) {
            const int n4 = std::min(std::min(max_clusters<FK, EW, false, ST, 4, TE, FP>(smem), sms / 4), p.total_items);
            if (n4 > 0) return launch_pair<FK, EW, false, ST, 4, TE, FP>(p, f, n4, s);
        } else {
            cudaGetLastError();
        }
    }
    return launch_pair<FK, EW, false, ST, 2, TE, FP>(p, f, std::min(p.total_tiles, sms / 2), s);
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmParams& p, int sms, bool multicast, bool tma_epilogue, cudaStream_t s) {
    // the symmetric products (Gram and polynomial) store through the exchange
    // blocks and give up one pipeline stage for them; the update (K = r) runs 5
    // stages too: the shared memory they leave lets more of the other
    // half-batch's elementwise CTAs run beside them
    const int npairs = std::min(p.total_tiles, sms / 2);
    if (p.mode == kUpdate) {
        if (tma_epilogue)
            return launch_update<kFinNone, kUpdateEpiWarps, kPairStages - 1, true>(p, NoFinal{0}, sms, multicast, s);
        return launch_update<kFinNone, kUpdateEpiWarps, kPairStages - 1, false>(p, NoFinal{0}, sms, multicast, s);
    }
    if (p.mode == kPoly || (p.mode == kGram && !p.fp8))
        return launch_pair<kFinNone, kEpiWarps, true, kPairStages - 1, 2, false>(p, NoFinal{0}, npairs, s);
    if (p.fp8) return launch_pair<kFinNone, kEpiWarps, false, kPairStages, 2, false, NoFinal, true>(p, NoFinal{0}, npairs, s);
    return launch_pair<kFinNone, kEpiWarps, false, kPairStages, 2, false>(p, NoFinal{0}, npairs, s);
}

cudaError_t launch_gemm_pair_final(const GemmParams& p, const FinalParams& f, int kind, int sms, bool multicast,
                                   cudaStream_t s) {
    if (p.mode != kUpdate) return cudaErrorInvalidValue;
    switch (kind) {
        case kFinStore: return launch_update<kFinStore, kEpiWarps, kPairStages - 1, false>(p, f, sms, multicast, s);
        case kFinWBf16: return launch_update<kFinWBf16, kEpiWarps, kPairStages - 1, false>(p, f, sms, multicast, s);
        case kFinWF32: return launch_update<kFinWF32, kEpiWarps, kPairStages - 1, false>(p, f, sms, multicast, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace muon
