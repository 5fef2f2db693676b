// Block-FP8 (W8A8) variant of the logprob path.
//
// The deployment recipe the vLLM blog describes for DeepSeek-V4 keeps the lm_head GEMM in
// block FP8 on both sides: the trainer quantises its master bf16 weights by the deployment
// rule on every forward and calls the inference GEMM, whose accumulation order does not depend
// on M ("Finish RL training faster", section 4.1).  The rule here is the DeepSeek block rule:
//   activations  1 x 128 blocks (one per token per 128 hidden columns),
//   weights      128 x 128 blocks,
//   scale s = amax / 448 (IEEE fp32 division; 1 for an all-zero block),
//   q = e4m3(x / s), round to nearest even, saturating to +-448.
// The GEMM keeps the K leaves and the fixed leaf tree:
//   B_kb[t,v] = sum_{k in block kb} qx[t,k] qw[v,k]           tcgen05.mma kind::f8f6f4, fp32
//   P_j       = sum_{kb in leaf j, ascending} (sx[t,kb] sw[v/128,kb]) B_kb
//               (first term a product, then one fma per block; computed as one fma per
//               block from -0, which gives the product's bits for the first term)
//   z         = fixed pairwise tree over P_0..P_{N-1}
// and the same 64-column tile log-sum-exp and vocabulary combine as the bf16 path.
//
//  quant_x_kernel        bf16 rows -> e4m3 rows + per-(row, block) scales
//  quant_w_kernel        bf16 lm_head -> e4m3 + per-(128 x 128 block) scales
//  leaf_gemm_fp8_kernel  persistent, warp-specialised: TMA producer warp, two MMA warps (one
//                        128-K block per TMEM buffer, two buffers: one warp issues the even
//                        blocks into buffer 0, the other the odd blocks into buffer 1), 8
//                        epilogue warps that apply the block scales, fold the leaves through
//                        the tree (TMEM slots L and S0, a shared-memory slot S1 for N = 8) and
//                        form the tile partials.
#pragma once

#include <cuda_fp8.h>

#include "kernels.cuh"

namespace lp {

constexpr int kQBlock = 128;              // quantisation block along K (and along V for W)
constexpr int kF8Stages = 5;              // 128-K pipeline stages: X 16 KB + W 16 KB each
constexpr int kF8Bufs = 2;                // TMEM block accumulators
constexpr uint32_t kF8ColL = 256;         // TMEM slot: the even leaf waiting for its pair
constexpr uint32_t kF8ColS0 = 384;        // TMEM slot: the first stack level of the tree
constexpr int kF8S1Bytes = kBM * kVT * 4; // shared-memory slot: the second stack level (N = 8)
// tcgen05 instruction descriptor, kind::f8f6f4: fp32 D (bits 4-5 = 1), A and B E4M3 (format
// code 0 in bits 7-9 and 10-12), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t kIdescF8 = (1u << 4) | ((static_cast<uint32_t>(kVT) >> 3) << 17) |
                              ((static_cast<uint32_t>(kBM) >> 4) << 24);

// Warp 0 copies, warps 1 and 2 issue the MMAs (block g by warp 1 + g % 2), warps 3-10 are the
// epilogue.  A block is only 256 tensor cycles; with one issuing warp its waits and commits
// left the tensor pipe idle between blocks, while two warps cover each other's gaps.
constexpr int kF8MmaWarps = 2;
constexpr int kF8FirstEpiWarp = 1 + kF8MmaWarps;
constexpr int kF8Threads = 32 * (kF8FirstEpiWarp + kEpiWarps);
static_assert(kF8Bufs == kF8MmaWarps, "each MMA warp owns one TMEM block buffer");
// A stage is used by both MMA warps in turn (5 stages, 2 warps).  A warp waits on the stage of
// block g only after its buffer's previous block g - 2 was released, and the epilogue releases
// blocks in order, so block g - 5 (the stage's previous use) has been issued and its phase has
// completed: the parity wait cannot match a stale phase.  Five stages keep 80 KB of W in flight
// per SM, which a weight stream (decode) needs; 230.5 KB of shared memory in all.
static_assert(kF8Stages >= kF8MmaWarps,
              "a stage's previous use must not follow the buffer's previous block");

__host__ __device__ constexpr int kF8NumBars() { return 2 * kF8Stages + 2 * kF8Bufs + kF8MmaWarps; }
__host__ __device__ constexpr int fp8_smem_bytes() {
    return 1024 + kF8Stages * 2 * kTileBytes + kF8S1Bytes + kF8NumBars() * 8 + 16;
}

// One 128-K block from a single elected lane: 4 MMAs of K = 32 (+32 bytes each), the first
// starting a fresh accumulator, then the commits that free the stage and hand the block's
// TMEM buffer to the epilogue.
__device__ __forceinline__ void umma_f8_block_elect(uint32_t d_tmem, uint64_t a, uint64_t b,
                                                    uint32_t idesc, uint64_t* stage_bar,
                                                    uint64_t* acc_bar) {
    asm volatile(
        "{\n\t.reg .pred e, f, t;\n\t.reg .b64 a1, b1;\n\t"
        "elect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 f, 0, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, f;\n\t"
        "add.s64 a1, %1, 2;\n\tadd.s64 b1, %2, 2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a1, b1, %3, t;\n\t"
        "add.s64 a1, %1, 4;\n\tadd.s64 b1, %2, 4;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a1, b1, %3, t;\n\t"
        "add.s64 a1, %1, 6;\n\tadd.s64 b1, %2, 6;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a1, b1, %3, t;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t}" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(smem_u32(stage_bar)), "r"(smem_u32(acc_bar))
        : "memory");
}

__device__ __forceinline__ float block_scale(float amax) {
    return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

__device__ __forceinline__ uint32_t e4m3(float v) {
    return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// One warp per (row, 128-column block); each lane converts 4 consecutive columns.
// grid: ceil(T * H/128 / 8), block 256.
static __global__ void __launch_bounds__(256) quant_x_kernel(const uint16_t* X, int64_t ldx,
                                                            int64_t T, int H, uint8_t* xq,
                                                            int64_t ldq, float* sx) {
    const int nkb = H / kQBlock;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (gw >= T * nkb) return;
    const int lane = threadIdx.x & 31;
    const int64_t t = gw / nkb;
    const int kb = static_cast<int>(gw - t * nkb);
    const uint2 raw = *reinterpret_cast<const uint2*>(X + t * ldx + kb * kQBlock + lane * 4);
    float v[4];
    v[0] = __uint_as_float(raw.x << 16);
    v[1] = __uint_as_float(raw.x & 0xffff0000u);
    v[2] = __uint_as_float(raw.y << 16);
    v[3] = __uint_as_float(raw.y & 0xffff0000u);
    float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    const float s = block_scale(a);
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) packed |= e4m3(__fdiv_rn(v[i], s)) << (8 * i);
    *reinterpret_cast<uint32_t*>(xq + t * ldq + kb * kQBlock + lane * 4) = packed;
    if (lane == 0) sx[t * nkb + kb] = s;
}

// One block of 256 threads per 128 x 128 weight block (rows past V excluded).
// grid: (H/128, ceil(V/128)).
static __global__ void __launch_bounds__(256) quant_w_kernel(const uint16_t* W, int V, int H,
                                                            uint8_t* wq, float* sw) {
    __shared__ float red[8];
    const int kb = blockIdx.x, vb = blockIdx.y;
    const int nkb = H / kQBlock;
    const int r0 = vb * kQBlock;
    const int rows = min(kQBlock, V - r0);
    // thread i covers 4 consecutive columns (i % 32) of rows i/32, i/32 + 8, ...
    const int c4 = (threadIdx.x & 31) * 4;
    float a = 0.0f;
    for (int r = threadIdx.x >> 5; r < rows; r += 8) {
        const uint2 raw = *reinterpret_cast<const uint2*>(
            W + static_cast<int64_t>(r0 + r) * H + kb * kQBlock + c4);
        a = fmaxf(a, fmaxf(fmaxf(fabsf(__uint_as_float(raw.x << 16)),
                                 fabsf(__uint_as_float(raw.x & 0xffff0000u))),
                           fmaxf(fabsf(__uint_as_float(raw.y << 16)),
                                 fabsf(__uint_as_float(raw.y & 0xffff0000u)))));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    a = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w]);
    const float s = block_scale(a);
    for (int r = threadIdx.x >> 5; r < rows; r += 8) {
        const int64_t off = static_cast<int64_t>(r0 + r) * H + kb * kQBlock + c4;
        const uint2 raw = *reinterpret_cast<const uint2*>(W + off);
        const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                            __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u)};
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) packed |= e4m3(__fdiv_rn(v[i], s)) << (8 * i);
        *reinterpret_cast<uint32_t*>(wq + off) = packed;
    }
    if (threadIdx.x == 0) sw[static_cast<int64_t>(vb) * nkb + kb] = s;
}

// The block-scaled leaf GEMM over the leaves [p.leaf_begin, p.leaf_begin + p.leaf_count),
// finished as in leaf_gemm_kernel: kModeLse (tile log-sum-exp partials and the sampled logit),
// kModeLseEnt (also the entropy partial) or kModeNode (the tree node z written to p.out).
// p.leaf_len is in elements (a multiple of 128); p.sx [T][nkb], p.sw [num_vocab_tiles][nkb].
template <int kMode>
__global__ void __launch_bounds__(kF8Threads, 1)
    leaf_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmX,
                         const __grid_constant__ CUtensorMap tmW, const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                                   // X  [kF8Stages][128 x 128] e4m3
    uint8_t* sB = smem + kF8Stages * kTileBytes;          // W  [kF8Stages][128 x 128] e4m3
    float* s1 = reinterpret_cast<float*>(smem + 2 * kF8Stages * kTileBytes);  // [col][row]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kF8Stages * kTileBytes + kF8S1Bytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + kF8Stages;
    uint64_t* acc_full = bars + 2 * kF8Stages;
    uint64_t* acc_empty = acc_full + kF8Bufs;
    uint64_t* drain = acc_empty + kF8Bufs;  // [kF8MmaWarps]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + kF8MmaWarps);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kF8Stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < kF8Bufs; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kEpiWarps);
        }
        for (int m = 0; m < kF8MmaWarps; ++m) mbar_init(&drain[m], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;

    const int num_tiles = p.num_row_tiles * p.num_vocab_tiles;
    const int nkb = p.nkb;                      // 128-K blocks over all of H
    const int bpl = p.leaf_len / kQBlock;       // blocks per leaf
    const int n = p.leaf_count;
    const int kb0 = p.leaf_begin * bpl;         // first block of the leaf range
    const int nkb_range = n * bpl;              // blocks per tile in the leaf range
    constexpr uint32_t kFull = 0xffffffffu;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (warp)
        const uint32_t tx_bytes = static_cast<uint32_t>(p.x_box_rows * kQBlock + kTileBytes);
        uint32_t stage = 0, phase = 0;
        uint64_t issued = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            int rt, vt;
            tile_coords(tile, p.num_row_tiles, p, rt, vt);
            const int row0 = rt * kBM, v0 = vt * kVT;
            for (int kb = kb0; kb < kb0 + nkb_range; ++kb) {
                ok = __all_sync(kFull, mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.timeout_ns));
                if (!ok) {
                    if (lane == 0) raise_timeout(p, abort_flag);
                    break;
                }
                mbar_arrive_expect_tx_elect(&full[stage], tx_bytes);
                tma_load_2d_elect(&tmX, &full[stage], sA + stage * kTileBytes, kb * kQBlock, row0);
                tma_load_2d_elect(&tmW, &full[stage], sB + stage * kTileBytes, kb * kQBlock, v0);
                ++issued;
                // test hook: stop as if this warp's own wait had run out (the consumers'
                // bounded waits then expire and the abort path runs)
                if (p.test_stop_after > 0 && issued >= uint64_t(p.test_stop_after)) {
                    ok = false;
                    break;
                }
                if (++stage == kF8Stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            const uint64_t first = issued > kF8Stages ? issued - kF8Stages : 0;
            for (uint64_t i = first; i < issued; ++i) {
                volatile int never = 0;
                mbar_wait(&full[i % kF8Stages], static_cast<uint32_t>((i / kF8Stages) & 1u), &never,
                          p.timeout_ns);
            }
        }
    } else if (warp < kF8FirstEpiWarp) {
        // ------------------------------------------------------------ MMA issuers (2 warps)
        // Block g of this CTA's sequence (tiles in order, 128-K blocks in order within a tile)
        // is issued by MMA warp g % 2 into TMEM buffer g % 2 from stage g % kF8Stages: 4 MMAs
        // of K = 32 (32 bytes of each 128-byte row), a fresh accumulator at the block's first
        // MMA, then the commits that free the stage and hand the buffer to the epilogue.  The
        // epilogue reads the blocks in order, so nothing about a block depends on which warp
        // issued it.
        const uint32_t me = static_cast<uint32_t>(warp - 1);
        const uint64_t descA = sw128_kmajor_desc(smem_u32(sA));
        const uint64_t descB = sw128_kmajor_desc(smem_u32(sB));
        constexpr uint32_t kStageDesc = kTileBytes >> 4;
        const uint32_t d_tmem = tmem_base + me * kVT;
        uint64_t g = 0;     // block index in the CTA's sequence
        uint32_t use = 0;   // blocks this warp has issued (uses of its buffer)
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            for (int kb = 0; ok && kb < nkb_range; ++kb, ++g) {
                if ((g % kF8MmaWarps) != me) continue;
                const uint32_t stage = static_cast<uint32_t>(g % kF8Stages);
                const uint32_t phase = static_cast<uint32_t>((g / kF8Stages) & 1u);
                // the buffer's previous block has been read (a fresh barrier passes at once)
                ok = __all_sync(kFull, mbar_wait(&acc_empty[me], (use & 1u) ^ 1u, abort_flag,
                                                 p.timeout_ns)) &&
                     __all_sync(kFull, mbar_wait(&full[stage], phase, abort_flag, p.timeout_ns));
                if (!ok) {
                    if (lane == 0) raise_timeout(p, abort_flag);
                    break;
                }
                tc_fence_after_sync();
                umma_f8_block_elect(d_tmem, descA + stage * kStageDesc, descB + stage * kStageDesc,
                                    kIdescF8, &empty[stage], &acc_full[me]);
                ++use;
            }
        }
        if (!ok) {
            volatile int never = 0;
            umma_commit_elect(&drain[me]);
            mbar_wait(&drain[me], 0, &never, p.timeout_ns);
        }
    } else {
        // ------------------------------------------------------------ epilogue (8 warps)
        const int q = warp & 3;  // TMEM lane quarter: warp w reaches lanes 32 (w % 4) ..
        const int h = (warp - kF8FirstEpiWarp) >> 2;
        const int r_in_tile = q * 32 + lane;
        const uint32_t lane_base =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * 64);
        float* s1_mine = s1 + (h * 64) * kBM + r_in_tile;   // column c at s1_mine[c * kBM]
        uint32_t g = 0;
        bool ok = true;
        const int npairs = n >> 1;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            int rt, vt;
            tile_coords(tile, p.num_row_tiles, p, rt, vt);
            const int row = rt * kBM + r_in_tile;
            const int v0 = vt * kVT;
            const bool row_ok = row < p.T;
            int ycol = -1;
            if (kMode != kModeNode && row_ok) {
                const int y = p.ids[row];
                if (y >= 0 && y < p.V) ycol = y - v0;
            }
            const float* sxr = p.sx + static_cast<int64_t>(row_ok ? row : 0) * nkb + kb0;
            const float* swr = p.sw + static_cast<int64_t>(vt) * nkb + kb0;
            // The block scales (this row's activation scale and the tile's weight scale) are
            // read kSxAhead blocks before they are used: with ~200 KB of shared memory per SM
            // they do not stay in L1, and a load issued at use would put an L2 round trip into
            // every block.
            constexpr int kSxAhead = 3;
            float sxq[kSxAhead], swq[kSxAhead];
#pragma unroll
            for (int i = 0; i < kSxAhead; ++i) {
                sxq[i] = i < nkb_range ? sxr[i] : 0.0f;
                swq[i] = i < nkb_range ? swr[i] : 0.0f;
            }
            int bi = 0;  // block index within the tile
            float R[64];
            for (int j = 0; ok && j < n; ++j) {
                // leaf j: P_j = sum over its blocks of (sx * sw) * B_kb.  The sum starts at -0:
                // fma(s, B, -0) rounds s * B + (-0) = s * B once, which is exactly the product
                // (a signed zero included), so every block is one fma and the first block gets
                // the bits of a plain product.
#pragma unroll
                for (int k = 0; k < 64; ++k) R[k] = -0.0f;
                for (int b = 0; b < bpl; ++b, ++g, ++bi) {
                    const uint32_t buf = g % kF8Bufs, use = g / kF8Bufs;
                    const float s = __fmul_rn(row_ok ? sxq[0] : 0.0f, swq[0]);
#pragma unroll
                    for (int i = 0; i + 1 < kSxAhead; ++i) {
                        sxq[i] = sxq[i + 1];
                        swq[i] = swq[i + 1];
                    }
                    const bool more = bi + kSxAhead < nkb_range;
                    sxq[kSxAhead - 1] = more ? sxr[bi + kSxAhead] : 0.0f;
                    swq[kSxAhead - 1] = more ? swr[bi + kSxAhead] : 0.0f;
                    if (!warp_wait(&acc_full[buf], use & 1u, p, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    {
                        // the block's 64 columns in one TMEM load (one instruction, one wait)
                        float P[64];
                        tmem_ld64(lane_base + buf * kVT, P);
                        const float* P0 = P;
                        const float* P1 = P + 32;
                        // two lanes per instruction: each lane of __ffma2_rn is one IEEE
                        // binary32 fma, so every element gets exactly the bits of __fmaf_rn
                        const float2 s2 = make_float2(s, s);
#pragma unroll
                        for (int k = 0; k < 32; k += 2) {
                            const float2 t = __ffma2_rn(s2, make_float2(P0[k], P0[k + 1]),
                                                        make_float2(R[k], R[k + 1]));
                            R[k] = t.x;
                            R[k + 1] = t.y;
                        }
#pragma unroll
                        for (int k = 0; k < 32; k += 2) {
                            const float2 t = __ffma2_rn(s2, make_float2(P1[k], P1[k + 1]),
                                                        make_float2(R[32 + k], R[33 + k]));
                            R[32 + k] = t.x;
                            R[33 + k] = t.y;
                        }
                    }
                    release_buf(&acc_empty[buf]);
                }
                if (!ok) break;
                if (n == 1) continue;
                if ((j & 1) == 0) {  // the even leaf waits for its partner
                    tmem_st64(lane_base + kF8ColL, R);
                    continue;
                }
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {  // pair sum P_{j-1} + P_j
                    float Lc[32];
                    tmem_ld32(lane_base + kF8ColL + cc * 32, Lc);
#pragma unroll
                    for (int k = 0; k < 32; ++k) R[cc * 32 + k] = __fadd_rn(Lc[k], R[cc * 32 + k]);
                }
                const int i = j >> 1;  // pair index
                if (npairs == 1) continue;
                if (i == 0 || (npairs == 4 && i == 1)) {
                    if (i == 1) {  // quad q0 = p0 + p1
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            float Sc[32];
                            tmem_ld32(lane_base + kF8ColS0 + cc * 32, Sc);
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                R[cc * 32 + k] = __fadd_rn(Sc[k], R[cc * 32 + k]);
                        }
                    }
                    tmem_st64(lane_base + kF8ColS0, R);  // p0 (N = 4) or q0 (N = 8)
                } else if (npairs == 2) {  // i == 1: root = p0 + p1
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        float Sc[32];
                        tmem_ld32(lane_base + kF8ColS0 + cc * 32, Sc);
#pragma unroll
                        for (int k = 0; k < 32; ++k) R[cc * 32 + k] = __fadd_rn(Sc[k], R[cc * 32 + k]);
                    }
                } else if (i == 2) {  // N = 8: p2 waits in shared memory
#pragma unroll
                    for (int k = 0; k < 64; ++k) s1_mine[k * kBM] = R[k];
                } else {  // N = 8, i == 3: q1 = p2 + p3, root = q0 + q1
#pragma unroll
                    for (int k = 0; k < 64; ++k) R[k] = __fadd_rn(s1_mine[k * kBM], R[k]);
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        float Sc[32];
                        tmem_ld32(lane_base + kF8ColS0 + cc * 32, Sc);
#pragma unroll
                        for (int k = 0; k < 32; ++k) R[cc * 32 + k] = __fadd_rn(Sc[k], R[cc * 32 + k]);
                    }
                }
            }
            if (!ok) break;
            const int col0 = v0 + h * 64;
            const int nv = p.V - col0;
            if constexpr (kMode == kModeNode) {
                if (row_ok && nv > 0) {
                    float* dst = p.out + static_cast<int64_t>(row) * p.ldo + col0;
                    if (nv >= 64) {
#pragma unroll
                        for (int i = 0; i < 64; i += 4)
                            *reinterpret_cast<float4*>(dst + i) =
                                make_float4(R[i], R[i + 1], R[i + 2], R[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if (i < nv) dst[i] = R[i];
                    }
                }
            } else if (row_ok && nv > 0) {
                float zy = 0.0f;
                const int yc = ycol - h * 64;
                const int64_t wi = static_cast<int64_t>(2 * vt + h) * p.ws_ld + row;
                if constexpr (kMode == kModeLseEnt) {
                    float u;
                    p.ws_ms[wi] = tile_lse64_ent(R, min(nv, kLT), yc, zy, u);
                    p.ws_u[wi] = u;
                } else {
                    p.ws_ms[wi] = tile_lse64(R, min(nv, kLT), yc, zy);
                }
                if (yc >= 0 && yc < kLT) p.zy[row] = zy;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace lp
