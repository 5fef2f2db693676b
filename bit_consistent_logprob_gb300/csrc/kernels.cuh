// kernels.cuh -- sm_103a kernels of the logprob path.
//
//  leaf_gemm_kernel<kMode>    persistent, warp-specialised tcgen05 GEMM over 128x128
//                             (token x vocab) tiles: TMA -> smem ring -> tcgen05.mma into
//                             TMEM, one accumulator per K leaf, the fixed leaf tree in
//                             the epilogue, then by mode: the per-tile log-sum-exp partial
//                             and the sampled logit (fused path; optionally the entropy
//                             partial too), the tree node written to global memory
//                             (tensor-parallel slice / leaf export), or the logprob
//                             gradient with respect to the logits (backward).
//  partials_lse_kernel        upper levels of the leaf tree over gathered slice partials,
//                             then the same per-tile log-sum-exp (emulated TP path).
//  lse_combine_kernel<ent>    fixed pairwise tree over the 64-column tiles of each row,
//                             logZ and the sampled-token logprob (and the row entropy).
//  wait_selftest_kernel       the bounded mbarrier wait on a barrier nothing arrives on
//                             (failure-detection self-test).
//  is_block_kernel /
//  is_final_kernel            importance weight per token and D3 over a fixed tree of
//                             1024-token blocks (double-float within a block, fp64 above).
#pragma once

// Non-template kernels are `static` (internal linkage): each translation unit that
// includes this header gets its own copy, compiled from the same source.

#include <cuda.h>
#include <cstdint>
#include <type_traits>

#include "numerics.cuh"
#include "ptx.cuh"

namespace lp {

constexpr int kEpiWarps = 8;                      // 2 per TMEM lane quarter, 64 columns each
constexpr int kGemmThreads = 64 + 32 * kEpiWarps; // TMA warp, MMA warp, 8 epilogue warps
constexpr int kTileBytes = kBM * kBK * 2;         // 16 KB per operand tile per stage
constexpr int kAccBufs = 3;                       // rotating TMEM leaf accumulators
constexpr int kTmemCols = 512;                    // buf0 | buf1 | buf2 | S0 (128 columns each)
constexpr uint32_t kColS0 = kAccBufs * kVT;       // TMEM slot of the deeper partial sum
constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kVT);

// What the epilogue does with each finished 128x128 tile of logits z.
constexpr int kModeNode = 0;     // write z (fp32) to out: a tree node of a leaf range
constexpr int kModeLse = 1;      // (max, sum-exp) per 64-column tile + the sampled logit
constexpr int kModeLseEnt = 2;   // kModeLse + sum e^(z-m)(z-m) per tile (row entropy)
constexpr int kModeGrad = 3;     // dl = g (onehot(y) - e^(z - logZ)) as bf16 to dl

struct GemmParams {
    int32_t T;                // rows of this launch
    int32_t V;
    int32_t leaf_len;         // H / N, a multiple of kBK
    int32_t leaf_begin;       // first leaf of the range (global leaf index)
    int32_t leaf_count;       // leaves in the range: 1, 2, 4 or 8
    int32_t num_row_tiles;    // ceil(T / 128)
    int32_t num_vocab_tiles;  // ceil(V / 128)
    int32_t num_lse_tiles;    // ceil(V / 64)
    int32_t band;             // scheduling units per band (along band_axis)
    int32_t band_axis;        // 0: bands of vocabulary tiles; 1: bands of rows (tiles or pairs)
    int32_t x_box_rows;       // rows per X TMA box (128, or T rounded up to 8 when T < 128)
    const int32_t* ids;       // [T] sampled ids (fused path)
    float2* ws_ms;            // [num_lse_tiles][ws_ld] (max, sum-exp) per 64-column tile (fused)
    int64_t ws_ld;
    float* zy;                // [T] sampled logit (fused path)
    float* out;               // [T][ldo] tree node (partial path)
    int64_t ldo;
    float* ws_u;              // [num_lse_tiles][ws_ld] entropy partial per tile (kModeLseEnt)
    const float* logZ;        // [T] per-row logZ of the forward pass (kModeGrad)
    const float* gout;        // [T] dLoss/dlogp per row (kModeGrad)
    uint16_t* dl;             // [T][ldd] bf16 gradient with respect to the logits (kModeGrad);
                              // kept for the host's record: the kernel writes dl only through
                              // the tmD tensor map and reads neither dl nor ldd
    int64_t ldd;
    const float* sx;          // [T][nkb] activation block scales (block-FP8 kernel)
    const float* sw;          // [num_vocab_tiles][nkb] weight block scales (block-FP8 kernel)
    int32_t nkb;              // 128-K blocks over H (block-FP8 kernel)
    int* sched;               // tile counter of a pair launch's dynamic schedule (zero at launch)
    int32_t test_stop_after;  // test hook: the producer stops after this many stages (0 = off)
    int* status;              // sticky device status word
    uint64_t timeout_ns;      // bound on every mbarrier wait
};

// A pair's tile schedule is dynamic: the leader's producer publishes each next tile in a ring
// of kTileSlots slots that every other warp of both CTAs reads (kTileReaders of them: the
// leader's MMA warp and 8 epilogue warps, the partner's producer, forwarder and 8 epilogue
// warps).
constexpr int kTileSlots = 4;
constexpr int kTileReaders = 2 * (1 + kEpiWarps) + 1;
__host__ __device__ constexpr int kNumBars(int stages) {
    return 2 * stages + 2 * kAccBufs + 1 + 2 * kTileSlots;
}

// A pipeline stage holds kSub 64-wide K sub-blocks of X and of W (4 MMAs of K = 16 per
// sub-block).  More MMAs per stage means fewer barrier synchronisations per MMA in the
// issuing thread; the MMA sequence of a leaf is the same for every kSub.  kSub = 2: three
// 128-K stages (192 KB); kSub = 1: seven 64-K stages (224 KB), the deeper ring for launches
// that stream W from DRAM.
// The gradient epilogue stages each warp's 32 x 64 bf16 block of dl in shared memory for a TMA
// store (8 warps: 32 KB), so its 64-K ring has six stages instead of seven.
// A CTA of a pair (cta_group::2, below) loads only 64 of the vocabulary tile's 128 W rows, so
// its stages are 24 KB per 64-K sub-block instead of 32 KB and its ring holds more of them:
// four 128-K stages or nine 64-K stages (eight beside the gradient staging).
constexpr int kGradWarpBytes = 32 * kLT * 2;
constexpr int kGradStageBytes = kEpiWarps * kGradWarpBytes;
constexpr int kHalfTileBytes = (kVT / 2) * kBK * 2;  // 8 KB: 64 W rows x 64 K
__host__ __device__ constexpr int gemm_stages(int sub, int mode = kModeLse, bool pair = false) {
    return pair ? (sub == 1 ? (mode == kModeGrad ? 8 : 9) : 4)
                : (sub == 1 ? (mode == kModeGrad ? 6 : 7) : 3);
}

// Bytes of one pipeline stage, both operands.
__host__ __device__ constexpr int gemm_stage_bytes(int sub, bool pair = false) {
    return sub * (kTileBytes + (pair ? kHalfTileBytes : kTileBytes));
}

__host__ __device__ constexpr int gemm_smem_bytes(int sub, int mode = kModeLse, bool pair = false) {
    return 1024 /* alignment slack */ + gemm_stages(sub, mode, pair) * gemm_stage_bytes(sub, pair) +
           (mode == kModeGrad ? kGradStageBytes : 0) + kNumBars(gemm_stages(sub, mode, pair)) * 8 +
           8 /* TMEM address, abort flag */ + 4 * kTileSlots /* tile slots */;
}
static_assert(gemm_smem_bytes(1, kModeGrad) <= 227 * 1024 &&
                  gemm_smem_bytes(2, kModeGrad) <= 227 * 1024 && gemm_smem_bytes(1) <= 227 * 1024 &&
                  gemm_smem_bytes(1, kModeGrad, true) <= 227 * 1024 &&
                  gemm_smem_bytes(2, kModeGrad, true) <= 227 * 1024 &&
                  gemm_smem_bytes(1, kModeLse, true) <= 227 * 1024,
              "leaf-GEMM shared memory exceeds the per-CTA limit");

// Tile schedule.  Vocabulary bands (band_axis 0): the vocabulary is cut into bands of `band`
// tiles; within a band the tiles run row by row (a row tile, or the two row tiles of a CTA
// pair), vocabulary fastest, so concurrent CTAs share the band's W tiles (kept in L2) and a
// few X rows; X is read once per band.  Row bands (band_axis 1): the rows are cut into bands of
// `band` rows; within a band the tiles run vocabulary tile by vocabulary tile, rows fastest,
// so the band's X rows stay in L2 and W is read once per band.  The schedule decides only
// which CTA computes a tile, never how.
__device__ __forceinline__ void tile_coords(int tile, int num_rows, const GemmParams& p, int& rt,
                                            int& vt) {
    if (p.band_axis == 0) {
        const int per_band = num_rows * p.band;
        const int b = tile / per_band;
        const int r = tile - b * per_band;
        const int vt0 = b * p.band;
        const int width = min(p.band, p.num_vocab_tiles - vt0);
        rt = r / width;
        vt = vt0 + (r - rt * width);
    } else {
        const int per_band = p.num_vocab_tiles * p.band;
        const int b = tile / per_band;
        const int r = tile - b * per_band;
        const int r0 = b * p.band;
        const int height = min(p.band, num_rows - r0);
        vt = r / height;
        rt = r0 + (r - vt * height);
    }
}

// A wait ran out: stop this CTA's warps (and, in a pair, the partner's) and record it.
template <bool kPair = false>
__device__ __forceinline__ void raise_timeout(const GemmParams& p, volatile int* abort_flag) {
    *abort_flag = 1;
    if constexpr (kPair)
        st_cluster_u32(cluster_addr(const_cast<int*>(abort_flag), cluster_ctarank() ^ 1u), 1u);
    atomicOr(p.status, kStatusTimeout);
}

// Bounded wait on a barrier and its non-blocking probe.  A pair's barriers also receive
// arrivals (and commits) from the partner CTA: the arriving side releases at cluster scope,
// and the waiting side keeps the CTA-scope acquire of every other wait.
template <bool kPair>
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint64_t timeout_ns) {
    return mbar_wait(bar, parity, abort_flag, timeout_ns);
}

template <bool kPair>
__device__ __forceinline__ bool bar_test(uint64_t* bar, uint32_t parity) {
    return mbar_test_wait(bar, parity);
}

// Number of trailing one bits of x.
__device__ __forceinline__ int trailing_ones(int x) { return __ffs(~x) - 1; }

// Warp-uniform bounded wait; on failure raises the abort flag (lane 0) and returns false.
template <bool kPair = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const GemmParams& p,
                                          volatile int* abort_flag) {
    bool got = bar_wait<kPair>(bar, parity, abort_flag, p.timeout_ns);
    got = __all_sync(0xffffffffu, got);
    if (!got && (threadIdx.x & 31) == 0) raise_timeout<kPair>(p, abort_flag);
    return got;
}

// Release a TMEM buffer to the MMA warp: this warp's loads from it have completed.  In a pair
// the MMA warp is the even CTA's, so both CTAs' warps arrive on its barrier.
template <bool kPair = false>
__device__ __forceinline__ void release_buf(uint64_t* bar) {
    tc_fence_before_sync();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        if constexpr (kPair)
            mbar_arrive_cluster(cluster_addr(bar, 0));
        else
            mbar_arrive(bar);
    }
}

// The k-th tile of this CTA (k = 0, 1, ...).  One CTA per tile: the static round robin
// tile0 + k * tile_step.  A pair: the tile the leader's producer published in slot
// k % kTileSlots; the slot is then released on the leader's barrier.  Returns -1 if the wait
// ran out (the abort flag is then raised).
template <bool kPair>
__device__ __forceinline__ int next_tile(uint32_t k, int tile0, int tile_step,
                                         const volatile int* slots, uint64_t* tile_full,
                                         uint32_t tile_empty_leader, const GemmParams& p,
                                         volatile int* abort_flag) {
    if constexpr (!kPair) {
        return tile0 + static_cast<int>(k) * tile_step;
    } else {
        const uint32_t s = k % kTileSlots;
        bool got = mbar_wait_cl(&tile_full[s], (k / kTileSlots) & 1u, abort_flag, p.timeout_ns);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
            if ((threadIdx.x & 31) == 0) raise_timeout<true>(p, abort_flag);
            return -1;
        }
        const int t = slots[s];
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive_cluster(tile_empty_leader + 8u * s);
        return t;
    }
}

// kPair = false: one CTA per 128 x 128 tile; each CTA loads its own X and W boxes.
// kPair = true: clusters of two CTAs (a pair) compute the two row tiles 2*rp and 2*rp + 1 of
// one vocabulary tile with tcgen05.mma.cta_group::2 (M = 256).  Each CTA loads its own
// 128-row X box and 64 of the tile's 128 W rows (tmW then has 64-row boxes) into its own
// shared memory and its own barrier; nothing is multicast.  The even CTA (the leader) issues
// the MMAs, which read both CTAs' shared memory and write each CTA's 128 rows of the
// accumulator into that CTA's TMEM; the odd CTA's MMA warp forwards its stage completions to
// the leader (one remote arrive per stage); the leader's commits free the stages and
// publish the accumulators in both CTAs (one commit per CTA's barrier), and both CTAs'
// epilogue warps release the TMEM buffers on the leader's barrier.  A CTA whose row tile lies
// past T still loads (zero-filled rows) and computes, but writes nothing.  Every element sees
// the same K = 16 MMA sequence, leaf tree and tile log-sum-exp as with one CTA per tile.
// A pair's tiles are handed out dynamically: the clusters do not all run at the same speed,
// and with a static round robin the tiles in flight drift apart over a launch (measured at
// the DS shape: 28 rounds of 76 clusters by the end) until the X rows they share fall out of
// L2.  The leader's producer takes each next tile from the zeroed counter p.sched (one atomic
// per tile, fetched a tile ahead) and publishes it to both CTAs (next_tile).
// tmD (kModeGrad only): dl as bf16 [T][ldd] with 64 x 32 boxes, 128-byte swizzle.
template <int kMode, int kSub, bool kPair = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
    leaf_gemm_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
    constexpr int kStages = gemm_stages(kSub, kMode, kPair);
    constexpr int kBTile = kPair ? kHalfTileBytes : kTileBytes;  // W bytes per 64-K sub-block
    constexpr int kStageA = kSub * kTileBytes;           // X bytes per stage
    constexpr int kStageB = kSub * kBTile;               // W bytes per stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                                  // X  [kStages][kSub][128 x 64] bf16
    uint8_t* sB = smem + kStages * kStageA;              // W  [kStages][kSub][128|64 x 64] bf16
    uint8_t* sD = sB + kStages * kStageB;                // dl staging [8 warps][32 x 64] bf16
    uint64_t* bars = reinterpret_cast<uint64_t*>(
        sD + (kMode == kModeGrad ? kGradStageBytes : 0));
    uint64_t* full = bars;                               // TMA -> MMA, per stage
    uint64_t* empty = bars + kStages;                    // MMA -> TMA, per stage
    uint64_t* acc_full = bars + 2 * kStages;             // MMA -> epilogue, per TMEM buffer
    uint64_t* acc_empty = acc_full + kAccBufs;           // epilogue -> MMA, per TMEM buffer
    uint64_t* drain = acc_empty + kAccBufs;              // MMA drain on abort
    uint64_t* tile_full = drain + 1;                     // pair: tile index published, per slot
    uint64_t* tile_empty = tile_full + kTileSlots;       // pair: slot read by every reader
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tile_empty + kTileSlots);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* tile_slot = abort_flag + 1;            // pair: [kTileSlots] tile indices

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = kPair ? cluster_ctarank() : 0u;
    const bool leader = crank == 0u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // the leader's stage is ready when its own copies landed and the partner forwarded
            // the completion of its copies
            mbar_init(&full[s], kPair && leader ? 2 : 1);
            mbar_init(&empty[s], 1);  // the MMA commit that frees the stage
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(&acc_full[b], 1);
            // every epilogue warp (of both CTAs of a pair) reads every buffer
            mbar_init(&acc_empty[b], kPair ? 2 * kEpiWarps : kEpiWarps);
        }
        mbar_init(drain, 1);
        for (int s = 0; s < kTileSlots; ++s) {
            mbar_init(&tile_full[s], 1);
            mbar_init(&tile_empty[s], kTileReaders);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        if constexpr (kPair) {
            tmem_alloc_pair(tmem_holder, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_holder, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kPair) cluster_sync_all();  // the partner's barriers exist before any signal
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;

    // scheduling rows: row tiles, or row-tile pairs
    const int num_rows = kPair ? (p.num_row_tiles + 1) >> 1 : p.num_row_tiles;
    const int num_tiles = num_rows * p.num_vocab_tiles;
    const int tile0 = static_cast<int>(kPair ? blockIdx.x >> 1 : blockIdx.x);
    const int tile_step = static_cast<int>(kPair ? gridDim.x >> 1 : gridDim.x);
    const uint32_t tile_empty_leader = kPair ? cluster_addr(tile_empty, 0) : 0u;
    const int nkb = p.leaf_len / (kBK * kSub);   // stages per leaf
    const int n = p.leaf_count;

    constexpr uint32_t kFull = 0xffffffffu;
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (warp)
        const uint32_t tx_bytes = static_cast<uint32_t>(kSub * (p.x_box_rows * kBK * 2 + kBTile));
        uint32_t stage = 0, phase = 0;
        uint64_t issued = 0;
        bool ok = true;
        // the leader of a pair publishes the tile sequence: tile0 first, then one counter value
        // per tile (taken a tile ahead, so the atomic's latency hides behind a tile of loads)
        const bool publish = kPair && leader;
        const uint32_t slot_peer = publish ? cluster_addr(const_cast<int*>(tile_slot), 1) : 0u;
        const uint32_t tfull_peer = publish ? cluster_addr(tile_full, 1) : 0u;
        int next = tile0;
        int ahead = 0;
        if (publish && lane == 0) ahead = atomicAdd(p.sched, 1);
        for (uint32_t k = 0; ok; ++k) {
            int tile;
            if (publish) {
                tile = next;
                const uint32_t s = k % kTileSlots;
                ok = __all_sync(kFull, mbar_wait(&tile_empty[s], ((k / kTileSlots) & 1u) ^ 1u,
                                                 abort_flag, p.timeout_ns));
                if (!ok) {
                    if (lane == 0) raise_timeout<kPair>(p, abort_flag);
                    break;
                }
                if (lane == 0) {
                    tile_slot[s] = tile;
                    st_cluster_u32(slot_peer + 4u * s, static_cast<uint32_t>(tile));
                    mbar_arrive(&tile_full[s]);
                    mbar_arrive_cluster_release(tfull_peer + 8u * s);
                }
                __syncwarp();
                if (tile >= num_tiles) break;
                next = tile_step + __shfl_sync(kFull, ahead, 0);
                if (lane == 0) ahead = atomicAdd(p.sched, 1);
            } else {
                tile = next_tile<kPair>(k, tile0, tile_step, tile_slot, tile_full,
                                        tile_empty_leader, p, abort_flag);
                if (tile < 0) {
                    ok = false;
                    break;
                }
                if (tile >= num_tiles) break;
            }
            int rt, vt;
            tile_coords(tile, num_rows, p, rt, vt);
            if constexpr (kPair) rt = 2 * rt + static_cast<int>(crank);
            const int row0 = rt * kBM;
            const int w0 = vt * kVT + static_cast<int>(crank) * (kVT / 2);  // this CTA's W rows
            for (int jj = 0; ok && jj < n; ++jj) {
                const int kbase = (p.leaf_begin + jj) * p.leaf_len;
                for (int kb = 0; kb < nkb; ++kb) {
                    ok = __all_sync(kFull, bar_wait<kPair>(&empty[stage], phase ^ 1u, abort_flag,
                                                           p.timeout_ns));
                    if (!ok) {
                        if (lane == 0) raise_timeout<kPair>(p, abort_flag);
                        break;
                    }
                    mbar_arrive_expect_tx_elect(&full[stage], tx_bytes);
#pragma unroll
                    for (int u = 0; u < kSub; ++u) {
                        const int k0 = kbase + (kb * kSub + u) * kBK;
                        uint8_t* xdst = sA + stage * kStageA + u * kTileBytes;
                        uint8_t* wdst = sB + stage * kStageB + u * kBTile;
                        tma_load_2d_elect(&tmX, &full[stage], xdst, k0, row0);
                        tma_load_2d_elect(&tmW, &full[stage], wdst, k0, w0);
                    }
                    ++issued;
                    // test hook: stop as if this warp's own wait had run out (the consumers'
                    // bounded waits then expire and the abort path runs)
                    if (p.test_stop_after > 0 && issued >= uint64_t(p.test_stop_after)) {
                        ok = false;
                        break;
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (!ok) {
            // Let the copies already in flight land before the CTA exits.  (A leader's stage
            // also counts the partner's forwarded arrival; if that never comes the wait runs
            // to its limit, long after the copies themselves have landed.)
            const uint64_t first = issued > kStages ? issued - kStages : 0;
            for (uint64_t i = first; i < issued; ++i) {
                volatile int never = 0;
                mbar_wait(&full[i % kStages], static_cast<uint32_t>((i / kStages) & 1u), &never,
                          p.timeout_ns);
            }
        }
    } else if (kPair && warp == 1 && !leader) {
        // ------------------------------------------------------------ forwarder (odd CTA)
        // Each time this CTA's copies of a stage have landed, arrive on the leader's barrier of
        // that stage (the leader's MMAs read this CTA's shared memory).  The stage sequence is
        // the producer's.
        const uint32_t full_leader = cluster_addr(full, 0);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (uint32_t k = 0; ok; ++k) {
            const int tile = next_tile<kPair>(k, tile0, tile_step, tile_slot, tile_full,
                                              tile_empty_leader, p, abort_flag);
            if (tile < 0) {
                ok = false;
                break;
            }
            if (tile >= num_tiles) break;
            for (int jj = 0; ok && jj < n; ++jj) {
                for (int kb = 0; kb < nkb; ++kb) {
                    ok = __all_sync(kFull, mbar_wait(&full[stage], phase, abort_flag, p.timeout_ns));
                    if (!ok) {
                        if (lane == 0) raise_timeout<kPair>(p, abort_flag);
                        break;
                    }
                    if (lane == 0) mbar_arrive_cluster(full_leader + 8u * stage);
                    __syncwarp();
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (warp)
        // The tensor core's instruction queue is shallow, so the issuing loop does as little
        // as possible between MMAs: descriptors are precomputed, buffer/stage indices advance
        // incrementally, every value is warp-uniform, and the barriers of the next stage and
        // of the next leaf's buffer are probed (non-blocking) while this stage's MMAs run.
        const uint64_t descA = sw128_kmajor_desc(smem_u32(sA));
        const uint64_t descB = sw128_kmajor_desc(smem_u32(sB));
        constexpr uint32_t kStageDescA = kStageA >> 4;  // descriptor units per stage
        constexpr uint32_t kStageDescB = kStageB >> 4;
        constexpr uint32_t kSubDesc = kTileBytes >> 4;  // ... per 64-K sub-block of X
        constexpr uint32_t kIdescRun = kPair ? idesc_bf16_f32(2 * kBM, kVT) : kIdesc;
        // the barriers a pair's commits arrive on: this CTA's and the partner's
        const uint32_t empty_own = smem_u32(empty), empty_peer = kPair ? cluster_addr(empty, 1) : 0u;
        const uint32_t accf_own = smem_u32(acc_full),
                       accf_peer = kPair ? cluster_addr(acc_full, 1) : 0u;
        uint32_t stage = 0, phase = 0;
        uint32_t buf = 0, bphase = 0;  // TMEM buffer of the current leaf, its use parity
        bool ok = true;
        bool ready = __all_sync(kFull, bar_test<kPair>(&full[0], 0));
        bool acc_ready = true;  // the first uses of every buffer find it free
        for (uint32_t k = 0; ok; ++k) {
            const int tile = next_tile<kPair>(k, tile0, tile_step, tile_slot, tile_full,
                                              tile_empty_leader, p, abort_flag);
            if (tile < 0) {
                ok = false;
                break;
            }
            if (tile >= num_tiles) break;
            for (int jj = 0; ok && jj < n; ++jj) {
                if (!acc_ready) {
                    ok = __all_sync(kFull, bar_wait<kPair>(&acc_empty[buf], bphase ^ 1u,
                                                           abort_flag, p.timeout_ns));
                    if (!ok) {
                        if (lane == 0) raise_timeout<kPair>(p, abort_flag);
                        break;
                    }
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + (buf << 7);
                const uint32_t nbuf = buf + 1 == kAccBufs ? 0u : buf + 1;
                const uint32_t nbphase = buf + 1 == kAccBufs ? bphase ^ 1u : bphase;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!ready) {
                        ok = __all_sync(kFull, bar_wait<kPair>(&full[stage], phase, abort_flag,
                                                               p.timeout_ns));
                        if (!ok) {
                            if (lane == 0) raise_timeout<kPair>(p, abort_flag);
                            break;
                        }
                    }
                    tc_fence_after_sync();
                    const uint32_t nstage = stage + 1 == kStages ? 0u : stage + 1;
                    const uint32_t nphase = stage + 1 == kStages ? phase ^ 1u : phase;
                    const uint64_t a = descA + stage * kStageDescA;
                    const uint64_t b = descB + stage * kStageDescB;
                    // +32 bytes (2 descriptor units) per K step of 16 bf16 inside a row;
                    // only the leaf's very first MMA starts a fresh accumulator; the commit
                    // frees the stage (in a pair: in both CTAs)
                    static_assert(kSubDesc == 1024, "sub-block stride assumed by the stage issue");
                    if constexpr (kPair)
                        umma_pair_stage_elect<kSub>(d_tmem, a, b, kIdescRun, kb != 0 ? 1u : 0u,
                                                    empty_own + 8u * stage,
                                                    empty_peer + 8u * stage);
                    else
                        umma_stage_elect<kSub>(d_tmem, a, b, kIdescRun, kb != 0 ? 1u : 0u,
                                               &empty[stage]);
                    // probe the next stage (and the next leaf's buffer) while these MMAs run
                    ready = __all_sync(kFull, bar_test<kPair>(&full[nstage], nphase));
                    if (kb == nkb - 1)
                        acc_ready =
                            __all_sync(kFull, bar_test<kPair>(&acc_empty[nbuf], nbphase ^ 1u));
                    stage = nstage;
                    phase = nphase;
                }
                if (!ok) break;
                if constexpr (kPair)
                    umma_commit2_pair_elect(accf_own + 8u * buf, accf_peer + 8u * buf);
                else
                    umma_commit_elect(&acc_full[buf]);
                buf = nbuf;
                bphase = nbphase;
            }
        }
        if (!ok) {
            // Wait for every MMA already issued before TMEM is released.
            volatile int never = 0;
            if constexpr (kPair)
                umma_commit_pair_elect(smem_u32(drain));
            else
                umma_commit_elect(drain);
            mbar_wait(drain, 0, &never, p.timeout_ns);
        }
    } else {
        // ------------------------------------------------------------ epilogue (8 warps)
        // Warp w may read TMEM lanes 32*(w%4)..+31; warps 2-5 take columns 0-63 of each
        // 128-column buffer, warps 6-9 columns 64-127.
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const int r_in_tile = q * 32 + lane;
        const uint32_t lane_base =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * 64);
        uint32_t g = 0;
        bool ok = true;
        for (uint32_t k = 0; ok; ++k) {
            const int tile = next_tile<kPair>(k, tile0, tile_step, tile_slot, tile_full,
                                              tile_empty_leader, p, abort_flag);
            if (tile < 0) {
                ok = false;
                break;
            }
            if (tile >= num_tiles) break;
            int rt, vt;
            tile_coords(tile, num_rows, p, rt, vt);
            if constexpr (kPair) rt = 2 * rt + static_cast<int>(crank);
            const int row = rt * kBM + r_in_tile;
            const int v0 = vt * kVT;
            const bool row_ok = row < p.T;
            int ycol = -1;
            if (kMode != kModeNode && row_ok) {
                const int y = p.ids[row];
                if (y >= 0 && y < p.V) ycol = y - v0;
            }
            // Leaf tree: every even leaf waits in its TMEM buffer for its odd partner, the
            // pair sum P_{2i} + P_{2i+1} is read from the two buffers, and the pair sums are
            // combined in post-order (the newest partial in registers R, the one below it in
            // TMEM slot S0) -- the same adds, in the same tree, as level-by-level pairing.
            float R[64];
            int depth = 0;
            const int npairs = n >> 1;
            for (int jj = 0; jj < n; ++jj, ++g) {
                const uint32_t buf = g % kAccBufs, use = g / kAccBufs;
                if (!warp_wait<kPair>(&acc_full[buf], use & 1u, p, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t colB = buf * kVT;
                if (n == 1) {
                    tmem_ld64(lane_base + colB, R);
                    release_buf<kPair>(&acc_empty[buf]);
                    continue;
                }
                if ((jj & 1) == 0) continue;  // wait for the partner leaf
                const uint32_t pbuf = (g + kAccBufs - 1) % kAccBufs;
                const uint32_t colP = pbuf * kVT;
                const int i = jj >> 1;  // pair index
                if ((i & 1) == 0 && i != npairs - 1) {
                    // push the pair sum (spilling the current top to S0): R is free, so both
                    // leaves load in one round trip
                    if (depth == 1) tmem_st64(lane_base + kColS0, R);
                    float b[64];
                    tmem_ld64x2(lane_base + colP, R, lane_base + colB, b);
                    add_rn_x2<64>(R, b);
                    ++depth;
                } else if (npairs == 1) {
                    // single pair: the node is P0 + P1
                    float b[64];
                    tmem_ld64x2(lane_base + colP, R, lane_base + colB, b);
                    add_rn_x2<64>(R, b);
                } else {
                    // odd pair index: close the subtrees that end at this pair
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        float a[32], b[32];
                        tmem_ld32x2(lane_base + colP + cc * 32, a, lane_base + colB + cc * 32, b);
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            R[cc * 32 + k] = __fadd_rn(R[cc * 32 + k], __fadd_rn(a[k], b[k]));
                    }
                    if (trailing_ones(i) >= 2) {
                        float b[64];
                        tmem_ld64(lane_base + kColS0, b);
                        add_rn_x2<64>(R, b);
                        --depth;
                    }
                }
                release_buf<kPair>(&acc_empty[pbuf]);
                release_buf<kPair>(&acc_empty[buf]);
            }
            if (!ok) break;
            {
                const int col0 = v0 + h * 64;
                if constexpr (kMode == kModeLse) {
                    // the 64-column log-sum-exp tile 2*vt + h of this row is entirely in R
                    const int nv = p.V - col0;
                    if (row_ok && nv > 0) {
                        float zy = 0.0f;
                        const int yc = ycol - h * 64;
                        const float2 ms = tile_lse64(R, min(nv, kLT), yc, zy);
                        p.ws_ms[static_cast<int64_t>(2 * vt + h) * p.ws_ld + row] = ms;
                        if (yc >= 0 && yc < kLT) p.zy[row] = zy;
                    }
                } else if constexpr (kMode == kModeLseEnt) {
                    const int nv = p.V - col0;
                    if (row_ok && nv > 0) {
                        float zy = 0.0f, u;
                        const int yc = ycol - h * 64;
                        const int64_t wi = static_cast<int64_t>(2 * vt + h) * p.ws_ld + row;
                        p.ws_ms[wi] = tile_lse64_ent(R, min(nv, kLT), yc, zy, u);
                        p.ws_u[wi] = u;
                        if (yc >= 0 && yc < kLT) p.zy[row] = zy;
                    }
                } else if constexpr (kMode == kModeGrad) {
                    // The warp's 32 rows x 64 columns of dl go to its shared-memory block in the
                    // 128-byte swizzled layout (16-byte chunk c of row r at chunk c ^ (r % 8):
                    // conflict-free), then one TMA store writes them; rows >= T and columns >= V
                    // fall outside the tensor map and are not written.
                    const int nv = p.V - col0;
                    const int wrow0 = rt * kBM + q * 32;
                    if (nv > 0 && wrow0 < p.T) {  // warp-uniform
                        uint32_t pk[32];
                        if (row_ok) {
                            const float lz = p.logZ[row], gg = p.gout[row];
                            const int yc = ycol - h * 64;
#pragma unroll
                            for (int i = 0; i < 64; i += 2) {
                                float d[2];
#pragma unroll
                                for (int k = 0; k < 2; ++k) {
                                    const float pr = __expf(__fsub_rn(R[i + k], lz));
                                    d[k] = __fmul_rn(gg, __fsub_rn(i + k == yc ? 1.0f : 0.0f, pr));
                                }
                                pk[i >> 1] = pack_bf16x2(d[0], d[1]);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) pk[i] = 0u;
                        }
                        uint8_t* blk = sD + (warp - 2) * kGradWarpBytes;
                        if (lane == 0) bulk_wait_read_all();  // the last store has read blk
                        __syncwarp();
                        uint8_t* myrow = blk + lane * (kLT * 2);
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4*>(myrow + ((c ^ (lane & 7)) << 4)) =
                                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmD, blk, col0, wrow0);
                            bulk_commit_group();
                        }
                    }
                } else if (row_ok) {
                    float* dst = p.out + static_cast<int64_t>(row) * p.ldo + col0;
                    if (col0 + 64 <= p.V) {
#pragma unroll
                        for (int i = 0; i < 64; i += 4)
                            *reinterpret_cast<float4*>(dst + i) =
                                make_float4(R[i], R[i + 1], R[i + 2], R[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if (col0 + i < p.V) dst[i] = R[i];
                    }
                }
            }
        }
        if constexpr (kMode == kModeGrad) {
            if (lane == 0) bulk_wait_all();  // this warp's dl stores have completed
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kPair) cluster_sync_all();  // no arrive or commit still targets either CTA
    if (warp == 1) {
        tc_fence_after_sync();
        if constexpr (kPair)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Upper levels of the leaf tree over gathered partials (one per slice), then the
// log-sum-exp partials of the two 64-column tiles and the sampled logit, exactly as the fused
// epilogue forms them.  grid: (num_vocab_tiles, ceil(T/128)); block: 128 threads, one row each.
struct PartialsParams {
    const float* parts;      // [n_parts] x [T][ldp]
    int64_t part_stride;
    int64_t ldp;
    int32_t n_parts;         // 1, 2, 4, 8
    int32_t T;
    int32_t V;
    const int32_t* ids;
    float2* ws_ms;
    float* ws_u;             // entropy partials (kEnt)
    int64_t ws_ld;
    float* zy;
};

template <int kParts, bool kEnt>
__global__ void __launch_bounds__(128) partials_lse_kernel(const PartialsParams p) {
    const int vt = blockIdx.x;
    const int row = blockIdx.y * 128 + threadIdx.x;
    if (row >= p.T) return;
    const int y = p.ids[row];
    const float* base = p.parts + static_cast<int64_t>(row) * p.ldp;
#pragma unroll 1
    for (int h = 0; h < kVT / kLT; ++h) {
        const int col0 = vt * kVT + h * kLT;
        const int nv = p.V - col0;
        if (nv <= 0) break;
        float z[kLT];
#pragma unroll
        for (int i = 0; i < kLT; ++i) {
            float node[kParts];
#pragma unroll
            for (int k = 0; k < kParts; ++k)
                node[k] = i < nv ? base[k * p.part_stride + col0 + i] : 0.0f;
#pragma unroll
            for (int w = kParts >> 1; w >= 1; w >>= 1)
#pragma unroll
                for (int k = 0; k < w; ++k) node[k] = __fadd_rn(node[2 * k], node[2 * k + 1]);
            z[i] = node[0];
        }
        const int ycol = (y >= 0 && y < p.V) ? y - col0 : -1;
        float zy = 0.0f;
        const int64_t wi = static_cast<int64_t>(2 * vt + h) * p.ws_ld + row;
        if constexpr (kEnt) {
            float u;
            p.ws_ms[wi] = tile_lse64_ent(z, min(nv, kLT), ycol, zy, u);
            p.ws_u[wi] = u;
        } else {
            p.ws_ms[wi] = tile_lse64(z, min(nv, kLT), ycol, zy);
        }
        if (ycol >= 0 && ycol < kLT) p.zy[row] = zy;
    }
}

// Fixed pairwise tree over the 64-column log-sum-exp tiles of each row (adjacent pairs
// first, level by level; an odd last entry moves up a level unchanged), logZ and logp.
//
// Level l of that tree holds one node per aligned block [j 2^l, (j+1) 2^l) of tiles (cut
// at the last tile), and two nodes merge exactly when their blocks are siblings.  So any
// split of the tiles into aligned power-of-two segments gives the same nodes in the same
// merge order: a thread folds one segment (8-tile rounds, each an in-register tree, joined
// by a binary counter whose final fold runs from the smallest block up), and the segments
// of a row meet in a shared-memory tree.  The split is chosen per launch for occupancy
// and coalescing; the bits do not depend on it.
// block: rows x nseg threads, thread (r, g) at g * rows + r; grid: ceil(T / rows).
struct CombineParams {
    const float2* ws_ms;
    const float* ws_u;        // entropy partials (entropy variant)
    int64_t ws_ld;
    const float* zy;
    const int32_t* ids;
    int32_t T;
    int32_t V;
    int32_t num_tiles;        // ceil(V / 64)
    int32_t rows;             // rows per block (power of two, <= 16)
    int32_t seg_log;          // tiles per segment = 2^seg_log, 3 <= seg_log <= kSegLogMax
    int32_t nseg;             // ceil(num_tiles / 2^seg_log); rows * nseg <= 512
    float* out_logp;
    float* out_logZ;          // may be null
    float* out_entropy;       // entropy variant only
    int* status;
};

constexpr int kCmbRound = 8;      // tiles per in-register tree
constexpr int kSegLogMax = 11;    // up to 2^11 tiles per thread
constexpr int kCmbMaxThreads = 512;

struct CombineLayout {
    int rows, seg_log, nseg;
};

// Rows per block: the largest power of two <= 16 that still gives every SM two blocks;
// segment length: the shortest that fits the block in 512 threads and the grid in about
// two waves of 2048 threads per SM.
__host__ inline CombineLayout combine_layout(int64_t T, int num_tiles, int num_sms) {
    CombineLayout c{1, 3, 0};
    while (c.rows < 16 && static_cast<int64_t>(c.rows) * 2 * num_sms <= T) c.rows *= 2;
    const int64_t groups = (T + c.rows - 1) / c.rows;
    for (;;) {
        c.nseg = (num_tiles + (1 << c.seg_log) - 1) >> c.seg_log;
        const int64_t threads = groups * c.rows * c.nseg;
        if (c.seg_log == kSegLogMax) break;
        if (c.rows * c.nseg <= kCmbMaxThreads && threads <= int64_t(4096) * num_sms) break;
        ++c.seg_log;
    }
    while (c.rows > 1 && c.rows * c.nseg > kCmbMaxThreads) c.rows /= 2;  // V beyond 2^21 only
    return c;
}

template <bool kEnt>
__global__ void __launch_bounds__(kCmbMaxThreads) lse_combine_kernel(const CombineParams p) {
    // (m, s) per tile, or (m, s, u) with the entropy partial; merged by the same tree
    using Acc = typename std::conditional<kEnt, float3, float2>::type;
    extern __shared__ __align__(16) uint8_t cmb_raw[];
    Acc* cmb = reinterpret_cast<Acc*>(cmb_raw);  // [nseg][rows]
    const auto load = [&](int b, int row) -> Acc {
        const int64_t i = static_cast<int64_t>(b) * p.ws_ld + row;
        const float2 ms = __ldg(p.ws_ms + i);
        if constexpr (kEnt) return make_float3(ms.x, ms.y, __ldg(p.ws_u + i));
        else return ms;
    };
    const auto merge = [](Acc a, Acc b) -> Acc {
        if constexpr (kEnt) return lse_merge_ent(a, b);
        else return lse_merge(a, b);
    };
    const int r = threadIdx.x % p.rows;
    const int g = threadIdx.x / p.rows;
    const int row = blockIdx.x * p.rows + r;
    const bool row_ok = row < p.T;
    if (row_ok) {
        const int b_end = min((g + 1) << p.seg_log, p.num_tiles);
        Acc stack[kSegLogMax - 2];     // counter levels: blocks of 8, 16, ..., 2^kSegLogMax
        uint32_t k = 0;                // rounds folded so far
        const int b_begin = g << p.seg_log;
        Acc nxt[kCmbRound];            // the next round's tiles, loaded one round ahead
#pragma unroll
        for (int i = 0; i < kCmbRound; ++i)
            if (b_begin + i < b_end) nxt[i] = load(b_begin + i, row);
        for (int b = b_begin; b < b_end; b += kCmbRound, ++k) {
            const int nv = min(kCmbRound, b_end - b);
            Acc v[kCmbRound];
#pragma unroll
            for (int i = 0; i < kCmbRound; ++i) v[i] = nxt[i];
            const int bn = b + kCmbRound;
#pragma unroll
            for (int i = 0; i < kCmbRound; ++i)
                if (bn + i < b_end) nxt[i] = load(bn + i, row);
#pragma unroll
            for (int w = 1; w < kCmbRound; w <<= 1)
#pragma unroll
                for (int i = 0; i < kCmbRound; i += 2 * w)
                    if (i + w < nv) v[i] = merge(v[i], v[i + w]);
            Acc carry = v[0];
            bool open = true;  // carry not yet stored
#pragma unroll
            for (int j = 0; j < kSegLogMax - 2; ++j) {
                if (open) {
                    if ((k >> j) & 1u) {
                        carry = merge(stack[j], carry);
                    } else {
                        stack[j] = carry;
                        open = false;
                    }
                }
            }
        }
        // blocks still open, smallest (rightmost) first
        Acc acc{};
        bool have = false;
#pragma unroll
        for (int j = 0; j < kSegLogMax - 2; ++j) {
            if ((k >> j) & 1u) {
                acc = have ? merge(stack[j], acc) : stack[j];
                have = true;
            }
        }
        cmb[g * p.rows + r] = acc;
    }
    __syncthreads();
    for (int s = 1; s < p.nseg; s <<= 1) {
        if (row_ok && (g & (2 * s - 1)) == 0 && g + s < p.nseg)
            cmb[g * p.rows + r] = merge(cmb[g * p.rows + r], cmb[(g + s) * p.rows + r]);
        __syncthreads();
    }
    if (row_ok && g == 0) {
        const Acc fin = cmb[r];
        const float lz = lse_finish(make_float2(fin.x, fin.y));
        const int y = p.ids[row];
        float lp;
        if (y >= 0 && y < p.V) {
            lp = __fsub_rn(p.zy[row], lz);
        } else {
            lp = __int_as_float(0x7fc00000);
            atomicOr(p.status, kStatusBadId);
        }
        p.out_logp[row] = lp;
        if (p.out_logZ) p.out_logZ[row] = lz;
        if constexpr (kEnt) p.out_entropy[row] = entropy_finish(fin);
    }
}

// Failure-detection self-test: one mbarrier that nothing ever arrives on (no copy, no MMA, no
// TMEM in flight), waited on with the same bounded wait as every pipeline barrier.  The wait
// must give up after timeout_ns, raise the sticky timeout bit and return, leaving the context
// usable.  One block of 32 threads.
static __global__ void __launch_bounds__(32) wait_selftest_kernel(int* status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const bool got = __all_sync(0xffffffffu, mbar_wait(&bar, 0, &abort_flag, timeout_ns));
    if (!got && threadIdx.x == 0) atomicOr(status, kStatusTimeout);
}

// ---------------------------------------------------------------------- IS / D3
constexpr int kIsBlock = 1024;       // tokens per D3 block (fixed; the tree is over blocks)
constexpr int kIsThreads = 256;      // 4 tokens per thread
constexpr int kIsChunk = 2048;       // block partials per level-wise pass of the final kernel

struct IsParams {
    const float* logp_pi;
    const float* logp_mu;
    const uint8_t* mask;     // may be null
    int64_t T;
    float* out_w;
    double* blk_sum;         // [num_blocks]
    long long* blk_cnt;      // [num_blocks]
};

// Per token: d = log pi - log mu, w = e^d, term = e^d - 1 - d.  Per block of 1024 tokens:
// each thread adds its 4 valid terms in order (double-float), a lane butterfly sums the warp
// (double-float), and a pairwise fp64 tree sums the 8 warps.
__device__ __forceinline__ double block_sum_8warps(df32 v, double* wsum) {
    v = warp_sum_df(v);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = df_to_f64(v);
    __syncthreads();
    const double s01 = __dadd_rn(wsum[0], wsum[1]), s23 = __dadd_rn(wsum[2], wsum[3]);
    const double s45 = __dadd_rn(wsum[4], wsum[5]), s67 = __dadd_rn(wsum[6], wsum[7]);
    return __dadd_rn(__dadd_rn(s01, s23), __dadd_rn(s45, s67));
}

static __global__ void __launch_bounds__(kIsThreads) is_block_kernel(const IsParams p) {
    __shared__ double wsum[kIsThreads / 32];
    __shared__ long long wcnt[kIsThreads / 32];
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kIsBlock + threadIdx.x * 4;
    df32 acc{0.0f, 0.0f};
    long long cnt = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t t = t0 + i;
        if (t < p.T) {
            const float d = __fsub_rn(p.logp_pi[t], p.logp_mu[t]);
            p.out_w[t] = expf(d);
            const bool valid = p.mask == nullptr || p.mask[t] != 0;
            if (valid) {
                acc = df_add(acc, d3_term(d));
                ++cnt;
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    if ((threadIdx.x & 31) == 0) wcnt[threadIdx.x >> 5] = cnt;
    const double total = block_sum_8warps(acc, wsum);
    if (threadIdx.x == 0) {
        p.blk_sum[blockIdx.x] = total;
        long long c = 0;
        for (int w = 0; w < kIsThreads / 32; ++w) c += wcnt[w];
        p.blk_cnt[blockIdx.x] = c;
    }
}

// Level-wise pairwise fp64 tree over n values in shared memory (in place), using the
// whole block.  Result in a[0].
__device__ __forceinline__ void block_tree_f64(double* a, int n) {
    while (n > 1) {
        const int half = n >> 1;
        for (int base = 0; base < half; base += blockDim.x) {
            const int i = base + threadIdx.x;
            double r = 0.0;
            if (i < half) r = __dadd_rn(a[2 * i], a[2 * i + 1]);
            __syncthreads();
            if (i < half) a[i] = r;
            __syncthreads();
        }
        if (n & 1) {
            if (threadIdx.x == 0) a[half] = a[n - 1];
            __syncthreads();
        }
        n = half + (n & 1);
    }
}

// The level-wise pairwise tree over n <= 2^21 block partials, taken in aligned chunks of
// kIsChunk (each chunk is a whole subtree of the level-wise tree, so the result is the
// same as one tree over every partial).  Called by a whole block of 1024 threads; `a`
// holds kIsChunk and `chunk_res` 1024 doubles of shared memory.  The result is returned
// to every thread.
__device__ __forceinline__ double tree_over_partials(const double* src, int n, double* a,
                                                     double* chunk_res) {
    const int num_chunks = (n + kIsChunk - 1) / kIsChunk;
    for (int ch = 0; ch < num_chunks; ++ch) {
        const int lo = ch * kIsChunk;
        const int len = min(kIsChunk, n - lo);
        for (int i = threadIdx.x; i < len; i += blockDim.x) a[i] = src[lo + i];
        __syncthreads();
        block_tree_f64(a, len);
        if (threadIdx.x == 0) chunk_res[ch] = a[0];
        __syncthreads();
    }
    if (num_chunks > 0) block_tree_f64(chunk_res, num_chunks);
    __syncthreads();
    const double r = num_chunks > 0 ? chunk_res[0] : 0.0;
    __syncthreads();
    return r;
}

// Exact sum of n counts (integer adds; the order does not matter).  Whole block of 1024.
__device__ __forceinline__ long long block_count_sum(const long long* src, int n,
                                                     long long* part) {
    long long c = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) c += src[i];
    part[threadIdx.x] = c;
    __syncthreads();
    for (int w = blockDim.x >> 1; w >= 1; w >>= 1) {
        if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    const long long r = part[0];
    __syncthreads();
    return r;
}

// One block: D3 = (tree over the block sums) / n_valid.
static __global__ void __launch_bounds__(1024) is_final_kernel(const double* blk_sum,
                                                        const long long* blk_cnt, int num_blocks,
                                                        double* out_d3, int64_t* out_nvalid) {
    __shared__ double a[kIsChunk];
    __shared__ double chunk_res[1024];
    __shared__ long long cnt_part[1024];
    const long long total = block_count_sum(blk_cnt, num_blocks, cnt_part);
    const double sum = tree_over_partials(blk_sum, num_blocks, a, chunk_res);
    if (threadIdx.x == 0) {
        *out_d3 = total > 0 ? __ddiv_rn(sum, static_cast<double>(total)) : 0.0;
        if (out_nvalid) *out_nvalid = total;
    }
}

}  // namespace lp
