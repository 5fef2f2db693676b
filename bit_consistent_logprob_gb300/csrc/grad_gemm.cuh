// grad_gemm.cuh -- the two GEMMs of the logprob backward on tcgen05, in CTA pairs
// (cta_group::2, one MMA of M = 256 over two SMs):
//
//   dX [rows][H]  = dl [rows][V]   . W [V][H]     M = rows, N = H, K = V     (A K-major)
//   dW [V][H]    += dl^T [V][rows] . X [rows][H]  M = V,    N = H, K = rows  (A M-major)
//
// dl is the bf16 gradient with respect to the logits written by the leaf GEMM's gradient
// epilogue.  B (W or X) is N-major in both (H contiguous), and so is dl^T as the A operand of
// dW (V contiguous in a row of dl), so those operand tiles are MN-major: TMA boxes of 64
// (M or N) x 64 (K) elements with the 128-byte swizzle, two boxes side by side for 128
// elements (the canonical MN-major layout: 128-byte K rows, 8-row groups 1 KB apart, the two
// 64-element halves 8 KB apart).
//
// One pair computes a 256 x 256 tile of D: each CTA loads its 128 rows of A and its 128 of
// the tile's 256 B columns into its own shared memory (six 64-K stages of 32 KB), the odd CTA
// forwards its stage completions to the even CTA with one remote arrive, the even CTA issues
// the MMAs (which read both CTAs' shared memory) and frees the stages and publishes the
// accumulator in both CTAs with one commit per CTA's barrier.  Each CTA holds its 128 rows x
// 256 fp32 columns in TMEM (two buffers: the epilogue of one tile overlaps the next tile's
// MMAs); eight epilogue warps per CTA write them to D, or add them to it.  The work units
// are (K slice, M tile, N tile), N fastest: a split K writes one fp32 partial per slice,
// which splitk_sum_kernel then adds in slice order.  Nothing depends on which CTA computes a
// unit, so the results do not depend on the launch.  Every wait is bounded.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "numerics.cuh"
#include "ptx.cuh"

namespace lp {

constexpr int kGgEpiWarps = 8;                        // 2 per TMEM lane quarter, 128 columns each
constexpr int kGgThreads = 64 + 32 * kGgEpiWarps;     // TMA warp, MMA/forwarder warp, epilogue
constexpr int kGgStages = 6;
constexpr int kGgHalfBytes = 128 * kBK * 2;           // 16 KB: 128 (M or N) x 64 K, bf16
constexpr int kGgStageBytes = 2 * kGgHalfBytes;       // A and B of one CTA
constexpr int kGgTileN = 256;                         // N of a pair tile (128 loaded per CTA)
constexpr int kGgTileM = 256;                         // M of a pair tile (128 per CTA)
constexpr int kGgAccBufs = 2;
constexpr int kGgTmemCols = kGgAccBufs * kGgTileN;    // 512
constexpr int kGgNumBars = 2 * kGgStages + 2 * kGgAccBufs + 1;
constexpr int kGgSmemBytes = 1024 + kGgStages * kGgStageBytes + kGgNumBars * 8 + 8;
static_assert(kGgSmemBytes <= 227 * 1024, "backward GEMM shared memory exceeds the per-CTA limit");

struct GradGemmParams {
    int32_t M, N, K;          // D is M x N; the sum runs over K
    int32_t k_slice;          // K per slice (a multiple of 64)
    int32_t num_m;            // ceil(M / 256)
    int32_t num_n;            // ceil(N / 256)
    int32_t num_slices;       // K slices (1 = no split)
    float* D;                 // [num_slices][M][ldd] (slice outputs slice_stride apart)
    int64_t ldd;
    int64_t slice_stride;
    int32_t accumulate;       // 1: D += the product, 0: D = the product
    int* status;              // sticky device status word
    uint64_t timeout_ns;      // bound on every mbarrier wait
};

// Shared-memory descriptor of an MN-major tile written by TMA with the 128-byte swizzle:
// 128-byte K rows of 64 elements, 8-row groups 1 KB apart (stride byte offset), the second
// 64-element half 8 KB further (leading byte offset).  Same field layout as sw128_kmajor_desc.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(8192u >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of the pair MMA: fp32 accumulator, bf16 A and B, M = 256, N = 256,
// A K-major (dX) or MN-major (dW), B MN-major.
__host__ __device__ constexpr uint32_t grad_idesc(bool a_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | (1u << 16) |
           ((uint32_t(kGgTileN) >> 3) << 17) | ((uint32_t(kGgTileM) >> 4) << 24);
}

// One 64-K stage of pair MMAs from one elected lane: 4 MMAs of K = 16, A advanced by OA and
// B by 128 descriptor units (2 KB: 16 MN-major K rows) per step; the first with the caller's
// accumulate flag; then one commit per CTA's stage barrier.
#define LP_GMMA(A, B, P) "@e tcgen05.mma.cta_group::2.kind::f16 [%0], " A ", " B ", %3, " P ";\n\t"
#define LP_GADV(OA, OB) "add.s64 a1, %1, " OA ";\n\tadd.s64 b1, %2, " OB ";\n\t"
#define LP_GHEAD                                                        \
    "{\n\t.reg .pred e, p, t;\n\t.reg .b64 a1, b1;\n\t"                \
    "elect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
#define LP_GTAIL                                                                          \
    "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t" \
    "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}"
template <bool kAMN>
__device__ __forceinline__ void grad_stage_elect(uint32_t d_tmem, uint64_t a, uint64_t b,
                                                 uint32_t idesc, uint32_t accumulate,
                                                 uint32_t bar_own, uint32_t bar_peer) {
    if constexpr (kAMN) {
        asm volatile(LP_GHEAD LP_GMMA("%1", "%2", "p") LP_GADV("128", "128")
                         LP_GMMA("a1", "b1", "t") LP_GADV("256", "256") LP_GMMA("a1", "b1", "t")
                             LP_GADV("384", "384") LP_GMMA("a1", "b1", "t") LP_GTAIL ::"r"(d_tmem),
                     "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(bar_own), "r"(bar_peer)
                     : "memory");
    } else {
        asm volatile(LP_GHEAD LP_GMMA("%1", "%2", "p") LP_GADV("2", "128") LP_GMMA("a1", "b1", "t")
                         LP_GADV("4", "256") LP_GMMA("a1", "b1", "t") LP_GADV("6", "384")
                             LP_GMMA("a1", "b1", "t") LP_GTAIL ::"r"(d_tmem),
                     "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(bar_own), "r"(bar_peer)
                     : "memory");
    }
}
#undef LP_GMMA
#undef LP_GADV
#undef LP_GHEAD
#undef LP_GTAIL

__device__ __forceinline__ void gg_unit_coords(int u, const GradGemmParams& p, int& s, int& mt,
                                               int& nt) {
    const int per_slice = p.num_m * p.num_n;
    s = u / per_slice;
    const int r = u - s * per_slice;
    mt = r / p.num_n;
    nt = r - mt * p.num_n;
}

// A wait ran out: stop this CTA's warps and the partner's, and record it.
__device__ __forceinline__ void gg_raise_timeout(const GradGemmParams& p, volatile int* abort_flag) {
    *abort_flag = 1;
    st_cluster_u32(cluster_addr(const_cast<int*>(abort_flag), cluster_ctarank() ^ 1u), 1u);
    atomicOr(p.status, kStatusTimeout);
}

__device__ __forceinline__ bool gg_warp_wait(uint64_t* bar, uint32_t parity,
                                             const GradGemmParams& p, volatile int* abort_flag) {
    bool got = mbar_wait(bar, parity, abort_flag, p.timeout_ns);
    got = __all_sync(0xffffffffu, got);
    if (!got && (threadIdx.x & 31) == 0) gg_raise_timeout(p, abort_flag);
    return got;
}

// tmA: K-major A (dX: dl, boxes of 64 K x 128 rows) or MN-major A (dW: dl seen as
// [K = rows][M = V], boxes of 64 M x 64 K); tmB: MN-major B ([K][N], boxes of 64 N x 64 K).
// grid: two CTAs per cluster, one cluster per pair of SMs (persistent); block: kGgThreads.
template <bool kAMN>
__global__ void __launch_bounds__(kGgThreads, 1)
    grad_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const GradGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                                     // [stage][16 KB]
    uint8_t* sB = smem + kGgStages * kGgHalfBytes;          // [stage][16 KB]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kGgStages * kGgStageBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + kGgStages;
    uint64_t* acc_full = bars + 2 * kGgStages;
    uint64_t* acc_empty = acc_full + kGgAccBufs;
    uint64_t* drain = acc_empty + kGgAccBufs;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const bool leader = crank == 0u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGgStages; ++s) {
            mbar_init(&full[s], leader ? 2 : 1);  // the leader also counts the partner's forward
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < kGgAccBufs; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 2 * kGgEpiWarps);  // every epilogue warp of both CTAs
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, kGgTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // the partner's barriers exist before any signal
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;

    const int num_units = p.num_slices * p.num_m * p.num_n;
    const int unit0 = static_cast<int>(blockIdx.x >> 1);
    const int unit_step = static_cast<int>(gridDim.x >> 1);
    constexpr uint32_t kFull = 0xffffffffu;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (warp)
        uint32_t stage = 0, phase = 0;
        uint64_t issued = 0;
        bool ok = true;
        for (int u = unit0; ok && u < num_units; u += unit_step) {
            int s, mt, nt;
            gg_unit_coords(u, p, s, mt, nt);
            const int k_begin = s * p.k_slice;
            const int k_len = min(p.k_slice, p.K - k_begin);
            const int nkb = (k_len + kBK - 1) / kBK;
            const int m0 = mt * kGgTileM + static_cast<int>(crank) * 128;  // this CTA's A rows
            const int n0 = nt * kGgTileN + static_cast<int>(crank) * 128;  // this CTA's B half
            for (int kb = 0; kb < nkb; ++kb) {
                ok = __all_sync(kFull, mbar_wait(&empty[stage], phase ^ 1u, abort_flag,
                                                 p.timeout_ns));
                if (!ok) {
                    if (lane == 0) gg_raise_timeout(p, abort_flag);
                    break;
                }
                mbar_arrive_expect_tx_elect(&full[stage], kGgStageBytes);
                const int k0 = k_begin + kb * kBK;
                uint8_t* a = sA + stage * kGgHalfBytes;
                uint8_t* b = sB + stage * kGgHalfBytes;
                if constexpr (kAMN) {
                    tma_load_2d_elect(&tmA, &full[stage], a, m0, k0);
                    tma_load_2d_elect(&tmA, &full[stage], a + kGgHalfBytes / 2, m0 + 64, k0);
                } else {
                    tma_load_2d_elect(&tmA, &full[stage], a, k0, m0);
                }
                tma_load_2d_elect(&tmB, &full[stage], b, n0, k0);
                tma_load_2d_elect(&tmB, &full[stage], b + kGgHalfBytes / 2, n0 + 64, k0);
                ++issued;
                if (++stage == kGgStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            // Let the copies already in flight land before the CTA exits.
            const uint64_t first = issued > kGgStages ? issued - kGgStages : 0;
            for (uint64_t i = first; i < issued; ++i) {
                volatile int never = 0;
                mbar_wait(&full[i % kGgStages], static_cast<uint32_t>((i / kGgStages) & 1u),
                          &never, p.timeout_ns);
            }
        }
    } else if (warp == 1 && !leader) {
        // ------------------------------------------------------------ forwarder (odd CTA)
        const uint32_t full_leader = cluster_addr(full, 0);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int u = unit0; ok && u < num_units; u += unit_step) {
            int s, mt, nt;
            gg_unit_coords(u, p, s, mt, nt);
            const int k_len = min(p.k_slice, p.K - s * p.k_slice);
            const int nkb = (k_len + kBK - 1) / kBK;
            for (int kb = 0; kb < nkb; ++kb) {
                ok = __all_sync(kFull, mbar_wait(&full[stage], phase, abort_flag, p.timeout_ns));
                if (!ok) {
                    if (lane == 0) gg_raise_timeout(p, abort_flag);
                    break;
                }
                if (lane == 0) mbar_arrive_cluster(full_leader + 8u * stage);
                __syncwarp();
                if (++stage == kGgStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        const uint64_t descA = kAMN ? sw128_mnmajor_desc(smem_u32(sA)) : sw128_kmajor_desc(smem_u32(sA));
        const uint64_t descB = sw128_mnmajor_desc(smem_u32(sB));
        constexpr uint32_t kStageDesc = kGgHalfBytes >> 4;
        constexpr uint32_t kIdescRun = grad_idesc(kAMN);
        const uint32_t empty_own = smem_u32(empty), empty_peer = cluster_addr(empty, 1);
        const uint32_t accf_own = smem_u32(acc_full), accf_peer = cluster_addr(acc_full, 1);
        uint32_t stage = 0, phase = 0;
        uint32_t buf = 0, bphase = 0;
        bool ok = true;
        for (int u = unit0; ok && u < num_units; u += unit_step) {
            int s, mt, nt;
            gg_unit_coords(u, p, s, mt, nt);
            const int k_len = min(p.k_slice, p.K - s * p.k_slice);
            const int nkb = (k_len + kBK - 1) / kBK;
            ok = __all_sync(kFull, mbar_wait(&acc_empty[buf], bphase ^ 1u, abort_flag, p.timeout_ns));
            if (!ok) {
                if (lane == 0) gg_raise_timeout(p, abort_flag);
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + buf * kGgTileN;
            for (int kb = 0; kb < nkb; ++kb) {
                ok = __all_sync(kFull, mbar_wait(&full[stage], phase, abort_flag, p.timeout_ns));
                if (!ok) {
                    if (lane == 0) gg_raise_timeout(p, abort_flag);
                    break;
                }
                tc_fence_after_sync();
                grad_stage_elect<kAMN>(d_tmem, descA + stage * kStageDesc, descB + stage * kStageDesc,
                                       kIdescRun, kb != 0 ? 1u : 0u, empty_own + 8u * stage,
                                       empty_peer + 8u * stage);
                if (++stage == kGgStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit2_pair_elect(accf_own + 8u * buf, accf_peer + 8u * buf);
            if (++buf == kGgAccBufs) {
                buf = 0;
                bphase ^= 1u;
            }
        }
        if (!ok) {
            volatile int never = 0;
            umma_commit_pair_elect(smem_u32(drain));
            mbar_wait(drain, 0, &never, p.timeout_ns);
        }
    } else {
        // ------------------------------------------------------------ epilogue (8 warps)
        // Warp w reads TMEM lanes 32*(w%4)..+31 (its 32 rows); warps 2-5 take accumulator
        // columns 0-127, warps 6-9 columns 128-255.
        const int q = warp & 3;
        const int hcol = (warp - 2) >> 2;
        const uint32_t acc_empty_leader = cluster_addr(acc_empty, 0);
        uint32_t buf = 0, bphase = 0;
        bool ok = true;
        for (int u = unit0; ok && u < num_units; u += unit_step) {
            int s, mt, nt;
            gg_unit_coords(u, p, s, mt, nt);
            if (!gg_warp_wait(&acc_full[buf], bphase, p, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const int row = mt * kGgTileM + static_cast<int>(crank) * 128 + q * 32 + lane;
            const int col0 = nt * kGgTileN + hcol * 128;
            float* drow = p.D + static_cast<int64_t>(s) * p.slice_stride +
                          static_cast<int64_t>(row) * p.ldd;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   buf * kGgTileN + static_cast<uint32_t>(hcol * 128);
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
                float v[32];
                tmem_ld32(taddr + static_cast<uint32_t>(c), v);
                const int n = col0 + c;
                if (row < p.M && n < p.N) {
                    float* dst = drow + n;
                    if (n + 32 <= p.N) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            float4 o = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                            if (p.accumulate) {
                                const float4 old = *reinterpret_cast<const float4*>(dst + i);
                                o.x = __fadd_rn(old.x, o.x);
                                o.y = __fadd_rn(old.y, o.y);
                                o.z = __fadd_rn(old.z, o.z);
                                o.w = __fadd_rn(old.w, o.w);
                            }
                            *reinterpret_cast<float4*>(dst + i) = o;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (n + i < p.N) dst[i] = p.accumulate ? __fadd_rn(dst[i], v[i]) : v[i];
                    }
                }
            }
            // this warp's TMEM reads are complete: release the buffer on the even CTA's barrier
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty_leader + 8u * buf);
            if (++buf == kGgAccBufs) {
                buf = 0;
                bphase ^= 1u;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // no arrive or commit still targets either CTA
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, kGgTmemCols);
    }
}

// out[i] = sum over s of part[s][i], added in slice order (a fixed left fold), n elements,
// n a multiple of 4 and every pointer 16-byte aligned.
static __global__ void splitk_sum_kernel(const float* __restrict__ part, int slices,
                                         int64_t slice_stride, int64_t n, float* __restrict__ out) {
    const int64_t n4 = n >> 2;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4;
         i += int64_t(gridDim.x) * blockDim.x) {
        float4 acc = reinterpret_cast<const float4*>(part)[i];
        for (int s = 1; s < slices; ++s) {
            const float4 v = reinterpret_cast<const float4*>(part + s * slice_stride)[i];
            acc.x = __fadd_rn(acc.x, v.x);
            acc.y = __fadd_rn(acc.y, v.y);
            acc.z = __fadd_rn(acc.z, v.z);
            acc.w = __fadd_rn(acc.w, v.w);
        }
        reinterpret_cast<float4*>(out)[i] = acc;
    }
}

}  // namespace lp
