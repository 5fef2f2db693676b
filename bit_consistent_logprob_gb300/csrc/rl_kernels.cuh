// Epilogues of the RL step that consume per-token logprobs.
//
//  stats_fused_kernel   acceptance statistics between two logprob vectors: max, mean and
//                       population std of |a - b| and the k3 estimate mean(r - 1 - log r),
//                       r = e^(a - b), over valid tokens (vLLM blog "Finish RL training
//                       faster", section 2: acceptance asks max, mean and std of the
//                       per-token difference to be 0; section 3.2: the k3 estimator).  Its
//                       block partials (stats_block_kernel) and its finish (stats_final_kernel)
//                       also run separately for the data-parallel path.
//  is_fused_kernel      importance weights and D3 in one launch: the per-token weights and
//                       block partials of is_block_kernel, then the last block to finish runs
//                       is_final_kernel's fixed tree over every block partial (same bits).
//  rz_seq_kernel        the REINFORCE Zero loss L = -(1/B) sum_i (1/T_i) sum_t A_i w_it with
//                       group-mean advantages, its gradient with respect to log pi, and the
//                       TIS / token-gate / sequence-gate options (REINFORCE Zero summary,
//                       section 4 and results table; vLLM blog, section 1); one block per
//                       response, the loss's fixed tree in the last block to finish.
//
// Per-token sums are double-float (fp32 pairs, error-free additions) within a thread and a
// warp and fp64 above, in a fixed order that depends only on token positions (1024-token
// blocks) or on the response itself (one block per response), never on the launch.
#pragma once

#include <cstdint>

#include "kernels.cuh"
#include "numerics.cuh"

namespace lp {

constexpr int kStatusBadOffsets = 4;  // a response's [offs[i], offs[i+1]) is not inside [0, T)

// ---------------------------------------------------------------------- one-launch finishing
// A kernel whose blocks each publish a partial can finish in its last block: every block
// fences and counts itself done, and the block that finds it was the last runs the fixed tree
// over all partials (reading them past L1), then zeroes the counter for the next launch.  The
// tree and its operands are those of the separate finishing kernels, so the bits are too.

// Thread 0 publishes this block's partials before the call; returns, to every thread, whether
// this block was the last of num_blocks to finish.
__device__ __forceinline__ bool finished_last(unsigned* done, int num_blocks, int* flag) {
    if (threadIdx.x == 0) {
        __threadfence();
        *flag = atomicAdd(done, 1u) == static_cast<unsigned>(num_blocks - 1);
    }
    __syncthreads();
    const bool last = *flag != 0;
    if (last) __threadfence();
    return last;
}

// The level-wise pairwise tree of block_tree_f64 (pairs (2i, 2i + 1), an odd last value
// carried up a level) is the aligned binary tree over the value indices: node (L, j) is the sum
// of the values [j 2^L, (j + 1) 2^L) that exist, formed as node (L - 1, 2j) + node (L - 1, 2j + 1),
// or as node (L - 1, 2j) alone when no value falls in the right half.  The last block of a
// launch (kIsThreads threads) evaluates each aligned chunk of kIsChunk values in that form:
// every thread its 8 consecutive values (levels 1-3) in registers, every warp levels 4-8 by a
// lane butterfly, thread 0 levels 9-11 over the 8 warp results; block_tree_f64 then joins the
// chunks.  The additions, their operands and their order are those of tree_over_partials, so
// are the bits, with one barrier per chunk instead of two per level.
static_assert(kIsChunk == 8 * kIsThreads, "a thread holds 8 consecutive values of a chunk");

// Node (3, t) of a chunk: v[k] is the chunk's value first + k (first = 8 t); `len` values exist.
__device__ __forceinline__ double tree_levels_1_3(const double (&v)[8], int first, int len) {
    double n1[4], n2[2];
#pragma unroll
    for (int m = 0; m < 4; ++m)
        n1[m] = first + 2 * m + 1 < len ? __dadd_rn(v[2 * m], v[2 * m + 1]) : v[2 * m];
#pragma unroll
    for (int m = 0; m < 2; ++m)
        n2[m] = first + 4 * m + 2 < len ? __dadd_rn(n1[2 * m], n1[2 * m + 1]) : n1[2 * m];
    return first + 4 < len ? __dadd_rn(n2[0], n2[1]) : n2[0];
}

// Levels 4-8: lane l of warp w enters with node (3, 32 w + l) and every lane leaves with node
// (8, w).  At distance `off` the lower lane of a pair of groups holds the left child and the
// upper lane the right one; both form left + right, or take the left child when the right
// half holds no value.
__device__ __forceinline__ double tree_levels_4_8(double v, int len) {
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int warp_first = static_cast<int>(threadIdx.x >> 5) * 256;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double o = __shfl_xor_sync(0xffffffffu, v, off);
        const bool low = (lane & off) == 0;
        const int right_first = warp_first + 8 * ((lane & ~(2 * off - 1)) + off);
        if (right_first < len) v = low ? __dadd_rn(v, o) : __dadd_rn(o, v);
        else if (!low) v = o;
    }
    return v;
}

// Levels 9-11 from r[w] = node (8, w), w < 8.
__device__ __forceinline__ double tree_levels_9_11(const double* r, int len) {
    double a[4], b[2];
#pragma unroll
    for (int m = 0; m < 4; ++m)
        a[m] = 256 * (2 * m + 1) < len ? __dadd_rn(r[2 * m], r[2 * m + 1]) : r[2 * m];
#pragma unroll
    for (int m = 0; m < 2; ++m)
        b[m] = 512 * (2 * m + 1) < len ? __dadd_rn(a[2 * m], a[2 * m + 1]) : a[2 * m];
    return 1024 < len ? __dadd_rn(b[0], b[1]) : b[0];
}

// The tree over n <= 2^21 partials (0 for n = 0), by the whole block; `chunk_res` holds 1024
// and `wres` 8 doubles of shared memory.  Every thread gets the result.
__device__ __forceinline__ double last_block_tree(const double* src, int n, double* chunk_res,
                                                  double* wres) {
    const int num_chunks = (n + kIsChunk - 1) / kIsChunk;
    const int first = 8 * static_cast<int>(threadIdx.x);
    for (int ch = 0; ch < num_chunks; ++ch) {
        const double* c = src + static_cast<int64_t>(ch) * kIsChunk;
        const int len = min(kIsChunk, n - ch * kIsChunk);
        double v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = first + k < len ? __ldcg(c + first + k) : 0.0;
        const double node = tree_levels_4_8(tree_levels_1_3(v, first, len), len);
        if ((threadIdx.x & 31) == 0) wres[threadIdx.x >> 5] = node;
        __syncthreads();
        if (threadIdx.x == 0) chunk_res[ch] = tree_levels_9_11(wres, len);
        __syncthreads();
    }
    if (num_chunks > 1) block_tree_f64(chunk_res, num_chunks);
    const double r = num_chunks > 0 ? chunk_res[0] : 0.0;
    __syncthreads();
    return r;
}

// Sum of n counts (integer adds, any order) by the whole block, each thread reading 8 at a
// time; `wcnt` holds 8 long longs of shared memory.  Every thread gets the result.
__device__ __forceinline__ long long last_block_count(const long long* src, int n,
                                                      long long* wcnt) {
    const int first = 8 * static_cast<int>(threadIdx.x);
    long long c = 0;
    for (int lo = 0; lo < n; lo += kIsChunk) {
        long long v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = lo + first + k < n ? __ldcg(src + lo + first + k) : 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) c += v[k];
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
    if ((threadIdx.x & 31) == 0) wcnt[threadIdx.x >> 5] = c;
    __syncthreads();
    long long r = 0;
#pragma unroll
    for (int w = 0; w < kIsThreads / 32; ++w) r += wcnt[w];
    __syncthreads();
    return r;
}

// Whether four consecutive elements starting at p can move as one 16-byte (or, for bytes,
// 4-byte) access.
template <typename T>
__device__ __forceinline__ bool aligned_x4(const T* p) {
    return (reinterpret_cast<uintptr_t>(p) & (4 * sizeof(T) - 1)) == 0;
}

// Thread j of a 1024-token block reads tokens t0 .. t0 + 3 (t0 = block * 1024 + 4 j): a = log pi
// (or the first logprob), b = log mu (or the second), valid = inside [0, T) and unmasked.  One
// vector load per input when the four are inside T and the pointers are aligned.
__device__ __forceinline__ void load_token_quad(const float* pa, const float* pb,
                                                const uint8_t* mask, int64_t T, int64_t t0,
                                                float (&a)[4], float (&b)[4], bool (&valid)[4],
                                                bool& vec) {
    vec = t0 + 3 < T && aligned_x4(pa) && aligned_x4(pb) && (mask == nullptr || aligned_x4(mask));
    if (vec) {
        const float4 va = *reinterpret_cast<const float4*>(pa + t0);
        const float4 vb = *reinterpret_cast<const float4*>(pb + t0);
        a[0] = va.x; a[1] = va.y; a[2] = va.z; a[3] = va.w;
        b[0] = vb.x; b[1] = vb.y; b[2] = vb.z; b[3] = vb.w;
        const uint32_t m = mask ? *reinterpret_cast<const uint32_t*>(mask + t0) : 0x01010101u;
#pragma unroll
        for (int i = 0; i < 4; ++i) valid[i] = ((m >> (8 * i)) & 0xffu) != 0;
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t t = t0 + i;
            a[i] = t < T ? pa[t] : 0.0f;
            b[i] = t < T ? pb[t] : 0.0f;
            valid[i] = t < T && (mask == nullptr || mask[t] != 0);
        }
    }
}

// ---------------------------------------------------------------------- acceptance statistics
struct StatsParams {
    const float* a;          // learner logprob (log pi)
    const float* b;          // rollout logprob (log mu)
    const uint8_t* mask;     // may be null
    int64_t T;
    double* blk_abs;         // [num_blocks] sum |d|
    double* blk_sq;          // [num_blocks] sum d^2
    double* blk_k3;          // [num_blocks] sum (e^d - 1 - d)
    float* blk_max;          // [num_blocks] max |d| (NaN if any valid |d| is NaN)
    long long* blk_cnt;      // [num_blocks] valid tokens
};

// max that keeps a NaN once seen (fmaxf would drop it); commutative for every input pair
__device__ __forceinline__ float nan_max(float m, float x) { return (x > m || x != x) ? x : m; }

// Max of n block maxima by the whole block, each thread reading 8 at a time; `wmax` holds 8
// floats of shared memory.  Every GPU-computed NaN has the same bits, so any order gives the
// same result.  Every thread gets it.
__device__ __forceinline__ float last_block_max(const float* src, int n, float* wmax) {
    const int first = 8 * static_cast<int>(threadIdx.x);
    float m = 0.0f;
    for (int lo = 0; lo < n; lo += kIsChunk) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = lo + first + k < n ? __ldcg(src + lo + first + k) : 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) m = nan_max(m, v[k]);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = nan_max(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    float r = 0.0f;
#pragma unroll
    for (int w = 0; w < kIsThreads / 32; ++w) r = nan_max(r, wmax[w]);
    __syncthreads();
    return r;
}

// Block sums with block_sum_8warps' arithmetic (each warp's lane butterfly of fp32 pairs,
// the pair widened to fp64, the 8-warp tree ((w0 + w1) + (w2 + w3)) + ((w4 + w5) + (w6 + w7))),
// for NS sums at once.  The fp64 pipe of a GB300 SM is narrow, and a warp instruction holds it
// for as long whatever its active lanes, so the fp64 steps run in warp 0 with lane 8s + w
// holding warp w's value of sum s: one instruction per step for every warp and sum (six in
// all) instead of a widening in each warp and a tree in one thread.
template <int NS>
struct BlockSums {
    static_assert(NS >= 1 && NS <= 4, "lane 8s + w of one warp per sum s and warp w");
    float hi[8 * NS], lo[8 * NS];
};

// Sum s of the calling warp: its lane butterfly, then lane 0 stores the warp's pair.
template <int NS>
__device__ __forceinline__ void stage_warp_sum(df32 v, int s, BlockSums<NS>& sh) {
    v = warp_sum_df(v);
    if ((threadIdx.x & 31) == 0) {
        sh.hi[8 * s + (threadIdx.x >> 5)] = v.hi;
        sh.lo[8 * s + (threadIdx.x >> 5)] = v.lo;
    }
}

// After a barrier that follows every stage_warp_sum, called by all lanes of warp 0: sum s ends
// in lane 8s (other lanes hold partial or unused values).
template <int NS>
__device__ __forceinline__ double finish_block_sums(const BlockSums<NS>& sh) {
    const int l = static_cast<int>(threadIdx.x & 31);
    double x = 0.0;
    if (l < 8 * NS) x = __dadd_rn(static_cast<double>(sh.hi[l]), static_cast<double>(sh.lo[l]));
#pragma unroll
    for (int off = 1; off <= 4; off <<= 1) {
        const double y = __shfl_down_sync(0xffffffffu, x, off);
        if ((l & (2 * off - 1)) == 0 && l < 8 * NS) x = __dadd_rn(x, y);
    }
    return x;
}

// Per block of 1024 tokens (4 per thread, in order): three double-float sums reduced exactly
// like the D3 block sum (is_block_kernel), so the k3 partials are bit-equal to the D3 partials
// of the same tokens; |d|^2 enters exactly (an fma recovers the product's rounding error);
// max and count are exact in any order.  Thread 0 writes the block's partials.  Warps 1-7
// return after the block barrier; warp 0 returns once it has formed the fp64 sums.
__device__ __forceinline__ void stats_block_body(const StatsParams& p, BlockSums<3>& s_w,
                                                 float* s_max, long long* s_cnt) {
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kIsBlock + threadIdx.x * 4;
    float a[4], b[4];
    bool valid[4], vec;
    load_token_quad(p.a, p.b, p.mask, p.T, t0, a, b, valid, vec);
    df32 acc_abs{0.0f, 0.0f}, acc_sq{0.0f, 0.0f}, acc_k3{0.0f, 0.0f};
    float mx = 0.0f;
    long long cnt = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (valid[i]) {
            const float d = __fsub_rn(a[i], b[i]);
            const float x = fabsf(d);
            acc_abs = df_add(acc_abs, x);
            acc_sq = df_add(acc_sq, square_exact(x));
            acc_k3 = df_add(acc_k3, d3_term(d));
            mx = nan_max(mx, x);
            ++cnt;
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        mx = nan_max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    }
    if ((threadIdx.x & 31) == 0) {
        s_max[threadIdx.x >> 5] = mx;
        s_cnt[threadIdx.x >> 5] = cnt;
    }
    stage_warp_sum(acc_abs, 0, s_w);
    stage_warp_sum(acc_sq, 1, s_w);
    stage_warp_sum(acc_k3, 2, s_w);
    __syncthreads();
    if (threadIdx.x >= 32) return;
    const double x = finish_block_sums(s_w);
    const double sum_sq = __shfl_sync(0xffffffffu, x, 8);
    const double sum_k3 = __shfl_sync(0xffffffffu, x, 16);
    if (threadIdx.x == 0) {
        p.blk_abs[blockIdx.x] = x;
        p.blk_sq[blockIdx.x] = sum_sq;
        p.blk_k3[blockIdx.x] = sum_k3;
        float m = 0.0f;
        long long c = 0;
        for (int w = 0; w < 8; ++w) {
            m = nan_max(m, s_max[w]);
            c += s_cnt[w];
        }
        p.blk_max[blockIdx.x] = m;
        p.blk_cnt[blockIdx.x] = c;
    }
}

static __global__ void __launch_bounds__(kIsThreads) stats_block_kernel(const StatsParams p) {
    __shared__ BlockSums<3> s_w;
    __shared__ float s_max[8];
    __shared__ long long s_cnt[8];
    stats_block_body(p, s_w, s_max, s_cnt);
}

// The statistics of stats_final_kernel from n_valid and the three sums.
__device__ __forceinline__ void stats_finish(double mx, long long n, double s_abs, double s_sq,
                                             double s_k3, double* out) {
    if (n == 0) {
        for (int i = 0; i < 5; ++i) out[i] = 0.0;
    } else {
        const double nd = static_cast<double>(n);
        const double mean = __ddiv_rn(s_abs, nd);
        const double var = __dsub_rn(__ddiv_rn(s_sq, nd), __dmul_rn(mean, mean));
        out[0] = mx;
        out[1] = mean;
        out[2] = var > 0.0 ? __dsqrt_rn(var) : (var == var ? 0.0 : var);
        out[3] = __ddiv_rn(s_k3, nd);
        out[4] = nd;
    }
}

// stats_block_kernel and stats_final_kernel in one launch: every block writes its partials,
// the last block to finish forms the statistics from all of them (same trees, same bits).
static __global__ void __launch_bounds__(kIsThreads, 8) stats_fused_kernel(const StatsParams p,
                                                                       int num_blocks,
                                                                       unsigned* done,
                                                                       double* out) {
    __shared__ BlockSums<3> s_w;
    __shared__ float s_max[8];
    __shared__ long long s_cnt[8];
    __shared__ int last;
    stats_block_body(p, s_w, s_max, s_cnt);
    if (!finished_last(done, num_blocks, &last)) return;
    // the block's own scratch is free again (finished_last synchronised the block)
    __shared__ double chunk_res[1024];
    const float mx = last_block_max(p.blk_max, num_blocks, s_max);
    const long long n = last_block_count(p.blk_cnt, num_blocks, s_cnt);
    __shared__ double wres[kIsThreads / 32];
    const double s_abs = last_block_tree(p.blk_abs, num_blocks, chunk_res, wres);
    const double s_sq = last_block_tree(p.blk_sq, num_blocks, chunk_res, wres);
    const double s_k3 = last_block_tree(p.blk_k3, num_blocks, chunk_res, wres);
    if (threadIdx.x == 0) {
        stats_finish(static_cast<double>(mx), n, s_abs, s_sq, s_k3, out);
        *done = 0u;
    }
}

// One block of 1024: the fixed trees over the block sums, then
// out[0] = max |d|, out[1] = mean |d|, out[2] = sqrt(max(0, mean d^2 - mean^2)),
// out[3] = k3, out[4] = n_valid; all zero when n_valid == 0.
static __global__ void __launch_bounds__(1024) stats_final_kernel(const StatsParams p,
                                                           int num_blocks, double* out) {
    __shared__ double a[kIsChunk];
    __shared__ double chunk_res[1024];
    __shared__ long long cnt_part[1024];
    __shared__ float max_part[1024];
    float m = 0.0f;
    for (int i = threadIdx.x; i < num_blocks; i += blockDim.x) m = nan_max(m, p.blk_max[i]);
    max_part[threadIdx.x] = m;
    const long long n = block_count_sum(p.blk_cnt, num_blocks, cnt_part);  // syncs
    for (int w = blockDim.x >> 1; w >= 1; w >>= 1) {
        if (threadIdx.x < w) max_part[threadIdx.x] = nan_max(max_part[threadIdx.x],
                                                             max_part[threadIdx.x + w]);
        __syncthreads();
    }
    const double s_abs = tree_over_partials(p.blk_abs, num_blocks, a, chunk_res);
    const double s_sq = tree_over_partials(p.blk_sq, num_blocks, a, chunk_res);
    const double s_k3 = tree_over_partials(p.blk_k3, num_blocks, a, chunk_res);
    if (threadIdx.x == 0) stats_finish(static_cast<double>(max_part[0]), n, s_abs, s_sq, s_k3, out);
}

// ---------------------------------------------------------------------- IS / D3, one launch
struct IsFusedParams {
    IsParams is;
    int num_blocks;          // ceil(T / kIsBlock) >= 1
    unsigned* done;          // blocks finished; zero at launch, zeroed again by the last block
    double* out_d3;
    int64_t* out_nvalid;     // may be null
};

// Per block of 1024 tokens (thread j takes tokens 4j .. 4j + 3 of the block, in order): w = e^d
// and the double-float sum of the valid tokens' D3 terms, reduced to the block partial by the
// lane butterfly and the 8-warp fp64 tree, with the valid count: the arithmetic of
// is_block_kernel, operation for operation (full groups of four move as one vector load of
// each input and one vector store of w).  The last block to finish then sums every block
// partial with is_final_kernel's tree and writes D3 = sum / n_valid.
static __global__ void __launch_bounds__(kIsThreads, 8) is_fused_kernel(const IsFusedParams q) {
    const IsParams& p = q.is;
    __shared__ BlockSums<1> bsum;
    __shared__ double wsum[kIsThreads / 32];
    __shared__ long long wcnt[kIsThreads / 32];
    __shared__ int last;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kIsBlock + threadIdx.x * 4;
    float a[4], b[4];
    bool valid[4], vec;
    load_token_quad(p.logp_pi, p.logp_mu, p.mask, p.T, t0, a, b, valid, vec);
    df32 acc{0.0f, 0.0f};
    long long cnt = 0;
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float d = __fsub_rn(a[i], b[i]);
        w[i] = expf(d);
        if (valid[i]) {
            acc = df_add(acc, d3_term(d));
            ++cnt;
        }
    }
    if (vec && aligned_x4(p.out_w)) {
        *reinterpret_cast<float4*>(p.out_w + t0) = make_float4(w[0], w[1], w[2], w[3]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (t0 + i < p.T) p.out_w[t0 + i] = w[i];
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    if ((threadIdx.x & 31) == 0) wcnt[threadIdx.x >> 5] = cnt;
    stage_warp_sum(acc, 0, bsum);
    __syncthreads();
    const double total = threadIdx.x < 32 ? finish_block_sums(bsum) : 0.0;
    if (threadIdx.x == 0) {
        long long c = 0;
        for (int k = 0; k < kIsThreads / 32; ++k) c += wcnt[k];
        p.blk_sum[blockIdx.x] = total;
        p.blk_cnt[blockIdx.x] = c;
    }
    if (!finished_last(q.done, q.num_blocks, &last)) return;
    // the block's own scratch is free again (finished_last synchronised the block)
    __shared__ double chunk_res[1024];
    const long long n = last_block_count(p.blk_cnt, q.num_blocks, wcnt);
    const double sum = last_block_tree(p.blk_sum, q.num_blocks, chunk_res, wsum);
    if (threadIdx.x == 0) {
        *q.out_d3 = n > 0 ? __ddiv_rn(sum, static_cast<double>(n)) : 0.0;
        if (q.out_nvalid) *q.out_nvalid = n;
        *q.done = 0u;  // ready for the next call (kernels on the stream run in order)
    }
}

// ---------------------------------------------------------------------- REINFORCE Zero
constexpr int kRzFlagTis = 1;        // w_hat = min(w, tis_cap)
constexpr int kRzFlagTokenGate = 2;  // w_hat = 0 unless tok_lo <= d <= tok_hi (fp32 d)
constexpr int kRzFlagSeqGate = 4;    // whole response zeroed unless seq_lo <= sum d <= seq_hi
constexpr int kRzThreads = 256;

struct RzParams {
    const float* logp_pi;
    const float* logp_mu;
    const uint8_t* mask;     // may be null
    int64_t T;
    const int64_t* offs;     // [B + 1]
    int64_t B;
    const float* rewards;    // [B]
    int32_t G;               // group size; B % G == 0
    int32_t flags;
    float tis_cap;
    float tok_lo, tok_hi;
    double seq_lo, seq_hi;
    float* out_w_hat;        // [T] or null
    float* out_grad;         // [T]
    double* out_adv;         // [B] or null
    double* seq_term;        // [B] workspace: A_i * sum_t w_hat / T_i (0 if empty or gated)
    long long* seq_kept;     // [B] workspace: 1 if the response passed the sequence gate
    int* status;
    unsigned* done;          // responses finished; zero at launch, zeroed again by the last block
    double* out_loss;
    int64_t* out_kept;       // may be null
};

// The token weight before the sequence gate: w = e^d (fp32), the token gate decided on the
// fp32 d, then the TIS cap.
__device__ __forceinline__ float rz_token_weight(const RzParams& p, float d) {
    float w = expf(d);
    if ((p.flags & kRzFlagTokenGate) && !(d >= p.tok_lo && d <= p.tok_hi)) w = 0.0f;
    if (p.flags & kRzFlagTis) w = fminf(w, p.tis_cap);
    return w;
}

// One block per response i.  Pass 1 (thread j takes tokens j, j + 256, ... in order, sixteen
// loads in flight): the
// valid-token count, the sequence log-ratio sum d (d exact as a double-float difference of the
// two fp32 inputs) and sum w_hat, each a double-float sum per thread, reduced by the lane
// butterfly and the 8-warp fp64 tree.  Then the gate, A_i = R_i - mean of the group's rewards
// (fp64, in order), and pass 2 writes w_hat and dL/dlog pi = -(A_i / (B T_i)) w_hat per token
// (the coefficient rounded to fp32 once, then one fp32 product).  The last response block to
// finish forms the loss L = -(fixed tree over the response terms) / B and the number of
// responses that passed the sequence gate, as rz_final_kernel does.
static __global__ void __launch_bounds__(kRzThreads, 4) rz_seq_kernel(const RzParams p) {
    static_assert(kRzThreads == kIsThreads, "the last-block finish runs on kIsThreads threads");
    __shared__ BlockSums<2> s_w;
    __shared__ long long s_n[8];
    __shared__ float s_coef;
    __shared__ int s_keep;
    __shared__ int last;
    const int64_t i = blockIdx.x;
    int64_t t_begin = p.offs[i], t_end = p.offs[i + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.T) {
        if (threadIdx.x == 0) atomicOr(p.status, kStatusBadOffsets);
        t_begin = t_end = 0;
    }
    df32 lr{0.0f, 0.0f}, ws{0.0f, 0.0f};
    long long n = 0;
    // sixteen tokens per round: their loads are issued together, then folded in token order
    // (64 registers: four blocks per SM, so all 512 responses of a 2 M-token batch are resident)
    constexpr int kU = 16;
    for (int64_t t0 = t_begin + threadIdx.x; t0 < t_end; t0 += kU * kRzThreads) {
        float a[kU], b[kU];
        bool valid[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t t = t0 + static_cast<int64_t>(u) * kRzThreads;
            valid[u] = t < t_end && (p.mask == nullptr || p.mask[t] != 0);
            a[u] = t < t_end ? p.logp_pi[t] : 0.0f;
            b[u] = t < t_end ? p.logp_mu[t] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (!valid[u]) continue;
            lr = df_add(lr, diff_exact(a[u], b[u]));
            ws = df_add(ws, rz_token_weight(p, __fsub_rn(a[u], b[u])));
            ++n;
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
    if ((threadIdx.x & 31) == 0) s_n[threadIdx.x >> 5] = n;
    stage_warp_sum(lr, 0, s_w);
    stage_warp_sum(ws, 1, s_w);
    __syncthreads();
    const double lr_ws = threadIdx.x < 32 ? finish_block_sums(s_w) : 0.0;
    const double ws_sum = __shfl_sync(0xffffffffu, lr_ws, 8);  // warp 0's lane 8
    // the response's fp64 scalars in thread 0 alone (the fp64 pipe is narrow): the two sums,
    // the gate, the advantage, the response term; the gate and the coefficient are broadcast
    if (threadIdx.x == 0) {
        const double lrd = lr_ws;
        const double wsd = ws_sum;
        long long nt = 0;
        for (int w = 0; w < 8; ++w) nt += s_n[w];
        const bool kp = !(p.flags & kRzFlagSeqGate) || (lrd >= p.seq_lo && lrd <= p.seq_hi);
        const int64_t g0 = (i / p.G) * p.G;
        double gsum = 0.0;
        for (int64_t j = g0; j < g0 + p.G; ++j)
            gsum = __dadd_rn(gsum, static_cast<double>(p.rewards[j]));
        const double A = __dsub_rn(static_cast<double>(p.rewards[i]),
                                   __ddiv_rn(gsum, static_cast<double>(p.G)));
        const double bn = __dmul_rn(static_cast<double>(p.B), static_cast<double>(nt));
        s_coef = (nt > 0 && kp) ? __double2float_rn(__ddiv_rn(-A, bn)) : 0.0f;
        s_keep = kp ? 1 : 0;
        p.seq_term[i] = (nt > 0 && kp) ? __ddiv_rn(__dmul_rn(A, wsd), static_cast<double>(nt)) : 0.0;
        p.seq_kept[i] = kp ? 1 : 0;
        if (p.out_adv) p.out_adv[i] = A;
    }
    __syncthreads();
    const bool keep = s_keep != 0;
    const float coef = s_coef;

    for (int64_t t0 = t_begin + threadIdx.x; t0 < t_end; t0 += kU * kRzThreads) {
        float d[kU];
        bool valid[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t t = t0 + static_cast<int64_t>(u) * kRzThreads;
            valid[u] = keep && t < t_end && (p.mask == nullptr || p.mask[t] != 0);
            d[u] = valid[u] ? __fsub_rn(p.logp_pi[t], p.logp_mu[t]) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t t = t0 + static_cast<int64_t>(u) * kRzThreads;
            if (t >= t_end) break;
            const float wh = valid[u] ? rz_token_weight(p, d[u]) : 0.0f;
            if (p.out_w_hat) p.out_w_hat[t] = wh;
            p.out_grad[t] = valid[u] ? __fmul_rn(coef, wh) : 0.0f;
        }
    }
    if (!finished_last(p.done, static_cast<int>(p.B), &last)) return;
    __shared__ double chunk_res[1024];
    __shared__ double wres[kIsThreads / 32];
    __shared__ long long wkept[kIsThreads / 32];
    const long long kept = last_block_count(p.seq_kept, static_cast<int>(p.B), wkept);
    const double sum = last_block_tree(p.seq_term, static_cast<int>(p.B), chunk_res, wres);
    if (threadIdx.x == 0) {
        *p.out_loss = __ddiv_rn(-sum, static_cast<double>(p.B));
        if (p.out_kept) *p.out_kept = kept;
        *p.done = 0u;
    }
}

// One block of 1024: L = -(fixed tree over the response terms) / B, and the number of
// responses that passed the sequence gate (used for B = 0; rz_seq_kernel finishes B > 0).
static __global__ void __launch_bounds__(1024) rz_final_kernel(const double* seq_term,
                                                        const long long* seq_kept, int B,
                                                        double* out_loss, int64_t* out_kept) {
    __shared__ double a[kIsChunk];
    __shared__ double chunk_res[1024];
    __shared__ long long cnt_part[1024];
    const long long kept = block_count_sum(seq_kept, B, cnt_part);
    const double sum = tree_over_partials(seq_term, B, a, chunk_res);
    if (threadIdx.x == 0) {
        *out_loss = B > 0 ? __ddiv_rn(-sum, static_cast<double>(B)) : 0.0;
        if (out_kept) *out_kept = kept;
    }
}

}  // namespace lp
