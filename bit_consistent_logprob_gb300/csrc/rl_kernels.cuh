// Epilogues of the RL step that consume per-token logprobs.
//
//  stats_block_kernel /
//  stats_final_kernel   acceptance statistics between two logprob vectors: max, mean and
//                       population std of |a - b| and the k3 estimate mean(r - 1 - log r),
//                       r = e^(a - b), over valid tokens (vLLM blog "Finish RL training
//                       faster", section 2: acceptance asks max, mean and std of the
//                       per-token difference to be 0; section 3.2: the k3 estimator).
//  rz_seq_kernel /
//  rz_final_kernel      the REINFORCE Zero loss L = -(1/B) sum_i (1/T_i) sum_t A_i w_it with
//                       group-mean advantages, its gradient with respect to log pi, and the
//                       TIS / token-gate / sequence-gate options (REINFORCE Zero summary,
//                       section 4 and results table; vLLM blog, section 1).
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

// Per block of 1024 tokens (4 per thread, in order): three double-float sums reduced exactly
// like the D3 block sum (is_block_kernel), so the k3 partials are bit-equal to the D3 partials
// of the same tokens; |d|^2 enters exactly (an fma recovers the product's rounding error);
// max and count are exact in any order.
static __global__ void __launch_bounds__(kIsThreads) stats_block_kernel(const StatsParams p) {
    __shared__ double s_w[8];
    __shared__ float s_max[8];
    __shared__ long long s_cnt[8];
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kIsBlock + threadIdx.x * 4;
    df32 acc_abs{0.0f, 0.0f}, acc_sq{0.0f, 0.0f}, acc_k3{0.0f, 0.0f};
    float mx = 0.0f;
    long long cnt = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t t = t0 + i;
        if (t < p.T && (p.mask == nullptr || p.mask[t] != 0)) {
            const float d = __fsub_rn(p.a[t], p.b[t]);
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
    const double sum_abs = block_sum_8warps(acc_abs, s_w);
    __syncthreads();
    const double sum_sq = block_sum_8warps(acc_sq, s_w);
    __syncthreads();
    const double sum_k3 = block_sum_8warps(acc_k3, s_w);
    if (threadIdx.x == 0) {
        p.blk_abs[blockIdx.x] = sum_abs;
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
    if (threadIdx.x == 0) {
        if (n == 0) {
            for (int i = 0; i < 5; ++i) out[i] = 0.0;
        } else {
            const double nd = static_cast<double>(n);
            const double mean = __ddiv_rn(s_abs, nd);
            const double var = __dsub_rn(__ddiv_rn(s_sq, nd), __dmul_rn(mean, mean));
            out[0] = static_cast<double>(max_part[0]);
            out[1] = mean;
            out[2] = var > 0.0 ? __dsqrt_rn(var) : (var == var ? 0.0 : var);
            out[3] = __ddiv_rn(s_k3, nd);
            out[4] = nd;
        }
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
};

// The token weight before the sequence gate: w = e^d (fp32), the token gate decided on the
// fp32 d, then the TIS cap.
__device__ __forceinline__ float rz_token_weight(const RzParams& p, float d) {
    float w = expf(d);
    if ((p.flags & kRzFlagTokenGate) && !(d >= p.tok_lo && d <= p.tok_hi)) w = 0.0f;
    if (p.flags & kRzFlagTis) w = fminf(w, p.tis_cap);
    return w;
}

// One block per response i.  Pass 1 (thread j takes tokens j, j + 256, ... in order, four
// loads in flight): the
// valid-token count, the sequence log-ratio sum d (d exact as a double-float difference of the
// two fp32 inputs) and sum w_hat, each a double-float sum per thread, reduced by the lane
// butterfly and the 8-warp fp64 tree.  Then the gate, A_i = R_i - mean of the group's rewards
// (fp64, in order), and pass 2 writes w_hat and dL/dlog pi = -(A_i / (B T_i)) w_hat per token
// (the coefficient rounded to fp32 once, then one fp32 product).
static __global__ void __launch_bounds__(kRzThreads) rz_seq_kernel(const RzParams p) {
    __shared__ double s_w[8];
    __shared__ long long s_n[8];
    const int64_t i = blockIdx.x;
    int64_t t_begin = p.offs[i], t_end = p.offs[i + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.T) {
        if (threadIdx.x == 0) atomicOr(p.status, kStatusBadOffsets);
        t_begin = t_end = 0;
    }
    df32 lr{0.0f, 0.0f}, ws{0.0f, 0.0f};
    long long n = 0;
    // four tokens per round: their loads are issued together, then folded in token order
    constexpr int kU = 4;
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
    const double lrd = block_sum_8warps(lr, s_w);
    __syncthreads();
    const double wsd = block_sum_8warps(ws, s_w);
    n = 0;
    for (int w = 0; w < 8; ++w) n += s_n[w];
    const bool keep = !(p.flags & kRzFlagSeqGate) || (lrd >= p.seq_lo && lrd <= p.seq_hi);

    const int64_t g0 = (i / p.G) * p.G;
    double gsum = 0.0;
    for (int64_t j = g0; j < g0 + p.G; ++j) gsum = __dadd_rn(gsum, static_cast<double>(p.rewards[j]));
    const double A = __dsub_rn(static_cast<double>(p.rewards[i]),
                               __ddiv_rn(gsum, static_cast<double>(p.G)));
    const double bn = __dmul_rn(static_cast<double>(p.B), static_cast<double>(n));
    const float coef = (n > 0 && keep) ? __double2float_rn(__ddiv_rn(-A, bn)) : 0.0f;

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
    if (threadIdx.x == 0) {
        p.seq_term[i] = (n > 0 && keep) ? __ddiv_rn(__dmul_rn(A, wsd), static_cast<double>(n)) : 0.0;
        p.seq_kept[i] = keep ? 1 : 0;
        if (p.out_adv) p.out_adv[i] = A;
    }
}

// One block of 1024: L = -(fixed tree over the response terms) / B, and the number of
// responses that passed the sequence gate.
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
