/*
 * oracle.c -- plain, slow, obviously correct CPU oracle (fp64) for the
 * sampled-token logprob path.  TEST INFRASTRUCTURE ONLY: the product path
 * (the CUDA library and its Python binding) never links, loads or calls this
 * file.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or helper with the CUDA sources.
 *
 * What it computes, and the passage each function follows:
 *
 *  - oracle_logits / oracle_logprobs / oracle_log_softmax:
 *      z[t,v] = sum_k X[t,k] * W[v,k] over ALL k in one plain fp64 loop (the
 *      products of two bf16 numbers are exact in fp64), then
 *      logZ = max_v z + log(sum_v exp(z - max)), logp = z[t, y_t] - logZ.
 *      The pages name "the final logprob" as a fused-kernel output (vLLM blog
 *      "Finish RL training faster: bit-consistent, high-throughput,
 *      agent-driven", section 3.1) and define diff over the logprob of every
 *      sampled token (same page, section 2); they print no formula, so this is
 *      the standard log-softmax definition.  The leaf split of K is a rounding
 *      schedule, not a change of the mathematical result, so the exact value
 *      is the plain sum.
 *
 *  - oracle_leaf_sums: the per-leaf sums P_j = sum_{k in leaf j} X[t,k]W[v,k]
 *      for K cut into N contiguous leaves (IsoExec blog summary, section
 *      "Parallelism-invariant kernels"; the contract example pins
 *      leaves = 8, leaf_dtype = fp32).
 *
 *  - oracle_tree_fp32: the fixed binary tree that combines N leaf partials in
 *      fp32: adjacent pairs first, level by level, e.g. for N = 8
 *      ((P0+P1)+(P2+P3))+((P4+P5)+(P6+P7)).  Same IsoExec section ("a fixed
 *      binary arithmetic schedule"); the pairing of adjacent leaves is the
 *      reading taken where the page only says "fixed binary tree".
 *      Compiled with -ffp-contract=off; every add is one IEEE binary32 add.
 *
 *  - oracle_importance_weights: w = pi/mu = exp(log pi - log mu), unclipped
 *      (REINFORCE Zero summary, sections 2 and 4), per-token term
 *      w - 1 - log w (the k3 form r - 1 - log r, vLLM blog section 3.2) and
 *      D3 = mean of the term over valid tokens (REINFORCE Zero summary,
 *      section 3).  log w is taken as exactly d = log pi - log mu, so the term
 *      is expm1(d) - d; it is 0 at w = 1.  No valid token gives D3 = 0.
 *
 *  - oracle_entropy: the entropy of each row's softmax, H = -sum_v p_v log p_v
 *      with log p = z - logZ (the actor entropy the vLLM blog tracks beside the
 *      train-inference KL, section 3.2 results).
 *
 *  - oracle_logprob_grad: the gradient of sum_t g_t logp_t with respect to X
 *      and W, from d logp_t / d z_tv = 1[v = y_t] - p_tv (the standard
 *      log-softmax derivative; the pages' recipe differentiates a training
 *      graph beside the inference forward, vLLM blog section 3.1):
 *        dl[t,v] = g_t (1[v = y_t] - p_tv), dX = dl W, dW = dl^T X.
 *      oracle_logprobs_f64 is the logprob definition on real-valued (fp64)
 *      inputs, used to check the gradient by finite differences.
 *
 *  - oracle_e4m3_encode / oracle_e4m3_decode / oracle_quantize_blocks /
 *    oracle_logprobs_fp8: the block-FP8 (W8A8) variant the vLLM blog keeps for
 *      DeepSeek-V4's deployment (section 4.1), with DeepSeek's block rule:
 *      activation blocks 1 x 128, weight blocks 128 x 128, scale = amax / 448
 *      in fp32 (1 for an all-zero block), q = e4m3(x / s) with x / s an fp32
 *      division, rounded to nearest even and saturated to +-448 (the OCP
 *      E4M3 format: bias 7, 3 mantissa bits, no infinities).  The quantised
 *      bytes are an integer decision, so they are made in the same fp32
 *      arithmetic the GPU uses.  The logits are the plain fp64 dot products
 *      of the dequantised values q * s.  oracle_entropy_fp8 is oracle_entropy
 *      over those logits.
 *
 *  - oracle_acceptance_stats: over the valid tokens, the max, mean and
 *      population standard deviation of |a - b| between two logprob vectors,
 *      and the k3 KL estimate mean(r - 1 - log r) with r = exp(a - b) (vLLM
 *      blog section 2: acceptance asks the max, mean and std of the per-token
 *      difference to be 0 over every valid sampled token; section 3.2: the k3
 *      estimator).  a is the learner's logprob, b the rollout's, so r = pi/mu
 *      and k3 is the same per-token term as D3.  A NaN difference on a valid
 *      token makes every statistic NaN; no valid token gives all zeros.
 *
 *  - oracle_reinforce_zero: the REINFORCE Zero loss (REINFORCE Zero summary,
 *      section 4) for B responses packed back to back,
 *        L = -(1/B) sum_i (1/T_i) sum_t A_i * w_it,
 *      A_i = R_i - mean of R over the response's group (groups of G
 *      consecutive responses), T_i = valid tokens of response i, w = pi/mu
 *      unclipped at token level, and dL/dlog pi_it = -(1/B)(1/T_i) A_i w_it.
 *      Options from the corrections the pages list beside it (vLLM blog
 *      section 1; REINFORCE Zero summary, results table): TIS truncates
 *      the weight at a cap, w_hat = min(w, C); a token gate zeroes tokens
 *      whose d = log pi - log mu (rounded to fp32, the precision the gate is
 *      decided in) lies outside [lo, hi]; a sequence gate (MIS) zeroes every
 *      token of a response whose sequence log-ratio sum_t d_t lies outside
 *      [lo, hi].  With any option the modified weight multiplies grad log pi
 *      (it is held constant under differentiation), so the gradient is
 *      -(1/B)(1/T_i) A_i w_hat_it and L uses w_hat in place of w.  Masked
 *      tokens get w_hat = 0 and gradient 0; a response with T_i = 0 adds 0.
 *
 * Every function is single-threaded per output element; rows are spread over
 * OpenMP threads, which changes no result (each row is computed alone).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> exact double (bf16 is the top half of a binary32). */
static double bf16_to_f64(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One logit: plain fp64 dot product of row t of X with row v of W. */
static double logit_f64(const uint16_t* xrow, const uint16_t* wrow, int64_t H) {
    double acc = 0.0;
    for (int64_t k = 0; k < H; ++k) acc += bf16_to_f64(xrow[k]) * bf16_to_f64(wrow[k]);
    return acc;
}

/* z[r, v] for the rows listed in `rows` (nrows of them); z is [nrows, V]. */
void oracle_logits(const uint16_t* X, int64_t ldx, const uint16_t* W, int64_t H, int64_t V,
                   const int64_t* rows, int64_t nrows, double* z) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        const uint16_t* xrow = X + rows[r] * ldx;
        for (int64_t v = 0; v < V; ++v) z[r * V + v] = logit_f64(xrow, W + v * H, H);
    }
}

/* log of the partition function of one row of logits: max + log sum exp(z - max). */
static double log_partition(const double* z, int64_t V) {
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v)
        if (z[v] > m || isnan(z[v])) m = z[v];
    if (isnan(m)) return NAN;
    if (isinf(m) && m < 0) return -INFINITY;
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) s += exp(z[v] - m);
    return m + log(s);
}

/*
 * Sampled-token logprob for the listed rows.  ids is indexed by the row number
 * (ids[rows[r]]); an id outside [0, V) gives NaN.  logp, logZ are [nrows].
 */
void oracle_logprobs(const uint16_t* X, int64_t ldx, const uint16_t* W, const int32_t* ids,
                     int64_t H, int64_t V, const int64_t* rows, int64_t nrows, double* logp,
                     double* logZ) {
#pragma omp parallel
    {
        double* z = (double*)malloc((size_t)V * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            const uint16_t* xrow = X + rows[r] * ldx;
            int32_t y = ids[rows[r]];
            for (int64_t v = 0; v < V; ++v) z[v] = logit_f64(xrow, W + v * H, H);
            double lz = log_partition(z, V);
            logZ[r] = lz;
            logp[r] = (y >= 0 && (int64_t)y < V) ? z[y] - lz : NAN;
        }
        free(z);
    }
}

/* Full log-softmax of the listed rows: out[r, v] = z[r,v] - logZ[r]. */
void oracle_log_softmax(const uint16_t* X, int64_t ldx, const uint16_t* W, int64_t H, int64_t V,
                        const int64_t* rows, int64_t nrows, double* out) {
    oracle_logits(X, ldx, W, H, V, rows, nrows, out);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        double lz = log_partition(out + r * V, V);
        for (int64_t v = 0; v < V; ++v) out[r * V + v] -= lz;
    }
}

/*
 * Leaf sums for one (row t, vocab v): leaf j covers k in [j*H/N, (j+1)*H/N).
 * out is [N].  Requires H % N == 0.
 */
void oracle_leaf_sums(const uint16_t* xrow, const uint16_t* wrow, int64_t H, int32_t N,
                      double* out) {
    int64_t L = H / N;
    for (int32_t j = 0; j < N; ++j) {
        double acc = 0.0;
        for (int64_t k = (int64_t)j * L; k < (int64_t)(j + 1) * L; ++k)
            acc += bf16_to_f64(xrow[k]) * bf16_to_f64(wrow[k]);
        out[j] = acc;
    }
}

/*
 * Fixed binary tree over N fp32 partials (N a power of two, N <= 64):
 * level by level, node i of the next level = node 2i + node 2i+1.
 * Returns NaN bits for an unsupported N.
 */
float oracle_tree_fp32(const float* P, int32_t N) {
    float buf[64];
    if (N < 1 || N > 64 || (N & (N - 1)) != 0) return NAN;
    for (int32_t i = 0; i < N; ++i) buf[i] = P[i];
    for (int32_t n = N; n > 1; n /= 2) {
        for (int32_t i = 0; i < n / 2; ++i) {
            volatile float a = buf[2 * i], b = buf[2 * i + 1];
            buf[i] = a + b; /* one binary32 add, round to nearest even */
        }
    }
    return buf[0];
}

/* Apply oracle_tree_fp32 to `count` independent groups of N partials: P is [count, N]. */
void oracle_tree_fp32_many(const float* P, int32_t N, int64_t count, float* out) {
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_tree_fp32(P + i * N, N);
}

/*
 * Importance weights and D3.  mask may be NULL (all tokens valid); a token is
 * valid when mask[t] != 0.  w and term are written for every token (term of an
 * invalid token is still computed but not counted).  d3 = sum(term over valid)
 * / n_valid, or 0 when n_valid == 0.
 */
void oracle_importance_weights(const float* logp_pi, const float* logp_mu, const uint8_t* mask,
                               int64_t T, double* w, double* term, double* d3,
                               int64_t* n_valid) {
    double sum = 0.0;
    int64_t n = 0;
    for (int64_t t = 0; t < T; ++t) {
        double d = (double)logp_pi[t] - (double)logp_mu[t];
        w[t] = exp(d);
        term[t] = expm1(d) - d;
        if (mask == NULL || mask[t] != 0) {
            sum += term[t];
            ++n;
        }
    }
    *n_valid = n;
    *d3 = n > 0 ? sum / (double)n : 0.0;
}

/* Max, mean, population std of |a-b| and mean of expm1(d) - d over valid tokens. */
void oracle_acceptance_stats(const float* a, const float* b, const uint8_t* mask, int64_t T,
                             double* out /* [5]: max, mean, std, k3, n_valid */) {
    int64_t n = 0;
    double mx = 0.0, sum = 0.0, k3 = 0.0;
    int any_nan = 0;
    for (int64_t t = 0; t < T; ++t) {
        if (mask != NULL && mask[t] == 0) continue;
        double d = (double)a[t] - (double)b[t];
        double x = fabs(d);
        if (isnan(x)) any_nan = 1;
        else if (x > mx) mx = x;
        sum += x;
        k3 += expm1(d) - d;
        ++n;
    }
    if (n == 0) {
        for (int i = 0; i < 5; ++i) out[i] = 0.0;
        return;
    }
    double mean = sum / (double)n;
    double ss = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        if (mask != NULL && mask[t] == 0) continue;
        double x = fabs((double)a[t] - (double)b[t]);
        ss += (x - mean) * (x - mean);
    }
    out[0] = any_nan ? NAN : mx;
    out[1] = mean;
    out[2] = sqrt(ss / (double)n);
    out[3] = k3 / (double)n;
    out[4] = (double)n;
}

enum { ORC_TIS = 1, ORC_TOKEN_GATE = 2, ORC_SEQ_GATE = 4 };

/* REINFORCE Zero loss with optional TIS / token gate / sequence gate.
 * offs[B+1]: response i holds tokens [offs[i], offs[i+1]). */
void oracle_reinforce_zero(const float* logp_pi, const float* logp_mu, const uint8_t* mask,
                           const int64_t* offs, int64_t B, const float* rewards, int G,
                           int flags, double tis_cap, float tok_lo, float tok_hi,
                           double seq_lo, double seq_hi,
                           double* w_hat, double* grad, double* adv, double* seq_logratio,
                           int32_t* kept, double* loss) {
    double total = 0.0;
    for (int64_t i = 0; i < B; ++i) {
        /* advantage: reward minus the mean reward of the response's group */
        int64_t g0 = (i / G) * G;
        double gsum = 0.0;
        for (int64_t j = g0; j < g0 + G; ++j) gsum += (double)rewards[j];
        double A = (double)rewards[i] - gsum / (double)G;
        adv[i] = A;

        int64_t n = 0;
        double lr = 0.0;
        for (int64_t t = offs[i]; t < offs[i + 1]; ++t) {
            if (mask != NULL && mask[t] == 0) continue;
            lr += (double)logp_pi[t] - (double)logp_mu[t];
            ++n;
        }
        seq_logratio[i] = lr;
        int keep = !(flags & ORC_SEQ_GATE) || (lr >= seq_lo && lr <= seq_hi);
        kept[i] = keep;

        double wsum = 0.0;
        for (int64_t t = offs[i]; t < offs[i + 1]; ++t) {
            int valid = mask == NULL || mask[t] != 0;
            double d = (double)logp_pi[t] - (double)logp_mu[t];
            double wh = exp(d);
            if (flags & ORC_TOKEN_GATE) {
                float d32 = (float)d;
                if (!(d32 >= tok_lo && d32 <= tok_hi)) wh = 0.0;
            }
            if ((flags & ORC_TIS) && wh > tis_cap) wh = tis_cap;
            if (!valid || !keep) wh = 0.0;
            w_hat[t] = wh;
            wsum += wh;
        }
        double coef = n > 0 ? -A / ((double)B * (double)n) : 0.0;
        for (int64_t t = offs[i]; t < offs[i + 1]; ++t) grad[t] = coef * w_hat[t];
        if (n > 0) total += A * wsum / (double)n;
    }
    *loss = B > 0 ? -total / (double)B : 0.0;
}

/* Entropy of the softmax of the listed rows: out[r] = -sum_v p log p, log p = z - logZ. */
void oracle_entropy(const uint16_t* X, int64_t ldx, const uint16_t* W, int64_t H, int64_t V,
                    const int64_t* rows, int64_t nrows, double* out) {
#pragma omp parallel
    {
        double* z = (double*)malloc((size_t)V * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            const uint16_t* xrow = X + rows[r] * ldx;
            for (int64_t v = 0; v < V; ++v) z[v] = logit_f64(xrow, W + v * H, H);
            double lz = log_partition(z, V);
            double h = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                double lp = z[v] - lz;
                double p = exp(lp);
                if (p > 0.0) h -= p * lp;
            }
            out[r] = h;
        }
        free(z);
    }
}

/* Sampled-token logprobs of fp64 inputs X [T, H], W [V, H] (plain definition). */
void oracle_logprobs_f64(const double* X, const double* W, const int32_t* ids, int64_t T,
                         int64_t H, int64_t V, double* logp) {
    double* z = (double*)malloc((size_t)V * sizeof(double));
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t v = 0; v < V; ++v) {
            double acc = 0.0;
            for (int64_t k = 0; k < H; ++k) acc += X[t * H + k] * W[v * H + k];
            z[v] = acc;
        }
        double lz = log_partition(z, V);
        int32_t y = ids[t];
        logp[t] = (y >= 0 && (int64_t)y < V) ? z[y] - lz : NAN;
    }
    free(z);
}

/* Gradient of L = sum_t g_t logp_t: dX [T, H] and dW [V, H] (fp64; X, W bf16 bits). */
void oracle_logprob_grad(const uint16_t* X, const uint16_t* W, const int32_t* ids,
                         const double* g, int64_t T, int64_t H, int64_t V, double* dX,
                         double* dW, double* dl /* [T, V] */) {
#pragma omp parallel
    {
        double* z = (double*)malloc((size_t)V * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t v = 0; v < V; ++v) z[v] = logit_f64(X + t * H, W + v * H, H);
            double lz = log_partition(z, V);
            for (int64_t v = 0; v < V; ++v) {
                double onehot = (v == (int64_t)ids[t]) ? 1.0 : 0.0;
                dl[t * V + v] = g[t] * (onehot - exp(z[v] - lz));
            }
            for (int64_t k = 0; k < H; ++k) {
                double acc = 0.0;
                for (int64_t v = 0; v < V; ++v) acc += dl[t * V + v] * bf16_to_f64(W[v * H + k]);
                dX[t * H + k] = acc;
            }
        }
        free(z);
    }
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t v = 0; v < V; ++v) {
        for (int64_t k = 0; k < H; ++k) {
            double acc = 0.0;
            for (int64_t t = 0; t < T; ++t) acc += dl[t * V + v] * bf16_to_f64(X[t * H + k]);
            dW[v * H + k] = acc;
        }
    }
}

/* OCP E4M3 (finite-only variant): value of one code. */
double oracle_e4m3_decode(uint8_t c) {
    int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -v : v;
}

/* Nearest E4M3 code to x (ties to even mantissa), saturating to +-448; NaN -> 0x7F. */
uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sgn = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0) return sgn | 0x7E;
    if (a < ldexp(1.0, -6)) {                    /* subnormal spacing 2^-9; k = 8 is 2^-6 */
        double k = nearbyint(a / ldexp(1.0, -9));
        return sgn | (uint8_t)k;
    }
    int E;
    frexp(a, &E);                                /* a = f 2^E, f in [0.5, 1) */
    int e = E - 1;                               /* a in [2^e, 2^(e+1)) */
    double m = nearbyint((a / ldexp(1.0, e) - 1.0) * 8.0);
    if (m == 8.0) {
        m = 0.0;
        e += 1;
    }
    int code = ((e + 7) << 3) | (int)m;
    if (code > 0x7E) code = 0x7E;
    return sgn | (uint8_t)code;
}

/* Block quantisation of a bf16 matrix [rows, cols] (row stride ld): blocks of block_rows x 128,
 * scales [ceil(rows / block_rows)][cols / 128]. */
void oracle_quantize_blocks(const uint16_t* src, int64_t rows, int64_t cols, int64_t ld,
                            int64_t block_rows, uint8_t* q, float* scales) {
    int64_t nkb = cols / 128, nrb = (rows + block_rows - 1) / block_rows;
    for (int64_t rb = 0; rb < nrb; ++rb) {
        for (int64_t kb = 0; kb < nkb; ++kb) {
            int64_t r0 = rb * block_rows, r1 = r0 + block_rows < rows ? r0 + block_rows : rows;
            float amax = 0.0f;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) {
                    float v = fabsf((float)bf16_to_f64(src[r * ld + k]));
                    if (v > amax) amax = v;
                }
            float s = amax > 0.0f ? amax / 448.0f : 1.0f;
            scales[rb * nkb + kb] = s;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
                    q[r * cols + k] = oracle_e4m3_encode((float)bf16_to_f64(src[r * ld + k]) / s);
        }
    }
}

/* Sampled-token logprobs from quantised operands: z = sum_k (qx sx)(qw sw) in fp64. */
void oracle_logprobs_fp8(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                         const int32_t* ids, int64_t H, int64_t V, const int64_t* rows,
                         int64_t nrows, double* logp, double* logZ) {
    int64_t nkb = H / 128;
#pragma omp parallel
    {
        double* z = (double*)malloc((size_t)V * sizeof(double));
        double* xd = (double*)malloc((size_t)H * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t t = rows[r];
            for (int64_t k = 0; k < H; ++k)
                xd[k] = oracle_e4m3_decode(xq[t * H + k]) * (double)sx[t * nkb + k / 128];
            for (int64_t v = 0; v < V; ++v) {
                double acc = 0.0;
                for (int64_t k = 0; k < H; ++k)
                    acc += xd[k] * (oracle_e4m3_decode(wq[v * H + k]) *
                                    (double)sw[(v / 128) * nkb + k / 128]);
                z[v] = acc;
            }
            double lz = log_partition(z, V);
            int32_t y = ids[t];
            logZ[r] = lz;
            logp[r] = (y >= 0 && (int64_t)y < V) ? z[y] - lz : NAN;
        }
        free(xd);
        free(z);
    }
}

/* Softmax entropy -sum_v p log p of the listed rows, over logits from the dequantised
 * block-FP8 operands: z[v] = sum_k (qx[k] sx) (qw[v][k] sw), all in fp64. */
void oracle_entropy_fp8(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                        int64_t H, int64_t V, const int64_t* rows, int64_t nrows, double* out) {
    int64_t nkb = H / 128;
#pragma omp parallel
    {
        double* z = (double*)malloc((size_t)V * sizeof(double));
        double* xd = (double*)malloc((size_t)H * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t t = rows[r];
            const float* sxrow = sx + t * nkb;
            for (int64_t k = 0; k < H; ++k)
                xd[k] = oracle_e4m3_decode(xq[t * H + k]) * (double)sxrow[k / 128];
            for (int64_t v = 0; v < V; ++v) {
                const uint8_t* wrow = wq + v * H;
                const float* swrow = sw + (v / 128) * nkb;
                double acc = 0.0;
                for (int64_t k = 0; k < H; ++k)
                    acc += xd[k] * (oracle_e4m3_decode(wrow[k]) * (double)swrow[k / 128]);
                z[v] = acc;
            }
            const double lz = log_partition(z, V);
            double h = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                const double lpv = z[v] - lz;
                const double pv = exp(lpv);
                if (pv > 0.0) h -= pv * lpv;
            }
            out[r] = h;
        }
        free(xd);
        free(z);
    }
}
