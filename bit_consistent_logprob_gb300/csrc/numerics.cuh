// numerics.cuh -- the pinned per-element arithmetic shared by every kernel.
//
// Bit-identity across batch size, row position, prefill/decode and the emulated
// tensor-parallel split holds because every path applies exactly these
// functions, in this order, to exactly the same fp32 values.  Every operation
// is an explicit IEEE binary32 operation (__fadd_rn / __fsub_rn / __fmul_rn /
// __fmaf_rn, fmaxf, and CUDA's __expf / expf / expm1f / logf), so no compiler
// contraction can differ between kernels.
#pragma once

#include <cstdint>

namespace lp {

constexpr int kVT = 128;     // vocabulary tile: MMA N
constexpr int kLT = 64;      // log-sum-exp tile: half a vocabulary tile
constexpr int kBM = 128;     // token rows per tile: MMA M
constexpr int kBK = 64;      // K elements per pipeline stage (128 bytes of bf16)
constexpr int kChunk = 32;   // columns per TMEM load
constexpr int kChunks = kVT / kChunk;
constexpr int kMaxLeaves = 8;

// Sticky device status bits (mapped to lp_status by the host).
constexpr int kStatusBadId = 1;
constexpr int kStatusTimeout = 2;

// Pairwise sum of 32 values, adjacent pairs first, level by level.  Destroys v.
__device__ __forceinline__ float tree_sum32(float (&v)[32]) {
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
#pragma unroll
        for (int i = 0; i < w; ++i) v[i] = __fadd_rn(v[2 * i], v[2 * i + 1]);
    }
    return v[0];
}

// Log-sum-exp partial of one 64-column log-sum-exp tile of one row, defined on its two
// 32-column chunks c = 0, 1 (columns at or beyond `nvalid`, i.e. vocabulary entries >= V,
// are excluded):
//   m_c = max of the chunk's valid logits, taken left to right from -inf
//   m   = max(m_0, m_1)
//   e_i = exp(z_i - m) for valid columns, 0 otherwise
//   s_c = pairwise tree sum of the chunk's 32 e_i (chunk_expsum)
//   s   = s_0 + s_1
// The fused GEMM epilogue (one thread holds a whole 64-column tile of its row) and the
// tensor-parallel kernel apply exactly these operations in this order.
__device__ __forceinline__ float chunk_max(const float (&v)[32], int nvalid) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; ++i)
        if (i < nvalid) m = fmaxf(m, v[i]);
    return m;
}

// Sum of exp(z - m) over the chunk's valid columns (pairwise tree); captures the logit in
// column `ycol` (chunk-relative) into zy.  Destroys v.  The exponential is CUDA's __expf
// intrinsic (argument <= 0 here; a few units in the last place, far inside the logprob
// tolerance), used identically by every kernel that forms a tile partial.
__device__ __forceinline__ float chunk_expsum(float (&v)[32], int nvalid, float m, int ycol,
                                              float& zy) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        if (i == ycol) zy = v[i];
        v[i] = (i < nvalid) ? __expf(__fsub_rn(v[i], m)) : 0.0f;
    }
    return tree_sum32(v);
}

// One 64-column log-sum-exp tile held by one thread (z[0..63]); nvalid counts its valid
// columns (> 0), ycol is the tile-relative column of the sampled token (or outside
// [0, 64)).  Destroys z.
__device__ __forceinline__ float2 tile_lse64(float (&z)[64], int nvalid, int ycol, float& zy) {
    float(&z0)[32] = *reinterpret_cast<float(*)[32]>(&z[0]);
    float(&z1)[32] = *reinterpret_cast<float(*)[32]>(&z[32]);
    const float m = fmaxf(chunk_max(z0, nvalid), chunk_max(z1, nvalid - 32));
    const float s0 = chunk_expsum(z0, nvalid, m, ycol, zy);
    const float s1 = chunk_expsum(z1, nvalid - 32, m, ycol - 32, zy);
    return make_float2(m, __fadd_rn(s0, s1));
}

// Merge two (max, sum-exp) pairs: m = max(m1, m2), s = s1 e^(m1-m) + s2 e^(m2-m).
// Two -inf maxima give (-inf, 0); a NaN propagates through s.
__device__ __forceinline__ float2 lse_merge(float2 a, float2 b) {
    const float m = fmaxf(a.x, b.x);
    if (m == -INFINITY) return make_float2(-INFINITY, 0.0f);
    const float s = __fadd_rn(__fmul_rn(a.y, expf(__fsub_rn(a.x, m))),
                              __fmul_rn(b.y, expf(__fsub_rn(b.x, m))));
    return make_float2(m, s);
}

// logZ of a fully merged pair.
__device__ __forceinline__ float lse_finish(float2 ms) { return __fadd_rn(ms.x, logf(ms.y)); }

// Per-token term of D3, e^d - 1 - d with d = log pi - log mu (w = e^d, log w = d).
// |d| < 1/4: its Taylor series d^2 (1/2! + d/3! + ... + d^7/9!) by Horner's rule
// (the next term is below 1e-11 relative); otherwise expm1f(d) - d, where the
// cancellation is at most ~9x.  Overflows to +inf above d ~ 88.7 (fp32 range).
__device__ __forceinline__ float d3_term(float d) {
    if (fabsf(d) < 0.25f) {
        float p = 1.0f / 362880.0f;                 // 1/9!
        p = __fmaf_rn(p, d, 1.0f / 40320.0f);       // 1/8!
        p = __fmaf_rn(p, d, 1.0f / 5040.0f);        // 1/7!
        p = __fmaf_rn(p, d, 1.0f / 720.0f);         // 1/6!
        p = __fmaf_rn(p, d, 1.0f / 120.0f);         // 1/5!
        p = __fmaf_rn(p, d, 1.0f / 24.0f);          // 1/4!
        p = __fmaf_rn(p, d, 1.0f / 6.0f);           // 1/3!
        p = __fmaf_rn(p, d, 0.5f);                  // 1/2!
        return __fmul_rn(__fmul_rn(d, d), p);
    }
    if (d == INFINITY) return INFINITY;
    return __fsub_rn(expm1f(d), d);
}

}  // namespace lp
