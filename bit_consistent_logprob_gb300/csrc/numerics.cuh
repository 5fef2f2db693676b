// numerics.cuh -- the pinned per-element arithmetic shared by every kernel.
//
// Bit-identity across batch size, row position, prefill/decode and the emulated
// tensor-parallel split holds because every path applies exactly these
// functions, in this order, to exactly the same fp32 values.  Every operation
// is an explicit IEEE binary32 operation (__fadd_rn / __fsub_rn / __fmul_rn /
// __fmaf_rn and the two-lane __fadd2_rn, fmaxf, and CUDA's __expf / expf / expm1f /
// logf), so no compiler contraction can differ between kernels.
#pragma once

#include <cuda_bf16.h>

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

// Element-wise r[i] = a[i] + r[i] over n (even) consecutive values, two lanes per
// instruction.  Each lane of __fadd2_rn is one IEEE binary32 round-to-nearest addition, so
// every element gets exactly the bits of __fadd_rn; the pairing only halves the additions
// issued (the leaf-tree adds of the bf16 epilogue).
template <int n>
__device__ __forceinline__ void add_rn_x2(float* r, const float* a) {
    static_assert(n % 2 == 0, "pairs of elements");
#pragma unroll
    for (int i = 0; i < n; i += 2) {
        const float2 t = __fadd2_rn(make_float2(a[i], a[i + 1]), make_float2(r[i], r[i + 1]));
        r[i] = t.x;
        r[i + 1] = t.y;
    }
}

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

// Entropy variant of tile_lse64: the same m and s (bit-equal: the same operations in the
// same order), and u = sum over valid columns of e_i * (z_i - m), e_i = exp(z_i - m), as a
// pairwise tree over each chunk's 32 products (level 0 formed pairwise on the fly), then
// u = u_0 + u_1.  The row entropy is log s - u / s once the tiles are merged.
__device__ __forceinline__ float chunk_expsum_ent(float (&v)[32], int nvalid, float m, int ycol,
                                                  float& zy, float& u) {
    float w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float t[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int c = 2 * i + k;
            if (c == ycol) zy = v[c];
            const float d = __fsub_rn(v[c], m);
            const float e = (c < nvalid) ? __expf(d) : 0.0f;
            t[k] = (c < nvalid) ? __fmul_rn(e, d) : 0.0f;
            v[c] = e;
        }
        w[i] = __fadd_rn(t[0], t[1]);
    }
#pragma unroll
    for (int l = 8; l >= 1; l >>= 1) {
#pragma unroll
        for (int i = 0; i < l; ++i) w[i] = __fadd_rn(w[2 * i], w[2 * i + 1]);
    }
    u = w[0];
    return tree_sum32(v);
}

__device__ __forceinline__ float2 tile_lse64_ent(float (&z)[64], int nvalid, int ycol, float& zy,
                                                 float& u) {
    float(&z0)[32] = *reinterpret_cast<float(*)[32]>(&z[0]);
    float(&z1)[32] = *reinterpret_cast<float(*)[32]>(&z[32]);
    const float m = fmaxf(chunk_max(z0, nvalid), chunk_max(z1, nvalid - 32));
    float u0, u1;
    const float s0 = chunk_expsum_ent(z0, nvalid, m, ycol, zy, u0);
    const float s1 = chunk_expsum_ent(z1, nvalid - 32, m, ycol - 32, zy, u1);
    u = __fadd_rn(u0, u1);
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

// Entropy-carrying merge of (m, s, u) triples: m and s exactly as lse_merge, and
// u = (u1 + (m1 - m) s1) e^(m1-m) + (u2 + (m2 - m) s2) e^(m2-m), the sum of e^(z-m)(z-m)
// rebased to the common maximum.
__device__ __forceinline__ float3 lse_merge_ent(float3 a, float3 b) {
    const float m = fmaxf(a.x, b.x);
    if (m == -INFINITY) return make_float3(-INFINITY, 0.0f, 0.0f);
    const float da = __fsub_rn(a.x, m), db = __fsub_rn(b.x, m);
    const float ea = expf(da), eb = expf(db);
    const float s = __fadd_rn(__fmul_rn(a.y, ea), __fmul_rn(b.y, eb));
    const float ua = __fmul_rn(__fadd_rn(a.z, __fmul_rn(da, a.y)), ea);
    const float ub = __fmul_rn(__fadd_rn(b.z, __fmul_rn(db, b.y)), eb);
    return make_float3(m, s, __fadd_rn(ua, ub));
}

// Row entropy from the fully merged triple: log s - u / s.
__device__ __forceinline__ float entropy_finish(float3 msu) {
    return __fsub_rn(logf(msu.y), __fdiv_rn(msu.z, msu.y));
}

// Double-float sums: a value hi + lo held as two non-overlapping fp32 numbers (about 48
// significant bits), added with error-free transformations (Knuth's two-sum) on the fp32
// pipes.  The GB300's fp64 rate is a small fraction of its fp32 rate, so per-token sums run in
// double-float and only the few per-warp results are widened to fp64 (exactly: hi + lo fits
// in a double).  Every operation is an explicit IEEE fp32 operation, so the result is the
// same on every launch.
struct df32 {
    float hi, lo;
};

__device__ __forceinline__ df32 two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

__device__ __forceinline__ df32 df_add(df32 x, df32 y) {
    const df32 s = two_sum(x.hi, y.hi);
    const float lo = __fadd_rn(__fadd_rn(x.lo, y.lo), s.lo);
    return two_sum(s.hi, lo);
}

__device__ __forceinline__ df32 df_add(df32 x, float v) { return df_add(x, df32{v, 0.0f}); }

// x * x exactly, as a double-float (the rounding error of the product by an fma).
__device__ __forceinline__ df32 square_exact(float x) {
    const float p = __fmul_rn(x, x);
    return {p, __fmaf_rn(x, x, -p)};
}

// a - b exactly, as a double-float.
__device__ __forceinline__ df32 diff_exact(float a, float b) { return two_sum(a, -b); }

__device__ __forceinline__ double df_to_f64(df32 x) {
    return __dadd_rn(static_cast<double>(x.hi), static_cast<double>(x.lo));
}

// Lane butterfly over a warp (xor 16, 8, ..., 1); every lane ends with the same sum.
__device__ __forceinline__ df32 warp_sum_df(df32 v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const df32 o{__shfl_xor_sync(0xffffffffu, v.hi, off), __shfl_xor_sync(0xffffffffu, v.lo, off)};
        // the lower lane adds (own, other), the upper (other, own): same operands in the same
        // order on both lanes, so they stay equal
        const bool low = (threadIdx.x & off) == 0;
        v = low ? df_add(v, o) : df_add(o, v);
    }
    return v;
}

// Two fp32 values rounded to bf16 (nearest even), packed low then high.// Two fp32 values rounded to bf16 (nearest even), packed low then high.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
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
