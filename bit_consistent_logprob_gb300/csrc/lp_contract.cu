// lp_contract.cu -- the execution contract of a configuration and its SHA-256 identities.
//
// The contract names every execution choice that can change a bit of the result, so that a
// trainer and a rollout engine can prove they run the same numerics by comparing digests
// (IsoExec, SkyRL blog summary, "unified execution contract": cases, composition of
// (region, case) -> implementation + pinned constants, claims, and identities that are
// SHA-256 digests of the serialised contract: semantic, numerical_policy, deployment).
// Here:
//   semantic          the logical computation: op, lm_head shape, outputs.
//   numerical_policy  cases, composition (implementations, versions, pinned constants) and
//                     claims (proven parallel sizes and phases, tolerances).
//   deployment        settings proven not to change bits (row chunk, scheduling band).
// The serialisation is canonical: fixed key order, no whitespace, integers in decimal.
// Host code only; SHA-256 follows FIPS 180-4, its round constants and initial hash values
// derived exactly (integer cube and square roots of the first primes).

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>

#include "lp.h"
#include "lp_internal.h"

namespace {

// ------------------------------------------------------------------------------- SHA-256
// floor(r * 2^32) mod 2^32 for r = the cube root (k = 3) or square root (k = 2) of p:
// the largest x with x^k <= p * 2^(32k), found by bisection on 128-bit integers.
uint32_t root_bits(unsigned p, int k) {
    using u128 = unsigned __int128;
    const u128 target = static_cast<u128>(p) << (32 * k);
    uint64_t lo = 0, hi = uint64_t(1) << (k == 3 ? 36 : 40);  // root * 2^32 < 2^36 (p < 2^12)
    while (hi - lo > 1) {
        const uint64_t mid = lo + (hi - lo) / 2;
        u128 v = static_cast<u128>(mid) * mid;
        if (k == 3) v *= mid;
        if (v <= target) lo = mid;
        else hi = mid;
    }
    return static_cast<uint32_t>(lo);
}

struct Sha256Tables {
    uint32_t k[64];
    uint32_t h0[8];
    Sha256Tables() {
        unsigned primes[64];
        int n = 0;
        for (unsigned c = 2; n < 64; ++c) {
            bool prime = true;
            for (unsigned d = 2; d * d <= c; ++d)
                if (c % d == 0) {
                    prime = false;
                    break;
                }
            if (prime) primes[n++] = c;
        }
        for (int i = 0; i < 64; ++i) k[i] = root_bits(primes[i], 3);
        for (int i = 0; i < 8; ++i) h0[i] = root_bits(primes[i], 2);
    }
};

const Sha256Tables& tables() {
    static const Sha256Tables t;
    return t;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

void sha256_block(uint32_t h[8], const uint8_t* blk) {
    const Sha256Tables& t = tables();
    uint32_t w[64];
    for (int i = 0; i < 16; ++i)
        w[i] = (uint32_t(blk[4 * i]) << 24) | (uint32_t(blk[4 * i + 1]) << 16) |
               (uint32_t(blk[4 * i + 2]) << 8) | uint32_t(blk[4 * i + 3]);
    for (int i = 16; i < 64; ++i) {
        const uint32_t s0 = rotr(w[i - 15], 7) ^ rotr(w[i - 15], 18) ^ (w[i - 15] >> 3);
        const uint32_t s1 = rotr(w[i - 2], 17) ^ rotr(w[i - 2], 19) ^ (w[i - 2] >> 10);
        w[i] = w[i - 16] + s0 + w[i - 7] + s1;
    }
    uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
    for (int i = 0; i < 64; ++i) {
        const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
        const uint32_t ch = (e & f) ^ (~e & g);
        const uint32_t t1 = hh + S1 + ch + t.k[i] + w[i];
        const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
        const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
        const uint32_t t2 = S0 + maj;
        hh = g;
        g = f;
        f = e;
        e = d + t1;
        d = c;
        c = b;
        b = a;
        a = t1 + t2;
    }
    h[0] += a; h[1] += b; h[2] += c; h[3] += d;
    h[4] += e; h[5] += f; h[6] += g; h[7] += hh;
}

void sha256(const void* data, size_t n, uint8_t out[32]) {
    uint32_t h[8];
    std::memcpy(h, tables().h0, sizeof h);
    const uint8_t* p = static_cast<const uint8_t*>(data);
    size_t off = 0;
    for (; off + 64 <= n; off += 64) sha256_block(h, p + off);
    uint8_t tail[128] = {0};
    const size_t rem = n - off;
    if (rem) std::memcpy(tail, p + off, rem);
    tail[rem] = 0x80;
    const size_t tl = rem + 9 <= 64 ? 64 : 128;
    const uint64_t bits = static_cast<uint64_t>(n) * 8;
    for (int i = 0; i < 8; ++i) tail[tl - 1 - i] = static_cast<uint8_t>(bits >> (8 * i));
    for (size_t o = 0; o < tl; o += 64) sha256_block(h, tail + o);
    for (int i = 0; i < 8; ++i) {
        out[4 * i] = static_cast<uint8_t>(h[i] >> 24);
        out[4 * i + 1] = static_cast<uint8_t>(h[i] >> 16);
        out[4 * i + 2] = static_cast<uint8_t>(h[i] >> 8);
        out[4 * i + 3] = static_cast<uint8_t>(h[i]);
    }
}

std::string hex(const uint8_t d[32]) {
    static const char* digits = "0123456789abcdef";
    std::string s;
    for (int i = 0; i < 32; ++i) {
        s += digits[d[i] >> 4];
        s += digits[d[i] & 15];
    }
    return s;
}

// ------------------------------------------------------------------------------- contract
std::string semantic_json(const lp_config* c) {
    char b[512];
    std::snprintf(b, sizeof b,
                  "{\"op\":\"sampled_token_logprob\",\"lm_head\":{\"V\":%d,\"H\":%d,"
                  "\"layout\":\"[V,H] row-major\"},\"outputs\":[\"logp\",\"logZ\",\"entropy\","
                  "\"importance_weight\",\"d3\"]}",
                  c->V, c->H);
    return b;
}

std::string policy_json(const lp_config* c, int precision) {
    const bool fp8 = precision == LP_PRECISION_FP8_BLOCK;
    std::string tp = "[1";
    for (int s = 2; s <= c->n_leaves; s *= 2) tp += "," + std::to_string(s);
    tp += "]";
    const char* lm_bf16 =
        "\"impl\":{\"id\":\"leaf_gemm_tcgen05\",\"version\":%d,\"arch\":\"sm_103a\"},"
        "\"constants\":{\"input_dtype\":\"bf16\",\"leaves\":%d,\"leaf_dtype\":\"fp32\","
        "\"leaf_len\":%d,\"leaf_order\":\"k ascending, tcgen05.mma kind::f16 m128n128k16\",";
    const char* lm_fp8 =
        "\"impl\":{\"id\":\"leaf_gemm_tcgen05_block_fp8\",\"version\":%d,\"arch\":\"sm_103a\"},"
        "\"constants\":{\"input_dtype\":\"e4m3\",\"quantization\":{\"activation_block\":"
        "\"1x128\",\"weight_block\":\"128x128\",\"scale\":\"fp32 amax/448, 1 if amax=0\","
        "\"rounding\":\"x/s in fp32, nearest even, saturate to 448\"},\"leaves\":%d,"
        "\"leaf_dtype\":\"fp32\",\"leaf_len\":%d,\"leaf_order\":\"128-k blocks ascending: "
        "tcgen05.mma kind::f8f6f4 m128n128k32 per block; (sx*sw)*B, first a product then one fma "
        "per block\",";
    char lm[1024];
    std::snprintf(lm, sizeof lm, fp8 ? lm_fp8 : lm_bf16, lp_version(), c->n_leaves,
                  c->H / c->n_leaves);
    char b[4096];
    std::snprintf(
        b, sizeof b,
        "{\"cases\":[\"engine_prefill\",\"engine_decode\",\"trainer_fwd\",\"trainer_fwd_tp\"],"
        "\"composition\":["
        "{\"region\":[\"lm_head\",\"log_softmax\",\"sampled_logprob\"],"
        "\"cases\":[\"engine_prefill\",\"engine_decode\",\"trainer_fwd\",\"trainer_fwd_tp\"],"
        "%s\"leaf_tree\":\"adjacent pairs, level by level\",\"lse_tile\":64,"
        "\"lse_tile_order\":\"2 chunks of 32: max left to right; sum of exp(z-m) by pairwise "
        "tree; s0+s1\",\"tile_exp\":\"__expf\",\"merge\":\"(m,s) with expf; aligned pairwise "
        "tree over tiles\",\"log\":\"logf\",\"logp\":\"z_y - (m + log s)\"}},"
        "{\"region\":[\"importance_weight\",\"d3\",\"acceptance_stats\"],"
        "\"cases\":[\"trainer_fwd\"],"
        "\"impl\":{\"id\":\"block_tree_f64\",\"version\":1,\"arch\":\"sm_103a\"},"
        "\"constants\":{\"block\":1024,\"sum_dtype\":\"fp64\",\"w\":\"expf(fp32 d)\","
        "\"term\":\"taylor to d^9/9! for |d|<1/4 else expm1f(d)-d\"}}],"
        "\"claims\":{\"topology\":{\"tp_slices\":%s},\"phases\":[\"prefill\",\"decode\"],"
        "\"batch_invariance\":\"bit_exact\",\"tolerances\":{\"oracle_logp_nats\":0.002}}}",
        lm, tp.c_str());
    return b;
}

std::string deployment_json(const lp_config* c) {
    char b[256];
    std::snprintf(b, sizeof b, "{\"max_tokens\":%lld,\"tp_slices\":%d}",
                  static_cast<long long>(c->max_tokens), c->tp_slices);
    return b;
}

std::string section(const lp_config* c, int precision, int which) {
    return which == LP_DIGEST_SEMANTIC ? semantic_json(c)
           : which == LP_DIGEST_NUMERICAL_POLICY ? policy_json(c, precision)
                                                 : deployment_json(c);
}

int check_args(const lp_config* cfg, int precision) {
    int rc = lp_internal_validate_config(cfg);
    if (rc != LP_OK) return rc;
    if (precision != LP_PRECISION_BF16 && precision != LP_PRECISION_FP8_BLOCK)
        return lp_internal_fail(LP_ERR_INVALID_ARG, "unknown precision %d", precision);
    if (precision == LP_PRECISION_FP8_BLOCK && cfg->H % (128 * cfg->n_leaves) != 0)
        return lp_internal_fail(LP_ERR_UNSUPPORTED, "block FP8 needs H %% (128 * n_leaves) == 0");
    return LP_OK;
}

}  // namespace

extern "C" {

void lp_sha256(const void* data, size_t n, uint8_t out[32]) { sha256(data, n, out); }

int lp_contract_digest(const lp_config* cfg, int precision, int which, uint8_t out[32]) {
    int rc = check_args(cfg, precision);
    if (rc != LP_OK) return rc;
    if (which < LP_DIGEST_SEMANTIC || which > LP_DIGEST_DEPLOYMENT || out == nullptr)
        return lp_internal_fail(LP_ERR_INVALID_ARG, "bad digest selector or NULL output");
    const std::string s = section(cfg, precision, which);
    sha256(s.data(), s.size(), out);
    return LP_OK;
}

int lp_contract(const lp_config* cfg, int precision, char* buf, size_t cap, size_t* len) {
    int rc = check_args(cfg, precision);
    if (rc != LP_OK) return rc;
    uint8_t d[3][32];
    std::string parts[3];
    for (int i = 0; i < 3; ++i) {
        parts[i] = section(cfg, precision, i);
        sha256(parts[i].data(), parts[i].size(), d[i]);
    }
    const std::string json = "{\"semantic\":" + parts[0] + ",\"numerical_policy\":" + parts[1] +
                             ",\"deployment\":" + parts[2] + ",\"identities\":{\"semantic\":\"" +
                             hex(d[0]) + "\",\"numerical_policy\":\"" + hex(d[1]) +
                             "\",\"deployment\":\"" + hex(d[2]) + "\"}}";
    if (len) *len = json.size();
    if (buf == nullptr) return LP_OK;  // size query
    if (cap < json.size() + 1)
        return lp_internal_fail(LP_ERR_INVALID_ARG, "buffer too small: %zu bytes needed",
                                json.size() + 1);
    std::memcpy(buf, json.c_str(), json.size() + 1);
    return LP_OK;
}

int lp_contract_check(const lp_config* cfg, int precision, const uint8_t peer_semantic[32],
                      const uint8_t peer_numerical_policy[32]) {
    uint8_t mine[32];
    int rc = lp_contract_digest(cfg, precision, LP_DIGEST_SEMANTIC, mine);
    if (rc != LP_OK) return rc;
    if (peer_semantic == nullptr || peer_numerical_policy == nullptr)
        return lp_internal_fail(LP_ERR_INVALID_ARG, "peer digests must not be NULL");
    if (std::memcmp(mine, peer_semantic, 32) != 0)
        return lp_internal_fail(LP_ERR_UNSUPPORTED, "semantic digest differs from the peer's");
    lp_contract_digest(cfg, precision, LP_DIGEST_NUMERICAL_POLICY, mine);
    if (std::memcmp(mine, peer_numerical_policy, 32) != 0)
        return lp_internal_fail(LP_ERR_UNSUPPORTED,
                                "numerical_policy digest differs from the peer's");
    return LP_OK;
}

}  // extern "C"
