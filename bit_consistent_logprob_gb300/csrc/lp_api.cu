// lp_api.cu -- host side of the C ABI declared in include/lp.h: argument checks, the
// fixed launch plan, workspace ownership, TMA descriptors and kernel launches for the
// logprob path (bf16 and block-FP8 handles), the RL epilogues, the backward (whose two plain
// GEMMs go to cuBLAS) and the failure-detection self-test.  The execution contract lives in
// lp_contract.cu, the handle-free entry point in lp_noalloc.cu.
//
// The plan depends only on (H, V, N, tp_slices, max_tokens) and on how many rows a
// call carries; the per-element arithmetic never depends on T, the SM count or the
// phase, so every row is bit-identical however it is batched.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "grad_gemm.cuh"
#include "kernels.cuh"
#include "lp.h"
#include "fp8_kernels.cuh"
#include "lp_internal.h"
#include "rl_kernels.cuh"

namespace {

constexpr int64_t kMaxIsTokens = (1LL << 31) - 1;
constexpr int64_t kTpRows = 1024;               // rows per pass of the emulated TP path
constexpr int kProfPairs = 4096;
constexpr int64_t kIsStage = 1 << 20;            // tokens per pass of the host IS call
constexpr int kShortStageRows = 256;              // leaf-GEMM launches up to here: 64-K stages
constexpr int64_t kHostFirstPiece = 512;  // lp_logprobs_host: rows of the first piece
constexpr int64_t kHostGrowth = 8;        // ... and the growth of each piece over the last

thread_local std::string g_last_error = "no error";

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    cudaGetLastError();  // clear the non-sticky error
    return fail(e == cudaErrorMemoryAllocation ? LP_ERR_OOM : LP_ERR_CUDA, "%s: %s (%s)", what,
                cudaGetErrorName(e), cudaGetErrorString(e));
}

#define LP_CUDA(call, what)                          \
    do {                                             \
        cudaError_t e_ = (call);                     \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// K-major bf16 matrix [rows, K] with a row stride of `ld` elements, read in 128 x 64
// boxes with 128-byte swizzling (the layout the tcgen05 descriptors expect).  Rows past
// `rows` read as zero.
// K-major 2-D tensor map with 128-byte-wide boxes (64 bf16 or 128 one-byte elements) and the
// 128-byte swizzle the MMA descriptors expect.
int encode_kmajor(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K, uint64_t ld,
                  uint32_t box_rows = lp::kBM, bool bytes = false) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return fail(LP_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const uint64_t esize = bytes ? 1 : 2;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {ld * esize};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     2, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return LP_OK;
}

}  // namespace

struct lp_handle {
    lp_config cfg{};
    const void* W = nullptr;
    int device = 0;
    int num_sms = 0;
    int num_vocab_tiles = 0;  // ceil(V / 128): MMA tiles
    int num_lse_tiles = 0;    // ceil(V / 64): log-sum-exp tiles
    int leaf_len = 0;
    uint64_t timeout_ns = 0;
    CUtensorMap tmW{};
    CUtensorMap tmW64{};  // the same W with 64-row boxes (a CTA pair's half of a W tile)
    double* host_scalars = nullptr;  // pinned host: D3 and n_valid of the host-buffer call
    // workspace (device)
    float2* ws_ms = nullptr;      // [num_lse_tiles][max_tokens]
    float* ws_u = nullptr;        // [num_lse_tiles][max_tokens] entropy partials
    // backward (lp_backward_reserve)
    uint16_t* dl = nullptr;       // [dl_rows][ldd] bf16 gradient with respect to the logits
    int64_t dl_rows = 0;
    int64_t ldd = 0;
    float* grad_part = nullptr;   // [kMaxGradSlices][dl_rows][H] fp32: dX partials of a K split
    float* zy = nullptr;          // [max_tokens]
    int* status = nullptr;        // sticky status word
    int* sched = nullptr;         // tile counter of the pair launches' dynamic schedule
    double* blk_sum = nullptr;    // [max_is_blocks]
    long long* blk_cnt = nullptr; // [max_is_blocks]
    unsigned* is_done = nullptr;  // blocks done in a one-launch epilogue (IS, statistics, loss); 0 between calls
    double* stat_blk = nullptr;   // [2][max_is_blocks]: sum |d|^2 and sum k3 per block
    float* stat_max = nullptr;    // [max_is_blocks]: max |d| per block
    int64_t max_is_blocks = 0;
    float* tp_parts = nullptr;    // [tp_slices][max_tokens][ldp] slice outputs
    float* tp_gather = nullptr;   // same shape: the "transported" copy
    int64_t tp_ldp = 0;
    int64_t chunk_rows = 0;       // rows per pass: max_tokens, or the TP sub-chunk
    // staging for lp_logprobs_host (device)
    void* x_stage = nullptr;
    int32_t* ids_stage = nullptr;
    float* logp_stage = nullptr;
    float* logz_stage = nullptr;
    // lp_logprobs_host pipeline: pieces alternate between the two halves of the staging
    // buffers; the copy of piece i+1 (on copy_stream) runs under the GEMM of piece i
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t stage_ready[2] = {nullptr, nullptr};  // half b holds its piece
    cudaEvent_t stage_free[2] = {nullptr, nullptr};   // half b's kernels are done with it
    cudaEvent_t host_entry = nullptr;                 // the caller's stream at entry
    float* is_stage = nullptr;      // [3][kIsStage]: log pi, log mu, w of one pass
    uint8_t* is_mask_stage = nullptr;
    double* scalars = nullptr;      // [2]: D3 and n_valid of the host IS call
    // block-FP8 handles (lp_init_fp8)
    bool fp8 = false;
    uint8_t* wq = nullptr;          // [V][H] e4m3 lm_head
    float* sw = nullptr;            // [num_vocab_tiles][H/128] weight block scales
    uint8_t* xq = nullptr;          // [max_tokens][H] e4m3 activations of one chunk
    float* sx = nullptr;            // [max_tokens][H/128] activation block scales
    CUtensorMap tmWq{};
    int band_fp8 = 0;
    cudaStream_t last_stream = nullptr;
    int64_t ws_bytes = 0;
    int32_t last_launches = 0;
    // launch-layout switches read from the environment at init (LP_FORCE_SINGLE_CTA,
    // LP_FORCE_SHORT_STAGES); they change only the schedule, never the arithmetic, and let
    // the tests prove that
    bool force_single_cta = false;
    bool force_sub1 = false;
    int test_stop_after = 0;  // LP_TEST_STOP_AFTER_STAGES: test hook of the abort path
    int band = 0;  // vocabulary tiles per scheduling band (even); schedule only
    int band_axis_env = -1;  // LP_BAND_AXIS: -1 = chosen per launch, 0 = vocabulary, 1 = rows
    int band_rows_env = 0;   // LP_BAND_ROWS: scheduling rows per row band (0 = from the budget)
    // profiling: event pairs around leaf-GEMM launches
    bool profiling = false;
    std::vector<cudaEvent_t> prof_events;  // 2 * kProfPairs, created on enable
    std::vector<int> prof_kind;            // what each pair brackets (LP_PROFILE_*)
    int prof_used = 0;                     // pairs recorded since the last read
};

namespace {

int validate_config(const lp_config* c) {
    if (c == nullptr) return fail(LP_ERR_INVALID_ARG, "config is NULL");
    if (c->H <= 0 || c->V <= 0) return fail(LP_ERR_INVALID_ARG, "H and V must be positive");
    if (c->max_tokens <= 0 || c->max_tokens > (1LL << 31) - 1)
        return fail(LP_ERR_INVALID_ARG, "max_tokens must be in [1, 2^31)");
    if (!(c->n_leaves == 1 || c->n_leaves == 2 || c->n_leaves == 4 || c->n_leaves == 8))
        return fail(LP_ERR_UNSUPPORTED, "n_leaves must be 1, 2, 4 or 8 (got %d)", c->n_leaves);
    if (c->H % (lp::kBK * c->n_leaves) != 0)
        return fail(LP_ERR_UNSUPPORTED, "H (%d) must be a multiple of 64 * n_leaves (%d)", c->H,
                    lp::kBK * c->n_leaves);
    if (!(c->tp_slices == 1 || c->tp_slices == 2 || c->tp_slices == 4 || c->tp_slices == 8) ||
        c->n_leaves % c->tp_slices != 0)
        return fail(LP_ERR_UNSUPPORTED, "tp_slices must be 1, 2, 4 or 8 and divide n_leaves");
    return LP_OK;
}

// Rows per X TMA box: a full 128-row tile, or for a batch smaller than one tile just its
// rows rounded up to 8 (the rows of the shared-memory tile past the box are never written;
// they only feed accumulator rows that are never read back).
uint32_t x_box_rows(int rows) {
    return rows >= lp::kBM ? lp::kBM : static_cast<uint32_t>((rows + 7) / 8 * 8);
}

// Scheduling band: enough vocabulary tiles for `mib` MiB of W, which stays L2-resident while
// every row tile of the batch sweeps across it.  Measured on GB300: 32 MiB for the bf16 kernel
// (18 tiles at H = 7168, 3 % faster than 16; at H = 2048 anything from 32 to 96 tiles is within
// 0.5 %), 28 MiB for the epilogue-bound block-FP8 kernel.  The band decides which CTA
// computes a tile, never how.
int scheduling_band(int H, int bytes_per_weight, int max_tiles, int mib) {
    const int64_t per_tile = static_cast<int64_t>(lp::kVT) * H * bytes_per_weight;
    int64_t b = (static_cast<int64_t>(mib) << 20) / per_tile;
    b = b < 8 ? 8 : (b > max_tiles ? max_tiles : b);
    return static_cast<int>(b) & ~1;
}

// Profiling: a pair of events on the launch stream around one timed kernel (or group).
bool prof_begin(lp_handle* h, cudaStream_t st, int kind) {
    if (!h->profiling || h->prof_used >= kProfPairs) return false;
    h->prof_kind[h->prof_used] = kind;
    return cudaEventRecord(h->prof_events[2 * h->prof_used], st) == cudaSuccess;
}

cudaError_t prof_end(lp_handle* h, cudaStream_t st) {
    const cudaError_t e = cudaEventRecord(h->prof_events[2 * h->prof_used + 1], st);
    ++h->prof_used;
    return e;
}

// The band of one bf16 leaf-GEMM launch (see tile_coords).  Vocabulary bands of h->band
// tiles (32 MiB of W) by default; LP_BAND_AXIS=rows switches to row bands of LP_BAND_ROWS
// scheduling rows (default: 32 MiB of X).  Measured on GB300 (DRAM reads per launch, time):
// at the 32 MiB budget row bands read less (H 2048, V 151936, 17627 rows: 1.3 GB against
// 2.0 GB; H 4096, V 151936, 32768 rows: 10.2 GB against 11.5 GB) but run 1-1.5 % slower at
// the larger shapes; resident bands beyond ~32 MiB, on either axis, thrash L2 (H 7168,
// V 129280, 16384 rows: 28 GB with 36 vocabulary tiles, 71 GB with 22 row pairs, against
// 15.8 GB).  The band moves data, never arithmetic.
constexpr int kBandMiB = 32;
void pick_band(const lp_handle* h, int rows, bool pair, int32_t& axis, int32_t& band) {
    (void)rows;
    axis = h->band_axis_env == 1 ? 1 : 0;
    if (axis == 0) {
        band = h->band;
        return;
    }
    const int64_t unit_rows = pair ? 2 * lp::kBM : lp::kBM;  // rows per scheduling row
    int64_t rband = h->band_rows_env > 0
                        ? h->band_rows_env
                        : (int64_t(kBandMiB) << 20) / (unit_rows * int64_t(h->cfg.H) * 2);
    band = static_cast<int32_t>(rband < 1 ? 1 : rband);
}

template <int kMode, int kSub, bool kPair = false>
cudaError_t launch_gemm_variant(int grid, cudaStream_t st, const CUtensorMap& tmX,
                                const CUtensorMap& tmW, const CUtensorMap& tmD,
                                const lp::GemmParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(lp::kGemmThreads);
    cfg.dynamicSmemBytes = lp::gemm_smem_bytes(kSub, kMode, kPair);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (kPair) {  // clusters of two CTAs: the pair of one cta_group::2 MMA
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, lp::leaf_gemm_kernel<kMode, kSub, kPair>, tmX, tmW, tmD, p);
}

template <int kMode>
int set_gemm_attributes() {
    const auto set = [](auto fn, int sub, bool pair) {
        return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    lp::gemm_smem_bytes(sub, kMode, pair));
    };
    cudaError_t e;
    if ((e = set(lp::leaf_gemm_kernel<kMode, 1>, 1, false)) != cudaSuccess ||
        (e = set(lp::leaf_gemm_kernel<kMode, 2>, 2, false)) != cudaSuccess ||
        (e = set(lp::leaf_gemm_kernel<kMode, 1, true>, 1, true)) != cudaSuccess ||
        (e = set(lp::leaf_gemm_kernel<kMode, 2, true>, 2, true)) != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(leaf_gemm_kernel)");
    return LP_OK;
}

// Extra per-mode operands of the leaf GEMM epilogue (kModeGrad).
struct GradArgs {
    const float* logZ = nullptr;
    const float* gout = nullptr;
    uint16_t* dl = nullptr;
    int64_t ldd = 0;
};

// The leaf GEMM over `rows` rows of X starting at `X` (row stride ldx).  Calls of more than
// one row tile run in CTA pairs (cta_group::2: each pair computes two row tiles of one
// vocabulary tile, each CTA loading half of the W tile, so the tensor core gets 256 rows per
// MMA instruction and each CTA fills 24 KB of shared memory per 64-K step instead of 32 KB);
// calls of at most one row tile (decode batches up to 128) run one CTA per 128 x 128 tile with
// the X box cut to their rows.  Stages are 128 K deep (8 MMAs per barrier synchronisation) when the leaf length allows.  Launches of
// at most kShortStageRows rows (decode batches) and odd leaf lengths take seven 64-K stages
// instead: such launches read each W tile from DRAM for one or two row tiles, and the deeper
// ring keeps 112 KB of W per CTA in flight instead of 96 KB (measured on GB300: decode
// batch 256 went from 66 % to 71 % of the copy bandwidth, batch 128 from 94 % to 98 %).  The
// stage depth changes only the schedule: every leaf sees the same MMA sequence.
template <int kMode>
int launch_leaf_gemm(lp_handle* h, const void* X, int64_t ldx, int rows, int leaf_begin,
                     int leaf_count, const int32_t* ids, float* out, int64_t ldo,
                     cudaStream_t st, const GradArgs& ga = GradArgs()) {
    lp::GemmParams p{};
    p.T = rows;
    p.V = h->cfg.V;
    p.leaf_len = h->leaf_len;
    p.leaf_begin = leaf_begin;
    p.leaf_count = leaf_count;
    p.num_row_tiles = static_cast<int32_t>(ceil_div(rows, lp::kBM));
    p.num_vocab_tiles = h->num_vocab_tiles;
    p.num_lse_tiles = h->num_lse_tiles;
    p.ids = ids;
    p.ws_ms = h->ws_ms;
    p.ws_ld = h->cfg.max_tokens;
    p.zy = h->zy;
    p.out = out;
    p.ldo = ldo;
    p.ws_u = h->ws_u;
    p.logZ = ga.logZ;
    p.gout = ga.gout;
    p.dl = ga.dl;
    p.ldd = ga.ldd;
    p.status = h->status;
    p.sched = h->sched;
    p.test_stop_after = h->test_stop_after;
    p.timeout_ns = h->timeout_ns;
    const bool sub2 = h->leaf_len % (2 * lp::kBK) == 0 && rows > kShortStageRows && !h->force_sub1;
    const bool pair = rows > lp::kBM && !h->force_single_cta;
    pick_band(h, rows, pair, p.band_axis, p.band);
    p.x_box_rows = static_cast<int32_t>(x_box_rows(rows));
    CUtensorMap tmX;
    int rc = encode_kmajor(&tmX, X, static_cast<uint64_t>(rows), h->cfg.H, ldx,
                           static_cast<uint32_t>(p.x_box_rows));
    if (rc != LP_OK) return rc;
    // the gradient epilogue's TMA stores: dl [rows][ldd] bf16 in 64-column x 32-row boxes
    CUtensorMap tmD{};
    if constexpr (kMode == lp::kModeGrad) {
        rc = encode_kmajor(&tmD, ga.dl, static_cast<uint64_t>(rows), h->cfg.V, ga.ldd, 32);
        if (rc != LP_OK) return rc;
    }
    // scheduling units: tiles, or (pairs) two row tiles of one vocabulary tile
    const int64_t tiles =
        (pair ? ceil_div(p.num_row_tiles, 2) : p.num_row_tiles) * int64_t(h->num_vocab_tiles);
    if (tiles > 0x7fffffff) return fail(LP_ERR_UNSUPPORTED, "too many tiles in one launch");
    const int64_t slots = pair ? h->num_sms / 2 : h->num_sms;
    const int grid = static_cast<int>((tiles < slots ? tiles : slots) * (pair ? 2 : 1));
    // a pair launch hands out its tiles from a counter that starts at zero
    if (pair) LP_CUDA(cudaMemsetAsync(h->sched, 0, sizeof(int), st), "tile counter reset");
    const bool prof = prof_begin(h, st, LP_PROFILE_LEAF_GEMM);
    cudaError_t e;
    if (pair)
        e = sub2 ? launch_gemm_variant<kMode, 2, true>(grid, st, tmX, h->tmW64, tmD, p)
                 : launch_gemm_variant<kMode, 1, true>(grid, st, tmX, h->tmW64, tmD, p);
    else
        e = sub2 ? launch_gemm_variant<kMode, 2>(grid, st, tmX, h->tmW, tmD, p)
                 : launch_gemm_variant<kMode, 1>(grid, st, tmX, h->tmW, tmD, p);
    LP_CUDA(e, "leaf_gemm_kernel launch");
    LP_CUDA(cudaGetLastError(), "leaf_gemm_kernel launch");
    if (prof) LP_CUDA(prof_end(h, st), "profile event");
    ++h->last_launches;
    return LP_OK;
}

int launch_combine(lp_handle* h, const int32_t* ids, int rows, float* out_logp, float* out_logZ,
                   float* out_entropy, cudaStream_t st) {
    lp::CombineParams c{};
    c.ws_ms = h->ws_ms;
    c.ws_u = h->ws_u;
    c.out_entropy = out_entropy;
    c.ws_ld = h->cfg.max_tokens;
    c.zy = h->zy;
    c.ids = ids;
    c.T = rows;
    c.V = h->cfg.V;
    c.num_tiles = h->num_lse_tiles;
    const lp::CombineLayout lay = lp::combine_layout(rows, h->num_lse_tiles, h->num_sms);
    c.rows = lay.rows;
    c.seg_log = lay.seg_log;
    c.nseg = lay.nseg;
    c.out_logp = out_logp;
    c.out_logZ = out_logZ;
    c.status = h->status;
    const size_t n = static_cast<size_t>(lay.rows) * lay.nseg;
    const dim3 grid(static_cast<unsigned>(ceil_div(rows, lay.rows)));
    const dim3 block(static_cast<unsigned>(lay.rows * lay.nseg));
    if (out_entropy)
        lp::lse_combine_kernel<true><<<grid, block, sizeof(float3) * n, st>>>(c);
    else
        lp::lse_combine_kernel<false><<<grid, block, sizeof(float2) * n, st>>>(c);
    LP_CUDA(cudaGetLastError(), "lse_combine_kernel launch");
    ++h->last_launches;
    return LP_OK;
}

int launch_partials_lse(lp_handle* h, const float* parts, int n_parts, int64_t part_stride,
                        int64_t ldp, const int32_t* ids, int rows, bool entropy, cudaStream_t st) {
    lp::PartialsParams q{};
    q.parts = parts;
    q.part_stride = part_stride;
    q.ldp = ldp;
    q.n_parts = n_parts;
    q.T = rows;
    q.V = h->cfg.V;
    q.ids = ids;
    q.ws_ms = h->ws_ms;
    q.ws_u = h->ws_u;
    q.ws_ld = h->cfg.max_tokens;
    q.zy = h->zy;
    dim3 grid(static_cast<unsigned>(h->num_vocab_tiles), static_cast<unsigned>(ceil_div(rows, 128)));
    if (entropy) {
        switch (n_parts) {
            case 1: lp::partials_lse_kernel<1, true><<<grid, 128, 0, st>>>(q); break;
            case 2: lp::partials_lse_kernel<2, true><<<grid, 128, 0, st>>>(q); break;
            case 4: lp::partials_lse_kernel<4, true><<<grid, 128, 0, st>>>(q); break;
            default: lp::partials_lse_kernel<8, true><<<grid, 128, 0, st>>>(q); break;
        }
    } else {
        switch (n_parts) {
            case 1: lp::partials_lse_kernel<1, false><<<grid, 128, 0, st>>>(q); break;
            case 2: lp::partials_lse_kernel<2, false><<<grid, 128, 0, st>>>(q); break;
            case 4: lp::partials_lse_kernel<4, false><<<grid, 128, 0, st>>>(q); break;
            default: lp::partials_lse_kernel<8, false><<<grid, 128, 0, st>>>(q); break;
        }
    }
    LP_CUDA(cudaGetLastError(), "partials_lse_kernel launch");
    ++h->last_launches;
    return LP_OK;
}

// Block-FP8 path for one chunk: quantise the rows (1 x 128 blocks), then the block-scaled leaf
// GEMM with the fused tile log-sum-exp (one CTA per tile, X box cut to the rows when T < 128).
// Quantise one chunk of X (rows <= max_tokens) into the handle's e4m3 activations and their
// 1 x 128 block scales.
int quantize_x_chunk(lp_handle* h, const void* X, int64_t ldx, int rows, cudaStream_t st) {
    const int H = h->cfg.H;
    const int nkb = H / lp::kQBlock;
    const int64_t warps = static_cast<int64_t>(rows) * nkb;
    lp::quant_x_kernel<<<static_cast<unsigned>(ceil_div(warps, 8)), 256, 0, st>>>(
        static_cast<const uint16_t*>(X), ldx, rows, H, h->xq, H, h->sx);
    LP_CUDA(cudaGetLastError(), "quant_x_kernel launch");
    ++h->last_launches;
    return LP_OK;
}

// The block-FP8 leaf GEMM over the leaves [leaf_begin, leaf_begin + leaf_count) of the chunk
// quantize_x_chunk left in the handle: tile partials (kModeLse, kModeLseEnt) or the tree node
// written to out (kModeNode).
template <int kMode>
int launch_fp8_gemm(lp_handle* h, int rows, int leaf_begin, int leaf_count, const int32_t* ids,
                    float* out, int64_t ldo, cudaStream_t st) {
    const int H = h->cfg.H;
    lp::GemmParams p{};
    p.T = rows;
    p.V = h->cfg.V;
    p.leaf_len = h->leaf_len;
    p.leaf_begin = leaf_begin;
    p.leaf_count = leaf_count;
    p.num_row_tiles = static_cast<int32_t>(ceil_div(rows, lp::kBM));
    p.num_vocab_tiles = h->num_vocab_tiles;
    p.num_lse_tiles = h->num_lse_tiles;
    p.band = h->band_fp8;
    p.test_stop_after = h->test_stop_after;
    p.x_box_rows = static_cast<int32_t>(x_box_rows(rows));
    p.ids = ids;
    p.ws_ms = h->ws_ms;
    p.ws_ld = h->cfg.max_tokens;
    p.zy = h->zy;
    p.ws_u = h->ws_u;
    p.out = out;
    p.ldo = ldo;
    p.sx = h->sx;
    p.sw = h->sw;
    p.nkb = H / lp::kQBlock;
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    CUtensorMap tmX;
    int rc = encode_kmajor(&tmX, h->xq, static_cast<uint64_t>(rows), H, H,
                           static_cast<uint32_t>(p.x_box_rows), true);
    if (rc != LP_OK) return rc;
    const int64_t tiles = static_cast<int64_t>(p.num_row_tiles) * h->num_vocab_tiles;
    if (tiles > 0x7fffffff) return fail(LP_ERR_UNSUPPORTED, "too many tiles in one launch");
    const int grid = static_cast<int>(tiles < h->num_sms ? tiles : h->num_sms);
    const bool prof = prof_begin(h, st, LP_PROFILE_LEAF_GEMM);
    lp::leaf_gemm_fp8_kernel<kMode><<<grid, lp::kF8Threads, lp::fp8_smem_bytes(), st>>>(
        tmX, h->tmWq, p);
    LP_CUDA(cudaGetLastError(), "leaf_gemm_fp8_kernel launch");
    if (prof) LP_CUDA(prof_end(h, st), "profile event");
    ++h->last_launches;
    return LP_OK;
}

// Quantise the referenced bf16 lm_head into the handle's e4m3 copy (128 x 128 blocks).
int quantize_weights(lp_handle* h, cudaStream_t st) {
    const dim3 grid(static_cast<unsigned>(h->cfg.H / lp::kQBlock),
                    static_cast<unsigned>(h->num_vocab_tiles));
    lp::quant_w_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(h->W), h->cfg.V,
                                             h->cfg.H, h->wq, h->sw);
    LP_CUDA(cudaGetLastError(), "quant_w_kernel launch");
    return LP_OK;
}

// Fused path or emulated tensor-parallel path for one chunk of rows (rows <= max_tokens).
int logprobs_chunk(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids, int rows,
                   float* out_logp, float* out_logZ, float* out_entropy, cudaStream_t st) {
    int rc;
    const int s = h->cfg.tp_slices;
    const int n = h->cfg.n_leaves;
    if (h->fp8 && (rc = quantize_x_chunk(h, X, ldx, rows, st)) != LP_OK) return rc;
    if (s == 1) {
        if (h->fp8)
            rc = out_entropy ? launch_fp8_gemm<lp::kModeLseEnt>(h, rows, 0, n, ids, nullptr, 0, st)
                             : launch_fp8_gemm<lp::kModeLse>(h, rows, 0, n, ids, nullptr, 0, st);
        else
            rc = out_entropy
                     ? launch_leaf_gemm<lp::kModeLseEnt>(h, X, ldx, rows, 0, n, ids, nullptr, 0, st)
                     : launch_leaf_gemm<lp::kModeLse>(h, X, ldx, rows, 0, n, ids, nullptr, 0, st);
        if (rc != LP_OK) return rc;
    } else {
        // Slice r owns leaves [r*N/s, (r+1)*N/s) and produces that node of the leaf tree;
        // the partials are then moved (a plain copy: data only, no arithmetic) into the
        // gathered buffer, where the upper levels of the same tree are applied.
        const int per = h->cfg.n_leaves / s;
        const int64_t part_stride = h->chunk_rows * h->tp_ldp;
        for (int r = 0; r < s; ++r) {
            float* part = h->tp_parts + r * part_stride;
            rc = h->fp8 ? launch_fp8_gemm<lp::kModeNode>(h, rows, r * per, per, nullptr, part,
                                                         h->tp_ldp, st)
                        : launch_leaf_gemm<lp::kModeNode>(h, X, ldx, rows, r * per, per, nullptr,
                                                          part, h->tp_ldp, st);
            if (rc != LP_OK) return rc;
        }
        for (int r = 0; r < s; ++r) {
            LP_CUDA(cudaMemcpyAsync(h->tp_gather + r * part_stride, h->tp_parts + r * part_stride,
                                    sizeof(float) * static_cast<size_t>(rows) * h->tp_ldp,
                                    cudaMemcpyDeviceToDevice, st),
                    "slice transport copy");
        }
        rc = launch_partials_lse(h, h->tp_gather, s, part_stride, h->tp_ldp, ids, rows,
                                 out_entropy != nullptr, st);
        if (rc != LP_OK) return rc;
    }
    return launch_combine(h, ids, rows, out_logp, out_logZ, out_entropy, st);
}

int check_x(const lp_handle* h, const void* X, int64_t ldx, int64_t T) {
    if (T < 0) return fail(LP_ERR_INVALID_ARG, "T must be >= 0");
    if (T == 0) return LP_OK;
    if (X == nullptr) return fail(LP_ERR_INVALID_ARG, "X is NULL");
    if (!aligned16(X)) return fail(LP_ERR_INVALID_ARG, "X must be 16-byte aligned");
    if (ldx < h->cfg.H || ldx % 8 != 0)
        return fail(LP_ERR_INVALID_ARG, "ldx must be >= H and a multiple of 8 (got %lld)",
                    (long long)ldx);
    return LP_OK;
}

}  // namespace

int lp_internal_validate_config(const lp_config* c) { return validate_config(c); }

int lp_internal_fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

extern "C" {

int lp_version(void) { return 100; }

const char* lp_last_error(void) { return g_last_error.c_str(); }

int64_t lp_workspace_bytes(const lp_handle* h) { return h ? h->ws_bytes : 0; }

int32_t lp_last_launch_count(const lp_handle* h) { return h ? h->last_launches : 0; }

void lp_free(lp_handle* h) {
    if (h == nullptr) return;
    cudaDeviceSynchronize();
    for (cudaEvent_t e : h->prof_events) cudaEventDestroy(e);
    for (cudaEvent_t e : {h->stage_ready[0], h->stage_ready[1], h->stage_free[0],
                          h->stage_free[1], h->host_entry})
        if (e) cudaEventDestroy(e);
    if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
    cudaFree(h->ws_ms);
    cudaFree(h->zy);
    cudaFree(h->status);
    cudaFree(h->sched);
    cudaFree(h->ws_u);
    cudaFree(h->wq);
    cudaFree(h->sw);
    cudaFree(h->xq);
    cudaFree(h->sx);
    cudaFree(h->dl);
    cudaFree(h->grad_part);
    cudaFree(h->blk_sum);
    cudaFree(h->blk_cnt);
    cudaFree(h->is_done);
    cudaFree(h->stat_blk);
    cudaFree(h->stat_max);
    cudaFree(h->tp_parts);
    cudaFree(h->tp_gather);
    cudaFree(h->x_stage);
    cudaFree(h->ids_stage);
    cudaFree(h->logp_stage);
    cudaFree(h->logz_stage);
    cudaFree(h->is_stage);
    cudaFree(h->is_mask_stage);
    if (h->host_scalars) cudaFreeHost(h->host_scalars);
    cudaFree(h->scalars);
    delete h;
}

namespace {
int init_impl(const lp_config* cfg, const void* W, void* stream, lp_handle** out, bool fp8) {
    if (out == nullptr) return fail(LP_ERR_INVALID_ARG, "out handle pointer is NULL");
    *out = nullptr;
    int rc = validate_config(cfg);
    if (rc != LP_OK) return rc;
    if (fp8 && cfg->H % (lp::kQBlock * cfg->n_leaves) != 0)
        return fail(LP_ERR_UNSUPPORTED,
                    "block FP8 needs H (%d) to be a multiple of 128 * n_leaves (%d)", cfg->H,
                    lp::kQBlock * cfg->n_leaves);
    if (W == nullptr) return fail(LP_ERR_INVALID_ARG, "W is NULL");
    if (!aligned16(W)) return fail(LP_ERR_INVALID_ARG, "W must be 16-byte aligned");

    int dev = 0;
    LP_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    cudaDeviceProp prop;
    LP_CUDA(cudaGetDeviceProperties(&prop, dev), "cudaGetDeviceProperties");
    if (!(prop.major == 10 && prop.minor == 3))
        return fail(LP_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300); device is sm_%d%d",
                    prop.major, prop.minor);

    lp_handle* h = new lp_handle();
    h->cfg = *cfg;
    h->W = W;
    h->device = dev;
    h->num_sms = prop.multiProcessorCount;
    h->num_vocab_tiles = static_cast<int>(ceil_div(cfg->V, lp::kVT));
    h->num_lse_tiles = static_cast<int>(ceil_div(cfg->V, lp::kLT));
    h->leaf_len = cfg->H / cfg->n_leaves;
    uint64_t timeout_ms = 2000;
    if (const char* e = std::getenv("LP_WAIT_TIMEOUT_MS")) {
        long long v = std::atoll(e);
        if (v > 0) timeout_ms = static_cast<uint64_t>(v);
    }
    h->timeout_ns = timeout_ms * 1000000ull;
    if (const char* e = std::getenv("LP_FORCE_SINGLE_CTA")) h->force_single_cta = e[0] == '1';
    if (const char* e = std::getenv("LP_FORCE_SHORT_STAGES")) h->force_sub1 = e[0] == '1';
    if (const char* e = std::getenv("LP_TEST_STOP_AFTER_STAGES")) {
        const int v = std::atoi(e);
        if (v > 0) h->test_stop_after = v;
    }
    h->band = scheduling_band(cfg->H, 2, 64, 32);
    if (const char* e = std::getenv("LP_BAND")) {
        const int b = std::atoi(e);
        if (b >= 2 && b <= 1024) h->band = b & ~1;
    }
    if (const char* e = std::getenv("LP_BAND_AXIS")) {
        if (std::strcmp(e, "vocab") == 0) h->band_axis_env = 0;
        if (std::strcmp(e, "rows") == 0) h->band_axis_env = 1;
    }
    if (const char* e = std::getenv("LP_BAND_ROWS")) {
        const int b = std::atoi(e);
        if (b >= 1 && b <= 1 << 20) h->band_rows_env = b;
    }
    h->band_fp8 = scheduling_band(cfg->H, 1, 128, 28);  // e4m3 weights: twice the tiles per byte
    h->fp8 = fp8;

    auto cleanup = [&](int code) {
        lp_free(h);
        return code;
    };
    rc = encode_kmajor(&h->tmW, W, static_cast<uint64_t>(cfg->V), cfg->H, cfg->H);
    if (rc != LP_OK) return cleanup(rc);
    rc = encode_kmajor(&h->tmW64, W, static_cast<uint64_t>(cfg->V), cfg->H, cfg->H, lp::kVT / 2);
    if (rc != LP_OK) return cleanup(rc);

    const int64_t mt = cfg->max_tokens;
    // LP_TEST_FAIL_ALLOC=<buffer name> reports that buffer's allocation as failed: a test hook
    // for the clean-up path (every buffer allocated so far is freed, nothing leaks)
    const char* fail_alloc = std::getenv("LP_TEST_FAIL_ALLOC");
    auto alloc = [&](void** p, size_t bytes, const char* what) -> int {
        if (fail_alloc != nullptr && std::strcmp(fail_alloc, what) == 0)
            return fail(LP_ERR_OOM, "%s: allocation of %zu bytes failed (test hook)", what, bytes);
        cudaError_t e = cudaMalloc(p, bytes);
        if (e != cudaSuccess) return cuda_fail(e, what);  // LP_ERR_OOM when out of memory
        h->ws_bytes += static_cast<int64_t>(bytes);
        return LP_OK;
    };
    h->max_is_blocks = ceil_div(kMaxIsTokens, lp::kIsBlock);
    if ((rc = alloc(reinterpret_cast<void**>(&h->ws_ms),
                    sizeof(float2) * static_cast<size_t>(h->num_lse_tiles) * mt, "ws_ms")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->ws_u),
                    sizeof(float) * static_cast<size_t>(h->num_lse_tiles) * mt, "ws_u")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->zy), sizeof(float) * mt, "zy")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->status), sizeof(int), "status")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->sched), sizeof(int), "sched")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->blk_sum), sizeof(double) * h->max_is_blocks,
                    "blk_sum")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->blk_cnt), sizeof(long long) * h->max_is_blocks,
                    "blk_cnt")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->is_done), sizeof(unsigned), "is_done")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->stat_blk), 2 * sizeof(double) * h->max_is_blocks,
                    "stat_blk")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->stat_max), sizeof(float) * h->max_is_blocks,
                    "stat_max")) ||
        (rc = alloc(&h->x_stage, sizeof(uint16_t) * static_cast<size_t>(mt) * cfg->H, "x_stage")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->ids_stage), sizeof(int32_t) * mt, "ids_stage")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->logp_stage), sizeof(float) * mt, "logp_stage")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->logz_stage), sizeof(float) * mt, "logz_stage")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->is_stage), sizeof(float) * 3 * kIsStage,
                    "is_stage")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->is_mask_stage), kIsStage, "is_mask_stage")) ||
        (rc = alloc(reinterpret_cast<void**>(&h->scalars), 2 * sizeof(double), "scalars")))
        return cleanup(rc);
    if (fail_alloc != nullptr && std::strcmp(fail_alloc, "host_scalars") == 0)
        return cleanup(fail(LP_ERR_OOM, "host_scalars: allocation failed (test hook)"));
    if (cudaError_t e = cudaMallocHost(reinterpret_cast<void**>(&h->host_scalars),
                                       2 * sizeof(double));
        e != cudaSuccess)
        return cleanup(cuda_fail(e, "host_scalars"));
    h->chunk_rows = mt;
    if (cfg->tp_slices > 1) {
        h->chunk_rows = mt < kTpRows ? mt : kTpRows;
        h->tp_ldp = ceil_div(cfg->V, 4) * 4;
        const size_t bytes =
            sizeof(float) * static_cast<size_t>(cfg->tp_slices) * h->chunk_rows * h->tp_ldp;
        if ((rc = alloc(reinterpret_cast<void**>(&h->tp_parts), bytes, "tp_parts")) ||
            (rc = alloc(reinterpret_cast<void**>(&h->tp_gather), bytes, "tp_gather")))
            return cleanup(rc);
    }

    {
        cudaError_t ce = cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking);
        for (cudaEvent_t* ev : {&h->stage_ready[0], &h->stage_ready[1], &h->stage_free[0],
                                &h->stage_free[1], &h->host_entry})
            if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (ce != cudaSuccess) return cleanup(cuda_fail(ce, "host staging stream and events"));
    }

    if ((rc = set_gemm_attributes<lp::kModeNode>()) != LP_OK ||
        (rc = set_gemm_attributes<lp::kModeLse>()) != LP_OK ||
        (rc = set_gemm_attributes<lp::kModeLseEnt>()) != LP_OK ||
        (rc = set_gemm_attributes<lp::kModeGrad>()) != LP_OK)
        return cleanup(rc);
    cudaError_t e;
    if (h->num_lse_tiles > (lp::kCmbMaxThreads << lp::kSegLogMax))
        return cleanup(fail(LP_ERR_UNSUPPORTED, "V too large (at most 2^26 columns)"));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((e = cudaMemsetAsync(h->status, 0, sizeof(int), st)) != cudaSuccess ||
        (e = cudaMemsetAsync(h->is_done, 0, sizeof(unsigned), st)) != cudaSuccess ||
        (e = cudaStreamSynchronize(st)) != cudaSuccess)
        return cleanup(cuda_fail(e, "status init"));
    if (fp8) {
        const int nkb = cfg->H / lp::kQBlock;
        if ((rc = alloc(reinterpret_cast<void**>(&h->wq),
                        static_cast<size_t>(cfg->V) * cfg->H, "wq")) ||
            (rc = alloc(reinterpret_cast<void**>(&h->sw),
                        sizeof(float) * static_cast<size_t>(h->num_vocab_tiles) * nkb, "sw")) ||
            (rc = alloc(reinterpret_cast<void**>(&h->xq), static_cast<size_t>(mt) * cfg->H, "xq")) ||
            (rc = alloc(reinterpret_cast<void**>(&h->sx), sizeof(float) * static_cast<size_t>(mt) * nkb,
                        "sx")))
            return cleanup(rc);
        if ((e = cudaFuncSetAttribute(lp::leaf_gemm_fp8_kernel<lp::kModeLse>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      lp::fp8_smem_bytes())) != cudaSuccess ||
            (e = cudaFuncSetAttribute(lp::leaf_gemm_fp8_kernel<lp::kModeLseEnt>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      lp::fp8_smem_bytes())) != cudaSuccess ||
            (e = cudaFuncSetAttribute(lp::leaf_gemm_fp8_kernel<lp::kModeNode>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      lp::fp8_smem_bytes())) != cudaSuccess)
            return cleanup(cuda_fail(e, "cudaFuncSetAttribute(leaf_gemm_fp8_kernel)"));
        if ((rc = encode_kmajor(&h->tmWq, h->wq, static_cast<uint64_t>(cfg->V), cfg->H, cfg->H,
                                lp::kBM, true)) != LP_OK ||
            (rc = quantize_weights(h, st)) != LP_OK)
            return cleanup(rc);
        if ((e = cudaStreamSynchronize(st)) != cudaSuccess)
            return cleanup(cuda_fail(e, "weight quantisation"));
    }
    h->last_stream = st;
    *out = h;
    return LP_OK;
}
}  // namespace

int lp_init(const lp_config* cfg, const void* W, void* stream, lp_handle** out) {
    return init_impl(cfg, W, stream, out, false);
}

int lp_init_fp8(const lp_config* cfg, const void* W, void* stream, lp_handle** out) {
    return init_impl(cfg, W, stream, out, true);
}

int lp_fp8_requantize(lp_handle* h, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (!h->fp8) return fail(LP_ERR_INVALID_ARG, "not a block-FP8 handle");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    h->last_launches = 1;
    return quantize_weights(h, st);
}

int lp_fp8_quantize_x(lp_handle* h, const void* X, int64_t ldx, int64_t T, uint8_t* xq, float* sx,
                      void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    int rc = check_x(h, X, ldx, T);
    if (rc != LP_OK) return rc;
    if (T > 0 && (xq == nullptr || sx == nullptr))
        return fail(LP_ERR_INVALID_ARG, "xq and sx must not be NULL");
    if (h->cfg.H % lp::kQBlock != 0) return fail(LP_ERR_UNSUPPORTED, "H must be a multiple of 128");
    if (reinterpret_cast<uintptr_t>(xq) % 4 != 0)
        return fail(LP_ERR_INVALID_ARG, "xq must be 4-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    h->last_launches = 0;
    if (T == 0) return LP_OK;
    const int64_t warps = T * (h->cfg.H / lp::kQBlock);
    if (ceil_div(warps, 8) > 0x7fffffff) return fail(LP_ERR_UNSUPPORTED, "T too large");
    lp::quant_x_kernel<<<static_cast<unsigned>(ceil_div(warps, 8)), 256, 0, st>>>(
        static_cast<const uint16_t*>(X), ldx, T, h->cfg.H, xq, h->cfg.H, sx);
    LP_CUDA(cudaGetLastError(), "quant_x_kernel launch");
    h->last_launches = 1;
    return LP_OK;
}

int lp_fp8_weights(const lp_handle* h, const uint8_t** wq, const float** sw) {
    if (h == nullptr || !h->fp8) return fail(LP_ERR_INVALID_ARG, "not a block-FP8 handle");
    if (wq) *wq = h->wq;
    if (sw) *sw = h->sw;
    return LP_OK;
}

namespace {
int logprobs_impl(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids, int64_t T,
                  float* out_logp, float* out_logZ, float* out_entropy, int phase, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    int rc = check_x(h, X, ldx, T);
    if (rc != LP_OK) return rc;
    if (phase < LP_PHASE_AUTO || phase > LP_PHASE_DECODE)
        return fail(LP_ERR_INVALID_ARG, "unknown phase %d", phase);
    h->last_launches = 0;
    if (T == 0) return LP_OK;
    if (ids == nullptr || out_logp == nullptr)
        return fail(LP_ERR_INVALID_ARG, "ids and out_logp must not be NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    const int64_t chunk = h->chunk_rows;
    const uint8_t* xb = static_cast<const uint8_t*>(X);
    for (int64_t r0 = 0; r0 < T; r0 += chunk) {
        const int rows = static_cast<int>(T - r0 < chunk ? T - r0 : chunk);
        rc = logprobs_chunk(h, xb + r0 * ldx * 2, ldx, ids + r0, rows, out_logp + r0,
                            out_logZ ? out_logZ + r0 : nullptr,
                            out_entropy ? out_entropy + r0 : nullptr, st);
        if (rc != LP_OK) return rc;
    }
    return LP_OK;
}
}  // namespace

int lp_logprobs(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids, int64_t T,
                float* out_logp, float* out_logZ, int phase, void* stream) {
    return logprobs_impl(h, X, ldx, ids, T, out_logp, out_logZ, nullptr, phase, stream);
}

int lp_logprobs_entropy(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids, int64_t T,
                        float* out_logp, float* out_logZ, float* out_entropy, int phase,
                        void* stream) {
    if (T > 0 && out_entropy == nullptr)
        return fail(LP_ERR_INVALID_ARG, "out_entropy must not be NULL");
    return logprobs_impl(h, X, ldx, ids, T, out_logp, out_logZ, out_entropy, phase, stream);
}

namespace {
// K splits of the dX GEMM: at most kMaxGradSlices fp32 partials of [rows][H].
constexpr int kMaxGradSlices = 4;

// Slices of K for a launch of `units` pair tiles on `clusters` SM pairs: the count that fills
// the most of its last wave (each slice costs one fp32 partial and its share of the sum); a
// larger count must win by 3 % of the cluster-waves.
int grad_slices(int64_t units, int64_t clusters, int64_t kblocks) {
    int best = 1;
    double best_eff = 0.0;
    for (int sl = 1; sl <= kMaxGradSlices && sl <= kblocks; ++sl) {
        const int64_t w = units * sl;
        const double eff = double(w) / double((w + clusters - 1) / clusters * clusters);
        if (eff > best_eff + 0.03) {
            best = sl;
            best_eff = eff;
        }
    }
    return best;
}

// One backward GEMM, D (+)= A . B over `slices` K slices (slice s writes D + s * slice_stride).
// tmA: K-major (a_mn = false) or MN-major A; tmB: MN-major B.  Returns the slice count used.
int launch_grad_gemm(lp_handle* h, bool a_mn, const CUtensorMap& tmA, const CUtensorMap& tmB,
                     int M, int N, int K, int slices, float* D, int64_t ldd, int64_t slice_stride,
                     int accumulate, cudaStream_t st, int* used) {
    lp::GradGemmParams g{};
    g.M = M;
    g.N = N;
    g.K = K;
    g.num_m = static_cast<int32_t>(ceil_div(M, lp::kGgTileM));
    g.num_n = static_cast<int32_t>(ceil_div(N, lp::kGgTileN));
    const int64_t kblocks = ceil_div(K, lp::kBK);
    const int64_t per = ceil_div(kblocks, slices);
    g.num_slices = static_cast<int32_t>(ceil_div(kblocks, per));  // no empty slice
    g.k_slice = static_cast<int32_t>(per * lp::kBK);
    g.D = D;
    g.ldd = ldd;
    g.slice_stride = slice_stride;
    g.accumulate = accumulate;
    g.status = h->status;
    g.timeout_ns = h->timeout_ns;
    const int64_t units = int64_t(g.num_slices) * g.num_m * g.num_n;
    if (units > 0x7fffffff) return fail(LP_ERR_UNSUPPORTED, "too many tiles in one launch");
    const int64_t clusters = units < h->num_sms / 2 ? units : h->num_sms / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    cfg.blockDim = dim3(lp::kGgThreads);
    cfg.dynamicSmemBytes = lp::kGgSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = a_mn ? cudaLaunchKernelEx(&cfg, lp::grad_gemm_kernel<true>, tmA, tmB, g)
                               : cudaLaunchKernelEx(&cfg, lp::grad_gemm_kernel<false>, tmA, tmB, g);
    LP_CUDA(e, "grad_gemm_kernel launch");
    ++h->last_launches;
    if (used) *used = g.num_slices;
    return LP_OK;
}

}  // namespace

int lp_backward_reserve(lp_handle* h, int64_t max_rows) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (max_rows < 1 || max_rows > (int64_t(1) << 31) - 1)
        return fail(LP_ERR_INVALID_ARG, "max_rows must be in [1, 2^31)");
    if (max_rows <= h->dl_rows) return LP_OK;
    const int64_t ldd = ceil_div(h->cfg.V, 8) * 8;
    void* p = nullptr;
    void* q = nullptr;
    const size_t bytes = sizeof(uint16_t) * static_cast<size_t>(max_rows) * ldd;
    const size_t pbytes =
        sizeof(float) * static_cast<size_t>(kMaxGradSlices) * max_rows * h->cfg.H;
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e == cudaSuccess) {
        e = cudaMalloc(&q, pbytes);
        if (e != cudaSuccess) cudaFree(p);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(LP_ERR_OOM, "backward workspace (%zu + %zu bytes): %s", bytes, pbytes,
                    cudaGetErrorString(e));
    }
    if (h->dl) {
        LP_CUDA(cudaDeviceSynchronize(), "device synchronize");
        cudaFree(h->dl);
        cudaFree(h->grad_part);
        h->ws_bytes -= static_cast<int64_t>(sizeof(uint16_t)) * h->dl_rows * h->ldd +
                       int64_t(sizeof(float)) * kMaxGradSlices * h->dl_rows * h->cfg.H;
    }
    h->dl = static_cast<uint16_t*>(p);
    h->grad_part = static_cast<float*>(q);
    h->dl_rows = max_rows;
    h->ldd = ldd;
    h->ws_bytes += static_cast<int64_t>(bytes + pbytes);
    for (const void* fn : {reinterpret_cast<const void*>(lp::grad_gemm_kernel<false>),
                           reinterpret_cast<const void*>(lp::grad_gemm_kernel<true>)})
        LP_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     lp::kGgSmemBytes),
                "cudaFuncSetAttribute(grad_gemm_kernel)");
    return LP_OK;
}

int lp_logprobs_backward(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids,
                         const float* logZ, const float* grad_logp, int64_t T, float* dX,
                         float* dW, int accumulate, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    int rc = check_x(h, X, ldx, T);
    if (rc != LP_OK) return rc;
    if (h->fp8) return fail(LP_ERR_UNSUPPORTED, "the backward is not built for block-FP8 handles");
    if (h->dl == nullptr)
        return fail(LP_ERR_INVALID_ARG, "call lp_backward_reserve before lp_logprobs_backward");
    if (T > 0 && (ids == nullptr || logZ == nullptr || grad_logp == nullptr))
        return fail(LP_ERR_INVALID_ARG, "ids, logZ and grad_logp must not be NULL");
    if ((dX != nullptr && !aligned16(dX)) || (dW != nullptr && !aligned16(dW)))
        return fail(LP_ERR_INVALID_ARG, "dX and dW must be 16-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    h->last_launches = 0;
    const int H = h->cfg.H, V = h->cfg.V;
    if (dW != nullptr && !accumulate)
        LP_CUDA(cudaMemsetAsync(dW, 0, sizeof(float) * static_cast<size_t>(V) * H, st), "dW clear");
    if (T == 0 || (dX == nullptr && dW == nullptr)) return LP_OK;
    const uint8_t* xb = static_cast<const uint8_t*>(X);
    // W as the B operand of dX: [K = V][N = H], MN-major 64 x 64 boxes (one tensor map for all
    // chunks)
    CUtensorMap tmWB;
    rc = encode_kmajor(&tmWB, h->W, static_cast<uint64_t>(V), H, H, 64);
    if (rc != LP_OK) return rc;
    for (int64_t r0 = 0; r0 < T; r0 += h->dl_rows) {
        const int rows = static_cast<int>(T - r0 < h->dl_rows ? T - r0 : h->dl_rows);
        const void* Xc = xb + r0 * ldx * 2;
        GradArgs ga;
        ga.logZ = logZ + r0;
        ga.gout = grad_logp + r0;
        ga.dl = h->dl;
        ga.ldd = h->ldd;
        rc = launch_leaf_gemm<lp::kModeGrad>(h, Xc, ldx, rows, 0, h->cfg.n_leaves, ids + r0,
                                             nullptr, 0, st, ga);
        if (rc != LP_OK) return rc;
        if (dX != nullptr) {
            // dX = dl W: A = dl [rows][V] K-major (64 x 128 boxes), split over K = V when the
            // tiles alone leave most of the last wave empty
            CUtensorMap tmA;
            rc = encode_kmajor(&tmA, h->dl, static_cast<uint64_t>(rows), V, h->ldd);
            if (rc != LP_OK) return rc;
            const int64_t units = ceil_div(rows, lp::kGgTileM) * ceil_div(H, lp::kGgTileN);
            const int slices = grad_slices(units, h->num_sms / 2, ceil_div(V, lp::kBK));
            float* dXc = dX + r0 * H;
            const bool prof = prof_begin(h, st, LP_PROFILE_GRAD_DX);
            int used = 1;
            rc = launch_grad_gemm(h, false, tmA, tmWB, rows, H, V, slices,
                                  slices == 1 ? dXc : h->grad_part, H, int64_t(rows) * H, 0, st,
                                  &used);
            if (rc != LP_OK) return rc;
            if (used > 1) {
                const int64_t n = int64_t(rows) * H;
                const int64_t blocks = ceil_div(n / 4, 256);
                lp::splitk_sum_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0,
                                        st>>>(h->grad_part, used, n, n, dXc);
                LP_CUDA(cudaGetLastError(), "splitk_sum_kernel launch");
                ++h->last_launches;
            }
            if (prof) LP_CUDA(prof_end(h, st), "profile event");
        }
        if (dW != nullptr) {
            // dW += dl^T X: A = dl seen as [K = rows][M = V], B = X as [K = rows][N = H], both
            // MN-major 64 x 64 boxes; one K slice, so each dW element has one writer per chunk
            CUtensorMap tmA, tmB;
            rc = encode_kmajor(&tmA, h->dl, static_cast<uint64_t>(rows), V, h->ldd, 64);
            if (rc == LP_OK) rc = encode_kmajor(&tmB, Xc, static_cast<uint64_t>(rows), H, ldx, 64);
            if (rc != LP_OK) return rc;
            const bool prof = prof_begin(h, st, LP_PROFILE_GRAD_DW);
            rc = launch_grad_gemm(h, true, tmA, tmB, V, H, rows, 1, dW, H, 0, 1, st, nullptr);
            if (rc != LP_OK) return rc;
            if (prof) LP_CUDA(prof_end(h, st), "profile event");
        }
    }
    return LP_OK;
}

int lp_logprobs_host(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids, int64_t T,
                     float* out_logp, float* out_logZ, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0) return fail(LP_ERR_INVALID_ARG, "T must be >= 0");
    h->last_launches = 0;
    if (T == 0) return LP_OK;
    if (X == nullptr || ids == nullptr || out_logp == nullptr)
        return fail(LP_ERR_INVALID_ARG, "X, ids and out_logp must not be NULL");
    if (ldx < h->cfg.H) return fail(LP_ERR_INVALID_ARG, "ldx must be >= H");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    const int H = h->cfg.H;
    // Pieces: a first piece of kHostFirstPiece rows, then each piece kHostGrowth times the
    // one before, each within one half of the staging buffers (max_tokens rows) and within
    // one pass (chunk_rows).  Only the first copy is exposed: the GEMM of a piece takes far
    // longer than the copy of a piece kHostGrowth times its size at large vocabularies.  With
    // max_tokens < 256 the halves are too small and pieces of max_tokens rows run one after
    // the other in the whole buffer.  A call of at most kHostFirstPiece rows that fits the
    // buffer is one piece: its copy is exposed either way, and a launch of so few rows streams
    // all of W, so every extra piece would read W again.  Pieces are row ranges: the results
    // do not depend on the split.
    const int64_t half = h->cfg.max_tokens / 2 / lp::kBM * lp::kBM;
    const bool one_piece = T <= kHostFirstPiece && T <= h->chunk_rows && T <= h->cfg.max_tokens;
    const int nbuf = half > 0 && !one_piece ? 2 : 1;
    const int64_t cap = nbuf == 2 ? (half < h->chunk_rows ? half : h->chunk_rows) : h->chunk_rows;
    const int64_t slot = nbuf == 2 ? half : 0;  // rows between the two halves
    const uint8_t* xb = static_cast<const uint8_t*>(X);
    uint16_t* xs = static_cast<uint16_t*>(h->x_stage);
    // Pieces are copied on the handle's copy stream, which starts after everything already
    // queued on the caller's stream; a single piece has nothing to overlap and is copied on the
    // caller's stream itself.
    cudaStream_t cs = one_piece ? st : h->copy_stream;
    if (!one_piece) {
        LP_CUDA(cudaEventRecord(h->host_entry, st), "host entry event");
        LP_CUDA(cudaStreamWaitEvent(h->copy_stream, h->host_entry, 0), "host entry wait");
    }
    int32_t launches = 0;
    int i = 0;
    int64_t piece = nbuf == 2 && kHostFirstPiece < cap ? kHostFirstPiece : cap;
    for (int64_t r0 = 0; r0 < T; r0 += piece, ++i) {
        if (i > 0) piece = piece * kHostGrowth < cap ? piece * kHostGrowth : cap;
        const int rows = static_cast<int>(T - r0 < piece ? T - r0 : piece);
        const int b = i % nbuf;
        const int64_t off = b * slot;
        if (i >= nbuf)
            LP_CUDA(cudaStreamWaitEvent(cs, h->stage_free[b], 0), "stage free wait");
        LP_CUDA(cudaMemcpy2DAsync(xs + off * H, static_cast<size_t>(H) * 2, xb + r0 * ldx * 2,
                                  static_cast<size_t>(ldx) * 2, static_cast<size_t>(H) * 2, rows,
                                  cudaMemcpyHostToDevice, cs),
                "X host-to-device copy");
        LP_CUDA(cudaMemcpyAsync(h->ids_stage + off, ids + r0, sizeof(int32_t) * rows,
                                cudaMemcpyHostToDevice, cs),
                "ids host-to-device copy");
        if (!one_piece) {
            LP_CUDA(cudaEventRecord(h->stage_ready[b], cs), "stage ready event");
            LP_CUDA(cudaStreamWaitEvent(st, h->stage_ready[b], 0), "stage ready wait");
        }
        int rc = logprobs_chunk(h, xs + off * H, H, h->ids_stage + off, rows, h->logp_stage + off,
                                h->logz_stage + off, nullptr, st);
        if (rc != LP_OK) return rc;
        launches += h->last_launches;
        h->last_launches = 0;
        if (!one_piece) LP_CUDA(cudaEventRecord(h->stage_free[b], st), "stage free event");
        // the results of this piece leave on the caller's stream, before any later kernel
        // there can overwrite them
        LP_CUDA(cudaMemcpyAsync(out_logp + r0, h->logp_stage + off, sizeof(float) * rows,
                                cudaMemcpyDeviceToHost, st),
                "logp device-to-host copy");
        if (out_logZ)
            LP_CUDA(cudaMemcpyAsync(out_logZ + r0, h->logz_stage + off, sizeof(float) * rows,
                                    cudaMemcpyDeviceToHost, st),
                    "logZ device-to-host copy");
    }
    h->last_launches = launches;
    LP_CUDA(cudaStreamSynchronize(st), "stream synchronize");
    return LP_OK;
}

int lp_logits_partial(lp_handle* h, const void* X, int64_t ldx, int64_t T, int32_t leaf_begin,
                      int32_t leaf_count, float* out, int64_t ldo, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    int rc = check_x(h, X, ldx, T);
    if (rc != LP_OK) return rc;
    if (!is_pow2(leaf_count) || leaf_begin < 0 || leaf_begin % leaf_count != 0 ||
        leaf_begin + leaf_count > h->cfg.n_leaves)
        return fail(LP_ERR_UNSUPPORTED,
                    "leaf range [%d, %d) is not an aligned node of the %d-leaf tree", leaf_begin,
                    leaf_begin + leaf_count, h->cfg.n_leaves);
    h->last_launches = 0;
    if (T == 0) return LP_OK;
    if (out == nullptr || !aligned16(out) || ldo < h->cfg.V || ldo % 4 != 0)
        return fail(LP_ERR_INVALID_ARG, "out must be 16-byte aligned with ldo >= V, ldo %% 4 == 0");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    const int64_t chunk = h->cfg.max_tokens;
    const uint8_t* xb = static_cast<const uint8_t*>(X);
    for (int64_t r0 = 0; r0 < T; r0 += chunk) {
        const int rows = static_cast<int>(T - r0 < chunk ? T - r0 : chunk);
        if (h->fp8) {
            rc = quantize_x_chunk(h, xb + r0 * ldx * 2, ldx, rows, st);
            if (rc == LP_OK)
                rc = launch_fp8_gemm<lp::kModeNode>(h, rows, leaf_begin, leaf_count, nullptr,
                                                    out + r0 * ldo, ldo, st);
        } else {
            rc = launch_leaf_gemm<lp::kModeNode>(h, xb + r0 * ldx * 2, ldx, rows, leaf_begin,
                                                 leaf_count, nullptr, out + r0 * ldo, ldo, st);
        }
        if (rc != LP_OK) return rc;
    }
    return LP_OK;
}

int lp_logprobs_from_partials(lp_handle* h, const float* partials, int32_t n_parts,
                              int64_t part_stride, int64_t ldp, const int32_t* ids, int64_t T,
                              float* out_logp, float* out_logZ, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (!(n_parts == 1 || n_parts == 2 || n_parts == 4 || n_parts == 8) ||
        h->cfg.n_leaves % n_parts != 0)
        return fail(LP_ERR_UNSUPPORTED, "n_parts must be 1, 2, 4 or 8 and divide n_leaves");
    if (T < 0 || T > h->cfg.max_tokens)
        return fail(LP_ERR_INVALID_ARG, "T must be in [0, max_tokens]");
    h->last_launches = 0;
    if (T == 0) return LP_OK;
    if (partials == nullptr || ids == nullptr || out_logp == nullptr)
        return fail(LP_ERR_INVALID_ARG, "partials, ids and out_logp must not be NULL");
    if (ldp < h->cfg.V || part_stride < ldp * T)
        return fail(LP_ERR_INVALID_ARG, "need ldp >= V and part_stride >= ldp * T");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    int rc = launch_partials_lse(h, partials, n_parts, part_stride, ldp, ids, static_cast<int>(T),
                                 false, st);
    if (rc != LP_OK) return rc;
    return launch_combine(h, ids, static_cast<int>(T), out_logp, out_logZ, nullptr, st);
}

int lp_importance_weights(lp_handle* h, const float* logp_pi, const float* logp_mu,
                          const uint8_t* mask, int64_t T, float* out_w, double* out_d3,
                          int64_t* out_nvalid, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0 || T > kMaxIsTokens) return fail(LP_ERR_INVALID_ARG, "T must be in [0, 2^31)");
    if (out_d3 == nullptr) return fail(LP_ERR_INVALID_ARG, "out_d3 must not be NULL");
    if (T > 0 && (logp_pi == nullptr || logp_mu == nullptr || out_w == nullptr))
        return fail(LP_ERR_INVALID_ARG, "logp_pi, logp_mu and out_w must not be NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    h->last_launches = 0;
    const int64_t nblk = ceil_div(T, lp::kIsBlock);
    if (nblk > 0) {
        // one launch: weights, block partials and (in the last block to finish) the fixed tree
        lp::IsFusedParams q{{logp_pi, logp_mu, mask, T, out_w, h->blk_sum, h->blk_cnt},
                            static_cast<int>(nblk), h->is_done, out_d3, out_nvalid};
        lp::is_fused_kernel<<<static_cast<unsigned>(nblk), lp::kIsThreads, 0, st>>>(q);
        LP_CUDA(cudaGetLastError(), "is_fused_kernel launch");
    } else {
        lp::is_final_kernel<<<1, 1024, 0, st>>>(h->blk_sum, h->blk_cnt, 0, out_d3, out_nvalid);
        LP_CUDA(cudaGetLastError(), "is_final_kernel launch");
    }
    ++h->last_launches;
    return LP_OK;
}

static_assert(sizeof(long long) == sizeof(int64_t), "block counts cross the ABI as int64_t");

int lp_vocab_partials(lp_handle* h, const void* X, int64_t ldx, const int32_t* ids_local,
                      int64_t T, void* out_ms, int64_t ld_ms, float* out_zy, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (h->fp8 || h->cfg.tp_slices != 1)
        return fail(LP_ERR_UNSUPPORTED, "vocabulary partials come from a bf16 handle with "
                                        "tp_slices = 1");
    int rc = check_x(h, X, ldx, T);
    if (rc != LP_OK) return rc;
    if (T > h->cfg.max_tokens) return fail(LP_ERR_INVALID_ARG, "T must be <= max_tokens");
    h->last_launches = 0;
    if (T == 0) return LP_OK;
    if (ids_local == nullptr || out_ms == nullptr || out_zy == nullptr || ld_ms < T ||
        !aligned16(out_ms))
        return fail(LP_ERR_INVALID_ARG,
                    "ids_local, out_ms (16-byte aligned, ld_ms >= T) and out_zy are required");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    const int rows = static_cast<int>(T);
    // the fused leaf GEMM of this slice; a row whose sampled id lies outside the slice is
    // not captured (its id belongs to another rank) and keeps the NaN written here
    LP_CUDA(cudaMemsetAsync(h->zy, 0xFF, sizeof(float) * static_cast<size_t>(rows), st),
            "sampled logits fill");
    rc = launch_leaf_gemm<lp::kModeLse>(h, X, ldx, rows, 0, h->cfg.n_leaves, ids_local, nullptr,
                                        0, st);
    if (rc != LP_OK) return rc;
    LP_CUDA(cudaMemcpy2DAsync(out_ms, sizeof(float2) * static_cast<size_t>(ld_ms), h->ws_ms,
                              sizeof(float2) * static_cast<size_t>(h->cfg.max_tokens),
                              sizeof(float2) * static_cast<size_t>(rows),
                              static_cast<size_t>(h->num_lse_tiles), cudaMemcpyDeviceToDevice, st),
            "tile partials copy");
    LP_CUDA(cudaMemcpyAsync(out_zy, h->zy, sizeof(float) * static_cast<size_t>(rows),
                            cudaMemcpyDeviceToDevice, st),
            "sampled logits copy");
    return LP_OK;
}

int lp_logprobs_from_vocab_partials(lp_handle* h, int32_t V_full, const void* ms, int64_t ld_ms,
                                    const float* zy, const int32_t* ids, int64_t T,
                                    float* out_logp, float* out_logZ, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (V_full <= 0) return fail(LP_ERR_INVALID_ARG, "V_full must be positive");
    const int64_t tiles = ceil_div(static_cast<int64_t>(V_full), lp::kLT);
    if (tiles > (lp::kCmbMaxThreads << lp::kSegLogMax))
        return fail(LP_ERR_UNSUPPORTED, "V too large (at most 2^26 columns)");
    if (T < 0 || T > (int64_t(1) << 31) - 1) return fail(LP_ERR_INVALID_ARG, "T out of range");
    h->last_launches = 0;
    if (T == 0) return LP_OK;
    if (ms == nullptr || zy == nullptr || ids == nullptr || out_logp == nullptr || ld_ms < T ||
        !aligned16(ms))
        return fail(LP_ERR_INVALID_ARG, "ms (16-byte aligned, ld_ms >= T), zy, ids and out_logp "
                                        "are required");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    // the fixed pairwise tree over all tiles of the full vocabulary, as in lp_logprobs
    const int rows = static_cast<int>(T);
    lp::CombineParams c{};
    c.ws_ms = static_cast<const float2*>(ms);
    c.ws_ld = ld_ms;
    c.zy = zy;
    c.ids = ids;
    c.T = rows;
    c.V = V_full;
    c.num_tiles = static_cast<int32_t>(tiles);
    const lp::CombineLayout lay = lp::combine_layout(rows, c.num_tiles, h->num_sms);
    c.rows = lay.rows;
    c.seg_log = lay.seg_log;
    c.nseg = lay.nseg;
    c.out_logp = out_logp;
    c.out_logZ = out_logZ;
    c.status = h->status;
    const dim3 grid(static_cast<unsigned>(ceil_div(rows, lay.rows)));
    const dim3 block(static_cast<unsigned>(lay.rows * lay.nseg));
    lp::lse_combine_kernel<false><<<grid, block, sizeof(float2) * lay.rows * lay.nseg, st>>>(c);
    LP_CUDA(cudaGetLastError(), "lse_combine_kernel launch");
    ++h->last_launches;
    return LP_OK;
}

int lp_importance_weights_partials(lp_handle* h, const float* logp_pi, const float* logp_mu,
                                   const uint8_t* mask, int64_t T, float* out_w,
                                   double* out_blk_sum, int64_t* out_blk_cnt, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0 || T > kMaxIsTokens) return fail(LP_ERR_INVALID_ARG, "T must be in [0, 2^31)");
    h->last_launches = 0;
    if (T == 0) return LP_OK;
    if (logp_pi == nullptr || logp_mu == nullptr || out_w == nullptr || out_blk_sum == nullptr ||
        out_blk_cnt == nullptr)
        return fail(LP_ERR_INVALID_ARG,
                    "logp_pi, logp_mu, out_w, out_blk_sum and out_blk_cnt must not be NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    const int64_t nblk = ceil_div(T, lp::kIsBlock);
    // the same block kernel as lp_importance_weights, its partials in the caller's arrays
    lp::IsParams p{logp_pi, logp_mu, mask, T, out_w, out_blk_sum,
                   reinterpret_cast<long long*>(out_blk_cnt)};
    lp::is_block_kernel<<<static_cast<unsigned>(nblk), lp::kIsThreads, 0, st>>>(p);
    LP_CUDA(cudaGetLastError(), "is_block_kernel launch");
    ++h->last_launches;
    return LP_OK;
}

int lp_d3_from_partials(lp_handle* h, const double* blk_sum, const int64_t* blk_cnt,
                        int64_t num_blocks, double* out_d3, int64_t* out_nvalid, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (num_blocks < 0 || num_blocks > ceil_div(kMaxIsTokens, lp::kIsBlock))
        return fail(LP_ERR_INVALID_ARG, "num_blocks must be in [0, 2^21]");
    if (out_d3 == nullptr) return fail(LP_ERR_INVALID_ARG, "out_d3 must not be NULL");
    if (num_blocks > 0 && (blk_sum == nullptr || blk_cnt == nullptr))
        return fail(LP_ERR_INVALID_ARG, "blk_sum and blk_cnt must not be NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    h->last_launches = 0;
    // the fixed fp64 tree over the gathered blocks, as in lp_importance_weights
    lp::is_final_kernel<<<1, 1024, 0, st>>>(blk_sum, reinterpret_cast<const long long*>(blk_cnt),
                                            static_cast<int>(num_blocks), out_d3, out_nvalid);
    LP_CUDA(cudaGetLastError(), "is_final_kernel launch");
    ++h->last_launches;
    return LP_OK;
}

int lp_acceptance_stats(lp_handle* h, const float* logp_a, const float* logp_b,
                        const uint8_t* mask, int64_t T, double* out_stats, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0 || T > kMaxIsTokens) return fail(LP_ERR_INVALID_ARG, "T must be in [0, 2^31)");
    if (out_stats == nullptr) return fail(LP_ERR_INVALID_ARG, "out_stats must not be NULL");
    if (T > 0 && (logp_a == nullptr || logp_b == nullptr))
        return fail(LP_ERR_INVALID_ARG, "logp_a and logp_b must not be NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    h->last_launches = 0;
    const int64_t nblk = ceil_div(T, lp::kIsBlock);
    lp::StatsParams p{logp_a, logp_b, mask, T, h->blk_sum, h->stat_blk,
                      h->stat_blk + h->max_is_blocks, h->stat_max, h->blk_cnt};
    if (nblk > 0) {
        // one launch: block partials, the statistics in the last block to finish
        lp::stats_fused_kernel<<<static_cast<unsigned>(nblk), lp::kIsThreads, 0, st>>>(
            p, static_cast<int>(nblk), h->is_done, out_stats);
        LP_CUDA(cudaGetLastError(), "stats_fused_kernel launch");
    } else {
        lp::stats_final_kernel<<<1, 1024, 0, st>>>(p, 0, out_stats);
        LP_CUDA(cudaGetLastError(), "stats_final_kernel launch");
    }
    ++h->last_launches;
    return LP_OK;
}

int lp_acceptance_stats_partials(lp_handle* h, const float* logp_a, const float* logp_b,
                                 const uint8_t* mask, int64_t T, double* out_blk,
                                 float* out_blk_max, int64_t* out_blk_cnt, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0 || T > kMaxIsTokens) return fail(LP_ERR_INVALID_ARG, "T must be in [0, 2^31)");
    h->last_launches = 0;
    if (T == 0) return LP_OK;
    if (logp_a == nullptr || logp_b == nullptr || out_blk == nullptr || out_blk_max == nullptr ||
        out_blk_cnt == nullptr)
        return fail(LP_ERR_INVALID_ARG,
                    "logp_a, logp_b, out_blk, out_blk_max and out_blk_cnt must not be NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    const int64_t nblk = ceil_div(T, lp::kIsBlock);
    // the block kernel of lp_acceptance_stats, its partials in the caller's arrays
    lp::StatsParams p{logp_a,          logp_b,          mask,        T,
                      out_blk,         out_blk + nblk,  out_blk + 2 * nblk, out_blk_max,
                      reinterpret_cast<long long*>(out_blk_cnt)};
    lp::stats_block_kernel<<<static_cast<unsigned>(nblk), lp::kIsThreads, 0, st>>>(p);
    LP_CUDA(cudaGetLastError(), "stats_block_kernel launch");
    ++h->last_launches;
    return LP_OK;
}

int lp_acceptance_stats_from_partials(lp_handle* h, const double* blk, const float* blk_max,
                                      const int64_t* blk_cnt, int64_t num_blocks,
                                      double* out_stats, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (num_blocks < 0 || num_blocks > ceil_div(kMaxIsTokens, lp::kIsBlock))
        return fail(LP_ERR_INVALID_ARG, "num_blocks must be in [0, 2^21]");
    if (out_stats == nullptr) return fail(LP_ERR_INVALID_ARG, "out_stats must not be NULL");
    if (num_blocks > 0 && (blk == nullptr || blk_max == nullptr || blk_cnt == nullptr))
        return fail(LP_ERR_INVALID_ARG, "blk, blk_max and blk_cnt must not be NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    h->last_launches = 0;
    // the final kernel only reads the block arrays
    double* b = const_cast<double*>(blk);
    lp::StatsParams p{nullptr, nullptr, nullptr, 0, b, b + num_blocks, b + 2 * num_blocks,
                      const_cast<float*>(blk_max),
                      reinterpret_cast<long long*>(const_cast<int64_t*>(blk_cnt))};
    lp::stats_final_kernel<<<1, 1024, 0, st>>>(p, static_cast<int>(num_blocks), out_stats);
    LP_CUDA(cudaGetLastError(), "stats_final_kernel launch");
    ++h->last_launches;
    return LP_OK;
}

int lp_reinforce_zero(lp_handle* h, const float* logp_pi, const float* logp_mu,
                      const uint8_t* mask, int64_t T, const int64_t* seq_offsets, int64_t B,
                      const float* rewards, int32_t group_size, const lp_rz_options* opt,
                      float* out_w_hat, float* out_grad, double* out_adv, double* out_loss,
                      int64_t* out_n_kept, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0 || T > kMaxIsTokens) return fail(LP_ERR_INVALID_ARG, "T must be in [0, 2^31)");
    if (B < 0 || B > h->max_is_blocks)
        return fail(LP_ERR_INVALID_ARG, "B must be in [0, %lld]", (long long)h->max_is_blocks);
    if (group_size < 1 || (B > 0 && B % group_size != 0))
        return fail(LP_ERR_INVALID_ARG, "group_size must be >= 1 and divide B");
    if (out_loss == nullptr) return fail(LP_ERR_INVALID_ARG, "out_loss must not be NULL");
    if (B > 0 && (seq_offsets == nullptr || rewards == nullptr))
        return fail(LP_ERR_INVALID_ARG, "seq_offsets and rewards must not be NULL");
    if (T > 0 && (logp_pi == nullptr || logp_mu == nullptr || out_grad == nullptr))
        return fail(LP_ERR_INVALID_ARG, "logp_pi, logp_mu and out_grad must not be NULL");
    lp::RzParams p{};
    p.logp_pi = logp_pi;
    p.logp_mu = logp_mu;
    p.mask = mask;
    p.T = T;
    p.offs = seq_offsets;
    p.B = B;
    p.rewards = rewards;
    p.G = group_size;
    p.flags = 0;
    p.tis_cap = INFINITY;
    p.tok_lo = -INFINITY;
    p.tok_hi = INFINITY;
    p.seq_lo = -INFINITY;
    p.seq_hi = INFINITY;
    if (opt != nullptr) {
        if (opt->flags & ~(LP_RZ_TIS | LP_RZ_TOKEN_GATE | LP_RZ_SEQ_GATE))
            return fail(LP_ERR_INVALID_ARG, "unknown flag in lp_rz_options.flags");
        if ((opt->flags & LP_RZ_TIS) && !(opt->tis_cap > 0.0f))
            return fail(LP_ERR_INVALID_ARG, "tis_cap must be > 0");
        if ((opt->flags & LP_RZ_TOKEN_GATE) && !(opt->token_log_lo <= opt->token_log_hi))
            return fail(LP_ERR_INVALID_ARG, "token gate needs token_log_lo <= token_log_hi");
        if ((opt->flags & LP_RZ_SEQ_GATE) && !(opt->seq_log_lo <= opt->seq_log_hi))
            return fail(LP_ERR_INVALID_ARG, "sequence gate needs seq_log_lo <= seq_log_hi");
        p.flags = opt->flags;
        p.tis_cap = opt->tis_cap;
        p.tok_lo = opt->token_log_lo;
        p.tok_hi = opt->token_log_hi;
        p.seq_lo = opt->seq_log_lo;
        p.seq_hi = opt->seq_log_hi;
    }
    p.out_w_hat = out_w_hat;
    p.out_grad = out_grad;
    p.out_adv = out_adv;
    p.seq_term = h->blk_sum;
    p.seq_kept = h->blk_cnt;
    p.status = h->status;
    p.done = h->is_done;
    p.out_loss = out_loss;
    p.out_kept = out_n_kept;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    h->last_launches = 0;
    if (B > 0) {
        // one launch: a block per response, the loss's tree in the last block to finish
        lp::rz_seq_kernel<<<static_cast<unsigned>(B), lp::kRzThreads, 0, st>>>(p);
        LP_CUDA(cudaGetLastError(), "rz_seq_kernel launch");
    } else {
        lp::rz_final_kernel<<<1, 1024, 0, st>>>(h->blk_sum, h->blk_cnt, 0, out_loss, out_n_kept);
        LP_CUDA(cudaGetLastError(), "rz_final_kernel launch");
    }
    ++h->last_launches;
    return LP_OK;
}

int lp_importance_weights_host(lp_handle* h, const float* logp_pi, const float* logp_mu,
                               const uint8_t* mask, int64_t T, float* out_w, double* out_d3,
                               int64_t* out_nvalid, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0 || T > kMaxIsTokens) return fail(LP_ERR_INVALID_ARG, "T must be in [0, 2^31)");
    if (out_d3 == nullptr) return fail(LP_ERR_INVALID_ARG, "out_d3 must not be NULL");
    if (T > 0 && (logp_pi == nullptr || logp_mu == nullptr || out_w == nullptr))
        return fail(LP_ERR_INVALID_ARG, "logp_pi, logp_mu and out_w must not be NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    h->last_launches = 0;
    // Stage in passes of kIsStage tokens (whole 1024-token blocks), so the block
    // partials and the tree over them are those of one device call.
    const int64_t chunk = kIsStage;
    float* a = h->is_stage;
    float* b = h->is_stage + kIsStage;
    float* wbuf = h->is_stage + 2 * kIsStage;
    uint8_t* mbuf = h->is_mask_stage;
    const int64_t nblk = ceil_div(T, lp::kIsBlock);
    for (int64_t t0 = 0; t0 < T; t0 += chunk) {
        const int64_t n = T - t0 < chunk ? T - t0 : chunk;
        LP_CUDA(cudaMemcpyAsync(a, logp_pi + t0, sizeof(float) * n, cudaMemcpyHostToDevice, st),
                "logp_pi host-to-device copy");
        LP_CUDA(cudaMemcpyAsync(b, logp_mu + t0, sizeof(float) * n, cudaMemcpyHostToDevice, st),
                "logp_mu host-to-device copy");
        if (mask)
            LP_CUDA(cudaMemcpyAsync(mbuf, mask + t0, n, cudaMemcpyHostToDevice, st),
                    "mask host-to-device copy");
        lp::IsParams p{a, b, mask ? mbuf : nullptr, n, wbuf, h->blk_sum + t0 / lp::kIsBlock,
                       h->blk_cnt + t0 / lp::kIsBlock};
        lp::is_block_kernel<<<static_cast<unsigned>(ceil_div(n, lp::kIsBlock)), lp::kIsThreads, 0,
                              st>>>(p);
        LP_CUDA(cudaGetLastError(), "is_block_kernel launch");
        ++h->last_launches;
        LP_CUDA(cudaMemcpyAsync(out_w + t0, wbuf, sizeof(float) * n, cudaMemcpyDeviceToHost, st),
                "w device-to-host copy");
    }
    double* d3_dev = h->scalars;
    lp::is_final_kernel<<<1, 1024, 0, st>>>(h->blk_sum, h->blk_cnt, static_cast<int>(nblk), d3_dev,
                                            reinterpret_cast<int64_t*>(d3_dev + 1));
    LP_CUDA(cudaGetLastError(), "is_final_kernel launch");
    ++h->last_launches;
    // D3 and n_valid land in pinned memory (a copy to pageable memory would be staged)
    double* res = h->host_scalars;
    LP_CUDA(cudaMemcpyAsync(res, d3_dev, 2 * sizeof(double), cudaMemcpyDeviceToHost, st),
            "D3 copy");
    LP_CUDA(cudaStreamSynchronize(st), "stream synchronize");
    *out_d3 = res[0];
    if (out_nvalid) std::memcpy(out_nvalid, &res[1], sizeof(int64_t));
    return LP_OK;
}

int lp_profile_enable(lp_handle* h, int enable) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (enable && h->prof_events.empty()) {
        h->prof_events.resize(2 * kProfPairs);
        h->prof_kind.assign(kProfPairs, 0);
        for (auto& e : h->prof_events) LP_CUDA(cudaEventCreate(&e), "cudaEventCreate");
    }
    h->profiling = enable != 0;
    h->prof_used = 0;
    return LP_OK;
}

int lp_profile_read_kind(lp_handle* h, int kind, double* ms_total, int32_t* count) {
    if (h == nullptr || ms_total == nullptr)
        return fail(LP_ERR_INVALID_ARG, "handle and ms_total must not be NULL");
    double total = 0.0;
    int32_t n = 0;
    for (int i = 0; i < h->prof_used; ++i) {
        if (h->prof_kind[i] != kind) continue;
        LP_CUDA(cudaEventSynchronize(h->prof_events[2 * i + 1]), "cudaEventSynchronize");
        float ms = 0.0f;
        LP_CUDA(cudaEventElapsedTime(&ms, h->prof_events[2 * i], h->prof_events[2 * i + 1]),
                "cudaEventElapsedTime");
        total += ms;
        ++n;
    }
    *ms_total = total;
    if (count) *count = n;
    return LP_OK;
}

int lp_profile_read(lp_handle* h, double* gemm_ms_total, int32_t* gemm_launches) {
    if (h == nullptr || gemm_ms_total == nullptr)
        return fail(LP_ERR_INVALID_ARG, "handle and gemm_ms_total must not be NULL");
    const int rc = lp_profile_read_kind(h, LP_PROFILE_LEAF_GEMM, gemm_ms_total, gemm_launches);
    h->prof_used = 0;
    return rc;
}

int lp_selftest_wait_timeout(lp_handle* h, int64_t timeout_us, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    if (timeout_us < 1 || timeout_us > 2000000)
        return fail(LP_ERR_INVALID_ARG, "timeout_us must be in [1, 2e6]");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    h->last_stream = st;
    lp::wait_selftest_kernel<<<1, 32, 0, st>>>(h->status, static_cast<uint64_t>(timeout_us) * 1000u);
    LP_CUDA(cudaGetLastError(), "wait_selftest_kernel launch");
    h->last_launches = 1;
    return LP_OK;
}

int lp_check(lp_handle* h) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    LP_CUDA(cudaStreamSynchronize(h->last_stream), "stream synchronize");
    int st = 0;
    LP_CUDA(cudaMemcpy(&st, h->status, sizeof(int), cudaMemcpyDeviceToHost), "status read");
    if (st & lp::kStatusTimeout)
        return fail(LP_ERR_TIMEOUT, "a device-side bounded wait expired; the kernel returned early");
    if (st & lp::kStatusBadId)
        return fail(LP_ERR_INVALID_ARG, "a sampled id was outside [0, V); its logprob is NaN");
    if (st & lp::kStatusBadOffsets)
        return fail(LP_ERR_INVALID_ARG,
                    "a response's token range [offs[i], offs[i+1]) was not inside [0, T)");
    return LP_OK;
}

int lp_clear_status(lp_handle* h, void* stream) {
    if (h == nullptr) return fail(LP_ERR_INVALID_ARG, "handle is NULL");
    LP_CUDA(cudaMemsetAsync(h->status, 0, sizeof(int), static_cast<cudaStream_t>(stream)),
            "status clear");
    return LP_OK;
}

}  // extern "C"
