// lp_noalloc.cu -- lp_logprobs_noalloc: the fused sampled-token logprob path for callers
// that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: runtimes whose device memory is planned ahead by
// their own allocator (which must not see allocations behind its back), and hosts that
// forbid allocation after start-up (a fixed memory budget checked once).  For them this
// entry point needs no handle and no workspace: the per-tile (max, sum-exp)
// partials, the sampled logits and the status word live in one file-scope device array
// of fixed size, g_lp_noalloc_scratch, which every GPU that loads the library holds until
// the process exits.  The caller still passes the inputs and the outputs.
//
// The kernels are the same templates as the handle-based path (same per-element
// arithmetic, so the results are bit-identical to lp_logprobs with tp_slices = 1).
//
// A bounded in-kernel wait that expires sets the timeout bit of the status word in the
// scratch; a last small kernel of the same call then turns every row's logp and logZ into
// NaN, so the caller sees it in the outputs without reading the status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>

#include "kernels.cuh"
#include "lp.h"

namespace {

constexpr int kBand = 32;
// Capacity of the static scratch (stated in include/lp.h):
constexpr int64_t kNoallocMaxTileRows = int64_t(1) << 20;  // T * ceil(V/64) (max, sum) pairs
constexpr int64_t kNoallocMaxRows = int64_t(1) << 15;      // T per call
constexpr size_t kMsBytes = static_cast<size_t>(kNoallocMaxTileRows) * sizeof(float2);  // 8 MiB
constexpr size_t kZyBytes = static_cast<size_t>(kNoallocMaxRows) * sizeof(float);       // 128 KiB
constexpr size_t kStatusBytes = 256;
constexpr size_t kScratchBytes = kMsBytes + kZyBytes + kStatusBytes;
constexpr int kMaxDevices = 64;

}  // namespace

// The scratch.  In host code this name is only a host-side stand-in for the device array:
// its address must come from cudaGetSymbolAddress (done once per device below).
static __device__ __align__(256) unsigned char g_lp_noalloc_scratch[kScratchBytes];

namespace {

thread_local std::string g_noalloc_error = "no error";

int nfail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_noalloc_error = buf;
    return code;
}

struct DeviceSetup {
    std::once_flag once;
    int status = LP_OK;
    std::string message;
    unsigned char* scratch = nullptr;  // device address of g_lp_noalloc_scratch on this device
    int num_sms = 0;
    uint64_t timeout_ns = 2000000000ull;  // bound on every in-kernel wait (LP_WAIT_TIMEOUT_MS)
    int status_init = 0;                  // the status word at the start of each call
};
DeviceSetup g_setup[kMaxDevices];

// Once per device, with that device current: resolve the scratch array's device address,
// check the architecture, raise the kernels' dynamic shared-memory limits and read the wait
// limit from the environment.  Nothing here allocates.
void setup_device(int dev, DeviceSetup& s) {
    if (const char* v = std::getenv("LP_WAIT_TIMEOUT_MS")) {
        const long long ms = std::atoll(v);
        if (ms > 0) s.timeout_ns = static_cast<uint64_t>(ms) * 1000000ull;
    }
    // test hook: every call starts as if one of its waits had expired, so the tests can check
    // what a caller sees on a timeout without making a GPU wait run out
    if (const char* v = std::getenv("LP_TEST_NOALLOC_MARK_TIMEOUT")) {
        if (v[0] == '1') s.status_init = lp::kStatusTimeout;
    }
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, dev);
    if (e == cudaSuccess && !(prop.major == 10 && prop.minor == 3)) {
        s.status = LP_ERR_UNSUPPORTED;
        s.message = "lp_logprobs_noalloc is built for sm_103a (GB300)";
        return;
    }
    void* ptr = nullptr;
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&ptr, g_lp_noalloc_scratch);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(lp::leaf_gemm_kernel<lp::kModeLse, 1>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 lp::gemm_smem_bytes(1));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(lp::leaf_gemm_kernel<lp::kModeLse, 2>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 lp::gemm_smem_bytes(2));
    if (e != cudaSuccess) {
        cudaGetLastError();
        s.status = LP_ERR_CUDA;
        s.message = std::string("no-alloc set-up failed: ") + cudaGetErrorString(e);
        return;
    }
    s.scratch = static_cast<unsigned char*>(ptr);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int encode(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K, uint64_t ld,
           uint32_t box_rows) {
    auto enc = encoder();
    if (enc == nullptr) return nfail(LP_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(lp::kBK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return nfail(LP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return LP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The status word's value at the start of a call (0, or the test hook's mark).
__global__ void noalloc_status_init_kernel(int* status, int value) { *status = value; }

// Last step of a call: if a bounded wait expired (timeout bit), every row's outputs become NaN.
__global__ void noalloc_timeout_nan_kernel(const int* status, float* logp, float* logZ, int T) {
    if ((*status & lp::kStatusTimeout) == 0) return;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T; i += gridDim.x * blockDim.x) {
        logp[i] = NAN;
        if (logZ != nullptr) logZ[i] = NAN;
    }
}

}  // namespace

extern "C" {

LP_API const char* lp_noalloc_last_error(void) { return g_noalloc_error.c_str(); }

LP_API int lp_logprobs_noalloc(const void* W, int32_t H, int32_t V, int32_t n_leaves, const void* X,
                        int64_t ldx, const int32_t* ids, int64_t T, float* out_logp,
                        float* out_logZ, void* stream) {
    // ---- host-side checks (before any CUDA call)
    if (!(n_leaves == 1 || n_leaves == 2 || n_leaves == 4 || n_leaves == 8))
        return nfail(LP_ERR_UNSUPPORTED, "n_leaves must be 1, 2, 4 or 8 (got %d)", n_leaves);
    if (H <= 0 || V <= 0 || H % (lp::kBK * n_leaves) != 0)
        return nfail(LP_ERR_UNSUPPORTED, "need H > 0, V > 0 and H %% (64 * n_leaves) == 0");
    if (T < 0) return nfail(LP_ERR_INVALID_ARG, "T must be >= 0");
    const int64_t nb = (static_cast<int64_t>(V) + lp::kLT - 1) / lp::kLT;  // log-sum-exp tiles
    if (T > kNoallocMaxRows || T * nb > kNoallocMaxTileRows)
        return nfail(LP_ERR_INVALID_ARG,
                     "T = %lld rows x %lld log-sum-exp tiles exceeds the static scratch "
                     "(at most %lld rows and %lld row-tiles; use lp_logprobs with a handle)",
                     (long long)T, (long long)nb, (long long)kNoallocMaxRows,
                     (long long)kNoallocMaxTileRows);
    if (T == 0) return LP_OK;
    if (W == nullptr || X == nullptr || ids == nullptr || out_logp == nullptr)
        return nfail(LP_ERR_INVALID_ARG, "W, X, ids and out_logp must not be NULL");
    if (!aligned16(W) || !aligned16(X) || ldx < H || ldx % 8 != 0)
        return nfail(LP_ERR_INVALID_ARG, "W and X must be 16-byte aligned, ldx >= H, ldx %% 8 == 0");
    if (nb > (int64_t(lp::kCmbMaxThreads) << lp::kSegLogMax))
        return nfail(LP_ERR_UNSUPPORTED, "V too large (at most 2^26 columns)");

    // ---- once-per-device set-up (the first call on a device; it must precede any capture)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return nfail(LP_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return nfail(LP_ERR_UNSUPPORTED, "device index too large");
    DeviceSetup& s = g_setup[dev];
    std::call_once(s.once, setup_device, dev, std::ref(s));
    if (s.status != LP_OK) return nfail(s.status, "%s", s.message.c_str());

    float2* ws_ms = reinterpret_cast<float2*>(s.scratch);
    float* zy = reinterpret_cast<float*>(s.scratch + kMsBytes);
    int* status = reinterpret_cast<int*>(s.scratch + kMsBytes + kZyBytes);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    CUtensorMap tmW, tmX;
    const int rows = static_cast<int>(T);
    const uint32_t box = rows >= lp::kBM ? lp::kBM : static_cast<uint32_t>((rows + 7) / 8 * 8);
    int rc = encode(&tmW, W, static_cast<uint64_t>(V), H, H, lp::kBM);
    if (rc == LP_OK) rc = encode(&tmX, X, static_cast<uint64_t>(rows), H, ldx, box);
    if (rc != LP_OK) return rc;

    // the status word starts at zero for every call (the array keeps the last call's data)
    noalloc_status_init_kernel<<<1, 1, 0, st>>>(status, s.status_init);
    e = cudaGetLastError();
    if (e != cudaSuccess) return nfail(LP_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));

    lp::GemmParams p{};
    p.T = rows;
    p.V = V;
    p.leaf_len = H / n_leaves;
    p.leaf_begin = 0;
    p.leaf_count = n_leaves;
    p.num_row_tiles = (rows + lp::kBM - 1) / lp::kBM;
    p.num_vocab_tiles = static_cast<int32_t>((V + lp::kVT - 1) / lp::kVT);
    p.num_lse_tiles = static_cast<int32_t>(nb);
    p.band = kBand;
    p.x_box_rows = static_cast<int32_t>(box);
    p.ids = ids;
    p.ws_ms = ws_ms;
    p.ws_ld = T;
    p.zy = zy;
    p.out = nullptr;
    p.ldo = 0;
    p.status = status;
    p.timeout_ns = s.timeout_ns;
    const int64_t tiles = static_cast<int64_t>(p.num_row_tiles) * p.num_vocab_tiles;
    const int grid = static_cast<int>(tiles < s.num_sms ? tiles : s.num_sms);
    if (p.leaf_len % (2 * lp::kBK) == 0)
        lp::leaf_gemm_kernel<lp::kModeLse, 2><<<grid, lp::kGemmThreads, lp::gemm_smem_bytes(2), st>>>(tmX, tmW, tmX, p);
    else
        lp::leaf_gemm_kernel<lp::kModeLse, 1><<<grid, lp::kGemmThreads, lp::gemm_smem_bytes(1), st>>>(tmX, tmW, tmX, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return nfail(LP_ERR_CUDA, "leaf_gemm_kernel launch: %s", cudaGetErrorString(e));

    lp::CombineParams c{};
    c.ws_ms = ws_ms;
    c.ws_ld = T;
    c.zy = zy;
    c.ids = ids;
    c.T = rows;
    c.V = V;
    c.num_tiles = static_cast<int32_t>(nb);
    const lp::CombineLayout lay = lp::combine_layout(rows, c.num_tiles, s.num_sms);
    c.rows = lay.rows;
    c.seg_log = lay.seg_log;
    c.nseg = lay.nseg;
    c.out_logp = out_logp;
    c.out_logZ = out_logZ;
    c.status = status;
    lp::lse_combine_kernel<false><<<static_cast<unsigned>((rows + lay.rows - 1) / lay.rows),
                             static_cast<unsigned>(lay.rows * lay.nseg),
                             sizeof(float2) * static_cast<size_t>(lay.rows) * lay.nseg, st>>>(c);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return nfail(LP_ERR_CUDA, "lse_combine_kernel launch: %s", cudaGetErrorString(e));
    const int nan_blocks = static_cast<int>((rows + 255) / 256 < 64 ? (rows + 255) / 256 : 64);
    noalloc_timeout_nan_kernel<<<nan_blocks, 256, 0, st>>>(status, out_logp, out_logZ, rows);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return nfail(LP_ERR_CUDA, "timeout check launch: %s", cudaGetErrorString(e));
    return LP_OK;
}

}  // extern "C"
