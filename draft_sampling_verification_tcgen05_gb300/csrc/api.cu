// C ABI of the DSpark hot path: argument validation, device facts, tensor-map
// encoding and the status word.  Compute happens only in the kernels of the
// other files; nothing here runs on the host in place of a kernel.
#include "confidence_common.cuh"
#include "device_common.cuh"
#include "host_common.h"

#include <cudaTypedefs.h>
#include <algorithm>
#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

namespace dspark {

namespace {
thread_local char g_error[512] = "";
std::mutex g_mu;
DeviceInfo g_dev_cache[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_error, sizeof(g_error), fmt, ap);
    va_end(ap);
}

dspark_status cuda_error(cudaError_t e, const char* what) {
    set_error("%s: %s (%d)", what, cudaGetErrorString(e), static_cast<int>(e));
    return DSPARK_ERR_CUDA;
}

bool current_device(DeviceInfo* info) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        set_error("no CUDA device: %s", cudaGetErrorString(e));
        return false;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev_cache[dev];
    if (d.device != dev) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) {
            set_error("cudaGetDeviceProperties: %s", cudaGetErrorString(e));
            return false;
        }
        if (prop.major != 10 || prop.minor != 3) {
            set_error("device %d is sm_%d%d; this library is built for sm_103a only", dev, prop.major, prop.minor);
            return false;
        }
        d.sm_count = prop.multiProcessorCount;
        d.cc_major = prop.major;
        d.cc_minor = prop.minor;
        d.smem_optin = prop.sharedMemPerBlockOptin;
        d.device = dev;
    }
    *info = d;
    return true;
}

bool make_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                     const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                     CUtensorMapSwizzle swizzle) {
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_encode == nullptr) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                             cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
                set_error("cuTensorMapEncodeTiled unavailable");
                return false;
            }
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    cuuint64_t d[5];
    cuuint64_t s[4];
    cuuint32_t bx[5];
    cuuint32_t es[5];
    for (uint32_t i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    const CUresult r = g_encode(map, dtype, rank, const_cast<void*>(base), d, s, bx, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
        return false;
    }
    return true;
}

namespace {

// Zeroes the first bytes of a workspace (16-byte stores, then the tail byte by byte).  A kernel
// rather than cudaMemsetAsync: in a CUDA graph a memset node ahead of each call's kernel measured
// about 4 us of dependency latency, a small kernel node well under 1 us.
__global__ void __launch_bounds__(256) clear_workspace_kernel(uint4* p, size_t n16, uint8_t* tail, size_t ntail) {
    const size_t i0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = i0; i < n16; i += stride) p[i] = make_uint4(0u, 0u, 0u, 0u);
    if (i0 < ntail) tail[i0] = 0;
}

}  // namespace

dspark_status clear_workspace(void* ws, size_t bytes, cudaStream_t stream) {
    if (bytes == 0) return DSPARK_OK;
    const size_t n16 = bytes / 16, ntail = bytes % 16;
    const size_t blocks = std::min<size_t>(std::max<size_t>((n16 + 1023) / 1024, 1), 608);
    clear_workspace_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<uint4*>(ws), n16, static_cast<uint8_t*>(ws) + n16 * 16, ntail);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(clear workspace)");
    return DSPARK_OK;
}

namespace {

__global__ void wait_selftest_kernel(WsHeader* ws, long long timeout_ns) {
    if (threadIdx.x != 0) return;
    const long long t0 = global_ns();
    while (ld_volatile_u32(&ws->never_set) == 0u) {
        if (global_ns() - t0 > timeout_ns) {
            atomicOr(&ws->status, DSPARK_STATUS_TIMEOUT);
            atomicExch(&ws->detail, 0x7E57u);
            return;
        }
        __nanosleep(1000);
    }
}

}  // namespace

dspark_status launch_wait_selftest(void* ws, long long timeout_ns, cudaStream_t stream) {
    dspark_status st = clear_workspace(ws, sizeof(WsHeader), stream);
    if (st != DSPARK_OK) return st;
    wait_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<WsHeader*>(ws), timeout_ns);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(wait_selftest)");
    return DSPARK_OK;
}

}  // namespace dspark

using namespace dspark;

namespace {

bool bad_ws(const void* ws, size_t ws_bytes, size_t need) {
    if (ws == nullptr || !aligned(ws, 256)) {
        set_error("workspace must be a non-null 256-byte aligned device pointer");
        return true;
    }
    if (ws_bytes < need) {
        set_error("workspace has %zu bytes, %zu needed", ws_bytes, need);
        return true;
    }
    return false;
}

#define DSPARK_REQUIRE(cond, ...)           \
    do {                                    \
        if (!(cond)) {                      \
            set_error(__VA_ARGS__);         \
            return DSPARK_ERR_INVALID_ARG;  \
        }                                   \
    } while (0)

}  // namespace

extern "C" {

size_t dspark_workspace_size(int op, int B, int N, int V, int r) {
    (void)r;
    if (B < 0 || N < 0) return 0;
    switch (op) {
        case DSPARK_OP_DRAFT_LOGITS:
            return sizeof(WsHeader);
        case DSPARK_OP_VERIFY:
            return V < 0 ? 0 : verify_workspace_bytes(B, V);
        case DSPARK_OP_MARKOV_SAMPLE:
            return markov_workspace_bytes(B, N);
        case DSPARK_OP_SCHEDULE:
            return schedule_workspace_bytes(B, N);
        case DSPARK_OP_VERIFY_GREEDY:
            return verify_greedy_workspace_bytes(B, N);
        case DSPARK_OP_CONFIDENCE:
            return sizeof(WsHeader);
        case DSPARK_OP_VERIFY_LOGITS:
            return verify_logits_workspace_bytes(B, N, V, r);
        case DSPARK_OP_VERIFY_GUMBEL:
            return verify_gumbel_workspace_bytes(B, N);
        default:
            return 0;
    }
}

dspark_status dspark_draft_logits(const void* hidden, const void* lm_head, dspark_dtype dtype, int M,
                                  int H, int V, float* logits, void* workspace, size_t ws_bytes,
                                  void* stream) {
    g_error[0] = '\0';
    DSPARK_REQUIRE(hidden && lm_head && logits, "draft_logits: null pointer");
    DSPARK_REQUIRE(dtype == DSPARK_F32 || dtype == DSPARK_BF16, "draft_logits: unknown dtype %d", (int)dtype);
    DSPARK_REQUIRE(M >= 1 && H >= 1 && V >= 1, "draft_logits: sizes must be positive (M=%d H=%d V=%d)", M, H, V);
    const size_t esize = dtype == DSPARK_F32 ? 4 : 2;
    DSPARK_REQUIRE((static_cast<size_t>(H) * esize) % 16 == 0,
                   "draft_logits: H*sizeof(dtype) must be a multiple of 16 bytes (H=%d)", H);
    DSPARK_REQUIRE(aligned(hidden, 16) && aligned(lm_head, 16) && aligned(logits, 4),
                   "draft_logits: hidden/lm_head must be 16-byte aligned, logits 4-byte aligned");
    if (bad_ws(workspace, ws_bytes, dspark_workspace_size(DSPARK_OP_DRAFT_LOGITS, 0, 0, 0, 0)))
        return DSPARK_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    dspark_status st = clear_workspace(workspace, sizeof(WsHeader), static_cast<cudaStream_t>(stream));
    if (st != DSPARK_OK) return st;
    return launch_draft_logits(hidden, lm_head, dtype, M, H, V, logits, workspace,
                               static_cast<cudaStream_t>(stream), dev);
}

dspark_status dspark_markov_sample(const float* base_logits, const int32_t* anchor, const void* w1,
                                   const void* w2, dspark_dtype wdtype, const float* temperature,
                                   uint64_t seed, uint64_t offset, int B, int N, int V, int r,
                                   int32_t* draft_tokens, float* lse, void* workspace, size_t ws_bytes,
                                   void* stream) {
    g_error[0] = '\0';
    DSPARK_REQUIRE(base_logits && anchor && w1 && w2 && temperature && draft_tokens,
                   "markov_sample: null pointer");
    DSPARK_REQUIRE(wdtype == DSPARK_F32 || wdtype == DSPARK_BF16, "markov_sample: unknown dtype %d", (int)wdtype);
    DSPARK_REQUIRE(B >= 1 && N >= 1 && N <= 65535 && V >= 2 && r >= 1 && r <= 1024,
                   "markov_sample: bad sizes (B=%d N=%d V=%d r=%d)", B, N, V, r);
    DSPARK_REQUIRE(offset < (1ull << 32), "markov_sample: offset must be below 2^32");
    DSPARK_REQUIRE(aligned(base_logits, 4) && aligned(w1, 16) && aligned(w2, 16),
                   "markov_sample: w1/w2 must be 16-byte aligned");
    if (bad_ws(workspace, ws_bytes, dspark_workspace_size(DSPARK_OP_MARKOV_SAMPLE, B, N, V, r)))
        return DSPARK_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    return launch_markov_sample(base_logits, anchor, w1, w2, wdtype, temperature, seed,
                                static_cast<uint32_t>(offset), B, N, V, r, draft_tokens, lse, nullptr, 0, V, nullptr,
                                workspace, static_cast<cudaStream_t>(stream), dev);
}

dspark_status dspark_markov_sample_conf(const float* base_logits, const int32_t* anchor, const void* w1,
                                        const void* w2, dspark_dtype wdtype, const float* temperature,
                                        uint64_t seed, uint64_t offset, int B, int N, int V, int r,
                                        const void* hidden, dspark_dtype hdtype, int H, const float* w_h,
                                        const float* w_e, float beta, const float* tau, int32_t* draft_tokens,
                                        float* conf, float* lse, void* workspace, size_t ws_bytes, void* stream) {
    g_error[0] = '\0';
    DSPARK_REQUIRE(base_logits && anchor && w1 && w2 && temperature && draft_tokens,
                   "markov_sample_conf: null pointer");
    DSPARK_REQUIRE(hidden && w_h && w_e && tau && conf, "markov_sample_conf: null confidence-head pointer");
    DSPARK_REQUIRE(wdtype == DSPARK_F32 || wdtype == DSPARK_BF16, "markov_sample_conf: unknown dtype %d", (int)wdtype);
    DSPARK_REQUIRE(hdtype == DSPARK_F32 || hdtype == DSPARK_BF16, "markov_sample_conf: unknown hidden dtype %d",
                   (int)hdtype);
    DSPARK_REQUIRE(B >= 1 && N >= 1 && N <= 65535 && V >= 2 && r >= 1 && r <= 1024 && H >= 1,
                   "markov_sample_conf: bad sizes (B=%d N=%d V=%d r=%d H=%d)", B, N, V, r, H);
    DSPARK_REQUIRE(offset < (1ull << 32), "markov_sample_conf: offset must be below 2^32");
    DSPARK_REQUIRE(aligned(base_logits, 4) && aligned(w1, 16) && aligned(w2, 16),
                   "markov_sample_conf: w1/w2 must be 16-byte aligned");
    if (bad_ws(workspace, ws_bytes, dspark_workspace_size(DSPARK_OP_MARKOV_SAMPLE, B, N, V, r)))
        return DSPARK_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    ConfHead head;
    head.hidden = hidden;
    head.hidden_bf16 = hdtype == DSPARK_BF16 ? 1 : 0;
    head.H = H;
    head.w_h = w_h;
    head.w_e = w_e;
    head.tau = tau;
    head.beta = beta;
    head.conf = conf;
    return launch_markov_sample(base_logits, anchor, w1, w2, wdtype, temperature, seed,
                                static_cast<uint32_t>(offset), B, N, V, r, draft_tokens, lse, nullptr, 0, V, &head,
                                workspace, static_cast<cudaStream_t>(stream), dev);
}

dspark_status dspark_markov_sample_reduced(const float* base_logits, const int32_t* anchor, const void* w1,
                                           const void* w2, dspark_dtype wdtype, const float* temperature,
                                           uint64_t seed, uint64_t offset, int B, int N, int V, int r,
                                           const int32_t* d2t, int d2t_mode, int V_target,
                                           int32_t* draft_tokens, float* lse, void* workspace, size_t ws_bytes,
                                           void* stream) {
    g_error[0] = '\0';
    DSPARK_REQUIRE(d2t != nullptr, "markov_sample_reduced: null d2t table");
    DSPARK_REQUIRE(d2t_mode == DSPARK_D2T_INDEX || d2t_mode == DSPARK_D2T_OFFSET,
                   "markov_sample_reduced: unknown table mode %d", d2t_mode);
    DSPARK_REQUIRE(V_target >= 1, "markov_sample_reduced: V_target must be positive");
    DSPARK_REQUIRE(base_logits && anchor && w1 && w2 && temperature && draft_tokens,
                   "markov_sample: null pointer");
    DSPARK_REQUIRE(wdtype == DSPARK_F32 || wdtype == DSPARK_BF16, "markov_sample: unknown dtype %d", (int)wdtype);
    DSPARK_REQUIRE(B >= 1 && N >= 1 && N <= 65535 && V >= 2 && r >= 1 && r <= 1024,
                   "markov_sample: bad sizes (B=%d N=%d V=%d r=%d)", B, N, V, r);
    DSPARK_REQUIRE(offset < (1ull << 32), "markov_sample: offset must be below 2^32");
    DSPARK_REQUIRE(aligned(base_logits, 4) && aligned(w1, 16) && aligned(w2, 16),
                   "markov_sample: w1/w2 must be 16-byte aligned");
    if (bad_ws(workspace, ws_bytes, dspark_workspace_size(DSPARK_OP_MARKOV_SAMPLE, B, N, V, r)))
        return DSPARK_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    return launch_markov_sample(base_logits, anchor, w1, w2, wdtype, temperature, seed,
                                static_cast<uint32_t>(offset), B, N, V, r, draft_tokens, lse, d2t,
                                d2t_mode == DSPARK_D2T_OFFSET ? 1 : 0, V_target, nullptr, workspace,
                                static_cast<cudaStream_t>(stream), dev);
}

dspark_status dspark_verify(const float* p_target, const float* p_draft, const int32_t* draft_tokens,
                            const int32_t* lengths, uint64_t seed, uint64_t offset, int B, int gamma, int V,
                            int32_t* out_tokens, int32_t* num_accepted, void* workspace, size_t ws_bytes,
                            void* stream) {
    g_error[0] = '\0';
    DSPARK_REQUIRE(p_target && p_draft && draft_tokens && out_tokens && num_accepted,
                   "verify: null pointer");
    DSPARK_REQUIRE(B >= 1 && gamma >= 1 && gamma <= 65535 && V >= 1 && V <= (1 << 24),
                   "verify: bad sizes (B=%d gamma=%d V=%d)", B, gamma, V);
    DSPARK_REQUIRE(offset < (1ull << 32), "verify: offset must be below 2^32");
    DSPARK_REQUIRE(aligned(p_target, 16) && aligned(p_draft, 16),
                   "verify: p_target/p_draft must be 16-byte aligned");
    if (bad_ws(workspace, ws_bytes, dspark_workspace_size(DSPARK_OP_VERIFY, B, gamma, V, 0)))
        return DSPARK_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    return launch_verify(p_target, p_draft, draft_tokens, lengths, seed, static_cast<uint32_t>(offset), B,
                         gamma, V, out_tokens, num_accepted, workspace, static_cast<cudaStream_t>(stream), dev);
}

dspark_status dspark_verify_greedy(const float* target, const int32_t* draft_tokens, const int32_t* lengths,
                                   int B, int gamma, int V, int32_t* out_tokens, int32_t* num_accepted,
                                   void* workspace, size_t ws_bytes, void* stream) {
    g_error[0] = '\0';
    DSPARK_REQUIRE(target && draft_tokens && out_tokens && num_accepted, "verify_greedy: null pointer");
    DSPARK_REQUIRE(B >= 1 && gamma >= 1 && gamma <= 65535 && V >= 1,
                   "verify_greedy: bad sizes (B=%d gamma=%d V=%d)", B, gamma, V);
    DSPARK_REQUIRE(aligned(target, 16), "verify_greedy: target must be 16-byte aligned");
    if (bad_ws(workspace, ws_bytes, dspark_workspace_size(DSPARK_OP_VERIFY_GREEDY, B, gamma, 0, 0)))
        return DSPARK_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    return launch_verify_greedy(target, draft_tokens, lengths, B, gamma, V, out_tokens, num_accepted, workspace,
                                static_cast<cudaStream_t>(stream), dev);
}

dspark_status dspark_verify_gumbel(const float* target_logits, const float* temperature,
                                   const int32_t* draft_tokens, const int32_t* lengths, uint64_t seed,
                                   uint64_t offset, int B, int gamma, int V, int32_t* out_tokens,
                                   int32_t* num_accepted, void* workspace, size_t ws_bytes, void* stream) {
    g_error[0] = '\0';
    DSPARK_REQUIRE(target_logits && temperature && draft_tokens && out_tokens && num_accepted,
                   "verify_gumbel: null pointer");
    DSPARK_REQUIRE(B >= 1 && B <= 65535 && gamma >= 1 && gamma <= 65535 && V >= 1 && V < (1 << 27),
                   "verify_gumbel: bad sizes (B=%d gamma=%d V=%d)", B, gamma, V);
    DSPARK_REQUIRE(offset < (1ull << 32), "verify_gumbel: offset must be below 2^32");
    DSPARK_REQUIRE(aligned(target_logits, 16), "verify_gumbel: target_logits must be 16-byte aligned");
    if (bad_ws(workspace, ws_bytes, dspark_workspace_size(DSPARK_OP_VERIFY_GUMBEL, B, gamma, 0, 0)))
        return DSPARK_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    return launch_verify_gumbel(target_logits, temperature, draft_tokens, lengths, seed, static_cast<uint32_t>(offset),
                                B, gamma, V, out_tokens, num_accepted, workspace, static_cast<cudaStream_t>(stream),
                                dev);
}

dspark_status dspark_verify_logits(const float* target_logits, const float* target_temperature,
                                   const float* base_logits, const int32_t* anchor, const void* w1, const void* w2,
                                   dspark_dtype wdtype, int r, const float* draft_temperature, const float* draft_lse,
                                   const int32_t* draft_tokens, const int32_t* lengths, uint64_t seed,
                                   uint64_t offset, int B, int gamma, int V, int32_t* out_tokens,
                                   int32_t* num_accepted, void* workspace, size_t ws_bytes, void* stream) {
    g_error[0] = '\0';
    DSPARK_REQUIRE(target_logits && target_temperature && base_logits && anchor && w1 && w2 && draft_temperature &&
                       draft_lse && draft_tokens && out_tokens && num_accepted,
                   "verify_logits: null pointer");
    DSPARK_REQUIRE(wdtype == DSPARK_F32 || wdtype == DSPARK_BF16, "verify_logits: unknown dtype %d", (int)wdtype);
    DSPARK_REQUIRE(B >= 1 && gamma >= 1 && gamma <= 65535 && V >= 2 && r >= 1 && r <= 1024,
                   "verify_logits: bad sizes (B=%d gamma=%d V=%d r=%d)", B, gamma, V, r);
    const size_t esize = wdtype == DSPARK_F32 ? 4 : 2;
    DSPARK_REQUIRE((static_cast<size_t>(r) * esize) % 16 == 0,
                   "verify_logits: r*sizeof(wdtype) must be a multiple of 16 bytes (r=%d)", r);
    DSPARK_REQUIRE(offset < (1ull << 32), "verify_logits: offset must be below 2^32");
    DSPARK_REQUIRE(aligned(target_logits, 16) && aligned(base_logits, 16) && aligned(w1, 16) && aligned(w2, 16),
                   "verify_logits: target_logits, base_logits, w1, w2 must be 16-byte aligned");
    if (bad_ws(workspace, ws_bytes, dspark_workspace_size(DSPARK_OP_VERIFY_LOGITS, B, gamma, V, r)))
        return DSPARK_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    return launch_verify_logits(target_logits, target_temperature, base_logits, anchor, w1, w2, wdtype,
                                draft_temperature, draft_lse, draft_tokens, lengths, seed,
                                static_cast<uint32_t>(offset), B, gamma, V, r, out_tokens, num_accepted, workspace,
                                static_cast<cudaStream_t>(stream), dev);
}

dspark_status dspark_confidence(const void* hidden, dspark_dtype hdtype, const void* w1, dspark_dtype wdtype,
                                const int32_t* anchor, const int32_t* draft_tokens, const float* w_h,
                                const float* w_e, float beta, const float* tau, int B, int N, int H, int V, int r,
                                float* conf, void* workspace, size_t ws_bytes, void* stream) {
    g_error[0] = '\0';
    DSPARK_REQUIRE(hidden && w1 && anchor && draft_tokens && w_h && w_e && tau && conf, "confidence: null pointer");
    DSPARK_REQUIRE((hdtype == DSPARK_F32 || hdtype == DSPARK_BF16) && (wdtype == DSPARK_F32 || wdtype == DSPARK_BF16),
                   "confidence: unknown dtype");
    DSPARK_REQUIRE(B >= 1 && N >= 1 && H >= 1 && V >= 1 && r >= 1 && static_cast<long long>(B) * N < (1ll << 31),
                   "confidence: bad sizes (B=%d N=%d H=%d V=%d r=%d)", B, N, H, V, r);
    if (bad_ws(workspace, ws_bytes, dspark_workspace_size(DSPARK_OP_CONFIDENCE, B, N, V, r)))
        return DSPARK_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    return launch_confidence(hidden, hdtype, w1, wdtype, anchor, draft_tokens, w_h, w_e, beta, tau, B, N, H, V, r,
                             conf, workspace, static_cast<cudaStream_t>(stream));
}

dspark_status dspark_schedule(const float* cond_accept, const double* sps, int S, int B, int N, int K_in,
                              float* survival, int32_t* K_out, int32_t* lengths, int32_t* selected,
                              void* workspace, size_t ws_bytes, void* stream) {
    g_error[0] = '\0';
    DSPARK_REQUIRE(cond_accept && survival && K_out && lengths && selected, "schedule: null pointer");
    DSPARK_REQUIRE(B >= 1 && N >= 1 && static_cast<long long>(B) * N <= (1ll << 20),
                   "schedule: need B, N >= 1 and B*N <= 2^20 (B=%d N=%d)", B, N);
    DSPARK_REQUIRE(K_in >= 0 || (sps != nullptr && S >= 1), "schedule: choosing K needs an SPS table (S >= 1)");
    if (bad_ws(workspace, ws_bytes, dspark_workspace_size(DSPARK_OP_SCHEDULE, B, N, 0, 0)))
        return DSPARK_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    return launch_schedule(cond_accept, sps, S, B, N, K_in, survival, K_out, lengths, selected, workspace,
                           static_cast<cudaStream_t>(stream), dev);
}

dspark_status dspark_read_status(const void* workspace, uint32_t* bits, void* stream) {
    g_error[0] = '\0';
    DSPARK_REQUIRE(workspace != nullptr, "read_status: null workspace");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "cudaStreamSynchronize");
    uint32_t w = 0;
    e = cudaMemcpy(&w, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_error(e, "cudaMemcpy(status)");
    if (bits) *bits = w;
    if (w & DSPARK_STATUS_TIMEOUT) return DSPARK_ERR_TIMEOUT;
    if (w & DSPARK_STATUS_NUMERIC) return DSPARK_ERR_NUMERIC;
    if (w & DSPARK_STATUS_INPUT_RANGE) return DSPARK_ERR_INPUT_RANGE;
    if (w & (DSPARK_STATUS_INTERNAL | DSPARK_STATUS_INDEX)) return DSPARK_ERR_CUDA;   // the library's own state
    return DSPARK_OK;
}

const char* dspark_status_string(dspark_status s) {
    switch (s) {
        case DSPARK_OK: return "ok";
        case DSPARK_ERR_INVALID_ARG: return "invalid argument";
        case DSPARK_ERR_UNSUPPORTED: return "unsupported";
        case DSPARK_ERR_CUDA: return "CUDA error";
        case DSPARK_ERR_TIMEOUT: return "device wait timed out";
        case DSPARK_ERR_NUMERIC: return "non-finite input or empty distribution";
        case DSPARK_ERR_INPUT_RANGE: return "input value out of range";
        default: return "unknown status";
    }
}

const char* dspark_last_error(void) { return g_error; }

dspark_status dspark_selftest_wait_timeout(void* workspace, size_t ws_bytes, long long timeout_ns, void* stream) {
    g_error[0] = '\0';
    if (bad_ws(workspace, ws_bytes, sizeof(WsHeader))) return DSPARK_ERR_INVALID_ARG;
    DSPARK_REQUIRE(timeout_ns >= 1000 && timeout_ns <= 10000000000LL, "selftest: timeout out of range");
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    return launch_wait_selftest(workspace, timeout_ns, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
