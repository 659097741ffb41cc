// Host-side helpers shared by the launchers: device facts, tensor-map
// encoding, error text, and the launcher entry points of each kernel file.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/dspark.h"

namespace dspark {

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0;
    int cc_minor = 0;
    size_t smem_optin = 0;
};

// Facts about the current device (cached per device).  Returns false and sets
// the error text when there is no usable device or it is not an sm_103 part.
bool current_device(DeviceInfo* info);

// Records a host-side error message for dspark_last_error().
void set_error(const char* fmt, ...);
dspark_status cuda_error(cudaError_t e, const char* what);

// 2-D / 3-D tiled tensor maps (dims and boxes innermost first; strides in
// bytes for dims 1..).  Returns false (with the error text set) on failure.
bool make_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                     const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                     CUtensorMapSwizzle swizzle);

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Clears the first `bytes` of a workspace on `stream` (status word, barrier,
// per-call scratch).
dspark_status clear_workspace(void* ws, size_t bytes, cudaStream_t stream);

// ---- launchers (one per kernel file); arguments are already validated ----
dspark_status launch_draft_logits(const void* hidden, const void* lm_head, dspark_dtype dtype,
                                  int M, int H, int V, float* logits, void* ws,
                                  cudaStream_t stream, const DeviceInfo& dev);

size_t markov_workspace_bytes(int B, int N);
dspark_status launch_markov_sample(const float* base_logits, const int32_t* anchor, const void* w1,
                                   const void* w2, dspark_dtype wdtype, const float* temperature,
                                   uint64_t seed, uint32_t offset, int B, int N, int V, int r,
                                   int32_t* draft_tokens, float* lse, const int32_t* d2t, int d2t_offset,
                                   int V_target, const struct ConfHead* head, void* ws, cudaStream_t stream,
                                   const DeviceInfo& dev);

size_t verify_workspace_bytes(int B, int V);
size_t verify_greedy_workspace_bytes(int B, int gamma);
size_t verify_gumbel_workspace_bytes(int B, int gamma);
dspark_status launch_verify_gumbel(const float* target_logits, const float* temperature, const int32_t* draft_tokens,
                                   const int32_t* lengths, uint64_t seed, uint32_t offset, int B, int gamma, int V,
                                   int32_t* out_tokens, int32_t* num_accepted, void* ws, cudaStream_t stream,
                                   const DeviceInfo& dev);
dspark_status launch_confidence(const void* hidden, dspark_dtype hdtype, const void* w1, dspark_dtype wdtype,
                                const int32_t* anchor, const int32_t* draft_tokens, const float* w_h,
                                const float* w_e, float beta, const float* tau, int B, int N, int H, int V, int r,
                                float* conf, void* ws, cudaStream_t stream);
dspark_status launch_verify_greedy(const float* target, const int32_t* draft_tokens, const int32_t* lengths,
                                   int B, int gamma, int V, int32_t* out_tokens, int32_t* num_accepted,
                                   void* ws, cudaStream_t stream, const DeviceInfo& dev);
dspark_status launch_verify(const float* p_target, const float* p_draft, const int32_t* draft_tokens,
                            const int32_t* lengths, uint64_t seed, uint32_t offset, int B, int gamma,
                            int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                            cudaStream_t stream, const DeviceInfo& dev);

size_t verify_logits_workspace_bytes(int B, int gamma, int V, int r);
dspark_status launch_verify_logits(const float* target_logits, const float* T_t, const float* base_logits,
                                   const int32_t* anchor, const void* w1, const void* w2, dspark_dtype wdtype,
                                   const float* T_d, const float* draft_lse, const int32_t* draft_tokens,
                                   const int32_t* lengths, uint64_t seed, uint32_t offset, int B, int gamma,
                                   int V, int r, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                                   cudaStream_t stream, const DeviceInfo& dev);

size_t schedule_workspace_bytes(int B, int N);
dspark_status launch_schedule(const float* cond_accept, const double* sps, int S, int B, int N,
                              int K_in, float* survival, int32_t* K_out, int32_t* lengths,
                              int32_t* selected, void* ws, cudaStream_t stream,
                              const DeviceInfo& dev);

dspark_status launch_wait_selftest(void* ws, long long timeout_ns, cudaStream_t stream);

}  // namespace dspark
