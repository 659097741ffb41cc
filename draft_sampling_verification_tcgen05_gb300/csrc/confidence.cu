// Calibrated confidence head: conditional acceptance probability of every draft token.
//
// "Speculative decoding: from zero to DSpark" §6: a linear projection of the
// backbone's hidden state together with the Markov embedding predicts each
// position's conditional acceptance probability, calibrated per position by
// temperature scaling; the scheduler chains them into survival probabilities.
//   c[b, i] = 1 / (1 + exp(-(w_h . hidden[b*N + i] + w_e . w1[prev] + beta) / tau[i]))
// with prev = anchor[b] for i = 0 and draft_tokens[b, i-1] after (the embedding
// the Markov head uses at step i).
//
// One warp per (request, position): 16-byte loads of the hidden row (the LM
// head's input row) and of w_h, eight in flight per lane, the r Markov
// features, a shuffle reduction, fp32 throughout (csrc/confidence_common.cuh,
// shared with the samplers that evaluate the head step by step).  The output
// feeds dspark_schedule's cond_accept directly.
#include "confidence_common.cuh"
#include "device_common.cuh"
#include "host_common.h"

#include <cuda_bf16.h>

namespace dspark {
namespace {

constexpr int kWarpsPerBlock = 8;

struct ConfArgs {
    const void* hidden;
    const void* w1;
    const int32_t* anchor;
    const int32_t* tokens;
    const float* w_h;
    const float* w_e;
    const float* tau;
    float* conf;
    WsHeader* ws;
    float beta;
    int B, N, H, V, r;
};

template <typename HT, typename WT>
__global__ void __launch_bounds__(32 * kWarpsPerBlock) confidence_kernel(ConfArgs a) {
    const int pair = static_cast<int>(blockIdx.x) * kWarpsPerBlock + static_cast<int>(warp_id());
    if (pair >= a.B * a.N) return;
    const uint32_t lane = lane_id();
    const int b = pair / a.N, i = pair % a.N;
    int prev = i == 0 ? a.anchor[b] : a.tokens[static_cast<size_t>(b) * a.N + i - 1];
    if (prev < 0 || prev >= a.V) {                       // read as token 0, flagged
        if (lane == 0) flag_input_index(a.ws);
        prev = 0;
    }
    const float s = conf_logit_sum<HT, WT>(static_cast<const HT*>(a.hidden) + static_cast<size_t>(pair) * a.H, a.w_h,
                                           a.H, static_cast<const WT*>(a.w1) + static_cast<size_t>(prev) * a.r, a.w_e,
                                           a.r, lane);
    if (lane == 0) a.conf[pair] = conf_probability(s, a.beta, a.tau[i], a.ws);
}

}  // namespace

dspark_status launch_confidence(const void* hidden, dspark_dtype hdtype, const void* w1, dspark_dtype wdtype,
                                const int32_t* anchor, const int32_t* draft_tokens, const float* w_h,
                                const float* w_e, float beta, const float* tau, int B, int N, int H, int V, int r,
                                float* conf, void* ws, cudaStream_t stream) {
    const dspark_status st = clear_workspace(ws, sizeof(WsHeader), stream);
    if (st != DSPARK_OK) return st;
    ConfArgs a;
    a.hidden = hidden;
    a.w1 = w1;
    a.anchor = anchor;
    a.tokens = draft_tokens;
    a.w_h = w_h;
    a.w_e = w_e;
    a.tau = tau;
    a.conf = conf;
    a.ws = static_cast<WsHeader*>(ws);
    a.beta = beta;
    a.B = B;
    a.N = N;
    a.H = H;
    a.V = V;
    a.r = r;
    const long long pairs = static_cast<long long>(B) * N;
    const unsigned grid = static_cast<unsigned>((pairs + kWarpsPerBlock - 1) / kWarpsPerBlock);
    const dim3 block(32 * kWarpsPerBlock);
    const bool hb = hdtype == DSPARK_BF16, wb = wdtype == DSPARK_BF16;
    if (hb && wb) confidence_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, block, 0, stream>>>(a);
    else if (hb) confidence_kernel<__nv_bfloat16, float><<<grid, block, 0, stream>>>(a);
    else if (wb) confidence_kernel<float, __nv_bfloat16><<<grid, block, 0, stream>>>(a);
    else confidence_kernel<float, float><<<grid, block, 0, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(confidence)");
    return DSPARK_OK;
}

}  // namespace dspark
