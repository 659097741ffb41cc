// The calibrated confidence head of one (request, position), evaluated by one warp.
//
// "Speculative decoding: from zero to DSpark" §6: a linear projection of the
// backbone's hidden state together with the Markov embedding predicts each draft
// position's conditional acceptance probability, calibrated per position by
// temperature scaling; the scheduler chains the values into survival
// probabilities.
//   c[b, i] = 1 / (1 + exp(-(w_h . hidden[b*N + i] + w_e . w1[prev] + beta) / tau[i]))
// with prev = anchor[b] for i = 0 and the draft token of step i - 1 after (the
// embedding the Markov head uses at step i).
//
// Used by the standalone head (csrc/confidence.cu) and by the Markov samplers,
// which evaluate it at each step from the previous token they already hold.
#pragma once

#include <cuda_bf16.h>

#include "device_common.cuh"

namespace dspark {

// The head's weights and output, as the samplers carry them (hidden == nullptr: no head).
struct ConfHead {
    const void* hidden;     // [B*N, H] (bf16 or fp32): the LM head's input rows
    int hidden_bf16;        // 1: hidden is bf16
    int H;
    const float* w_h;       // [H]
    const float* w_e;       // [r]
    const float* tau;       // [N], > 0: per-position calibration temperatures
    float beta;
    float* conf;            // [B, N] output
};

template <typename T> __device__ __forceinline__ float conf_as_f(T x);
template <> __device__ __forceinline__ float conf_as_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float conf_as_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// Partial dot product of one lane over a row of n elements of type T against fp32 weights:
// 16-byte pieces where the row allows it, then the tail element by element.
template <typename T>
__device__ __forceinline__ float conf_lane_dot(const T* row, const float* w, int n, uint32_t lane) {
    constexpr int kPer = 16 / static_cast<int>(sizeof(T));          // elements per 16-byte piece
    float acc0 = 0.f, acc1 = 0.f;
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(row) & 15) == 0 && (reinterpret_cast<uintptr_t>(w) & 15) == 0) {
        const int pieces = n / kPer;
#pragma unroll 8
        for (int p = static_cast<int>(lane); p < pieces; p += 32) {
            const uint4 q = *reinterpret_cast<const uint4*>(row + p * kPer);
            const T* e = reinterpret_cast<const T*>(&q);
#pragma unroll
            for (int k = 0; k < kPer; k += 4) {
                const float4 wv = *reinterpret_cast<const float4*>(w + p * kPer + k);
                acc0 = fmaf(conf_as_f<T>(e[k + 0]), wv.x, acc0);
                acc1 = fmaf(conf_as_f<T>(e[k + 1]), wv.y, acc1);
                acc0 = fmaf(conf_as_f<T>(e[k + 2]), wv.z, acc0);
                acc1 = fmaf(conf_as_f<T>(e[k + 3]), wv.w, acc1);
            }
        }
        done = pieces * kPer;
    }
    for (int k = done + static_cast<int>(lane); k < n; k += 32) acc0 = fmaf(conf_as_f<T>(row[k]), w[k], acc0);
    return acc0 + acc1;
}

// Logit sum s = w_h . hidden_row + w_e . w1_row, reduced over the warp (every lane gets it).
template <typename HT, typename WT>
__device__ __forceinline__ float conf_logit_sum(const HT* hidden_row, const float* w_h, int H, const WT* w1_row,
                                                const float* w_e, int r, uint32_t lane) {
    float s = conf_lane_dot<HT>(hidden_row, w_h, H, lane) + conf_lane_dot<WT>(w1_row, w_e, r, lane);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    return s;
}

// Calibrated probability from the warp-reduced logit sum; a temperature that is not positive and
// finite gives 0 and sets NUMERIC, as does a NaN result.
__device__ __forceinline__ float conf_probability(float s, float beta, float tau, WsHeader* ws) {
    float c = 0.f;
    if (tau > 0.f && tau < INFINITY) {
        const float z = __fdiv_rn(__fadd_rn(s, beta), tau);
        c = 1.f / (1.f + expf(-z));
    } else {
        set_status(ws, DSPARK_STATUS_NUMERIC);
    }
    if (c != c) set_status(ws, DSPARK_STATUS_NUMERIC);
    return c;
}

// c[b, i] of the head for hidden row `row` (= b*N + i) and embedding row prev of w1 (type WT), by the
// calling warp; lane 0 writes it.
template <typename WT>
__device__ __forceinline__ void conf_eval_warp(const ConfHead& h, WsHeader* ws, size_t row, int i, const WT* w1_row,
                                               int r, uint32_t lane) {
    float s;
    if (h.hidden_bf16)
        s = conf_logit_sum<__nv_bfloat16, WT>(static_cast<const __nv_bfloat16*>(h.hidden) + row * h.H, h.w_h, h.H,
                                              w1_row, h.w_e, r, lane);
    else
        s = conf_logit_sum<float, WT>(static_cast<const float*>(h.hidden) + row * h.H, h.w_h, h.H, w1_row, h.w_e, r,
                                      lane);
    if (lane == 0) h.conf[row] = conf_probability(s, h.beta, h.tau[i], ws);
}

}  // namespace dspark
