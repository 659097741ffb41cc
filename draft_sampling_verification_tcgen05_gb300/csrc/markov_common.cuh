// Shared pieces of the two Markov-sampler kernels (CUDA-core and tensor-core
// paths): workspace layout, arguments, Gumbel variate of an element, step
// slots and the log-sum-exp partials.
#pragma once

#include "confidence_common.cuh"
#include "device_common.cuh"
#include "host_common.h"

namespace dspark {
namespace markov {

constexpr int kMaxGrid = 1024;                         // workspace is sized for this many blocks
constexpr uint32_t kWaitStep = 0x200;                  // + step index (grid barrier)
constexpr int kExchangeMaxBN = 64;                     // B * N limit of the candidate exchange
constexpr int kPubStride = 16;                         // publication counters per step (one per request chunk)

struct MarkovLayout {
    unsigned long long* slots;   // [N][B] argmax keys
    uint32_t* lb;                // [N][B] order bits of the published lower bound
    uint32_t* pub;               // [N][kPubStride] blocks that have published a chunk's bounds (tensor path)
    unsigned long long* cand;    // [N][grid][B] per-block candidates (exchange; B * N <= kExchangeMaxBN)
    float2* lse_part;            // [2][kMaxGrid][B] (max, sum) partials
    float* conf_h;               // [B][N] w_h . hidden row of each pair (confidence head, CUDA-core path)
};

__host__ __device__ inline size_t markov_cand_entries(int B, int N) {
    return static_cast<size_t>(B) * N <= static_cast<size_t>(kExchangeMaxBN)
               ? static_cast<size_t>(N) * kMaxGrid * B : 0;
}

__host__ __device__ inline MarkovLayout markov_layout(void* ws, int B, int N) {
    uint8_t* p = static_cast<uint8_t*>(ws) + sizeof(WsHeader);
    MarkovLayout L;
    L.slots = reinterpret_cast<unsigned long long*>(p);
    p += sizeof(unsigned long long) * static_cast<size_t>(N) * B;
    L.lb = reinterpret_cast<uint32_t*>(p);
    p += sizeof(uint32_t) * static_cast<size_t>(N) * B;
    L.pub = reinterpret_cast<uint32_t*>(p);
    p += sizeof(uint32_t) * static_cast<size_t>(N) * kPubStride;
    p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 15) & ~static_cast<uintptr_t>(15));
    L.cand = reinterpret_cast<unsigned long long*>(p);
    p += sizeof(unsigned long long) * markov_cand_entries(B, N);
    L.lse_part = reinterpret_cast<float2*>(p);
    p += sizeof(float2) * 2 * static_cast<size_t>(kMaxGrid) * B;
    L.conf_h = reinterpret_cast<float*>(p);
    return L;
}

struct MarkovArgs {
    const float* base;          // [B, N, V]
    const int32_t* anchor;      // [B]
    const void* w1;             // [V, r]
    const void* w2;             // [V, r]
    const float* temperature;   // [B]
    int32_t* tokens;            // [B, N]
    float* lse;                 // [B, N] or null
    WsHeader* ws;
    MarkovLayout lay;
    uint64_t seed;
    uint32_t offset;
    int B, N, V, r;
    int slice;                  // vocabulary entries per block
    int w2_cached;              // w2 slice lives in shared memory
    int w2_pitch;               // bytes per cached w2 row (padded)
    int z_stored;               // z rows live in shared memory
    int single_pass;            // noise on every element in one pass (few elements per block)
    int exchange;               // blocks publish per-step candidates and poll each other's
                                // (instead of step slots and a grid barrier)
    int w2_split;               // cached w2 rows stored even rows first, then odd rows
    const int32_t* d2t;         // [V] draft-to-target table, or null (tokens are draft ids)
    int d2t_offset;             // 0: target = d2t[d]; 1: target = d + d2t[d]
    int V_target;               // range of the mapped ids
    ConfHead head;              // calibrated confidence head evaluated at every step (head.hidden null: none)
    long long timeout_ns;
};

// The token written for sampled draft id d: d itself, or its target-vocabulary id through the
// table ("DSpark implementation and evaluation" §5 index table; EAGLE-3's offset table); a
// mapped id outside [0, V_target) is written as -1 and flagged.
__device__ __forceinline__ int32_t output_token(const MarkovArgs& a, int d) {
    if (a.d2t == nullptr) return d;
    const long long t = a.d2t_offset ? static_cast<long long>(d) + a.d2t[d] : static_cast<long long>(a.d2t[d]);
    if (t < 0 || t >= a.V_target) {
        flag_input_index(a.ws);
        return -1;
    }
    return static_cast<int32_t>(t);
}

__device__ __forceinline__ float gumbel_at(const MarkovArgs& a, int b, int i, int v) {
    return draft_gumbel(a.seed, a.offset, static_cast<uint32_t>(b), static_cast<uint32_t>(i), static_cast<uint32_t>(v));
}

__device__ __forceinline__ float2 lse_merge(float2 a, float2 b) {
    if (a.y == 0.f) return b;
    if (b.y == 0.f) return a;
    const float m = fmaxf(a.x, b.x);
    return make_float2(m, a.y * __expf(a.x - m) + b.y * __expf(b.x - m));
}

// Reads a token from a step slot; key 0 means no finite candidate existed.
__device__ __forceinline__ int slot_token(const MarkovArgs& a, int i, int b) {
    const unsigned long long k = __ldcg(a.lay.slots + static_cast<size_t>(i) * a.B + b);
    if (k == 0ull) {
        set_status(a.ws, DSPARK_STATUS_NUMERIC);
        return 0;
    }
    const int x = static_cast<int>(key_index(k));
    return own_index_ok(x, a.V, a.ws) ? x : 0;
}

// Combine the lse partials of step i: one warp per request, the lanes over the blocks' partials,
// then a butterfly merge.  `tid`/`nthreads`: this thread's index among the block's participating
// threads (whole warps).
__device__ inline void finish_lse(const MarkovArgs& a, int i, int tid, int nthreads) {
    if (a.lse == nullptr) return;
    const float2* part = a.lay.lse_part + static_cast<size_t>(i & 1) * kMaxGrid * a.B;
    const int lane = tid & 31, warps = nthreads >> 5;
    for (int b = static_cast<int>(blockIdx.x) * warps + (tid >> 5); b < a.B; b += static_cast<int>(gridDim.x) * warps) {
        float2 m = make_float2(0.f, 0.f);
        for (int c = lane; c < static_cast<int>(gridDim.x); c += 32) m = lse_merge(m, __ldcg(part + static_cast<size_t>(c) * a.B + b));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float2 other;
            other.x = __shfl_xor_sync(0xFFFFFFFFu, m.x, o);
            other.y = __shfl_xor_sync(0xFFFFFFFFu, m.y, o);
            m = lse_merge(m, other);
        }
        if (lane == 0) a.lse[static_cast<size_t>(b) * a.N + i] = m.y > 0.f ? m.x + logf(m.y) : -INFINITY;
    }
}

}  // namespace markov

// Tensor-core path (csrc/markov_tc.cu): bf16 Markov head, 16 <= B <= 256.
bool markov_tc_eligible(int B, int N, int V, int r, dspark_dtype wdtype, const float* base, const float* lse,
                        int sm_count);
dspark_status launch_markov_tc(const markov::MarkovArgs& a, cudaStream_t stream, const DeviceInfo& dev);

}  // namespace dspark
