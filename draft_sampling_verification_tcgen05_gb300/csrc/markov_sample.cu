// Sequential Markov-biased Gumbel-max sampling of N draft tokens per request.
//
// "DSpark implementation and evaluation" §2.2 (_sample_sequential): for
// i = 0..N-1, bias = markov_w2 . markov_w1[prev] is added to base_logits[:, i],
// a token is Gumbel-sampled and becomes prev; §3: markov_w1 is an
// Embedding(V, r), markov_w2 a bias-free r -> V linear.
//
// One persistent cooperative kernel runs all N steps.  Block c owns a
// contiguous vocabulary slice [v_lo, v_hi) for the whole call; per step:
//   1. prev_b (the anchor, or the previous step's winner) -> w1 row gather
//      into shared memory (E[b, :])
//   2. pass 1: z = (base + w2 . E[b]) / T_b for every v of the slice, kept in
//      shared memory; the block's argmax of z is perturbed with its own Gumbel
//      noise, giving a real candidate value y*, published as a lower bound
//      LB[i][b] (atomicMax) and as a candidate key
//   3. pass 2: Gumbel noise only for elements that can still win:
//      z + G_max >= LB (G_max bounds every variate), each candidate (value,
//      index) folded into a 64-bit key; block reduction, then one atomicMax
//      per (block, b) into the step's slot -- the two-level argmax
//   4. grid barrier; every block reads the B winners as the next prev.
// Rows of z never leave the block: no [B, V] array is written to memory.
// Ties go to the lowest index through the key encoding; the result does not
// depend on which elements were skipped, because a skipped element is
// strictly below the bound, which is itself a value some element reaches.
#include "device_common.cuh"
#include "host_common.h"
#include "markov_common.cuh"

#include <algorithm>
#include <type_traits>

namespace dspark {
namespace {

using namespace markov;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr size_t kW2CacheBytes = 144 * 1024;           // w2 slice kept in shared memory when it fits
constexpr size_t kZStoreBytes = 32 * 1024;             // z rows kept in shared memory when they fit
constexpr int kMaxEFloats = 16384;                     // B * r limit of the shared E matrix

// Decode tensor path (one request, bf16 head, r = 64): the block's w2 slice stays in tensor
// memory for the whole call as the A operand of eight 128 x 16 x 64 tcgen05 MMAs per step,
// E = w1[prev] is row 0 of the 16-row B operand in shared memory (128-byte swizzle), and the
// bias of each entry is column 0 of its tile's accumulator.  Tensor memory: accumulators in
// columns [0, 128) (16 per tile), the slice in [128, 384) (32 per tile: 64 bf16 per lane).
constexpr int kTcRows = 2 * kThreads;                   // 1024 slice entries, 8 tiles of 128
constexpr int kTcTiles = kTcRows / 128;
constexpr int kTcR = 64;
constexpr int kTcN = 16;
constexpr uint32_t kTcCols = 512;
constexpr uint32_t kTcACol = 128;
constexpr size_t kTcBBytes = static_cast<size_t>(kTcN) * kTcR * 2;
constexpr size_t kTcStageBytes = static_cast<size_t>(kTcRows) * kTcR * 2;   // slice staging (also
                                                        // keeps one block per SM, which holds all of TMEM)
constexpr uint32_t kWaitDecodeMma = 0x311;
constexpr long long kPollHoldCycles = 800;              // about 0.4 us at 2 GHz

// Entry 2 tid + h of the slice (thread tid, warp w) is row 32 (w mod 4) + lane of tile w / 4 + 4 h:
// the two entries of a thread share a noise group word, and warp w reads exactly tensor-memory
// lanes 32 (w mod 4) + lane.


template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// dot(w2 row, E row) over r in fp32: four independent partial sums (k mod 8 in
// {0,1}, {2,3}, {4,5}, {6,7} of each 16-byte piece) added at the end, so the
// dependent FMA chain is a quarter as long.
template <typename WT>
__device__ __forceinline__ float bias_dot(const uint8_t* row, const float* e, int r) {
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    int k = 0;
    if constexpr (sizeof(WT) == 2) {
        if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
            for (; k + 8 <= r; k += 8) {
                const uint4 q = *reinterpret_cast<const uint4*>(row + 2 * k);
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
                const float2 f0 = __bfloat1622float2(h[0]), f1 = __bfloat1622float2(h[1]);
                const float2 f2 = __bfloat1622float2(h[2]), f3 = __bfloat1622float2(h[3]);
                acc0 = fmaf(f0.x, e[k + 0], acc0);
                acc1 = fmaf(f1.x, e[k + 2], acc1);
                acc2 = fmaf(f2.x, e[k + 4], acc2);
                acc3 = fmaf(f3.x, e[k + 6], acc3);
                acc0 = fmaf(f0.y, e[k + 1], acc0);
                acc1 = fmaf(f1.y, e[k + 3], acc1);
                acc2 = fmaf(f2.y, e[k + 5], acc2);
                acc3 = fmaf(f3.y, e[k + 7], acc3);
            }
        }
        for (; k < r; ++k)
            acc0 = fmaf(__bfloat162float(reinterpret_cast<const __nv_bfloat16*>(row)[k]), e[k], acc0);
    } else {
        if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
            for (; k + 4 <= r; k += 4) {
                const float4 q = *reinterpret_cast<const float4*>(row + 4 * k);
                acc0 = fmaf(q.x, e[k], acc0);
                acc1 = fmaf(q.y, e[k + 1], acc1);
                acc2 = fmaf(q.z, e[k + 2], acc2);
                acc3 = fmaf(q.w, e[k + 3], acc3);
            }
        }
        for (; k < r; ++k) acc0 = fmaf(reinterpret_cast<const float*>(row)[k], e[k], acc0);
    }
    return (acc0 + acc1) + (acc2 + acc3);
}

// Two bf16 rows of fixed width R against the same E row, fully unrolled: every shared-memory
// load is issued before the first multiply-add, and four independent chains per row.
template <int R>
__device__ __forceinline__ void bias_dot2_fixed(const uint8_t* row0, const uint8_t* row1, const float* e,
                                                float& out0, float& out1) {
    uint4 q0[R / 8], q1[R / 8];
#pragma unroll
    for (int c = 0; c < R / 8; ++c) {
        q0[c] = *reinterpret_cast<const uint4*>(row0 + 16 * c);
        q1[c] = *reinterpret_cast<const uint4*>(row1 + 16 * c);
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < R / 8; ++c) {
        const float4 e0 = *reinterpret_cast<const float4*>(e + 8 * c);
        const float4 e1 = *reinterpret_cast<const float4*>(e + 8 * c + 4);
        const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
        const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&q0[c]);
        const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&q1[c]);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float2 f0 = __bfloat1622float2(h0[p]);
            const float2 f1 = __bfloat1622float2(h1[p]);
            acc[(p & 1) * 2 + 0] = fmaf(f0.x, ev[2 * p], acc[(p & 1) * 2 + 0]);
            acc[(p & 1) * 2 + 1] = fmaf(f0.y, ev[2 * p + 1], acc[(p & 1) * 2 + 1]);
            acc[4 + (p & 1) * 2 + 0] = fmaf(f1.x, ev[2 * p], acc[4 + (p & 1) * 2 + 0]);
            acc[4 + (p & 1) * 2 + 1] = fmaf(f1.y, ev[2 * p + 1], acc[4 + (p & 1) * 2 + 1]);
        }
    }
    out0 = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    out1 = (acc[4] + acc[5]) + (acc[6] + acc[7]);
}

// Two rows against the same E row at once (independent chains, shared E reads).
template <typename WT>
__device__ __forceinline__ void bias_dot2(const uint8_t* row0, const uint8_t* row1, const float* e, int r,
                                          float& out0, float& out1) {
    if constexpr (sizeof(WT) == 2) {
        if (((reinterpret_cast<uintptr_t>(row0) | reinterpret_cast<uintptr_t>(row1)) & 15) == 0 &&
            (reinterpret_cast<uintptr_t>(e) & 15) == 0 && r == 64) {
            bias_dot2_fixed<64>(row0, row1, e, out0, out1);
            return;
        }
        if (((reinterpret_cast<uintptr_t>(row0) | reinterpret_cast<uintptr_t>(row1)) & 15) == 0 && (r & 7) == 0 &&
            (reinterpret_cast<uintptr_t>(e) & 15) == 0) {
            float a0 = 0.f, a1 = 0.f, c0 = 0.f, c1 = 0.f;
            for (int k = 0; k < r; k += 8) {
                const uint4 q0 = *reinterpret_cast<const uint4*>(row0 + 2 * k);
                const uint4 q1 = *reinterpret_cast<const uint4*>(row1 + 2 * k);
                const float4 e0 = *reinterpret_cast<const float4*>(e + k);
                const float4 e1 = *reinterpret_cast<const float4*>(e + k + 4);
                const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&q0);
                const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&q1);
                float2 f;
                f = __bfloat1622float2(h0[0]); a0 = fmaf(f.x, e0.x, a0); c0 = fmaf(f.y, e0.y, c0);
                f = __bfloat1622float2(h0[1]); a0 = fmaf(f.x, e0.z, a0); c0 = fmaf(f.y, e0.w, c0);
                f = __bfloat1622float2(h0[2]); a0 = fmaf(f.x, e1.x, a0); c0 = fmaf(f.y, e1.y, c0);
                f = __bfloat1622float2(h0[3]); a0 = fmaf(f.x, e1.z, a0); c0 = fmaf(f.y, e1.w, c0);
                f = __bfloat1622float2(h1[0]); a1 = fmaf(f.x, e0.x, a1); c1 = fmaf(f.y, e0.y, c1);
                f = __bfloat1622float2(h1[1]); a1 = fmaf(f.x, e0.z, a1); c1 = fmaf(f.y, e0.w, c1);
                f = __bfloat1622float2(h1[2]); a1 = fmaf(f.x, e1.x, a1); c1 = fmaf(f.y, e1.y, c1);
                f = __bfloat1622float2(h1[3]); a1 = fmaf(f.x, e1.z, a1); c1 = fmaf(f.y, e1.w, c1);
            }
            out0 = a0 + c0;
            out1 = a1 + c1;
            return;
        }
    }
    out0 = bias_dot<WT>(row0, e, r);
    out1 = bias_dot<WT>(row1, e, r);
}

// Block maximum, valid in thread 0 only (the only reader).  One barrier: callers rotate over
// four `red` buffers (request parity x pass), so the barrier of an intermediate call always
// separates thread 0's read of a buffer from the next writes to it.
__device__ __forceinline__ unsigned long long block_max_u64_t0(unsigned long long k, unsigned long long* red) {
    k = warp_max_u64(k);
    if (lane_id() == 0) red[warp_id()] = k;
    __syncthreads();
    unsigned long long m = 0;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) m = red[w] > m ? red[w] : m;
    }
    return m;
}


__device__ __forceinline__ float2 block_lse(float2 v, float2* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float2 other;
        other.x = __shfl_xor_sync(0xFFFFFFFFu, v.x, o);
        other.y = __shfl_xor_sync(0xFFFFFFFFu, v.y, o);
        v = lse_merge(v, other);
    }
    __syncthreads();
    if (lane_id() == 0) red[warp_id()] = v;
    __syncthreads();
    float2 m = make_float2(0.f, 0.f);
    for (int w = 0; w < kWarps; ++w) m = lse_merge(m, red[w]);
    return m;
}


// Shared-memory slot of local w2 row t.  With w2_split the even rows come first and the odd
// rows after them, so the threads of a warp that take adjacent row pairs (2t, 2t+1) read
// consecutive slots: no bank conflicts with the 16-byte row padding.
__device__ __forceinline__ int w2_slot(const MarkovArgs& a, int t) {
    return a.w2_split ? ((t & 1) ? (a.slice >> 1) + (t >> 1) : (t >> 1)) : t;
}

template <typename WT, bool kTC>
__global__ void __launch_bounds__(kThreads, 1) markov_generic_kernel(MarkovArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sp = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~static_cast<uintptr_t>(15));
    __shared__ unsigned long long s_red[4][kWarps];   // [request parity][pass]: see block_max_u64_t0
    __shared__ float2 s_red2[kWarps];
    __shared__ float s_bcast[2];
    __shared__ float s_temp[256];                     // temperatures of the first 256 requests
    __shared__ float s_inv[256];                      // their reciprocals (1 for greedy)
    __shared__ unsigned long long s_win[kExchangeMaxBN];  // exchange: the step's best key per request
    __shared__ int s_tok[kExchangeMaxBN];                  // exchange: winners [step][request]
    __shared__ __align__(8) uint64_t s_mma_bar;            // tensor path: the step's MMAs completed
    __shared__ uint32_t s_tmem;                            // tensor path: accumulator base

    const int v_lo = blockIdx.x * a.slice;
    const int v_hi = min(a.V, v_lo + a.slice);
    const int n_local = max(0, v_hi - v_lo);
    const int tid = threadIdx.x;

    // shared-memory carve-up: [w2 cache][z store][E][prev]; the tensor path keeps the slice in
    // tensor memory and has the 1024-byte aligned B operand in place of the w2 cache
    uint8_t* w2s = sp;
    uint8_t* bop = nullptr;
    uint8_t* stage = nullptr;
    if constexpr (kTC) {
        bop = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sp) + 1023) & ~static_cast<uintptr_t>(1023));
        stage = bop + kTcBBytes;
        sp = stage + kTcStageBytes;
    } else {
        sp += a.w2_cached ? static_cast<size_t>(a.slice) * a.w2_pitch : 0;
    }
    float* zs = reinterpret_cast<float*>(sp);
    sp += a.z_stored ? sizeof(float) * static_cast<size_t>(a.slice) * a.B : 0;
    float* E = reinterpret_cast<float*>(sp);
    sp += sizeof(float) * static_cast<size_t>(a.B) * a.r;
    int* prev = reinterpret_cast<int*>(sp);

    const size_t row_bytes = sizeof(WT) * static_cast<size_t>(a.r);
    const size_t row_bytes_w1 = row_bytes;
    // Decode fast path (one request, one pair of entries per thread): the base logits and
    // the noise of step i+1 do not depend on the token of step i, so they are fetched and
    // drawn while the block waits at step i's grid barrier.
    const bool fast = a.B == 1 && a.single_pass && a.lse == nullptr && 2 * kThreads >= n_local;
    float pl0 = 0.f, pl1 = 0.f, pg0 = 0.f, pg1 = 0.f;       // this step's logits and noise
    auto prepare = [&](int j, float& l0, float& l1, float& g0, float& g1) {
        const int t = 2 * tid;
        if (t >= n_local) return;
        const int v = v_lo + t;
        const bool two = t + 1 < n_local;
        const float* lr = a.base + static_cast<size_t>(j) * a.V;
        l0 = __ldcs(lr + v);
        l1 = two ? __ldcs(lr + v + 1) : 0.f;
        draft_gumbel_pair(a.seed, a.offset, 0u, static_cast<uint32_t>(j), static_cast<uint32_t>(v), g0, g1);
        if (!two) g1 = 0.f;
    };
    // step 0's inputs are fetched before anything waits on memory: the first request's
    // temperature and anchor per thread, and (tensor path) the anchor's w1 row
    const float T_first = tid < a.B ? __ldg(a.temperature + tid) : 0.f;
    const int anchor_first = tid < a.B ? __ldg(a.anchor + tid) : 0;
    uint4 e_first = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (kTC) {
        if (tid < 8) {
            const int p = __ldg(a.anchor);
            e_first = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.w1) +
                                                           static_cast<size_t>(p >= 0 && p < a.V ? p : 0) * (2 * kTcR)) + tid);
        }
    }
    if constexpr (kTC) {
        // warp w's entries [64 w, 64 w + 64) (its threads' pairs) are 8 KB of contiguous rows: copied
        // in 512-byte warp-wide pieces into the staging area, chunk c of entry e at chunk
        // c ^ ((e / 2) mod 8) of its 128-byte row, so that the row-per-thread reads below are free of
        // bank conflicts; rows past the slice are zero.  The copies land while step 0's noise is
        // drawn and tensor memory is allocated.
        const uint8_t* src = static_cast<const uint8_t*>(a.w2) + static_cast<size_t>(v_lo) * (2 * kTcR);
        const int e_base = 64 * static_cast<int>(warp_id());
        const int lane = static_cast<int>(lane_id());
#pragma unroll 4
        for (int j = 0; j < 16; ++j) {
            const int e = e_base + 4 * j + (lane >> 3), c = lane & 7;
            uint8_t* dst = stage + static_cast<size_t>(e) * 128 + 16 * (c ^ ((e >> 1) & 7));
            if (e < n_local)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                             :: "r"(smem_u32(dst)), "l"(src + static_cast<size_t>(e) * 128 + 16 * c) : "memory");
            else
                *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    if (fast) prepare(0, pl0, pl1, pg0, pg1);
    if constexpr (kTC) {
        for (int idx = tid; idx < static_cast<int>(kTcBBytes / 16); idx += kThreads)
            reinterpret_cast<uint4*>(bop)[idx] = make_uint4(0u, 0u, 0u, 0u);
        if (tid == 0) {
            mbar_init(&s_mma_bar, 1);
            fence_mbarrier_init();
        }
        if (warp_id() == 0) {
            tmem_alloc(&s_tmem, kTcCols);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // entry 2 tid + h into lane 32 (w mod 4) + lane of tile w / 4 + 4 h: 32 columns of bf16
        // pairs in K order
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncwarp();
        const uint32_t w = warp_id();
        const uint32_t lanes = (32u * (w & 3u)) << 16;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = 2 * tid + h;
            const uint8_t* row = stage + static_cast<size_t>(e) * 128;
            uint32_t rw[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 q = *reinterpret_cast<const uint4*>(row + 16 * (c ^ ((e >> 1) & 7)));
                rw[4 * c] = q.x;
                rw[4 * c + 1] = q.y;
                rw[4 * c + 2] = q.z;
                rw[4 * c + 3] = q.w;
            }
            tmem_st32(s_tmem + lanes + kTcACol + 32u * ((w >> 2) + 4u * h), rw);
        }
        tmem_wait_st();
    } else if (a.w2_cached) {
        // load this block's w2 rows once; rows padded to w2_pitch bytes
        const uint8_t* src = static_cast<const uint8_t*>(a.w2) + static_cast<size_t>(v_lo) * row_bytes;
        const int chunks = static_cast<int>(row_bytes / 16);
        // asynchronous 16-byte copies (many in flight); completed before step 0's first pass
        for (int idx = tid; idx < n_local * chunks; idx += kThreads) {
            const int v = idx / chunks, c = idx % chunks;
            const uint32_t dst = smem_u32(w2s + static_cast<size_t>(w2_slot(a, v)) * a.w2_pitch + 16 * c);
            const uint8_t* g = src + static_cast<size_t>(v) * row_bytes + 16 * c;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(g) : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }

    for (int b = tid; b < 256 && b < a.B; b += kThreads) {
        float T = b == tid ? T_first : __ldg(a.temperature + b);
        if (!(T >= 0.f) || isinf(T)) {
            set_status(a.ws, DSPARK_STATUS_NUMERIC);
            T = 0.f;
        }
        s_temp[b] = T;
        s_inv[b] = T > 0.f ? __frcp_rn(T) : 1.f;
    }
    if (a.exchange)
        for (int b = tid; b < a.B; b += kThreads) s_win[b] = 0ull;
    if (a.head.hidden != nullptr) {
        // the calibrated confidence head of "Speculative decoding: from zero to DSpark" §6: the
        // hidden-state half of its logit does not depend on any token, so each block computes it
        // now for the (request, position) pairs it owns (pair p belongs to block p mod grid); the
        // embedding half is added at each step from the E row the block holds then
        const long long pairs = static_cast<long long>(a.B) * a.N;
        const uint32_t lane = lane_id();
        for (long long pr = blockIdx.x + static_cast<long long>(warp_id()) * gridDim.x; pr < pairs;
             pr += static_cast<long long>(kWarps) * gridDim.x) {
            float hs = a.head.hidden_bf16
                           ? conf_lane_dot<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(a.head.hidden) + pr * a.head.H,
                                                          a.head.w_h, a.head.H, lane)
                           : conf_lane_dot<float>(static_cast<const float*>(a.head.hidden) + pr * a.head.H, a.head.w_h,
                                                  a.head.H, lane);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) hs += __shfl_xor_sync(0xFFFFFFFFu, hs, o);
            if (lane == 0) a.lay.conf_h[pr] = hs;
        }
    }
    bool alive = true;
    int tc_fail = 0;                                  // tensor path: an MMA wait timed out
    for (int i = 0; i < a.N && alive; ++i) {
        // ---- 1. previous tokens and the Markov embedding E[b] = w1[prev_b] ----
        for (int b = tid; b < a.B; b += kThreads) {
            int p;
            if (i == 0) {
                p = b == tid ? anchor_first : a.anchor[b];
                if (p < 0 || p >= a.V) {
                    flag_input_index(a.ws);
                    p = 0;
                }
            } else {
                p = a.exchange ? s_tok[(i - 1) * a.B + b] : slot_token(a, i - 1, b);
            }
            prev[b] = p;
        }
        if (i > 0) finish_lse(a, i - 1, tid, kThreads);
        __syncthreads();
        float tb0 = 0.f, tb1 = 0.f;                  // tensor path: this thread's two biases
        if constexpr (kTC) {
            // E = w1[prev] (bf16, unconverted) is row 0 of the B operand: the anchor's row here,
            // later steps' rows were put there by the exchange
            if (i == 0 && tid < 8) reinterpret_cast<uint4*>(bop)[tid] = e_first;
            if (i > 0 && tid == 0) s_win[0] = 0ull;  // every thread read the last winner before the barrier above
            fence_proxy_async_smem();                // operand writes -> the tensor core's view
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            const uint32_t tmem = s_tmem;
            if (tid == 0) {
                constexpr uint32_t idesc = mma_idesc(128, kTcN, false);
                const uint32_t b0 = smem_u32(bop);
#pragma unroll
                for (int m = 0; m < kTcTiles; ++m)
#pragma unroll
                    for (int kk = 0; kk < kTcR / 16; ++kk)
                        mma_issue_ta(tmem + static_cast<uint32_t>(kTcN * m),
                                     tmem + kTcACol + static_cast<uint32_t>(32 * m + 8 * kk),
                                     sw128_kmajor_desc(b0 + static_cast<uint32_t>(32 * kk)), idesc,
                                     kk > 0 ? 1u : 0u);
                mma_commit(&s_mma_bar);
            }
            if (!mbar_wait(&s_mma_bar, static_cast<uint32_t>(i & 1), a.ws, a.timeout_ns, kWaitDecodeMma))
                tc_fail = 1;
            tc_fence_after();
            const uint32_t w = warp_id();
            const uint32_t lanes = (32u * (w & 3u)) << 16;
            if (a.head.hidden != nullptr && w == 1) {
                // one request: E = w1[prev] in bf16 is row 0 of the B operand (unswizzled for row 0)
                const long long pr = static_cast<long long>(i);
                if (pr % gridDim.x == blockIdx.x) {
                    const uint32_t ln = lane_id();
                    float es = conf_lane_dot<__nv_bfloat16>(reinterpret_cast<const __nv_bfloat16*>(bop), a.head.w_e, a.r, ln);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) es += __shfl_xor_sync(0xFFFFFFFFu, es, o);
                    if (ln == 0) a.head.conf[pr] = conf_probability(a.lay.conf_h[pr] + es, a.head.beta, a.head.tau[i], a.ws);
                }
            }
            tb0 = __uint_as_float(tmem_ld1(tmem + lanes + static_cast<uint32_t>(kTcN * (w >> 2))));
            tb1 = __uint_as_float(tmem_ld1(tmem + lanes + static_cast<uint32_t>(kTcN * ((w >> 2) + 4))));
            tmem_wait_ld();
            tc_fence_before();                       // the next step's MMAs overwrite these columns
        } else {
            for (int idx = tid; idx < a.B * a.r; idx += kThreads) {
                const int b = idx / a.r, k = idx % a.r;
                E[idx] = to_f<WT>(static_cast<const WT*>(a.w1)[static_cast<size_t>(prev[b]) * a.r + k]);
            }
            if (i == 0 && a.w2_cached) asm volatile("cp.async.wait_all;" ::: "memory");
            __syncthreads();
            if (a.head.hidden != nullptr) {
                // the embedding half of each owned pair's confidence logit, from E (fp32 in shared memory)
                const uint32_t w = warp_id(), ln = lane_id();
                for (int b = static_cast<int>(w); b < a.B; b += kWarps) {
                    const long long pr = static_cast<long long>(b) * a.N + i;
                    if (pr % gridDim.x != blockIdx.x) continue;
                    float es = conf_lane_dot<float>(E + static_cast<size_t>(b) * a.r, a.head.w_e, a.r, ln);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) es += __shfl_xor_sync(0xFFFFFFFFu, es, o);
                    if (ln == 0) a.head.conf[pr] = conf_probability(a.lay.conf_h[pr] + es, a.head.beta, a.head.tau[i], a.ws);
                }
            }
        }

        unsigned long long* slot = a.lay.slots + static_cast<size_t>(i) * a.B;
        uint32_t* lbs = a.lay.lb + static_cast<size_t>(i) * a.B;
        float2* lse_part = a.lay.lse_part + static_cast<size_t>(i & 1) * kMaxGrid * a.B;

        for (int b = 0; b < a.B; ++b) {
            float T, invT;
            if (b < 256) {
                T = s_temp[b];
                invT = s_inv[b];
            } else {
                T = __ldg(a.temperature + b);
                if (!(T >= 0.f) || isinf(T)) {
                    if (tid == 0) set_status(a.ws, DSPARK_STATUS_NUMERIC);
                    T = 0.f;
                }
                invT = T > 0.f ? __frcp_rn(T) : 1.f;
            }
            const bool hot = T > 0.f;
            const float* lrow = a.base + (static_cast<size_t>(b) * a.N + i) * a.V;
            const float* e = E + static_cast<size_t>(b) * a.r;

            // ---- 2. pass 1: z for the slice, block argmax of z ----
            unsigned long long best = 0ull;
            float2 ls = make_float2(0.f, 0.f);
            bool bad = false;
            if ((hot || kTC) && a.single_pass && a.lse == nullptr) {
                // one pass with noise on every entry; each thread takes two adjacent entries,
                // which share their group word and element counter and interleave for ILP
                // (the tensor path takes greedy requests here too, without the noise)
                for (int t = 2 * tid; t < n_local; t += 2 * kThreads) {
                    const int v = v_lo + t;
                    const bool two = t + 1 < n_local;
                    const uint8_t* wrow0 = a.w2_cached ? w2s + static_cast<size_t>(w2_slot(a, t)) * a.w2_pitch
                                                       : static_cast<const uint8_t*>(a.w2) + static_cast<size_t>(v) * row_bytes;
                    const uint8_t* wrow1 = a.w2_cached ? w2s + static_cast<size_t>(w2_slot(a, t + 1)) * a.w2_pitch
                                                       : wrow0 + row_bytes;
                    float b0, b1;
                    if constexpr (kTC) {
                        b0 = tb0;
                        b1 = tb1;
                    } else {
                        bias_dot2<WT>(wrow0, two ? wrow1 : wrow0, e, a.r, b0, b1);
                    }
                    float l0, l1, g0, g1;
                    if (fast) {
                        l0 = pl0; l1 = pl1; g0 = pg0; g1 = pg1;
                    } else {
                        l0 = __ldcs(lrow + v);
                        l1 = two ? __ldcs(lrow + v + 1) : 0.f;
                        draft_gumbel_pair(a.seed, a.offset, static_cast<uint32_t>(b), static_cast<uint32_t>(i),
                                          static_cast<uint32_t>(v), g0, g1);
                        if (!two) g1 = 0.f;
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h == 1 && !two) break;
                        const uint32_t vv = static_cast<uint32_t>(v + h);
                        const float z = __fmul_rn(__fadd_rn(h ? l1 : l0, h ? b1 : b0), invT);
                        if (z != z) { bad = true; continue; }
                        const float y = hot ? __fadd_rn(z, h ? g1 : g0) : z;
                        if (y != y) continue;
                        const unsigned long long k = argmax_key(y, vv);
                        best = k > best ? k : best;
                    }
                }
            } else
            for (int t = tid; t < n_local; t += kThreads) {
                const int v = v_lo + t;
                const uint8_t* wrow = a.w2_cached ? w2s + static_cast<size_t>(w2_slot(a, t)) * a.w2_pitch
                                                  : static_cast<const uint8_t*>(a.w2) + static_cast<size_t>(v) * row_bytes;
                const float bias = bias_dot<WT>(wrow, e, a.r);
                const float s = __fadd_rn(__ldcs(lrow + v), bias);
                const float z = hot ? __fmul_rn(s, invT) : s;
                if (a.z_stored) zs[static_cast<size_t>(b) * a.slice + t] = z;
                if (z != z) { bad = true; continue; }
                if (a.lse != nullptr && z > -INFINITY) ls = lse_merge(ls, make_float2(z, 1.f));
                // single pass (few elements per block): perturb every element right away
                const float key_val = (hot && a.single_pass) ? __fadd_rn(z, gumbel_at(a, b, i, v)) : z;
                if (key_val != key_val) continue;
                const unsigned long long k = argmax_key(key_val, static_cast<uint32_t>(v));
                best = k > best ? k : best;
            }
            if (bad) set_status(a.ws, DSPARK_STATUS_NUMERIC);
            best = block_max_u64_t0(best, s_red[(b & 1) * 2]);
            if (a.lse != nullptr) {
                ls = block_lse(ls, s_red2);
                if (tid == 0) lse_part[static_cast<size_t>(blockIdx.x) * a.B + b] = ls;
            }
            if (tid == 0 && best != 0ull) {
                const uint32_t vb = key_index(best);
                // the next step may gather this row: bring it into L2 now
                for (size_t l = 0; l < row_bytes_w1; l += 128)
                    prefetch_l2(static_cast<const uint8_t*>(a.w1) + static_cast<size_t>(vb) * row_bytes_w1 + l);
                if (hot && !a.single_pass) {
                    const float zb = float_from_order_bits(static_cast<uint32_t>(best >> 32));
                    const float y = __fadd_rn(zb, gumbel_at(a, b, i, static_cast<int>(vb)));
                    atomicMax(lbs + b, float_order_bits(y));
                    atomicMax(slot + b, argmax_key(y, vb));
                } else if (!a.exchange) {
                    atomicMax(slot + b, best);
                }
            }
            if (a.exchange && tid == 0)   // 1 = this block has no finite candidate (below every key)
                st_relaxed_u64(a.lay.cand + (static_cast<size_t>(i) * gridDim.x + blockIdx.x) * a.B + b,
                               best != 0ull ? best : 1ull);
            if (!hot || a.single_pass) continue;

            // ---- 3. pass 2: Gumbel noise where the element can still win ----
            __syncthreads();
            if (tid == 0) s_bcast[0] = float_from_order_bits(__ldcg(lbs + b));
            __syncthreads();
            const float lb = s_bcast[0];
            best = 0ull;
            for (int t = tid; t < n_local; t += kThreads) {
                const int v = v_lo + t;
                float z;
                if (a.z_stored) {
                    z = zs[static_cast<size_t>(b) * a.slice + t];
                } else {
                    const uint8_t* wrow = a.w2_cached ? w2s + static_cast<size_t>(w2_slot(a, t)) * a.w2_pitch
                                                      : static_cast<const uint8_t*>(a.w2) + static_cast<size_t>(v) * row_bytes;
                    z = __fmul_rn(__fadd_rn(__ldg(lrow + v), bias_dot<WT>(wrow, e, a.r)), invT);
                }
                if (!(__fadd_rn(z, kDraftGumbelMax) >= lb)) continue;  // cannot win (or NaN)
                const float y = __fadd_rn(z, gumbel_at(a, b, i, v));
                if (y != y) continue;
                const unsigned long long k = argmax_key(y, static_cast<uint32_t>(v));
                best = k > best ? k : best;
            }
            best = block_max_u64_t0(best, s_red[(b & 1) * 2 + 1]);
            if (tid == 0 && best != 0ull) atomicMax(slot + b, best);
        }

        // ---- 4. all blocks agree on the step's winners ----
        if (a.exchange) {
            // every block's candidates for this step, polled (bounded) and reduced here
            // the next step's logits and noise do not depend on this step's token: drawn
            // while the other blocks finish
            if (fast && i + 1 < a.N) {
                prepare(i + 1, pl0, pl1, pg0, pg1);
            } else {
                // nothing to prefetch: polling the moment this block has published delays the
                // publications of the others (measured: about 3 us instead of 1.5 us at 149
                // blocks); the first poll waits as long as the prefetch would have taken
                const long long c0 = clock64();
                while (clock64() - c0 < kPollHoldCycles) {
                }
            }
            const int n_ent = static_cast<int>(gridDim.x) * a.B;
            const unsigned long long* cs = a.lay.cand + static_cast<size_t>(i) * n_ent;
            int fail = 0;
            // tensor path: a candidate that beats every one this block has seen so far has its w1
            // row fetched at once, so the winner's row (the next B operand) is in flight while the
            // last candidates arrive
            unsigned long long row_key = 0ull;
            uint4 row[8];
            for (int e = tid; e < n_ent; e += kThreads) {
                unsigned long long k = ld_relaxed_u64(cs + e);
                const long long t0 = global_ns();
                uint32_t spins = 0;
                while (k == 0ull) {
                    if ((++spins & 63u) == 0) {
                        if (aborted(a.ws)) { fail = 1; break; }
                        if (global_ns() - t0 > a.timeout_ns) {
                            atomicOr(&a.ws->status, DSPARK_STATUS_TIMEOUT);
                            atomicExch(&a.ws->detail, kWaitStep + static_cast<uint32_t>(i));
                            fail = 1;
                            break;
                        }
                    }
                    k = ld_relaxed_u64(cs + e);
                }
                if (k > 1ull) {
                    const unsigned long long old = atomicMax(&s_win[e % a.B], k);
                    if constexpr (kTC) {
                        if (k > old && own_index_ok(key_index(k), a.V, a.ws)) {
                            const uint4* src = reinterpret_cast<const uint4*>(
                                static_cast<const uint8_t*>(a.w1) + static_cast<size_t>(key_index(k)) * (2 * kTcR));
#pragma unroll
                            for (int c = 0; c < 8; ++c) row[c] = __ldg(src + c);
                            row_key = k;
                        }
                    }
                }
            }
            alive = __syncthreads_or(fail | tc_fail) == 0;
            if constexpr (kTC) {
                const unsigned long long kw = s_win[0];
                if (kw == 0ull) {                     // no finite candidate: token 0's row
                    if (tid < 8)
                        reinterpret_cast<uint4*>(bop)[tid] = __ldg(reinterpret_cast<const uint4*>(a.w1) + tid);
                } else if (row_key == kw) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) reinterpret_cast<uint4*>(bop)[c] = row[c];
                }
            }
            for (int b = tid; b < a.B; b += kThreads) {
                const unsigned long long k = s_win[b];
                int x = 0;
                if (k == 0ull) set_status(a.ws, DSPARK_STATUS_NUMERIC);    // no finite candidate at all
                else if (own_index_ok(key_index(k), a.V, a.ws)) x = static_cast<int>(key_index(k));
                s_tok[i * a.B + b] = x;
                if constexpr (!kTC) s_win[b] = 0ull;
            }
        } else {
            grid_arrive(a.ws);
            if (fast && i + 1 < a.N) prepare(i + 1, pl0, pl1, pg0, pg1);
            alive = grid_wait(a.ws, static_cast<uint32_t>(i), a.timeout_ns, kWaitStep + i);
        }
    }
    if constexpr (kTC) {
        tc_fence_before();
        __syncthreads();
        if (warp_id() == 0) {
            tc_fence_after();
            tmem_dealloc(s_tmem, kTcCols);
        }
    }
    if (!alive) return;
    __threadfence();
    finish_lse(a, a.N - 1, tid, kThreads);
    if (blockIdx.x == 0) {
        if (a.exchange) __syncthreads();          // the last step's winners, written by other threads
        for (int idx = tid; idx < a.B * a.N; idx += kThreads) {
            const int b = idx / a.N, i = idx % a.N;
            a.tokens[idx] = output_token(a, a.exchange ? s_tok[i * a.B + b] : slot_token(a, i, b));
        }
    }
}

template <typename WT>
dspark_status run_generic(MarkovArgs& a, cudaStream_t stream, const DeviceInfo& dev) {
    // one block per SM; each block owns ceil(V / grid) vocabulary entries (multiple of 32)
    int grid = std::min(dev.sm_count, (a.V + 255) / 256);
    grid = std::max(1, std::min(grid, kMaxGrid));
    a.slice = ((a.V + grid - 1) / grid + 31) & ~31;
    grid = (a.V + a.slice - 1) / a.slice;
    const size_t row_bytes = sizeof(WT) * static_cast<size_t>(a.r);
    a.w2_pitch = static_cast<int>(row_bytes + 16);
    a.w2_cached = (row_bytes % 16 == 0) && static_cast<size_t>(a.slice) * a.w2_pitch <= kW2CacheBytes;
    a.z_stored = sizeof(float) * static_cast<size_t>(a.slice) * a.B <= kZStoreBytes;
    // at most 8 elements per thread and step: one pass with noise on every element is
    // cheaper than publishing a bound and making a second pass
    a.single_pass = static_cast<size_t>(a.slice) * a.B <= static_cast<size_t>(8 * kThreads);
    // few requests and steps, one pass: blocks trade candidates directly (one poll per block
    // and request) instead of atomics on step slots plus a grid barrier
    a.exchange = a.single_pass && a.lse == nullptr && markov_cand_entries(a.B, a.N) > 0 &&
                 static_cast<long long>(grid) * a.B <= kThreads;
    a.w2_split = a.w2_cached && (a.slice % 2 == 0);
    if (static_cast<size_t>(a.B) * a.r > static_cast<size_t>(kMaxEFloats)) {
        set_error("markov_sample: B*r = %d exceeds the %d the sampler holds on chip", a.B * a.r, kMaxEFloats);
        return DSPARK_ERR_UNSUPPORTED;
    }
    // one request with a bf16 head of rank 64 whose slice fits eight 128-row tiles: the bias on
    // the tensor cores
    bool tc = false;
    if constexpr (std::is_same<WT, __nv_bfloat16>::value)
        tc = a.B == 1 && a.r == kTcR && a.single_pass && a.lse == nullptr && a.exchange && a.slice <= kTcRows;
    size_t smem = 16;
    smem += tc ? 1023 + kTcBBytes + kTcStageBytes : a.w2_cached ? static_cast<size_t>(a.slice) * a.w2_pitch : 0;
    smem += a.z_stored ? sizeof(float) * static_cast<size_t>(a.slice) * a.B : 0;
    smem += sizeof(float) * static_cast<size_t>(a.B) * a.r + sizeof(int) * static_cast<size_t>(a.B);
    if (smem > dev.smem_optin) {
        set_error("markov_sample: needs %zu bytes of shared memory", smem);
        return DSPARK_ERR_UNSUPPORTED;
    }
    auto kernel = markov_generic_kernel<WT, false>;
    if constexpr (std::is_same<WT, __nv_bfloat16>::value)
        if (tc) kernel = markov_generic_kernel<WT, true>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(markov_sample)");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
    if (e != cudaSuccess) return cuda_error(e, "occupancy(markov_sample)");
    if (per_sm * dev.sm_count < grid) {
        set_error("markov_sample: %d blocks cannot be co-resident", grid);
        return DSPARK_ERR_UNSUPPORTED;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess) return cuda_error(e, "launch(markov_sample)");
    return DSPARK_OK;
}

}  // namespace

size_t markov_workspace_bytes(int B, int N) {
    const size_t nb = static_cast<size_t>(B) * N;
    size_t bytes = sizeof(WsHeader) + nb * sizeof(unsigned long long) + nb * sizeof(uint32_t) +
                   sizeof(uint32_t) * static_cast<size_t>(N) * kPubStride;
    bytes = (bytes + 15) & ~static_cast<size_t>(15);
    bytes += sizeof(unsigned long long) * markov_cand_entries(B, N);
    bytes += 2 * static_cast<size_t>(kMaxGrid) * B * sizeof(float2);
    bytes += nb * sizeof(float);                      // confidence head: hidden-row dot per pair
    return bytes;
}

dspark_status launch_markov_sample(const float* base_logits, const int32_t* anchor, const void* w1,
                                   const void* w2, dspark_dtype wdtype, const float* temperature,
                                   uint64_t seed, uint32_t offset, int B, int N, int V, int r,
                                   int32_t* draft_tokens, float* lse, const int32_t* d2t, int d2t_offset,
                                   int V_target, const ConfHead* head, void* ws, cudaStream_t stream,
                                   const DeviceInfo& dev) {
    // clear header, slots, bounds, publication counters and the candidate entries a grid of
    // at most one block per SM uses (the lse partials need no clearing)
    const MarkovLayout lay = markov_layout(ws, B, N);
    size_t clear = static_cast<size_t>(reinterpret_cast<uint8_t*>(lay.cand) - static_cast<uint8_t*>(ws));
    if (markov_cand_entries(B, N) > 0)
        clear += sizeof(unsigned long long) * static_cast<size_t>(N) * std::min(dev.sm_count, kMaxGrid) * B;
    dspark_status st = clear_workspace(ws, clear, stream);
    if (st != DSPARK_OK) return st;
    MarkovArgs a = {};
    a.base = base_logits;
    a.anchor = anchor;
    a.w1 = w1;
    a.w2 = w2;
    a.temperature = temperature;
    a.tokens = draft_tokens;
    a.lse = lse;
    a.ws = static_cast<WsHeader*>(ws);
    a.lay = markov_layout(ws, B, N);
    a.seed = seed;
    a.offset = offset;
    a.B = B;
    a.N = N;
    a.V = V;
    a.r = r;
    a.d2t = d2t;
    a.d2t_offset = d2t_offset;
    a.V_target = V_target;
    if (head != nullptr) a.head = *head;
    a.timeout_ns = kDefaultTimeoutNs;
    if (markov_tc_eligible(B, N, V, r, wdtype, base_logits, lse, dev.sm_count))
        return launch_markov_tc(a, stream, dev);
    if (wdtype == DSPARK_BF16) return run_generic<__nv_bfloat16>(a, stream, dev);
    return run_generic<float>(a, stream, dev);
}

}  // namespace dspark
