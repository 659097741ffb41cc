// Lossless speculative verification, one block per request.
//
// "Speculative decoding: from zero to DSpark" §2: draft token x_k is accepted
// with probability min(1, p_t(x_k)/p_d(x_k)); the first rejection k* draws a
// correction from norm(max(0, p_t - p_d)); if all tested tokens pass, a bonus
// token is drawn from p_t at the position after the block.
//
// Per request (block):
//   1. all tested positions k < L_b are checked at once (one thread each):
//      fl32(u_k * p_d[x_k]) < p_t[x_k]; k* = the smallest failing k (shared atomicMin)
//   2. one streaming pass over the residual (or bonus) row: each warp turns 128
//      consecutive entries into integer masses q_v = floor(w_v * 2^40) and
//      stores their sum; Q = sum over the row
//   3. t = floor(R * Q / 2^64); a block-wide exclusive scan over the 128-entry
//      sums finds the segment holding t; one warp re-reads that segment and an
//      inclusive warp scan picks the token.
// Integer masses make the result independent of the summation order, so the
// token equals the CPU reference bit for bit.
#include "device_common.cuh"
#include "host_common.h"

#include <algorithm>

namespace dspark {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kSeg = 128;                        // entries per warp segment (4 per lane)
constexpr int kMaxSegs = (1 << 24) / kSeg;       // V <= 2^24

struct VerifyArgs {
    const float* p_t;
    const float* p_d;
    const int32_t* tokens;
    const int32_t* lengths;
    int32_t* out;
    int32_t* n_acc;
    WsHeader* ws;
    uint64_t seed;
    uint32_t offset;
    int B, gamma, V;
};

// Four consecutive entries starting at e (a multiple of 4), zero past the end.
__device__ __forceinline__ float4 load4(const float* row, int e, int V, bool vec) {
    if (vec && e + 4 <= V) return __ldcs(reinterpret_cast<const float4*>(row + e));
    float4 f;
    f.x = e + 0 < V ? __ldcs(row + e + 0) : 0.f;
    f.y = e + 1 < V ? __ldcs(row + e + 1) : 0.f;
    f.z = e + 2 < V ? __ldcs(row + e + 2) : 0.f;
    f.w = e + 3 < V ? __ldcs(row + e + 3) : 0.f;
    return f;
}

// q = floor(w * 2^40) for w in [0, 1]; w * 2^40 is exact, the conversion truncates.
__device__ __forceinline__ unsigned long long mass(float w) {
    return __float2ull_rz(__fmul_rn(w, 0x1p40f));
}

__device__ __forceinline__ void masses4(const float* rt, const float* rd, int e, int V, bool vec,
                                        unsigned long long (&q)[4]) {
    const float4 t = load4(rt, e, V, vec);
    if (rd != nullptr) {
        const float4 d = load4(rd, e, V, vec);
        q[0] = mass(fmaxf(0.f, __fsub_rn(t.x, d.x)));
        q[1] = mass(fmaxf(0.f, __fsub_rn(t.y, d.y)));
        q[2] = mass(fmaxf(0.f, __fsub_rn(t.z, d.z)));
        q[3] = mass(fmaxf(0.f, __fsub_rn(t.w, d.w)));
    } else {
        q[0] = mass(fmaxf(0.f, t.x));
        q[1] = mass(fmaxf(0.f, t.y));
        q[2] = mass(fmaxf(0.f, t.z));
        q[3] = mass(fmaxf(0.f, t.w));
    }
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
}

__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long x) {
    const uint32_t lane = lane_id();
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= static_cast<uint32_t>(o)) x += y;
    }
    return x;
}

// Pass over the row: per-segment sums into seg[] and the total.
__device__ unsigned long long segment_sums(const float* rt, const float* rd, int V, bool vec,
                                           unsigned long long* seg, unsigned long long* red) {
    const int n_seg = (V + kSeg - 1) / kSeg;
    const uint32_t warp = warp_id(), lane = lane_id();
    unsigned long long total = 0;
    for (int sgi = warp; sgi < n_seg; sgi += kWarps) {
        unsigned long long q[4];
        masses4(rt, rd, sgi * kSeg + 4 * static_cast<int>(lane), V, vec, q);
        const unsigned long long s = warp_sum_u64(q[0] + q[1] + q[2] + q[3]);
        if (lane == 0) seg[sgi] = s;
        total += s;
    }
    __syncthreads();
    if (lane == 0) red[warp] = total;
    __syncthreads();
    unsigned long long Q = 0;
    for (int w = 0; w < kWarps; ++w) Q += red[w];
    __syncthreads();
    return Q;
}

__global__ void __launch_bounds__(kThreads) verify_kernel(VerifyArgs a) {
    extern __shared__ unsigned long long seg[];           // [n_seg] segment sums
    __shared__ unsigned long long s_red[kWarps];
    __shared__ unsigned long long s_scan[kWarps];
    __shared__ int s_kstar, s_bad, s_pick;
    __shared__ unsigned long long s_tloc;

    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const int V = a.V, g = a.gamma;
    int32_t* out = a.out + static_cast<size_t>(b) * (g + 1);

    int Lb = a.lengths != nullptr ? a.lengths[b] : g;
    if (tid == 0) {
        s_kstar = (Lb >= 0 && Lb <= g) ? Lb : 0;
        s_bad = (Lb < 0 || Lb > g) ? 1 : 0;
        s_pick = -1;
    }
    __syncthreads();
    if (s_bad) Lb = 0;

    // ---- 1. ratio test at every tested position ----
    for (int k = tid; k < Lb; k += kThreads) {
        const int x = a.tokens[static_cast<size_t>(b) * g + k];
        if (x < 0 || x >= V) {
            atomicExch(&s_bad, 1);
            continue;
        }
        const uint4 w = philox_at(a.seed, a.offset, 0u, static_cast<uint32_t>(b), kStreamAccept,
                                  static_cast<uint32_t>(k));
        const float u = uniform_from_word(w.x);
        const float pd = a.p_d[(static_cast<size_t>(b) * g + k) * V + x];
        const float pt = a.p_t[(static_cast<size_t>(b) * (g + 1) + k) * V + x];
        if (!(__fmul_rn(u, pd) < pt)) atomicMin(&s_kstar, k);
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) set_status(a.ws, DSPARK_STATUS_INPUT_RANGE);
        for (int k = tid; k <= g; k += kThreads) out[k] = -1;
        if (tid == 0) a.n_acc[b] = 0;
        return;
    }
    const int kstar = s_kstar;
    const bool rej = kstar < Lb;

    // ---- 2. residual (or bonus) row -> segment masses ----
    const float* rt = a.p_t + (static_cast<size_t>(b) * (g + 1) + kstar) * V;
    const float* rd = rej ? a.p_d + (static_cast<size_t>(b) * g + kstar) * V : nullptr;
    const bool vec = (V & 3) == 0;
    unsigned long long Q = segment_sums(rt, rd, V, vec, seg, s_red);
    if (Q == 0 && rd != nullptr) {                 // residual without mass: use the p_t row
        rd = nullptr;
        Q = segment_sums(rt, rd, V, vec, seg, s_red);
    }

    int y;
    if (Q == 0) {
        // no mass at all: argmax of p_t (lowest index on ties)
        unsigned long long best = 0;
        for (int v = tid; v < V; v += kThreads) {
            const unsigned long long k = argmax_key(rt[v], static_cast<uint32_t>(v));
            best = k > best ? k : best;
        }
        best = warp_max_u64(best);
        if (lane_id() == 0) s_red[warp_id()] = best;
        __syncthreads();
        unsigned long long m = 0;
        for (int w = 0; w < kWarps; ++w) m = s_red[w] > m ? s_red[w] : m;
        y = static_cast<int>(key_index(m));
        if (tid == 0) set_status(a.ws, DSPARK_STATUS_NUMERIC);
    } else {
        // ---- 3. inverse CDF: t = floor(R * Q / 2^64) ----
        const uint4 w = philox_at(a.seed, a.offset, 0u, static_cast<uint32_t>(b), kStreamResample,
                                  static_cast<uint32_t>(kstar));
        const unsigned long long R = (static_cast<unsigned long long>(w.x) << 32) | w.y;
        const unsigned long long t = __umul64hi(R, Q);
        // block-wide exclusive scan over segment sums, each thread owning a run of segments
        const int n_seg = (V + kSeg - 1) / kSeg;
        const int per = (n_seg + kThreads - 1) / kThreads;
        const int s0 = tid * per, s1 = min(n_seg, s0 + per);
        unsigned long long mine = 0;
        for (int s = s0; s < s1; ++s) mine += seg[s];
        const unsigned long long incl = warp_incl_scan_u64(mine);
        if (lane_id() == 31) s_scan[warp_id()] = incl;
        __syncthreads();
        unsigned long long before = incl - mine;
        for (int w2 = 0; w2 < static_cast<int>(warp_id()); ++w2) before += s_scan[w2];
        for (int s = s0; s < s1; ++s) {
            const unsigned long long sv = seg[s];
            if (before <= t && t < before + sv) {   // exactly one segment holds t
                s_pick = s;
                s_tloc = t - before;
            }
            before += sv;
        }
        __syncthreads();
        const int s = s_pick;
        if (warp_id() == 0) {
            const unsigned long long tl = s_tloc;
            unsigned long long q[4];
            masses4(rt, rd, s * kSeg + 4 * static_cast<int>(lane_id()), V, vec, q);
            const unsigned long long lane_sum = q[0] + q[1] + q[2] + q[3];
            const unsigned long long incl_l = warp_incl_scan_u64(lane_sum);
            unsigned long long run = incl_l - lane_sum;
            int pick = -1;
            for (int j = 0; j < 4; ++j) {
                run += q[j];
                if (pick < 0 && run > tl) pick = j;
            }
            const bool has = (incl_l - lane_sum <= tl) && (tl < incl_l);
            const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, has);
            const int src = __ffs(ballot) - 1;
            const int pj = __shfl_sync(0xFFFFFFFFu, pick, src < 0 ? 0 : src);
            if (lane_id() == 0) s_pick = src < 0 ? -1 : s * kSeg + 4 * src + pj;
        }
        __syncthreads();
        y = s_pick;
        if (y < 0 || y >= V) {            // cannot happen when Q > 0; kept as a guard
            if (tid == 0) set_status(a.ws, DSPARK_STATUS_INTERNAL);
            y = 0;
        }
    }

    // ---- outputs: accepted prefix, the correction / bonus token, then -1 ----
    for (int k = tid; k <= g; k += kThreads) {
        int v = -1;
        if (k < kstar) v = a.tokens[static_cast<size_t>(b) * g + k];
        else if (k == kstar) v = y;
        out[k] = v;
    }
    if (tid == 0) a.n_acc[b] = kstar;
}

}  // namespace

dspark_status launch_verify(const float* p_target, const float* p_draft, const int32_t* draft_tokens,
                            const int32_t* lengths, uint64_t seed, uint32_t offset, int B, int gamma,
                            int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                            cudaStream_t stream, const DeviceInfo& dev) {
    dspark_status st = clear_workspace(ws, sizeof(WsHeader), stream);
    if (st != DSPARK_OK) return st;
    const int n_seg = (V + kSeg - 1) / kSeg;
    if (n_seg > kMaxSegs) {
        set_error("verify: V=%d too large", V);
        return DSPARK_ERR_UNSUPPORTED;
    }
    const size_t smem = sizeof(unsigned long long) * static_cast<size_t>(n_seg);
    if (smem > dev.smem_optin) {
        set_error("verify: V=%d needs %zu bytes of shared memory", V, smem);
        return DSPARK_ERR_UNSUPPORTED;
    }
    cudaError_t e = cudaFuncSetAttribute(verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(verify)");
    VerifyArgs a;
    a.p_t = p_target;
    a.p_d = p_draft;
    a.tokens = draft_tokens;
    a.lengths = lengths;
    a.out = out_tokens;
    a.n_acc = num_accepted;
    a.ws = static_cast<WsHeader*>(ws);
    a.seed = seed;
    a.offset = offset;
    a.B = B;
    a.gamma = gamma;
    a.V = V;
    verify_kernel<<<B, kThreads, smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(verify)");
    return DSPARK_OK;
}

}  // namespace dspark
