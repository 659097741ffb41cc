// Lossless speculative verification.
//
// "Speculative decoding: from zero to DSpark" §2: draft token x_k is accepted
// with probability min(1, p_t(x_k)/p_d(x_k)); the first rejection k* draws a
// correction from norm(max(0, p_t - p_d)); if all tested tokens pass, a bonus
// token is drawn from p_t at the position after the block.
//
// S blocks per request (S = 1 when the batch alone fills the GPU, more when it
// does not, so a single request still streams its 1-2 vocabulary rows at full
// bandwidth).  Every block of request b:
//   1. checks all tested positions k < L_b at once (one thread each):
//      fl32(u_k * p_d[x_k]) < p_t[x_k]; k* = the smallest failing k
//   2. streams its share of the residual (or bonus) row: each warp turns 128
//      consecutive entries into integer masses q_v = floor(w_v * 2^40) and
//      writes their sum to the workspace
// The last block of the request to finish (an atomic counter) then
//   3. sums the segment masses, t = floor(R * Q / 2^64), finds the segment
//      holding t with a block-wide exclusive scan, re-reads that segment with
//      one warp and picks the token with an inclusive warp scan.
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

struct VerifyArgs {
    const float* p_t;
    const float* p_d;
    const int32_t* tokens;
    const int32_t* lengths;
    int32_t* out;
    int32_t* n_acc;
    WsHeader* ws;
    uint32_t* done;              // [B] blocks finished per request
    unsigned long long* seg;     // [B][n_seg] segment masses
    uint64_t seed;
    uint32_t offset;
    int B, gamma, V, n_seg, splits;
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

// Masses of segments [s0, s1) of the row into dst[segment].
__device__ void segment_sums(const float* rt, const float* rd, int V, bool vec, int s0, int s1,
                             unsigned long long* dst) {
    const uint32_t warp = warp_id(), lane = lane_id();
    for (int sgi = s0 + static_cast<int>(warp); sgi < s1; sgi += kWarps) {
        unsigned long long q[4];
        masses4(rt, rd, sgi * kSeg + 4 * static_cast<int>(lane), V, vec, q);
        const unsigned long long s = warp_sum_u64(q[0] + q[1] + q[2] + q[3]);
        if (lane == 0) dst[sgi] = s;
    }
}

__device__ unsigned long long block_sum_u64(unsigned long long x, unsigned long long* red) {
    x = warp_sum_u64(x);
    __syncthreads();
    if (lane_id() == 0) red[warp_id()] = x;
    __syncthreads();
    unsigned long long s = 0;
    for (int w = 0; w < kWarps; ++w) s += red[w];
    return s;
}

__global__ void __launch_bounds__(kThreads) verify_kernel(VerifyArgs a) {
    extern __shared__ unsigned long long s_seg[];         // [n_seg] (last block only)
    __shared__ unsigned long long s_red[kWarps];
    __shared__ unsigned long long s_scan[kWarps];
    __shared__ int s_kstar, s_bad, s_pick, s_last;
    __shared__ unsigned long long s_tloc;

    const int b = blockIdx.x / a.splits;
    const int split = blockIdx.x % a.splits;
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
        if (split == 0) {
            if (tid == 0) set_status(a.ws, DSPARK_STATUS_INPUT_RANGE);
            for (int k = tid; k <= g; k += kThreads) out[k] = -1;
            if (tid == 0) a.n_acc[b] = 0;
        }
        return;
    }
    const int kstar = s_kstar;
    const bool rej = kstar < Lb;

    // ---- 2. this block's share of the residual (or bonus) row ----
    const float* rt = a.p_t + (static_cast<size_t>(b) * (g + 1) + kstar) * V;
    const float* rd = rej ? a.p_d + (static_cast<size_t>(b) * g + kstar) * V : nullptr;
    const bool vec = (V & 3) == 0;
    const int n_seg = a.n_seg;
    unsigned long long* seg = a.seg + static_cast<size_t>(b) * n_seg;
    const int s0 = static_cast<int>((static_cast<long long>(split) * n_seg) / a.splits);
    const int s1 = static_cast<int>((static_cast<long long>(split + 1) * n_seg) / a.splits);
    segment_sums(rt, rd, V, vec, s0, s1, seg);

    // ---- the last block of the request finishes it ----
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(a.done + b, 1u) == static_cast<uint32_t>(a.splits - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    unsigned long long mine = 0;
    for (int s = tid; s < n_seg; s += kThreads) {
        const unsigned long long v = __ldcg(seg + s);
        s_seg[s] = v;
        mine += v;
    }
    unsigned long long Q = block_sum_u64(mine, s_red);
    if (Q == 0 && rd != nullptr) {                 // residual without mass: use the p_t row
        rd = nullptr;
        __syncthreads();
        segment_sums(rt, rd, V, vec, 0, n_seg, s_seg);
        __syncthreads();
        mine = 0;
        for (int s = tid; s < n_seg; s += kThreads) mine += s_seg[s];
        Q = block_sum_u64(mine, s_red);
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
        __syncthreads();
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
        // block-wide exclusive scan over segment masses, each thread owning a run of segments
        const int per = (n_seg + kThreads - 1) / kThreads;
        const int r0 = tid * per, r1 = min(n_seg, r0 + per);
        unsigned long long run = 0;
        for (int s = r0; s < r1; ++s) run += s_seg[s];
        const unsigned long long incl = warp_incl_scan_u64(run);
        if (lane_id() == 31) s_scan[warp_id()] = incl;
        __syncthreads();
        unsigned long long before = incl - run;
        for (int w2 = 0; w2 < static_cast<int>(warp_id()); ++w2) before += s_scan[w2];
        for (int s = r0; s < r1; ++s) {
            const unsigned long long sv = s_seg[s];
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
            unsigned long long acc = incl_l - lane_sum;
            int pick = -1;
            for (int j = 0; j < 4; ++j) {
                acc += q[j];
                if (pick < 0 && acc > tl) pick = j;
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

int n_segments(int V) { return (V + kSeg - 1) / kSeg; }

size_t done_bytes(int B) { return (sizeof(uint32_t) * static_cast<size_t>(B) + 15) & ~static_cast<size_t>(15); }

}  // namespace

size_t verify_workspace_bytes(int B, int V) {
    return sizeof(WsHeader) + done_bytes(B) + sizeof(unsigned long long) * static_cast<size_t>(B) * n_segments(V);
}

dspark_status launch_verify(const float* p_target, const float* p_draft, const int32_t* draft_tokens,
                            const int32_t* lengths, uint64_t seed, uint32_t offset, int B, int gamma,
                            int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                            cudaStream_t stream, const DeviceInfo& dev) {
    const int n_seg = n_segments(V);
    const size_t smem = sizeof(unsigned long long) * static_cast<size_t>(n_seg);
    if (smem > dev.smem_optin) {
        set_error("verify: V=%d needs %zu bytes of shared memory", V, smem);
        return DSPARK_ERR_UNSUPPORTED;
    }
    dspark_status st = clear_workspace(ws, sizeof(WsHeader) + done_bytes(B), stream);
    if (st != DSPARK_OK) return st;
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
    a.done = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + sizeof(WsHeader));
    a.seg = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + sizeof(WsHeader) + done_bytes(B));
    a.seed = seed;
    a.offset = offset;
    a.B = B;
    a.gamma = gamma;
    a.V = V;
    a.n_seg = n_seg;
    // enough blocks to cover the GPU twice, but at least 8 segments (1024 entries) per block
    a.splits = B >= dev.sm_count ? 1 : std::max(1, std::min((2 * dev.sm_count + B - 1) / B, n_seg / 8));
    const long long grid = static_cast<long long>(B) * a.splits;
    if (grid > 0x7FFFFFFFLL) {
        set_error("verify: too many requests (%d)", B);
        return DSPARK_ERR_UNSUPPORTED;
    }
    verify_kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(verify)");
    return DSPARK_OK;
}

}  // namespace dspark
