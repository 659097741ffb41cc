// Lossless speculative verification.
//
// "Speculative decoding: from zero to DSpark" §2: draft token x_k is accepted
// with probability min(1, p_t(x_k)/p_d(x_k)); the first rejection k* draws a
// correction from norm(max(0, p_t - p_d)); if all tested tokens pass, a bonus
// token is drawn from p_t at the position after the block.
//
// One launch (two blocks per SM).  The B * ceil(V / 512) segments of the rows to
// stream -- residual rows p_t[k*], p_d[k*] for a rejection, the bonus row p_t[L_b]
// otherwise -- are cut into equal contiguous ranges, one per block.  A block first
// decides the requests its range touches, one warp per request checking all tested
// positions k < L_b at once, one lane each: fl32(u_k * p_d[x_k]) < p_t[x_k]; k* = the
// smallest failing k (every block touching a request reaches the same k*, so no
// decision crosses blocks).  Each warp then turns 512 consecutive entries into
// integer masses q_v = floor(w_v * 2^40) and writes their sum to the workspace.  The block that completes a request's
// segment count (an atomic counter) then sums the segment masses,
// t = floor(R * Q / 2^64), finds the segment holding t with a block-wide
// exclusive scan, re-reads that segment with one warp (128 entries at a time)
// and picks the token with an inclusive warp scan.  Integer masses make the
// result independent of the summation order, so the token equals the CPU
// reference bit for bit.
#include "device_common.cuh"
#include "host_common.h"

#include <algorithm>

namespace dspark {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kSeg = 512;                        // entries per warp segment (16 per lane)
constexpr int kSlice = 128;                      // a segment is 4 slices of 4 consecutive entries per lane

struct VerifyArgs {
    const float* p_t;
    const float* p_d;
    const int32_t* tokens;
    const int32_t* lengths;
    int32_t* out;
    int32_t* n_acc;
    WsHeader* ws;
    uint32_t* done;              // [B] segments finished per request
    unsigned long long* seg;     // [B][n_seg] segment masses
    uint64_t seed;
    uint32_t offset;
    int B, gamma, V, n_seg, grid;
    long long total_seg;         // B * n_seg
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

// q = floor(w * 2^40) for w >= 0 (never NaN: it comes out of fmaxf(0, .)), read off the
// float's bits with integer operations only: w = m * 2^(e - 150) for a normal w with biased
// exponent e and 24-bit significand m, so w * 2^40 = m * 2^(e - 110).  Subnormals give 0;
// values whose product reaches 2^64 (only possible for w > 1, i.e. bad input) saturate as a
// float-to-integer conversion would.  A float-to-u64 conversion runs on the FP64 pipe, which
// is narrow on this GPU; this keeps the row stream memory-bound.
__device__ __forceinline__ unsigned long long mass(float w) {
    const uint32_t bits = __float_as_uint(w) & 0x7FFFFFFFu;      // -0 (fmaxf may keep it) is 0
    const int e = static_cast<int>(bits >> 23);
    const unsigned long long m = (bits & 0x7FFFFFu) | 0x800000u;
    const int sh = e - 110;
    if (e == 0 || sh <= -24) return 0ull;
    if (sh >= 41) return ~0ull;
    return sh >= 0 ? m << sh : m >> -sh;
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

__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long x) {
    const uint32_t lane = lane_id();
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= static_cast<uint32_t>(o)) x += y;
    }
    return x;
}

// Masses of segments [s0, s1) of the row into dst[segment], one warp per segment: a lane's
// 16 entries are four float4 of each row, all loaded before any is used.
__device__ void segment_sums(const float* rt, const float* rd, int V, bool vec, int s0, int s1,
                             unsigned long long* dst) {
    const uint32_t warp = warp_id(), lane = lane_id();
    for (int sgi = s0 + static_cast<int>(warp); sgi < s1; sgi += kWarps) {
        const int e0 = sgi * kSeg + 4 * static_cast<int>(lane);
        float4 t[4], d[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) t[i] = load4(rt, e0 + i * kSlice, V, vec);
        if (rd != nullptr) {
#pragma unroll
            for (int i = 0; i < 4; ++i) d[i] = load4(rd, e0 + i * kSlice, V, vec);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) d[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        unsigned long long sum = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sum += mass(fmaxf(0.f, __fsub_rn(t[i].x, d[i].x))) + mass(fmaxf(0.f, __fsub_rn(t[i].y, d[i].y))) +
                   mass(fmaxf(0.f, __fsub_rn(t[i].z, d[i].z))) + mass(fmaxf(0.f, __fsub_rn(t[i].w, d[i].w)));
        }
        sum = warp_sum_u64(sum);
        if (lane == 0) dst[sgi] = sum;
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

// Decision of request b, (k* << 1) | rejected, or -1 for bad input (then INPUT_RANGE is set);
// warp-collective, one lane per tested position, the result in every lane.
__device__ int decide_request(const VerifyArgs& a, int b) {
    const uint32_t lane = lane_id();
    const int V = a.V, g = a.gamma;
    const int Lb = a.lengths != nullptr ? a.lengths[b] : g;
    bool bad = Lb < 0 || Lb > g;
    int kmin = bad ? 0 : Lb;
    if (!bad) {
        for (int k = static_cast<int>(lane); k < Lb; k += 32) {
            const int x = a.tokens[static_cast<size_t>(b) * g + k];
            if (x < 0 || x >= V) {
                bad = true;
                continue;
            }
            const uint4 w = philox_at(a.seed, a.offset, 0u, static_cast<uint32_t>(b), kStreamAccept,
                                      static_cast<uint32_t>(k));
            const float u = uniform_from_word(w.x);
            const float pd = a.p_d[(static_cast<size_t>(b) * g + k) * V + x];
            const float pt = a.p_t[(static_cast<size_t>(b) * (g + 1) + k) * V + x];
            if (!(__fmul_rn(u, pd) < pt)) kmin = min(kmin, k);
        }
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    if (bad && lane == 0) flag_input_index(a.ws);
    return bad ? -1 : ((kmin << 1) | (kmin < Lb ? 1 : 0));
}

// The last block to stream a request draws its token and writes its outputs.
__device__ void finish_request(const VerifyArgs& a, int b, int dec, unsigned long long* s_seg,
                               unsigned long long* s_red, unsigned long long* s_scan, int* s_pick,
                               unsigned long long* s_tloc) {
    const int tid = threadIdx.x;
    const int V = a.V, g = a.gamma, n_seg = a.n_seg;
    int32_t* out = a.out + static_cast<size_t>(b) * (g + 1);
    if (dec < 0) {                               // bad input: nothing accepted, no token
        for (int k = tid; k <= g; k += kThreads) out[k] = -1;
        if (tid == 0) a.n_acc[b] = 0;
        return;
    }
    const int kstar = dec >> 1;
    const float* rt = a.p_t + (static_cast<size_t>(b) * (g + 1) + kstar) * V;
    const float* rd = (dec & 1) ? a.p_d + (static_cast<size_t>(b) * g + kstar) * V : nullptr;
    const bool vec = (V & 3) == 0;
    const unsigned long long* seg = a.seg + static_cast<size_t>(b) * n_seg;

    unsigned long long mine = 0;
    for (int s = tid; s < n_seg; s += kThreads) {
        const unsigned long long v = __ldcg(seg + s);
        s_seg[s] = v;
        mine += v;
    }
    unsigned long long Q = block_sum_u64(mine, s_red);
    if (Q == 0 && rd != nullptr) {               // residual without mass: use the p_t row
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
        // ---- inverse CDF: t = floor(R * Q / 2^64) ----
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
                *s_pick = s;
                *s_tloc = t - before;
            }
            before += sv;
        }
        __syncthreads();
        const int s = *s_pick;
        if (warp_id() == 0) {
            // the segment's four 128-entry slices are loaded at once (one memory round trip),
            // then walked to the one holding tl, and tl is picked inside it
            unsigned long long tl = *s_tloc;
            int pick_v = -1;
            unsigned long long qs[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                masses4(rt, rd, s * kSeg + i * kSlice + 4 * static_cast<int>(lane_id()), V, vec, qs[i]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (pick_v >= 0) break;
                const unsigned long long (&q)[4] = qs[i];
                const int e = s * kSeg + i * kSlice;
                const unsigned long long lane_sum = q[0] + q[1] + q[2] + q[3];
                const unsigned long long incl_l = warp_incl_scan_u64(lane_sum);
                const unsigned long long slice = __shfl_sync(0xFFFFFFFFu, incl_l, 31);
                if (tl >= slice) {
                    tl -= slice;
                    continue;
                }
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
                pick_v = src < 0 ? -2 : e + 4 * src + pj;
            }
            if (lane_id() == 0) *s_pick = pick_v < 0 ? -1 : pick_v;
        }
        __syncthreads();
        y = *s_pick;
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

// Streams block blockIdx.x's contiguous range of the B * n_seg row segments.
__global__ void __launch_bounds__(kThreads, 2) verify_stream_kernel(VerifyArgs a) {
    extern __shared__ unsigned long long s_seg[];         // [n_seg] (finishing blocks only), then the
                                                          // decisions of the block's requests
    __shared__ unsigned long long s_red[kWarps];
    __shared__ unsigned long long s_scan[kWarps];
    __shared__ int s_pick, s_last;
    __shared__ unsigned long long s_tloc;

    const int tid = threadIdx.x;
    const int V = a.V, g = a.gamma, n_seg = a.n_seg;
    const bool vec = (V & 3) == 0;
    const long long T = a.total_seg;
    long long f = T * blockIdx.x / a.grid;
    const long long f1 = T * (blockIdx.x + 1) / a.grid;
    int* s_dec = reinterpret_cast<int*>(s_seg + n_seg);

    // the decisions of the requests [b_first, b_last] this block streams, one warp each
    const int b_first = static_cast<int>(f / n_seg);
    const int n_req = f < f1 ? static_cast<int>((f1 - 1) / n_seg) - b_first + 1 : 0;
    for (int j = static_cast<int>(warp_id()); j < n_req; j += kWarps) {
        const int dec = decide_request(a, b_first + j);
        if (lane_id() == 0) s_dec[j] = dec;
    }
    __syncthreads();
    while (f < f1) {
        const int b = static_cast<int>(f / n_seg);
        const int s0 = static_cast<int>(f - static_cast<long long>(b) * n_seg);
        const int s1 = static_cast<int>(min(static_cast<long long>(n_seg), s0 + (f1 - f)));
        const int dec = s_dec[b - b_first];
        if (dec >= 0) {
            const int kstar = dec >> 1;
            const float* rt = a.p_t + (static_cast<size_t>(b) * (g + 1) + kstar) * V;
            const float* rd = (dec & 1) ? a.p_d + (static_cast<size_t>(b) * g + kstar) * V : nullptr;
            segment_sums(rt, rd, V, vec, s0, s1, a.seg + static_cast<size_t>(b) * n_seg);
        }
        __syncthreads();
        if (tid == 0) {                                   // release the block's sums, acquire the others'
            const uint32_t cnt = static_cast<uint32_t>(s1 - s0);
            s_last = atom_add_acq_rel(a.done + b, cnt) + cnt == static_cast<uint32_t>(n_seg);
        }
        __syncthreads();
        if (s_last) {
            finish_request(a, b, dec, s_seg, s_red, s_scan, &s_pick, &s_tloc);
            __syncthreads();                              // shared scratch is reused by the next request
        }
        f += s1 - s0;
    }
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
    const long long total_seg = static_cast<long long>(B) * n_seg;
    // two resident blocks per SM, each streaming at least 2 segments (1024 row entries)
    const int grid = static_cast<int>(std::max(1LL, std::min(2LL * dev.sm_count, (total_seg + 1) / 2)));
    // a block's range of at most ceil(total / grid) segments touches at most this many requests
    const long long per_block = (total_seg + grid - 1) / grid;
    const long long max_req = (per_block + n_seg - 1) / n_seg + 1;
    const size_t smem = sizeof(unsigned long long) * static_cast<size_t>(n_seg) + sizeof(int) * static_cast<size_t>(max_req);
    if (smem > dev.smem_optin) {
        set_error("verify: V=%d needs %zu bytes of shared memory", V, smem);
        return DSPARK_ERR_UNSUPPORTED;
    }
    dspark_status st = clear_workspace(ws, sizeof(WsHeader) + done_bytes(B), stream);
    if (st != DSPARK_OK) return st;
    cudaError_t e = cudaFuncSetAttribute(verify_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    uint8_t* p = static_cast<uint8_t*>(ws) + sizeof(WsHeader);
    a.done = reinterpret_cast<uint32_t*>(p);
    a.seg = reinterpret_cast<unsigned long long*>(p + done_bytes(B));
    a.seed = seed;
    a.offset = offset;
    a.B = B;
    a.gamma = gamma;
    a.V = V;
    a.n_seg = n_seg;
    a.total_seg = total_seg;
    a.grid = grid;
    verify_stream_kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(verify)");
    return DSPARK_OK;
}

}  // namespace dspark
