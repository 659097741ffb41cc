// Lossless verification straight from logits, the draft distribution recomputed where needed.
//
// "Speculative decoding: from zero to DSpark" §2 gives the rule (accept x_k with
// probability min(1, p_t(x_k)/p_d(x_k)), draw the correction from
// norm(max(0, p_t - p_d)) at the first rejection, a bonus token from p_t after a
// fully accepted block).  "DSpark implementation and evaluation" §2.2 / §5: the
// draft distribution of position k is softmax((base_logits[:, k] +
// markov_w2 . markov_w1[prev]) / T_d), which the sampler never writes out; its
// log-sum-exp is the sampler's lse output.  So nothing of size [B, gamma, V]
// exists on the draft side: p_d(x_k) is recomputed at one point per tested
// position, and at the rejected position only at the entries that can still
// win the draw.
//
// Two launches after the workspace clear:
//  1. rounds kernel (persistent, cooperative, one block per SM): round j streams
//     target row j of every request still undecided, as warp items of 2048
//     entries giving (max, sum of 2^((t - max) c)), c = log2(e)/T_t; the warp
//     completing a request's row merges the partials into the row's log2
//     normaliser and runs the acceptance test fl32(u_j p_d(x_j)) < p_t(x_j)
//     (u_j from Philox stream 1, p_d(x_j) from the base logit, one r-long dot
//     product for the bias and the sampler's lse).  A rejection fixes k* = j, an
//     acceptance of position L_b - 1 fixes k* = L_b (bonus), otherwise the
//     request joins the next round; a grid barrier separates the rounds.  Only
//     the rows k <= k* are read (a bonus row needs no normaliser: the draw is
//     invariant to a constant shift).
//  2. draw kernel (warp items of 512 entries of row k*, L2-resident shared
//     lower bound per request): y_v = ln w_v + g_v with w = max(0, p_t - p_d)
//     (rejection) or p_t (bonus), g_v the Gumbel variate of Philox stream 4.
//     Since w_v <= p_t(v) and g_v is increasing in its word, ln p_t(v) plus a
//     table bound of g over the word's top byte bounds y_v; only entries whose
//     bound reaches the best value seen so far are evaluated exactly, and only
//     for those is the draft probability formed (the base logit and one r-long
//     dot product for the bias, computed by the whole warp).  The chunk's
//     largest key goes to the request's slot with one atomicMax, and the warp
//     completing a request's chunks writes its tokens.
//     ln w_v = a_v ln 2 + log1p(-2^(b_v - a_v)) with a_v = log2 p_t(v),
//     b_v = log2 p_d(v), so no cancellation is formed in the linear domain.
// A greedy draft (T_d = 0) has the point mass at its token as distribution: its
// acceptance probability is p_t(x_k) and its residual is p_t without x_{k*}.
#include "device_common.cuh"
#include "host_common.h"

#include <algorithm>

namespace dspark {
namespace {

constexpr int kThreads = 512;                        // rounds kernel
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 2048;                         // rounds warp item: 16 float4 per lane
constexpr int kDrawThreads = 256;                    // draw kernel (one thread per table entry)
constexpr int kDrawWarps = kDrawThreads / 32;
constexpr int kDrawChunk = 512;                      // draw warp item: 4 float4 per lane
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct RowSel {                                      // what the draw of request b needs
    float c_t;                                       // log2(e) / T_t
    float lse2_t;                                    // log2 of the target normaliser of row k*
    float c_d;                                       // log2(e) / T_d (0 for a greedy draft)
    float lse2_d;                                    // sampler lse of position k*, times log2(e)
    int prev;                                        // the token before position k*
    int xk;                                          // draft token at k* (rejections only)
    int pad[2];
};

struct VLArgs {
    const float* t;                                  // [B, g+1, V] target logits
    const float* T_t;                                // [B]
    const float* L;                                  // [B, g, V] draft base logits
    const int32_t* anchor;                           // [B]
    const void* w1;                                  // [V, r]
    const void* w2;                                  // [V, r]
    const float* T_d;                                // [B]
    const float* lse_d;                              // [B, g] sampler lse (natural log)
    const int32_t* tokens;                           // [B, g]
    const int32_t* lengths;                          // [B] or null
    int32_t* out;                                    // [B, g+1]
    int32_t* n_acc;                                  // [B]
    WsHeader* ws;
    // workspace
    unsigned long long* keys;                        // [B] draw keys (zeroed)
    uint32_t* done3;                                 // [B] draw chunks counted (zeroed)
    uint32_t* done;                                  // [B] chunk items counted over all rounds (zeroed)
    uint32_t* rowcnt;                                // [B][g] chunks counted per row (zeroed)
    uint32_t* rejm;                                  // [B] window positions rejected (zeroed)
    uint32_t* badm;                                  // [B] window positions with non-finite inputs (zeroed)
    uint32_t* count;                                 // [rounds + 1] requests entering each round (zeroed)
    int32_t* list;                                   // [2][B] requests of the current / next round
    float* lse2w;                                    // [B][R] log2 normalisers of the window's rows
    int32_t* decision;                               // [B] 2 + decision (see write_decision; zeroed)
    RowSel* sel;                                     // [B]
    float2* part;                                    // [B][R][n_chunk] (max t, sum) of the window's rows
    uint64_t seed;
    uint32_t offset;
    long long timeout_ns;
    int B, g, V, r, wbf16, n_chunk, n_chunk3, warps1, warps3;
    int R;                                           // rows per round (window), <= 32
    long long total3;                                // B * n_chunk3
};

// decision encoding: -1 bad request; else (k* << 2) | (rejected << 0) | (sampled draft << 1)
__device__ __forceinline__ int dec_kstar(int d) { return d >> 2; }
__device__ __forceinline__ bool dec_rejected(int d) { return (d & 1) != 0; }
__device__ __forceinline__ bool dec_sampled(int d) { return (d & 2) != 0; }

__device__ __forceinline__ float warp_sum_f(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
}

__device__ __forceinline__ float warp_max_f(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    return x;
}

// Four consecutive entries at e (a multiple of 4) with `fill` past the end.
__device__ __forceinline__ float4 load4(const float* row, int e, int V, bool vec, float fill) {
    if (vec && e + 4 <= V) return __ldcs(reinterpret_cast<const float4*>(row + e));
    float4 f;
    f.x = e + 0 < V ? __ldcs(row + e + 0) : fill;
    f.y = e + 1 < V ? __ldcs(row + e + 1) : fill;
    f.z = e + 2 < V ? __ldcs(row + e + 2) : fill;
    f.w = e + 3 < V ? __ldcs(row + e + 3) : fill;
    return f;
}

// ---------------------------------------------------------------------------
// 1. target normalisers and the acceptance tests
// ---------------------------------------------------------------------------

// (max, sum 2^((x - max) c)) of one lane's 64 entries of a chunk, merged over the warp.
__device__ __forceinline__ float2 chunk_lse(const float* row, int e0, int V, bool vec, float c) {
    float4 f[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) f[j] = load4(row, e0 + 128 * j, V, vec, -INFINITY);
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j) m = fmaxf(m, fmaxf(fmaxf(f[j].x, f[j].y), fmaxf(f[j].z, f[j].w)));
    const float M = warp_max_f(m);
    float s = 0.f;
    if (M > -INFINITY) {
        const float mc = M * c;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            s += exp2f(fmaf(f[j].x, c, -mc)) + exp2f(fmaf(f[j].y, c, -mc)) + exp2f(fmaf(f[j].z, c, -mc)) +
                 exp2f(fmaf(f[j].w, c, -mc));
        }
    }
    return make_float2(M, warp_sum_f(s));
}

// log2 of the normaliser of window row `slot` of request b from its chunk partials (whole warp).
__device__ float row_lse2(const VLArgs& a, int b, int slot, float c) {
    const float2* p = a.part + (static_cast<size_t>(b) * a.R + slot) * a.n_chunk;
    float m = -INFINITY;
    for (int i = static_cast<int>(lane_id()); i < a.n_chunk; i += 32) m = fmaxf(m, __ldcg(&p[i].x));
    const float M = warp_max_f(m);
    float s = 0.f;
    if (M > -INFINITY)
        for (int i = static_cast<int>(lane_id()); i < a.n_chunk; i += 32) {
            const float2 q = __ldcg(&p[i]);
            s += q.y * exp2f((q.x - M) * c);
        }
    s = warp_sum_f(s);
    return fmaf(M, c, log2f(s));
}

// Sum over j < r of w2[x, j] * w1[prev, j] (whole warp, one 16-byte piece of each row per lane
// per step; rows are whole multiples of 16 bytes and 16-byte aligned).  The butterfly leaves
// the same sum in every lane.
__device__ float point_bias(const VLArgs& a, int x, int prev) {
    float s0 = 0.f, s1 = 0.f;
    if (a.wbf16) {
        const uint4* rx = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.w2) + static_cast<size_t>(x) * a.r);
        const uint4* re = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.w1) + static_cast<size_t>(prev) * a.r);
        for (int p = static_cast<int>(lane_id()); p < a.r / 8; p += 32) {
            const uint4 qx = __ldg(rx + p), qe = __ldg(re + p);
            const __nv_bfloat162* hx = reinterpret_cast<const __nv_bfloat162*>(&qx);
            const __nv_bfloat162* he = reinterpret_cast<const __nv_bfloat162*>(&qe);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 fx = __bfloat1622float2(hx[i]), fe = __bfloat1622float2(he[i]);
                s0 = fmaf(fx.x, fe.x, s0);
                s1 = fmaf(fx.y, fe.y, s1);
            }
        }
    } else {
        const float4* rx = reinterpret_cast<const float4*>(static_cast<const float*>(a.w2) + static_cast<size_t>(x) * a.r);
        const float4* re = reinterpret_cast<const float4*>(static_cast<const float*>(a.w1) + static_cast<size_t>(prev) * a.r);
        for (int p = static_cast<int>(lane_id()); p < a.r / 4; p += 32) {
            const float4 fx = __ldg(rx + p), fe = __ldg(re + p);
            s0 = fmaf(fx.x, fe.x, s0);
            s1 = fmaf(fx.y, fe.y, s1);
            s0 = fmaf(fx.z, fe.z, s0);
            s1 = fmaf(fx.w, fe.w, s1);
        }
    }
    return warp_sum_f(s0 + s1);
}

enum : int { kBadRange = 1, kBadNumeric = 2 };

// Decisions are stored plus 2, so that the cleared value 0 reads as "never decided" (only after
// a grid barrier gave up).
__device__ void write_decision(const VLArgs& a, int b, int dec, const RowSel& sl) {
    if (lane_id() == 0) {
        a.sel[b] = sl;
        a.decision[b] = dec + 2;
    }
}

__device__ __forceinline__ int read_decision(const VLArgs& a, int b) {
    const int d = a.decision[b] - 2;
    if (d == -2) {                                       // undecided: treated as a bad request
        set_status(a.ws, DSPARK_STATUS_INTERNAL);
        return -1;
    }
    return d;
}

__device__ void write_bad(const VLArgs& a, int b, int bad) {
    if (lane_id() == 0) {
        if (bad & kBadNumeric) set_status(a.ws, DSPARK_STATUS_NUMERIC);
        if (bad & kBadRange) flag_input_index(a.ws);
        a.decision[b] = -1 + 2;
    }
}

// Lengths, temperatures and anchor of request b usable (its rows can be streamed).
__device__ __forceinline__ bool request_ok(const VLArgs& a, int b) {
    const int Lb = a.lengths != nullptr ? a.lengths[b] : a.g;
    const float Tt = a.T_t[b], Td = a.T_d[b];
    const int anc = a.anchor[b];
    return Lb >= 0 && Lb <= a.g && Tt > 0.f && Tt < INFINITY && Td >= 0.f && Td < INFINITY && anc >= 0 &&
           anc < a.V;
}

// The warp that completed row k (window slot k - k0) of request b: its normaliser and the
// acceptance test of position k (whole warp).  The previous token is known, so every row of a
// window is tested independently; the first rejection is chosen once the window is complete.
__device__ void decide_row(const VLArgs& a, int b, int k, int k0) {
    const int g = a.g, V = a.V;
    const float Td = a.T_d[b];
    const bool sampled = Td > 0.f;
    const float c_t = kLog2e / a.T_t[b];
    const float lse2 = row_lse2(a, b, k - k0, c_t);
    const uint32_t bit = 1u << (k - k0);
    if (lane_id() == 0) a.lse2w[static_cast<size_t>(b) * a.R + (k - k0)] = lse2;
    if (!(fabsf(lse2) < INFINITY)) {                     // NaN in the row or no finite entry
        if (lane_id() == 0) atomicOr(a.badm + b, bit);
        return;
    }
    const int x = a.tokens[static_cast<size_t>(b) * g + k];
    const int prev = k == 0 ? a.anchor[b] : a.tokens[static_cast<size_t>(b) * g + k - 1];
    if (x < 0 || x >= V || prev < 0 || prev >= V) {     // the request is voided when its window ends
        if (lane_id() == 0) atomicOr(a.badm + b, bit);
        return;
    }
    const float pt = exp2f(fmaf(__ldg(a.t + (static_cast<size_t>(b) * (g + 1) + k) * V + x), c_t, -lse2));
    float pd = 1.f;
    if (sampled) {
        const float lse_d = a.lse_d[static_cast<size_t>(b) * g + k];
        if (!(fabsf(lse_d) < INFINITY)) {
            if (lane_id() == 0) atomicOr(a.badm + b, bit);
            return;
        }
        const float z = __fadd_rn(__ldg(a.L + (static_cast<size_t>(b) * g + k) * V + x), point_bias(a, x, prev));
        pd = exp2f(fmaf(z, kLog2e / Td, -lse_d * kLog2e));
    }
    const uint4 wd = philox_at(a.seed, a.offset, 0u, static_cast<uint32_t>(b), kStreamAccept,
                               static_cast<uint32_t>(k));
    const float u = uniform_from_word(wd.x);
    if (!(__fmul_rn(u, pd) < pt) && lane_id() == 0) atomicOr(a.rejm + b, bit);
}

// The warp that completed request b's window [k0, k0 + R) decides what comes next (whole warp).
__device__ void decide_request(const VLArgs& a, int b, int j, int next_slot_base) {
    const uint32_t lane = lane_id();
    const int g = a.g;
    const int Lb = a.lengths != nullptr ? a.lengths[b] : g;
    const float Td = a.T_d[b];
    const int anc = a.anchor[b];
    const bool sampled = Td > 0.f;
    const int k0 = j * a.R;
    RowSel sl;
    sl.c_t = kLog2e / a.T_t[b];
    sl.c_d = sampled ? kLog2e / Td : 0.f;
    sl.lse2_t = 0.f;
    sl.lse2_d = 0.f;
    sl.prev = anc;
    sl.xk = -1;
    sl.pad[0] = sl.pad[1] = 0;
    if (j == 0) {
        // the first round checks the whole request: lengths, temperatures, anchor, every token
        bool bad = !request_ok(a, b);
        for (int k = static_cast<int>(lane); !bad && k < Lb; k += 32) {
            const int x = a.tokens[static_cast<size_t>(b) * g + k];
            bad = x < 0 || x >= a.V;
        }
        if (__any_sync(0xFFFFFFFFu, bad)) {
            write_bad(a, b, kBadRange);
            return;
        }
        if (Lb == 0) {                                   // nothing to test: a bonus draw from row 0
            write_decision(a, b, (0 << 2) | (sampled ? 2 : 0), sl);
            return;
        }
    }
    const uint32_t rej = __ldcg(a.rejm + b), bad = __ldcg(a.badm + b);
    const uint32_t stop = rej | bad;
    if (stop != 0u) {
        const int p = __ffs(stop) - 1;                   // the first position that ends the block
        if (bad & (1u << p)) {
            write_bad(a, b, kBadNumeric);
            return;
        }
        const int kstar = k0 + p;
        sl.lse2_t = __ldcg(a.lse2w + static_cast<size_t>(b) * a.R + p);
        sl.lse2_d = sampled ? a.lse_d[static_cast<size_t>(b) * g + kstar] * kLog2e : 0.f;
        sl.prev = kstar == 0 ? anc : a.tokens[static_cast<size_t>(b) * g + kstar - 1];
        sl.xk = a.tokens[static_cast<size_t>(b) * g + kstar];
        write_decision(a, b, (kstar << 2) | (sampled ? 2 : 0) | 1, sl);
    } else if (k0 + a.R >= Lb) {                         // all accepted: the bonus row L_b
        write_decision(a, b, (Lb << 2) | (sampled ? 2 : 0), sl);
    } else if (lane == 0) {                              // on to the next window
        const uint32_t slot = atomicAdd(a.count + j + 1, 1u);
        a.list[next_slot_base + static_cast<int>(slot)] = b;
    }
}

__global__ void __launch_bounds__(kThreads, 1) vl_rounds_kernel(VLArgs a) {
    const int gw = static_cast<int>(blockIdx.x) * kWarps + static_cast<int>(warp_id());
    const uint32_t lane = lane_id();
    const bool vec = (a.V & 3) == 0;
    const int per_req = a.R * a.n_chunk;                 // chunk items of one request per round
    const int rounds = (a.g + a.R - 1) / a.R;
    for (int j = 0; j < rounds; ++j) {
        // round j: rows [j R, j R + R) of the requests undecided after round j - 1 (all in round 0)
        const int k0 = j * a.R;
        const int n_active = j == 0 ? a.B : static_cast<int>(__ldcg(a.count + j));
        if (n_active == 0) break;
        const int32_t* list = a.list + (j & 1) * a.B;
        const int next_base = ((j + 1) & 1) * a.B;
        const long long total = static_cast<long long>(n_active) * per_req;
        long long f = total * gw / a.warps1;
        const long long f1 = total * (gw + 1) / a.warps1;
        while (f < f1) {
            const int li = static_cast<int>(f / per_req);
            const int b = j == 0 ? li : __ldcg(list + li);
            const long long req_end = min(static_cast<long long>(li + 1) * per_req, f1);
            if (!own_index_ok(b, a.B, a.ws)) {                      // a work-list entry out of range
                f = req_end;
                continue;
            }
            const uint32_t count = static_cast<uint32_t>(req_end - f);
            const int Lb = a.lengths != nullptr ? a.lengths[b] : a.g;
            const bool ok = j > 0 || (request_ok(a, b) && Lb > 0);
            const float c = kLog2e / a.T_t[b];
            while (f < req_end) {
                // the part of this row that falls in the warp's range
                const int rem = static_cast<int>(f - static_cast<long long>(li) * per_req);
                const int kk = rem / a.n_chunk, k = k0 + kk;
                const long long row_end = min(static_cast<long long>(li) * per_req + (kk + 1) * a.n_chunk, req_end);
                const uint32_t rcount = static_cast<uint32_t>(row_end - f);
                const bool live = ok && k < Lb;
                const float* row = a.t + (static_cast<size_t>(b) * (a.g + 1) + k) * a.V;
                for (; f < row_end; ++f) {
                    if (!live) continue;
                    const int ch = static_cast<int>(f - static_cast<long long>(li) * per_req) - kk * a.n_chunk;
                    const float2 p = chunk_lse(row, ch * kChunk + 4 * static_cast<int>(lane), a.V, vec, c);
                    if (lane == 0) a.part[(static_cast<size_t>(b) * a.R + kk) * a.n_chunk + ch] = p;
                }
                if (live) {
                    uint32_t last = 0;
                    if (lane == 0)                       // release this warp's partials, acquire the others'
                        last = atom_add_acq_rel(a.rowcnt + static_cast<size_t>(b) * a.g + k, rcount) + rcount ==
                                       static_cast<uint32_t>(a.n_chunk) ? 1u : 0u;
                    __syncwarp();
                    if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
                        decide_row(a, b, k, k0);
                    }
                }
            }
            uint32_t last = 0;
            if (lane == 0)
                last = atom_add_acq_rel(a.done + b, count) + count == static_cast<uint32_t>((j + 1) * per_req) ? 1u : 0u;
            __syncwarp();
            if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
                decide_request(a, b, j, next_base);
            }
        }
        if (j + 1 == rounds) break;
        if (!grid_barrier(a.ws, static_cast<uint32_t>(j), a.timeout_ns, 0x5600u + static_cast<uint32_t>(j))) return;
    }
}

// ---------------------------------------------------------------------------
// 3. the Gumbel-max draw of the correction / bonus token
// ---------------------------------------------------------------------------

// Perturbed value ln w_v + g_v of entry v (-inf where w_v = 0), from log2 p_t = a and
// log2 p_d = bb (bb = -inf: no draft mass to subtract).  Never above
// __fadd_rn(__fmul_rn(a, ln 2), g): the log1p term is <= 0 and rounding is monotone.
__device__ __forceinline__ float perturbed(float a, float bb, uint32_t word) {
    float lnw;
    if (bb == -INFINITY) lnw = __fmul_rn(a, kLn2);
    else if (bb >= a) lnw = -INFINITY;
    else lnw = fmaf(a, kLn2, log1pf(-exp2f(bb - a)));
    return __fadd_rn(lnw, gumbel_from_word(word));
}

__device__ __forceinline__ uint32_t word_sel(uint4 w, int j) {
    return j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w;
}

__device__ __forceinline__ float key_value(unsigned long long key) {
    return key == 0ull ? -INFINITY : float_from_order_bits(static_cast<uint32_t>(key >> 32));
}

// Sum over j < r of w2[v, j] * w1[prev, j] by one lane (16-byte pieces; rows are whole
// multiples of 16 bytes and 16-byte aligned).
__device__ __forceinline__ float lane_bias(const VLArgs& a, int v, int prev) {
    float s0 = 0.f, s1 = 0.f;
    if (a.wbf16) {
        const uint4* x = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.w2) + static_cast<size_t>(v) * a.r);
        const uint4* e = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.w1) + static_cast<size_t>(prev) * a.r);
#pragma unroll 4
        for (int p = 0; p < a.r / 8; ++p) {
            const uint4 qx = __ldg(x + p), qe = __ldg(e + p);
            const __nv_bfloat162* hx = reinterpret_cast<const __nv_bfloat162*>(&qx);
            const __nv_bfloat162* he = reinterpret_cast<const __nv_bfloat162*>(&qe);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 fx = __bfloat1622float2(hx[i]), fe = __bfloat1622float2(he[i]);
                s0 = fmaf(fx.x, fe.x, s0);
                s1 = fmaf(fx.y, fe.y, s1);
            }
        }
    } else {
        const float4* x = reinterpret_cast<const float4*>(static_cast<const float*>(a.w2) + static_cast<size_t>(v) * a.r);
        const float4* e = reinterpret_cast<const float4*>(static_cast<const float*>(a.w1) + static_cast<size_t>(prev) * a.r);
#pragma unroll 4
        for (int p = 0; p < a.r / 4; ++p) {
            const float4 fx = __ldg(x + p), fe = __ldg(e + p);
            s0 = fmaf(fx.x, fe.x, s0);
            s1 = fmaf(fx.y, fe.y, s1);
            s0 = fmaf(fx.z, fe.z, s0);
            s1 = fmaf(fx.w, fe.w, s1);
        }
    }
    return s0 + s1;
}

// The draft's log2 probability at entry v of row k* (one lane).
__device__ __forceinline__ float draft_log2p(const VLArgs& a, int b, int dec, const RowSel& s, int v) {
    if (!dec_rejected(dec)) return -INFINITY;
    if (!dec_sampled(dec)) return v == s.xk ? 0.f : -INFINITY;
    const int kstar = dec_kstar(dec);
    const float l = __ldg(a.L + (static_cast<size_t>(b) * a.g + kstar) * a.V + v);
    return fmaf(__fadd_rn(l, lane_bias(a, v, s.prev)), s.c_d, -s.lse2_d);
}

// The draft's log2 probability at entry v of row k* (whole warp; v uniform).
__device__ __forceinline__ float draft_log2p_warp(const VLArgs& a, int b, int dec, const RowSel& s, int v) {
    if (!dec_rejected(dec)) return -INFINITY;
    if (!dec_sampled(dec)) return v == s.xk ? 0.f : -INFINITY;
    const int kstar = dec_kstar(dec);
    const float l = __ldg(a.L + (static_cast<size_t>(b) * a.g + kstar) * a.V + v);
    return fmaf(__fadd_rn(l, point_bias(a, v, s.prev)), s.c_d, -s.lse2_d);
}

// Bound of the Gumbel variate of `word`: by its top byte, and for top byte 255 (where the
// variate ranges up to its maximum) by its second byte.
__device__ __forceinline__ float gumbel_bound(const float* gtab, uint32_t word) {
    const uint32_t hi = word >> 24;
    return hi != 255u ? gtab[hi] : gtab[256 + ((word >> 16) & 255u)];
}

__device__ __forceinline__ float comp(const float4& f, int i) { return i == 0 ? f.x : i == 1 ? f.y : i == 2 ? f.z : f.w; }

// Entry q (= 4 j + i) of a lane's 16 loaded target logits, q not a compile-time constant.
__device__ __forceinline__ float entry_of(const float4 (&tv)[4], int q) {
    float x = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k)
        if (k == q) x = comp(tv[k >> 2], k & 3);
    return x;
}

__device__ __forceinline__ uint32_t residual_word(const VLArgs& a, int b, int kstar, int v) {
    return word_sel(philox_at(a.seed, a.offset, static_cast<uint32_t>(v >> 2), static_cast<uint32_t>(b),
                              kStreamResidual, static_cast<uint32_t>(kstar)),
                    v & 3);
}

// One 512-entry chunk of row k* whose target logits tv the lane holds (lane l: entries
// e0 + 128 j + 0..3, j < 4).  best / LB are warp-uniform: the largest key found so far and its
// value, which every exact value must reach to matter.
__device__ __forceinline__ void chunk_draw(const VLArgs& a, int b, int dec, const RowSel& s, int e0,
                                           const float4 (&tv)[4], const float* gtab, unsigned long long& best,
                                           float& LB, bool& nan_seen) {
    const int V = a.V;
    const int kstar = dec_kstar(dec);
    float bnd[16];
    uint32_t cand = 0;                                   // bit 4 j + i: entry e0 + 128 j + i may win
    int pick = -1;                                       // the lane's candidate of largest bound
    float pb = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float av[4];
        float hi = -INFINITY;
        bool odd = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            av[i] = fmaf(comp(tv[j], i), s.c_t, -s.lse2_t);
            hi = fmaxf(hi, av[i]);
            odd |= av[i] != av[i];
            bnd[4 * j + i] = -INFINITY;
        }
        const int e = e0 + 128 * j;
        // no word can lift this group to LB: skip its Philox call (NaN entries are kept)
        if (e >= V || (!odd && __fadd_rn(__fmul_rn(hi, kLn2), kGumbelMax) < LB)) continue;
        const uint4 w = philox_at(a.seed, a.offset, static_cast<uint32_t>(e >> 2), static_cast<uint32_t>(b),
                                  kStreamResidual, static_cast<uint32_t>(kstar));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float bound = __fadd_rn(__fmul_rn(av[i], kLn2), gumbel_bound(gtab, word_sel(w, i)));
            bnd[4 * j + i] = bound;
            if (e + i < V && !(bound < LB)) {
                cand |= 1u << (4 * j + i);
                if (pick < 0 || bound > pb) {
                    pick = 4 * j + i;
                    pb = bound;
                }
            }
        }
    }
    if (LB == -INFINITY) {
        // nothing known yet: every lane evaluates its candidate of largest bound, at once
        unsigned long long mine = 0;
        if (pick >= 0) {
            cand &= ~(1u << pick);
            const int v = e0 + 128 * (pick >> 2) + (pick & 3);
            const float y = perturbed(fmaf(entry_of(tv, pick), s.c_t, -s.lse2_t), draft_log2p(a, b, dec, s, v),
                                      residual_word(a, b, kstar, v));
            if (y != y) nan_seen = true;
            else if (y > -INFINITY) mine = argmax_key(y, static_cast<uint32_t>(v));
        }
        mine = warp_max_u64(mine);
        if (mine > best) {
            best = mine;
            LB = key_value(best);
        }
    }
    // drop what LB now excludes, then the rest one at a time across the warp
#pragma unroll
    for (int q = 0; q < 16; ++q)
        if (bnd[q] < LB) cand &= ~(1u << q);
    uint32_t m = __ballot_sync(0xFFFFFFFFu, cand != 0u);
    while (m != 0u) {
        const int src = __ffs(m) - 1;
        const int bit = __ffs(__shfl_sync(0xFFFFFFFFu, cand, src)) - 1;
        const float tc = __shfl_sync(0xFFFFFFFFu, entry_of(tv, bit), src);
        const int v = e0 - 4 * static_cast<int>(lane_id()) + 4 * src + 128 * (bit >> 2) + (bit & 3);
        const float y = perturbed(fmaf(tc, s.c_t, -s.lse2_t), draft_log2p_warp(a, b, dec, s, v),
                                  residual_word(a, b, kstar, v));
        if (static_cast<int>(lane_id()) == src) cand &= cand - 1u;
        if (y != y) {
            nan_seen = true;
        } else if (y > -INFINITY) {
            const unsigned long long key = argmax_key(y, static_cast<uint32_t>(v));
            if (key > best) {
                best = key;
                LB = y;
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    if (bnd[q] < LB) cand &= ~(1u << q);
            }
        }
        m = __ballot_sync(0xFFFFFFFFu, cand != 0u);
    }
}

// Fallback of a residual without positive mass (float32 rounding only): the bonus form over row
// k*, one warp over the whole row.
__device__ unsigned long long row_draw_bonus(const VLArgs& a, int b, int dec, const RowSel& s) {
    const int V = a.V, kstar = dec_kstar(dec);
    const float* rt = a.t + (static_cast<size_t>(b) * (a.g + 1) + kstar) * V;
    unsigned long long best = 0;
    for (int v = static_cast<int>(lane_id()); v < V; v += 32) {
        const uint4 w = philox_at(a.seed, a.offset, static_cast<uint32_t>(v >> 2), static_cast<uint32_t>(b),
                                  kStreamResidual, static_cast<uint32_t>(kstar));
        const float y = perturbed(fmaf(rt[v], s.c_t, -s.lse2_t), -INFINITY, word_sel(w, v & 3));
        if (y == y && y > -INFINITY) {
            const unsigned long long key = argmax_key(y, static_cast<uint32_t>(v));
            best = key > best ? key : best;
        }
    }
    return warp_max_u64(best);
}

__device__ void finish(const VLArgs& a, int b, int dec) {
    const uint32_t lane = lane_id();
    const int g = a.g;
    int32_t* out = a.out + static_cast<size_t>(b) * (g + 1);
    if (dec < 0) {
        for (int k = static_cast<int>(lane); k <= g; k += 32) out[k] = -1;
        if (lane == 0) a.n_acc[b] = 0;
        return;
    }
    const int kstar = dec_kstar(dec);
    unsigned long long key = __ldcg(a.keys + b);
    if (key == 0ull && dec_rejected(dec)) key = row_draw_bonus(a, b, dec, a.sel[b]);
    int y = 0;
    if (key == 0ull) {
        if (lane == 0) set_status(a.ws, DSPARK_STATUS_NUMERIC);      // no entry with positive mass
    } else {
        y = static_cast<int>(key_index(key));
    }
    for (int k = static_cast<int>(lane); k <= g; k += 32) {
        int v = -1;
        if (k < kstar) v = a.tokens[static_cast<size_t>(b) * g + k];
        else if (k == kstar) v = y;
        out[k] = v;
    }
    if (lane == 0) a.n_acc[b] = kstar;
}

__global__ void __launch_bounds__(kDrawThreads, 2) vl_draw_kernel(VLArgs a) {
    __shared__ float gtab[512];
    {
        // bound of the Gumbel variate over the words with top byte k (entry k) and over those with
        // top bytes 255, k (entry 256 + k): the value at the largest such word, plus a margin for
        // the rounding of the two logarithms (the variate increases with the word)
        const uint32_t k = threadIdx.x;                  // blockDim.x == 256
        gtab[k] = __fadd_rn(gumbel_from_word(((k + 1u) << 24) - 1u), 1e-3f);
        gtab[256 + k] = __fadd_rn(gumbel_from_word(((0xFF00u + k + 1u) << 16) - 1u), 1e-3f);
    }
    __syncthreads();
    const int gw = static_cast<int>(blockIdx.x) * kDrawWarps + static_cast<int>(warp_id());
    const uint32_t lane = lane_id();
    const bool vec = (a.V & 3) == 0;
    long long f = a.total3 * gw / a.warps3;
    const long long f1 = a.total3 * (gw + 1) / a.warps3;
    bool nan_seen = false;
    while (f < f1) {
        const int b = static_cast<int>(f / a.n_chunk3);
        const long long req_end = min(static_cast<long long>(b + 1) * a.n_chunk3, f1);
        const uint32_t count = static_cast<uint32_t>(req_end - f);
        const int dec = read_decision(a, b);
        if (dec >= 0) {
            const RowSel s = a.sel[b];
            const float* rt = a.t + (static_cast<size_t>(b) * (a.g + 1) + dec_kstar(dec)) * a.V;
            unsigned long long best = 0, published = 0;
            float4 cur[4], nxt[4];
            int e0 = static_cast<int>(f - static_cast<long long>(b) * a.n_chunk3) * kDrawChunk + 4 * static_cast<int>(lane);
#pragma unroll
            for (int j = 0; j < 4; ++j) cur[j] = load4(rt, e0 + 128 * j, a.V, vec, -INFINITY);
            for (; f < req_end; ++f) {
                // the next chunk's loads are in flight while this one is processed
                const bool more = f + 1 < req_end;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    nxt[j] = more ? load4(rt, e0 + kDrawChunk + 128 * j, a.V, vec, -INFINITY) : cur[j];
                // the request's best so far (any warp's) bounds what can still win
                const unsigned long long shared_best = __ldcg(a.keys + b);
                if (shared_best > best) best = shared_best;
                float LB = key_value(best);
                chunk_draw(a, b, dec, s, e0, cur, gtab, best, LB, nan_seen);
                if (best > published && best > shared_best) {
                    if (lane == 0) atomicMax(a.keys + b, best);
                    published = best;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) cur[j] = nxt[j];
                e0 += kDrawChunk;
            }
        }
        f = req_end;
        uint32_t last = 0;
        if (lane == 0)
            last = atom_add_acq_rel(a.done3 + b, count) + count == static_cast<uint32_t>(a.n_chunk3) ? 1u : 0u;
        __syncwarp();
        if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
            finish(a, b, dec);
        }
    }
    if (__any_sync(0xFFFFFFFFu, nan_seen) && lane == 0) set_status(a.ws, DSPARK_STATUS_NUMERIC);
}

size_t al(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct VLLayout {
    size_t keys, done3, done, rowcnt, rejm, badm, count, decision, clear_end, sel, list, lse2w, part, total;
};

// Rows per round: all drafted rows at once while they are few (their bytes cost less than the
// extra rounds would), else one row per round so that only rows k <= k* are streamed.
int rows_per_round(int B, int gamma, int V) {
    const double all_rows = 4.0 * B * static_cast<double>(gamma) * V;
    return all_rows <= 64.0 * (1 << 20) ? std::min(gamma, 32) : 1;
}

VLLayout vl_layout(int B, int gamma, int V) {
    const size_t n_chunk = (static_cast<size_t>(V) + kChunk - 1) / kChunk;
    const int R = rows_per_round(B, gamma, V);
    const int rounds = (gamma + R - 1) / R;
    VLLayout l;
    size_t p = sizeof(WsHeader);
    l.keys = p;
    p = al(p + sizeof(unsigned long long) * B);
    l.done3 = p;
    p = al(p + sizeof(uint32_t) * B);
    l.done = p;
    p = al(p + sizeof(uint32_t) * B);
    l.rowcnt = p;
    p = al(p + sizeof(uint32_t) * static_cast<size_t>(B) * gamma);
    l.rejm = p;
    p = al(p + sizeof(uint32_t) * B);
    l.badm = p;
    p = al(p + sizeof(uint32_t) * B);
    l.count = p;
    p = al(p + sizeof(uint32_t) * (static_cast<size_t>(rounds) + 1));
    l.decision = p;
    p = al(p + sizeof(int32_t) * B);
    l.clear_end = p;
    l.sel = p;
    p = al(p + sizeof(RowSel) * B);
    l.list = p;
    p = al(p + sizeof(int32_t) * 2 * static_cast<size_t>(B));
    l.lse2w = p;
    p = al(p + sizeof(float) * static_cast<size_t>(B) * R);
    l.part = p;
    p = al(p + sizeof(float2) * static_cast<size_t>(B) * R * n_chunk);
    l.total = p;
    return l;
}

}  // namespace

size_t verify_logits_workspace_bytes(int B, int gamma, int V, int r) {
    if (B < 1 || gamma < 1 || V < 1 || r < 1) return 0;
    (void)r;
    return vl_layout(B, gamma, V).total;
}

dspark_status launch_verify_logits(const float* target_logits, const float* T_t, const float* base_logits,
                                   const int32_t* anchor, const void* w1, const void* w2, dspark_dtype wdtype,
                                   const float* T_d, const float* draft_lse, const int32_t* draft_tokens,
                                   const int32_t* lengths, uint64_t seed, uint32_t offset, int B, int gamma,
                                   int V, int r, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                                   cudaStream_t stream, const DeviceInfo& dev) {
    const VLLayout l = vl_layout(B, gamma, V);
    dspark_status st = clear_workspace(ws, l.clear_end, stream);
    if (st != DSPARK_OK) return st;
    uint8_t* base = static_cast<uint8_t*>(ws);
    VLArgs a;
    a.t = target_logits;
    a.T_t = T_t;
    a.L = base_logits;
    a.anchor = anchor;
    a.w1 = w1;
    a.w2 = w2;
    a.T_d = T_d;
    a.lse_d = draft_lse;
    a.tokens = draft_tokens;
    a.lengths = lengths;
    a.out = out_tokens;
    a.n_acc = num_accepted;
    a.ws = static_cast<WsHeader*>(ws);
    a.keys = reinterpret_cast<unsigned long long*>(base + l.keys);
    a.done3 = reinterpret_cast<uint32_t*>(base + l.done3);
    a.decision = reinterpret_cast<int32_t*>(base + l.decision);
    a.sel = reinterpret_cast<RowSel*>(base + l.sel);
    a.done = reinterpret_cast<uint32_t*>(base + l.done);
    a.rowcnt = reinterpret_cast<uint32_t*>(base + l.rowcnt);
    a.rejm = reinterpret_cast<uint32_t*>(base + l.rejm);
    a.badm = reinterpret_cast<uint32_t*>(base + l.badm);
    a.count = reinterpret_cast<uint32_t*>(base + l.count);
    a.list = reinterpret_cast<int32_t*>(base + l.list);
    a.lse2w = reinterpret_cast<float*>(base + l.lse2w);
    a.part = reinterpret_cast<float2*>(base + l.part);
    a.seed = seed;
    a.offset = offset;
    a.timeout_ns = kDefaultTimeoutNs;
    a.B = B;
    a.g = gamma;
    a.V = V;
    a.r = r;
    a.wbf16 = wdtype == DSPARK_BF16 ? 1 : 0;
    a.n_chunk = (V + kChunk - 1) / kChunk;
    a.R = rows_per_round(B, gamma, V);
    a.n_chunk3 = (V + kDrawChunk - 1) / kDrawChunk;
    a.total3 = static_cast<long long>(B) * a.n_chunk3;
    // rounds: one co-resident 512-thread block per SM at most; draw: up to two 256-thread
    // blocks per SM, each warp at least one 512-entry chunk
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vl_rounds_kernel, kThreads, 0);
    if (e != cudaSuccess) return cuda_error(e, "occupancy(verify_logits rounds)");
    if (per_sm < 1) {
        set_error("verify_logits: the rounds kernel does not fit on an SM");
        return DSPARK_ERR_UNSUPPORTED;
    }
    const long long want1 = (static_cast<long long>(B) * a.R * a.n_chunk + kWarps - 1) / kWarps;
    const int blocks1 = static_cast<int>(std::max(1LL, std::min(static_cast<long long>(dev.sm_count), want1)));
    const int blocks3 = static_cast<int>(std::max(1LL, std::min(2LL * dev.sm_count,
                                                                 (a.total3 + kDrawWarps - 1) / kDrawWarps)));
    a.warps1 = blocks1 * kWarps;
    a.warps3 = blocks3 * kDrawWarps;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks1));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;          // the rounds meet at grid barriers
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, vl_rounds_kernel, a);
    if (e != cudaSuccess) return cuda_error(e, "launch(verify_logits rounds)");
    vl_draw_kernel<<<blocks3, kDrawThreads, 0, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(verify_logits draw)");
    return DSPARK_OK;
}

}  // namespace dspark
