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
// position, and the full draft row only at the rejected position.
//
// Three launches after the workspace clear:
//  1. lse kernel (one block per SM, warp items of 2048 entries): per-chunk
//     (max, sum of 2^((t - max) c)) of the target rows k <= L_b, c = log2(e)/T_t.
//     The warp completing a request's items decides it: it merges the chunk
//     partials into log2-normalisers row by row and runs the acceptance tests
//     fl32(u_k p_d(x_k)) < p_t(x_k) in order (u_k from Philox stream 1, p_d(x_k)
//     from the base logit, one r-long dot product for the bias and the sampler's
//     lse), stopping at the first rejection k*.  It writes the decision, the
//     normalisers of row k* and, for a rejection by a sampled draft, the row
//     markov_w1[prev_{k*}] for step 2.
//  2. the tcgen05 GEMM of the draft logits (same kernel) computes the bias rows
//     markov_w2 . markov_w1[prev_{k*}] of every request, [B, V] fp32.
//  3. draw kernel (one block per SM, warp items of 2048 entries of row k*):
//     y_v = ln w_v + g_v with w = max(0, p_t - p_d) (rejection) or p_t (bonus),
//     g_v the Gumbel variate of Philox stream 4; the chunk's largest key goes to
//     the request's slot with one atomicMax, and the warp completing a request's
//     chunks writes its tokens.  ln w_v = a_v ln 2 + log1p(-2^(b_v - a_v)) with
//     a_v = log2 p_t(v), b_v = log2 p_d(v), so no cancellation is formed in the
//     linear domain.
// A greedy draft (T_d = 0) has the point mass at its token as distribution: its
// acceptance probability is p_t(x_k) and its residual is p_t without x_{k*}.
#include "device_common.cuh"
#include "host_common.h"

#include <algorithm>

namespace dspark {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 2048;                         // entries per warp item: 16 float4 per lane
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct RowSel {                                      // what the draw of request b needs
    float c_t;                                       // log2(e) / T_t
    float lse2_t;                                    // log2 of the target normaliser of row k*
    float c_d;                                       // log2(e) / T_d (0 for a greedy draft)
    float lse2_d;                                    // sampler lse of position k*, times log2(e)
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
    uint32_t* done1;                                 // [B] lse items counted (zeroed)
    uint32_t* done3;                                 // [B] draw chunks counted (zeroed)
    int32_t* decision;                               // [B] see dec_kstar / dec_rejected / dec_sampled
    RowSel* sel;                                     // [B]
    float2* part;                                    // [B][g+1][n_chunk] (max t, sum)
    void* eg;                                        // [B, r] gathered markov_w1 rows (GEMM operand)
    const float* bias;                               // [B, V] bias rows (GEMM output)
    uint64_t seed;
    uint32_t offset;
    int B, g, V, r, wbf16, n_chunk, warps1, warps3;
    long long total1;                                // B * (g+1) * n_chunk
    long long total3;                                // B * n_chunk
};

// decision encoding: -1 bad request; else (k* << 2) | (rejected << 0) | (sampled draft << 1)
__device__ __forceinline__ int dec_kstar(int d) { return d >> 2; }
__device__ __forceinline__ bool dec_rejected(int d) { return (d & 1) != 0; }
__device__ __forceinline__ bool dec_sampled(int d) { return (d & 2) != 0; }

__device__ __forceinline__ float wval(const void* w, bool bf16, size_t i) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(w)[i]) : static_cast<const float*>(w)[i];
}

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

// log2 of the normaliser of target row k of request b from its chunk partials (whole warp).
__device__ float row_lse2(const VLArgs& a, int b, int k, float c) {
    const float2* p = a.part + (static_cast<size_t>(b) * (a.g + 1) + k) * a.n_chunk;
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

// Sum over j < r of w2[x, j] * w1[prev, j] (whole warp).
__device__ float point_bias(const VLArgs& a, int x, int prev) {
    const bool bf = a.wbf16 != 0;
    const size_t rx = static_cast<size_t>(x) * a.r, rp = static_cast<size_t>(prev) * a.r;
    float s = 0.f;
    for (int j = static_cast<int>(lane_id()); j < a.r; j += 32) s = fmaf(wval(a.w2, bf, rx + j), wval(a.w1, bf, rp + j), s);
    return warp_sum_f(s);
}

// The warp that completed request b's normaliser items decides the request.
__device__ void decide(const VLArgs& a, int b) {
    const uint32_t lane = lane_id();
    const int g = a.g, V = a.V;
    const int Lb = a.lengths != nullptr ? a.lengths[b] : g;
    const float Tt = a.T_t[b], Td = a.T_d[b];
    const int anc = a.anchor[b];
    bool bad = !(Lb >= 0 && Lb <= g) || !(Tt > 0.f && Tt < INFINITY) || !(Td >= 0.f && Td < INFINITY) ||
               anc < 0 || anc >= V;
    const bool sampled = Td > 0.f;
    const float c_t = kLog2e / Tt;
    const float c_d = sampled ? kLog2e / Td : 0.f;
    int kstar = Lb, prev_star = anc;
    bool rejected = false, numeric = false;
    float lse2_star = 0.f, lsed2_star = 0.f;
    int prev = anc;
    for (int k = 0; !bad && k <= Lb; ++k) {
        const float lse2 = row_lse2(a, b, k, c_t);
        if (!(fabsf(lse2) < INFINITY)) {                 // NaN in the row or no finite entry
            numeric = bad = true;
            break;
        }
        if (k == Lb) {                                  // every tested token accepted: bonus row
            lse2_star = lse2;
            break;
        }
        const int x = a.tokens[static_cast<size_t>(b) * g + k];
        if (x < 0 || x >= V) {
            bad = true;
            break;
        }
        const float pt = exp2f(fmaf(__ldg(a.t + (static_cast<size_t>(b) * (g + 1) + k) * V + x), c_t, -lse2));
        float pd = 1.f;
        float lsed2 = 0.f;
        if (sampled) {
            const float lse_d = a.lse_d[static_cast<size_t>(b) * g + k];
            if (!(fabsf(lse_d) < INFINITY)) {
                numeric = bad = true;
                break;
            }
            lsed2 = lse_d * kLog2e;
            const float z = __fadd_rn(__ldg(a.L + (static_cast<size_t>(b) * g + k) * V + x), point_bias(a, x, prev));
            pd = exp2f(fmaf(z, c_d, -lsed2));
        }
        const uint4 w = philox_at(a.seed, a.offset, 0u, static_cast<uint32_t>(b), kStreamAccept,
                                  static_cast<uint32_t>(k));
        const float u = uniform_from_word(w.x);
        if (!(__fmul_rn(u, pd) < pt)) {
            kstar = k;
            rejected = true;
            prev_star = prev;
            lse2_star = lse2;
            lsed2_star = lsed2;
            break;
        }
        prev = x;
    }
    // the GEMM operand row: markov_w1[prev_{k*}] for a rejection by a sampled draft, else zeros
    const bool gather = !bad && rejected && sampled;
    const size_t esz = a.wbf16 ? 2 : 4;
    const size_t row_bytes = esz * static_cast<size_t>(a.r);
    uint8_t* dst = static_cast<uint8_t*>(a.eg) + row_bytes * static_cast<size_t>(b);
    if (gather) {                                        // prev_star is a checked token id here
        const uint8_t* src = static_cast<const uint8_t*>(a.w1) + row_bytes * static_cast<size_t>(prev_star);
        for (size_t i = 4 * lane; i < row_bytes; i += 128)    // rows are whole multiples of 16 bytes
            *reinterpret_cast<uint32_t*>(dst + i) = *reinterpret_cast<const uint32_t*>(src + i);
    } else {
        for (size_t i = 4 * lane; i < row_bytes; i += 128) *reinterpret_cast<uint32_t*>(dst + i) = 0u;
    }
    if (lane == 0) {
        if (bad) set_status(a.ws, numeric ? DSPARK_STATUS_NUMERIC : DSPARK_STATUS_INPUT_RANGE);
        RowSel s;
        s.c_t = c_t;
        s.lse2_t = lse2_star;
        s.c_d = c_d;
        s.lse2_d = lsed2_star;
        a.sel[b] = s;
        a.decision[b] = bad ? -1 : ((kstar << 2) | (sampled ? 2 : 0) | (rejected ? 1 : 0));
    }
}

__global__ void __launch_bounds__(kThreads, 1) vl_lse_kernel(VLArgs a) {
    const int gw = static_cast<int>(blockIdx.x) * kWarps + static_cast<int>(warp_id());
    const uint32_t lane = lane_id();
    const long long per_req = static_cast<long long>(a.g + 1) * a.n_chunk;
    const bool vec = (a.V & 3) == 0;
    long long f = a.total1 * gw / a.warps1;
    const long long f1 = a.total1 * (gw + 1) / a.warps1;
    while (f < f1) {
        const int b = static_cast<int>(f / per_req);
        const long long req_end = min(static_cast<long long>(b + 1) * per_req, f1);
        const uint32_t count = static_cast<uint32_t>(req_end - f);
        const int Lb = a.lengths != nullptr ? a.lengths[b] : a.g;
        const float Tt = a.T_t[b];
        const bool ok = Lb >= 0 && Lb <= a.g && Tt > 0.f && Tt < INFINITY;
        const float c = kLog2e / Tt;
        for (; f < req_end; ++f) {
            const long long rem = f - static_cast<long long>(b) * per_req;
            const int k = static_cast<int>(rem / a.n_chunk), ch = static_cast<int>(rem % a.n_chunk);
            if (!ok || k > Lb) continue;                     // rows past L_b are not needed
            const float* row = a.t + (static_cast<size_t>(b) * (a.g + 1) + k) * a.V;
            const float2 p = chunk_lse(row, ch * kChunk + 4 * static_cast<int>(lane), a.V, vec, c);
            if (lane == 0) a.part[(static_cast<size_t>(b) * (a.g + 1) + k) * a.n_chunk + ch] = p;
        }
        uint32_t last = 0;
        if (lane == 0) {
            __threadfence();
            last = atomicAdd(a.done1 + b, count) + count == static_cast<uint32_t>(per_req) ? 1u : 0u;
        }
        if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
            __threadfence();
            decide(a, b);
        }
    }
}

// ---------------------------------------------------------------------------
// 3. the Gumbel-max draw of the correction / bonus token
// ---------------------------------------------------------------------------

// Perturbed value ln w_v + g_v of entry v (-inf where w_v = 0), from log2 p_t = a and
// log2 p_d = bb (bb = -inf: no draft mass to subtract).
__device__ __forceinline__ float perturbed(float a, float bb, uint32_t word) {
    float lnw;
    if (bb == -INFINITY) lnw = a * kLn2;
    else if (bb >= a) lnw = -INFINITY;
    else lnw = fmaf(a, kLn2, log1pf(-exp2f(bb - a)));
    return lnw + gumbel_from_word(word);
}

__device__ __forceinline__ uint32_t word_sel(uint4 w, int j) {
    return j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w;
}

// Largest key of the chunk starting at lane entry e0 (lane l: e0 + 128 q + 0..3, q < 16).
__device__ __forceinline__ unsigned long long chunk_draw(const VLArgs& a, int b, int dec, const RowSel& s,
                                                         int e0, bool vec, bool& nan_seen) {
    const int V = a.V, g = a.g;
    const int kstar = dec_kstar(dec);
    const bool rej = dec_rejected(dec), smp = dec_sampled(dec);
    const float* rt = a.t + (static_cast<size_t>(b) * (g + 1) + kstar) * V;
    const float* rl = a.L + (static_cast<size_t>(b) * g + kstar) * V;
    const float* rb = a.bias + static_cast<size_t>(b) * V;
    const int xk = rej && !smp ? a.tokens[static_cast<size_t>(b) * g + kstar] : -1;
    unsigned long long best = 0;
#pragma unroll 1
    for (int q0 = 0; q0 < 16; q0 += 4) {
        float4 tv[4], lv[4], bv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) tv[j] = load4(rt, e0 + 128 * (q0 + j), V, vec, -INFINITY);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            lv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            bv[j] = lv[j];
        }
        if (rej && smp) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lv[j] = load4(rl, e0 + 128 * (q0 + j), V, vec, 0.f);
                bv[j] = load4(rb, e0 + 128 * (q0 + j), V, vec, 0.f);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + 128 * (q0 + j);
            if (e >= V) continue;
            const uint4 w = philox_at(a.seed, a.offset, static_cast<uint32_t>(e >> 2), static_cast<uint32_t>(b),
                                      kStreamResidual, static_cast<uint32_t>(kstar));
            const float tt[4] = {tv[j].x, tv[j].y, tv[j].z, tv[j].w};
            const float ll[4] = {lv[j].x, lv[j].y, lv[j].z, lv[j].w};
            const float bb4[4] = {bv[j].x, bv[j].y, bv[j].z, bv[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int v = e + i;
                if (v >= V) break;
                const float av = fmaf(tt[i], s.c_t, -s.lse2_t);
                float bb = -INFINITY;
                if (rej) {
                    if (smp) bb = fmaf(__fadd_rn(ll[i], bb4[i]), s.c_d, -s.lse2_d);
                    else bb = v == xk ? 0.f : -INFINITY;
                }
                const float y = perturbed(av, bb, word_sel(w, i));
                if (y != y) {
                    nan_seen = true;
                    continue;
                }
                if (y == -INFINITY) continue;
                const unsigned long long key = argmax_key(y, static_cast<uint32_t>(v));
                best = key > best ? key : best;
            }
        }
    }
    return best;
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

__global__ void __launch_bounds__(kThreads, 1) vl_draw_kernel(VLArgs a) {
    const int gw = static_cast<int>(blockIdx.x) * kWarps + static_cast<int>(warp_id());
    const uint32_t lane = lane_id();
    const bool vec = (a.V & 3) == 0;
    long long f = a.total3 * gw / a.warps3;
    const long long f1 = a.total3 * (gw + 1) / a.warps3;
    bool nan_seen = false;
    while (f < f1) {
        const int b = static_cast<int>(f / a.n_chunk);
        const long long req_end = min(static_cast<long long>(b + 1) * a.n_chunk, f1);
        const uint32_t count = static_cast<uint32_t>(req_end - f);
        const int dec = a.decision[b];
        if (dec >= 0) {
            const RowSel s = a.sel[b];
            unsigned long long best = 0;
            for (; f < req_end; ++f) {
                const int ch = static_cast<int>(f - static_cast<long long>(b) * a.n_chunk);
                const unsigned long long k =
                    chunk_draw(a, b, dec, s, ch * kChunk + 4 * static_cast<int>(lane), vec, nan_seen);
                best = k > best ? k : best;
            }
            best = warp_max_u64(best);
            if (lane == 0 && best != 0ull) atomicMax(a.keys + b, best);
        }
        f = req_end;
        uint32_t last = 0;
        if (lane == 0) {
            __threadfence();
            last = atomicAdd(a.done3 + b, count) + count == static_cast<uint32_t>(a.n_chunk) ? 1u : 0u;
        }
        if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
            __threadfence();
            finish(a, b, dec);
        }
    }
    if (__any_sync(0xFFFFFFFFu, nan_seen) && lane == 0) set_status(a.ws, DSPARK_STATUS_NUMERIC);
}

size_t al(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct VLLayout {
    size_t keys, done1, done3, clear_end, decision, sel, part, eg, bias, total;
};

VLLayout vl_layout(int B, int gamma, int V, int r) {
    const size_t n_chunk = (static_cast<size_t>(V) + kChunk - 1) / kChunk;
    VLLayout l;
    size_t p = sizeof(WsHeader);
    l.keys = p;
    p = al(p + sizeof(unsigned long long) * B);
    l.done1 = p;
    p = al(p + sizeof(uint32_t) * B);
    l.done3 = p;
    p = al(p + sizeof(uint32_t) * B);
    l.clear_end = p;
    l.decision = p;
    p = al(p + sizeof(int32_t) * B);
    l.sel = p;
    p = al(p + sizeof(RowSel) * B);
    l.part = p;
    p = al(p + sizeof(float2) * static_cast<size_t>(B) * (gamma + 1) * n_chunk);
    l.eg = p;
    p = al(p + sizeof(float) * static_cast<size_t>(B) * r);          // sized for fp32 weights
    l.bias = p;
    p = al(p + sizeof(float) * static_cast<size_t>(B) * V);
    l.total = p;
    return l;
}

}  // namespace

size_t verify_logits_workspace_bytes(int B, int gamma, int V, int r) {
    if (B < 1 || gamma < 1 || V < 1 || r < 1) return 0;
    return vl_layout(B, gamma, V, r).total;
}

dspark_status launch_verify_logits(const float* target_logits, const float* T_t, const float* base_logits,
                                   const int32_t* anchor, const void* w1, const void* w2, dspark_dtype wdtype,
                                   const float* T_d, const float* draft_lse, const int32_t* draft_tokens,
                                   const int32_t* lengths, uint64_t seed, uint32_t offset, int B, int gamma,
                                   int V, int r, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                                   cudaStream_t stream, const DeviceInfo& dev) {
    const VLLayout l = vl_layout(B, gamma, V, r);
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
    a.done1 = reinterpret_cast<uint32_t*>(base + l.done1);
    a.done3 = reinterpret_cast<uint32_t*>(base + l.done3);
    a.decision = reinterpret_cast<int32_t*>(base + l.decision);
    a.sel = reinterpret_cast<RowSel*>(base + l.sel);
    a.part = reinterpret_cast<float2*>(base + l.part);
    a.eg = base + l.eg;
    float* bias = reinterpret_cast<float*>(base + l.bias);
    a.bias = bias;
    a.seed = seed;
    a.offset = offset;
    a.B = B;
    a.g = gamma;
    a.V = V;
    a.r = r;
    a.wbf16 = wdtype == DSPARK_BF16 ? 1 : 0;
    a.n_chunk = (V + kChunk - 1) / kChunk;
    a.total1 = static_cast<long long>(B) * (gamma + 1) * a.n_chunk;
    a.total3 = static_cast<long long>(B) * a.n_chunk;
    auto blocks_for = [&](long long items) {
        const long long want = (items + 3) / 4;                      // at least 4 chunks a warp
        return static_cast<int>(std::max(1LL, std::min(static_cast<long long>(dev.sm_count),
                                                        (want + kWarps - 1) / kWarps)));
    };
    const int blocks1 = blocks_for(a.total1), blocks3 = blocks_for(a.total3);
    a.warps1 = blocks1 * kWarps;
    a.warps3 = blocks3 * kWarps;

    vl_lse_kernel<<<blocks1, kThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(verify_logits lse)");
    st = launch_draft_logits(a.eg, w2, wdtype, B, r, V, bias, ws, stream, dev);
    if (st != DSPARK_OK) return st;
    vl_draw_kernel<<<blocks3, kThreads, 0, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(verify_logits draw)");
    return DSPARK_OK;
}

}  // namespace dspark
