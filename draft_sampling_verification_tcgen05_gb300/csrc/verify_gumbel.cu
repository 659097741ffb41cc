// Verification with the draft's own Gumbel noise.
//
// "DSpark implementation and evaluation" §5: the draft samples with the
// Gumbel-max trick and the target verifies with the same Gumbel seed, so the
// output keeps the target's distribution.  Here the target draws its own token
// at position k with the noise the draft drew at step k,
//   y_k = argmax_v (t[b, k, v] / T_b + g(b, k, v))   (plain argmax when T_b = 0),
// drafted tokens are accepted while x_k = y_k, and y at the first mismatch
// (at L_b when every tested token matches) is appended: the output is the
// target's own Gumbel-max sample sequence.
//
// One kernel, bound by reading the rows, with the item / count / decide
// structure of the greedy verifier: every warp of a grid of three 256-thread
// blocks per SM (24 warps: more loads in flight than one 512-thread block at
// the register count the noise test needs) takes an equal contiguous range of
// the B * (gamma+1) * n_chunk chunks of
// 2048 entries (rows k <= L_b only).  The draft noise comes in groups of 16
// entries whose group word bounds the group's largest variate (see
// draft_gumbel in device_common.cuh); per chunk one Philox round per lane
// draws the 128 group words (lane l: counter 32 c + l), the four lanes of a
// group take its largest z by two shuffles, and a group is drawn exactly only
// when that z plus a table bound on its largest variate reaches the best
// exact value the row has reached so far (seeded from the row's key and raised
// by each group's largest variate, which is exact at the group's position p).
// The chunk's best key goes to the row's key by atomicMax; the warp that
// completes a request's chunk count decides it.
#include "device_common.cuh"
#include "host_common.h"

#include <algorithm>

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 3;                      // 24 warps per SM (registers capped at 80)
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 2048;                         // entries per warp item: 16 float4 per lane

struct GumbelArgs {
    const float* t;                                  // [B, gamma+1, V] target logits
    const float* temperature;                        // [B]
    const int32_t* tokens;                           // [B, gamma]
    const int32_t* lengths;                          // [B] or null
    int32_t* out;                                    // [B, gamma+1]
    int32_t* n_acc;                                  // [B]
    WsHeader* ws;
    unsigned long long* keys;                        // [B][gamma+1] row keys (zeroed)
    uint32_t* done;                                  // [B] chunks counted (zeroed)
    uint64_t seed;
    uint32_t offset;
    int B, gamma, V, n_chunk, warps_total;
    long long total;                                 // B * (gamma+1) * n_chunk
};

__device__ __forceinline__ void take(unsigned long long& best, float y, int v) {
    if (y == y) {
        const unsigned long long k = argmax_key(y, static_cast<uint32_t>(v));
        best = k > best ? k : best;
    }
}

// Running argmax of one lane over entries it sees in increasing index order: a strict comparison
// keeps the lowest index, NaN never wins.
__device__ __forceinline__ void argmax_take(float x, int e, float& best, int& idx) {
    const bool take_it = (x == x) & ((idx < 0) | (x > best));
    best = take_it ? x : best;
    idx = take_it ? e : idx;
}

struct Running {
    float lb;                                        // best exact score the row has reached
    unsigned long long best;                         // this lane's best key
};

// The groups of one step of the chunk loop that the table could not rule out (rare; out of line
// so the unrolled loop stays small): the exact largest variate first (exact for the entry at
// position p, which becomes a candidate), the bound raised to the best of them over the warp,
// then the lane's entries that can still reach it draw their own variate.  Called by the whole
// warp.
__device__ __noinline__ Running draw_groups(const GumbelArgs& a, int b, int k, int e, uint32_t W, float z0, float z1,
                                            float z2, float z3, bool pass, Running run) {
    const uint32_t lane = lane_id();
    const float z[4] = {z0, z1, z2, z3};
    const float e_min = group_e_min(W);
    const float g_top = -logf(e_min);
    const uint32_t p = W & 15u;
    const uint32_t kpos0 = 4u * (lane & 3u);                    // this lane's first position in the group
    if (pass && p - kpos0 < 4u) {
        const int q = static_cast<int>(p - kpos0);
        take(run.best, __fadd_rn(z[q], g_top), e + q);
    }
    const unsigned long long top = warp_max_u64(run.best);
    if (top != 0ull) run.lb = fmaxf(run.lb, float_from_order_bits(static_cast<uint32_t>(top >> 32)));
    if (pass) {
        const uint32_t G = static_cast<uint32_t>(e) >> 4;
        uint4 ew = make_uint4(0, 0, 0, 0);
        bool have = false;
        for (int q = 0; q < 4; ++q) {
            if (kpos0 + static_cast<uint32_t>(q) == p) continue;
            if (!(__fadd_rn(__fadd_rn(z[q], g_top), 1e-3f) >= run.lb)) continue;    // can not reach it (or NaN)
            if (!have) {
                ew = philox_at(a.seed, a.offset, (G << 2) | (lane & 3u), static_cast<uint32_t>(b), kStreamGumbelLo,
                               static_cast<uint32_t>(k));
                have = true;
            }
            take(run.best, __fadd_rn(z[q], draft_gumbel_of_entry(e_min, word_of(ew, static_cast<uint32_t>(q)))), e + q);
        }
    }
    return run;
}

// Best key of one chunk of row (b, k) scored by z = t * invT plus the draft noise of step k.
// Lane l holds entries e0 + 128 j + 4 l .. + 3 (j = 0..15); the four lanes 4m..4m+3 hold one
// noise group for every j.
__device__ unsigned long long chunk_gumbel(const GumbelArgs& a, const float* row, int b, int k, int c, float invT,
                                           float lb, const float* gtab, uint4* wbuf) {
    const uint32_t lane = lane_id();
    const int e0 = c * kChunk + 4 * static_cast<int>(lane);
    const bool whole = (a.V & 3) == 0 && c * kChunk + kChunk <= a.V;
    // group words of the chunk's 128 groups: lane l draws groups 4l .. 4l+3
    const uint4 gw = philox_at(a.seed, a.offset, static_cast<uint32_t>(c * 32) + lane, static_cast<uint32_t>(b),
                               kStreamGumbel, static_cast<uint32_t>(k));
    // through the warp's 512-byte buffer: lane l later reads word (l >> 2) & 3 of lane 2 jj + (l >> 4)
    __syncwarp();
    wbuf[lane] = gw;
    __syncwarp();
    const uint32_t* wsrc = reinterpret_cast<const uint32_t*>(wbuf) + 4 * (lane >> 4) + ((lane >> 2) & 3u);
    Running run = {lb, 0ull};
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        float4 f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = e0 + 128 * (8 * half + j);
            if (whole) {
                f[j] = __ldcs(reinterpret_cast<const float4*>(row + e));
            } else {
                const float nan = __int_as_float(0x7FC00000);
                f[j].x = e + 0 < a.V ? __ldcs(row + e + 0) : nan;
                f[j].y = e + 1 < a.V ? __ldcs(row + e + 1) : nan;
                f[j].z = e + 2 < a.V ? __ldcs(row + e + 2) : nan;
                f[j].w = e + 3 < a.V ? __ldcs(row + e + 3) : nan;
            }
        }
        // the eight group tests of this half first (independent of each other), against the
        // bound reached before the half; then the rare groups that pass are drawn in order
        uint32_t Ws[8];
        uint32_t passm = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int jj = 8 * half + j;
            f[j].x = __fmul_rn(f[j].x, invT);
            f[j].y = __fmul_rn(f[j].y, invT);
            f[j].z = __fmul_rn(f[j].z, invT);
            f[j].w = __fmul_rn(f[j].w, invT);
            Ws[j] = wsrc[8 * jj];                        // the group word of this lane's group
            float gm = fmaxf(fmaxf(f[j].x, f[j].y), fmaxf(f[j].z, f[j].w));   // NaN (and past-V) never win
            gm = fmaxf(gm, __shfl_xor_sync(0xFFFFFFFFu, gm, 1));
            gm = fmaxf(gm, __shfl_xor_sync(0xFFFFFFFFu, gm, 2));
            const bool pass = __fadd_rn(gm, gtab[Ws[j] >> 24]) >= run.lb;
            passm |= (pass ? 1u : 0u) << j;
        }
        const uint32_t warpm = __reduce_or_sync(0xFFFFFFFFu, passm);
        if (warpm == 0u) continue;                                        // uniform over the warp
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if ((warpm >> j) & 1u)
                run = draw_groups(a, b, k, e0 + 128 * (8 * half + j), Ws[j], f[j].x, f[j].y, f[j].z, f[j].w,
                                  ((passm >> j) & 1u) != 0u, run);
    }
    return warp_max_u64(run.best);
}

// Plain argmax of one chunk (a greedy request): lowest index on ties, NaN never wins.  The loads
// of each half are all issued before any is compared.
__device__ unsigned long long chunk_argmax(const GumbelArgs& a, const float* row, int c) {
    const uint32_t lane = lane_id();
    const int e0 = c * kChunk + 4 * static_cast<int>(lane);
    const bool whole = (a.V & 3) == 0 && c * kChunk + kChunk <= a.V;
    float bv = 0.f;
    int bi = -1;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float4 f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = e0 + 128 * (8 * half + j);
            if (whole) {
                f[j] = __ldcs(reinterpret_cast<const float4*>(row + e));
            } else {
                const float nan = __int_as_float(0x7FC00000);
                f[j].x = e + 0 < a.V ? __ldcs(row + e + 0) : nan;
                f[j].y = e + 1 < a.V ? __ldcs(row + e + 1) : nan;
                f[j].z = e + 2 < a.V ? __ldcs(row + e + 2) : nan;
                f[j].w = e + 3 < a.V ? __ldcs(row + e + 3) : nan;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = e0 + 128 * (8 * half + j);
            argmax_take(f[j].x, e, bv, bi);
            argmax_take(f[j].y, e + 1, bv, bi);
            argmax_take(f[j].z, e + 2, bv, bi);
            argmax_take(f[j].w, e + 3, bv, bi);
        }
    }
    const unsigned long long best = bi >= 0 ? argmax_key(bv, static_cast<uint32_t>(bi)) : 0ull;
    return warp_max_u64(best);
}

// One warp decides request b from its row keys (the target's token of each row).
__device__ void decide(const GumbelArgs& a, int b) {
    const uint32_t lane = lane_id();
    const int g = a.gamma;
    int32_t* out = a.out + static_cast<size_t>(b) * (g + 1);
    const int Lb = a.lengths != nullptr ? a.lengths[b] : g;
    bool bad = !(Lb >= 0 && Lb <= g);
    const unsigned long long* keys = a.keys + static_cast<size_t>(b) * (g + 1);
    int kstar = Lb;
    bool no_entry = false;
    for (int k0 = 0; !bad && k0 < Lb; k0 += 32) {
        const int k = k0 + static_cast<int>(lane);
        bool mismatch = false, invalid = false;
        if (k < Lb) {
            const int x = a.tokens[static_cast<size_t>(b) * g + k];
            invalid = x < 0 || x >= a.V;
            const unsigned long long key = __ldcg(keys + k);
            no_entry |= key == 0ull;
            mismatch = x != (key == 0ull ? 0 : static_cast<int>(key_index(key)));
        }
        bad = __any_sync(0xFFFFFFFFu, invalid);
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, mismatch);
        if (m != 0u && kstar == Lb) kstar = min(kstar, k0 + __ffs(m) - 1);
    }
    if (bad) {
        if (lane == 0) flag_input_index(a.ws);
        for (int k = static_cast<int>(lane); k <= g; k += 32) out[k] = -1;
        if (lane == 0) a.n_acc[b] = 0;
        return;
    }
    const unsigned long long kk = __ldcg(keys + kstar);
    const int y = kk == 0ull ? 0 : static_cast<int>(key_index(kk));
    if (__any_sync(0xFFFFFFFFu, no_entry) || kk == 0ull)
        if (lane == 0) set_status(a.ws, DSPARK_STATUS_NUMERIC);          // a row without a scored entry
    for (int k = static_cast<int>(lane); k <= g; k += 32) {
        int v = -1;
        if (k < kstar) v = a.tokens[static_cast<size_t>(b) * g + k];
        else if (k == kstar) v = y;
        out[k] = v;
    }
    if (lane == 0) a.n_acc[b] = kstar;
}

__global__ void __launch_bounds__(kThreads, kBlocksPerSm) verify_gumbel_kernel(GumbelArgs a) {
    // gtab[k]: bound on the largest variate -log(E_min) of a noise group whose group word has
    // top byte k (that of the largest such word, plus a margin for logf's rounding)
    __shared__ float gtab[256];
    __shared__ uint4 s_words[kWarps][32];                // per-warp transpose of the chunk's group words
    for (int k = threadIdx.x; k < 256; k += kThreads)
        gtab[k] = k == 255 ? kDraftGumbelMax : -logf(group_e_min((static_cast<uint32_t>(k + 1) << 24) - 1u)) + 1e-3f;
    __syncthreads();
    const int gw = static_cast<int>(blockIdx.x) * kWarps + static_cast<int>(warp_id());
    const uint32_t lane = lane_id();
    const long long per_req = static_cast<long long>(a.gamma + 1) * a.n_chunk;
    long long f = a.total * gw / a.warps_total;
    const long long f1 = a.total * (gw + 1) / a.warps_total;
    while (f < f1) {
        const int b = static_cast<int>(f / per_req);
        const long long req_end = min(static_cast<long long>(b + 1) * per_req, f1);
        const uint32_t count = static_cast<uint32_t>(req_end - f);
        const int Lb = a.lengths != nullptr ? a.lengths[b] : a.gamma;
        const bool len_ok = Lb >= 0 && Lb <= a.gamma;
        float T = a.temperature[b];
        if (!(T >= 0.f) || isinf(T)) {                  // NaN, negative or infinite: scored greedily
            if (lane == 0) set_status(a.ws, DSPARK_STATUS_NUMERIC);
            T = 0.f;
        }
        const float invT = T > 0.f ? __frcp_rn(T) : 0.f;
        for (; f < req_end; ++f) {
            const long long rem = f - static_cast<long long>(b) * per_req;
            const int k = static_cast<int>(rem / a.n_chunk), c = static_cast<int>(rem % a.n_chunk);
            if (!len_ok || k > Lb) continue;                      // rows past L_b are not needed
            const float* row = a.t + (static_cast<size_t>(b) * (a.gamma + 1) + k) * a.V;
            unsigned long long* slot = a.keys + static_cast<size_t>(b) * (a.gamma + 1) + k;
            if (f + 1 < req_end) {
                // bring the warp's next chunk of this request into L2 while this one is scored
                const long long rn = rem + 1;
                const int kn = static_cast<int>(rn / a.n_chunk), cn = static_cast<int>(rn % a.n_chunk);
                if (kn <= Lb) {
                    const float* nrow = a.t + (static_cast<size_t>(b) * (a.gamma + 1) + kn) * a.V;
                    const int e = cn * kChunk + 64 * static_cast<int>(lane);
                    if (e < a.V) prefetch_l2(nrow + e);
                    if (e + 32 < a.V) prefetch_l2(nrow + e + 32);
                }
            }
            unsigned long long key;
            if (invT > 0.f) {
                // the best exact value another chunk of the row has reached already
                const unsigned long long seen = __ldcg(slot);
                const float lb = seen != 0ull ? float_from_order_bits(static_cast<uint32_t>(seen >> 32)) : -INFINITY;
                key = chunk_gumbel(a, row, b, k, c, invT, lb, gtab, s_words[warp_id()]);
            } else {
                key = chunk_argmax(a, row, c);
            }
            if (lane == 0 && key != 0ull) atomicMax(slot, key);
        }
        // count this warp's chunks of request b; the warp completing the count decides it
        uint32_t last = 0;
        if (lane == 0)                                   // release this warp's keys, acquire the others'
            last = atom_add_acq_rel(a.done + b, count) + count == static_cast<uint32_t>(per_req) ? 1u : 0u;
        __syncwarp();                                    // the other lanes read after lane 0's acquire
        if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
            decide(a, b);
        }
    }
}

}  // namespace

size_t verify_gumbel_workspace_bytes(int B, int gamma) {
    const size_t keys = sizeof(unsigned long long) * static_cast<size_t>(B) * (gamma + 1);
    const size_t done = (sizeof(uint32_t) * static_cast<size_t>(B) + 15) & ~static_cast<size_t>(15);
    return sizeof(WsHeader) + keys + done;
}

dspark_status launch_verify_gumbel(const float* target_logits, const float* temperature, const int32_t* draft_tokens,
                                   const int32_t* lengths, uint64_t seed, uint32_t offset, int B, int gamma, int V,
                                   int32_t* out_tokens, int32_t* num_accepted, void* ws, cudaStream_t stream,
                                   const DeviceInfo& dev) {
    const dspark_status st = clear_workspace(ws, verify_gumbel_workspace_bytes(B, gamma), stream);
    if (st != DSPARK_OK) return st;
    GumbelArgs a;
    a.t = target_logits;
    a.temperature = temperature;
    a.tokens = draft_tokens;
    a.lengths = lengths;
    a.out = out_tokens;
    a.n_acc = num_accepted;
    a.ws = static_cast<WsHeader*>(ws);
    uint8_t* p = static_cast<uint8_t*>(ws) + sizeof(WsHeader);
    a.keys = reinterpret_cast<unsigned long long*>(p);
    a.done = reinterpret_cast<uint32_t*>(p + sizeof(unsigned long long) * static_cast<size_t>(B) * (gamma + 1));
    a.seed = seed;
    a.offset = offset;
    a.B = B;
    a.gamma = gamma;
    a.V = V;
    a.n_chunk = (V + kChunk - 1) / kChunk;
    a.total = static_cast<long long>(B) * (gamma + 1) * a.n_chunk;
    const long long want = (a.total + 3) / 4;                    // at least 4 chunks a warp
    const int blocks = static_cast<int>(std::max(1LL, std::min(static_cast<long long>(dev.sm_count) * kBlocksPerSm,
                                                                (want + kWarps - 1) / kWarps)));
    a.warps_total = blocks * kWarps;
    verify_gumbel_kernel<<<blocks, kThreads, 0, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(verify_gumbel)");
    return DSPARK_OK;
}

}  // namespace dspark
