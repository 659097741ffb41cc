// Greedy (temperature-0) verification of a drafted block.
//
// "xserv/docs/25-speculative-methods-comparison.md" §2: the target scores every
// drafted position at once; the longest prefix of draft tokens that each equal
// the target's argmax at their position is accepted, and the target's argmax at
// the first failing position (the position after the block when none fails) is
// appended.  Row k of the target input scores position k; the rows may be logits
// or probabilities, only their argmax is used.
//
// One kernel, bound by reading the rows.  The rows a request needs (k <= L_b)
// are cut into chunks of 2048 entries; every warp of a grid of one block per SM
// takes an equal contiguous range of the B * (gamma+1) * n_chunk chunks, finds
// each chunk's argmax (lowest index on ties, NaN never wins), folds it into the
// row's 64-bit key with one atomicMax and adds its chunk count to the request's
// counter; the warp that completes a request's count decides it.
#include "device_common.cuh"
#include "host_common.h"

#include <algorithm>

namespace dspark {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 2048;                         // entries per warp item: 16 float4 per lane

struct GreedyArgs {
    const float* t;                                  // [B, gamma+1, V]
    const int32_t* tokens;                           // [B, gamma]
    const int32_t* lengths;                          // [B] or null
    int32_t* out;                                    // [B, gamma+1]
    int32_t* n_acc;                                  // [B]
    WsHeader* ws;
    unsigned long long* keys;                        // [B][gamma+1] row argmax keys (zeroed)
    uint32_t* done;                                  // [B] chunks counted (zeroed)
    int B, gamma, V, n_chunk, warps_total;
    long long total;                                 // B * (gamma+1) * n_chunk
};

// Running argmax of one lane over entries it sees in increasing index order: branch-free, a
// strict comparison keeps the lowest index, NaN never wins.
__device__ __forceinline__ void argmax_take(float x, int e, float& best, int& idx) {
    const bool take = (x == x) & ((idx < 0) | (x > best));
    best = take ? x : best;
    idx = take ? e : idx;
}

// Argmax over one 2048-entry chunk: lane l sees entries e0 + 128 j .. + 3 (j = 0..15); the loads
// of each half are all issued before any is compared.
__device__ __forceinline__ void chunk_argmax(const float* row, int e0, int V, bool vec, float& best, int& idx) {
    const bool whole = vec && e0 + 128 * 15 + 4 <= V;            // every load of the chunk in range
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
                f[j].x = e + 0 < V ? __ldcs(row + e + 0) : nan;
                f[j].y = e + 1 < V ? __ldcs(row + e + 1) : nan;
                f[j].z = e + 2 < V ? __ldcs(row + e + 2) : nan;
                f[j].w = e + 3 < V ? __ldcs(row + e + 3) : nan;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = e0 + 128 * (8 * half + j);
            argmax_take(f[j].x, e, best, idx);
            argmax_take(f[j].y, e + 1, best, idx);
            argmax_take(f[j].z, e + 2, best, idx);
            argmax_take(f[j].w, e + 3, best, idx);
        }
    }
}

// One warp decides request b from its row keys.
__device__ void decide(const GreedyArgs& a, int b) {
    const uint32_t lane = lane_id();
    const int g = a.gamma;
    int32_t* out = a.out + static_cast<size_t>(b) * (g + 1);
    const int Lb = a.lengths != nullptr ? a.lengths[b] : g;
    bool bad = !(Lb >= 0 && Lb <= g);
    const unsigned long long* keys = a.keys + static_cast<size_t>(b) * (g + 1);
    // first position whose draft token is not the row's argmax (Lb if none)
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
            const int am = key == 0ull ? 0 : static_cast<int>(key_index(key));
            mismatch = x != am;
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
    const int correction = kk == 0ull ? 0 : static_cast<int>(key_index(kk));
    if (__any_sync(0xFFFFFFFFu, no_entry) || kk == 0ull)
        if (lane == 0) set_status(a.ws, DSPARK_STATUS_NUMERIC);          // a row without a non-NaN entry
    for (int k = static_cast<int>(lane); k <= g; k += 32) {
        int v = -1;
        if (k < kstar) v = a.tokens[static_cast<size_t>(b) * g + k];
        else if (k == kstar) v = correction;
        out[k] = v;
    }
    if (lane == 0) a.n_acc[b] = kstar;
}

__global__ void __launch_bounds__(kThreads, 1) verify_greedy_kernel(GreedyArgs a) {
    const int gw = static_cast<int>(blockIdx.x) * kWarps + static_cast<int>(warp_id());
    const uint32_t lane = lane_id();
    const long long per_req = static_cast<long long>(a.gamma + 1) * a.n_chunk;
    const bool vec = (a.V & 3) == 0;
    long long f = a.total * gw / a.warps_total;
    const long long f1 = a.total * (gw + 1) / a.warps_total;
    while (f < f1) {
        const int b = static_cast<int>(f / per_req);
        const long long req_end = min(static_cast<long long>(b + 1) * per_req, f1);
        const uint32_t count = static_cast<uint32_t>(req_end - f);
        const int Lb = a.lengths != nullptr ? a.lengths[b] : a.gamma;
        const bool len_ok = Lb >= 0 && Lb <= a.gamma;
        for (; f < req_end; ++f) {
            const long long rem = f - static_cast<long long>(b) * per_req;
            const int k = static_cast<int>(rem / a.n_chunk), c = static_cast<int>(rem % a.n_chunk);
            if (!len_ok || k > Lb) continue;                      // rows past L_b are not needed
            const float* row = a.t + (static_cast<size_t>(b) * (a.gamma + 1) + k) * a.V;
            float best = 0.f;
            int idx = -1;
            chunk_argmax(row, c * kChunk + 4 * static_cast<int>(lane), a.V, vec, best, idx);
            unsigned long long key = idx >= 0 ? argmax_key(best, static_cast<uint32_t>(idx)) : 0ull;
            key = warp_max_u64(key);
            if (lane == 0 && key != 0ull) atomicMax(a.keys + static_cast<size_t>(b) * (a.gamma + 1) + k, key);
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

size_t verify_greedy_workspace_bytes(int B, int gamma) {
    const size_t keys = sizeof(unsigned long long) * static_cast<size_t>(B) * (gamma + 1);
    const size_t done = (sizeof(uint32_t) * static_cast<size_t>(B) + 15) & ~static_cast<size_t>(15);
    return sizeof(WsHeader) + keys + done;
}

dspark_status launch_verify_greedy(const float* target, const int32_t* draft_tokens, const int32_t* lengths,
                                   int B, int gamma, int V, int32_t* out_tokens, int32_t* num_accepted,
                                   void* ws, cudaStream_t stream, const DeviceInfo& dev) {
    const dspark_status st = clear_workspace(ws, verify_greedy_workspace_bytes(B, gamma), stream);
    if (st != DSPARK_OK) return st;
    GreedyArgs a;
    a.t = target;
    a.tokens = draft_tokens;
    a.lengths = lengths;
    a.out = out_tokens;
    a.n_acc = num_accepted;
    a.ws = static_cast<WsHeader*>(ws);
    uint8_t* p = static_cast<uint8_t*>(ws) + sizeof(WsHeader);
    a.keys = reinterpret_cast<unsigned long long*>(p);
    a.done = reinterpret_cast<uint32_t*>(p + sizeof(unsigned long long) * static_cast<size_t>(B) * (gamma + 1));
    a.B = B;
    a.gamma = gamma;
    a.V = V;
    a.n_chunk = (V + kChunk - 1) / kChunk;
    a.total = static_cast<long long>(B) * (gamma + 1) * a.n_chunk;
    const long long want = (a.total + 3) / 4;                    // at least 4 chunks a warp
    const int blocks = static_cast<int>(std::max(1LL, std::min(static_cast<long long>(dev.sm_count),
                                                                (want + kWarps - 1) / kWarps)));
    a.warps_total = blocks * kWarps;
    verify_greedy_kernel<<<blocks, kThreads, 0, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(verify_greedy)");
    return DSPARK_OK;
}

}  // namespace dspark
