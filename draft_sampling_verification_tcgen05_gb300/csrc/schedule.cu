// Confidence-scheduled admission of draft tokens.
//
// "Speculative decoding: from zero to DSpark" §6: conditional acceptance
// probabilities are chained into survival probabilities; all candidates of all
// requests are pooled, sorted by survival and admitted from the top; the
// verify capacity maximises expected tokens x SPS(batch size).  §7: the SPS
// curve is jagged, so every K is evaluated; K may also be fixed ahead of time
// and only the fill done now.  No token value is read at any point.
//
// Every kernel takes the same steps:
//   1. survival chain per request (fp32, round to nearest, no contraction);
//      sort key (~bits(s)) per candidate, index order
//   2. stable sort of the candidates by that key (the index breaks survival
//      ties): LSD radix passes of 8 bits whose per-key ranks come from warp
//      ballots, or a bitonic network over (key << 32 | index) for small pools
//   3. if K is to be chosen: fixed-point masses floor(s * 2^32) from the float
//      bits, prefix sums, f(K) = float64(B * 2^32 + prefix) * SPS[K-1] for
//      every K with the rounding done in integer arithmetic (the FP64 pipe of
//      this GPU is narrow), argmax with ties to the smallest K
//   4. fill: selected in rank order, lengths of the admitted prefixes
// and differ in where the keys live:
//   <= 32 candidates        one warp, one candidate per lane
//   <= 2048                 one block, shared memory (bitonic sort above 256)
//   <= 16384 (2049 and up)  a cluster of 16 (or 8) blocks, distributed shared memory
//                           (one block with shared memory where a block's share
//                           of the requests does not fit)
//   <= 2^20                 one block, keys in the workspace (global memory, L2)
#include "device_common.cuh"
#include "host_common.h"

#include <cooperative_groups.h>
#include <mutex>

namespace dspark {
namespace {

constexpr int kRadix = 256;

struct ScheduleArgs {
    const float* c;
    const double* sps;
    float* survival;
    int32_t* K_out;
    int32_t* lengths;
    int32_t* selected;
    unsigned long long* keys0;
    unsigned long long* keys1;
    WsHeader* ws;
    int S, B, N, K_in;
};

__device__ __forceinline__ float clamp_prob(float x, bool& bad) {
    if (!(x >= 0.f)) { bad = true; return 0.f; }     // negative or NaN
    if (x > 1.f) { bad = true; return 1.f; }
    return x;
}

// Sort key of a survival value: smaller key = earlier in the admission order.  -0 and +0
// are one value (the key of +0).
__device__ __forceinline__ uint32_t order_key(float s) {
    return 0xFFFFFFFFu - __float_as_uint(__fadd_rn(s, 0.f));
}

// Survival back from its key.
__device__ __forceinline__ float key_survival(uint32_t key) { return __uint_as_float(0xFFFFFFFFu - key); }

// floor(s * 2^32) for s in [0, 1] from the float's bits (s = m * 2^(e - 150) for biased
// exponent e and 24-bit significand m, so s * 2^32 = m * 2^(e - 118)); subnormals give 0.
__device__ __forceinline__ unsigned long long mass32(float s) {
    const uint32_t bits = __float_as_uint(s) & 0x7FFFFFFFu;
    const int e = static_cast<int>(bits >> 23);
    const unsigned long long m = (bits & 0x7FFFFFu) | 0x800000u;
    const int sh = e - 118;
    if (e == 0 || sh <= -24) return 0ull;
    return sh >= 0 ? m << sh : m >> -sh;          // s <= 1 keeps sh <= 9
}

constexpr unsigned long long kMant52 = 0xFFFFFFFFFFFFFull;

// Bits of float64(E), round to nearest even, for E >= 1 (integer operations only).
__device__ __forceinline__ unsigned long long u64_to_f64_bits(unsigned long long E) {
    const int lz = __clzll(static_cast<long long>(E));
    const unsigned long long m = E << lz;          // leading one at bit 63
    unsigned long long hi = m >> 11;               // 53 significant bits
    const unsigned long long rem = m & 0x7FFull;
    int ex = 63 - lz;
    if (rem > 0x400ull || (rem == 0x400ull && (hi & 1ull))) {
        ++hi;
        if (hi >> 53) {
            hi >>= 1;
            ++ex;
        }
    }
    return (static_cast<unsigned long long>(ex + 1023) << 52) | (hi & kMant52);
}

// Bits of fl64(a * b), round to nearest even, for a positive normal double a (bits ab) when
// b (bits bb) is a positive normal double and the rounded product is normal; returns false
// in every other case, where the caller multiplies with __dmul_rn instead.  The significands
// (53 bits each) multiply exactly into 106 bits, which are cut back to 53 with the
// round-half-even rule.
__device__ __forceinline__ bool f64_mul_bits(unsigned long long ab, unsigned long long bb,
                                             unsigned long long* out) {
    const int eb = static_cast<int>((bb >> 52) & 0x7FFull);
    if ((bb >> 63) != 0ull || eb == 0 || eb == 0x7FF) return false;
    const int ea = static_cast<int>(ab >> 52);
    const unsigned long long ma = (ab & kMant52) | (1ull << 52);
    const unsigned long long mb = (bb & kMant52) | (1ull << 52);
    const unsigned long long lo = ma * mb, hi = __umul64hi(ma, mb);      // product in [2^104, 2^106)
    const int top = static_cast<int>((hi >> 41) & 1ull);                  // product >= 2^105
    const int sh = 52 + top;
    unsigned long long r = (hi << (64 - sh)) | (lo >> sh);                // 53 bits
    const unsigned long long rest = lo & ((1ull << sh) - 1ull);
    const unsigned long long half = 1ull << (sh - 1);
    int e = ea + eb - 1023 + top;                                         // biased exponent
    if (rest > half || (rest == half && (r & 1ull))) {
        ++r;
        if (r >> 53) {
            r >>= 1;
            ++e;
        }
    }
    if (e <= 0 || e >= 0x7FF) return false;
    *out = (static_cast<unsigned long long>(e) << 52) | (r & kMant52);
    return true;
}

// f(K) = float64(E) * sps as a key that orders like the double (larger key = larger f);
// 0 for a NaN or -inf product, which never wins (the search starts below every f > -inf).
__device__ __forceinline__ unsigned long long objective_key(unsigned long long E, double sps) {
    const unsigned long long eb = u64_to_f64_bits(E);
    unsigned long long fb;
    if (!f64_mul_bits(eb, static_cast<unsigned long long>(__double_as_longlong(sps)), &fb)) {
        const double f = __dmul_rn(__longlong_as_double(static_cast<long long>(eb)), sps);
        if (!(f > -INFINITY)) return 0ull;
        fb = static_cast<unsigned long long>(__double_as_longlong(f));
        if ((fb << 1) == 0ull) fb = 0ull;                               // -0 is +0
    }
    return (fb >> 63) ? ~fb : (fb | 0x8000000000000000ull);
}

// The warp's largest key and, among the lanes holding it, the smallest K (to every lane), by the
// hardware's 32-bit reduce instructions rather than shuffle rounds (on this GPU a shuffle occupies
// its sub-partition for about seven issue cycles, a vote about fourteen).
__device__ __forceinline__ void warp_best_key(unsigned long long& key, int& K) {
    const uint32_t hi = static_cast<uint32_t>(key >> 32), lo = static_cast<uint32_t>(key);
    const uint32_t mhi = __reduce_max_sync(0xFFFFFFFFu, hi);
    const uint32_t mlo = __reduce_max_sync(0xFFFFFFFFu, hi == mhi ? lo : 0u);
    const bool top = hi == mhi && lo == mlo;
    K = static_cast<int>(__reduce_min_sync(0xFFFFFFFFu, top ? static_cast<uint32_t>(K) : 0xFFFFFFFFu));
    key = (static_cast<unsigned long long>(mhi) << 32) | mlo;
}

// Capacity K* over the sorted order (sorted(j) = the sort key of the j-th candidate), shared by
// the one-block kernels.  Thread t owns the contiguous K range [t per, (t + 1) per): it sums its
// masses, one block scan of the thread sums gives each range its starting prefix, and a second
// walk forms every E(K) and keeps the best f(K) (ascending K, so a strict comparison keeps the
// smallest K).  The reductions over the block use the hardware's 32-bit reduce instructions.
// Returns K* to every thread.
template <int kThreads, typename SortedKey>
__device__ int choose_capacity(const ScheduleArgs& a, int n, SortedKey sorted, unsigned long long* s_wsum,
                               unsigned long long* s_bk, int* s_bK, int* s_K) {
    constexpr int kWarps = kThreads / 32;
    const int tid = threadIdx.x;
    const uint32_t lane = lane_id(), warp = warp_id();
    const int Kmax = a.S < n ? a.S : n;
    const int per = (Kmax + kThreads - 1) / kThreads;
    const int j0 = min(Kmax, tid * per), j1 = min(Kmax, j0 + per);
    unsigned long long part = 0;
    for (int j = j0; j < j1; ++j) part += mass32(key_survival(sorted(j)));
    // block exclusive scan of the thread sums
    unsigned long long incl = part;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= static_cast<uint32_t>(o)) incl += y;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const unsigned long long v = lane < static_cast<uint32_t>(kWarps) ? s_wsum[lane] : 0ull;
        unsigned long long x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= static_cast<uint32_t>(o)) x += y;
        }
        if (lane < static_cast<uint32_t>(kWarps)) s_wsum[lane] = x - v;
    }
    __syncthreads();
    unsigned long long E = (static_cast<unsigned long long>(a.B) << 32) + s_wsum[warp] + incl - part;
    unsigned long long best_key = 0ull;                   // below every f > -inf
    int best_K = 0x7FFFFFFF;
    for (int j = j0; j < j1; ++j) {
        E += mass32(key_survival(sorted(j)));
        const unsigned long long k = objective_key(E, __ldg(a.sps + j));
        if (k > best_key) {
            best_key = k;
            best_K = j + 1;
        }
    }
    warp_best_key(best_key, best_K);
    if (lane == 0) {
        s_bk[warp] = best_key;
        s_bK[warp] = best_K;
    }
    __syncthreads();
    if (warp == 0) {
        unsigned long long bkey = lane < static_cast<uint32_t>(kWarps) ? s_bk[lane] : 0ull;
        int bK = lane < static_cast<uint32_t>(kWarps) ? s_bK[lane] : 0x7FFFFFFF;
        warp_best_key(bkey, bK);
        if (lane == 0) {
            if (bK == 0x7FFFFFFF) {             // every f was NaN or -inf: K = 1, flagged
                set_status(a.ws, DSPARK_STATUS_NUMERIC);
                bK = 1;
            }
            *s_K = bK;
        }
    }
    __syncthreads();
    return *s_K;
}

// ---------------------------------------------------------------------------
// Pools of at most 32 candidates (a few decode requests): one warp, one candidate per lane,
// no block barrier at all.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32) schedule_warp_kernel(ScheduleArgs a) {
    __shared__ int s_at_rank[32];
    const int lane = static_cast<int>(threadIdx.x);
    if (lane == 0) a.ws->status = 0u;            // this call's status word; only lane 0 sets bits
    const int B = a.B, N = a.N, n = B * N;
    const bool valid = lane < n;
    const int k = lane % N;
    bool bad = false;
    const float c = valid ? clamp_prob(__ldg(a.c + lane), bad) : 1.f;
    // survival chain: at step t the lanes with k == t multiply their left neighbour's
    // (final) survival by their own confidence
    float s = c;
    for (int t = 1; t < N; ++t) {
        const float left = __shfl_up_sync(0xFFFFFFFFu, s, 1);
        if (k == t) s = __fmul_rn(left, c);
    }
    if (valid) a.survival[lane] = s;
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) set_status(a.ws, DSPARK_STATUS_INPUT_RANGE);
    // rank = keys before this one in (key, index) order; empty lanes sort last
    const uint32_t my = valid ? order_key(s) : 0xFFFFFFFFu;
    int rank = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t other = __shfl_sync(0xFFFFFFFFu, my, i);
        rank += (other < my || (other == my && i < lane)) ? 1 : 0;
    }
    s_at_rank[rank] = lane;
    __syncwarp();
    const int at = s_at_rank[lane];                        // candidate at rank `lane`
    const float s_at = __shfl_sync(0xFFFFFFFFu, s, at);
    int K;
    if (a.K_in >= 0) {
        K = a.K_in < n ? a.K_in : n;
    } else {
        const int Kmax = a.S < n ? a.S : n;
        const bool in = lane < Kmax;
        unsigned long long incl = in ? mass32(s_at) : 0ull;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        unsigned long long best_key = in ? objective_key((static_cast<unsigned long long>(B) << 32) + incl,
                                                         __ldg(a.sps + lane))
                                         : 0ull;
        int best_K = best_key != 0ull ? lane + 1 : 0x7FFFFFFF;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long ok = __shfl_xor_sync(0xFFFFFFFFu, best_key, o);
            const int oK = __shfl_xor_sync(0xFFFFFFFFu, best_K, o);
            if (ok > best_key || (ok == best_key && oK < best_K)) {
                best_key = ok;
                best_K = oK;
            }
        }
        if (best_K == 0x7FFFFFFF) {                       // every f was NaN or -inf: K = 1, flagged
            if (lane == 0) set_status(a.ws, DSPARK_STATUS_NUMERIC);
            best_K = 1;
        }
        K = best_K;
    }
    if (valid) a.selected[lane] = lane < K ? at : -1;
    const unsigned long long admitted = __ballot_sync(0xFFFFFFFFu, valid && rank < K);
    if (lane < B) {
        const unsigned long long mask = (N >= 64 ? ~0ull : ((1ull << N) - 1ull)) << (lane * N);
        a.lengths[lane] = __popcll(admitted & mask);
    }
    if (lane == 0) a.K_out[0] = K;
}

// ---------------------------------------------------------------------------
// Pools of up to kSmemMaxCandidates: everything in shared memory.
// ---------------------------------------------------------------------------
constexpr int kSmemMaxCandidates = 16384;
constexpr int kBitonicMax = 2048;                                   // pools sorted by the bitonic network
constexpr int kMaxRounds = kSmemMaxCandidates / (32 * 32);       // rounds of 32 keys per warp (1024 threads)

// Dynamic shared memory: key[nn] u32 | idxA[nn] u16 | idxB[nn] u16 | cnt[kWarps][256] u16, nn = n
// rounded up to 32 (whole swizzle rows)
size_t smem_schedule_bytes(int n, int warps) {
    const size_t nn = (static_cast<size_t>(n) + 31) & ~static_cast<size_t>(31);
    return 4 * nn + 2 * 2 * nn + 2 * static_cast<size_t>(warps) * kRadix;
}

// Lanes of the warp holding the same 8-bit digit as this lane (bit 8 set = no digit: such a
// lane matches only lanes that also have no digit), from nine ballots; a warp match would do
// the same in one instruction, but it is far slower on this GPU.
__device__ __forceinline__ uint32_t same_digit_lanes(uint32_t d) {
    uint32_t peers = 0xFFFFFFFFu;
#pragma unroll
    for (int bit = 0; bit < 9; ++bit) {
        const uint32_t ones = __ballot_sync(0xFFFFFFFFu, (d >> bit) & 1u);
        peers &= ((d >> bit) & 1u) ? ones : ~ones;
    }
    return peers;
}

// Shared-memory slot of candidate id's key: rows of 32 words are permuted by the row index, so
// one thread per request walking its N consecutive keys (lanes N words apart) does not hit
// the same bank from every lane.
__device__ __forceinline__ int swz(int id) { return id ^ ((id >> 5) & 31); }

template <int kThreads>
__global__ void __launch_bounds__(kThreads, 1) schedule_smem_kernel(ScheduleArgs a) {
    constexpr int kWarps = kThreads / 32;
    constexpr int kQuarters = kThreads / kRadix;        // (digit, quarter) threads of the scan
    constexpr int kWarpsPerQuarter = kWarps / kQuarters;
    static_assert(kWarpsPerQuarter * kQuarters == kWarps, "scan layout");
    // rounds of 32 keys per warp: 16 at 1024 threads (16384 keys), 1 at 256 threads (256 keys)
    constexpr int kRounds = kThreads == 1024 ? kMaxRounds : 1;
    extern __shared__ __align__(16) unsigned char s_dyn[];
    __shared__ uint32_t s_qs[kQuarters][kRadix];
    __shared__ uint32_t s_wt[kRadix / 32];
    __shared__ unsigned long long s_wsum[kWarps];
    __shared__ unsigned long long s_bk[kWarps];
    __shared__ int s_bK[kWarps];
    __shared__ int s_K;
    __shared__ int s_bad;

    const int tid = threadIdx.x;
    const uint32_t lane = lane_id(), warp = warp_id();
    const int B = a.B, N = a.N;
    const int n = B * N;
    const int nn = (n + 31) & ~31;
    uint32_t* key = reinterpret_cast<uint32_t*>(s_dyn);   // key[swz(id)], nn words
    uint16_t* idxA = reinterpret_cast<uint16_t*>(key + nn);
    uint16_t* idxB = idxA + nn;
    uint16_t* cnt = idxB + nn;                           // [kWarps][kRadix]

    // the SPS table is read late (step 3): start pulling it into L2 now
    if (a.K_in < 0) {
        const int Kmax = a.S < n ? a.S : n;
        for (int j = tid * 16; j < Kmax; j += kThreads * 16) prefetch_l2(a.sps + j);
    }

    // ---- 1. coalesced load of c, survival chain (one thread per request), keys ----
    if (tid == 0) {
        s_bad = 0;
        a.ws->status = 0u;                       // this call's status word; only thread 0 sets bits
    }
    for (int j = tid; j < n; j += kThreads) {
        key[swz(j)] = __float_as_uint(__ldg(a.c + j));
        idxA[j] = static_cast<uint16_t>(j);
    }
    __syncthreads();
    bool bad = false;
    for (int b = tid; b < B; b += kThreads) {
        float s = 1.f;
        for (int k0 = 0; k0 < N; k0 += 8) {                      // eight loads in flight, then the chain
            uint32_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = k0 + u < N ? key[swz(b * N + k0 + u)] : 0u;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (k0 + u < N) {
                    const float c = clamp_prob(__uint_as_float(v[u]), bad);
                    s = (k0 + u == 0) ? c : __fmul_rn(s, c);
                    a.survival[b * N + k0 + u] = s;
                    v[u] = order_key(s);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (k0 + u < N) key[swz(b * N + k0 + u)] = v[u];
        }
    }
    if (bad) s_bad = 1;
    __syncthreads();
    if (tid == 0 && s_bad) set_status(a.ws, DSPARK_STATUS_INPUT_RANGE);

    uint16_t* src = idxA;
    if (kThreads == 1024 && n <= kBitonicMax) {
        // ---- 2'. pools of up to 2048: bitonic sort of (key << 32 | index) in the counter area.
        //      Equal keys fall to the lower index, as in the stable radix sort.  Pair i of a stage with
        //      partner distance jj <= 32 lies in its warp's 64-entry window, so those stages
        //      need only a warp barrier ----
        unsigned long long* sk = reinterpret_cast<unsigned long long*>(cnt);
        int P = 64;
        while (P < n) P <<= 1;
        for (int j = tid; j < P; j += kThreads)
            sk[j] = j < n ? (static_cast<unsigned long long>(key[swz(j)]) << 32) | static_cast<unsigned long long>(j)
                          : ~0ull;
        __syncthreads();
        for (int k = 2; k <= P; k <<= 1) {
            for (int jj = k >> 1; jj > 0; jj >>= 1) {
                for (int i = tid; i < P / 2; i += kThreads) {
                    const int pos = 2 * i - (i & (jj - 1));
                    const unsigned long long x = sk[pos], y = sk[pos + jj];
                    if ((x > y) == ((pos & k) == 0)) {
                        sk[pos] = y;
                        sk[pos + jj] = x;
                    }
                }
                // the next stage crosses warps when its distance is 64 or more
                const int next = jj > 1 ? jj >> 1 : k;
                if (jj >= 64 || next >= 64) __syncthreads(); else __syncwarp();
            }
        }
        __syncthreads();
        for (int j = tid; j < n; j += kThreads) idxA[j] = static_cast<uint16_t>(sk[j] & 0xFFFFull);
        __syncthreads();
    } else {
    // ---- 2. stable LSD radix sort of the indices by key ----
    // warp w ranks the run [w0, w1) of the current order; chunk is a multiple of 32
    const int chunk = (((n + kWarps - 1) / kWarps) + 31) & ~31;
    const int w0 = static_cast<int>(warp) * chunk;
    const int w1 = min(n, w0 + chunk);
    const int rounds = w1 > w0 ? (w1 - w0 + 31) / 32 : 0;
    uint16_t* dst = idxB;
    uint16_t* mycnt = cnt + warp * kRadix;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 8 * pass;
        for (int i = tid; i < kWarps * kRadix / 2; i += kThreads) reinterpret_cast<uint32_t*>(cnt)[i] = 0u;
        // (a) digits of this warp's keys, all loads first
        uint32_t slot[kRounds];
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
            const int j = w0 + r * 32 + static_cast<int>(lane);
            slot[r] = (r < rounds && j < w1) ? ((key[swz(src[j])] >> shift) & 0xFFu) : (0x100u | lane);
        }
        __syncthreads();                                  // counters cleared
        // per-warp digit counts; each key keeps (digit << 16 | offset within the warp's digit)
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
            if (r < rounds) {
                const uint32_t d = slot[r];
                const bool valid = d < 0x100u;
                const uint32_t peers = same_digit_lanes(d);
                const uint32_t below = peers & ((1u << lane) - 1u);
                const uint32_t base = valid ? mycnt[d] : 0u;
                __syncwarp();
                if (valid && below == 0u) mycnt[d] = static_cast<uint16_t>(base + __popc(peers));
                __syncwarp();
                slot[r] = (d << 16) | (base + __popc(below));
            }
        }
        __syncthreads();
        // (b) output position of (warp, digit): digit start + the same digit in earlier warps
        const int sd = tid & (kRadix - 1), sq = tid / kRadix;
        {
            uint32_t run = 0;
#pragma unroll
            for (int i = 0; i < kWarpsPerQuarter; ++i) {
                uint16_t* c = cnt + (sq * kWarpsPerQuarter + i) * kRadix + sd;
                const uint32_t v = *c;
                *c = static_cast<uint16_t>(run);
                run += v;
            }
            s_qs[sq][sd] = run;
        }
        __syncthreads();
        uint32_t digit_excl = 0;                      // digits below this one, within this warp's 32
        if (tid < kRadix) {
            uint32_t tot = 0;
#pragma unroll
            for (int q = 0; q < kQuarters; ++q) {     // quarters: exclusive prefix in place
                const uint32_t v = s_qs[q][tid];
                s_qs[q][tid] = tot;
                tot += v;
            }
            uint32_t incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= static_cast<uint32_t>(o)) incl += y;
            }
            if (lane == 31) s_wt[warp] = incl;
            digit_excl = incl - tot;
        }
        __syncthreads();
        if (tid < kRadix) {
            uint32_t before = digit_excl;
            for (int w = 0; w < static_cast<int>(warp); ++w) before += s_wt[w];
#pragma unroll
            for (int q = 0; q < kQuarters; ++q) s_qs[q][tid] += before;
        }
        __syncthreads();
        {
            const uint32_t add = s_qs[sq][sd];
#pragma unroll
            for (int i = 0; i < kWarpsPerQuarter; ++i) {
                uint16_t* c = cnt + (sq * kWarpsPerQuarter + i) * kRadix + sd;
                *c = static_cast<uint16_t>(*c + add);
            }
        }
        __syncthreads();
        // (c) scatter
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
            if (r < rounds) {
                const int j = w0 + r * 32 + static_cast<int>(lane);
                if (j < w1) {
                    const uint32_t d = slot[r] >> 16;
                    const int pos = mycnt[d] + static_cast<int>(slot[r] & 0xFFFFu);
                    if (own_index_ok(pos, n, a.ws)) dst[pos] = src[j];
                }
            }
        }
        __syncthreads();
        uint16_t* t = src;
        src = dst;
        dst = t;
    }
    }
    // sorted candidate indices are in src

    // ---- 3. capacity K ----
    int K;
    if (a.K_in >= 0) {
        K = a.K_in < n ? a.K_in : n;
    } else {
        K = choose_capacity<kThreads>(a, n, [&](int j) { return key[swz(src[j])]; }, s_wsum, s_bk, s_bK, &s_K);
    }

    // ---- 4. fill: selected in rank order; admitted flags (in the key slots) give the lengths ----
    __syncthreads();
    for (int j = tid; j < n; j += kThreads) {
        const int idx = src[j];
        a.selected[j] = j < K ? idx : -1;
        if (own_index_ok(idx, n, a.ws)) key[swz(idx)] = j < K ? 1u : 0u;
    }
    __syncthreads();
    for (int b = tid; b < B; b += kThreads) {
        int len = 0;
        for (int k = 0; k < N; ++k) len += static_cast<int>(key[swz(b * N + k)]);
        a.lengths[b] = len;
    }
    if (tid == 0) a.K_out[0] = K;
}

// ---------------------------------------------------------------------------
// Pools of 2049 .. 16384 candidates on a cluster of C = 16 blocks (one per SM; 8 where the GPU
// cannot place 16), everything in distributed shared memory.  Block c owns a contiguous range of requests (their survival
// chains and keys) and, after the sort, sorted positions [c * P, (c + 1) * P), P = ceil(n / C).
// Blocks exchange small tables by writing them into every block's shared memory, so that reads
// stay local after each cluster barrier; only the sorted keys themselves cross the cluster.
//   1. survival chain and the 64-bit key (order key << 32 | flat index) of each candidate
//   2. stable LSD radix sort over the cluster: survival lies in [+0, 1], so the two top bits of
//      its order key are always one and 4 passes of 8, 8, 8 and 6 bits cover the rest; per pass
//      each warp ranks its 64 keys by digit (warp ballots), each block hands its per-digit totals to every block,
//      orders its keys by digit locally, then writes runs of equal digits to consecutive
//      positions in the shared memory of the block owning them; two cluster barriers per pass,
//      split so that local work fills their wait
//   3. capacity: fixed-point masses of the block's sorted positions, a block scan, the blocks'
//      totals for the carry, f(K) for the block's K range, the best (f, smallest K) over the
//      cluster
//   4. fill: selected for the block's positions; the admitted set is every key up to the one at
//      sorted position K - 1, so each block counts its own requests' admitted candidates
//      against that one key
// ---------------------------------------------------------------------------
constexpr int kClusterThreads = 1024;
constexpr int kClusterChunk = 2048;                 // keys a block holds (per-block capacity)
constexpr int kClusterWarps = kClusterThreads / 32;
constexpr int kCQuarters = kClusterThreads / kRadix;                 // (digit, quarter) threads
constexpr int kCWarpsPerQuarter = kClusterWarps / kCQuarters;
constexpr size_t kClusterKeyBytes = kClusterChunk * sizeof(unsigned long long);
constexpr size_t kClusterCntBytes = static_cast<size_t>(kClusterWarps) * kRadix * sizeof(uint16_t);
// keys [2][chunk] | digit-ordered staging [chunk] | per-warp counters | survival [chunk] | SPS [chunk]
constexpr size_t kClusterSpsOffset = 3 * kClusterKeyBytes + kClusterCntBytes + kClusterChunk * sizeof(float);
constexpr size_t kClusterSmemBytes = kClusterSpsOffset + kClusterChunk * sizeof(double);
static_assert(kCQuarters * kRadix == kClusterThreads && kCWarpsPerQuarter * kCQuarters == kClusterWarps,
              "digit scan layout");

// Requests [lo, hi) of block c when B requests are split into kCtas contiguous ranges.
template <int kCtas>
__device__ __forceinline__ void cluster_requests(int B, int c, int& lo, int& hi) {
    lo = static_cast<int>((static_cast<long long>(c) * B) / kCtas);
    hi = static_cast<int>((static_cast<long long>(c + 1) * B) / kCtas);
}

// Lanes of the warp whose digit (nbits bits, nbits <= 8) equals this lane's, among the lanes of
// `valid`, one ballot per bit.
__device__ __forceinline__ uint32_t same_digit_lanes_masked(uint32_t d, int nbits, uint32_t valid) {
    uint32_t peers = valid;
#pragma unroll
    for (int bit = 0; bit < 8; ++bit) {
        if (bit < nbits) {
            const uint32_t ones = __ballot_sync(0xFFFFFFFFu, (d >> bit) & 1u);
            peers &= ((d >> bit) & 1u) ? ones : ~ones;
        }
    }
    return peers;
}

// Split cluster barrier: arrive (release: this thread's shared-memory writes, local and remote,
// become visible to every thread that waits), then wait (acquire) for every thread of the cluster.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

template <int kClusterCtas>
__global__ void __launch_bounds__(kClusterThreads, 1) schedule_cluster_kernel(ScheduleArgs a) {
    static_assert(kClusterCtas <= 32 && kClusterCtas * kRadix / 8 <= kClusterThreads,
                  "one lane per block in the exchanges, one thread per 16-byte piece of the totals");
    namespace cg = cooperative_groups;
    constexpr int kWarps = kClusterWarps;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ __align__(16) unsigned char s_dyn[];
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(s_dyn);              // [2][kClusterChunk]
    unsigned long long* stage = keys + 2 * kClusterChunk;                                 // [kClusterChunk]
    uint16_t* cnt = reinterpret_cast<uint16_t*>(s_dyn + 3 * kClusterKeyBytes);            // [kWarps][kRadix]
    float* surv = reinterpret_cast<float*>(s_dyn + 3 * kClusterKeyBytes + kClusterCntBytes);   // [swz(j)]
    double* s_sps = reinterpret_cast<double*>(s_dyn + kClusterSpsOffset);                // this block's K range
    __shared__ __align__(16) uint16_t s_alltot[kClusterCtas][kRadix];   // every block's per-digit totals
    __shared__ uint32_t s_q[kCQuarters][kRadix];                // per-quarter digit counts, then offsets
    __shared__ __align__(16) uint16_t s_tot[kRadix];            // this block's per-digit totals
    __shared__ uint32_t s_pos[kRadix];                          // start of (digit, this block) in the output
    __shared__ uint32_t s_lstart[kRadix];                       // start of the digit in this block's keys
    __shared__ uint32_t s_gsum[kRadix / 32], s_lsum[kRadix / 32];
    __shared__ unsigned long long s_allpart[kClusterCtas];      // mass of every block's sorted positions
    __shared__ unsigned long long s_allbest[kClusterCtas];      // every block's best objective key
    __shared__ int s_allK[kClusterCtas];
    __shared__ unsigned long long s_allT[kClusterCtas];         // every block's key at its best K - 1
    __shared__ unsigned long long s_wsum[kWarps];
    __shared__ unsigned long long s_best[kWarps];
    __shared__ int s_bestK[kWarps];
    __shared__ unsigned long long s_T;                          // key at sorted position K - 1
    __shared__ int s_Kfill;                                     // K, for every thread of the fill
    __shared__ int s_bad;

    const int tid = threadIdx.x;
    const uint32_t lane = lane_id(), warp = warp_id();
    const int c = static_cast<int>(cluster.block_rank());
    const int B = a.B, N = a.N;
    const int n = B * N;
    const int P = (n + kClusterCtas - 1) / kClusterCtas;        // sorted positions per block
    // pos / P as a multiply-high: exact for pos < 2^16 and P <= 2^11 (the error term stays below 1 / P)
    const uint32_t magicP = static_cast<uint32_t>((0x100000000ull + P - 1) / static_cast<unsigned long long>(P));
    int r_lo, r_hi;
    cluster_requests<kClusterCtas>(B, c, r_lo, r_hi);
    const int Kmax = a.K_in >= 0 ? 0 : (a.S < n ? a.S : n);

    // the SPS entries of this block's K range are read in step 3: copied into shared memory now,
    // asynchronously (8-byte pieces: the range may start at an odd entry)
    for (int j = c * P + tid; j < min(Kmax, (c + 1) * P); j += kClusterThreads)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;"
                     :: "r"(smem_u32(s_sps + (j - c * P))), "l"(a.sps + j) : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");

    // ---- 1. survival chain (one thread per request, in row-permuted slots), keys in flat order ----
    int m = (r_hi - r_lo) * N;                                   // keys this block holds now
    const int base = r_lo * N;
    float cin[kClusterChunk / kClusterThreads];                  // loads in flight while counters clear
#pragma unroll
    for (int r = 0; r < kClusterChunk / kClusterThreads; ++r) {
        const int j = tid + r * kClusterThreads;
        cin[r] = j < m ? __ldg(a.c + base + j) : 0.f;
    }
    if (tid == 0) s_bad = 0;
    // this call's status word: cleared by block 0 before the first cluster barrier; every bit is
    // set after it
    if (c == 0 && tid == 0) a.ws->status = 0u;
    for (int i = tid; i < static_cast<int>(kClusterCntBytes / 16); i += kClusterThreads)
        reinterpret_cast<uint4*>(cnt)[i] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int r = 0; r < kClusterChunk / kClusterThreads; ++r) {
        const int j = tid + r * kClusterThreads;
        if (j < m) surv[swz(j)] = cin[r];
    }
    __syncthreads();
    bool bad = false;
    for (int b = tid; b < r_hi - r_lo; b += kClusterThreads) {
        float sv = 1.f;
        for (int k0 = 0; k0 < N; k0 += 8) {                      // eight loads in flight, then the chain
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = k0 + u < N ? surv[swz(b * N + k0 + u)] : 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (k0 + u < N) {
                    const float cp = clamp_prob(v[u], bad);
                    sv = (k0 + u == 0) ? cp : __fmul_rn(sv, cp);
                    v[u] = sv;
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (k0 + u < N) surv[swz(b * N + k0 + u)] = v[u];
        }
    }
    if (bad) s_bad = 1;
    __syncthreads();
    for (int j = tid; j < m; j += kClusterThreads)
        keys[j] = (static_cast<unsigned long long>(order_key(surv[swz(j)])) << 32) | static_cast<unsigned long long>(base + j);
    __syncthreads();

    // ---- 2. stable LSD radix sort over the cluster ----
    int cur = 0;
    // the warp's keys: a contiguous run of one or two rounds of 32, so that every warp ranks keys
    const int rounds = m > 32 * kWarps || (n + kClusterCtas - 1) / kClusterCtas > 32 * kWarps ? 2 : 1;
    const int w0 = static_cast<int>(warp) * 32 * rounds;
    uint16_t* mycnt = cnt + warp * kRadix;
    const int sd = tid & (kRadix - 1), sq = tid / kRadix;        // (digit, quarter) of this thread
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 32 + 8 * pass;
        const int nbits = pass == 3 ? 6 : 8;                     // key bits 62 and 63 never vary
        const uint32_t dmask = (1u << nbits) - 1u;
        uint32_t slot[2];
        unsigned long long kv[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int j = w0 + r * 32 + static_cast<int>(lane);
            kv[r] = r < rounds && j < m ? keys[cur * kClusterChunk + j] : 0ull;
            slot[r] = static_cast<uint32_t>(kv[r] >> shift) & dmask;
        }
        // (a) per-warp digit counts; each key keeps (digit << 16 | offset within the warp's digit)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int live = r < rounds ? min(32, max(0, m - (w0 + r * 32))) : 0;   // lanes with a key
            if (live > 0) {
                const uint32_t vmask = live == 32 ? 0xFFFFFFFFu : ((1u << live) - 1u);
                const bool valid = lane < static_cast<uint32_t>(live);
                const uint32_t d = slot[r];
                const uint32_t peers = same_digit_lanes_masked(d, nbits, vmask);
                const uint32_t below = peers & ((1u << lane) - 1u);
                const uint32_t before = valid ? mycnt[d] : 0u;
                __syncwarp();
                if (valid && below == 0u) mycnt[d] = static_cast<uint16_t>(before + __popc(peers));
                __syncwarp();
                slot[r] = (d << 16) | (before + __popc(below));
            }
        }
        __syncthreads();
        // (b) block totals per digit, from four quarters of the warps; handed to every block
        {
            uint32_t sum = 0;
#pragma unroll
            for (int i = 0; i < kCWarpsPerQuarter; ++i) sum += cnt[(sq * kCWarpsPerQuarter + i) * kRadix + sd];
            s_q[sq][sd] = sum;
        }
        __syncthreads();
        if (tid < kRadix) {
            uint32_t tot = 0;
#pragma unroll
            for (int q = 0; q < kCQuarters; ++q) {                   // quarters: exclusive prefix in place
                const uint32_t v = s_q[q][tid];
                s_q[q][tid] = tot;
                tot += v;
            }
            s_tot[tid] = static_cast<uint16_t>(tot);
            // 16-byte pieces of 8 totals gathered by shuffles: lane l holds piece l & 3 of its warp's
            // 32 digits and sends it to the blocks l >> 2, (l >> 2) + 8, ...
            const uint32_t pair = tot | (__shfl_down_sync(0xFFFFFFFFu, tot, 1) << 16);
            const int src = static_cast<int>(lane & 3u) * 8;
            uint4 piece;
            piece.x = __shfl_sync(0xFFFFFFFFu, pair, src + 0);
            piece.y = __shfl_sync(0xFFFFFFFFu, pair, src + 2);
            piece.z = __shfl_sync(0xFFFFFFFFu, pair, src + 4);
            piece.w = __shfl_sync(0xFFFFFFFFu, pair, src + 6);
#pragma unroll
            for (int cc = static_cast<int>(lane >> 2); cc < kClusterCtas; cc += 8)
                reinterpret_cast<uint4*>(cluster.map_shared_rank(&s_alltot[c][0], cc))[warp * 4 + (lane & 3u)] = piece;
        }
        cluster_arrive();
        __syncthreads();
        {                                                            // counters: exclusive prefix over warps
            uint32_t run = s_q[sq][sd];
#pragma unroll
            for (int i = 0; i < kCWarpsPerQuarter; ++i) {
                uint16_t* cp = cnt + (sq * kCWarpsPerQuarter + i) * kRadix + sd;
                const uint32_t v = *cp;
                *cp = static_cast<uint16_t>(run);
                run += v;
            }
        }
        cluster_wait();
        if (pass == 0 && tid == 0 && s_bad) set_status(a.ws, DSPARK_STATUS_INPUT_RANGE);
        // (c) per digit: start in the output (smaller digits anywhere, then this digit in the
        //     blocks before this one) and start in this block's digit order
        uint32_t all_d = 0, tot_d = 0, incl_g = 0, incl_l = 0;
        if (tid < kRadix) {
            uint32_t mine_before = 0;
#pragma unroll
            for (int cc = 0; cc < kClusterCtas; ++cc) {
                const uint32_t v = s_alltot[cc][tid];
                all_d += v;
                if (cc < c) mine_before += v;
            }
            tot_d = s_tot[tid];
            incl_g = all_d;
            incl_l = tot_d;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t yg = __shfl_up_sync(0xFFFFFFFFu, incl_g, o);
                const uint32_t yl = __shfl_up_sync(0xFFFFFFFFu, incl_l, o);
                if (lane >= static_cast<uint32_t>(o)) {
                    incl_g += yg;
                    incl_l += yl;
                }
            }
            if (lane == 31) {
                s_gsum[warp] = incl_g;
                s_lsum[warp] = incl_l;
            }
            incl_g += mine_before;
        }
        __syncthreads();
        if (tid < kRadix) {
            uint32_t g = 0, l = 0;
            for (int w = 0; w < static_cast<int>(warp); ++w) {
                g += s_gsum[w];
                l += s_lsum[w];
            }
            s_pos[tid] = g + incl_g - all_d;
            s_lstart[tid] = l + incl_l - tot_d;
        }
        __syncthreads();
        // (d) this block's keys in digit order (stable), then each run of a digit written to
        //     consecutive output positions in the block owning them
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int j = w0 + r * 32 + static_cast<int>(lane);
            if (r < rounds && j < m) {
                const uint32_t d = slot[r] >> 16;
                stage[s_lstart[d] + mycnt[d] + (slot[r] & 0xFFFFu)] = kv[r];
            }
        }
        __syncthreads();
        // Two keys of one digit run that land on an even slot and the next one go as one 16-byte
        // store (remote stores cost per request, not per byte); the second key's thread skips.
        unsigned long long* nxt = keys + (cur ^ 1) * kClusterChunk;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int t = tid + r * kClusterThreads;
            if (t < m) {
                const unsigned long long key = stage[t];
                const uint32_t d = static_cast<uint32_t>(key >> shift) & dmask;
                const uint32_t pos = s_pos[d] + static_cast<uint32_t>(t) - s_lstart[d];
                const uint32_t owner = __umulhi(pos, magicP);
                const uint32_t slot_o = pos - owner * static_cast<uint32_t>(P);
                if (!own_index_ok(owner, kClusterCtas, a.ws) || !own_index_ok(slot_o, P, a.ws)) continue;
                unsigned long long* dst = cluster.map_shared_rank(nxt, static_cast<int>(owner)) + slot_o;
                if ((slot_o & 1u) == 0u) {
                    const bool pair = t + 1 < m && slot_o + 1 < static_cast<uint32_t>(P) &&
                                      (static_cast<uint32_t>(stage[t + 1] >> shift) & dmask) == d;
                    if (pair) *reinterpret_cast<ulonglong2*>(dst) = make_ulonglong2(key, stage[t + 1]);
                    else *dst = key;
                } else {
                    const bool second = t > 0 && (static_cast<uint32_t>(stage[t - 1] >> shift) & dmask) == d;
                    if (!second) *dst = key;
                }
            }
        }
        cluster_arrive();
        if (pass < 3)                                            // counters were last read before staging
            for (int i = tid; i < static_cast<int>(kClusterCntBytes / 16); i += kClusterThreads)
                reinterpret_cast<uint4*>(cnt)[i] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
        cluster_wait();                                          // every key landed
        cur ^= 1;
        m = max(0, min(P, n - c * P));
    }
    // this block now holds sorted positions [c * P, c * P + m)
    const unsigned long long* sorted = keys + cur * kClusterChunk;

    // ---- 3. capacity K ----
    int K;
    bool have_T = false;
    if (a.K_in >= 0) {
        K = a.K_in < n ? a.K_in : n;
    } else {
        // kPer consecutive positions per thread (one for 16 blocks, whose share is at most 1024)
        constexpr int kPer = (kSmemMaxCandidates / kClusterCtas + kClusterThreads - 1) / kClusterThreads;
        const int j_lo = c * P, j_hi = min(Kmax, c * P + m);        // this block's K - 1 range
        const int jl0 = kPer * tid;
        asm volatile("cp.async.wait_all;" ::: "memory");            // this thread's SPS pieces landed
        unsigned long long q[kPer];
        unsigned long long sum = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            q[i] = j_lo + jl0 + i < j_hi ? mass32(key_survival(static_cast<uint32_t>(sorted[jl0 + i] >> 32))) : 0ull;
            sum += q[i];
        }
        unsigned long long incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= static_cast<uint32_t>(o)) incl += y;
        }
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();                                              // also: every thread's SPS pieces landed
        if (warp == 0) {
            const unsigned long long v = s_wsum[lane];
            unsigned long long x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= static_cast<uint32_t>(o)) x += y;
            }
            s_wsum[lane] = x - v;                                     // exclusive prefix of the warps
            const unsigned long long total = __shfl_sync(0xFFFFFFFFu, x, 31);
            if (lane < static_cast<uint32_t>(kClusterCtas))          // the block's total mass, to every block
                cluster.map_shared_rank(&s_allpart[c], static_cast<int>(lane))[0] = total;
        }
        cluster.sync();
        // masses of the blocks before this one: one entry per lane and a warp sum in every warp
        // (a loop over the entries in every thread costs more: 32 warps of broadcast loads)
        const unsigned long long before = warp_sum_u64(lane < static_cast<uint32_t>(c) ? s_allpart[lane] : 0ull);
        unsigned long long carry = (static_cast<unsigned long long>(a.B) << 32) + before;
        carry += s_wsum[warp] + incl - sum;                           // masses before this thread's positions
        unsigned long long best = 0ull;
        int bestK = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            carry += q[i];
            if (j_lo + jl0 + i < j_hi) {
                const unsigned long long k = objective_key(carry, s_sps[jl0 + i]);
                if (k > best) { best = k; bestK = j_lo + jl0 + i + 1; }
            }
        }
        warp_best_key(best, bestK);
        if (lane == 0) { s_best[warp] = best; s_bestK[warp] = bestK; }
        __syncthreads();
        if (warp == 0) {
            best = s_best[lane];
            bestK = s_bestK[lane];
            warp_best_key(best, bestK);
            // the block's best with the key at its position K - 1 (local), to every block
            const unsigned long long T = bestK != 0x7FFFFFFF ? sorted[bestK - 1 - j_lo] : 0ull;
            if (lane < static_cast<uint32_t>(kClusterCtas)) {
                cluster.map_shared_rank(&s_allbest[c], static_cast<int>(lane))[0] = best;
                cluster.map_shared_rank(&s_allK[c], static_cast<int>(lane))[0] = bestK;
                cluster.map_shared_rank(&s_allT[c], static_cast<int>(lane))[0] = T;
            }
        }
        cluster.sync();
        // the best over the blocks (one entry per lane) by warp 0; the fill reads K from shared memory
        K = 0;
        if (warp == 0) {
            const unsigned long long mine = lane < static_cast<uint32_t>(kClusterCtas) ? s_allbest[lane] : 0ull;
            const int mineK = lane < static_cast<uint32_t>(kClusterCtas) ? s_allK[lane] : 0x7FFFFFFF;
            unsigned long long bk = mine;
            int bK = mineK;
            warp_best_key(bk, bK);
            const uint32_t holder = __ballot_sync(0xFFFFFFFFu, mine == bk && mineK == bK);
            if (bK == 0x7FFFFFFF) {                                   // every f was NaN or -inf: K = 1, flagged
                if (c == 0 && lane == 0) set_status(a.ws, DSPARK_STATUS_NUMERIC);
                bK = 1;
            } else if (lane == 0) {
                s_T = s_allT[__ffs(holder) - 1];
                have_T = true;
            }
            K = bK;
        }
    }

    // ---- 4. fill ----
    if (tid == 0) {
        s_Kfill = K;
        if (K > 0 && !have_T) {                                       // K fixed, or the flagged K = 1
            const uint32_t last = static_cast<uint32_t>(K - 1);
            const uint32_t owner = __umulhi(last, magicP);
            s_T = cluster.map_shared_rank(keys + cur * kClusterChunk, static_cast<int>(owner))[last - owner * P];
        }
    }
    __syncthreads();
    K = s_Kfill;
    cluster_arrive();                                                 // no remote access after this point
    // global stores only from here on: the release fences of the cluster barriers above never wait
    // for them
    for (int jl = tid; jl < m; jl += kClusterThreads) {
        const int j = c * P + jl;
        a.selected[j] = j < K ? static_cast<int>(sorted[jl] & 0xFFFFFFFFull) : -1;
    }
    // Candidate k of a request is admitted iff its key is at most T.  Survival never grows along a
    // request (each factor is at most one) and equal survivals order by index, so the admitted
    // candidates of a request are a prefix: the thread of its last admitted candidate (or of its
    // first candidate, when none is) writes the length.
    const unsigned long long T = s_T;
    for (int jj = tid; jj < (r_hi - r_lo) * N; jj += kClusterThreads) {
        const float sv = surv[swz(jj)];
        a.survival[base + jj] = sv;
        const int b = jj / N, k = jj - b * N;
        const bool adm = K > 0 && ((static_cast<unsigned long long>(order_key(sv)) << 32) |
                                   static_cast<unsigned long long>(base + jj)) <= T;
        const bool adm_next = k + 1 < N && K > 0 &&
                              ((static_cast<unsigned long long>(order_key(surv[swz(jj + 1)])) << 32) |
                               static_cast<unsigned long long>(base + jj + 1)) <= T;
        if (adm && !adm_next) a.lengths[r_lo + b] = k + 1;
        if (k == 0 && !adm) a.lengths[r_lo + b] = 0;
    }
    if (c == 0 && tid == 0) a.K_out[0] = K;
    cluster_wait();                                                   // no block leaves while another reads it
}

// ---------------------------------------------------------------------------
// Pools above kSmemMaxCandidates: 64-bit keys (order key << 32 | index) in the workspace.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024, 1) schedule_global_kernel(ScheduleArgs a) {
    constexpr int kThreads = 1024;
    constexpr int kWarps = kThreads / 32;
    __shared__ uint32_t s_cnt[kWarps][kRadix];
    __shared__ uint32_t s_base[kRadix];
    __shared__ uint32_t s_tmp[kRadix];
    __shared__ unsigned long long s_wsum[kWarps];
    __shared__ unsigned long long s_bk[kWarps];
    __shared__ int s_bK[kWarps];
    __shared__ int s_K;

    const int tid = threadIdx.x;
    const uint32_t lane = lane_id(), warp = warp_id();
    const int B = a.B, N = a.N;
    const int n = B * N;

    // ---- 1. survival chain and keys ----
    if (tid == 0) a.ws->status = 0u;             // this call's status word, cleared before any bit is set
    __syncthreads();
    bool bad = false;
    for (int b = tid; b < B; b += kThreads) {
        float s = 1.f;
        for (int k = 0; k < N; ++k) {
            const size_t idx = static_cast<size_t>(b) * N + k;
            const float c = clamp_prob(a.c[idx], bad);
            s = (k == 0) ? c : __fmul_rn(s, c);
            a.survival[idx] = s;
            a.keys0[idx] = (static_cast<unsigned long long>(order_key(s)) << 32) | static_cast<unsigned long long>(idx);
        }
        a.lengths[b] = 0;
    }
    if (bad) set_status(a.ws, DSPARK_STATUS_INPUT_RANGE);
    for (int i = tid; i < kWarps * kRadix; i += kThreads) (&s_cnt[0][0])[i] = 0;
    __syncthreads();

    // ---- 2. stable LSD radix sort on the upper 32 bits (rounds of 1024 keys) ----
    unsigned long long* src = a.keys0;
    unsigned long long* dst = a.keys1;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 32 + 8 * pass;
        if (tid < kRadix) s_base[tid] = 0;
        __syncthreads();
        for (int j = tid; j < n; j += kThreads)
            atomicAdd(&s_base[static_cast<uint32_t>(src[j] >> shift) & 0xFFu], 1u);
        __syncthreads();
        uint32_t hv = 0, hincl = 0;
        if (tid < kRadix) {
            hv = s_base[tid];
            hincl = hv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, hincl, o);
                if (lane >= static_cast<uint32_t>(o)) hincl += y;
            }
            s_tmp[tid] = hincl;
        }
        __syncthreads();
        if (tid < kRadix) {
            uint32_t before = 0;
            for (int w = 0; w < static_cast<int>(tid >> 5); ++w) before += s_tmp[w * 32 + 31];
            s_base[tid] = before + hincl - hv;
        }
        __syncthreads();
        for (int r0 = 0; r0 < n; r0 += kThreads) {
            const int j = r0 + tid;
            const bool valid = j < n;
            const unsigned long long k = valid ? src[j] : 0ull;
            const uint32_t d = valid ? (static_cast<uint32_t>(k >> shift) & 0xFFu) : (0x100u | lane);
            const uint32_t peers = same_digit_lanes(d);
            const uint32_t rank = __popc(peers & ((1u << lane) - 1u));
            if (valid && rank == 0) s_cnt[warp][d] = __popc(peers);
            __syncthreads();
            if (tid < kRadix) {
                uint32_t run = s_base[tid];
                for (int w = 0; w < kWarps; ++w) {
                    const uint32_t c = s_cnt[w][tid];
                    s_cnt[w][tid] = run;
                    run += c;
                }
                s_base[tid] = run;
            }
            __syncthreads();
            if (valid) dst[s_cnt[warp][d] + rank] = k;
            __syncthreads();
            for (int i = tid; i < kWarps * kRadix; i += kThreads) (&s_cnt[0][0])[i] = 0;
            __syncthreads();
        }
        unsigned long long* t = src;
        src = dst;
        dst = t;
    }

    // ---- 3. capacity K ----
    int K;
    if (a.K_in >= 0) {
        K = a.K_in < n ? a.K_in : n;
    } else {
        K = choose_capacity<kThreads>(a, n, [&](int j) { return static_cast<uint32_t>(src[j] >> 32); },
                                      s_wsum, s_bk, s_bK, &s_K);
    }

    // ---- 4. fill ----
    for (int j = tid; j < n; j += kThreads) {
        const int idx = static_cast<int>(src[j] & 0xFFFFFFFFull);
        if (j < K) {
            a.selected[j] = idx;
            if (own_index_ok(idx, n, a.ws)) atomicAdd(a.lengths + idx / N, 1);
        } else {
            a.selected[j] = -1;
        }
    }
    if (tid == 0) a.K_out[0] = K;
}

}  // namespace

template <int kCtas>
cudaLaunchConfig_t cluster_config(cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCtas, 1, 1);
    cfg.blockDim = dim3(kClusterThreads, 1, 1);
    cfg.dynamicSmemBytes = kClusterSmemBytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int kCtas>
cudaError_t prepare_cluster_kernel() {
    cudaError_t e = cudaFuncSetAttribute(schedule_cluster_kernel<kCtas>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kClusterSmemBytes));
    if (e == cudaSuccess && kCtas > 8)
        e = cudaFuncSetAttribute(schedule_cluster_kernel<kCtas>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

template <int kCtas>
cudaError_t launch_cluster(const ScheduleArgs& a, cudaStream_t stream) {
    const cudaError_t e = prepare_cluster_kernel<kCtas>();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = cluster_config<kCtas>(stream, attr);
    return cudaLaunchKernelEx(&cfg, schedule_cluster_kernel<kCtas>, a);
}

// Whether the device can place a cluster of 16 of these blocks (16 SMs of one GPU processing
// cluster, each with the block's shared memory), asked once per device.
bool cluster16_fits(int device) {
    static std::mutex mu;
    static int known[64] = {};                                    // 0 unknown, 1 fits, 2 does not
    if (device < 0 || device >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (known[device] == 0) {
        int clusters = 0;
        cudaError_t e = prepare_cluster_kernel<16>();
        if (e == cudaSuccess) {
            cudaLaunchAttribute attr[1];
            const cudaLaunchConfig_t cfg = cluster_config<16>(nullptr, attr);
            e = cudaOccupancyMaxActiveClusters(&clusters, schedule_cluster_kernel<16>, &cfg);
        }
        if (e != cudaSuccess) (void)cudaGetLastError();           // not sticky: fall back to 8
        known[device] = (e == cudaSuccess && clusters >= 1) ? 1 : 2;
    }
    return known[device] == 1;
}

size_t schedule_workspace_bytes(int B, int N) {
    return sizeof(WsHeader) + 2 * sizeof(unsigned long long) * static_cast<size_t>(B) * N;
}

dspark_status launch_schedule(const float* cond_accept, const double* sps, int S, int B, int N,
                              int K_in, float* survival, int32_t* K_out, int32_t* lengths,
                              int32_t* selected, void* ws, cudaStream_t stream, const DeviceInfo& dev) {
    // no separate clear: every schedule kernel zeroes its status word itself before setting a bit
    ScheduleArgs a;
    a.c = cond_accept;
    a.sps = sps;
    a.survival = survival;
    a.K_out = K_out;
    a.lengths = lengths;
    a.selected = selected;
    uint8_t* p = static_cast<uint8_t*>(ws) + sizeof(WsHeader);
    a.keys0 = reinterpret_cast<unsigned long long*>(p);
    a.keys1 = a.keys0 + static_cast<size_t>(B) * N;
    a.ws = static_cast<WsHeader*>(ws);
    a.S = S;
    a.B = B;
    a.N = N;
    a.K_in = K_in;
    const long long n = static_cast<long long>(B) * N;
    if (n <= 32) {
        schedule_warp_kernel<<<1, 32, 0, stream>>>(a);
    } else if (n <= 256) {                    // one block: 256 threads are plenty for small pools
        schedule_smem_kernel<256><<<1, 256, smem_schedule_bytes(static_cast<int>(n), 8), stream>>>(a);
    } else if (n > kBitonicMax && n <= kSmemMaxCandidates &&
               ((B + 7) / 8) * static_cast<long long>(N) <= kClusterChunk) {
        // every block's requests and every block's share of the sorted order fit its key buffers
        const bool wide = ((B + 15) / 16) * static_cast<long long>(N) <= kClusterChunk && cluster16_fits(dev.device);
        const cudaError_t e = wide ? launch_cluster<16>(a, stream) : launch_cluster<8>(a, stream);
        if (e != cudaSuccess) return cuda_error(e, "launch(schedule cluster)");
    } else if (n <= kSmemMaxCandidates) {
        const size_t smem = smem_schedule_bytes(static_cast<int>(n), 32);
        const cudaError_t e = cudaFuncSetAttribute(schedule_smem_kernel<1024>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem_schedule_bytes(kSmemMaxCandidates, 32)));
        if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(schedule)");
        schedule_smem_kernel<1024><<<1, 1024, smem, stream>>>(a);
    } else {
        schedule_global_kernel<<<1, 1024, 0, stream>>>(a);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(schedule)");
    return DSPARK_OK;
}

}  // namespace dspark

// ---------------------------------------------------------------------------
// Allocation-free variant of dspark_schedule.
//
// Some callers cannot hand this library a workspace: a serving loop that must
// never block (cudaMalloc and cudaFree can synchronise with work already queued
// on the device), or a host whose device memory is entirely reserved by another
// allocator (a framework's memory pool), where a fresh allocation would fail.
// For them the scratch that dspark_schedule takes from its workspace lives here
// instead, in one fixed array that every GPU loading the library holds until the
// process exits.  Pools of up to kSmemMaxCandidates candidates sort in shared
// memory, so the only global scratch they use is the workspace header (status
// word and wait bookkeeping); the array is exactly that header.
// ---------------------------------------------------------------------------

namespace dspark {
namespace {

constexpr int kNoAllocMaxCandidates = 16384;                 // B * N limit
static_assert(kNoAllocMaxCandidates <= kSmemMaxCandidates,
              "allocation-free pools must stay on the shared-memory kernels (no global key buffers)");
constexpr size_t kNoAllocScratchBytes = sizeof(WsHeader);

static __device__ __align__(256) unsigned char g_schedule_scratch[kNoAllocScratchBytes];

// The array's device address, looked up once per CUDA context.  A context is named by the
// driver's context id (unique for the life of the process), so a device reset, or another
// context made current on the same device, gets a lookup of its own rather than a stale address.
using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

struct ScratchEntry {
    unsigned long long ctx_id;
    void* addr;
};

constexpr int kScratchEntries = 64;
std::mutex g_scratch_mu;
ScratchEntry g_scratch_cache[kScratchEntries] = {};
int g_scratch_used = 0, g_scratch_next = 0;
PfnCtxGetCurrent g_ctx_get_current = nullptr;
PfnCtxGetId g_ctx_get_id = nullptr;

template <typename F>
bool driver_fn(const char* name, F* out) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
        set_error("driver entry point %s unavailable", name);
        return false;
    }
    *out = reinterpret_cast<F>(fn);
    return true;
}

// Device address of g_schedule_scratch in the current context.
dspark_status schedule_scratch(void** out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_ctx_get_current == nullptr && !driver_fn("cuCtxGetCurrent", &g_ctx_get_current))
        return DSPARK_ERR_UNSUPPORTED;
    if (g_ctx_get_id == nullptr && !driver_fn("cuCtxGetId", &g_ctx_get_id)) return DSPARK_ERR_UNSUPPORTED;
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) {
        set_error("cuCtxGetCurrent failed");
        return DSPARK_ERR_CUDA;
    }
    void* p = nullptr;
    if (ctx == nullptr) {
        // no context yet: the runtime makes the device's primary context current on this lookup
        const cudaError_t e = cudaGetSymbolAddress(&p, g_schedule_scratch);
        if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(schedule scratch)");
        if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
            set_error("no current CUDA context");
            return DSPARK_ERR_CUDA;
        }
    }
    unsigned long long id = 0;
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) {
        set_error("cuCtxGetId failed");
        return DSPARK_ERR_CUDA;
    }
    for (int k = 0; k < g_scratch_used; ++k)
        if (g_scratch_cache[k].ctx_id == id) {
            *out = g_scratch_cache[k].addr;
            return DSPARK_OK;
        }
    if (p == nullptr) {
        const cudaError_t e = cudaGetSymbolAddress(&p, g_schedule_scratch);
        if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(schedule scratch)");
    }
    const int slot = g_scratch_used < kScratchEntries ? g_scratch_used++ : (g_scratch_next++ % kScratchEntries);
    g_scratch_cache[slot] = ScratchEntry{id, p};
    *out = p;
    return DSPARK_OK;
}

}  // namespace
}  // namespace dspark

extern "C" dspark_status dspark_schedule_noalloc(const float* cond_accept, const double* sps, int S, int B,
                                                 int N, int K_in, float* survival, int32_t* K_out,
                                                 int32_t* lengths, int32_t* selected, void* stream) {
    using namespace dspark;
    set_error("%s", "");
    if (!(cond_accept && survival && K_out && lengths && selected)) {
        set_error("schedule_noalloc: null pointer");
        return DSPARK_ERR_INVALID_ARG;
    }
    if (B < 1 || N < 1 || static_cast<long long>(B) * N > kNoAllocMaxCandidates) {
        set_error("schedule_noalloc: B*N must be between 1 and %d (got B=%d N=%d); "
                  "larger pools need dspark_schedule with a workspace", kNoAllocMaxCandidates, B, N);
        return DSPARK_ERR_INVALID_ARG;
    }
    if (K_in < 0 && (sps == nullptr || S < 1)) {
        set_error("schedule_noalloc: choosing K needs an SPS table (S >= 1)");
        return DSPARK_ERR_INVALID_ARG;
    }
    DeviceInfo dev;
    if (!current_device(&dev)) return DSPARK_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const dspark_status st = schedule_scratch(&scratch);
    if (st != DSPARK_OK) return st;
    return launch_schedule(cond_accept, sps, S, B, N, K_in, survival, K_out, lengths, selected, scratch,
                           static_cast<cudaStream_t>(stream), dev);
}
