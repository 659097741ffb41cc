// Confidence-scheduled admission of draft tokens, one block.
//
// "Speculative decoding: from zero to DSpark" §6: conditional acceptance
// probabilities are chained into survival probabilities; all candidates of all
// requests are pooled, sorted by survival and admitted from the top; the
// verify capacity maximises expected tokens x SPS(batch size).  §7: the SPS
// curve is jagged, so every K is evaluated; K may also be fixed ahead of time
// and only the fill done now.  No token value is read at any point.
//
// Steps (one block of 1024 threads, 256 for pools of at most 256 candidates):
//   1. survival chain per request (fp32, round to nearest, no contraction)
//      and 64-bit keys ((~survival bits) << 32 | b*N+k), in index order
//   2. stable LSD radix sort of the keys on their upper 32 bits (4 passes of
//      8 bits; rounds of 1024 keys ranked with warp match + per-warp digit
//      counts), ping-ponging between two workspace buffers (L2-resident);
//      pools of at most 1024 candidates are ranked by counting, in shared memory
//   3. if K is to be chosen: block-wide prefix sum of floor(s * 2^32) over the
//      sorted order, f(K) = float64(B * 2^32 + prefix) * SPS[K-1] for every K,
//      block argmax with ties to the smallest K
//   4. fill: the first K sorted candidates are admitted; lengths by counting.
#include "device_common.cuh"
#include "host_common.h"

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

// Exclusive block scan of one u64 per thread; returns the exclusive prefix, *total the sum.
__device__ unsigned long long block_excl_scan_u64(unsigned long long x, unsigned long long* sm,
                                                  unsigned long long* total) {
    const uint32_t lane = lane_id(), warp = warp_id();
    unsigned long long incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= static_cast<uint32_t>(o)) incl += y;
    }
    __syncthreads();
    if (lane == 31) sm[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        unsigned long long w = lane < blockDim.x / 32 ? sm[lane] : 0ull;
        unsigned long long wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= static_cast<uint32_t>(o)) wi += y;
        }
        sm[lane] = wi - w;                 // exclusive prefix of warp totals
        if (lane == 31) sm[32] = wi;
    }
    __syncthreads();
    *total = sm[32];
    return sm[warp] + incl - x;
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads, 1) schedule_kernel(ScheduleArgs a) {
    constexpr int kWarps = kThreads / 32;
    __shared__ uint32_t s_cnt[kWarps][kRadix];
    __shared__ uint32_t s_base[kRadix];
    __shared__ uint32_t s_tmp[kRadix];
    __shared__ unsigned long long s_scan[33];                 // 32 warp slots + total
    __shared__ double s_bf[kWarps];
    __shared__ int s_bk[kWarps];
    __shared__ int s_K;

    const int tid = threadIdx.x;
    const uint32_t lane = lane_id(), warp = warp_id();
    const int B = a.B, N = a.N;
    const int n = B * N;

    // ---- 1. survival chain and keys (small pools keep their keys in shared memory) ----
    const bool small = n <= kThreads;
    unsigned long long* sk = reinterpret_cast<unsigned long long*>(&s_cnt[0][0]);   // [2][kThreads] when small
    unsigned long long* keys = small ? sk : a.keys0;
    bool bad = false;
    for (int b = tid; b < B; b += kThreads) {
        float s = 1.f;
        for (int k = 0; k < N; ++k) {
            const size_t idx = static_cast<size_t>(b) * N + k;
            const float c = clamp_prob(a.c[idx], bad);
            s = (k == 0) ? c : __fmul_rn(s, c);
            a.survival[idx] = s;
            keys[idx] = (static_cast<unsigned long long>(0xFFFFFFFFu - __float_as_uint(s)) << 32) |
                        static_cast<unsigned long long>(idx);
        }
        a.lengths[b] = 0;
    }
    if (bad) set_status(a.ws, DSPARK_STATUS_INPUT_RANGE);
    if (!small)
        for (int i = tid; i < kWarps * kRadix; i += kThreads) (&s_cnt[0][0])[i] = 0;
    __syncthreads();

    // ---- 2. sort: keys are unique (the index is part of the key) ----
    unsigned long long* src = a.keys0;
    unsigned long long* dst = a.keys1;
    if (small) {
        // rank of each key = number of smaller keys (one key per thread), all in shared memory
        const unsigned long long mine = tid < n ? sk[tid] : 0ull;
        if (tid < n) {
            int rank = 0;
            for (int j = 0; j < n; ++j) rank += sk[j] < mine ? 1 : 0;
            sk[kThreads + rank] = mine;
        }
        __syncthreads();
        src = sk + kThreads;
    }
    for (int pass = 0; pass < (small ? 0 : 4); ++pass) {
        const int shift = 32 + 8 * pass;
        if (tid < kRadix) s_base[tid] = 0;
        __syncthreads();
        for (int j = tid; j < n; j += kThreads)
            atomicAdd(&s_base[static_cast<uint32_t>(src[j] >> shift) & 0xFFu], 1u);
        __syncthreads();
        // exclusive scan of the 256-bin histogram (8 warps, then warp totals)
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
            const unsigned long long key = valid ? src[j] : 0ull;
            const uint32_t d = valid ? (static_cast<uint32_t>(key >> shift) & 0xFFu) : (0x100u | lane);
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d);
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
            if (valid) dst[s_cnt[warp][d] + rank] = key;
            __syncthreads();
            for (int i = tid; i < kWarps * kRadix; i += kThreads) (&s_cnt[0][0])[i] = 0;
            __syncthreads();
        }
        unsigned long long* t = src;
        src = dst;
        dst = t;
    }
    // sorted keys are in src (keys0 after the 4 radix passes, shared memory after the rank sort)

    // ---- 3. capacity K ----
    if (a.K_in >= 0) {
        if (tid == 0) s_K = a.K_in < n ? a.K_in : n;
    } else {
        const int Kmax = a.S < n ? a.S : n;
        const int per = (Kmax + kThreads - 1) / kThreads;
        const int j0 = tid * per, j1 = min(Kmax, j0 + per);
        unsigned long long mine = 0;
        for (int j = j0; j < j1; ++j) {
            const float s = __uint_as_float(0xFFFFFFFFu - static_cast<uint32_t>(src[j] >> 32));
            mine += __double2ull_rz(static_cast<double>(s) * 4294967296.0);
        }
        unsigned long long total;
        unsigned long long prefix = block_excl_scan_u64(mine, s_scan, &total);
        double best_f = -INFINITY;
        int best_K = 0x7FFFFFFF;
        const unsigned long long base = static_cast<unsigned long long>(a.B) << 32;
        for (int j = j0; j < j1; ++j) {
            const float s = __uint_as_float(0xFFFFFFFFu - static_cast<uint32_t>(src[j] >> 32));
            prefix += __double2ull_rz(static_cast<double>(s) * 4294967296.0);
            const double f = __dmul_rn(static_cast<double>(base + prefix), a.sps[j]);
            if (f > best_f) { best_f = f; best_K = j + 1; }      // ascending K: strict keeps smallest
        }
        // block argmax (larger f, then smaller K)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const double of = __shfl_xor_sync(0xFFFFFFFFu, best_f, o);
            const int ok = __shfl_xor_sync(0xFFFFFFFFu, best_K, o);
            if (of > best_f || (of == best_f && ok < best_K)) { best_f = of; best_K = ok; }
        }
        if (lane == 0) { s_bf[warp] = best_f; s_bk[warp] = best_K; }
        __syncthreads();
        if (tid == 0) {
            double bf = s_bf[0];
            int bk = s_bk[0];
            for (int w = 1; w < kWarps; ++w)
                if (s_bf[w] > bf || (s_bf[w] == bf && s_bk[w] < bk)) { bf = s_bf[w]; bk = s_bk[w]; }
            if (bk == 0x7FFFFFFF) {          // every f was NaN
                set_status(a.ws, DSPARK_STATUS_NUMERIC);
                bk = 1;
            }
            s_K = bk;
        }
    }
    __syncthreads();
    const int K = s_K;

    // ---- 4. fill ----
    for (int j = tid; j < n; j += kThreads) {
        const int idx = static_cast<int>(src[j] & 0xFFFFFFFFull);
        if (j < K) {
            a.selected[j] = idx;
            atomicAdd(a.lengths + idx / N, 1);
        } else {
            a.selected[j] = -1;
        }
    }
    if (tid == 0) a.K_out[0] = K;
}

}  // namespace

size_t schedule_workspace_bytes(int B, int N) {
    return sizeof(WsHeader) + 2 * sizeof(unsigned long long) * static_cast<size_t>(B) * N;
}

dspark_status launch_schedule(const float* cond_accept, const double* sps, int S, int B, int N,
                              int K_in, float* survival, int32_t* K_out, int32_t* lengths,
                              int32_t* selected, void* ws, cudaStream_t stream, const DeviceInfo& dev) {
    (void)dev;
    dspark_status st = clear_workspace(ws, sizeof(WsHeader), stream);
    if (st != DSPARK_OK) return st;
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
    // one block: 256 threads are plenty for pools of up to 256 candidates
    if (static_cast<long long>(B) * N <= 256)
        schedule_kernel<256><<<1, 256, 0, stream>>>(a);
    else
        schedule_kernel<1024><<<1, 1024, 0, stream>>>(a);
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
// For them the scratch that dspark_schedule takes from its workspace (a status
// header and two radix-sort key buffers) lives here instead, in one fixed array
// that every GPU loading the library holds until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace dspark {
namespace {

constexpr int kNoAllocMaxCandidates = 16384;                 // B * N limit
constexpr size_t kNoAllocScratchBytes =
    sizeof(WsHeader) + 2 * sizeof(unsigned long long) * static_cast<size_t>(kNoAllocMaxCandidates);

static __device__ __align__(256) unsigned char g_schedule_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {};

// Device address of g_schedule_scratch on the current device, looked up once per device.
dspark_status schedule_scratch(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) {
        set_error("device index %d out of range", dev);
        return DSPARK_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_schedule_scratch);
        if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(schedule scratch)");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
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
