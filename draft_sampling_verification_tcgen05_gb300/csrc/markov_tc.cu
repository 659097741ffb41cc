// Tensor-core path of the sequential Markov sampler (bf16 Markov head,
// 16 <= B <= 256 requests): the per-step bias markov_w2 . markov_w1[prev]
// ("DSpark implementation and evaluation" §2.2, §3) is a [V, r] x [r, B]
// product of 2*V*r*B FLOP per step -- 5 GFLOP at V=151936, r=256, B=64 --
// which belongs on the 5th-generation tensor cores.
//
// One persistent cooperative kernel for all N steps.  Block c owns vocabulary
// tiles [tile_lo, tile_hi) of 128 entries for the whole call.
//   warp 0        one thread streams, ahead of use and across steps, the w2
//                 tiles of the block (TMA, 128-byte swizzle, kept in L2 with
//                 evict_last) into a shared-memory ring
//   last warp     one thread streams the base-logit tiles [16 requests x 128 v]
//                 (3-D TMA, evict_first) into one ring per epilogue group
//   warp 1        allocates tensor memory; per step one thread issues, for
//                 every local tile, tcgen05.mma (M=128 vocab rows, N=B rounded
//                 to 16, K=16) with A = w2 tile and B = E = w1[prev] (gathered
//                 by the block into a swizzled shared-memory operand), into its
//                 own TMEM columns
//   warps 2..17   epilogue in four groups of four warps (one per TMEM lane
//                 quadrant); group g handles request chunks g, g+4, ...:
//                 pass 1   bias (tcgen05.ld) + base logit -> z = (base + bias)/T,
//                          written back in place (tcgen05.st): TMEM holds the
//                          block's whole [tiles x 128, B] slab of z for the step;
//                          per-request argmax of z -> one real perturbed value
//                          published as the lower bound LB (atomicMax)
//                 pass 2   z from TMEM; per 16-entry noise group one group word
//                          (its top byte bounds the group's largest variate by a
//                          table); only groups whose largest z plus that bound
//                          reaches LB draw exact variates (rare); block argmax ->
//                          one atomicMax per (block, request);
//                          with an lse output, also the block's sum of
//                          exp(z - block max z) per request, merged over the
//                          blocks at the start of the next step
//   last warp     (aux) evaluates the calibrated confidence head of the (request, step) pairs
//                 the block owns, from the previous tokens the step's bias uses
//   then a grid barrier among the step's warps; the producers keep streaming.
// No [B, V] row is written to device memory.
#include "confidence_common.cuh"
#include "device_common.cuh"
#include "host_common.h"
#include "markov_common.cuh"

#include <algorithm>

namespace dspark {
namespace {

using namespace markov;

constexpr int kGroups = 4;
constexpr int kEpiWarps = 4 * kGroups;
constexpr int kLProdWarp = 2 + kEpiWarps;                    // base-logit producer
constexpr int kAuxWarp = 3 + kEpiWarps;                      // last warp: the confidence head
constexpr int kThreadsTC = 32 * (4 + kEpiWarps);
constexpr uint32_t kStepThreads = 32 * (2 + kEpiWarps);      // warps 1 .. 1 + kEpiWarps and the aux warp
constexpr int kW2Stages = 6;                    // upper bound of the w2 ring (the stream from L2 is bound by bytes in flight)
constexpr int kLStages = 3;                      // upper bound per epilogue group; the launcher picks 2 or 3
constexpr int kTileV = 128;
constexpr int kChunk = 16;                       // requests per epilogue chunk
constexpr int kInterleave = 1;                   // tiles whose bias MMAs are issued k-block by k-block together
constexpr int kKbPerStage = 2;                   // 64-wide K blocks of w2 per ring stage
constexpr int kMaxLocalTiles = 32;
constexpr int kZtPitch = 36;                     // floats per request row of the transpose buffer (no bank conflicts)
constexpr uint32_t kW2BoxBytes = kTileV * 128;               // 128 rows x 64 bf16
constexpr uint32_t kW2StageBytes = kKbPerStage * kW2BoxBytes;
constexpr uint32_t kLStageBytes = kTileV * kChunk * 4;       // 16 requests x 128 fp32
constexpr uint32_t kGtabBytes = 256 * 4;                     // bound table of the group words
constexpr uint32_t kBarStep = 1;
constexpr uint32_t kBarGroup0 = 2;
constexpr uint32_t kBarEpi = kBarGroup0 + kGroups;   // all epilogue warps
constexpr uint32_t kWaitProducer = 0x301, kWaitMma = 0x302, kWaitEpi = 0x303;
constexpr size_t kEMaxBytes = 64 * 1024;
constexpr float kLog2eF = 1.4426950408889634f;

struct TcArgs {
    int w2_stages;        // depth of the w2 ring
    int l_stages;         // depth of each base-logit ring
    int B_pad;            // B rounded up to 16 (MMA N)
    int n_tiles;          // ceil(V / 128)
    uint32_t tmem_cols;   // power of two >= max tiles per block * B_pad
};

__device__ __forceinline__ void tile_range(const TcArgs& t, int& lo, int& hi) {
    lo = static_cast<int>((static_cast<long long>(blockIdx.x) * t.n_tiles) / gridDim.x);
    hi = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * t.n_tiles) / gridDim.x);
}

// Stream-0 counter of the two noise groups of local tile `tile` that TMEM lane quadrant `quad`
// holds (rows quad * 32 .. quad * 32 + 31 of the tile: groups 8 tile + 2 quad and + 1).
__device__ __forceinline__ uint32_t group_counter(int tile, uint32_t quad) {
    return static_cast<uint32_t>((tile * kTileV + static_cast<int>(quad * 32u)) >> 6);
}

// Exact candidates of one noise group that the table test could not rule out (rare), drawn by
// the whole warp: one TMEM column load gives lane l the z of row quad * 32 + l for the request,
// so each of the group's 16 lanes (half `gsel` of the warp) tests its own entry.  The group's
// largest variate -log(E_min) is exact for the entry at position p and bounds every other one,
// so an entry is drawn only when z + that variate still reaches lb (the 1e-3 covers the rounding
// of z + g and of logf).  The best key goes to `best_slot`.  Called by the whole warp.
__device__ __forceinline__ void group_candidates(const MarkovArgs& a, int b, int i, uint32_t taddr, int v_row0,
                                                 uint32_t gsel, uint32_t W, float lb, unsigned long long* best_slot) {
    const uint32_t lane = lane_id();
    const float z = __uint_as_float(tmem_ld1(taddr));
    tmem_wait_ld();
    const int v = v_row0 + static_cast<int>(lane);
    const uint32_t k = lane & 15u;
    const float e_min = group_e_min(W);
    const float g_top = -logf(e_min);
    unsigned long long key = 0ull;
    if ((lane >> 4) == gsel && v < a.V && __fadd_rn(__fadd_rn(z, g_top), 1e-3f) >= lb) {
        float g = g_top;
        if (k != (W & 15u)) {
            const uint32_t G = static_cast<uint32_t>(v) >> 4;
            g = draft_gumbel_of_entry(e_min, word_of(philox_at(a.seed, a.offset, (G << 2) | (k >> 2),
                                                               static_cast<uint32_t>(b), kStreamGumbelLo,
                                                               static_cast<uint32_t>(i)), k & 3u));
        }
        const float y = __fadd_rn(z, g);
        if (y == y) key = argmax_key(y, static_cast<uint32_t>(v));
    }
    key = warp_max_u64(key);
    if (lane == 0 && key != 0ull) atomicMax(best_slot, key);
}

// Half h of a tile-chunk seen transposed: the warp holds z for its 32 rows (one per lane) and 16
// requests (r[0..15], from TMEM); afterwards lane (jj = lane >> 2, q = lane & 3) holds z of rows
// 8q..8q+7 for request 8h + jj -- the 8 entries whose noise comes from one Philox counter.
__device__ __forceinline__ void transpose_half(float* zt, const uint32_t (&r)[16], int h, uint32_t lane,
                                               float (&zz)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) zt[j * kZtPitch + static_cast<int>(lane)] = __uint_as_float(r[8 * h + j]);
    __syncwarp();
    const float* src = zt + (lane >> 2) * kZtPitch + 8 * (lane & 3u);
    const float4 a = *reinterpret_cast<const float4*>(src);
    const float4 b = *reinterpret_cast<const float4*>(src + 4);
    __syncwarp();
    zz[0] = a.x; zz[1] = a.y; zz[2] = a.z; zz[3] = a.w;
    zz[4] = b.x; zz[5] = b.y; zz[6] = b.z; zz[7] = b.w;
}

__global__ void __launch_bounds__(kThreadsTC, 1)
markov_tc_kernel(const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmW2k,
                 const __grid_constant__ CUtensorMap tmL, MarkovArgs a, TcArgs t) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* w2s = base;
    uint8_t* Ls = w2s + t.w2_stages * kW2StageBytes;
    // gtab[k]: bound on the largest variate of a noise group whose group word has top byte k
    float* gtab = reinterpret_cast<float*>(Ls + kGroups * t.l_stages * kLStageBytes);
    uint8_t* Es = Ls + kGroups * t.l_stages * kLStageBytes + kGtabBytes;

    __shared__ uint64_t bar_w2_full[kW2Stages], bar_w2_empty[kW2Stages];
    __shared__ uint64_t bar_L_full[kGroups][kLStages], bar_L_empty[kGroups][kLStages];
    __shared__ uint64_t bar_tile[kMaxLocalTiles];
    __shared__ uint32_t s_tmem;
    __shared__ int s_prev[256];
    __shared__ float s_invT[256];
    __shared__ float s_lb[kGroups][kChunk];
    __shared__ uint32_t s_lbv[256];                                    // the step's bounds, as read by the wait
    __shared__ unsigned long long s_part[kGroups][4][kChunk];
    __shared__ unsigned long long s_best[kGroups][kChunk];
    __shared__ float s_zmax[256];                                      // block max of z per request
    __shared__ float s_lsum[kGroups][4][kChunk];                       // per-warp sums of exp(z - zmax)
    __shared__ __align__(16) float s_zt[kEpiWarps][8 * kZtPitch];      // z of 8 requests x 32 rows, transposed
    __shared__ int s_ok;

    const uint32_t warp = warp_id(), lane = lane_id();
    const int Bp = t.B_pad;
    const int n_chunks = Bp / kChunk;
    const int rounds = (n_chunks + kGroups - 1) / kGroups;
    const int kblocks = a.r / 64;
    const int kstages = (kblocks + kKbPerStage - 1) / kKbPerStage;      // ring stages per tile
    const uint32_t e_kb_bytes = static_cast<uint32_t>(Bp) * 128u;
    int tile_lo, tile_hi;
    tile_range(t, tile_lo, tile_hi);
    const int nt = tile_hi - tile_lo;

    // ---------------- set-up ----------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < kW2Stages; ++s) {
            mbar_init(&bar_w2_full[s], 1);
            mbar_init(&bar_w2_empty[s], 1);
        }
        for (int g = 0; g < kGroups; ++g)
            for (int s = 0; s < kLStages; ++s) {
                mbar_init(&bar_L_full[g][s], 1);
                mbar_init(&bar_L_empty[g][s], 128);
            }
        for (int i = 0; i < kMaxLocalTiles; ++i) mbar_init(&bar_tile[i], 1);
        fence_mbarrier_init();
        prefetch_tensormap(&tmW2);
        prefetch_tensormap(&tmW2k);
        prefetch_tensormap(&tmL);
    }
    bool bad_t = false;
    for (int b = threadIdx.x; b < 256; b += kThreadsTC) {
        float inv = 0.f;
        if (b < a.B) {
            float T = a.temperature[b];
            if (!(T >= 0.f) || isinf(T)) {
                bad_t = true;
                T = 0.f;
            }
            inv = T > 0.f ? __frcp_rn(T) : 0.f;          // 0 marks a greedy request
        }
        s_invT[b] = inv;
    }
    if (bad_t) set_status(a.ws, DSPARK_STATUS_NUMERIC);
    // gtab[k][.] bounds the largest variate -log(E_min) of a noise group whose group word has top
    // byte k: that of the largest such word (it increases with the word) plus a margin for logf's
    // rounding; the top bin is capped by the global bound
    for (int k = threadIdx.x; k < 256; k += kThreadsTC) {
        const float g = k == 255 ? kDraftGumbelMax
                                 : -logf(group_e_min((static_cast<uint32_t>(k + 1) << 24) - 1u)) + 1e-3f;
        gtab[k] = g;
    }
    {   // zero E once: padding rows (b >= B) stay zero for the whole call
        uint4* e4 = reinterpret_cast<uint4*>(Es);
        const int n16 = Bp * a.r * 2 / 16;
        for (int k = threadIdx.x; k < n16; k += kThreadsTC) e4[k] = make_uint4(0, 0, 0, 0);
    }
    if (warp == 1) {
        tmem_alloc(&s_tmem, t.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- w2 producer: the block's w2 tiles, every step ----------------
            const uint64_t pol_keep = l2_policy_evict_last();
            int ws = 0;
            uint32_t wph = 0;
            bool ok = true;
            // (in the order the MMA warp consumes them: k-block by k-block across each group
            // of kInterleave tiles)
            for (int i = 0; i < a.N && ok; ++i) {
                for (int t0 = 0; t0 < nt && ok; t0 += kInterleave) {
                    const int gsz = min(kInterleave, nt - t0);
                    for (int ks = 0; ks < kstages && ok; ++ks) {
                        const int nkb = min(kKbPerStage, kblocks - ks * kKbPerStage);
                        for (int u = 0; u < gsz; ++u) {
                            if (!mbar_wait(&bar_w2_empty[ws], wph ^ 1u, a.ws, a.timeout_ns, kWaitProducer)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&bar_w2_full[ws], static_cast<uint32_t>(nkb) * kW2BoxBytes);
                            if (nkb == kKbPerStage) {
                                // one copy of the stage's k-blocks (slabs of 16 KB): a TMA-issuing thread
                                // pays a large fixed cost per copy, so fewer, larger copies stream faster
                                tma_load_3d(w2s + ws * kW2StageBytes, &tmW2k, 0, (tile_lo + t0 + u) * kTileV,
                                            ks * kKbPerStage, &bar_w2_full[ws], pol_keep);
                            } else {
                                for (int j = 0; j < nkb; ++j)
                                    tma_load_2d(w2s + ws * kW2StageBytes + j * kW2BoxBytes, &tmW2, (ks * kKbPerStage + j) * 64,
                                                (tile_lo + t0 + u) * kTileV, &bar_w2_full[ws], pol_keep);
                            }
                            if (++ws == t.w2_stages) { ws = 0; wph ^= 1u; }
                        }
                    }
                }
            }
            if (!ok) {
                // let copies already issued land before the block exits: stages before the
                // ring position were last filled in the current phase, the rest one phase
                // earlier (or never, which reads as complete)
                const long long t0 = global_ns();
                for (int s = 0; s < t.w2_stages; ++s)
                    while (!mbar_try_wait(&bar_w2_full[s], s < ws ? wph : (wph ^ 1u)) &&
                           global_ns() - t0 < a.timeout_ns) {
                    }
            }
        }
    } else if (warp == kLProdWarp) {
        if (lane == 0) {
            // ---------------- logit producer: base-logit tiles for every step ----------------
            const uint64_t pol_stream = l2_policy_evict_first();
            int ls[kGroups];
            uint32_t lph[kGroups];
            for (int g = 0; g < kGroups; ++g) { ls[g] = 0; lph[g] = 0; }
            bool ok = true;
            // (no L2 prefetch a step ahead: w2 must stay L2-resident across steps, and a
            // second step of logits in L2 would push it out)
            for (int i = 0; i < a.N && ok; ++i) {
                for (int ro = 0; ro < rounds && ok; ++ro) {
                    for (int tl = 0; tl < nt && ok; ++tl) {
                        const int v0 = (tile_lo + tl) * kTileV;
                        for (int g = 0; g < kGroups && ok; ++g) {
                            const int c = ro * kGroups + g;
                            if (c >= n_chunks) continue;
                            if (!mbar_wait(&bar_L_empty[g][ls[g]], lph[g] ^ 1u, a.ws, a.timeout_ns, kWaitProducer)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&bar_L_full[g][ls[g]], kLStageBytes);
                            tma_load_3d(Ls + (g * t.l_stages + ls[g]) * kLStageBytes, &tmL, v0, i, c * kChunk,
                                        &bar_L_full[g][ls[g]], pol_stream);
                            if (++ls[g] == t.l_stages) { ls[g] = 0; lph[g] ^= 1u; }
                        }
                    }
                }
            }
            if (!ok) {
                const long long t0 = global_ns();
                for (int g = 0; g < kGroups; ++g)
                    for (int s = 0; s < t.l_stages; ++s)
                        while (!mbar_try_wait(&bar_L_full[g][s], s < ls[g] ? lph[g] : (lph[g] ^ 1u)) &&
                               global_ns() - t0 < a.timeout_ns) {
                        }
            }
        }
    } else {
        // ---------------- MMA warp, epilogue warps, aux warp: the N sequential steps ----------------
        const bool is_aux = warp == static_cast<uint32_t>(kAuxWarp);
        const int stid = is_aux ? static_cast<int>(32 * (1 + kEpiWarps) + lane) : static_cast<int>(threadIdx.x) - 32;
        const bool is_mma = warp == 1;
        const int epi = static_cast<int>(warp) - 2;
        const int grp = epi >= 0 ? epi / 4 : 0;
        const uint32_t quad = warp & 3u;
        const bool grp_lead = epi >= 0 && (epi % 4) == 0;
        int w2st = 0, lsg = 0;
        uint32_t w2ph = 0, lphg = 0;
        bool alive = true, dead = false, nan_seen = false;
        // one MMA covers all B_pad requests: measured on sm_103a, a tcgen05.mma of
        // M=128, K=16 costs about the same time for N=32, 64 or 256, so the widest N wins
        const uint32_t idesc = mma_idesc(128, Bp, false);
        const uint64_t dw2 = sw128_kmajor_desc(smem_u32(w2s));    // ring base (every offset keeps it below 256 KB)
        const uint64_t dE = sw128_kmajor_desc(smem_u32(Es));
        const int chunks16 = a.r / 8;                         // 16-byte pieces of a w1 row

        for (int i = 0; i < a.N && alive; ++i) {
            if (i > 0) finish_lse(a, i - 1, stid, static_cast<int>(kStepThreads));
            // ---- previous tokens, then E = w1[prev] in the swizzled K-major operand layout ----
            for (int b = stid; b < a.B; b += kStepThreads) {
                int p;
                if (i == 0) {
                    p = a.anchor[b];
                    if (p < 0 || p >= a.V) {
                        flag_input_index(a.ws);
                        p = 0;
                    }
                } else {
                    p = slot_token(a, i - 1, b);
                }
                s_prev[b] = p;
            }
            named_bar_sync(kBarStep, kStepThreads);
            // 16-byte cp.async copies: all of a thread's pieces are in flight at once and none
            // passes through registers
            for (int idx = stid; idx < a.B * chunks16; idx += kStepThreads) {
                const int b = idx / chunks16, c16 = idx % chunks16;
                const int kb = c16 >> 3, cc = c16 & 7;
                uint8_t* dst = Es + kb * e_kb_bytes + (b >> 3) * 1024 + (b & 7) * 128 + ((cc ^ (b & 7)) << 4);
                const uint8_t* src = static_cast<const uint8_t*>(a.w1) + (static_cast<size_t>(s_prev[b]) * a.r + c16 * 8) * 2;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
            fence_proxy_async_smem();
            named_bar_sync(kBarStep, kStepThreads);

            if (is_aux) {
                // ---- calibrated confidence head of the (request, step) pairs this block owns: the
                //      hidden row and the embedding of the previous token this step's bias uses ----
                if (a.head.hidden != nullptr) {
                    for (int b0 = 0; b0 < a.B; b0 += 32) {
                        const int bl = b0 + static_cast<int>(lane);
                        const bool mine = bl < a.B && (static_cast<long long>(bl) * a.N + i) % gridDim.x == blockIdx.x;
                        uint32_t m = __ballot_sync(0xFFFFFFFFu, mine);
                        while (m != 0u) {
                            const int b = b0 + __ffs(m) - 1;
                            m &= m - 1u;
                            conf_eval_warp<__nv_bfloat16>(a.head, a.ws, static_cast<size_t>(b) * a.N + i, i,
                                                          static_cast<const __nv_bfloat16*>(a.w1) +
                                                              static_cast<size_t>(s_prev[b]) * a.r,
                                                          a.r, lane);
                        }
                    }
                }
            } else if (is_mma) {
                // ---- bias for every local tile: D[tile] = w2_tile (128 x r) . E^T (r x Bp) ----
                if (lane == 0 && !dead) {
                    tc_fence_after();
                    // the k-blocks of kInterleave tiles alternate, so their accumulation chains
                    // (independent TMEM columns) overlap in the tensor pipe
                    for (int t0 = 0; t0 < nt && !dead; t0 += kInterleave) {
                        const int gsz = min(kInterleave, nt - t0);
                        for (int ks = 0; ks < kstages && !dead; ++ks) {
                            const int nkb = min(kKbPerStage, kblocks - ks * kKbPerStage);
                            for (int u = 0; u < gsz; ++u) {
                                if (!mbar_wait(&bar_w2_full[w2st], w2ph, a.ws, a.timeout_ns, kWaitMma)) {
                                    dead = true;
                                    break;
                                }
                                tc_fence_after();
                                const uint32_t d = tmem + static_cast<uint32_t>((t0 + u) * Bp);
                                // descriptors differ only in the start-address field (address >> 4)
                                const uint64_t da = dw2 + ((static_cast<uint32_t>(w2st) * kW2StageBytes) >> 4);
                                for (int j = 0; j < nkb; ++j) {
                                    const int kb = ks * kKbPerStage + j;
                                    const uint64_t dja = da + (static_cast<uint32_t>(j) * kW2BoxBytes >> 4);
                                    const uint64_t djb = dE + (static_cast<uint32_t>(kb) * e_kb_bytes >> 4);
#pragma unroll
                                    for (int k = 0; k < 4; ++k)
                                        mma_issue<false>(d, dja + 2 * k, djb + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
                                }
                                mma_commit(&bar_w2_empty[w2st]);
                                if (++w2st == t.w2_stages) { w2st = 0; w2ph ^= 1u; }
                            }
                        }
                        if (!dead)
                            for (int u = 0; u < gsz; ++u) mma_commit(&bar_tile[t0 + u]);
                    }
                }
                __syncwarp();
            } else {
                unsigned long long* slot = a.lay.slots + static_cast<size_t>(i) * a.B;
                uint32_t* lbs = a.lay.lb + static_cast<size_t>(i) * a.B;
                const int row_lines = a.r * 2 / 128;                   // 128-byte lines of a w1 row
                // ---- pass 1 over this group's chunks: z = (base + bias) / T into TMEM, argmax of z ----
                for (int ro = 0; ro < rounds; ++ro) {
                    const int c = ro * kGroups + grp;
                    if (c >= n_chunks) continue;                       // uniform over the group
                    float bz[kChunk];
                    int bv[kChunk];
#pragma unroll
                    for (int j = 0; j < kChunk; ++j) { bz[j] = -INFINITY; bv[j] = -1; }
                    for (int tl = 0; tl < nt; ++tl) {
                        const int v = (tile_lo + tl) * kTileV + static_cast<int>(quad * 32 + lane);
                        bool okw = !dead;
                        if (okw) okw = mbar_wait(&bar_tile[tl], static_cast<uint32_t>(i & 1), a.ws, a.timeout_ns, kWaitEpi);
                        if (okw) okw = mbar_wait(&bar_L_full[grp][lsg], lphg, a.ws, a.timeout_ns, kWaitEpi);
                        // lane 0's outcome decides for the warp (a shuffle, not a vote): when it saw
                        // both phases complete the data is there for every lane
                        dead = __shfl_sync(0xFFFFFFFFu, okw ? 0 : 1, 0) != 0;
                        if (!dead) {
                            tc_fence_after();
                            const uint32_t taddr = tmem + ((quad * 32u) << 16) + static_cast<uint32_t>(tl * Bp + c * kChunk);
                            uint32_t r[kChunk];
                            tmem_ld16(taddr, r);
                            tmem_wait_ld();
                            const float* Lt = reinterpret_cast<const float*>(Ls + (grp * t.l_stages + lsg) * kLStageBytes);
#pragma unroll
                            for (int j = 0; j < kChunk; ++j) {
                                const float s = __fadd_rn(Lt[j * kTileV + quad * 32 + lane], __uint_as_float(r[j]));
                                const float inv = s_invT[c * kChunk + j];
                                const float z = inv > 0.f ? __fmul_rn(s, inv) : s;
                                r[j] = __float_as_uint(z);
                                if (z != z) nan_seen = true;
                                if (v < a.V && z > bz[j]) { bz[j] = z; bv[j] = v; }
                            }
                            tmem_st16(taddr, r);
                        }
                        mbar_arrive(&bar_L_empty[grp][lsg]);
                        if (++lsg == t.l_stages) { lsg = 0; lphg ^= 1u; }
                    }
                    if (!dead) tmem_wait_st();
#pragma unroll
                    for (int j = 0; j < kChunk; ++j) {
                        const unsigned long long k = warp_max_u64(bv[j] >= 0 ? argmax_key(bz[j], static_cast<uint32_t>(bv[j])) : 0ull);
                        if (lane == 0) s_part[grp][quad][j] = k;
                    }
                    named_bar_sync(kBarGroup0 + grp, 128);
                    if (grp_lead && lane < kChunk) {
                        // the block's best z, perturbed by its own noise, is a value some element
                        // reaches: publish it as a lower bound of the step's maximum
                        const int b = c * kChunk + static_cast<int>(lane);
                        unsigned long long k = 0;
                        for (int q = 0; q < 4; ++q) k = s_part[grp][q][lane] > k ? s_part[grp][q][lane] : k;
                        if (b < a.B) s_zmax[b] = k != 0ull ? float_from_order_bits(static_cast<uint32_t>(k >> 32)) : -INFINITY;
                        if (b < a.B && k != 0ull) {
                            const uint32_t vb = key_index(k);
                            if (s_invT[b] > 0.f) {
                                const float zb = float_from_order_bits(static_cast<uint32_t>(k >> 32));
                                const float y = __fadd_rn(zb, gumbel_at(a, b, i, static_cast<int>(vb)));
                                atomicMax(lbs + b, float_order_bits(y));
                                atomicMax(slot + b, argmax_key(y, vb));
                            } else {
                                atomicMax(slot + b, k);                 // greedy: argmax of z is the token
                            }
                            // the next step may gather this row: bring it into L2 now
                            for (int l = 0; l < row_lines; ++l)
                                prefetch_l2(static_cast<const uint8_t*>(a.w1) + static_cast<size_t>(vb) * a.r * 2 + 128 * l);
                        }
                    }
                    named_bar_sync(kBarGroup0 + grp, 128);
                }

                // ---- wait (bounded) until every block has published its bounds for this step.  The
                //      bounds are read in the same polls as the count, so pass 2 starts without
                //      another round trip: every published bound is a value some element reaches, so
                //      a read that missed a late bound (or a wait that ran out) only weakens the
                //      pruning, and the result stays exact ----
                named_bar_sync(kBarEpi, 32 * kEpiWarps);
                if (epi == 0) {
                    uint32_t* pub = a.lay.pub + static_cast<size_t>(i) * kPubStride;
                    // release: covers the bounds the group leads published before the named barrier
                    if (lane == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(pub) : "memory");
                    __syncwarp();
                    const long long t0 = global_ns();
                    uint32_t lbv[8];
                    while (true) {
                        const uint32_t cnt = ld_volatile_u32(pub);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int b = static_cast<int>(lane) + 32 * j;
                            lbv[j] = b < a.B ? ld_volatile_u32(lbs + b) : 0u;
                        }
                        const bool stop = cnt >= gridDim.x || aborted(a.ws) || global_ns() - t0 >= a.timeout_ns;
                        if (__any_sync(0xFFFFFFFFu, stop)) break;
                        __nanosleep(32);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int b = static_cast<int>(lane) + 32 * j;
                        if (b < a.B) s_lbv[b] = lbv[j];
                    }
                }
                named_bar_sync(kBarEpi, 32 * kEpiWarps);

                // ---- pass 2 over this group's chunks: noise only where z can still beat the
                //      bound.  One group word per 16 entries bounds the group's largest variate
                //      (a table on its top byte); a group whose largest z plus that bound
                //      reaches LB is drawn exactly by the whole warp (rare) ----
                for (int ro = 0; ro < rounds; ++ro) {
                    const int c = ro * kGroups + grp;
                    if (c >= n_chunks) continue;
                    if (grp_lead && lane < kChunk) {
                        const int b = c * kChunk + static_cast<int>(lane);
                        s_lb[grp][lane] = (b < a.B && s_invT[b] > 0.f) ? float_from_order_bits(s_lbv[b]) : INFINITY;
                        s_best[grp][lane] = 0ull;
                    }
                    named_bar_sync(kBarGroup0 + grp, 128);
                    bool any = false;
#pragma unroll
                    for (int j = 0; j < kChunk; ++j) any |= s_lb[grp][j] < INFINITY;
                    const bool want_lse = a.lse != nullptr;
                    const int jj = static_cast<int>(lane >> 2), q = static_cast<int>(lane & 3u);
                    const int b0 = c * kChunk + jj, b1 = b0 + 8;
                    float ls0 = 0.f, ls1 = 0.f;               // sums of exp(z - block max z)
                    if ((any || want_lse) && !dead) {
                        // lane (jj, q) takes rows 8q..8q+7 of requests jj and 8 + jj; lanes q and
                        // q ^ 1 hold the two halves of one 16-entry noise group, whose group word
                        // bounds every variate of the group.  Lane l draws the stream-0 counter of
                        // the warp's two groups for request l & 15 of the chunk (lanes 16-31 one
                        // tile ahead) and passes the group words to the lanes that hold them.
                        const float lb0 = s_lb[grp][jj], lb1 = s_lb[grp][8 + jj];
                        const float m0 = want_lse && b0 < a.B ? s_zmax[b0] : -INFINITY;
                        const float m1 = want_lse && b1 < a.B ? s_zmax[b1] : -INFINITY;
                        const uint32_t pw = (quad * 2u) & 3u;            // word of the warp's first group
                        const int bsrc = c * kChunk + static_cast<int>(lane & 15u);
                        const bool draw = any && s_lb[grp][lane & 15u] < INFINITY;
                        uint32_t wa = 0, wb = 0;
                        for (int tl = 0; tl < nt; ++tl) {
                            const int v0 = (tile_lo + tl) * kTileV + static_cast<int>(quad * 32) + 8 * q;
                            const uint32_t taddr = tmem + ((quad * 32u) << 16) + static_cast<uint32_t>(tl * Bp + c * kChunk);
                            uint32_t r[kChunk];
                            tmem_ld16(taddr, r);
                            tmem_wait_ld();
                            float z0[8], z1[8];
                            transpose_half(s_zt[epi], r, 0, lane, z0);
                            transpose_half(s_zt[epi], r, 1, lane, z1);
                            if (want_lse) {
#pragma unroll
                                for (int k = 0; k < 8; ++k) {
                                    if (v0 + k < a.V) {
                                        if (m0 > -INFINITY) ls0 += exp2f(__fmul_rn(__fsub_rn(z0[k], m0), kLog2eF));
                                        if (m1 > -INFINITY) ls1 += exp2f(__fmul_rn(__fsub_rn(z1[k], m1), kLog2eF));
                                    }
                                }
                            }
                            if ((tl & 1) == 0) {
                                // one Philox round serves two tiles: lanes 0-15 draw this tile's group
                                // words, lanes 16-31 the next tile's
                                const int td = tl + static_cast<int>(lane >> 4);
                                wa = 0;
                                wb = 0;
                                if (draw && td < nt) {
                                    const uint4 w = philox_at(a.seed, a.offset, group_counter(tile_lo + td, quad),
                                                              static_cast<uint32_t>(bsrc), kStreamGumbel, static_cast<uint32_t>(i));
                                    wa = word_of(w, pw);
                                    wb = word_of(w, pw + 1u);
                                }
                            }
                            const int wo = (tl & 1) ? 16 : 0;
                            const uint32_t a0 = __shfl_sync(0xFFFFFFFFu, wa, wo + jj), c0 = __shfl_sync(0xFFFFFFFFu, wb, wo + jj);
                            const uint32_t a1 = __shfl_sync(0xFFFFFFFFu, wa, wo + 8 + jj), c1 = __shfl_sync(0xFFFFFFFFu, wb, wo + 8 + jj);
                            const uint32_t W0 = (q >> 1) ? c0 : a0, W1 = (q >> 1) ? c1 : a1;
                            // the group's largest z (entries past V left out), from both halves
                            float gm0 = -INFINITY, gm1 = -INFINITY;
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                if (v0 + k < a.V) {
                                    gm0 = fmaxf(gm0, z0[k]);
                                    gm1 = fmaxf(gm1, z1[k]);
                                }
                            }
                            gm0 = fmaxf(gm0, __shfl_xor_sync(0xFFFFFFFFu, gm0, 1));
                            gm1 = fmaxf(gm1, __shfl_xor_sync(0xFFFFFFFFu, gm1, 1));
                            // the table bounds the group's largest variate by the top byte of its word
                            const bool T0 = lb0 < INFINITY && __fadd_rn(gm0, gtab[W0 >> 24]) >= lb0;
                            const bool T1 = lb1 < INFINITY && __fadd_rn(gm1, gtab[W1 >> 24]) >= lb1;
                            // both lanes of a pair know both groups: the even lane reports the first,
                            // the odd lane the second, in one vote; the warp draws them one by one
                            const uint32_t mm = __ballot_sync(0xFFFFFFFFu, (q & 1) ? T1 : T0);
                            uint32_t m0 = mm & 0x55555555u;
                            uint32_t m1 = (mm & 0xAAAAAAAAu) >> 1;
                            const int row0 = (tile_lo + tl) * kTileV + static_cast<int>(quad * 32);
                            while ((m0 | m1) != 0u) {
                                const bool second = m0 == 0u;
                                const int src = __ffs(second ? m1 : m0) - 1;
                                if (second) m1 &= m1 - 1u; else m0 &= m0 - 1u;
                                const int j = (src >> 2) + (second ? 8 : 0);           // request in the chunk
                                const uint32_t Wg = __shfl_sync(0xFFFFFFFFu, second ? W1 : W0, src);
                                group_candidates(a, c * kChunk + j, i, taddr + static_cast<uint32_t>(j), row0,
                                                 static_cast<uint32_t>(src >> 1) & 1u, Wg, s_lb[grp][j], &s_best[grp][j]);
                            }
                        }
                    }
                    if (a.lse != nullptr) {
                        // the four lanes of a request pair, then the four warps of the group (fixed order)
                        ls0 += __shfl_xor_sync(0xFFFFFFFFu, ls0, 1);
                        ls0 += __shfl_xor_sync(0xFFFFFFFFu, ls0, 2);
                        ls1 += __shfl_xor_sync(0xFFFFFFFFu, ls1, 1);
                        ls1 += __shfl_xor_sync(0xFFFFFFFFu, ls1, 2);
                        if (q == 0) {
                            s_lsum[grp][quad][jj] = ls0;
                            s_lsum[grp][quad][8 + jj] = ls1;
                        }
                    }
                    named_bar_sync(kBarGroup0 + grp, 128);
                    if (grp_lead && lane < kChunk) {
                        const int b = c * kChunk + static_cast<int>(lane);
                        if (a.lse != nullptr && b < a.B) {
                            const float S = ((s_lsum[grp][0][lane] + s_lsum[grp][1][lane]) + s_lsum[grp][2][lane]) +
                                            s_lsum[grp][3][lane];
                            a.lay.lse_part[(static_cast<size_t>(i & 1) * kMaxGrid + blockIdx.x) * a.B + b] =
                                make_float2(s_zmax[b], s_zmax[b] > -INFINITY ? S : 0.f);
                        }
                        const unsigned long long k = s_best[grp][lane];
                        if (b < a.B && k != 0ull) {
                            atomicMax(slot + b, k);
                            const uint32_t vb = key_index(k);
                            for (int l = 0; l < row_lines; ++l)
                                prefetch_l2(static_cast<const uint8_t*>(a.w1) + static_cast<size_t>(vb) * a.r * 2 + 128 * l);
                        }
                    }
                }
            }
            // ---- every block agrees on the step's winners ----
            tc_fence_before();
            alive = grid_barrier_named(a.ws, static_cast<uint32_t>(i), a.timeout_ns, kWaitStep + i, kBarStep,
                                       kStepThreads, threadIdx.x == 32, &s_ok);
            tc_fence_after();
        }
        if (nan_seen) set_status(a.ws, DSPARK_STATUS_NUMERIC);
        if (alive) finish_lse(a, a.N - 1, stid, static_cast<int>(kStepThreads));
        if (alive && blockIdx.x == 0) {
            for (int idx = stid; idx < a.B * a.N; idx += kStepThreads) {
                const int b = idx / a.N, i = idx % a.N;
                a.tokens[idx] = output_token(a, slot_token(a, i, b));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, t.tmem_cols);
    }
}

// Ring depths: the w2 ring gets what the E operand leaves (the w2 stream from L2 is bound by the
// bytes in flight, and a deeper ring lets the next step's first tiles land during pass 2).
void tc_rings(int B_pad, int r, int* w2_stages, int* l_stages) {
    const bool small_e = static_cast<size_t>(B_pad) * r * 2 <= 32 * 1024;
    *w2_stages = (small_e ? 6 : 4) / kKbPerStage;
    *l_stages = 2;
}

size_t tc_smem_bytes(int B_pad, int r) {
    int w2s, ls;
    tc_rings(B_pad, r, &w2s, &ls);
    return 1024 + static_cast<size_t>(w2s) * kW2StageBytes + static_cast<size_t>(kGroups) * ls * kLStageBytes +
           kGtabBytes + static_cast<size_t>(B_pad) * r * 2;
}

}  // namespace

bool markov_tc_eligible(int B, int N, int V, int r, dspark_dtype wdtype, const float* base, const float* lse,
                        int sm_count) {
    (void)lse;
    if (wdtype != DSPARK_BF16) return false;
    if (B < 16 || B > 256 || r % 64 != 0 || r > 256 || V % 4 != 0 || V < kTileV || V >= (1 << 27))
        return false;
    if (N > 65535 || !aligned(base, 16)) return false;
    const int B_pad = (B + 15) & ~15;
    if (static_cast<size_t>(B_pad) * r * 2 > kEMaxBytes) return false;
    const int n_tiles = (V + kTileV - 1) / kTileV;
    const int grid = std::min(sm_count, n_tiles);
    const int max_local = (n_tiles + grid - 1) / grid;
    return max_local <= kMaxLocalTiles && max_local * B_pad <= 512;
}

dspark_status launch_markov_tc(const MarkovArgs& a, cudaStream_t stream, const DeviceInfo& dev) {
    TcArgs t;
    t.B_pad = (a.B + 15) & ~15;
    tc_rings(t.B_pad, a.r, &t.w2_stages, &t.l_stages);
    t.n_tiles = (a.V + kTileV - 1) / kTileV;
    const int grid = std::min(dev.sm_count, t.n_tiles);
    const int max_local = (t.n_tiles + grid - 1) / grid;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(max_local * t.B_pad)) cols *= 2;
    t.tmem_cols = cols;

    CUtensorMap tmW2, tmW2k, tmL;
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(a.r), static_cast<uint64_t>(a.V)};
        const uint64_t strides[1] = {static_cast<uint64_t>(a.r) * 2};
        const uint32_t box[2] = {64, static_cast<uint32_t>(kTileV)};
        if (!make_tensor_map(&tmW2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.w2, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
            return DSPARK_ERR_UNSUPPORTED;
    }
    {
        // w2 seen as (64 elements of a k-block, row, k-block): a box of (64, 128, kKbPerStage) is one
        // ring stage, landing as kKbPerStage slabs of 128 rows x 128 bytes in the swizzled layout
        const uint64_t dims[3] = {64, static_cast<uint64_t>(a.V), static_cast<uint64_t>(a.r / 64)};
        const uint64_t strides[2] = {static_cast<uint64_t>(a.r) * 2, 128};
        const uint32_t box[3] = {64, static_cast<uint32_t>(kTileV), static_cast<uint32_t>(std::min(kKbPerStage, a.r / 64))};
        if (!make_tensor_map(&tmW2k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.w2, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
            return DSPARK_ERR_UNSUPPORTED;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(a.V), static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.B)};
        const uint64_t strides[2] = {static_cast<uint64_t>(a.V) * 4, static_cast<uint64_t>(a.N) * a.V * 4};
        const uint32_t box[3] = {static_cast<uint32_t>(kTileV), 1, static_cast<uint32_t>(kChunk)};
        if (!make_tensor_map(&tmL, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.base, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_NONE))
            return DSPARK_ERR_UNSUPPORTED;
    }
    const size_t smem = tc_smem_bytes(t.B_pad, a.r);
    if (smem > dev.smem_optin) {
        set_error("markov_sample (tensor path): needs %zu bytes of shared memory", smem);
        return DSPARK_ERR_UNSUPPORTED;
    }
    cudaError_t e = cudaFuncSetAttribute(markov_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(markov_tc)");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, markov_tc_kernel, kThreadsTC, smem);
    if (e != cudaSuccess) return cuda_error(e, "occupancy(markov_tc)");
    if (per_sm < 1 || per_sm * dev.sm_count < grid) {
        set_error("markov_sample (tensor path): %d blocks cannot be co-resident", grid);
        return DSPARK_ERR_UNSUPPORTED;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsTC);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, markov_tc_kernel, tmW2, tmW2k, tmL, a, t);
    if (e != cudaSuccess) return cuda_error(e, "launch(markov_tc)");
    return DSPARK_OK;
}

}  // namespace dspark
