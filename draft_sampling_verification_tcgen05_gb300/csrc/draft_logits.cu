// Base logits of the draft LM head on the 5th-generation tensor cores.
//
// "DSpark implementation and evaluation" §2.2 / §4: compute_draft_logits runs
// every drafted position of every request through the LM head in one
// contraction, logits[m, v] = sum_h hidden[m, h] * lm_head[v, h].
//
// Design (sm_103a): a persistent, warp-specialised tcgen05 GEMM.
//   warp 0      one thread issues TMA loads of 128-byte K slices of both
//               operands (128-byte swizzle) into a ring of shared-memory stages
//               (one slice per stage; four or two adjacent slices per stage in
//               the decode shapes)
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma
//               (M = 128, N = BN, K = 16 for bf16 / 8 for tf32) into one of two
//               fp32 accumulators in TMEM and commits each stage back to the
//               producer and each finished tile to the epilogue
//   warps 2-5   read the accumulator with tcgen05.ld (one TMEM lane quadrant
//               per warp) and write fp32 logits
// Two shapes:
//   M <= 256 (decode: a few requests x N positions): "swap" -- A = lm_head rows
//     (128 vocabulary entries per tile), B = all M hidden rows padded to BN;
//     the kernel streams lm_head once from HBM (memory bound).
//   M > 256 (batched drafting): 256 x 256 output tiles on a CTA pair
//     (tcgen05.mma.cta_group::2, gemm_pair_kernel below) for bf16 inputs, 128 x 256
//     tiles on one CTA for fp32 (tf32) inputs; tiles ordered so that the tiles
//     sharing an lm_head slice run together and re-read it from L2 (tensor bound).
#include "device_common.cuh"
#include "host_common.h"

#include <algorithm>

namespace dspark {
namespace {

constexpr int kTileA = 128;          // accumulator rows = MMA M
constexpr int kRowBytes = 128;       // one swizzle row: 64 bf16 or 32 fp32 of K per stage
constexpr int kThreads = 192;
constexpr uint32_t kWaitProducer = 0x101, kWaitMma = 0x102, kWaitEpilogue = 0x103;

struct GemmArgs {
    float* out;
    int M, V, H;
    int swap;
    int tiles_a, tiles_b, k_blocks;
    WsHeader* ws;
    long long timeout_ns;
};

// A stage holds kSlices adjacent 128-byte K slices of both operands, the A slices copied back to
// back, so the memory-bound decode shapes read each lm_head row in runs of kSlices x 128 bytes.
// Measured on the decode GEMM (M = 8 and M = 24, H = 4096, V = 151936): four slices in three
// 72 KB stages (BN = 16) and two in five 40 KB stages (BN = 32) run about 2 us (1 %) faster than
// one slice in ten or nine stages; four slices at BN = 32 leave two stages and run slower.
template <int BN>
constexpr int slices_for() { return BN <= 16 ? 4 : BN <= 32 ? 2 : 1; }

template <int BN>
struct GemmCfg {
    static constexpr int kSlices = slices_for<BN>();
    static constexpr uint32_t kSliceBytes = (kTileA + BN) * kRowBytes;
    static constexpr uint32_t kStageBytes = kSlices * kSliceBytes;
    static constexpr int kStages = std::min<int>(12, (kSlices == 1 ? 192 * 1024 : 216 * 1024) / kStageBytes);
    static constexpr uint32_t kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
};

template <int BN>
struct GemmSmem {
    alignas(1024) uint8_t a[GemmCfg<BN>::kStages][GemmCfg<BN>::kSlices][kTileA * kRowBytes];
    alignas(1024) uint8_t b[GemmCfg<BN>::kStages][GemmCfg<BN>::kSlices][BN * kRowBytes];
    uint64_t full[GemmCfg<BN>::kStages];
    uint64_t empty[GemmCfg<BN>::kStages];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
};

template <int BN, bool kTF32>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    GemmArgs p) {
    using Cfg = GemmCfg<BN>;
    using Smem = GemmSmem<BN>;
    constexpr int kStages = Cfg::kStages;
    constexpr int kSlices = Cfg::kSlices;
    constexpr int kKElems = kTF32 ? 32 : 64;                 // K elements per slice
    constexpr int kMmaK = kTF32 ? 8 : 16;                    // K per MMA instruction
    constexpr int kMmaPerSlice = kKElems / kMmaK;            // 4
    constexpr uint32_t kIdesc = mma_idesc(kTileA, BN, kTF32);

    extern __shared__ uint8_t smem_raw[];
    Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
    const uint32_t warp = warp_id(), lane = lane_id();
    const int total = p.tiles_a * p.tiles_b;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tmem_full[i], 1);
            mbar_init(&s.tmem_empty[i], 128);
        }
        mbar_init(&s.drain, 1);
        fence_mbarrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(&s.tmem_base, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            const uint64_t keep = l2_policy_evict_last();
            const uint64_t stream_once = l2_policy_evict_first();
            // swap: A = lm_head (read once), B = hidden (reused by every tile)
            const uint64_t pol_a = p.swap ? stream_once : keep;
            const uint64_t pol_b = p.swap ? keep : keep;
            uint32_t issued_parity[kStages];
            bool issued[kStages];
            for (int i = 0; i < kStages; ++i) { issued[i] = false; issued_parity[i] = 0; }
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
                const int a_tile = t % p.tiles_a, b_tile = t / p.tiles_a;
                for (int kb = 0; kb < p.k_blocks; kb += kSlices) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1u, p.ws, p.timeout_ns, kWaitProducer)) {
                        ok = false;
                        break;
                    }
                    const int ns = p.k_blocks - kb < kSlices ? p.k_blocks - kb : kSlices;
                    mbar_arrive_expect_tx(&s.full[stage], static_cast<uint32_t>(ns) * Cfg::kSliceBytes);
                    for (int j = 0; j < ns; ++j)
                        tma_load_2d(s.a[stage][j], &tmA, (kb + j) * kKElems, a_tile * kTileA, &s.full[stage], pol_a);
                    for (int j = 0; j < ns; ++j)
                        tma_load_2d(s.b[stage][j], &tmB, (kb + j) * kKElems, b_tile * BN, &s.full[stage], pol_b);
                    issued[stage] = true;
                    issued_parity[stage] = phase;
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // give copies already in flight time to land before the block exits
                for (int i = 0; i < kStages; ++i) {
                    if (!issued[i]) continue;
                    const long long t0 = global_ns();
                    while (!mbar_try_wait(&s.full[i], issued_parity[i]) &&
                           global_ns() - t0 < p.timeout_ns) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
                if (!mbar_wait(&s.tmem_empty[acc], acc_phase ^ 1u, p.ws, p.timeout_ns, kWaitMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < p.k_blocks; kb += kSlices) {
                    if (!mbar_wait(&s.full[stage], phase, p.ws, p.timeout_ns, kWaitMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int ns = p.k_blocks - kb < kSlices ? p.k_blocks - kb : kSlices;
                    for (int j = 0; j < ns; ++j) {
                        const uint32_t a_addr = smem_u32(s.a[stage][j]);
                        const uint32_t b_addr = smem_u32(s.b[stage][j]);
#pragma unroll
                        for (int k = 0; k < kMmaPerSlice; ++k) {
                            const uint64_t adesc = sw128_kmajor_desc(a_addr + k * 32);
                            const uint64_t bdesc = sw128_kmajor_desc(b_addr + k * 32);
                            mma_issue<kTF32>(d_tmem, adesc, bdesc, kIdesc, (kb | j | k) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(&s.empty[stage]);          // stage reusable once these MMAs finish
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(&s.tmem_full[acc]);            // accumulator complete
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // wait until every MMA this thread issued has completed
            mma_commit(&s.drain);
            const long long t0 = global_ns();
            while (!mbar_try_wait(&s.drain, 0) && global_ns() - t0 < p.timeout_ns) {
            }
        }
    } else {
        // ---------------- epilogue: warps 2..5 ----------------
        const uint32_t quad = warp & 3u;                  // TMEM lanes this warp may access
        const uint32_t row = quad * 32u + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const int a_tile = t % p.tiles_a, b_tile = t / p.tiles_a;
            // every lane waits; the vote keeps the warp converged for the .sync.aligned loads
            const bool ready = mbar_wait(&s.tmem_full[acc], acc_phase, p.ws, p.timeout_ns, kWaitEpilogue);
            if (!__all_sync(0xFFFFFFFFu, ready)) break;
            tc_fence_after();
            const int a_row = a_tile * kTileA + static_cast<int>(row);
            const uint32_t taddr = tmem_base + ((quad * 32u) << 16) + static_cast<uint32_t>(acc * BN);
            if (p.swap) {
                // accumulator row = vocabulary entry v, column = hidden row m
                const int v = a_row;
                for (int c0 = 0; c0 < BN && c0 < p.M; c0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(taddr + c0, r);
                    tmem_wait_ld();
                    if (v < p.V) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int m = c0 + j;
                            if (m < p.M) p.out[static_cast<size_t>(m) * p.V + v] = __uint_as_float(r[j]);
                        }
                    }
                }
            } else {
                // accumulator row = hidden row m, column = vocabulary entry v
                const int m = a_row;
                float* orow = p.out + static_cast<size_t>(m) * p.V;
                const bool vec = (p.V & 3) == 0;
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(taddr + c0, r);
                    tmem_wait_ld();
                    const int v0 = b_tile * BN + c0;
                    if (m < p.M) {
                        if (vec && v0 + 16 <= p.V) {
#pragma unroll
                            for (int j = 0; j < 16; j += 4) {
                                *reinterpret_cast<float4*>(orow + v0 + j) =
                                    make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                                __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (v0 + j < p.V) orow[v0 + j] = __uint_as_float(r[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&s.tmem_empty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// CTA-pair variant for the batched bf16 shape.  Two CTAs of a cluster share
// one 256 x 256 output tile: each holds 128 hidden rows (its half of M) and
// 128 lm_head rows (its half of N) per stage, and the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), which reads A and B
// from both CTAs' shared memory and writes each CTA's 128 accumulator rows
// into its own tensor memory.  A stage is 32 KB per CTA instead of 48 KB for
// a 128 x 256 tile, so six stages fit: the ring covers the operand latency,
// and each CTA moves 2/3 of the bytes per output element.
// ---------------------------------------------------------------------------
constexpr int kStages2 = 6;
constexpr int kTile2 = 256;                                    // pair tile: M and N
constexpr uint32_t kHalfBytes2 = 128 * kRowBytes;              // one operand half per CTA
constexpr uint32_t kTmemCols2 = 2 * kTile2;                    // two accumulators

struct Gemm2Smem {
    alignas(1024) uint8_t a[kStages2][128 * kRowBytes];
    alignas(1024) uint8_t b[kStages2][128 * kRowBytes];
    uint64_t full[kStages2];        // the even CTA's: both CTAs' copies complete on it
    uint64_t empty[kStages2];       // each CTA's own, signalled by the pair's MMA commit
    uint64_t tmem_full[2];          // each CTA's own, signalled by the pair's MMA commit
    uint64_t tmem_empty[2];         // the even CTA's: both CTAs' epilogues arrive on it
    uint64_t drain;
    uint32_t tmem_base;
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of both CTAs: release this CTA's prior writes, wait for the peer's.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_smem(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// 2-D tiled TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier that may live in the peer CTA (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar_cluster, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;"
        :: "r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster),
           "r"(x), "r"(y), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void mma_issue_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive once on the mbarrier at `bar`'s offset in every CTA of `mask` when the pair's
// tcgen05 operations issued so far by this thread complete.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 :: "r"(smem_u32(bar)), "h"(mask) : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(smem_result)), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(bar_cluster) : "memory");
}

// Pair tiles t = (m2, n): hidden rows [256 m2, 256 m2 + 256), lm_head rows [256 n, 256 n + 256);
// the CTAs of a cluster take tiles t = pair, pair + pairs, ...  Even CTA (rank 0): MMA issuer and
// owner of the pair's full/tmem_empty barriers; both CTAs load their halves and write their rows.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs p) {
    constexpr uint32_t kIdesc = mma_idesc(kTile2, kTile2, false);
    extern __shared__ uint8_t smem_raw[];
    Gemm2Smem& s = *reinterpret_cast<Gemm2Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                 ~static_cast<uintptr_t>(1023));
    const uint32_t warp = warp_id(), lane = lane_id();
    const uint32_t rank = cluster_ctarank();
    const int pair = static_cast<int>(blockIdx.x >> 1), pairs = static_cast<int>(gridDim.x >> 1);
    const int total = p.tiles_a * p.tiles_b;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages2; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tmem_full[i], 1);
            mbar_init(&s.tmem_empty[i], 2 * 128);
        }
        mbar_init(&s.drain, 1);
        fence_mbarrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(&s.tmem_base, kTmemCols2);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();                     // both CTAs' barriers are initialised before any use
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs): this CTA's halves of A and B ----------------
            const uint64_t keep = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, any = false;
            for (int t = pair; ok && t < total; t += pairs) {
                const int m2 = t % p.tiles_a, n = t / p.tiles_a;
                const int a_row = m2 * kTile2 + static_cast<int>(rank) * 128;
                const int b_row = n * kTile2 + static_cast<int>(rank) * 128;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1u, p.ws, p.timeout_ns, kWaitProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_bar = peer_smem(&s.full[stage], 0);
                    if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], 4 * kHalfBytes2);   // both CTAs' copies
                    tma_load_2d_pair(s.a[stage], &tmA, kb * 64, a_row, full_bar, keep);
                    tma_load_2d_pair(s.b[stage], &tmB, kb * 64, b_row, full_bar, keep);
                    any = true;
                    if (++stage == kStages2) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok && any) {
                // copies in flight complete on the even CTA's barriers: give them time to land
                // before this CTA can leave
                const long long t0 = global_ns();
                while (global_ns() - t0 < 200000) __nanosleep(1000);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (even CTA) ----------------
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = pair; ok && t < total; t += pairs) {
                if (!mbar_wait(&s.tmem_empty[acc], acc_phase ^ 1u, p.ws, p.timeout_ns, kWaitMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kTile2);
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&s.full[stage], phase, p.ws, p.timeout_ns, kWaitMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(s.a[stage]);
                    const uint32_t b_addr = smem_u32(s.b[stage]);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_issue_pair(d_tmem, sw128_kmajor_desc(a_addr + k * 32), sw128_kmajor_desc(b_addr + k * 32),
                                       kIdesc, (kb | k) != 0 ? 1u : 0u);
                    mma_commit_pair(&s.empty[stage], 0x3);     // both CTAs may refill the stage
                    if (++stage == kStages2) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair(&s.tmem_full[acc], 0x3);       // both halves of the accumulator done
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            mma_commit_pair(&s.drain, 0x1);
            const long long t0 = global_ns();
            while (!mbar_try_wait(&s.drain, 0) && global_ns() - t0 < p.timeout_ns) {
            }
        }
    } else {
        // ---------------- epilogue: warps 2..5 of both CTAs ----------------
        const uint32_t quad = warp & 3u;
        const uint32_t row = quad * 32u + lane;
        const bool vec = (p.V & 3) == 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = pair; t < total; t += pairs) {
            const int m2 = t % p.tiles_a, n = t / p.tiles_a;
            const bool ready = mbar_wait(&s.tmem_full[acc], acc_phase, p.ws, p.timeout_ns, kWaitEpilogue);
            if (!__all_sync(0xFFFFFFFFu, ready)) break;
            tc_fence_after();
            const int m = m2 * kTile2 + static_cast<int>(rank) * 128 + static_cast<int>(row);
            float* orow = p.out + static_cast<size_t>(m) * p.V;
            const uint32_t taddr = tmem_base + ((quad * 32u) << 16) + static_cast<uint32_t>(acc * kTile2);
            for (int c0 = 0; c0 < kTile2; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(taddr + c0, r);
                tmem_wait_ld();
                const int v0 = n * kTile2 + c0;
                if (m < p.M) {
                    if (vec && v0 + 16 <= p.V) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4*>(orow + v0 + j) =
                                make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                            __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (v0 + j < p.V) orow[v0 + j] = __uint_as_float(r[j]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive_cluster(peer_smem(&s.tmem_empty[acc], 0));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    // neither CTA leaves while the pair's MMAs, copies or arrivals may still touch the other
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols2);
    }
}

template <int BN, bool kTF32>
dspark_status run_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& args,
                       cudaStream_t stream, const DeviceInfo& dev) {
    auto kernel = gemm_tcgen05_kernel<BN, kTF32>;
    const size_t smem = sizeof(GemmSmem<BN>) + 1024;
    if (smem > dev.smem_optin) {
        set_error("draft_logits: needs %zu bytes of shared memory, device allows %zu", smem, dev.smem_optin);
        return DSPARK_ERR_UNSUPPORTED;
    }
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(draft_logits)");
    const int total = args.tiles_a * args.tiles_b;
    const int grid = std::max(1, std::min(total, dev.sm_count));
    kernel<<<grid, kThreads, smem, stream>>>(ta, tb, args);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(draft_logits)");
    return DSPARK_OK;
}

dspark_status run_gemm_pair(const void* hidden, const void* lm_head, GemmArgs args, cudaStream_t stream,
                            const DeviceInfo& dev) {
    CUtensorMap ta, tb;
    const uint64_t dims_a[2] = {static_cast<uint64_t>(args.H), static_cast<uint64_t>(args.M)};
    const uint64_t dims_b[2] = {static_cast<uint64_t>(args.H), static_cast<uint64_t>(args.V)};
    const uint64_t stride[1] = {static_cast<uint64_t>(args.H) * 2};
    const uint32_t box[2] = {64, 128};
    if (!make_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, hidden, dims_a, stride, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lm_head, dims_b, stride, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
        return DSPARK_ERR_UNSUPPORTED;
    args.swap = 0;
    args.tiles_a = (args.M + kTile2 - 1) / kTile2;
    args.tiles_b = (args.V + kTile2 - 1) / kTile2;
    const size_t smem = sizeof(Gemm2Smem) + 1024;
    if (smem > dev.smem_optin) {
        set_error("draft_logits: needs %zu bytes of shared memory, device allows %zu", smem, dev.smem_optin);
        return DSPARK_ERR_UNSUPPORTED;
    }
    cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(draft_logits pair)");
    const int total = args.tiles_a * args.tiles_b;
    const int grid = 2 * std::max(1, std::min(total, dev.sm_count / 2));
    gemm_pair_kernel<<<grid, kThreads, smem, stream>>>(ta, tb, args);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "launch(draft_logits pair)");
    return DSPARK_OK;
}

}  // namespace

dspark_status launch_draft_logits(const void* hidden, const void* lm_head, dspark_dtype dtype, int M,
                                  int H, int V, float* logits, void* ws, cudaStream_t stream,
                                  const DeviceInfo& dev) {
    const bool tf32 = dtype == DSPARK_F32;
    const uint32_t esize = tf32 ? 4u : 2u;
    const uint32_t kelems = kRowBytes / esize;
    const bool swap = M <= 256;
    int BN = 256;
    if (swap) {
        BN = 16;
        while (BN < M) BN *= 2;
    }
    const CUtensorMapDataType ttype = tf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const void* a_ptr = swap ? lm_head : hidden;
    const void* b_ptr = swap ? hidden : lm_head;
    const uint64_t a_rows = swap ? static_cast<uint64_t>(V) : static_cast<uint64_t>(M);
    const uint64_t b_rows = swap ? static_cast<uint64_t>(M) : static_cast<uint64_t>(V);
    CUtensorMap ta, tb;
    const uint64_t dims_a[2] = {static_cast<uint64_t>(H), a_rows};
    const uint64_t dims_b[2] = {static_cast<uint64_t>(H), b_rows};
    const uint64_t stride[1] = {static_cast<uint64_t>(H) * esize};
    const uint32_t box_a[2] = {kelems, static_cast<uint32_t>(kTileA)};
    const uint32_t box_b[2] = {kelems, static_cast<uint32_t>(BN)};
    if (!make_tensor_map(&ta, ttype, 2, a_ptr, dims_a, stride, box_a, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&tb, ttype, 2, b_ptr, dims_b, stride, box_b, CU_TENSOR_MAP_SWIZZLE_128B))
        return DSPARK_ERR_UNSUPPORTED;

    GemmArgs args;
    args.out = logits;
    args.M = M;
    args.V = V;
    args.H = H;
    args.swap = swap ? 1 : 0;
    args.tiles_a = static_cast<int>((a_rows + kTileA - 1) / kTileA);
    args.tiles_b = static_cast<int>((b_rows + BN - 1) / BN);
    args.k_blocks = static_cast<int>((static_cast<uint32_t>(H) + kelems - 1) / kelems);
    args.ws = static_cast<WsHeader*>(ws);
    args.timeout_ns = kDefaultTimeoutNs;
    if (!swap && !tf32 && dev.sm_count >= 2) return run_gemm_pair(hidden, lm_head, args, stream, dev);

#define DSPARK_GEMM_CASE(bn)                                                          \
    case bn:                                                                          \
        return tf32 ? run_gemm<bn, true>(ta, tb, args, stream, dev)                   \
                    : run_gemm<bn, false>(ta, tb, args, stream, dev);
    switch (BN) {
        DSPARK_GEMM_CASE(16)
        DSPARK_GEMM_CASE(32)
        DSPARK_GEMM_CASE(64)
        DSPARK_GEMM_CASE(128)
        DSPARK_GEMM_CASE(256)
        default:
            set_error("draft_logits: no tile for M=%d", M);
            return DSPARK_ERR_UNSUPPORTED;
    }
#undef DSPARK_GEMM_CASE
}

}  // namespace dspark
