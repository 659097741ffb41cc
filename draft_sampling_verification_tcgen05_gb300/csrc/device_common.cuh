// Device-side building blocks shared by the kernels of the DSpark hot path:
// status word, bounded waits, grid barrier, Philox4x32-10, argmax keys, and
// thin inline-PTX wrappers for mbarrier, TMA and tcgen05 (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/dspark.h"

namespace dspark {

// ---------------------------------------------------------------------------
// Workspace header (first 256 bytes of every workspace).
// ---------------------------------------------------------------------------
struct WsHeader {
    uint32_t status;        // DSPARK_STATUS_* bits
    uint32_t barrier;       // grid-barrier arrival counter
    uint32_t detail;        // where a wait gave up (kernel-specific code)
    uint32_t never_set;     // flag that nothing writes (wait self-test)
    uint32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr long long kDefaultTimeoutNs = 2000000000LL;   // 2 s for any single wait

__device__ __forceinline__ long long global_ns() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_status(WsHeader* ws, uint32_t bits) {
    atomicOr(&ws->status, bits);
}

// Index checks at gather sites.  An index taken from the caller (an anchor, a draft token, a
// length, a table entry) is always checked: out of range it sets INPUT_RANGE (and INDEX in a
// checked build) and the kernel substitutes a safe value.  An index the library computed itself
// (a token read back from a step slot, a sorted candidate, a request from a work list) is checked
// only in a library built with -DDSPARK_CHECKED: out of range it sets INDEX and the access is
// skipped.  Neither kind ever traps.
#ifdef DSPARK_CHECKED
constexpr bool kCheckedBuild = true;
#else
constexpr bool kCheckedBuild = false;
#endif

__device__ __forceinline__ void flag_input_index(WsHeader* ws) {
    set_status(ws, DSPARK_STATUS_INPUT_RANGE | (kCheckedBuild ? DSPARK_STATUS_INDEX : 0u));
}

__device__ __forceinline__ bool own_index_ok(long long i, long long n, WsHeader* ws) {
    if (!kCheckedBuild || (i >= 0 && i < n)) return true;
    set_status(ws, DSPARK_STATUS_INDEX);
    return false;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

// Relaxed (GPU-scope, L1-bypassing) 64-bit store and load: for a value that is itself the whole
// message, with no other data to order behind it.
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Counter increment with release (every write the thread, or its block or warp through a barrier
// before it, made is visible first) and acquire (the caller's later reads see what the other
// incrementers released): the "last one to finish" pattern without separate fences.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
    return *reinterpret_cast<const volatile uint32_t*>(p);
}

// True once another part of the kernel has recorded a timeout (all waits give up then).
__device__ __forceinline__ bool aborted(const WsHeader* ws) {
    return (ld_volatile_u32(&ws->status) & DSPARK_STATUS_TIMEOUT) != 0;
}

// ---------------------------------------------------------------------------
// Grid barrier for a cooperative (co-resident) grid.  The arrival counter in
// the workspace header starts at 0 for every call (the host clears it);
// barrier number `phase` (0, 1, ...) waits until (phase+1)*gridDim.x blocks
// have arrived.  The spin is bounded: after timeout_ns it records TIMEOUT and
// returns false, and every other block gives up as soon as it sees the flag.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool grid_barrier(WsHeader* ws, uint32_t phase, long long timeout_ns,
                                             uint32_t where) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        // release on arrival, acquire on the poll; the block barriers carry both to every thread
        int ok = 1;
        const uint32_t target = (phase + 1u) * gridDim.x;
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(&ws->barrier) : "memory");
        long long t0 = global_ns();
        uint32_t spins = 0;
        while (ld_acquire_u32(&ws->barrier) < target) {
            if ((++spins & 63u) == 0) {
                if (aborted(ws)) { ok = 0; break; }
                if (global_ns() - t0 > timeout_ns) {
                    atomicOr(&ws->status, DSPARK_STATUS_TIMEOUT);
                    atomicExch(&ws->detail, where);
                    ok = 0;
                    break;
                }
            }
            __nanosleep(64);
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// The same barrier in two halves, so a block can do work that does not depend
// on the other blocks between arriving and waiting.
__device__ __forceinline__ void grid_arrive(WsHeader* ws) {
    __syncthreads();
    if (threadIdx.x == 0)                        // release: covers the block's writes before the barrier
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(&ws->barrier) : "memory");
}

__device__ __forceinline__ bool grid_wait(WsHeader* ws, uint32_t phase, long long timeout_ns, uint32_t where) {
    __shared__ int s_ok2;
    if (threadIdx.x == 0) {
        int ok = 1;
        const uint32_t target = (phase + 1u) * gridDim.x;
        const long long t0 = global_ns();
        uint32_t spins = 0;
        while (ld_acquire_u32(&ws->barrier) < target) {
            if ((++spins & 63u) == 0) {
                if (aborted(ws)) { ok = 0; break; }
                if (global_ns() - t0 > timeout_ns) {
                    atomicOr(&ws->status, DSPARK_STATUS_TIMEOUT);
                    atomicExch(&ws->detail, where);
                    ok = 0;
                    break;
                }
            }
            __nanosleep(32);
        }
        s_ok2 = ok;                              // the acquire above orders the block's later reads
    }
    __syncthreads();
    return s_ok2 != 0;
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// Grid barrier among a subset of every block's threads: the `nthreads`
// participants of named barrier `bar_id` (a multiple of 32), of which exactly
// one has `leader` set.  Same bounded spin and abort rules as grid_barrier.
__device__ __forceinline__ bool grid_barrier_named(WsHeader* ws, uint32_t phase, long long timeout_ns,
                                                   uint32_t where, uint32_t bar_id, uint32_t nthreads,
                                                   bool leader, volatile int* s_ok) {
    named_bar_sync(bar_id, nthreads);
    if (leader) {
        // the release of the arrival covers every write the block's threads made before the named
        // barrier, and the acquire of the poll every read after it: no separate fences
        int ok = 1;
        const uint32_t target = (phase + 1u) * gridDim.x;
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(&ws->barrier) : "memory");
        const long long t0 = global_ns();
        uint32_t spins = 0;
        while (ld_acquire_u32(&ws->barrier) < target) {
            if ((++spins & 63u) == 0) {
                if (aborted(ws)) { ok = 0; break; }
                if (global_ns() - t0 > timeout_ns) {
                    atomicOr(&ws->status, DSPARK_STATUS_TIMEOUT);
                    atomicExch(&ws->detail, where);
                    ok = 0;
                    break;
                }
            }
            __nanosleep(32);
        }
        *s_ok = ok;
    }
    named_bar_sync(bar_id, nthreads);
    return *s_ok != 0;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplications on counter
// words 0 and 2, with the key bumped by the Weyl constants between rounds.
// ---------------------------------------------------------------------------
constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = c.x * kPhiloxM0;
        const uint32_t hi0 = __umulhi(c.x, kPhiloxM0);
        const uint32_t lo1 = c.z * kPhiloxM1;
        const uint32_t hi1 = __umulhi(c.z, kPhiloxM1);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
    return c;
}

// Counter layout of this library: (j, b, (stream << 16) | i, offset).
enum : uint32_t {
    kStreamGumbel = 0,
    kStreamAccept = 1,
    kStreamResample = 2,
    kStreamGumbelLo = 3,
    kStreamResidual = 4,        // from-logits resample: word v & 3 of counter j = v >> 2
};

__device__ __forceinline__ uint4 philox_at(uint64_t seed, uint32_t offset, uint32_t j, uint32_t b,
                                           uint32_t stream, uint32_t i) {
    return philox4x32_10(make_uint4(j, b, (stream << 16) | i, offset),
                         static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
}

// u = ((w >> 9) + 1/2) * 2^-23 in [2^-24, 1 - 2^-24]; every step is exact in fp32.
__device__ __forceinline__ float uniform_from_word(uint32_t w) {
    return __fmul_rn(__fadd_rn(static_cast<float>(w >> 9), 0.5f), 0x1p-23f);
}

// Standard Gumbel variate -log(-log(u)) with CUDA's (accurate) logf.
__device__ __forceinline__ float gumbel_from_word(uint32_t w) {
    const float u = uniform_from_word(w);
    return -logf(-logf(u));
}

// Draft noise, in groups of 16 entries (group G = v >> 4, position k = v & 15).
// The group word is word G & 3 of stream-0 counter G >> 2: its bits 0-3 give
// the position p of the group's largest variate and its uniform u0 the
// group's smallest exponential E_min = -log(u0) / 16.  Entry k != p adds its
// own exponential: E_k = E_min - log(u_k), u_k from word k & 3 of stream-3
// counter (G << 2) | (k >> 2); E_p = E_min; g = -log(E).  The 16 E's are
// independent Exp(1) variates (the smallest of 16 is Exp(16), at a uniform
// position, and the rest exceed it by independent Exp(1) amounts), so the g's
// are independent standard Gumbels, and -log(E_min) bounds the whole group.
__device__ __forceinline__ uint32_t word_of(const uint4& w, uint32_t s) {
    return s == 0 ? w.x : s == 1 ? w.y : s == 2 ? w.z : w.w;
}

__device__ __forceinline__ uint32_t draft_group_word(uint64_t seed, uint32_t offset, uint32_t b, uint32_t i,
                                                     uint32_t G) {
    return word_of(philox_at(seed, offset, G >> 2, b, kStreamGumbel, i), G & 3u);
}

// E_min of a group word (the scaling by 1/16 is exact).
__device__ __forceinline__ float group_e_min(uint32_t W) {
    return __fmul_rn(-logf(uniform_from_word(W)), 0.0625f);
}

// Gumbel variate of an entry other than the group's largest, from its element word.
__device__ __forceinline__ float draft_gumbel_of_entry(float e_min, uint32_t w) {
    return -logf(__fadd_rn(e_min, -logf(uniform_from_word(w))));
}

// Gumbel variate of entry k of group G whose group word is W (E_min = group_e_min(W)).
__device__ __forceinline__ float draft_gumbel_in_group(uint64_t seed, uint32_t offset, uint32_t b, uint32_t i,
                                                       uint32_t G, uint32_t k, uint32_t W, float e_min) {
    if (k == (W & 15u)) return -logf(e_min);
    return draft_gumbel_of_entry(e_min, word_of(philox_at(seed, offset, (G << 2) | (k >> 2), b, kStreamGumbelLo, i),
                                                k & 3u));
}

__device__ __forceinline__ float draft_gumbel(uint64_t seed, uint32_t offset, uint32_t b, uint32_t i, uint32_t v) {
    const uint32_t G = v >> 4;
    const uint32_t W = draft_group_word(seed, offset, b, i, G);
    return draft_gumbel_in_group(seed, offset, b, i, G, v & 15u, W, group_e_min(W));
}

// Draft variates of the adjacent entries v and v + 1 (v even: one group word and one
// element counter serve both).
__device__ __forceinline__ void draft_gumbel_pair(uint64_t seed, uint32_t offset, uint32_t b, uint32_t i,
                                                  uint32_t v, float& g0, float& g1) {
    const uint32_t G = v >> 4, k = v & 15u;
    const uint32_t W = draft_group_word(seed, offset, b, i, G);
    const float e_min = group_e_min(W);
    const uint4 w = philox_at(seed, offset, (G << 2) | (k >> 2), b, kStreamGumbelLo, i);
    const uint32_t p = W & 15u;
    g0 = k == p ? -logf(e_min) : draft_gumbel_of_entry(e_min, word_of(w, k & 3u));
    g1 = k + 1u == p ? -logf(e_min) : draft_gumbel_of_entry(e_min, word_of(w, (k + 1u) & 3u));
}

// Bound on every draft variate: E_min >= -log(1 - 2^-24) / 16, so g <= 19.41; logf is
// accurate to a few ulp, so 19.5 leaves a wide margin.
constexpr float kDraftGumbelMax = 19.5f;

// Every standard Gumbel variate of one word (gumbel_from_word) is below this
// bound: the largest u is 1 - 2^-24, for which -log(-log(u)) = 16.6355..; logf
// is accurate to a few ulp, so 16.75 leaves a wide margin.  Used only to skip
// elements that can not win an argmax.
constexpr float kGumbelMax = 16.75f;

// ---------------------------------------------------------------------------
// Argmax keys: a 64-bit key whose unsigned order is (value ascending, index
// descending), so atomicMax picks the largest value and, among equal values,
// the lowest index.  Key 0 is below every real value (it decodes to a NaN).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t float_order_bits(float x) {
    x = __fadd_rn(x, 0.0f);                        // -0 -> +0
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float float_from_order_bits(uint32_t o) {
    const uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    return __uint_as_float(b);
}

__device__ __forceinline__ unsigned long long argmax_key(float value, uint32_t index) {
    return (static_cast<unsigned long long>(float_order_bits(value)) << 32) |
           static_cast<unsigned long long>(0xFFFFFFFFu - index);
}

__device__ __forceinline__ uint32_t key_index(unsigned long long key) {
    return 0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull);
}

// Two hardware reduces (the high words, then the low words of the lanes holding the largest high
// word) instead of five shuffle rounds of two words each: a shuffle occupies its SM sub-partition
// for several issue cycles.
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long k) {
    const uint32_t hi = static_cast<uint32_t>(k >> 32), lo = static_cast<uint32_t>(k);
    const uint32_t mhi = __reduce_max_sync(0xFFFFFFFFu, hi);
    const uint32_t mlo = __reduce_max_sync(0xFFFFFFFFu, hi == mhi ? lo : 0u);
    return (static_cast<unsigned long long>(mhi) << 32) | mlo;
}

// Sum over the warp, modulo 2^64 like a shuffle-tree sum, by three hardware reduces: the value in
// parts of 21, 21 and 22 bits, whose 32-lane sums cannot overflow 32 bits.
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long x) {
    const uint32_t s0 = __reduce_add_sync(0xFFFFFFFFu, static_cast<uint32_t>(x & 0x1FFFFFull));
    const uint32_t s1 = __reduce_add_sync(0xFFFFFFFFu, static_cast<uint32_t>((x >> 21) & 0x1FFFFFull));
    const uint32_t s2 = __reduce_add_sync(0xFFFFFFFFu, static_cast<uint32_t>(x >> 42));
    return static_cast<unsigned long long>(s0) + (static_cast<unsigned long long>(s1) << 21) +
           (static_cast<unsigned long long>(s2) << 42);
}

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarrier and TMA.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity.  On timeout (or when the
// kernel is already aborting) records TIMEOUT/`where` and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, WsHeader* ws,
                                          long long timeout_ns, uint32_t where) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = global_ns();
    uint32_t spins = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++spins & 255u) == 0) {
            if (aborted(ws)) return false;
            if (global_ns() - t0 > timeout_ns) {
                atomicOr(&ws->status, DSPARK_STATUS_TIMEOUT);
                atomicExch(&ws->detail, where);
                return false;
            }
        }
    }
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2-D tiled TMA load global -> shared, completing on `bar` (x = innermost coordinate).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;"
        :: "r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)),
           "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// 3-D tiled TMA load (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;"
        :: "r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)),
           "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

// 3-D tiled prefetch of a box into L2 (no shared memory, no completion tracking).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

// Make generic-proxy writes to shared memory visible to the async proxy
// (tensor core operand reads, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads/stores.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(smem_result)), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.  The
// tile base must be 1024-byte aligned; a K offset inside the 128-byte row is
// added to the start address.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);      // start address   [0,14)
    d |= static_cast<uint64_t>(1) << 16;                          // leading offset  [16,30) (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                  // stride offset   [32,46)
    d |= static_cast<uint64_t>(1) << 46;                          // descriptor version (sm_100 family)
    d |= static_cast<uint64_t>(2) << 61;                          // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::f16 (bf16 inputs) or kind::tf32, fp32
// accumulation, both operands K-major, M x N tile.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, bool tf32) {
    return (1u << 4)                                    // D format: f32
         | ((tf32 ? 2u : 1u) << 7)                      // A format: bf16 = 1, tf32 = 2
         | ((tf32 ? 2u : 1u) << 10)                     // B format
         | (static_cast<uint32_t>(N >> 3) << 17)        // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);       // M / 16
}

template <bool kTF32>
__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    if constexpr (kTF32) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
            :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
            :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
    }
}

// kind::f16 MMA whose A operand (M rows x 16 K elements) sits in tensor memory at a_tmem: row m
// in lane m, K elements 2c and 2c + 1 in column c (lower half first); B from shared memory.
__device__ __forceinline__ void mma_issue_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp gets lane
// (quadrant*32 + t) columns [col, col+16).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// 32 lanes x 32 bits, one column: thread t of the warp gets lane (quadrant*32 + t) of column col.
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
    return r;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
           "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
           "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// 32 lanes x 32 bits, 32 consecutive columns from r[0..31]: thread t of the warp writes lane
// (quadrant*32 + t) columns [col, col+32).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
           "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
           "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
           "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]),
           "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t warp_id() { return threadIdx.x >> 5; }
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

}  // namespace dspark
