// gdn_common.cuh -- device helpers and parameter blocks shared by the forward and
// backward kernels of the gated delta rule library (internal; not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

namespace gdn {

constexpr unsigned kFullMask = 0xffffffffu;

// Thread layout of every state tile: a warp owns kRowsPerWarp rows of one value head's
// [Dv, Dk] state; lane l holds columns l, l+32, ..., l+32*(E-1) of each of those rows
// (E = Dk/32). Row dot products (S k, S q, Sh k) are therefore sums across the 32
// lanes; column sums (for dq, dk) are sums over a thread's rows, then over warps.
constexpr int kRowsPerWarp = 8;
// Steps per forward staging tile (a multiple of 16).
constexpr int kFwdTile = 32;
constexpr int kMaxChunk = 128;
constexpr int kMaxDv = 4096;

struct FwdParams {
    const void *q, *k, *v, *g, *beta;
    const float *S0;
    void *y;
    float *S_T, *ckpt;      // ckpt may be null (no backward follows: nothing is saved)
    float *resid;           // [B, T, Hv, Dv] v_t - u_t, kept for the backward; may be null
    int *status;            // device status word (bounded-wait timeouts), may be null
    int B, T, Hk, Hv, Dv, C, NC;
};

struct BwdParams {
    const void *q, *k, *v, *g, *beta;
    const float *ckpt;
    const float *resid;     // [B, T, Hv, Dv] v_t - u_t as written by the forward
    const void *dy;
    const float *dS_T;
    float *dS0;
    float *ws_dq, *ws_dk;   // [B, T, Hv, nsplit, Dk] per-CTA column partials
    float *ws_dg, *ws_db;   // [B, T, Hv, nsplit]
    float *ws_state;        // per CTA: nsub_max sub-block start states of RB x Dk (pair layout)
    void *dv;
    int *status;            // device status word (bounded-wait timeouts), may be null
    int B, T, Hk, Hv, Dv, C, NC, nsplit, nsub_max;
    int slots;              // depth of the per-step partial-sum ring (2..4)
};

// Backward geometry, shared by host and device. A lane holds Dk/32 columns of each of
// its rows as bwd_pairs(Dk) column pairs (the last pair only on lanes 0..15 when Dk/32
// is odd). A sub-block of bwd_sub(Dk) steps keeps bwd_sub - 1 states in tensor memory
// (256 columns per thread: 8 rows x 2 x pairs columns per state) and one in registers.
__host__ __device__ constexpr int bwd_pairs(int Dk) { return (Dk / 32 + 1) / 2; }
__host__ __device__ constexpr int bwd_sub(int Dk) {
    return 256 / (16 * bwd_pairs(Dk)) + 1 > 8 ? 8 : 256 / (16 * bwd_pairs(Dk)) + 1;
}
constexpr int kBwdRowsPerWarp = 8;
// The backward CTA: two warpgroups of compute warps (8 rows each, 64 rows per CTA) and one
// service warpgroup. Registers are rebalanced with setmaxnreg after launch: the launch
// gives every thread kBwdLaunchRegs; the compute warpgroups raise theirs to
// kBwdComputeRegs and the service warpgroup lowers its to kBwdServiceRegs, and the two
// shares add up to no more than the launch's total.
constexpr int kBwdComputeWarps = 8;
constexpr int kBwdThreads = (kBwdComputeWarps + 4) * 32;
constexpr int kBwdRows = kBwdComputeWarps * kBwdRowsPerWarp;
constexpr int kBwdLaunchRegs = 168;
constexpr int kBwdComputeRegs = 208;
constexpr int kBwdServiceRegs = 88;
static_assert(kBwdComputeWarps * 32 * kBwdComputeRegs + 128 * kBwdServiceRegs <= kBwdThreads * kBwdLaunchRegs,
              "register split exceeds the launch's registers");

// Chunkwise tensor-core forward (bf16 inputs, chunks of 64 steps). Per (b, h, chunk), in the
// saved buffer: lam, the in-chunk log-decay prefix [64]; and bf16 matrices in their shared-memory
// (core-matrix) layout: pkm [(Q K^T) o E_incl; (K K^T) o E_strict] [128][64], wm -W [64][Dk]
// (W = T diag(beta exp Lam) K), tm T = (I + A)^-1 [64][64], tcm T diag(beta) [64][64]; per
// (b, h, chunk, block of 64 value rows) s0m, the chunk-start state in bf16 [64][Dk]; and per
// (b, kv head, chunk) qkm, [Q; K] of the chunk [128][Dk].
struct ChunkParams {
    const void *q, *k, *v, *g, *beta;
    const float *S0;
    void *y;
    float *S_T, *ckpt, *resid;
    float *maps_M, *maps_Mt;   // the lite sweep's maps and their transposes ([B][Hv][Dk][Dk] each)
    const float *conv;         // prep in the re-computation backward: these fp32 checkpoints go to
                               // s0m as operand tiles, and W and T diag(beta) are not formed (else null)
    float *lam;
    __nv_bfloat16 *pkm, *wm, *tm, *tcm, *s0m, *qkm;
    int *status;
    int B, T, Hk, Hv, Dv, NC;
};

// Chunkwise tensor-core backward (same sizes as the chunkwise forward; consumes its saved
// buffer). nsplit = Dv / 64 blocks of value rows.
struct ChunkBwdParams {
    const void *dy, *beta;
    const float *resid, *lam;
    const __nv_bfloat16 *tm, *pkm, *s0m, *qkm;
    const float *dS_T;
    float *dS0;
    void *dv, *dg, *dq, *dk, *dbeta;
    float *ws_db, *ws_f;       // [B, T, Hv, nsplit, 2]: per 32 value rows (the halves of a 64-row block)
    __nv_bfloat16 *ws_yu;      // [B, Hv, NC, nsplit][128 x 64]: [dY; dU] of the block, operand layout
    __nv_bfloat16 *ws_dl;      // [B, Hv, NC, nsplit][64 x 64]: Delta = diag(beta) (v - u), operand layout
    __nv_bfloat16 *ws_dsl;     // [B, Hv, NC, nsplit][64 x Dk]: dS at each chunk end, operand layout
    // Hand-off from the reverse sweep to the gradient kernel when it runs alongside it: ready[(b
    // * Hv + h) * NC + c] counts the reverse-sweep CTAs (nsplit in all) that have published chunk
    // c of (b, h); ready null: the sweep publishes nothing and the gradient kernel waits for it
    // to finish. next hands out the gradient kernel's groups. Both zero when the sweep starts.
    unsigned *ready;
    int *next;
    int *status;
    int B, T, Hk, Hv, Dv, NC, nsplit;
};

// Gate map (a, b, A_log, dt_bias -> g, beta) and its VJP; a, b, g, beta, dg, dbeta, da, db
// are [rows = B*T, Hv] in the input type, the per-head parameters fp32.
struct GatesParams {
    const void *a, *b;
    const float *A_log, *dt_bias;
    void *g, *beta;
    const void *dg, *dbeta;
    void *da, *db;
    float *dA_log, *ddt_bias;
    int rows, Hv;
};

struct ReduceParams {
    const float *ws_dq, *ws_dk, *ws_dg, *ws_db;
    void *dq, *dk, *dg, *dbeta;
    int B, T, Hk, Hv, Dk, nsplit;
};

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Sum N values (N a power of two, 2 <= N <= 32) across the 32 lanes of a warp with
// (N - 1) + (5 - log2 N) shuffles instead of 5 N: at each of the first log2(N) levels a
// lane keeps half of its values, sends the other half to its partner (lane ^ m) and
// adds what it receives. Afterwards lane l holds the full sum of value index
// (l >> (5 - log2 N)) -- bit i of the index is lane bit (5 - log2 N + i) -- and the
// 32/N lanes that share that index hold the same sum. Summation order is fixed.
template <int N>
__device__ __forceinline__ float transpose_reduce(float (&v)[N], int lane) {
    static_assert(N >= 2 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two");
    int m = 16;
#pragma unroll
    for (int n = N; n > 1; n >>= 1, m >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(kFullMask, send, m);
        }
    }
    float x = v[0];
#pragma unroll
    for (; m >= 1; m >>= 1) x += __shfl_xor_sync(kFullMask, x, m);
    return x;
}

// Same as transpose_reduce, within aligned groups of G lanes (G = 16 or 32): afterwards
// lane l holds the group sum of value index ((l & (G-1)) >> (log2 G - log2 N)).
template <int N, int G>
__device__ __forceinline__ float group_transpose_reduce(float (&v)[N], int lane) {
    static_assert(N >= 1 && N <= G && (N & (N - 1)) == 0 && (G == 16 || G == 32), "bad sizes");
    int m = G / 2;
#pragma unroll
    for (int n = N; n > 1; n >>= 1, m >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(kFullMask, send, m);
        }
    }
    float x = v[0];
#pragma unroll
    for (; m >= 1; m >>= 1) x += __shfl_xor_sync(kFullMask, x, m);
    return x;
}

// ---------------------------------------------------------------- TMA and mbarriers
// Spin limit of every mbarrier wait: far above any legitimate copy latency. A wait that
// runs out records GDN_ERR_TIMEOUT (-6) in the status word and the CTA stops early.
constexpr unsigned kWaitLimit = 1u << 24;
constexpr int kStatusTimeout = -6;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Barrier `id` (1-15; 0 is __syncthreads) among the `n` threads (whole warps) that reach it.
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Bounded wait for the phase with the given parity to complete (at most `limit` polls); false
// on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, unsigned limit = kWaitLimit) {
    const uint32_t a = smem_addr(bar);
    for (unsigned it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// 4-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
        : "memory");
}

// 5-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                            int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], "
        "[%7];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_addr(bar))
        : "memory");
}

// Fetch a tensor map (a kernel parameter) into the descriptor cache ahead of its first use.
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// L2 eviction priorities for global traffic: streamed data (read or written once) is
// marked evict-first so that it does not push out data that is re-read soon (evict-last).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ float2 ld_hint(const float2 *ptr, uint64_t pol) {
    float2 v;
    asm("ld.global.L2::cache_hint.v2.f32 {%0, %1}, [%2], %3;" : "=f"(v.x), "=f"(v.y) : "l"(ptr), "l"(pol));
    return v;
}
__device__ __forceinline__ uint4 ld_hint(const uint4 *ptr, uint64_t pol) {
    uint4 v;
    asm("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr), "l"(pol));
    return v;
}
__device__ __forceinline__ uint2 ld_hint(const uint2 *ptr, uint64_t pol) {
    uint2 v;
    asm("ld.global.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;" : "=r"(v.x), "=r"(v.y) : "l"(ptr), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_hint(float2 *ptr, float2 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(ptr), "f"(v.x), "f"(v.y), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void st_hint(float *ptr, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(pol) : "memory");
}

// 1-D bulk copy global -> shared with an L2 eviction priority for the source.
__device__ __forceinline__ void bulk_load_hint(void *dst, const void *src, unsigned bytes, uint64_t *bar,
                                               uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

// 16-byte asynchronous copy global -> shared; the bytes past src_bytes (0 or 16) are zero.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 1-D bulk copy shared -> global (16-byte aligned addresses, size a multiple of 16), in the
// issuing thread's current bulk async-group.
__device__ __forceinline__ void bulk_store(void *dst, const void *src, unsigned bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
                 "r"(smem_addr(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's bulk stores have read their shared-memory source (the buffer may be
// reused), or have completed entirely.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The same, leaving this thread's N most recent bulk groups possibly still reading.
template <int N>
__device__ __forceinline__ void bulk_wait_read_but() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups are pending (the others' writes complete).
template <int N>
__device__ __forceinline__ void bulk_wait_but() { asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory"); }

// 2-D tiled TMA store of one box from shared memory (the box's layout as the tensor map's
// swizzle mode describes), in the issuing thread's current bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_addr(src))
                 : "memory");
}

// 5-D tiled TMA store of one box from shared memory, in the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_5d(const CUtensorMap *map, const void *src, int c0, int c1, int c2, int c3,
                                             int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4, %5}], [%6];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_addr(src))
        : "memory");
}

// 4-D tiled TMA store of one box from shared memory, in the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, const void *src, int c0, int c1, int c2,
                                             int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(src))
        : "memory");
}

// Orders this thread's earlier generic-proxy global writes before later async-proxy
// (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Counter hand-off between CTAs at GPU scope: the producer's earlier writes (its own, its bulk
// stores once complete, and those of other threads of its CTA that it has synchronised with)
// are visible to a consumer that reads the incremented value with load_acquire_gpu.
__device__ __forceinline__ void add_release_gpu(unsigned *ctr, unsigned v) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ctr), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned load_acquire_gpu(const unsigned *ctr) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    return v;
}
// Polling form: relaxed loads (several in flight at once), then fence_acquire_gpu once every
// value read is the one waited for.
__device__ __forceinline__ unsigned load_relaxed_gpu(const unsigned *ctr) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// ---------------------------------------------------------------- tensor memory
// Allocation is warp-collective (one warp); the allocated base address is written to
// shared memory. 32x32b accesses: warp w reaches TMEM lanes 32*(w%4) .. +31, one lane
// per thread, N consecutive 32-bit columns per access.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float2 (&v)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "f"(v[0].x), "f"(v[0].y), "f"(v[1].x), "f"(v[1].y), "f"(v[2].x), "f"(v[2].y), "f"(v[3].x), "f"(v[3].y),
        "f"(v[4].x), "f"(v[4].y), "f"(v[5].x), "f"(v[5].y), "f"(v[6].x), "f"(v[6].y), "f"(v[7].x), "f"(v[7].y)
        : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float2 (&v)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(v[0].x), "=f"(v[0].y), "=f"(v[1].x), "=f"(v[1].y), "=f"(v[2].x), "=f"(v[2].y),
                   "=f"(v[3].x), "=f"(v[3].y)
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float2 (&v)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=f"(v[0].x), "=f"(v[0].y), "=f"(v[1].x), "=f"(v[1].y), "=f"(v[2].x), "=f"(v[2].y), "=f"(v[3].x),
          "=f"(v[3].y), "=f"(v[4].x), "=f"(v[4].y), "=f"(v[5].x), "=f"(v[5].y), "=f"(v[6].x), "=f"(v[6].y),
          "=f"(v[7].x), "=f"(v[7].y)
        : "r"(taddr)
        : "memory");
}

// Per-thread register limit of the executing warpgroup (all four warps execute it).
template <int N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

// Programmatic dependent launch. A kernel launched with launch_pdl may begin (set-up: barrier
// initialisation, tensor-memory allocation, descriptor prefetch) while the previous kernel on the
// stream finishes; griddep_wait blocks until that kernel has completed and its memory writes are
// visible, so every kernel calls it before its first global memory access. griddep_launch lets
// the next kernel on the stream begin its own set-up.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` on stream s with programmatic stream serialization allowed (see griddep_wait).
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

__device__ __forceinline__ void report_status(int *status, int code) {
    if (status != nullptr) atomicExch(status, code);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(kFullMask, x, m);
    return x;
}

// Per-kernel timing (gdn_timing_enable): every launcher calls timing_mark(name, 0, s) just
// before and timing_mark(name, 1, s) just after each kernel launch; a no-op while timing is
// off. Defined with the C ABI.
void timing_mark(const char *kernel, int phase, cudaStream_t s);

// Launchers (one per kernel family); each returns the cudaError_t of its launch.
// tm_q / tm_k: 4-D tensor maps of q and k ([B, T, Hk, Dk], box {Dk, 1, kFwdTile, 1}).
// One decode step (T = 1, nothing saved): a streaming pass over the state (gdn_decode.cu), for
// Dk in {64, 128, 192, 256} (decode_takes).
bool decode_takes(int Dk);
cudaError_t launch_decode(const FwdParams &p, int Dk, int dtype, cudaStream_t s);
cudaError_t launch_fwd(const FwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k, int Dk, int dtype,
                       int warps, cudaStream_t s);
// tm_q / tm_k: tensor maps with box {Dk, 1, bwd_sub(Dk) + 1, 1}.
// Fails with cudaErrorInvalidConfiguration if the compiled kernel was given fewer
// registers per thread than the register split assumes.
cudaError_t launch_bwd(const BwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k, int Dk, int dtype,
                       cudaStream_t s);
// Depth of the backward's partial-sum ring for checkpoint interval C: the deepest (4, 3
// or 2 steps) whose shared-memory layout fits `limit` bytes, 0 if none does; and the
// shared-memory bytes of that layout.
int bwd_slots(int Dk, int C, int dtype, size_t limit);
size_t bwd_smem_bytes(int Dk, int C, int dtype, int slots);
cudaError_t launch_reduce(const ReduceParams &p, int dtype, cudaStream_t s);
cudaError_t launch_gates_fwd(const GatesParams &p, int dtype, cudaStream_t s);
// Chunkwise forward: Dk in {64, 128, 192}, Dv a multiple of 64 up to 256, bf16, C = 64.
// Tensor maps. Read by TMA loads in 1 KB core-matrix columns of 64 rows (no swizzle): k and q as
// 5-D column blocks of [B][T][Hk][Dk] {8, T, Dk / 8, Hk, B}, box {8, 64, Dk / 8, 1, 1}. vb: v as
// [B][T][Hv][Dv] bf16, 4-D {Dv, Hv, T, B}, box {64, 1, 64, 1} (64 value columns of 64 steps),
// 128-byte swizzle. qk, the [Q; K] buffer as {256, 2, 2 halves (Q, K), Dk / 8 chunks, B*Hk*NC blocks},
// box {256, 2, 1, Dk / 8, 1} (a half's 64 rows of a K chunk are 1 KB contiguous): written by
// TMA stores from an operand tile of 64 rows, read back the same way.
// Written by TMA stores, 128-byte swizzle: y as [B][T][Hv][Dv] bf16, box {64, 1, 64, 1}; r (v - u)
// as 5-D column blocks of [B][T][Hv][Dv] fp32 {32, T, Dv / 32, Hv, B}, box {32, 64, 2, 1, 1}.
// ck, the fp32 checkpoints [B][Hv][NC][Dv][Dk] as 2-D {Dk, B*Hv*NC*Dv}, box {32, 64}, 128-byte
// swizzle: written by TMA stores from staged [64][32] boxes.
struct ChunkFwdMaps {
    CUtensorMap vb, k, q, qk, y, r, ck;
};
// The chunkwise forward's kernels to launch (a bit set): prep (per-chunk products into the saved
// buffer), the sweep (states, checkpoints, y, v - u, S_T), and the lite sweep of the
// sequence-parallel form (every row's end state from a zero start into p.S_T, the state maps into
// p.maps_M and their transposes into p.maps_Mt, [B][Hv][Dk][Dk] each; nothing else is written).
constexpr int kStagePrep = 1, kStageSweep = 2, kStageLite = 4;
cudaError_t launch_chunk_fwd(const ChunkParams &p, const ChunkFwdMaps &maps, int Dk, cudaStream_t s,
                             int stages = kStagePrep | kStageSweep);
size_t chunk_prep_smem(int Dk, int Dv);
size_t chunk_sweep_smem(int Dk);
// Chunkwise backward: the reverse sweep over chunks (dS), the per-chunk gradient products
// and the fixed-order sums over value heads and row blocks.
// Tensor maps of [B][T][Hv][Dv] tensors: tm_dv dv (bf16, 4-D, box {64, 1, 64, 1}, 128-byte
// swizzle); tm_dy dy (bf16, 5-D column blocks {8, T, Dv / 8, Hv, B}, box {8, 128, 8, 1, 1}, no
// swizzle). tm_qk, tm_pk: the saved [Q; K] blocks (per b, kv head, chunk) and [P; KKm] blocks
// (per b, value head, chunk) as {256, 2, 2 halves, columns / 8, blocks}, box one half: a
// [64][columns] operand tile (Q or K; P).
// tm_dq, tm_dk: dq and dk as [B][T][Hk][Dk] bf16, 4-D, box {64, 1, 64, 1}, 128-byte swizzle.
// stages: the reverse sweep (dS, dD, dv, dbeta, f, dS0, the workspace) and the gradient kernel.
constexpr int kStageDsweep = 1, kStageGrad = 2;
cudaError_t launch_chunk_bwd(const ChunkBwdParams &p, const CUtensorMap &tm_dv, const CUtensorMap &tm_dy,
                             const CUtensorMap &tm_qk, const CUtensorMap &tm_pk, const CUtensorMap &tm_dq,
                             const CUtensorMap &tm_dk, int Dk, cudaStream_t s, int stages = kStageDsweep | kStageGrad);
// The scan over segments of the sequence-parallel form: forward X_0 = X0 (zero if null),
// X_s = X_{s-1} M_{s-1} + C_{s-1}; reverse X_{P-1} = X0, X_s = X_{s+1} M_{s+1}^T + C_{s+1}. X, C:
// [B*P][Hv][rows][Dk] fp32 (rows a multiple of 64), X0: [B][Hv][rows][Dk]. M: [B*P][Hv][Dk][Dk]
// fp32, the maps for the forward scan and their transposes for the reverse one (the kernel reads
// M row by row either way). A bounded wait that gives up writes kStatusTimeout to *status.
cudaError_t launch_segment_scan(const float *X0, const float *M, const float *C, float *X, int B, int P, int Hv,
                                int rows, int Dk, bool reverse, int *status, cudaStream_t s);
size_t chunk_dsweep_smem(int Dk);
size_t chunk_grad_smem(int Dk, int Dv);
cudaError_t launch_gates_bwd(const GatesParams &p, int dtype, cudaStream_t s);
// Diagnostics (gdn_diag.cu): a CTA whose bounded wait cannot succeed (the timeout path), and
// the FP32 FMA issue rate of the whole GPU.
cudaError_t launch_wait_probe(int *status, unsigned polls, cudaStream_t s);
cudaError_t measure_fma_rate(int packed, double *tflops);

}  // namespace gdn
