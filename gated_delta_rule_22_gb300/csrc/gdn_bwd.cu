// gdn_bwd.cu -- reverse-time VJP of the gated delta rule.
//
// The backward is the chain rule applied in reverse time to the recurrence of mlx issue
// #4614 ("Recurrence used for the references"); the pages print no backward formula.
// With Sh = dL/dS_t gathered from later steps, step t (going backwards) is
//     Sc     = Sh + dy_t q_t^T                     y_t = S_t q_t
//     ddelta = Sc k_t       dv_t = beta_t ddelta    dbeta_t = ddelta . (v_t - u_t)
//     du     = -beta_t ddelta
//     dA     = Sc + du k_t^T
//     dq_t  += S_t^T dy_t = g_t S_{t-1}^T dy_t + k_t (delta_t . dy_t)
//     dk_t  += Sc^T delta_t + g_t S_{t-1}^T du
//     dg_t   = <dA, S_{t-1}>
//     Sh     = g_t dA                                (= dL/dS_{t-1})
// Every element of the [Dv, Dk] tile is touched once per step in one fused pass of 8
// packed f32x2 operations per two elements; ddelta needs Sc k_t = Sh k_t + dy_t (q_t . k_t),
// so the row dot Sh k_t is formed in the previous step's pass (against k_{t-1}) and is the
// only cross-lane reduction on the serial chain.
//
// Checkpointing (mlx-lm PR #1217, "What this PR adds": forward-with-save, then a reverse
// sweep in the same chunked layout). Per chunk, going backwards:
//   pass A  re-runs the chunk from its checkpoint with the forward's own residuals
//           v_t - u_t (delta_t = beta_t (v_t - u_t), so no prediction dot: the states are
//           the forward's, bit for bit), keeping delta_t and v_t - u_t per row and step in
//           shared memory and the state at the start of every sub-block of
//           SUB = bwd_sub(Dk) steps in an L2-resident scratch;
//   per sub-block, going backwards:
//     pass B  takes the sub-block's start state (1-D TMA bulk copy, issued one sub-block
//             ahead) and re-builds the states inside it with the kept delta
//             (S <- g S + delta k^T), writing them to tensor memory (TMEM); the last one
//             stays in registers;
//     core    runs the reverse steps, reading S_{t-1} from TMEM in two halves (rows 0-3,
//             rows 4-7 of each warp) so that one half loads while the other is used.
//
// Warp roles. A CTA owns RB = 64 rows of one (b, h): two warpgroups of compute warps
// (8 rows each) and a service warpgroup, registers moved from the second to the first by
// setmaxnreg. Lane l of a compute warp holds the column pairs (2l + 64m, 2l + 1 + 64m) of
// each of its rows, so row dot products are 32-lane reductions and a warp's column sums
// are complete per lane. What a compute warp keeps between steps (delta, v - u, its rows
// of the states) is its own, so compute warps never wait for one another.
//   stager warp   stages every tile one tile ahead into a double buffer (k and q rows by
//                 TMA, widened to fp32; v - u or dy, g, beta and k . q per step, the global
//                 loads issued a tile earlier still) and issues the start-state copies;
//   reducer warp  sums the compute warps' per-step partials (columns of dq and dk, dg,
//                 dbeta) in ascending warp order out of a ring of slots into fp32
//                 scratch per (b, t, h, row split), and writes dv.
// reduce_kernel then adds the row splits (ascending) and the value heads of each kv head
// (ascending). Every hand-off is an mbarrier with a bounded wait; there are no atomics and
// no block-wide barriers between set-up and tear-down.
#include <type_traits>

#include "gdn_common.cuh"

namespace gdn {

namespace {

constexpr int kMaxSlots = 4;
// mbarriers
constexpr int kBarRaw = 0;          // [2] k (and q) rows of a tile landed in raw buffer b (TMA)
constexpr int kBarFull = 2;         // [2] tile buffer b staged for the compute warps (1 arrival)
constexpr int kBarEmpty = 4;        // [2] compute warps done with tile buffer b (ncw arrivals)
constexpr int kBarScb = 6;          // a sub-block start state landed in scb (bulk copy)
constexpr int kBarScbEmpty = 7;     // compute warps took their rows of scb (ncw arrivals)
constexpr int kBarStart = 8;        // a chunk's last sub-block start state is in scratch (ncw)
constexpr int kBarSlotFull = 9;     // [kMaxSlots] a step's partials are in the slot (ncw)
constexpr int kBarSlotEmpty = 9 + kMaxSlots;   // [kMaxSlots] slot reduced (1 arrival)
constexpr int kNumBars = 9 + 2 * kMaxSlots;

template <typename T>
struct IsF32B { static constexpr bool value = false; };
template <>
struct IsF32B<float> { static constexpr bool value = true; };

template <typename T>
struct QuadB;
template <>
struct QuadB<float> {
    using type = float4;
    static __device__ __forceinline__ type zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    static __device__ __forceinline__ float4 unpack(const type &q) { return q; }
};
template <>
struct QuadB<__nv_bfloat16> {
    using type = uint2;
    static __device__ __forceinline__ type zero() { return make_uint2(0u, 0u); }
    static __device__ __forceinline__ float4 unpack(const type &q) {
        return make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u),
                           __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
    }
};

__host__ __device__ inline size_t align_upb(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared-memory layout of bwd_kernel (byte offsets from a 128-byte aligned base).
struct BwdSmem {
    size_t raw, kfq, xrow, gsc, dl, vm, scb, ring, ring_stride, bar, tslot, total;
    __host__ __device__ BwdSmem(int DK, int esize, int C, int slots) {
        const int ncw = kBwdComputeWarps, RB = kBwdRows;
        const int P2 = bwd_pairs(DK), SUB = bwd_sub(DK), TR = SUB + 1;
        size_t o = 0;
        raw = o; o += align_upb((size_t)2 * 2 * TR * DK * esize, 128);   // [buf][k|q][TR][DK], input type
        kfq = o; o += (size_t)2 * 2 * TR * DK * 4;                        // [buf][k|q][TR][DK], fp32
        xrow = o; o += (size_t)2 * SUB * RB * 4;                           // [buf][SUB][RB]: v - u or dy
        gsc = o; o += (size_t)2 * 4 * SUB * 4;                             // [buf][g | beta | k.q | -][SUB]
        dl = o; o += (size_t)C * RB * 4;                                   // delta per step and row
        vm = o; o += (size_t)C * RB * 4;                                   // v - u per step and row
        o = align_upb(o, 128);
        scb = o; o += (size_t)RB * P2 * 64 * 4;                            // sub-block start state
        // slot: column partials [ncw][dk | dq][DK], (dg, dbeta) [ncw], dv [RB]
        ring_stride = align_upb((size_t)ncw * 2 * DK * 4 + (size_t)ncw * 8 + (size_t)RB * 4, 16);
        ring = o; o += (size_t)slots * ring_stride;
        bar = align_upb(o, 8); o = bar + kNumBars * 8;
        tslot = o; o += 16;
        total = o + 128;
    }
};

struct TileRef {
    int kind;  // 0 = pass A, 1 = reverse, -1 = none
    int c, m;
};

}  // namespace

template <int E, typename TIn>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, BwdParams p) {
    constexpr int R = kBwdRowsPerWarp;
    constexpr int DK = 32 * E;
    constexpr int P2 = bwd_pairs(DK);
    constexpr int SUB = bwd_sub(DK);
    constexpr int TR = SUB + 1;
    constexpr int NPAIR = R * P2;         // float2 pairs of one state per thread
    constexpr int SW = 2 * NPAIR;         // TMEM columns of one state per thread
    constexpr bool kOdd = (DK % 64) != 0; // the last pair exists only on lanes 0..15
    static_assert(R == 8, "the compute-warp layout assumes 8 rows per warp");
    static_assert(NPAIR % 8 == 0, "state must be a whole number of 16-column TMEM chunks");
    static_assert((SUB - 1) * SW <= 256, "sub-block states exceed the TMEM share");
    static_assert(SUB <= 8, "k . q of a tile is reduced as 8 values");

    constexpr int ncw = kBwdComputeWarps;
    constexpr int RB = kBwdRows;
    constexpr int kStager = ncw, kReducer = ncw + 1;   // service warps; ncw + 2, ncw + 3 idle
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int row0 = split * RB, hk = h / (p.Hv / p.Hk);
    const int T = p.T, Dv = p.Dv, C = p.C, Hv = p.Hv, nsplit = p.nsplit, slots = p.slots;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(align_upb(reinterpret_cast<size_t>(smem_raw), 128));
    const BwdSmem L(DK, (int)sizeof(TIn), C, slots);
    TIn *raw = reinterpret_cast<TIn *>(base + L.raw);
    float *kfq = reinterpret_cast<float *>(base + L.kfq);
    float *xrow = reinterpret_cast<float *>(base + L.xrow);
    float *gsc = reinterpret_cast<float *>(base + L.gsc);
    float *dl_s = reinterpret_cast<float *>(base + L.dl);
    float *vm_s = reinterpret_cast<float *>(base + L.vm);
    float *scb = reinterpret_cast<float *>(base + L.scb);
    unsigned char *ring = base + L.ring;
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + L.bar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + L.tslot);

    const size_t head = (size_t)b * Hv + h;
    const size_t cta = head * nsplit + split;
    const size_t slot_floats = (size_t)RB * P2 * 64;
    float *scratch = p.ws_state + cta * (size_t)p.nsub_max * slot_floats;
    // ring slot s: column partials, then (dg, dbeta) per warp, then dv per row (fp32)
    auto slot_cp = [&](int s) { return reinterpret_cast<float *>(ring + (size_t)s * L.ring_stride); };
    auto slot_gp = [&](int s) { return reinterpret_cast<float2 *>(slot_cp(s) + (size_t)ncw * 2 * DK); };
    auto slot_dv = [&](int s) { return reinterpret_cast<float *>(slot_gp(s) + ncw); };

    // ---- set-up: barriers, tensor memory
    if (tid == 0) {
        mbar_init(&bar[kBarRaw], 1);
        mbar_init(&bar[kBarRaw + 1], 1);
        mbar_init(&bar[kBarFull], 1);
        mbar_init(&bar[kBarFull + 1], 1);
        mbar_init(&bar[kBarEmpty], ncw);
        mbar_init(&bar[kBarEmpty + 1], ncw);
        mbar_init(&bar[kBarScb], 1);
        mbar_init(&bar[kBarScbEmpty], ncw);
        mbar_init(&bar[kBarStart], ncw);
        for (int s = 0; s < kMaxSlots; ++s) {
            mbar_init(&bar[kBarSlotFull + s], ncw);
            mbar_init(&bar[kBarSlotEmpty + s], 1);
        }
        fence_mbar_init();
    }
    if (warp == kStager) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    bool failed = false;
    int raw_issued[2] = {0, 0}, scb_loads = 0;   // stager: copies issued (for the drain)
    // Streamed data (checkpoints, residuals, dy, partial sums) is evicted first from L2; the
    // sub-block start states, written and read back within a chunk, are kept.
    const uint64_t pol_stream = l2_policy_evict_first();
    const uint64_t pol_keep = l2_policy_evict_last();

    // Each role's code sits under its own setmaxnreg, so that it is compiled for that
    // role's register limit.
    if (warp >= ncw) {
    regs_dec<kBwdServiceRegs>();
    if (warp == kStager) {
        // =============================== stager warp ===============================
        const float *resid = p.resid;
        const TIn *dy = static_cast<const TIn *>(p.dy);
        const TIn *g = static_cast<const TIn *>(p.g);
        const TIn *beta = static_cast<const TIn *>(p.beta);
        using QuadT = typename QuadB<TIn>::type;
        constexpr int kQ = (SUB * RB / 4 + 31) / 32;   // row quads per lane

        auto nsub_of = [&](int c) { return (min(C, T - c * C) + SUB - 1) / SUB; };
        auto tile_after = [&](TileRef t) -> TileRef {
            if (t.kind == 0) {
                if (t.m + 1 < nsub_of(t.c)) return {0, t.c, t.m + 1};
                return {1, t.c, nsub_of(t.c) - 1};
            }
            if (t.m > 0) return {1, t.c, t.m - 1};
            if (t.c > 0) return {0, t.c - 1, 0};
            return {-1, 0, 0};
        };
        auto slice_of = [&](TileRef t, int &s0, int &slen) {
            s0 = t.c * C + t.m * SUB;
            slen = min(SUB, min(t.c * C + C, T) - s0);
        };
        // TMA of a tile's k (and, for reverse tiles, q) rows s0 - 1 .. s0 + SUB - 1 (lane 0)
        auto issue_raw = [&](TileRef t, int rb) {
            int s0, slen;
            slice_of(t, s0, slen);
            TIn *dst = raw + (size_t)rb * 2 * TR * DK;
            fence_proxy_async();
            mbar_expect_tx(&bar[kBarRaw + rb], (t.kind == 1 ? 2u : 1u) * TR * DK * (unsigned)sizeof(TIn));
            tma_load_4d(dst, &tm_k, &bar[kBarRaw + rb], 0, hk, s0 - 1, b);
            if (t.kind == 1) tma_load_4d(dst + TR * DK, &tm_q, &bar[kBarRaw + rb], 0, hk, s0 - 1, b);
            ++raw_issued[rb];
        };
        // per-step inputs of a tile, loaded into registers one tile before they are staged:
        // dy (input type) for reverse tiles, v - u (fp32) for pass-A tiles
        constexpr bool kWide = IsF32B<TIn>::value;   // dy quads are 16 bytes (else 8)
        uint4 xq[kQ];                               // raw bits of 4 consecutive rows
        float gq = 1.f, bq = 0.f;
        auto fetch = [&](TileRef t) {
            int s0, slen;
            slice_of(t, s0, slen);
            constexpr int nq = RB / 4;
#pragma unroll
            for (int i = 0; i < kQ; ++i) {
                const int e = lane + 32 * i, j = e / nq, r4 = (e - j * nq) * 4;
                const size_t o = (((size_t)b * T + s0 + j) * Hv + h) * Dv + row0 + r4;
                const bool in = j < slen && row0 + r4 < Dv;
                if (t.kind == 1 && !kWide) {
                    const uint2 u = in ? ld_hint(reinterpret_cast<const uint2 *>(dy + o), pol_stream) : make_uint2(0u, 0u);
                    xq[i] = make_uint4(u.x, u.y, 0u, 0u);
                } else {
                    const void *src = t.kind == 1 ? static_cast<const void *>(dy + o) : static_cast<const void *>(resid + o);
                    xq[i] = in ? ld_hint(reinterpret_cast<const uint4 *>(src), pol_stream) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
            gq = lane < slen ? to_f32(g[((size_t)b * T + s0 + lane) * Hv + h]) : 1.f;
            bq = lane < slen ? to_f32(beta[((size_t)b * T + s0 + lane) * Hv + h]) : 0.f;
        };
        // Stage tile t (the x-th tile) into buffer x & 1, then fetch the tile after it and
        // send the raw rows of the tile two ahead. Returns false on a timeout.
        auto prepare = [&](TileRef t, int x) -> bool {
            const int bx = x & 1, fx = x >> 1;
            int s0, slen;
            slice_of(t, s0, slen);
            if (fx >= 1 && !mbar_wait(&bar[kBarEmpty + bx], (fx - 1) & 1)) return false;
            float *xr = xrow + (size_t)bx * SUB * RB;
            float *gs = gsc + (size_t)bx * 4 * SUB;
            constexpr int nq = RB / 4;
#pragma unroll
            for (int i = 0; i < kQ; ++i) {
                const int e = lane + 32 * i;
                if (e < SUB * nq) {
                    const uint4 u = xq[i];
                    *reinterpret_cast<float4 *>(xr + 4 * e) =
                        (t.kind == 1 && !kWide)
                            ? make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                                          __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u))
                            : make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                          __uint_as_float(u.w));
                }
            }
            if (lane < SUB) {
                gs[lane] = gq;
                gs[SUB + lane] = bq;
            }
            const TileRef nt = tile_after(t);
            if (nt.kind >= 0) fetch(nt);
            if (!mbar_wait(&bar[kBarRaw + bx], fx & 1)) return false;
            // widen the k (and q) rows to fp32: 16 bytes of input per access, the loads of a
            // batch issued back to back (trip counts are compile-time per tile kind)
            float *dstf = kfq + (size_t)bx * 2 * TR * DK;
            const TIn *src = raw + (size_t)bx * 2 * TR * DK;
            auto widen = [&](auto rows_c) {
                constexpr int ROWS = decltype(rows_c)::value;
                constexpr int EPC = IsF32B<TIn>::value ? 4 : 8;   // elements per 16 bytes
                constexpr int NCH = ROWS * DK / EPC;
                constexpr int PER = (NCH + 31) / 32;
                constexpr int BATCH = 4;
#pragma unroll
                for (int i0 = 0; i0 < PER; i0 += BATCH) {
                    uint4 w[BATCH];
#pragma unroll
                    for (int u = 0; u < BATCH; ++u) {
                        const int i = lane + 32 * (i0 + u);
                        if (i0 + u < PER && i < NCH) w[u] = reinterpret_cast<const uint4 *>(src)[i];
                    }
#pragma unroll
                    for (int u = 0; u < BATCH; ++u) {
                        const int i = lane + 32 * (i0 + u);
                        if (i0 + u < PER && i < NCH) {
                            if (IsF32B<TIn>::value) {
                                reinterpret_cast<uint4 *>(dstf)[i] = w[u];
                            } else {
                                float4 *d = reinterpret_cast<float4 *>(dstf + 8 * i);
                                d[0] = make_float4(__uint_as_float(w[u].x << 16), __uint_as_float(w[u].x & 0xffff0000u),
                                                   __uint_as_float(w[u].y << 16), __uint_as_float(w[u].y & 0xffff0000u));
                                d[1] = make_float4(__uint_as_float(w[u].z << 16), __uint_as_float(w[u].z & 0xffff0000u),
                                                   __uint_as_float(w[u].w << 16), __uint_as_float(w[u].w & 0xffff0000u));
                            }
                        }
                    }
                }
            };
            if (t.kind == 1) widen(std::integral_constant<int, 2 * TR>{});
            else widen(std::integral_constant<int, TR>{});
            __syncwarp();
            if (t.kind == 1) {
                // k_t . q_t for the tile's steps (all SUB rows; those past the tile's end are
                // never used): lane partials, one transpose reduction
                float part[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float a = 0.f;
                    if (j < SUB) {
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            a = fmaf(dstf[(j + 1) * DK + lane + 32 * e], dstf[(TR + j + 1) * DK + lane + 32 * e], a);
                    }
                    part[j] = a;
                }
                const float kq = group_transpose_reduce<8, 32>(part, lane);
                if ((lane & 3) == 0 && (lane >> 2) < SUB) gs[2 * SUB + (lane >> 2)] = kq;
                __syncwarp();
            }
            if (lane == 0) {
                mbar_arrive(&bar[kBarFull + bx]);
                if (nt.kind >= 0) {
                    const TileRef n2 = tile_after(nt);
                    if (n2.kind >= 0) issue_raw(n2, bx);   // raw buffer bx is free again
                }
            }
            __syncwarp();
            return true;
        };

        const TileRef first{0, p.NC - 1, 0};
        if (lane == 0) {
            issue_raw(first, 0);
            const TileRef t1 = tile_after(first);
            if (t1.kind >= 0) issue_raw(t1, 1);
        }
        __syncwarp();
        fetch(first);
        failed = !prepare(first, 0);
        int chunks_started = 0, x = 0;
        for (TileRef t = first; t.kind >= 0 && !failed; t = tile_after(t), ++x) {
            const TileRef nt = tile_after(t);
            if (nt.kind >= 0) {
                if (!prepare(nt, x + 1)) { failed = true; break; }
                if (nt.kind == 1) {
                    // the next reverse tile's start state, once pass A has written it
                    if (nt.m == nsub_of(nt.c) - 1) {
                        if (!mbar_wait(&bar[kBarStart], chunks_started & 1)) { failed = true; break; }
                        ++chunks_started;
                    }
                    if (scb_loads >= 1 && !mbar_wait(&bar[kBarScbEmpty], (scb_loads - 1) & 1)) { failed = true; break; }
                    if (lane == 0) {
                        fence_proxy_async_global();
                        fence_proxy_async();
                        mbar_expect_tx(&bar[kBarScb], (unsigned)(slot_floats * 4));
                        bulk_load_hint(scb, scratch + (size_t)nt.m * slot_floats, (unsigned)(slot_floats * 4), &bar[kBarScb],
                                       pol_keep);
                    }
                    ++scb_loads;
                    __syncwarp();
                }
            }
        }
    } else if (warp == kReducer) {
        // =============================== reducer warp ===============================
        // Steps arrive in the compute warps' order: chunks, sub-blocks and steps descending.
        TIn *dv = static_cast<TIn *>(p.dv);
        int gstep = 0;
        for (int c = p.NC - 1; c >= 0 && !failed; --c) {
            const int t0 = c * C, t1 = min(t0 + C, T);
            for (int tt = t1 - 1; tt >= t0; --tt, ++gstep) {
                const int s = gstep % slots, n = gstep / slots;
                if (!mbar_wait(&bar[kBarSlotFull + s], n & 1)) { failed = true; break; }
                const float *cp = slot_cp(s);
                const float2 *gp = slot_gp(s);
                const float *dvs = slot_dv(s);
                const size_t og = (((size_t)b * T + tt) * Hv + h) * nsplit + split;
#pragma unroll
                for (int m = 0; m < P2; ++m) {
                    const int col = 2 * lane + 64 * m;
                    if (col < DK) {
                        float2 a = make_float2(0.f, 0.f), q2 = a;
#pragma unroll
                        for (int w = 0; w < ncw; ++w) {
                            const float2 x1 = *reinterpret_cast<const float2 *>(cp + w * 2 * DK + col);
                            const float2 x2 = *reinterpret_cast<const float2 *>(cp + w * 2 * DK + DK + col);
                            a.x += x1.x; a.y += x1.y;
                            q2.x += x2.x; q2.y += x2.y;
                        }
                        st_hint(reinterpret_cast<float2 *>(p.ws_dk + og * DK + col), a, pol_stream);
                        st_hint(reinterpret_cast<float2 *>(p.ws_dq + og * DK + col), q2, pol_stream);
                    }
                }
                if (lane == 0) {
                    float dgs = 0.f, dbs = 0.f;
#pragma unroll
                    for (int w = 0; w < ncw; ++w) {
                        dgs += gp[w].x;
                        dbs += gp[w].y;
                    }
                    st_hint(p.ws_dg + og, dgs, pol_stream);
                    st_hint(p.ws_db + og, dbs, pol_stream);
                }
#pragma unroll
                for (int i = 0; i < RB / 32; ++i) {
                    const int rr = lane + 32 * i;
                    if (row0 + rr < Dv) dv[(((size_t)b * T + tt) * Hv + h) * Dv + row0 + rr] = from_f32<TIn>(dvs[rr]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kBarSlotEmpty + s]);
            }
        }
    }
    } else {
        // =============================== compute warps ===============================
        regs_inc<kBwdComputeRegs>();
        const TIn *k = static_cast<const TIn *>(p.k);
        const int wrow = warp * R;
        const int my_row = lane >> 2;   // row held by this lane after a transpose reduction of 8
        const int pair_off = wrow * P2 * 64 + 2 * lane;   // pair (r, m) of this thread at + (r * P2 + m) * 64
        const int pc = 2 * lane;                          // first column of this lane's pair 0
        const uint32_t tmem = *tslot + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * 256);
        auto pvalid = [&](int m) { return !kOdd || m < P2 - 1 || lane < 16; };
        auto load_pair = [&](const float *rowbase, int m) {
            return pvalid(m) ? *reinterpret_cast<const float2 *>(rowbase + pc + 64 * m) : make_float2(0.f, 0.f);
        };

        // ---- adjoint state Sh from dS_T, and its first row dot with k_{T-1}
        float2 Sh[R][P2];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = row0 + wrow + r;
#pragma unroll
            for (int m = 0; m < P2; ++m)
                Sh[r][m] = (p.dS_T != nullptr && row < Dv && pvalid(m))
                               ? *reinterpret_cast<const float2 *>(p.dS_T + (head * Dv + row) * DK + pc + 64 * m)
                               : make_float2(0.f, 0.f);
        }
        float p_own;   // Sh . k_t of row my_row, for the next reverse step t
        {
            float part[R];
            float2 kk[P2];
            const TIn *src = k + (((size_t)b * T + T - 1) * p.Hk + hk) * DK;
#pragma unroll
            for (int m = 0; m < P2; ++m) {
                kk[m].x = pvalid(m) ? to_f32(src[pc + 64 * m]) : 0.f;
                kk[m].y = pvalid(m) ? to_f32(src[pc + 64 * m + 1]) : 0.f;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int m = 0; m < P2; ++m) acc = __ffma2_rn(Sh[r][m], kk[m], acc);
                part[r] = acc.x + acc.y;
            }
            p_own = group_transpose_reduce<R, 32>(part, lane);
        }

        int x = 0, scb_reads = 0, gstep = 0;
        for (int c = p.NC - 1; c >= 0 && !failed; --c) {
            const int t0 = c * C, len = min(C, T - t0), nsub = (len + SUB - 1) / SUB;

            // ============ pass A: forward through the chunk from its checkpoint ============
            {
                float2 S[R][P2];
                const float *ck = p.ckpt + (head * p.NC + c) * (size_t)Dv * DK;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int row = row0 + wrow + r;
#pragma unroll
                    for (int m = 0; m < P2; ++m)
                        S[r][m] = (row < Dv && pvalid(m))
                                      ? ld_hint(reinterpret_cast<const float2 *>(ck + (size_t)row * DK + pc + 64 * m), pol_stream)
                                      : make_float2(0.f, 0.f);
                }
                for (int sm = 0; sm < nsub; ++sm, ++x) {
                    const int bx = x & 1;
                    const int s0 = t0 + sm * SUB, slen = min(SUB, t0 + len - s0);
                    float *slot = scratch + (size_t)sm * slot_floats + pair_off;
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int m = 0; m < P2; ++m) st_hint(reinterpret_cast<float2 *>(slot + (r * P2 + m) * 64), S[r][m], pol_keep);
                    if (sm == nsub - 1) {
                        // the reverse sweep starts from this state: hand it to the bulk copy
                        fence_proxy_async_global();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar[kBarStart]);
                    }
                    if (!mbar_wait(&bar[kBarFull + bx], (x >> 1) & 1)) { failed = true; break; }
                    const float *kf = kfq + (size_t)bx * 2 * TR * DK;   // row i = step s0 - 1 + i
                    const float *xr = xrow + (size_t)bx * SUB * RB;
                    const float *gs = gsc + (size_t)bx * 4 * SUB;
                    for (int j = 0; j < slen; ++j) {
                        float2 kv[P2];
#pragma unroll
                        for (int m = 0; m < P2; ++m) kv[m] = load_pair(kf + (j + 1) * DK, m);
                        const float gt = gs[j], bt = gs[SUB + j];
                        // v - u of the warp's rows (the forward's residuals); delta = beta (v - u)
                        const float *xw = xr + j * RB + wrow;
                        if (lane < R) {
                            const float x = xw[lane];
                            dl_s[(s0 - t0 + j) * RB + wrow + lane] = bt * x;
                            vm_s[(s0 - t0 + j) * RB + wrow + lane] = x;
                        }
                        const float4 x0 = *reinterpret_cast<const float4 *>(xw);
                        const float4 x1 = *reinterpret_cast<const float4 *>(xw + 4);
                        const float xv[R] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                        const float2 gg = make_float2(gt, gt);
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const float d = bt * xv[r];
                            const float2 dd = make_float2(d, d);
#pragma unroll
                            for (int m = 0; m < P2; ++m) S[r][m] = __ffma2_rn(dd, kv[m], __fmul2_rn(gg, S[r][m]));
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[kBarEmpty + bx]);
                }
            }
            if (failed) break;

            // ============ reverse sweep over the chunk's sub-blocks ============
            for (int sm = nsub - 1; sm >= 0; --sm, ++x) {
                const int bx = x & 1;
                const int s0 = t0 + sm * SUB, slen = min(SUB, t0 + len - s0);
                if (!mbar_wait(&bar[kBarFull + bx], (x >> 1) & 1)) { failed = true; break; }
                const float *kf = kfq + (size_t)bx * 2 * TR * DK;   // row i = step s0 - 1 + i
                const float *qf = kf + TR * DK;
                const float *xr = xrow + (size_t)bx * SUB * RB;
                const float *gs = gsc + (size_t)bx * 4 * SUB;
                // the sub-block's start state: rows 0-3 (X) and rows 4-7 (Y) of this warp
                if (!mbar_wait(&bar[kBarScb], scb_reads & 1)) { failed = true; break; }
                ++scb_reads;
                float2 X[R / 2][P2], Y[R / 2][P2];
#pragma unroll
                for (int r = 0; r < R / 2; ++r)
#pragma unroll
                    for (int m = 0; m < P2; ++m) {
                        X[r][m] = *reinterpret_cast<const float2 *>(scb + pair_off + (r * P2 + m) * 64);
                        Y[r][m] = *reinterpret_cast<const float2 *>(scb + pair_off + ((r + R / 2) * P2 + m) * 64);
                    }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kBarScbEmpty]);

                // ---- pass B: states before steps s0 .. s0+slen-2 to TMEM; the last stays in X, Y
                for (int j = 0; j + 1 < slen; ++j) {
                    const uint32_t ts = tmem + (uint32_t)(j * SW);
#pragma unroll
                    for (int q = 0; q < NPAIR / 8; ++q) {
                        float2 chunk[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int f = q * 8 + i;   // pair index in the state: rows 0-3 then rows 4-7
                            chunk[i] = f < NPAIR / 2 ? X[f / P2][f % P2] : Y[(f - NPAIR / 2) / P2][(f - NPAIR / 2) % P2];
                        }
                        tmem_st16(ts + q * 16, chunk);
                    }
                    const float gt = gs[j];
                    const float2 gg = make_float2(gt, gt);
                    float2 kv[P2];
#pragma unroll
                    for (int m = 0; m < P2; ++m) kv[m] = load_pair(kf + (j + 1) * DK, m);
#pragma unroll
                    for (int r = 0; r < R / 2; ++r) {
                        const float d0 = dl_s[(s0 - t0 + j) * RB + wrow + r];
                        const float d1 = dl_s[(s0 - t0 + j) * RB + wrow + r + R / 2];
                        const float2 dd0 = make_float2(d0, d0), dd1 = make_float2(d1, d1);
#pragma unroll
                        for (int m = 0; m < P2; ++m) {
                            X[r][m] = __ffma2_rn(dd0, kv[m], __fmul2_rn(gg, X[r][m]));
                            Y[r][m] = __ffma2_rn(dd1, kv[m], __fmul2_rn(gg, Y[r][m]));
                        }
                    }
                }
                tmem_wait_st();

                // half hh (0: rows 0-3, 1: rows 4-7) of the state before step s0 + j, from TMEM
                auto tmem_load_half = [&](int j, int hh, float2 (&dst)[R / 2][P2]) {
                    const uint32_t ts = tmem + (uint32_t)(j * SW + hh * (SW / 2));
#pragma unroll
                    for (int q = 0; q < NPAIR / 8; ++q) {   // NPAIR / 2 pairs in chunks of 4
                        float2 chunk[4];
                        tmem_ld8(ts + q * 8, chunk);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[(q * 4 + i) / P2][(q * 4 + i) % P2] = chunk[i];
                    }
                };

                // ---- core: reverse steps j = slen-1 .. 0
                for (int j = slen - 1; j >= 0; --j, ++gstep) {
                    const int tc = s0 + j - t0;
                    const float gt = gs[j], bt = gs[SUB + j];
                    // owner lane: ddelta of its row; then every lane takes all 8 rows' values
                    const float ddo = p_own + xr[j * RB + wrow + my_row] * gs[2 * SUB + j];
                    // this warp's rows of dy_t, delta_t and v_t - u_t (read per row, broadcast)
                    const float *dyw = xr + j * RB + wrow;
                    const float *dlw = dl_s + tc * RB + wrow;
                    const float *vmw = vm_s + tc * RB + wrow;
                    float2 kt[P2], qt[P2], kp[P2];
#pragma unroll
                    for (int m = 0; m < P2; ++m) {
                        kt[m] = load_pair(kf + (j + 1) * DK, m);
                        qt[m] = load_pair(qf + (j + 1) * DK, m);
                        kp[m] = load_pair(kf + j * DK, m);
                    }
                    float2 dkacc[P2], dqacc[P2];
#pragma unroll
                    for (int m = 0; m < P2; ++m) dkacc[m] = dqacc[m] = make_float2(0.f, 0.f);
                    float2 dg2 = make_float2(0.f, 0.f);
                    float s_dy = 0.f, s_db = 0.f;   // over the warp's rows: delta . dy and ddelta . (v - u)
                    float pn[R];
                    const float2 gg = make_float2(gt, gt);
                    // one row of the fused reverse step, with that row's S_{t-1} in sprow
                    auto row_step = [&](int r, const float2 (&sprow)[P2]) {
                        const float dd = __shfl_sync(kFullMask, ddo, 4 * r);
                        const float du = -bt * dd;
                        const float dyv = dyw[r], dlv = dlw[r];
                        s_dy = fmaf(dlv, dyv, s_dy);
                        s_db = fmaf(dd, vmw[r], s_db);
                        const float2 du2 = make_float2(du, du), dy2 = make_float2(dyv, dyv);
                        const float2 dr2 = make_float2(dlv, dlv);
                        const float2 gdu2 = make_float2(gt * du, gt * du), gdy2 = make_float2(gt * dyv, gt * dyv);
                        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                        for (int m = 0; m < P2; ++m) {
                            const float2 sp = sprow[m];
                            const float2 sc = __ffma2_rn(dy2, qt[m], Sh[r][m]);
                            dkacc[m] = __ffma2_rn(sc, dr2, dkacc[m]);
                            const float2 dA = __ffma2_rn(du2, kt[m], sc);
                            dg2 = __ffma2_rn(dA, sp, dg2);
                            dkacc[m] = __ffma2_rn(sp, gdu2, dkacc[m]);
                            dqacc[m] = __ffma2_rn(sp, gdy2, dqacc[m]);
                            const float2 shn = __fmul2_rn(gg, dA);
                            Sh[r][m] = shn;
                            acc = __ffma2_rn(shn, kp[m], acc);
                        }
                        pn[r] = acc.x + acc.y;
                    };
                    // rows 0-3 (X, in registers) while rows 4-7 load; then the next step's
                    // rows 0-3 load while rows 4-7 (Y) are used
                    const bool last_built = j == slen - 1;   // X, Y come from pass B
                    if (!last_built) tmem_load_half(j, 1, Y);
#pragma unroll
                    for (int r = 0; r < R / 2; ++r) row_step(r, X[r]);
                    if (!last_built) tmem_wait_ld();
                    if (j >= 1) tmem_load_half(j - 1, 0, X);
#pragma unroll
                    for (int r = 0; r < R / 2; ++r) row_step(r + R / 2, Y[r]);
                    if (j >= 1) tmem_wait_ld();

                    // hand the step's partials to the service warp
                    const int s = gstep % slots, n = gstep / slots;
                    if (n >= 1 && !mbar_wait(&bar[kBarSlotEmpty + s], (n - 1) & 1)) { failed = true; break; }
                    const float2 sdy2 = make_float2(s_dy, s_dy);   // dq_t also carries k_t (delta_t . dy_t)
                    float *cpw = slot_cp(s) + (size_t)warp * 2 * DK + pc;
#pragma unroll
                    for (int m = 0; m < P2; ++m) {
                        if (pvalid(m)) {
                            *reinterpret_cast<float2 *>(cpw + 64 * m) = dkacc[m];
                            *reinterpret_cast<float2 *>(cpw + DK + 64 * m) = __ffma2_rn(kt[m], sdy2, dqacc[m]);
                        }
                    }
                    const float dgs = warp_sum(dg2.x + dg2.y);
                    if (lane == 0) slot_gp(s)[warp] = make_float2(dgs, s_db);
                    if ((lane & 3) == 0) slot_dv(s)[wrow + my_row] = bt * ddo;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[kBarSlotFull + s]);
                    p_own = group_transpose_reduce<R, 32>(pn, lane);
                }
                if (failed) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kBarEmpty + bx]);
            }
        }

        if (!failed && p.dS0 != nullptr) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int row = row0 + wrow + r;
                if (row < Dv) {
                    float *dst = p.dS0 + (head * Dv + row) * DK;
#pragma unroll
                    for (int m = 0; m < P2; ++m)
                        if (pvalid(m)) *reinterpret_cast<float2 *>(dst + pc + 64 * m) = Sh[r][m];
                }
            }
        }
    }

    // ---- tear-down. After a timeout, wait (bounded) for the copies still in flight into
    // this CTA's shared memory before it exits; then release tensor memory.
    if (__syncthreads_or(failed)) {
        if (tid == 0) report_status(p.status, kStatusTimeout);
        if (warp == kStager && lane == 0) {
            for (int rb = 0; rb < 2; ++rb)
                if (raw_issued[rb] >= 1) mbar_wait(&bar[kBarRaw + rb], (raw_issued[rb] - 1) & 1);
            if (scb_loads >= 1) mbar_wait(&bar[kBarScb], (scb_loads - 1) & 1);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kStager) tmem_dealloc(*tslot, 512);
}

// dq[b,t,hk,:] = sum over h in the kv head's group (ascending) of the sum over row splits
// (ascending) of the per-CTA partials; the same for dk. dg and dbeta sum the row splits.
template <typename TOut>
__global__ void __launch_bounds__(256) reduce_kernel(ReduceParams p) {
    const size_t nqk = (size_t)p.B * p.T * p.Hk * p.Dk;
    const size_t ngate = (size_t)p.B * p.T * p.Hv;
    const int rep = p.Hv / p.Hk;
    TOut *dq = static_cast<TOut *>(p.dq);
    TOut *dk = static_cast<TOut *>(p.dk);
    TOut *dg = static_cast<TOut *>(p.dg);
    TOut *db = static_cast<TOut *>(p.dbeta);
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nqk + ngate;
         i += (size_t)gridDim.x * blockDim.x) {
        if (i < nqk) {
            const int j = (int)(i % p.Dk);
            const size_t bthk = i / p.Dk;
            const int hk = (int)(bthk % p.Hk);
            const size_t bt = bthk / p.Hk;
            float sq = 0.f, sk = 0.f;
            for (int h = hk * rep; h < (hk + 1) * rep; ++h) {
                float hq = 0.f, hkk = 0.f;
                for (int s = 0; s < p.nsplit; ++s) {
                    const size_t o = ((bt * p.Hv + h) * p.nsplit + s) * p.Dk + j;
                    hq += p.ws_dq[o];
                    hkk += p.ws_dk[o];
                }
                sq += hq;
                sk += hkk;
            }
            dq[i] = from_f32<TOut>(sq);
            dk[i] = from_f32<TOut>(sk);
        } else {
            const size_t gi = i - nqk;
            float sg = 0.f, sb = 0.f;
            for (int s = 0; s < p.nsplit; ++s) {
                sg += p.ws_dg[gi * p.nsplit + s];
                sb += p.ws_db[gi * p.nsplit + s];
            }
            dg[gi] = from_f32<TOut>(sg);
            db[gi] = from_f32<TOut>(sb);
        }
    }
}

size_t bwd_smem_bytes(int Dk, int C, int dtype, int slots) {
    return BwdSmem(Dk, dtype == 0 ? 4 : 2, C, slots).total;
}

int bwd_slots(int Dk, int C, int dtype, size_t limit) {
    for (int s = kMaxSlots; s >= 2; --s)
        if (bwd_smem_bytes(Dk, C, dtype, s) <= limit) return s;
    return 0;
}

template <int E, typename TIn>
static cudaError_t launch_bwd_t(const BwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk, cudaStream_t s) {
    if (p.slots < 2 || p.slots > kMaxSlots) return cudaErrorInvalidValue;
    // the register split waits for registers that only a launch of kBwdLaunchRegs per
    // thread provides
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, bwd_kernel<E, TIn>);
    if (err != cudaSuccess) return err;
    if (fa.numRegs < kBwdLaunchRegs || fa.maxThreadsPerBlock < kBwdThreads) return cudaErrorInvalidConfiguration;
    const size_t smem = bwd_smem_bytes(32 * E, p.C, IsF32B<TIn>::value ? 0 : 1, p.slots);
    err = cudaFuncSetAttribute(bwd_kernel<E, TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid(p.nsplit, p.Hv, p.B);
    timing_mark("seq_bwd", 0, s);
    bwd_kernel<E, TIn><<<grid, kBwdThreads, smem, s>>>(tq, tk, p);
    timing_mark("seq_bwd", 1, s);
    return cudaGetLastError();
}

template <typename TIn>
static cudaError_t launch_bwd_dk(const BwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk, int Dk,
                                 cudaStream_t s) {
    switch (Dk) {
        case 32: return launch_bwd_t<1, TIn>(p, tq, tk, s);
        case 64: return launch_bwd_t<2, TIn>(p, tq, tk, s);
        case 96: return launch_bwd_t<3, TIn>(p, tq, tk, s);
        case 128: return launch_bwd_t<4, TIn>(p, tq, tk, s);
        case 160: return launch_bwd_t<5, TIn>(p, tq, tk, s);
        case 192: return launch_bwd_t<6, TIn>(p, tq, tk, s);
        case 224: return launch_bwd_t<7, TIn>(p, tq, tk, s);
        case 256: return launch_bwd_t<8, TIn>(p, tq, tk, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd(const BwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k, int Dk, int dtype,
                       cudaStream_t s) {
    return dtype == 0 ? launch_bwd_dk<float>(p, tm_q, tm_k, Dk, s)
                      : launch_bwd_dk<__nv_bfloat16>(p, tm_q, tm_k, Dk, s);
}

cudaError_t launch_reduce(const ReduceParams &p, int dtype, cudaStream_t s) {
    const size_t n = (size_t)p.B * p.T * p.Hk * p.Dk + (size_t)p.B * p.T * p.Hv;
    const int threads = 256;
    const size_t want = (n + threads - 1) / threads;
    const int blocks = (int)(want < 152 * 16 ? want : 152 * 16);
    timing_mark("seq_reduce", 0, s);
    if (dtype == 0) reduce_kernel<float><<<blocks, threads, 0, s>>>(p);
    else reduce_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>(p);
    timing_mark("seq_reduce", 1, s);
    return cudaGetLastError();
}

}  // namespace gdn
