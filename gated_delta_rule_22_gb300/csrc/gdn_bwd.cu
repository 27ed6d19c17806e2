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
//   pass A  re-runs the chunk from its checkpoint, keeping delta_t and v_t - u_t per row
//           and step in shared memory and the state at the start of every sub-block of
//           SUB = bwd_sub(Dk) steps in an L2-resident scratch;
//   per sub-block, going backwards:
//     pass B  brings the sub-block's start state back (1-D TMA bulk copy, prefetched one
//             sub-block ahead) and re-builds the states inside it with the kept delta
//             (S <- g S + delta k^T), writing them to tensor memory (TMEM); the last one
//             stays in registers;
//     core    runs the reverse steps, reading S_{t-1} from TMEM in two halves (rows 0-3,
//             rows 4-7 of each warp) so that one half loads while the other is used.
//
// Layout: a CTA owns RB = 8 * warps rows of one (b, h); a warp owns 8 rows; lane l holds
// the column pairs (2l + 64m, 2l + 1 + 64m) of each row, so row dot products are 32-lane
// reductions and a warp's column sums are complete per lane. Each warp folds the row
// sums delta . dy and ddelta . (v - u) of its rows into its partials in the same pass;
// column sums (dq, dk), dg and dbeta are then reduced over the warps in shared memory in
// ascending warp order and written per (b, t, h, row split) to fp32 scratch;
// reduce_kernel adds the row splits (ascending) and the value heads of each kv head
// (ascending). No atomics.
//
// Staging: k and q tiles of SUB + 1 steps arrive by TMA (tiled tensor maps, one tile
// ahead, two buffers); v or dy, g and beta are loaded one tile ahead into registers.
#include "gdn_common.cuh"

namespace gdn {

namespace {

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
    size_t raw, kf, scb, dl, vm, xs, dd, cp, gp, gs, bs, kq, bar, tslot, total;
    __host__ __device__ BwdSmem(int DK, int RB, int nw, int esize, int C, int F) {
        const int P2 = bwd_pairs(DK), SUB = bwd_sub(DK), TR = SUB + 1;
        size_t o = 0;
        raw = o; o += align_upb((size_t)2 * 2 * TR * DK * esize, 128);   // [buf][k|q][TR][DK], input type
        kf = o; if (esize != 4) o += (size_t)2 * TR * DK * 4;              // widened k rows then q rows
        o = align_upb(o, 128);
        scb = o; o += (size_t)RB * P2 * 64 * 4;                            // incoming sub-block start state
        dl = o; o += (size_t)C * RB * 4;
        vm = o; o += (size_t)C * RB * 4;
        xs = o; o += (size_t)SUB * RB * 4;                                  // v (pass A) or dy (reverse)
        dd = o; o += (size_t)SUB * RB * 4;
        cp = o; o += (size_t)F * nw * 2 * DK * 4;                           // [F][warp][dk|dq][DK]
        gp = o; o += (size_t)F * nw * 8;                                    // [F][warp] (dg, dbeta)
        gs = o; o += SUB * 4;
        bs = o; o += SUB * 4;
        kq = o; o += SUB * 4;
        bar = align_upb(o, 8); o = bar + 3 * 8;
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
__global__ void __launch_bounds__(256, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, BwdParams p) {
    constexpr int R = kBwdRowsPerWarp;
    constexpr int DK = 32 * E;
    constexpr int P2 = bwd_pairs(DK);
    constexpr int SUB = bwd_sub(DK);
    constexpr int TR = SUB + 1;
    constexpr int NPAIR = R * P2;         // float2 pairs of one state per thread
    constexpr int SW = 2 * NPAIR;         // TMEM columns of one state per thread
    constexpr bool kConv = !IsF32B<TIn>::value;
    constexpr bool kOdd = (DK % 64) != 0;   // the last pair exists only on lanes 0..15
    using QuadT = typename QuadB<TIn>::type;
    static_assert(NPAIR % 8 == 0, "state must be a whole number of 16-column TMEM chunks");
    static_assert((SUB - 1) * SW <= 256, "sub-block states exceed the TMEM share");

    const int tid = threadIdx.x, nthreads = blockDim.x, nw = nthreads >> 5;
    const int warp = tid >> 5, lane = tid & 31;
    const int RB = nw * R;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int row0 = split * RB, hk = h / (p.Hv / p.Hk);
    const int T = p.T, Dv = p.Dv, C = p.C, Hv = p.Hv, nsplit = p.nsplit, F = p.flush;
    const int wrow = warp * R;
    const int my_row = lane >> 2;         // row held by this lane after a transpose reduction of 8

    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(align_upb(reinterpret_cast<size_t>(smem_raw), 128));
    const BwdSmem L(DK, RB, nw, (int)sizeof(TIn), C, F);
    TIn *raw = reinterpret_cast<TIn *>(base + L.raw);
    float *kfq = reinterpret_cast<float *>(base + L.kf);   // widened k rows then q rows (bf16 input)
    float *scb = reinterpret_cast<float *>(base + L.scb);
    float *dl_s = reinterpret_cast<float *>(base + L.dl);
    float *vm_s = reinterpret_cast<float *>(base + L.vm);
    float *xs = reinterpret_cast<float *>(base + L.xs);
    float *dd_s = reinterpret_cast<float *>(base + L.dd);
    float *cp_s = reinterpret_cast<float *>(base + L.cp);
    float2 *gp_s = reinterpret_cast<float2 *>(base + L.gp);
    float *g_s = reinterpret_cast<float *>(base + L.gs);
    float *b_s = reinterpret_cast<float *>(base + L.bs);
    float *kq_s = reinterpret_cast<float *>(base + L.kq);
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + L.bar);   // [0], [1]: tiles; [2]: sub-block state
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + L.tslot);

    const TIn *v = static_cast<const TIn *>(p.v);
    const TIn *g = static_cast<const TIn *>(p.g);
    const TIn *beta = static_cast<const TIn *>(p.beta);
    const TIn *dy = static_cast<const TIn *>(p.dy);
    const TIn *k = static_cast<const TIn *>(p.k);
    TIn *dv = static_cast<TIn *>(p.dv);

    const size_t head = (size_t)b * Hv + h;
    const size_t cta = head * nsplit + split;
    const size_t slot_floats = (size_t)RB * P2 * 64;
    float *scratch = p.ws_state + cta * (size_t)p.nsub_max * slot_floats;
    const int pair_off = wrow * P2 * 64 + 2 * lane;   // this thread's pair (r, m) is at + (r * P2 + m) * 64
    const int pc = 2 * lane;                          // first column of this lane's pair 0
    auto pvalid = [&](int m) { return !kOdd || m < P2 - 1 || lane < 16; };

    // ---- set-up: barriers, tensor memory
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init(&bar[2], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * 256);

    auto nsub_of = [&](int c) {
        const int len = min(C, T - c * C);
        return (len + SUB - 1) / SUB;
    };
    auto tile_after = [&](TileRef t) -> TileRef {
        if (t.kind == 0) {
            if (t.m + 1 < nsub_of(t.c)) return {0, t.c, t.m + 1};
            return {1, t.c, nsub_of(t.c) - 1};
        }
        if (t.m > 0) return {1, t.c, t.m - 1};
        if (t.c > 0) return {0, t.c - 1, 0};
        return {-1, 0, 0};
    };

    // register prefetch of one tile's per-row input (v for pass A, dy for reverse), g, beta
    const int nquads = SUB * (RB / 4);
    QuadT xq = QuadB<TIn>::zero();
    float gq = 1.f, bq = 0.f;
    auto issue_tile = [&](TileRef t, int buf) {
        const int s0 = t.c * C + t.m * SUB;
        const int slen = min(SUB, min(t.c * C + C, T) - s0);
        if (tid == 0) {
            fence_proxy_async();
            TIn *dst = raw + (size_t)buf * 2 * TR * DK;
            mbar_expect_tx(&bar[buf], (t.kind == 1 ? 2u : 1u) * TR * DK * (unsigned)sizeof(TIn));
            tma_load_4d(dst, &tm_k, &bar[buf], 0, hk, s0 - 1, b);
            if (t.kind == 1) tma_load_4d(dst + TR * DK, &tm_q, &bar[buf], 0, hk, s0 - 1, b);
        }
        const TIn *x = t.kind == 1 ? dy : v;
        xq = QuadB<TIn>::zero();
        if (tid < nquads) {
            const int j = tid / (RB / 4), r4 = (tid % (RB / 4)) * 4;
            if (j < slen && row0 + r4 < Dv)
                xq = *reinterpret_cast<const QuadT *>(x + ((((size_t)b * T + s0 + j) * Hv + h) * Dv + row0 + r4));
        }
        if (tid < SUB) {
            gq = tid < slen ? to_f32(g[((size_t)b * T + s0 + tid) * Hv + h]) : 1.f;
            bq = tid < slen ? to_f32(beta[((size_t)b * T + s0 + tid) * Hv + h]) : 0.f;
        }
    };
    // Consume the tile in `buf`: stage the prefetched registers, wait for and widen the TMA
    // rows into the pair layout, then start the next tile. Returns false on a timeout.
    unsigned tile_phase0 = 0u, tile_phase1 = 0u;
    auto begin_tile = [&](TileRef t, int buf) -> bool {
        __syncthreads();   // the previous tile's staging buffers are no longer read
        if (tid < nquads) {
            const float4 f = QuadB<TIn>::unpack(xq);
            *reinterpret_cast<float4 *>(xs + (tid / (RB / 4)) * RB + (tid % (RB / 4)) * 4) = f;
        }
        if (tid < SUB) {
            g_s[tid] = gq;
            b_s[tid] = bq;
        }
        const bool ok = mbar_wait(&bar[buf], buf ? tile_phase1 : tile_phase0);
        if (buf) tile_phase1 ^= 1u;
        else tile_phase0 ^= 1u;
        if (ok && kConv) {
            // widen 8 bf16 (16 bytes) at a time: k rows then q rows
            const uint4 *src = reinterpret_cast<const uint4 *>(raw + (size_t)buf * 2 * TR * DK);
            const int nchunks = (t.kind == 1 ? 2 * TR : TR) * DK / 8;
            for (int i = tid; i < nchunks; i += nthreads) {
                const uint4 w = src[i];
                float4 *dst = reinterpret_cast<float4 *>(kfq + 8 * i);
                dst[0] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
                dst[1] = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u),
                                     __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
            }
        }
        if (__syncthreads_or(!ok)) return false;
        const TileRef nt = tile_after(t);
        if (nt.kind >= 0) issue_tile(nt, buf ^ 1);
        return true;
    };
    // row tiles of the current tile: k rows 0..TR-1 (row i = step s0 - 1 + i), q rows likewise
    const float *kf = kfq, *qf = kfq + TR * DK;
    auto set_tile_rows = [&](int buf) {
        if (!kConv) {
            kf = reinterpret_cast<const float *>(raw + (size_t)buf * 2 * TR * DK);
            qf = kf + TR * DK;
        }
    };
    auto load_pair = [&](const float *rowbase, int m) {
        return pvalid(m) ? *reinterpret_cast<const float2 *>(rowbase + pc + 64 * m) : make_float2(0.f, 0.f);
    };

    // ---- adjoint state Sh from dS_T, and its first row dot with k_{T-1}
    float2 Sh[R][P2];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int row = row0 + wrow + r;
#pragma unroll
        for (int m = 0; m < P2; ++m) {
            Sh[r][m] = (p.dS_T != nullptr && row < Dv && pvalid(m))
                           ? *reinterpret_cast<const float2 *>(p.dS_T + (head * Dv + row) * DK + pc + 64 * m)
                           : make_float2(0.f, 0.f);
        }
    }
    float p_own;   // Sh . k_t of row my_row, for the next reverse step t
    {
        float part[R];
        float2 kk[P2];
#pragma unroll
        for (int m = 0; m < P2; ++m) {
            const TIn *src = k + (((size_t)b * T + T - 1) * p.Hk + hk) * DK;
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

    bool failed = false;
    unsigned scb_phase = 0u;
    int buf = 0;
    issue_tile(TileRef{0, p.NC - 1, 0}, 0);

    for (int c = p.NC - 1; c >= 0 && !failed; --c) {
        const int t0 = c * C, len = min(C, T - t0), nsub = (len + SUB - 1) / SUB;

        // ============ pass A: forward through the chunk from its checkpoint ============
        float2 S[R][P2];
        {
            const float *ck = p.ckpt + (head * p.NC + c) * (size_t)Dv * DK;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int row = row0 + wrow + r;
#pragma unroll
                for (int m = 0; m < P2; ++m) {
                    S[r][m] = (row < Dv && pvalid(m))
                                  ? *reinterpret_cast<const float2 *>(ck + (size_t)row * DK + pc + 64 * m)
                                  : make_float2(0.f, 0.f);
                }
            }
        }
        for (int m = 0; m < nsub; ++m) {
            const int s0 = t0 + m * SUB, slen = min(SUB, t0 + len - s0);
            if (!begin_tile(TileRef{0, c, m}, buf)) { failed = true; break; }
            set_tile_rows(buf);
            float *slot = scratch + (size_t)m * slot_floats + pair_off;
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int mm = 0; mm < P2; ++mm) *reinterpret_cast<float2 *>(slot + (r * P2 + mm) * 64) = S[r][mm];
            for (int j = 0; j < slen; ++j) {
                float2 kv[P2];
#pragma unroll
                for (int mm = 0; mm < P2; ++mm) kv[mm] = load_pair(kf + (j + 1) * DK, mm);
                float part[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int mm = 0; mm < P2; ++mm) acc = __ffma2_rn(S[r][mm], kv[mm], acc);
                    part[r] = acc.x + acc.y;
                }
                const float a = group_transpose_reduce<R, 32>(part, lane);
                const float gt = g_s[j], bt = b_s[j];
                const float vmv = xs[j * RB + wrow + my_row] - gt * a;
                const float dlv = bt * vmv;
                if ((lane & 3) == 0) {
                    dl_s[(s0 - t0 + j) * RB + wrow + my_row] = dlv;
                    vm_s[(s0 - t0 + j) * RB + wrow + my_row] = vmv;
                }
                const float2 gg = make_float2(gt, gt);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float d = __shfl_sync(kFullMask, dlv, 4 * r);
                    const float2 dd = make_float2(d, d);
#pragma unroll
                    for (int mm = 0; mm < P2; ++mm) S[r][mm] = __ffma2_rn(dd, kv[mm], __fmul2_rn(gg, S[r][mm]));
                }
            }
            buf ^= 1;
        }
        if (failed) break;
        fence_proxy_async_global();   // the sub-block start states are read back by TMA

        // ============ reverse sweep over the chunk's sub-blocks ============
        for (int m = nsub - 1; m >= 0; --m) {
            const int s0 = t0 + m * SUB, slen = min(SUB, t0 + len - s0);
            if (!begin_tile(TileRef{1, c, m}, buf)) { failed = true; break; }
            set_tile_rows(buf);
            if (m == nsub - 1 && tid == 0) {
                mbar_expect_tx(&bar[2], (unsigned)(slot_floats * 4));
                bulk_load(scb, scratch + (size_t)m * slot_floats, (unsigned)(slot_floats * 4), &bar[2]);
            }
            // per-step k_t . q_t
            for (int j = warp; j < slen; j += nw) {
                float a = 0.f;
                for (int i = lane; i < DK; i += 32) a = fmaf(kf[(j + 1) * DK + i], qf[(j + 1) * DK + i], a);
                a = warp_sum(a);
                if (lane == 0) kq_s[j] = a;
            }
            // the sub-block's start state
            const bool ok = mbar_wait(&bar[2], scb_phase);
            scb_phase ^= 1u;
            // the state of the warp's rows 0-3 (X) and rows 4-7 (Y)
            float2 X[R / 2][P2], Y[R / 2][P2];
#pragma unroll
            for (int r = 0; r < R / 2; ++r)
#pragma unroll
                for (int mm = 0; mm < P2; ++mm) {
                    X[r][mm] = *reinterpret_cast<const float2 *>(scb + pair_off + (r * P2 + mm) * 64);
                    Y[r][mm] = *reinterpret_cast<const float2 *>(scb + pair_off + ((r + R / 2) * P2 + mm) * 64);
                }
            if (__syncthreads_or(!ok)) { failed = true; break; }
            if (m > 0 && tid == 0) {
                fence_proxy_async();
                mbar_expect_tx(&bar[2], (unsigned)(slot_floats * 4));
                bulk_load(scb, scratch + (size_t)(m - 1) * slot_floats, (unsigned)(slot_floats * 4), &bar[2]);
            }

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
                const float gt = g_s[j];
                const float2 gg = make_float2(gt, gt);
                float2 kv[P2];
#pragma unroll
                for (int mm = 0; mm < P2; ++mm) kv[mm] = load_pair(kf + (j + 1) * DK, mm);
#pragma unroll
                for (int r = 0; r < R / 2; ++r) {
                    const float d0 = dl_s[(s0 - t0 + j) * RB + wrow + r];
                    const float d1 = dl_s[(s0 - t0 + j) * RB + wrow + r + R / 2];
                    const float2 dd0 = make_float2(d0, d0), dd1 = make_float2(d1, d1);
#pragma unroll
                    for (int mm = 0; mm < P2; ++mm) {
                        X[r][mm] = __ffma2_rn(dd0, kv[mm], __fmul2_rn(gg, X[r][mm]));
                        Y[r][mm] = __ffma2_rn(dd1, kv[mm], __fmul2_rn(gg, Y[r][mm]));
                    }
                }
            }
            tmem_wait_st();

            // ---- core: reverse steps j = slen-1 .. 0, S_{t-1} in Sa / Sb alternately
            // half h (0: rows 0-3, 1: rows 4-7) of the state before step s0 + j, from TMEM
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
            // Reduce the warps' partials of steps jlo .. jhi (the batch's highest step, jhi, sits
            // in partial slot 0; step j in slot jhi - j), write them out, and free the slots.
            auto flush = [&](int jlo, int jhi) {
                __syncthreads();
                const int nst = jhi - jlo + 1;
                for (int i = tid; i < nst * (DK / 4); i += nthreads) {
                    const int jj = i / (DK / 4), c4 = (i - jj * (DK / 4)) * 4;
                    const int j = jhi - jj, t = s0 + j;
                    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), q4 = a;
#pragma unroll
                    for (int w = 0; w < kBwdMaxWarps; ++w) {
                        if (w < nw) {
                            const float4 x = *reinterpret_cast<const float4 *>(cp_s + ((size_t)(jj * nw + w) * 2) * DK + c4);
                            const float4 y = *reinterpret_cast<const float4 *>(cp_s + ((size_t)(jj * nw + w) * 2 + 1) * DK + c4);
                            a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
                            q4.x += y.x; q4.y += y.y; q4.z += y.z; q4.w += y.w;
                        }
                    }
                    const size_t o = ((((size_t)b * T + t) * Hv + h) * nsplit + split) * DK + c4;
                    *reinterpret_cast<float4 *>(p.ws_dk + o) = a;
                    *reinterpret_cast<float4 *>(p.ws_dq + o) = q4;
                }
                if (tid < nst) {
                    const int jj = tid, j = jhi - jj, t = s0 + j;
                    float dgs = 0.f, dbs = 0.f;
#pragma unroll
                    for (int w = 0; w < kBwdMaxWarps; ++w) {
                        if (w < nw) {
                            dgs += gp_s[jj * nw + w].x;
                            dbs += gp_s[jj * nw + w].y;
                        }
                    }
                    const size_t o = (((size_t)b * T + t) * Hv + h) * nsplit + split;
                    p.ws_dg[o] = dgs;
                    p.ws_db[o] = dbs;
                }
                for (int i = tid; i < nst * RB; i += nthreads) {
                    const int jj = i / RB, rr = i - jj * RB, j = jhi - jj, row = row0 + rr;
                    if (row < Dv)
                        dv[(((size_t)b * T + s0 + j) * Hv + h) * Dv + row] = from_f32<TIn>(b_s[j] * dd_s[j * RB + rr]);
                }
                __syncthreads();
            };
            int jf = 0;   // partial slot of the next core step
            auto core_step = [&](int j) {
                const int tc = s0 + j - t0;
                const float gt = g_s[j], bt = b_s[j];
                // owner lane: ddelta of its row; then every lane takes all 8 rows' values
                const float ddo = p_own + xs[j * RB + wrow + my_row] * kq_s[j];
                if ((lane & 3) == 0) dd_s[j * RB + wrow + my_row] = ddo;
                float dyr[R], drr[R], vmr[R];
#pragma unroll
                for (int h4 = 0; h4 < R / 4; ++h4) {
                    const float4 a = *reinterpret_cast<const float4 *>(xs + j * RB + wrow + 4 * h4);
                    const float4 d = *reinterpret_cast<const float4 *>(dl_s + tc * RB + wrow + 4 * h4);
                    const float4 u = *reinterpret_cast<const float4 *>(vm_s + tc * RB + wrow + 4 * h4);
                    dyr[4 * h4] = a.x; dyr[4 * h4 + 1] = a.y; dyr[4 * h4 + 2] = a.z; dyr[4 * h4 + 3] = a.w;
                    drr[4 * h4] = d.x; drr[4 * h4 + 1] = d.y; drr[4 * h4 + 2] = d.z; drr[4 * h4 + 3] = d.w;
                    vmr[4 * h4] = u.x; vmr[4 * h4 + 1] = u.y; vmr[4 * h4 + 2] = u.z; vmr[4 * h4 + 3] = u.w;
                }
                float2 kt[P2], qt[P2], kp[P2];
#pragma unroll
                for (int mm = 0; mm < P2; ++mm) {
                    kt[mm] = load_pair(kf + (j + 1) * DK, mm);
                    qt[mm] = load_pair(qf + (j + 1) * DK, mm);
                    kp[mm] = load_pair(kf + j * DK, mm);
                }
                float2 dkacc[P2], dqacc[P2];
#pragma unroll
                for (int mm = 0; mm < P2; ++mm) dkacc[mm] = dqacc[mm] = make_float2(0.f, 0.f);
                float2 dg2 = make_float2(0.f, 0.f);
                float s_dy = 0.f, s_db = 0.f;   // sum over the warp's rows of delta.dy and ddelta.(v - u)
                float pn[R];
                const float2 gg = make_float2(gt, gt);
                // one row of the fused reverse step, with that row's S_{t-1} in sprow
                auto row_step = [&](int r, const float2 (&sprow)[P2]) {
                    const float dd = __shfl_sync(kFullMask, ddo, 4 * r);
                    const float du = -bt * dd;
                    s_dy = fmaf(drr[r], dyr[r], s_dy);
                    s_db = fmaf(dd, vmr[r], s_db);
                    const float2 du2 = make_float2(du, du), dy2 = make_float2(dyr[r], dyr[r]);
                    const float2 dr2 = make_float2(drr[r], drr[r]);
                    const float2 gdu2 = make_float2(gt * du, gt * du), gdy2 = make_float2(gt * dyr[r], gt * dyr[r]);
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int mm = 0; mm < P2; ++mm) {
                        const float2 sp = sprow[mm];
                        const float2 sc = __ffma2_rn(dy2, qt[mm], Sh[r][mm]);
                        dkacc[mm] = __ffma2_rn(sc, dr2, dkacc[mm]);
                        const float2 dA = __ffma2_rn(du2, kt[mm], sc);
                        dg2 = __ffma2_rn(dA, sp, dg2);
                        dkacc[mm] = __ffma2_rn(sp, gdu2, dkacc[mm]);
                        dqacc[mm] = __ffma2_rn(sp, gdy2, dqacc[mm]);
                        const float2 shn = __fmul2_rn(gg, dA);
                        Sh[r][mm] = shn;
                        acc = __ffma2_rn(shn, kp[mm], acc);
                    }
                    pn[r] = acc.x + acc.y;
                };
                // rows 0-3 (X, already in registers) while rows 4-7 load; then the next step's
                // rows 0-3 load while rows 4-7 (Y) are used
                const bool first = j == slen - 1;   // X, Y come from pass B
                if (!first) tmem_load_half(j, 1, Y);
#pragma unroll
                for (int r = 0; r < R / 2; ++r) row_step(r, X[r]);
                if (!first) tmem_wait_ld();
                if (j >= 1) tmem_load_half(j - 1, 0, X);
#pragma unroll
                for (int r = 0; r < R / 2; ++r) row_step(r + R / 2, Y[r]);
                if (j >= 1) tmem_wait_ld();
                // dq_t also carries k_t (delta_t . dy_t) over the warp's rows
                const float2 sdy2 = make_float2(s_dy, s_dy);
                float *cpw = cp_s + (size_t)(jf * nw + warp) * 2 * DK + pc;
#pragma unroll
                for (int mm = 0; mm < P2; ++mm) {
                    if (pvalid(mm)) {
                        *reinterpret_cast<float2 *>(cpw + 64 * mm) = dkacc[mm];
                        *reinterpret_cast<float2 *>(cpw + DK + 64 * mm) = __ffma2_rn(kt[mm], sdy2, dqacc[mm]);
                    }
                }
                const float dgs = warp_sum(dg2.x + dg2.y);
                if (lane == 0) gp_s[jf * nw + warp] = make_float2(dgs, s_db);
                p_own = group_transpose_reduce<R, 32>(pn, lane);
                if (jf == F - 1 || j == 0) {
                    flush(j, j + jf);
                    jf = 0;
                } else {
                    ++jf;
                }
            };
            for (int j = slen - 1; j >= 0; --j) core_step(j);
            buf ^= 1;
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
    if (failed && tid == 0) report_status(p.status, kStatusTimeout);
    // release tensor memory on every path
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(*tslot, 512);
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

size_t bwd_smem_bytes(int Dk, int warps, int C, int F, int dtype) {
    return BwdSmem(Dk, warps * kBwdRowsPerWarp, warps, dtype == 0 ? 4 : 2, C, F).total;
}

template <int E, typename TIn>
static cudaError_t launch_bwd_t(const BwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk, int warps,
                                cudaStream_t s) {
    const size_t smem = bwd_smem_bytes(32 * E, warps, p.C, p.flush, IsF32B<TIn>::value ? 0 : 1);
    cudaError_t err = cudaFuncSetAttribute(bwd_kernel<E, TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid(p.nsplit, p.Hv, p.B);
    bwd_kernel<E, TIn><<<grid, warps * 32, smem, s>>>(tq, tk, p);
    return cudaGetLastError();
}

template <typename TIn>
static cudaError_t launch_bwd_dk(const BwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk, int Dk,
                                 int warps, cudaStream_t s) {
    switch (Dk) {
        case 32: return launch_bwd_t<1, TIn>(p, tq, tk, warps, s);
        case 64: return launch_bwd_t<2, TIn>(p, tq, tk, warps, s);
        case 96: return launch_bwd_t<3, TIn>(p, tq, tk, warps, s);
        case 128: return launch_bwd_t<4, TIn>(p, tq, tk, warps, s);
        case 160: return launch_bwd_t<5, TIn>(p, tq, tk, warps, s);
        case 192: return launch_bwd_t<6, TIn>(p, tq, tk, warps, s);
        case 224: return launch_bwd_t<7, TIn>(p, tq, tk, warps, s);
        case 256: return launch_bwd_t<8, TIn>(p, tq, tk, warps, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd(const BwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k, int Dk, int dtype,
                       int warps, cudaStream_t s) {
    return dtype == 0 ? launch_bwd_dk<float>(p, tm_q, tm_k, Dk, warps, s)
                      : launch_bwd_dk<__nv_bfloat16>(p, tm_q, tm_k, Dk, warps, s);
}

cudaError_t launch_reduce(const ReduceParams &p, int dtype, cudaStream_t s) {
    const size_t n = (size_t)p.B * p.T * p.Hk * p.Dk + (size_t)p.B * p.T * p.Hv;
    const int threads = 256;
    const size_t want = (n + threads - 1) / threads;
    const int blocks = (int)(want < 152 * 16 ? want : 152 * 16);
    if (dtype == 0) reduce_kernel<float><<<blocks, threads, 0, s>>>(p);
    else reduce_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
