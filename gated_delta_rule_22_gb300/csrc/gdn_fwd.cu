// gdn_fwd.cu -- forward of the gated delta rule with chunk checkpoints.
//
// Recurrence (mlx issue #4614, "Recurrence used for the references"), per value head h
// with kv head h / (Hv/Hk):  S <- g_t S;  S <- S + (beta_t (v_t - S k_t)) k_t^T;
// y_t = S q_t.  Checkpoints (mlx-lm PR #1217, "What this PR adds"): the state before
// every C-th step is written to HBM for the reverse sweep.
//
// One CTA owns RB = 8 * warps rows of one (b, h) state and keeps them in registers for
// the whole sequence. A warp holds 8 rows as two groups of 16 lanes; each lane holds
// 4 rows x Dk/16 columns (column pairs 2j, 2j+1 + 32m), so a row dot product is a
// 16-lane reduction. Per step every element is read and written once, in packed f32x2
// arithmetic (one instruction per two elements):
//     S_t = g_t S_{t-1} + delta_t k_t^T           (FMUL2 + FFMA2)
//     ya  = S_t . q_t      -> y_t                   (FFMA2)
//     an  = S_t . k_{t+1}  -> prediction u_{t+1} = g_{t+1} an   (FFMA2)
// The 8 row partials (4 rows x {ya, an}) are reduced across the 16 lanes by a transpose
// reduction; the lane that ends up with row r's `an` computes
// delta_{t+1} = beta_{t+1} (v_{t+1} - g_{t+1} an) and shares it with a shuffle.
//
// Residuals: v_t - u_t of every step and row is kept (fp32, staged per tile like y) for the
// backward, whose re-computation then applies the same delta_t = beta_t (v_t - u_t) as the
// forward instead of forming the prediction dot again.
//
// Staging: k and q arrive by TMA (tiled 4-D tensor maps, one tile of kFwdTile steps
// ahead, two buffers, mbarrier completion); v, g and beta are loaded one tile ahead into
// registers. Each tile starts with a prediction dot against its first k, so no tile
// needs its successor's data.
#include "gdn_common.cuh"

namespace gdn {

namespace {

constexpr int kRowsF = 4;    // rows per thread
constexpr int kGroupF = 16;  // lanes per row group

template <typename T>
struct IsF32 { static constexpr bool value = false; };
template <>
struct IsF32<float> { static constexpr bool value = true; };

// four consecutive elements of v, as loaded in one vector access
template <typename T>
struct Quad;
template <>
struct Quad<float> {
    using type = float4;
    static __device__ __forceinline__ type zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    static __device__ __forceinline__ void unpack(const type &q, float (&o)[4]) {
        o[0] = q.x; o[1] = q.y; o[2] = q.z; o[3] = q.w;
    }
};
template <>
struct Quad<__nv_bfloat16> {
    using type = uint2;
    static __device__ __forceinline__ type zero() { return make_uint2(0u, 0u); }
    static __device__ __forceinline__ void unpack(const type &q, float (&o)[4]) {
        o[0] = __uint_as_float(q.x << 16); o[1] = __uint_as_float(q.x & 0xffff0000u);
        o[2] = __uint_as_float(q.y << 16); o[3] = __uint_as_float(q.y & 0xffff0000u);
    }
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared-memory layout of fwd_kernel (byte offsets from a 128-byte aligned base).
struct FwdSmem {
    size_t raw, fk, fq, fv, fy, fr, fg, fb, bar, total;
    __host__ __device__ FwdSmem(int DK, int RB, int esize, bool conv) {
        const int TS = kFwdTile;
        size_t o = 0;
        raw = o; o += align_up((size_t)2 * 2 * TS * DK * esize, 128);     // [buf][k|q][TS][DK]
        fk = o; if (conv) o += (size_t)(TS + 1) * DK * 4;                  // fp32 k rows (+1 spare)
        fq = o; if (conv) o += (size_t)TS * DK * 4;                        // fp32 q rows
        fv = o; o += (size_t)TS * RB * 4;
        fy = o; o += (size_t)TS * RB * 4;
        fr = o; o += (size_t)TS * RB * 4;                                  // v - u per step and row
        fg = o; o += TS * 4;
        fb = o; o += TS * 4;
        bar = align_up(o, 8); o = bar + 2 * 8;
        total = o + 128;                                                   // + alignment slack
    }
};

}  // namespace

template <int P, typename TIn>
__global__ void __launch_bounds__(256, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, FwdParams p) {
    constexpr int R = kRowsF, G = kGroupF, DK = 32 * P, TS = kFwdTile;
    constexpr bool kConv = !IsF32<TIn>::value;
    using QuadT = typename Quad<TIn>::type;
    const int tid = threadIdx.x, nthreads = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, gl = lane & (G - 1);
    const int RB = (nthreads >> 5) * 8;
    const int b = blockIdx.z, h = blockIdx.y, row0 = blockIdx.x * RB;
    const int hk = h / (p.Hv / p.Hk);
    const int T = p.T, Dv = p.Dv, Hv = p.Hv;
    const int lrow = warp * 8 + (lane >> 4) * R;          // first CTA-local row of this thread
    const int own_row = lrow + (gl >> 2);                  // row whose reduced sums this lane holds
    const int col = 2 * gl;                                // first column of this lane's pairs

    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(align_up(reinterpret_cast<size_t>(smem_raw), 128));
    const FwdSmem L(DK, RB, (int)sizeof(TIn), kConv);
    TIn *raw = reinterpret_cast<TIn *>(base + L.raw);
    float *fk = reinterpret_cast<float *>(base + L.fk);
    float *fq = reinterpret_cast<float *>(base + L.fq);
    float *fv = reinterpret_cast<float *>(base + L.fv);
    float *fy = reinterpret_cast<float *>(base + L.fy);
    float *fr = reinterpret_cast<float *>(base + L.fr);
    float *fg = reinterpret_cast<float *>(base + L.fg);
    float *fb = reinterpret_cast<float *>(base + L.fb);
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + L.bar);

    const TIn *v = static_cast<const TIn *>(p.v);
    const TIn *g = static_cast<const TIn *>(p.g);
    const TIn *beta = static_cast<const TIn *>(p.beta);
    TIn *y = static_cast<TIn *>(p.y);
    const size_t head = (size_t)b * Hv + h;
    const int ntiles = (T + TS - 1) / TS;
    const unsigned tile_bytes = 2u * TS * DK * sizeof(TIn);

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    if (kConv)
        for (int i = tid; i < DK; i += nthreads) fk[TS * DK + i] = 0.f;   // spare row, never a real k
    __syncthreads();
    if (tid == 0) {
        mbar_expect_tx(&bar[0], tile_bytes);
        tma_load_4d(raw, &tm_k, &bar[0], 0, hk, 0, b);
        tma_load_4d(raw + TS * DK, &tm_q, &bar[0], 0, hk, 0, b);
    }

    // v (groups of 4 consecutive rows of one step), g and beta of a tile, one tile ahead.
    // A tile holds TS * RB / 4 = (TS / 16) * nthreads quads: QPT per thread.
    constexpr int QPT = TS / 16;
    QuadT vq[QPT];
    float gq = 1.f, bq = 0.f;
    auto prefetch = [&](int i) {
#pragma unroll
        for (int j = 0; j < QPT; ++j) {
            const int qd = tid + j * nthreads, q_tt = qd / (RB / 4), q_r = (qd % (RB / 4)) * 4;
            const int t = i * TS + q_tt;
            vq[j] = Quad<TIn>::zero();
            if (t < T && row0 + q_r < Dv)
                vq[j] = *reinterpret_cast<const QuadT *>(v + ((((size_t)b * T + t) * Hv + h) * Dv + row0 + q_r));
        }
        if (tid < TS) {
            const int tg = i * TS + tid;
            gq = tg < T ? to_f32(g[((size_t)b * T + tg) * Hv + h]) : 1.f;
            bq = tg < T ? to_f32(beta[((size_t)b * T + tg) * Hv + h]) : 0.f;
        }
    };
    prefetch(0);

    float2 S[R][P];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int row = row0 + lrow + r;
#pragma unroll
        for (int m = 0; m < P; ++m)
            S[r][m] = (p.S0 != nullptr && row < Dv)
                          ? *reinterpret_cast<const float2 *>(p.S0 + (head * Dv + row) * DK + col + 32 * m)
                          : make_float2(0.f, 0.f);
    }
    float delta[R];      // delta_t of the thread's 4 rows
    int to_ckpt = 0;     // steps until the next checkpoint

    for (int i = 0; i < ntiles; ++i) {
        const int t0 = i * TS, tl = min(TS, T - t0);
        const int buf = i & 1;
        // stage the prefetched registers; wait for and widen this tile's k and q
#pragma unroll
        for (int j = 0; j < QPT; ++j) {
            const int qd = tid + j * nthreads;
            float o[4];
            Quad<TIn>::unpack(vq[j], o);
            *reinterpret_cast<float4 *>(fv + (qd / (RB / 4)) * RB + (qd % (RB / 4)) * 4) = make_float4(o[0], o[1], o[2], o[3]);
        }
        if (tid < TS) {
            fg[tid] = gq;
            fb[tid] = bq;
        }
        const bool ok = mbar_wait(&bar[buf], (i >> 1) & 1);
        const TIn *rk = raw + (size_t)buf * 2 * TS * DK;
        if (kConv && ok) {
            const uint32_t *src = reinterpret_cast<const uint32_t *>(rk);   // bf16 pairs, k then q
            for (int e = tid; e < TS * DK; e += nthreads) {                // e indexes pairs
                const uint32_t w = src[e];
                float2 f = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
                float *dst = e < TS * DK / 2 ? fk + 2 * e : fq + 2 * (e - TS * DK / 2);
                *reinterpret_cast<float2 *>(dst) = f;
            }
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) report_status(p.status, kStatusTimeout);
            return;
        }
        if (tid == 0 && i + 1 < ntiles) {
            fence_proxy_async();
            TIn *dst = raw + (size_t)(buf ^ 1) * 2 * TS * DK;
            mbar_expect_tx(&bar[buf ^ 1], tile_bytes);
            tma_load_4d(dst, &tm_k, &bar[buf ^ 1], 0, hk, t0 + TS, b);
            tma_load_4d(dst + TS * DK, &tm_q, &bar[buf ^ 1], 0, hk, t0 + TS, b);
        }
        if (i + 1 < ntiles) prefetch(i + 1);
        const float *kt = kConv ? fk : reinterpret_cast<const float *>(rk);
        const float *qt = kConv ? fq : reinterpret_cast<const float *>(rk) + TS * DK;
        // prediction of the tile's first step: delta_{t0} = beta (v - g S k_{t0})
        {
            float part[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int m = 0; m < P; ++m)
                    acc = __ffma2_rn(S[r][m], *reinterpret_cast<const float2 *>(kt + col + 32 * m), acc);
                part[r] = acc.x + acc.y;
            }
            const float a = group_transpose_reduce<R, G>(part, lane);      // row lrow + (gl >> 2)
            const float r0 = fv[own_row] - fg[0] * a;
            const float d0 = fb[0] * r0;
            if ((gl & 3) == 0) fr[own_row] = r0;
#pragma unroll
            for (int r = 0; r < R; ++r) delta[r] = __shfl_sync(kFullMask, d0, (lane & 16) + 4 * r);
        }

        float2 kc[P];
#pragma unroll
        for (int m = 0; m < P; ++m) kc[m] = *reinterpret_cast<const float2 *>(kt + col + 32 * m);
        for (int tt = 0; tt < tl; ++tt) {
            const int t = t0 + tt;
            if (to_ckpt == 0) {
                // checkpoint: the state before step t (none without a saved-for-backward buffer)
                to_ckpt = p.C;
                if (p.ckpt != nullptr) {
                    float *ck = p.ckpt + (head * p.NC + t / p.C) * (size_t)Dv * DK;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const int row = row0 + lrow + r;
                        if (row < Dv) {
#pragma unroll
                            for (int m = 0; m < P; ++m)
                                *reinterpret_cast<float2 *>(ck + (size_t)row * DK + col + 32 * m) = S[r][m];
                        }
                    }
                }
            }
            --to_ckpt;
            float2 qv[P], kn[P];
#pragma unroll
            for (int m = 0; m < P; ++m) {
                qv[m] = *reinterpret_cast<const float2 *>(qt + tt * DK + col + 32 * m);
                kn[m] = *reinterpret_cast<const float2 *>(kt + (tt + 1) * DK + col + 32 * m);
            }
            const float gc = fg[tt];
            const float2 gg = make_float2(gc, gc);
            float red[2 * R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float2 dd = make_float2(delta[r], delta[r]);
                float2 ya = make_float2(0.f, 0.f), an = make_float2(0.f, 0.f);
#pragma unroll
                for (int m = 0; m < P; ++m) {
                    const float2 s = __ffma2_rn(dd, kc[m], __fmul2_rn(gg, S[r][m]));
                    S[r][m] = s;
                    ya = __ffma2_rn(s, qv[m], ya);
                    an = __ffma2_rn(s, kn[m], an);
                }
                red[2 * r] = ya.x + ya.y;
                red[2 * r + 1] = an.x + an.y;
            }
#pragma unroll
            for (int m = 0; m < P; ++m) kc[m] = kn[m];   // k_{t+1} is the next step's k_t
            // lane holds value (gl >> 1) = 2 * (row offset) + kind; kind 1 = prediction
            const float tot = group_transpose_reduce<2 * R, G>(red, lane);
            if ((gl & 3) == 0) fy[tt * RB + own_row] = tot;
            if (tt + 1 < tl) {
                const float rn = fv[(tt + 1) * RB + own_row] - fg[tt + 1] * tot;
                const float dn = fb[tt + 1] * rn;
                if ((gl & 3) == 2) fr[(tt + 1) * RB + own_row] = rn;
#pragma unroll
                for (int r = 0; r < R; ++r) delta[r] = __shfl_sync(kFullMask, dn, (lane & 16) + 4 * r + 2);
            }
        }
        __syncthreads();
        // y and the residuals of the tile, four consecutive rows per access (Dv % 4 == 0)
        for (int e = tid; e < tl * (RB / 4); e += nthreads) {
            const int tt = e / (RB / 4), rr = (e - tt * (RB / 4)) * 4, row = row0 + rr;
            if (row < Dv) {
                const size_t o = (((size_t)b * T + t0 + tt) * Hv + h) * Dv + row;
                const float4 yv = *reinterpret_cast<const float4 *>(fy + tt * RB + rr);
                if (kConv) {
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(yv.x, yv.y), hi = __floats2bfloat162_rn(yv.z, yv.w);
                    uint2 u;
                    u.x = *reinterpret_cast<const uint32_t *>(&lo);
                    u.y = *reinterpret_cast<const uint32_t *>(&hi);
                    *reinterpret_cast<uint2 *>(y + o) = u;
                } else {
                    *reinterpret_cast<float4 *>(y + o) = yv;
                }
                if (p.resid != nullptr)
                    *reinterpret_cast<float4 *>(p.resid + o) = *reinterpret_cast<const float4 *>(fr + tt * RB + rr);
            }
        }
    }
    if (p.S_T != nullptr) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = row0 + lrow + r;
            if (row < Dv) {
#pragma unroll
                for (int m = 0; m < P; ++m)
                    *reinterpret_cast<float2 *>(p.S_T + (head * Dv + row) * DK + col + 32 * m) = S[r][m];
            }
        }
    }
}

template <int P, typename TIn>
static cudaError_t launch_fwd_t(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk, int warps,
                                cudaStream_t s) {
    const int RB = warps * 8;
    const FwdSmem L(32 * P, RB, (int)sizeof(TIn), !IsF32<TIn>::value);
    cudaError_t err =
        cudaFuncSetAttribute(fwd_kernel<P, TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
    if (err != cudaSuccess) return err;
    dim3 grid((p.Dv + RB - 1) / RB, p.Hv, p.B);
    timing_mark("seq_fwd", 0, s);
    fwd_kernel<P, TIn><<<grid, warps * 32, L.total, s>>>(tq, tk, p);
    timing_mark("seq_fwd", 1, s);
    return cudaGetLastError();
}

template <typename TIn>
static cudaError_t launch_fwd_dk(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk, int Dk,
                                 int warps, cudaStream_t s) {
    switch (Dk) {
        case 32: return launch_fwd_t<1, TIn>(p, tq, tk, warps, s);
        case 64: return launch_fwd_t<2, TIn>(p, tq, tk, warps, s);
        case 96: return launch_fwd_t<3, TIn>(p, tq, tk, warps, s);
        case 128: return launch_fwd_t<4, TIn>(p, tq, tk, warps, s);
        case 160: return launch_fwd_t<5, TIn>(p, tq, tk, warps, s);
        case 192: return launch_fwd_t<6, TIn>(p, tq, tk, warps, s);
        case 224: return launch_fwd_t<7, TIn>(p, tq, tk, warps, s);
        case 256: return launch_fwd_t<8, TIn>(p, tq, tk, warps, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_fwd(const FwdParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_k, int Dk, int dtype,
                       int warps, cudaStream_t s) {
    return dtype == 0 ? launch_fwd_dk<float>(p, tm_q, tm_k, Dk, warps, s)
                      : launch_fwd_dk<__nv_bfloat16>(p, tm_q, tm_k, Dk, warps, s);
}

}  // namespace gdn
