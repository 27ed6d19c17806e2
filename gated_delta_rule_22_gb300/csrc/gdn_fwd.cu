// gdn_fwd.cu -- forward of the gated delta rule with chunk checkpoints.
//
// Recurrence (mlx issue #4614, "Recurrence used for the references"), per value head h
// with kv head h / (Hv/Hk):  S <- g_t S;  S <- S + (beta_t (v_t - S k_t)) k_t^T;
// y_t = S q_t.  Checkpoints (mlx-lm PR #1217, "What this PR adds"): the state before
// every C-th step is written to HBM for the reverse sweep.
//
// One CTA owns RB = 8 * warps rows of one (b, h) state and keeps them in registers for
// the whole sequence. Per step every element of S is read once and written once in a
// fused pass that also forms both row dot products the recurrence needs next:
//     S_t = g_t S_{t-1} + delta_t k_t^T         (FMUL + FFMA)
//     ya  = S_t . q_t   -> y_t                   (FFMA)
//     an  = S_t . k_{t+1} -> prediction u_{t+1} = g_{t+1} an   (FFMA)
// The two dots of the warp's 8 rows (16 partial sums per lane) are reduced across the
// 32 lanes by one transpose-reduction; the lane that ends up holding row r's `an`
// computes delta_{t+1} = beta_{t+1} (v_{t+1} - g_{t+1} an) and shares it with a shuffle.
// Inputs are staged per tile of kFwdTile steps in shared memory as fp32.
#include "gdn_common.cuh"

namespace gdn {

template <int E, typename TIn>
__global__ void __launch_bounds__(256, 1) fwd_kernel(FwdParams p) {
    constexpr int RW = kRowsPerWarp;
    constexpr int DK = 32 * E;
    constexpr int TS = kFwdTile;
    const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RB = nw * RW;
    const int b = blockIdx.z, h = blockIdx.y, row0 = blockIdx.x * RB;
    const int rep = p.Hv / p.Hk, hk = h / rep;
    const int T = p.T, Dv = p.Dv;

    extern __shared__ float smem[];
    float *k_s = smem;                  // [TS+1][DK]  k_{t0} .. k_{t0+TS}
    float *q_s = k_s + (TS + 1) * DK;   // [TS][DK]
    float *v_s = q_s + TS * DK;         // [TS+1][RB]
    float *y_s = v_s + (TS + 1) * RB;   // [TS][RB]
    float *g_s = y_s + TS * RB;         // [TS+1]
    float *b_s = g_s + (TS + 1);        // [TS+1]

    const TIn *q = static_cast<const TIn *>(p.q);
    const TIn *k = static_cast<const TIn *>(p.k);
    const TIn *v = static_cast<const TIn *>(p.v);
    const TIn *g = static_cast<const TIn *>(p.g);
    const TIn *beta = static_cast<const TIn *>(p.beta);
    TIn *y = static_cast<TIn *>(p.y);

    const int wrow = warp * RW;                             // first row of this warp in the CTA
    const size_t state_off = ((size_t)b * p.Hv + h) * Dv;   // row offset of this head's state
    const size_t ckpt_off = ((size_t)b * p.Hv + h) * p.NC * (size_t)Dv;

    float S[RW][E];
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        const int row = row0 + wrow + r;
#pragma unroll
        for (int e = 0; e < E; ++e)
            S[r][e] = (p.S0 != nullptr && row < Dv) ? p.S0[(state_off + row) * DK + lane + 32 * e] : 0.f;
    }

    float kc[E];        // k_t of the step about to run
    float delta[RW];    // delta_t of this warp's rows (same on every lane)
    float gc = 1.f;     // g_t
    // after transpose_reduce<16> lane l holds value (l >> 1) = 2 * row + kind,
    // kind 0 = readout partial, kind 1 = prediction partial
    const int my_row = lane >> 2;
    const bool holds_pred = (lane >> 1) & 1;

    for (int t0 = 0; t0 < T; t0 += TS) {
        const int tl = min(TS, T - t0);
        __syncthreads();  // previous tile fully consumed
        for (int i = threadIdx.x; i < (tl + 1) * DK; i += blockDim.x) {
            const int tt = i / DK, c = i - tt * DK, t = t0 + tt;
            k_s[i] = t < T ? to_f32(k[(((size_t)b * T + t) * p.Hk + hk) * DK + c]) : 0.f;
        }
        for (int i = threadIdx.x; i < tl * DK; i += blockDim.x) {
            const int tt = i / DK, c = i - tt * DK, t = t0 + tt;
            q_s[i] = to_f32(q[(((size_t)b * T + t) * p.Hk + hk) * DK + c]);
        }
        for (int i = threadIdx.x; i < (tl + 1) * RB; i += blockDim.x) {
            const int tt = i / RB, rr = i - tt * RB, t = t0 + tt, row = row0 + rr;
            v_s[i] = (t < T && row < Dv) ? to_f32(v[(((size_t)b * T + t) * p.Hv + h) * Dv + row]) : 0.f;
        }
        for (int i = threadIdx.x; i < tl + 1; i += blockDim.x) {
            const int t = t0 + i;
            g_s[i] = t < T ? to_f32(g[((size_t)b * T + t) * p.Hv + h]) : 1.f;
            b_s[i] = t < T ? to_f32(beta[((size_t)b * T + t) * p.Hv + h]) : 0.f;
        }
        __syncthreads();

        if (t0 == 0) {
            // prediction of step 0 from S_0
            float part[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) a = fmaf(S[r][e], k_s[lane + 32 * e], a);
                part[r] = a;
            }
            const float a0 = transpose_reduce<RW>(part, lane);   // row lane >> 2
            const float d0 = b_s[0] * (v_s[wrow + (lane >> 2)] - g_s[0] * a0);
#pragma unroll
            for (int r = 0; r < RW; ++r) delta[r] = __shfl_sync(kFullMask, d0, 4 * r);
#pragma unroll
            for (int e = 0; e < E; ++e) kc[e] = k_s[lane + 32 * e];
            gc = g_s[0];
        }

        for (int tt = 0; tt < tl; ++tt) {
            const int t = t0 + tt;
            if (t % p.C == 0) {
                // checkpoint: state before step t
                float *ck = p.ckpt + (ckpt_off + (size_t)(t / p.C) * Dv) * DK;
#pragma unroll
                for (int r = 0; r < RW; ++r) {
                    const int row = row0 + wrow + r;
                    if (row < Dv) {
#pragma unroll
                        for (int e = 0; e < E; ++e) ck[(size_t)row * DK + lane + 32 * e] = S[r][e];
                    }
                }
            }
            float qv[E], kn[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                qv[e] = q_s[tt * DK + lane + 32 * e];
                kn[e] = k_s[(tt + 1) * DK + lane + 32 * e];
            }
            float red[2 * RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                float ya = 0.f, an = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float s = fmaf(delta[r], kc[e], gc * S[r][e]);
                    S[r][e] = s;
                    ya = fmaf(s, qv[e], ya);
                    an = fmaf(s, kn[e], an);
                }
                red[2 * r] = ya;
                red[2 * r + 1] = an;
            }
            const float tot = transpose_reduce<2 * RW>(red, lane);
            if (!holds_pred && (lane & 1) == 0) y_s[tt * RB + wrow + my_row] = tot;
            const float gn = g_s[tt + 1];
            const float dn = b_s[tt + 1] * (v_s[(tt + 1) * RB + wrow + my_row] - gn * tot);
#pragma unroll
            for (int r = 0; r < RW; ++r) delta[r] = __shfl_sync(kFullMask, dn, 4 * r + 2);
#pragma unroll
            for (int e = 0; e < E; ++e) kc[e] = kn[e];
            gc = gn;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < tl * RB; i += blockDim.x) {
            const int tt = i / RB, rr = i - tt * RB, row = row0 + rr;
            if (row < Dv) y[(((size_t)b * T + t0 + tt) * p.Hv + h) * Dv + row] = from_f32<TIn>(y_s[i]);
        }
    }
    if (p.S_T != nullptr) {
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const int row = row0 + wrow + r;
            if (row < Dv) {
#pragma unroll
                for (int e = 0; e < E; ++e) p.S_T[(state_off + row) * DK + lane + 32 * e] = S[r][e];
            }
        }
    }
}

static size_t fwd_smem_bytes(int DK, int RB) {
    const int TS = kFwdTile;
    return sizeof(float) * ((size_t)(2 * TS + 1) * DK + (size_t)(2 * TS + 1) * RB + 2 * (TS + 1));
}

template <int E, typename TIn>
static cudaError_t launch_fwd_t(const FwdParams &p, int warps, cudaStream_t s) {
    const int RB = warps * kRowsPerWarp;
    const size_t smem = fwd_smem_bytes(32 * E, RB);
    cudaError_t err = cudaFuncSetAttribute(fwd_kernel<E, TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid((p.Dv + RB - 1) / RB, p.Hv, p.B);
    fwd_kernel<E, TIn><<<grid, warps * 32, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename TIn>
static cudaError_t launch_fwd_dk(const FwdParams &p, int Dk, int warps, cudaStream_t s) {
    switch (Dk) {
        case 32: return launch_fwd_t<1, TIn>(p, warps, s);
        case 64: return launch_fwd_t<2, TIn>(p, warps, s);
        case 96: return launch_fwd_t<3, TIn>(p, warps, s);
        case 128: return launch_fwd_t<4, TIn>(p, warps, s);
        case 160: return launch_fwd_t<5, TIn>(p, warps, s);
        case 192: return launch_fwd_t<6, TIn>(p, warps, s);
        case 224: return launch_fwd_t<7, TIn>(p, warps, s);
        case 256: return launch_fwd_t<8, TIn>(p, warps, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_fwd(const FwdParams &p, int Dk, int dtype, int warps, cudaStream_t s) {
    return dtype == 0 ? launch_fwd_dk<float>(p, Dk, warps, s) : launch_fwd_dk<__nv_bfloat16>(p, Dk, warps, s);
}

}  // namespace gdn
