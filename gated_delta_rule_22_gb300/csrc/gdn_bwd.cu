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
// FP32 operations; ddelta needs Sc k_t = Sh k_t + dy_t (q_t . k_t), so the row dot
// Sh k_t is formed in the previous step's pass (against k_{t-1}) and is the only
// cross-lane reduction on the serial chain.
//
// Checkpointing (mlx-lm PR #1217, "What this PR adds": forward-with-save, then a reverse
// sweep in the same chunked layout): for each chunk, going backwards,
//   pass A  re-runs the chunk from its checkpoint, keeping delta_t and v_t - u_t per row
//           and step in shared memory and the state at every kSub-th step (sub-block
//           start) in scratch;
//   pass B  for each sub-block, going backwards, re-builds the states inside it from its
//           start state with the kept delta (S <- g S + delta k^T: 2 FP32 ops/element);
//   core    runs the reverse steps of the sub-block reading S_{t-1} from scratch.
//
// Reductions: a CTA owns RB rows of one (b, h). Column sums (dq, dk) are summed over a
// thread's rows in registers, over the CTA's warps in shared memory in ascending warp
// order, and written per (b, t, h, row split) to fp32 scratch; dg and dbeta likewise.
// reduce_kernel then adds the row splits (ascending) and the value heads of each kv
// head (ascending) and rounds to the output type. No atomics anywhere.
#include "gdn_common.cuh"

namespace gdn {

template <int E, typename TIn>
__global__ void __launch_bounds__(256, 1) bwd_kernel(BwdParams p) {
    constexpr int RW = kRowsPerWarp;
    constexpr int DK = 32 * E;
    constexpr int SUB = kSub;
    const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RB = nw * RW;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int row0 = split * RB;
    const int rep = p.Hv / p.Hk, hk = h / rep;
    const int T = p.T, Dv = p.Dv, C = p.C, Hv = p.Hv, nsplit = p.nsplit;
    const int wrow = warp * RW;
    const int my_row = lane >> 2;   // row held by this lane after a transpose_reduce<RW>

    extern __shared__ float smem[];
    float *dl_s = smem;                      // [C][RB]   delta_t per row (pass A)
    float *vm_s = dl_s + C * RB;             // [C][RB]   v_t - u_t per row (pass A)
    float *k_s = vm_s + C * RB;              // [SUB+1][DK]
    float *q_s = k_s + (SUB + 1) * DK;       // [SUB][DK]
    float *v_s = q_s + SUB * DK;             // [SUB][RB]  (pass A)
    float *dy_s = v_s + SUB * RB;            // [SUB][RB]
    float *dd_s = dy_s + SUB * RB;           // [SUB][RB]  ddelta per row
    float *cp_s = dd_s + SUB * RB;           // [SUB][nw][2][DK] per-warp column partials (dk, dq)
    float *gp_s = cp_s + SUB * nw * 2 * DK;  // [SUB][nw] per-warp dg partials
    float *g_s = gp_s + SUB * nw;            // [SUB]
    float *b_s = g_s + SUB;                  // [SUB]
    float *kq_s = b_s + SUB;                 // [SUB] k_t . q_t
    float *dd2_s = kq_s + SUB;               // [SUB] delta_t . dy_t over the CTA's rows

    const TIn *q = static_cast<const TIn *>(p.q);
    const TIn *k = static_cast<const TIn *>(p.k);
    const TIn *v = static_cast<const TIn *>(p.v);
    const TIn *g = static_cast<const TIn *>(p.g);
    const TIn *beta = static_cast<const TIn *>(p.beta);
    const TIn *dy = static_cast<const TIn *>(p.dy);
    TIn *dv = static_cast<TIn *>(p.dv);

    const size_t state_off = ((size_t)b * Hv + h) * Dv;
    const size_t cta = ((size_t)b * Hv + h) * nsplit + split;
    const int nslots = p.nsub_max + SUB - 1;
    float *scratch = p.ws_state + cta * nslots * (size_t)RB * DK;
    // element (r, e) of this thread inside a scratch state slot is my_off + r*DK + 32*e
    const int my_off = wrow * DK + lane;

    float Sh[RW][E];
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        const int row = row0 + wrow + r;
#pragma unroll
        for (int e = 0; e < E; ++e)
            Sh[r][e] = (p.dS_T != nullptr && row < Dv) ? p.dS_T[(state_off + row) * DK + lane + 32 * e] : 0.f;
    }
    float p_own;  // (Sh k_t) of row my_row for the next reverse step t
    {
        float part[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) part[r] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float kk = to_f32(k[(((size_t)b * T + T - 1) * p.Hk + hk) * DK + lane + 32 * e]);
#pragma unroll
            for (int r = 0; r < RW; ++r) part[r] = fmaf(Sh[r][e], kk, part[r]);
        }
        p_own = transpose_reduce<RW>(part, lane);
    }

    for (int c = p.NC - 1; c >= 0; --c) {
        const int t0 = c * C, len = min(C, T - t0), nsub = (len + SUB - 1) / SUB;

        // ---------------- pass A: forward through the chunk from its checkpoint ----------------
        float S[RW][E];
        {
            const float *ck = p.ckpt + ((state_off * p.NC) + (size_t)c * Dv) * DK;
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int row = row0 + wrow + r;
#pragma unroll
                for (int e = 0; e < E; ++e) S[r][e] = row < Dv ? ck[(size_t)row * DK + lane + 32 * e] : 0.f;
            }
        }
        for (int m = 0; m < nsub; ++m) {
            const int s0 = t0 + m * SUB, slen = min(SUB, t0 + len - s0);
            float *slot = scratch + (size_t)m * RB * DK + my_off;
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int e = 0; e < E; ++e) slot[r * DK + 32 * e] = S[r][e];
            __syncthreads();
            for (int i = threadIdx.x; i < slen * DK; i += blockDim.x) {
                const int j = i / DK, col = i - j * DK;
                k_s[i] = to_f32(k[(((size_t)b * T + s0 + j) * p.Hk + hk) * DK + col]);
            }
            for (int i = threadIdx.x; i < slen * RB; i += blockDim.x) {
                const int j = i / RB, rr = i - j * RB, row = row0 + rr;
                v_s[i] = row < Dv ? to_f32(v[(((size_t)b * T + s0 + j) * Hv + h) * Dv + row]) : 0.f;
            }
            for (int i = threadIdx.x; i < slen; i += blockDim.x) {
                g_s[i] = to_f32(g[((size_t)b * T + s0 + i) * Hv + h]);
                b_s[i] = to_f32(beta[((size_t)b * T + s0 + i) * Hv + h]);
            }
            __syncthreads();
            for (int j = 0; j < slen; ++j) {
                float kv[E];
#pragma unroll
                for (int e = 0; e < E; ++e) kv[e] = k_s[j * DK + lane + 32 * e];
                float part[RW];
#pragma unroll
                for (int r = 0; r < RW; ++r) {
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) a = fmaf(S[r][e], kv[e], a);
                    part[r] = a;
                }
                const float a = transpose_reduce<RW>(part, lane);
                const float gt = g_s[j], bt = b_s[j];
                const float vm = v_s[j * RB + wrow + my_row] - gt * a;
                const float dl = bt * vm;
                if ((lane & 3) == 0) {
                    dl_s[(s0 - t0 + j) * RB + wrow + my_row] = dl;
                    vm_s[(s0 - t0 + j) * RB + wrow + my_row] = vm;
                }
                float d[RW];
#pragma unroll
                for (int r = 0; r < RW; ++r) d[r] = __shfl_sync(kFullMask, dl, 4 * r);
#pragma unroll
                for (int r = 0; r < RW; ++r)
#pragma unroll
                    for (int e = 0; e < E; ++e) S[r][e] = fmaf(d[r], kv[e], gt * S[r][e]);
            }
        }

        // ---------------- reverse sweep over the chunk's sub-blocks ----------------
        for (int m = nsub - 1; m >= 0; --m) {
            const int s0 = t0 + m * SUB, slen = min(SUB, t0 + len - s0);
            __syncthreads();
            for (int i = threadIdx.x; i < (slen + 1) * DK; i += blockDim.x) {
                const int j = i / DK, col = i - j * DK, t = s0 - 1 + j;
                k_s[i] = t >= 0 ? to_f32(k[(((size_t)b * T + t) * p.Hk + hk) * DK + col]) : 0.f;
            }
            for (int i = threadIdx.x; i < slen * DK; i += blockDim.x) {
                const int j = i / DK, col = i - j * DK;
                q_s[i] = to_f32(q[(((size_t)b * T + s0 + j) * p.Hk + hk) * DK + col]);
            }
            for (int i = threadIdx.x; i < slen * RB; i += blockDim.x) {
                const int j = i / RB, rr = i - j * RB, row = row0 + rr;
                dy_s[i] = row < Dv ? to_f32(dy[(((size_t)b * T + s0 + j) * Hv + h) * Dv + row]) : 0.f;
            }
            for (int i = threadIdx.x; i < slen; i += blockDim.x) {
                g_s[i] = to_f32(g[((size_t)b * T + s0 + i) * Hv + h]);
                b_s[i] = to_f32(beta[((size_t)b * T + s0 + i) * Hv + h]);
            }
            __syncthreads();
            for (int j = warp; j < slen; j += nw) {
                float a = 0.f;
                for (int col = lane; col < DK; col += 32) a = fmaf(k_s[(j + 1) * DK + col], q_s[j * DK + col], a);
                a = warp_sum(a);
                if (lane == 0) kq_s[j] = a;
            }

            // pass B: states before steps s0+1 .. s0+slen-1, from the sub-block's start state
            {
                float S2[RW][E];
                const float *slot0 = scratch + (size_t)m * RB * DK + my_off;
#pragma unroll
                for (int r = 0; r < RW; ++r)
#pragma unroll
                    for (int e = 0; e < E; ++e) S2[r][e] = slot0[r * DK + 32 * e];
                for (int j = 0; j + 1 < slen; ++j) {
                    const float gt = g_s[j];
                    float *slot = scratch + (size_t)(p.nsub_max + j) * RB * DK + my_off;
#pragma unroll
                    for (int r = 0; r < RW; ++r) {
                        const float d = dl_s[(s0 - t0 + j) * RB + wrow + r];
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            S2[r][e] = fmaf(d, k_s[(j + 1) * DK + lane + 32 * e], gt * S2[r][e]);
                            slot[r * DK + 32 * e] = S2[r][e];
                        }
                    }
                }
            }
            __syncthreads();

            // core: reverse steps of the sub-block
            for (int j = slen - 1; j >= 0; --j) {
                const float *sp = scratch + (size_t)(j == 0 ? m : p.nsub_max + j - 1) * RB * DK + my_off;
                const float gt = g_s[j], bt = b_s[j];
                const float dyo = dy_s[j * RB + wrow + my_row];
                const float ddo = p_own + dyo * kq_s[j];
                const float duo = -bt * ddo;
                if ((lane & 3) == 0) dd_s[j * RB + wrow + my_row] = ddo;
                float kt[E], qt[E], kp[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    kt[e] = k_s[(j + 1) * DK + lane + 32 * e];
                    qt[e] = q_s[j * DK + lane + 32 * e];
                    kp[e] = k_s[j * DK + lane + 32 * e];
                }
                float dkacc[E], dqacc[E], pn[RW];
#pragma unroll
                for (int e = 0; e < E; ++e) dkacc[e] = dqacc[e] = 0.f;
                float dgacc = 0.f;
                const int tc = s0 + j - t0;
#pragma unroll
                for (int r = 0; r < RW; ++r) {
                    const float du = __shfl_sync(kFullMask, duo, 4 * r);
                    const float dyr = dy_s[j * RB + wrow + r];
                    const float dr = dl_s[tc * RB + wrow + r];
                    const float gdu = gt * du, gdy = gt * dyr;
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float spe = sp[r * DK + 32 * e];
                        const float sc = fmaf(dyr, qt[e], Sh[r][e]);
                        dkacc[e] = fmaf(sc, dr, dkacc[e]);
                        const float dA = fmaf(du, kt[e], sc);
                        dgacc = fmaf(dA, spe, dgacc);
                        dkacc[e] = fmaf(spe, gdu, dkacc[e]);
                        dqacc[e] = fmaf(spe, gdy, dqacc[e]);
                        const float shn = gt * dA;
                        Sh[r][e] = shn;
                        acc = fmaf(shn, kp[e], acc);
                    }
                    pn[r] = acc;
                }
                float *cp = cp_s + (size_t)(j * nw + warp) * 2 * DK + lane;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    cp[32 * e] = dkacc[e];
                    cp[DK + 32 * e] = dqacc[e];
                }
                dgacc = warp_sum(dgacc);
                if (lane == 0) gp_s[j * nw + warp] = dgacc;
                p_own = transpose_reduce<RW>(pn, lane);
            }
            __syncthreads();

            // fixed-order reductions of the sub-block's per-step partials
            for (int j = warp; j < slen; j += nw) {
                const int t = s0 + j, tc = t - t0;
                float s1 = 0.f, s2 = 0.f;
                for (int rr = lane; rr < RB; rr += 32) {
                    s1 = fmaf(dl_s[tc * RB + rr], dy_s[j * RB + rr], s1);
                    s2 = fmaf(dd_s[j * RB + rr], vm_s[tc * RB + rr], s2);
                }
                s1 = warp_sum(s1);
                s2 = warp_sum(s2);
                if (lane == 0) {
                    float dgs = 0.f;
                    for (int w = 0; w < nw; ++w) dgs += gp_s[j * nw + w];
                    const size_t o = (((size_t)b * T + t) * Hv + h) * nsplit + split;
                    p.ws_dg[o] = dgs;
                    p.ws_db[o] = s2;
                    dd2_s[j] = s1;
                }
            }
            __syncthreads();
            for (int i = threadIdx.x; i < slen * DK; i += blockDim.x) {
                const int j = i / DK, col = i - j * DK, t = s0 + j;
                float a = 0.f, bq = 0.f;
                for (int w = 0; w < nw; ++w) {
                    a += cp_s[((size_t)(j * nw + w) * 2) * DK + col];
                    bq += cp_s[((size_t)(j * nw + w) * 2 + 1) * DK + col];
                }
                bq = fmaf(k_s[(j + 1) * DK + col], dd2_s[j], bq);
                const size_t o = ((((size_t)b * T + t) * Hv + h) * nsplit + split) * DK + col;
                p.ws_dk[o] = a;
                p.ws_dq[o] = bq;
            }
            for (int i = threadIdx.x; i < slen * RB; i += blockDim.x) {
                const int j = i / RB, rr = i - j * RB, row = row0 + rr;
                if (row < Dv)
                    dv[(((size_t)b * T + s0 + j) * Hv + h) * Dv + row] = from_f32<TIn>(b_s[j] * dd_s[j * RB + rr]);
            }
        }
    }
    if (p.dS0 != nullptr) {
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const int row = row0 + wrow + r;
            if (row < Dv) {
#pragma unroll
                for (int e = 0; e < E; ++e) p.dS0[(state_off + row) * DK + lane + 32 * e] = Sh[r][e];
            }
        }
    }
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

size_t bwd_smem_bytes(int DK, int nw, int C) {
    const int RB = nw * kRowsPerWarp, SUB = kSub;
    const size_t floats = (size_t)2 * C * RB + (size_t)(2 * SUB + 1) * DK + (size_t)3 * SUB * RB +
                          (size_t)SUB * nw * 2 * DK + (size_t)SUB * nw + 4 * SUB;
    return floats * sizeof(float);
}

template <int E, typename TIn>
static cudaError_t launch_bwd_t(const BwdParams &p, int warps, cudaStream_t s) {
    const size_t smem = bwd_smem_bytes(32 * E, warps, p.C);
    cudaError_t err = cudaFuncSetAttribute(bwd_kernel<E, TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid(p.nsplit, p.Hv, p.B);
    bwd_kernel<E, TIn><<<grid, warps * 32, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename TIn>
static cudaError_t launch_bwd_dk(const BwdParams &p, int Dk, int warps, cudaStream_t s) {
    switch (Dk) {
        case 32: return launch_bwd_t<1, TIn>(p, warps, s);
        case 64: return launch_bwd_t<2, TIn>(p, warps, s);
        case 96: return launch_bwd_t<3, TIn>(p, warps, s);
        case 128: return launch_bwd_t<4, TIn>(p, warps, s);
        case 160: return launch_bwd_t<5, TIn>(p, warps, s);
        case 192: return launch_bwd_t<6, TIn>(p, warps, s);
        case 224: return launch_bwd_t<7, TIn>(p, warps, s);
        case 256: return launch_bwd_t<8, TIn>(p, warps, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd(const BwdParams &p, int Dk, int dtype, int warps, cudaStream_t s) {
    return dtype == 0 ? launch_bwd_dk<float>(p, Dk, warps, s) : launch_bwd_dk<__nv_bfloat16>(p, Dk, warps, s);
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
