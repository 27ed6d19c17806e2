// gdn_chunk.cu -- the forward of the gated delta rule in its chunkwise (dense) form on the
// 5th-generation tensor cores, for bf16 inputs and chunks of 64 steps.
//
// The recurrence is that of mlx issue #4614 ("Recurrence used for the references"); the
// chunkwise form is derived from it (the pages do not give it). Per value head and chunk of
// L = 64 steps with start state S0 [Dv, Dk] (lam_t = log g_t, Lam its in-chunk prefix sum,
// E(s, i) = exp(Lam_s - Lam_i) <= 1, never a division by a decay):
//     A[t, i] = beta_t (k_t . k_i) E(t, i)  (i < t),   T = (I + A)^-1
//     W = T diag(beta exp Lam) K,   U = T diag(beta) V,   Delta = U - W S0^T
//     y = diag(exp Lam) (Q S0^T) + ((Q K^T) o E_incl) Delta
//     u = diag(exp Lam) (K S0^T) + ((K K^T) o E_strict) Delta      (u_t = g_t S_{t-1} k_t)
//     S_L = exp(Lam_L) S0 + (diag(E(L, .)) Delta)^T K
// chunk_prep_kernel computes what depends on neither the state nor V, for all chunks at once;
// chunk_sweep_kernel carries the state through the chunks of one head and forms
// Delta = (T diag(beta)) V - W S0^T as one accumulation on the tensor cores. Products run with
// bf16 operands and fp32 accumulators in tensor memory; T is formed in fp32 on the CUDA cores.
// The outputs (y, the chunk-start states, v - u) are those of the sequential forward, so the
// backward consumes them unchanged.
#include "gdn_umma.cuh"

namespace gdn {

namespace {

constexpr int kL = 64;           // chunk length of the tensor-core forward
constexpr int kP = 68;           // row of prep's fp32 64 x 64 work matrices (16-byte aligned, conflict-free float4 columns)
// Both kernels hold all 512 tensor-memory columns, so each must be alone on its SM: they ask
// for more than half of the shared memory.
constexpr size_t kOneCtaSmem = 120 * 1024;

__host__ __device__ inline size_t al(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Prep runs two CTAs per SM (each 256 tensor-memory columns and under half of the shared
// memory), so that one CTA's serial steps (the inversion, the products' round trips) overlap
// the other's.
struct PrepSmem {
    size_t kc, qc, am, ts, xs, tcw, tcu, lam, bar, tslot, total;
    __host__ __device__ PrepSmem(int DK) {
        size_t o = 0;
        kc = o; o += (size_t)kL * DK * 2;           // K of the chunk, bf16 operand [64][DK]
        qc = o; o += (size_t)kL * DK * 2;           // Q of the chunk
        am = o; o += (size_t)kL * kP * 4;           // A
        ts = o; o += (size_t)kL * kP * 4;           // T = (I + A)^-1 (blocks above the diagonal not written)
        xs = o; o += (size_t)32 * 32 * 4;           // block products of the inversion
        tcw = o; o += (size_t)kL * kL * 2;          // T diag(beta exp Lam), bf16 operand [64][64]
        tcu = o; o += (size_t)kL * kL * 2;          // T diag(beta), bf16 operand [64][64] (stored for the sweep)
        lam = o; o += 4 * kL * 4;                   // log g, Lam, exp Lam, beta
        bar = al(o, 8); o = bar + 2 * 8;            // MMA, copies of K and Q
        tslot = o; o += 16;
        total = o + 1024;
    }
};

__device__ __forceinline__ uint4 pack8_bf16(const float (&x)[8]) {
    uint4 u;
    __nv_bfloat162 h;
    h = __floats2bfloat162_rn(x[0], x[1]); u.x = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2bfloat162_rn(x[2], x[3]); u.y = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2bfloat162_rn(x[4], x[5]); u.z = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2bfloat162_rn(x[6], x[7]); u.w = *reinterpret_cast<uint32_t *>(&h);
    return u;
}

// T = (I + A)^-1 for the strictly lower 64 x 64 A (row stride kP), in two levels of 2 x 2
// block recursion: the four diagonal 16 x 16 blocks by forward substitution (a column per
// thread, rows above the column's diagonal exactly zero); then the two 32 x 32 diagonal blocks, and then the 64 x 64, each by
//     T_21 = -T_22 (A_21 T_11)
// as two dependent products with four consecutive columns of one row per thread (a scalar
// and a float4 load per four multiply-adds). Blocks of T above the diagonal are not written,
// and the products skip them. Called by all 256 threads; xs holds 32 x 32 floats. Threads
// 64-255, idle during the diagonal blocks, run `other` meanwhile.
template <class Other>
__device__ void invert_unit_lower(const float *am, float *ts, float *xs, int tid, Other &&other) {
    if (tid >= kL) other();
    if (tid < kL) {
        // column c of the block's inverse, right-looking: once x_i is final it updates every
        // later row at once, so the dependent chain is 16 multiply-adds long (not 120)
        const int b0 = 16 * (tid >> 4), c = tid & 15;
        float acc[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) acc[r] = r == c ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < 15; ++i) {
            const float xi = acc[i];
#pragma unroll
            for (int r = i + 1; r < 16; ++r) acc[r] = fmaf(-am[(b0 + r) * kP + b0 + i], xi, acc[r]);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) ts[(b0 + r) * kP + b0 + c] = acc[r];
    }
    __syncthreads();
    // ---- level 1: the 32 x 32 diagonal blocks b = 0, 1 (threads 0-127)
    {
        const int b = tid >> 6, r = (tid >> 2) & 15, c4 = 4 * (tid & 3), o = 32 * b;
        if (tid < 128) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float a = am[(o + 16 + r) * kP + o + k];
                const float4 t4 = *reinterpret_cast<const float4 *>(ts + (o + k) * kP + o + c4);
                acc.x = fmaf(a, t4.x, acc.x); acc.y = fmaf(a, t4.y, acc.y);
                acc.z = fmaf(a, t4.z, acc.z); acc.w = fmaf(a, t4.w, acc.w);
            }
            *reinterpret_cast<float4 *>(xs + (b * 16 + r) * 16 + c4) = acc;
        }
        __syncthreads();
        if (tid < 128) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float a = ts[(o + 16 + r) * kP + o + 16 + k];
                const float4 x4 = *reinterpret_cast<const float4 *>(xs + (b * 16 + k) * 16 + c4);
                acc.x = fmaf(a, x4.x, acc.x); acc.y = fmaf(a, x4.y, acc.y);
                acc.z = fmaf(a, x4.z, acc.z); acc.w = fmaf(a, x4.w, acc.w);
            }
            *reinterpret_cast<float4 *>(ts + (o + 16 + r) * kP + o + c4) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        __syncthreads();
    }
    // ---- level 2: rows 32-63, columns 0-31 (all threads: row r, columns c4 .. c4 + 3)
    {
        const int r = tid >> 3, c4 = 4 * (tid & 7);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        // X = A_21 T_11: T_11[k][c] = 0 for k in a 16-block above c's
        for (int k = 16 * (c4 >> 4); k < 32; ++k) {
            const float a = am[(32 + r) * kP + k];
            const float4 t4 = *reinterpret_cast<const float4 *>(ts + k * kP + c4);
            acc.x = fmaf(a, t4.x, acc.x); acc.y = fmaf(a, t4.y, acc.y);
            acc.z = fmaf(a, t4.z, acc.z); acc.w = fmaf(a, t4.w, acc.w);
        }
        *reinterpret_cast<float4 *>(xs + r * 32 + c4) = acc;
        __syncthreads();
        // T_21 = -T_22 X: T_22[r][k] = 0 for k in a 16-block right of r's
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const int kend = 16 * ((r >> 4) + 1);
        for (int k = 0; k < kend; ++k) {
            const float a = ts[(32 + r) * kP + 32 + k];
            const float4 x4 = *reinterpret_cast<const float4 *>(xs + k * 32 + c4);
            acc.x = fmaf(a, x4.x, acc.x); acc.y = fmaf(a, x4.y, acc.y);
            acc.z = fmaf(a, x4.z, acc.z); acc.w = fmaf(a, x4.w, acc.w);
        }
        *reinterpret_cast<float4 *>(ts + (32 + r) * kP + c4) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        __syncthreads();
    }
}

}  // namespace

// Persistent: two CTAs per SM, each over a contiguous range of units (batch row, chunk, kv head,
// value head), value head fastest. When a unit starts a new (batch row, chunk, kv head) group
// the CTA stores [Q; K] for the sweeps and the gradient kernel (K and Q fetched by TMA while the
// previous group's last unit was read back). Per unit (value head) it forms K K^T and Q K^T on
// the tensor cores (again per unit: tensor memory holds them only until the unit's W), reads
// them straight from tensor memory into the decay-weighted matrices and A, inverts, and forms
// W = (T diag(beta exp Lam)) K (the row scalings folded into T's columns, K read as an MN-major
// operand), stored negated for the sweep's single Delta accumulation; it stores T and
// T diag(beta) (the sweep forms U from the latter and V).
template <int E>
__global__ void __launch_bounds__(256, 2) chunk_prep_kernel(ChunkParams p, int units,
                                                            const __grid_constant__ ChunkFwdMaps maps) {
    constexpr int DK = 32 * E;
    static_assert(DK <= 256, "W fits the 256 tensor-memory columns of a CTA");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.T, Hv = p.Hv, Hk = p.Hk, NC = p.NC, rep = p.Hv / p.Hk;
    const int u_begin = (int)((long long)blockIdx.x * units / gridDim.x);
    const int u_end = (int)((long long)(blockIdx.x + 1) * units / gridDim.x);

    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(al(reinterpret_cast<size_t>(smem_raw), 1024));
    const PrepSmem L(DK);
    unsigned char *kc = base + L.kc, *qc = base + L.qc, *tcw = base + L.tcw, *tcu = base + L.tcu;
    float *am = reinterpret_cast<float *>(base + L.am);
    float *ts = reinterpret_cast<float *>(base + L.ts);
    float *xs = reinterpret_cast<float *>(base + L.xs);
    float *lg = reinterpret_cast<float *>(base + L.lam);     // log g
    float *Lm = lg + kL;                                      // Lam (inclusive prefix)
    float *gm = Lm + kL;                                      // exp(Lam)
    float *bt = gm + kL;                                      // beta
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + L.bar), *cbKQ = bar + 1;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + L.tslot);

    const __nv_bfloat16 *g = static_cast<const __nv_bfloat16 *>(p.g);
    const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(p.beta);

    // unit u = ((b * NC + c) * Hk + hk) * rep + hh, value head h = hk * rep + hh
    struct Unit { int b, c, hk, h, t0, len; };
    auto unit_of = [&](int u) {
        Unit x;
        const int hh = u % rep, grp = u / rep;
        x.hk = grp % Hk;
        const int bc = grp / Hk;
        x.c = bc % NC;
        x.b = bc / NC;
        x.h = x.hk * rep + hh;
        x.t0 = x.c * kL;
        x.len = min(kL, T - x.t0);
        return x;
    };

    if (tid == 0) {
        for (int j = 0; j < 2; ++j) mbar_init(bar + j, 1);
        fence_mbar_init();
    }
    if (tid == 32) {
        tma_prefetch_map(&maps.k);
        tma_prefetch_map(&maps.q);
        tma_prefetch_map(&maps.qk);
    }
    if (warp == 0) tmem_alloc(tslot, 256);
    const uint32_t lead = warp == 0 ? elect_one_sync() : 0u;   // the lane of warp 0 that issues products
    int nKQ = 0, wKQ = 0;
    // log g and beta of a unit (warp 0, two steps per lane), raw
    __nv_bfloat16 graw[2], braw[2];
    auto fetch_gb = [&](const Unit &x) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = 2 * lane + u;
            const size_t o = ((size_t)x.b * T + x.t0 + (t < x.len ? t : 0)) * Hv + x.h;
            graw[u] = g[o];
            braw[u] = beta[o];
        }
    };
    // K and Q of a (batch row, chunk, kv head) into kc and qc in their operand layout, one TMA
    // box each (5-D: the box walks 8-column blocks, rows past T are zeros), issued by thread 32
    auto fetch_kq = [&](const Unit &x) {
        if (tid == 32) {
            mbar_expect_tx(cbKQ, 2 * kL * DK * 2);
            tma_load_5d(kc, &maps.k, cbKQ, 0, x.t0, 0, x.hk, x.b);
            tma_load_5d(qc, &maps.q, cbKQ, 0, x.t0, 0, x.hk, x.b);
        }
        ++nKQ;
    };
    unsigned phase = 0;
    bool ok = true;
    uint32_t tmem = 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tmem = *tslot;
    griddep_wait();                                           // the previous kernel's writes are visible
    griddep_launch();
    // the first unit's g, beta, K and Q
    if (u_begin < u_end && warp == 0) fetch_gb(unit_of(u_begin));
    if (u_begin < u_end) fetch_kq(unit_of(u_begin));

    const uint32_t lo16 = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's M = 64 rows in tensor memory
    const M64Frag fa(warp, lane, kL);   // this thread's values of K K^T and Q K^T (M = 64, 64 columns)
    const M64Frag fw(warp, lane, DK);   // and of W (M = 64, DK columns)
    for (int u = u_begin, i = 0; u < u_end && ok; ++u, ++i) {
        const Unit x = unit_of(u);
        const int b = x.b, c = x.c, h = x.h, len = x.len;
        const bool newg = i == 0 || (u - 1) / rep != u / rep;
        const size_t chk = ((size_t)b * Hv + h) * NC + c;   // (b, h, c)
        if (newg) {
            // K and Q of the group have landed; [Q; K] leaves for the sweeps and the gradient kernel
            // (K chunk j: the 64 rows of Q, then the 64 rows of K; a group split between two CTAs is
            // written by both, alike)
            const bool w = mbar_wait(cbKQ, wKQ & 1);
            ++wKQ;
            ok = !__syncthreads_or(!w);
            if (!ok) break;
            if (tid == 32) {
                const size_t ckv = ((size_t)b * Hk + x.hk) * NC + c;
                tma_store_5d(&maps.qk, qc, 0, 0, 0, 0, (int)ckv);
                tma_store_5d(&maps.qk, kc, 0, 0, 1, 0, (int)ckv);
                bulk_commit();
            }
        }
        // K K^T -> columns [0, 64), Q K^T -> [64, 128) (M = 64: row m in lane m % 16 + 32 (m / 16))
        if (warp == 0) {
            constexpr uint32_t id = umma_idesc(1, kL, kL);
            umma_gemm_w(tmem, CmOp{kc, kL, 0, 0, false}, CmOp{kc, kL, 0, 0, false}, DK, id, false, lead);
            umma_gemm_w(tmem + kL, CmOp{qc, kL, 0, 0, false}, CmOp{kc, kL, 0, 0, false}, DK, id, false, lead);
            umma_commit_w(bar, lead);
        }
        // the re-computation backward: this unit's checkpoint rows as the gradient kernel's bf16
        // operand tiles while the products run (block of 64 rows s: element (r, c) at
        // s * 64 * DK + (c / 8) * 512 + r * 8 + c % 8; a warp writes 512 contiguous bytes)
        if (p.conv != nullptr && warp > 0) {
            const float *src = p.conv + chk * p.Dv * DK;
            __nv_bfloat16 *dst = p.s0m + chk * p.Dv * DK;
            const int per_blk = kL * (DK / 8), items = (p.Dv / kL) * per_blk;
#pragma unroll 4
            for (int it = tid - 32; it < items; it += 224) {
                const int blk = it / per_blk, w = it - blk * per_blk, ch = w / kL, row = w - ch * kL;
                const float *sp = src + (size_t)(blk * kL + row) * DK + 8 * ch;
                const float4 a = __ldcs(reinterpret_cast<const float4 *>(sp));
                const float4 b2 = __ldcs(reinterpret_cast<const float4 *>(sp + 4));
                const float x8[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w};
                *reinterpret_cast<uint4 *>(dst + (size_t)blk * kL * DK + ch * (kL * 8) + row * 8) = pack8_bf16(x8);
            }
        }
        // log g, beta and the in-chunk prefix Lam (warp 0: two steps per lane, a shuffle scan)
        if (warp == 0) {
            float l2[2], b2[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int t = 2 * lane + j;
                const bool in = t < len;
                l2[j] = in ? fmaxf(logf(__bfloat162float(graw[j])), -200.f) : 0.f;   // g = 0: exp(-200) = 0 in fp32; a nonzero bf16 g has log g > -93
                b2[j] = in ? __bfloat162float(braw[j]) : 0.f;
            }
            if (u + 1 < u_end) fetch_gb(unit_of(u + 1));   // used one unit later
            float s = l2[0] + l2[1];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y2 = __shfl_up_sync(kFullMask, s, off);
                if (lane >= off) s += y2;
            }
            const float e0 = s - l2[1];                       // inclusive prefix at step 2 lane
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int t = 2 * lane + j;
                const float Lt = j == 0 ? e0 : s;
                Lm[t] = Lt;
                gm[t] = expf(Lt);
                bt[t] = b2[j];
                p.lam[chk * kL + t] = Lt;
            }
        }
        tc_fence_before();
        ok = !__syncthreads_or(!mbar_wait(bar, phase & 1));
        ++phase;
        tc_fence_after();
        if (!ok) break;
        // A, and the decay-weighted Q K^T (i <= t) and K K^T (i < t) as bf16 operands stacked in
        // one 128-row core-matrix layout ([P; KKm]: row t of P, row 64 + t of KKm), straight from
        // tensor memory: a thread's 16x256b fragment, two columns per 4-byte store (a warp's store
        // covers one 128-byte core matrix)
        {
            float kx[16], qx[16];
            tmem_ld16x256_x4(tmem + lo16 + 32 * (warp >> 2), kx);
            tmem_ld16x256_x4(tmem + lo16 + kL + 32 * (warp >> 2), qx);
            tmem_wait_ld();
            unsigned char *PK = reinterpret_cast<unsigned char *>(p.pkm + chk * 2 * kL * kL);
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                const int t = fa.row(2 * k2);
                const float lt = Lm[t], bb = bt[t];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i0 = fa.col(j, 0);
                    float e2[2], a2[2], p2[2], m2[2];
#pragma unroll
                    for (int k1 = 0; k1 < 2; ++k1) {
                        const int ii = i0 + k1;
                        const float kk = kx[4 * j + 2 * k2 + k1], qq = qx[4 * j + 2 * k2 + k1];
                        e2[k1] = ii <= t ? expf(lt - Lm[ii]) : 0.f;
                        a2[k1] = ii < t ? bb * kk * e2[k1] : 0.f;
                        p2[k1] = qq * e2[k1];
                        m2[k1] = ii < t ? kk * e2[k1] : 0.f;
                    }
                    *reinterpret_cast<float2 *>(am + t * kP + i0) = make_float2(a2[0], a2[1]);
                    *reinterpret_cast<uint32_t *>(PK + cm_off(t, 2 * i0, 2 * kL)) = pack2_bf16(p2[0], p2[1]);
                    *reinterpret_cast<uint32_t *>(PK + cm_off(kL + t, 2 * i0, 2 * kL)) = pack2_bf16(m2[0], m2[1]);
                }
            }
        }
        if (tid == 32) bulk_wait_read();   // the last unit's store of T diag(beta) has read tcu
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // T = (I + A)^-1
        invert_unit_lower(am, ts, xs, tid, [] {});
        // T (for the backward), T diag(beta exp Lam) (W's operand) and T diag(beta) (stored for
        // the sweep) as bf16 operands; the blocks of T above the diagonal are zero
        {
            unsigned char *Tg = reinterpret_cast<unsigned char *>(p.tm + chk * kL * kL);
            for (int e = tid; e < kL * 8; e += 256) {
                const int t = e & (kL - 1), ch = e >> 6;
                float x8[8], w8[8], u8[8];
                if ((8 * ch) >> 4 <= t >> 4) {
                    const float4 a = *reinterpret_cast<const float4 *>(ts + t * kP + 8 * ch);
                    const float4 a2 = *reinterpret_cast<const float4 *>(ts + t * kP + 8 * ch + 4);
                    x8[0] = a.x; x8[1] = a.y; x8[2] = a.z; x8[3] = a.w; x8[4] = a2.x; x8[5] = a2.y; x8[6] = a2.z; x8[7] = a2.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) x8[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int col = 8 * ch + j;
                    u8[j] = x8[j] * bt[col];
                    w8[j] = u8[j] * gm[col];
                }
                const uint32_t o = cm_off(t, 16 * ch, kL);
                if (p.conv == nullptr) {
                    *reinterpret_cast<uint4 *>(tcw + o) = pack8_bf16(w8);
                    *reinterpret_cast<uint4 *>(tcu + o) = pack8_bf16(u8);
                }
                *reinterpret_cast<uint4 *>(Tg + o) = pack8_bf16(x8);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const bool kq_next = u + 1 < u_end && (u + 1) / rep != u / rep;
        if (p.conv != nullptr) {
            // the re-computation backward needs neither W nor T diag(beta); K and Q are free
            // (their products are done) once the stores of [Q; K] have read them
            if (tid == 32 && kq_next) bulk_wait_read();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (kq_next) fetch_kq(unit_of(u + 1));
            continue;
        }
        // W -> columns [0, DK) (K K^T and Q K^T are dead); T diag(beta) leaves by a bulk store
        if (warp == 0) {
            umma_gemm_w(tmem, CmOp{tcw, kL, 0, 0, false}, CmOp{kc, kL, 0, 0, true}, kL,
                        umma_idesc_t(1, kL, DK, false, true), false, lead);
            umma_commit_w(bar, lead);
        }
        // when the next unit starts another group, its K and Q are fetched into kc and qc
        // (free once this product is done) while this unit's W is read back
        if (tid == 32) {
            bulk_store(p.tcm + chk * kL * kL, tcu, kL * kL * 2);
            bulk_commit();
            if (kq_next) bulk_wait_read();                // the stores of [Q; K] have read kc, qc
        }
        ok = !__syncthreads_or(!mbar_wait(bar, phase & 1));
        ++phase;
        tc_fence_after();
        if (ok && kq_next) fetch_kq(unit_of(u + 1));
        if (ok) {
            // -W in its operand layout: a 4-byte pair of columns per value, a warp's store
            // covering one 128-byte core matrix
            unsigned char *Wg = reinterpret_cast<unsigned char *>(p.wm + chk * kL * DK);
#pragma unroll
            for (int r = 0; r < DK / 64; ++r) {
                float xw[16];
                tmem_ld16x256_x4(tmem + lo16 + (DK / 2) * (warp >> 2) + 32 * r, xw);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int k2 = 0; k2 < 2; ++k2) {
                        const int row = fw.row(2 * k2), col = fw.col(4 * r + j, 0);
                        *reinterpret_cast<uint32_t *>(Wg + cm_off(row, 2 * col, kL)) =
                            pack2_bf16(-xw[4 * j + 2 * k2], -xw[4 * j + 2 * k2 + 1]);
                    }
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (!ok && tid == 32) {
        report_status(p.status, kStatusTimeout);
        // copies still in flight land before the CTA exits (each wait bounded)
        if (nKQ > wKQ) mbar_wait(cbKQ, (nKQ - 1) & 1);
    }
    if (tid == 32) bulk_wait_all();   // no store still reads shared memory when the CTA exits
    if (!ok && warp == 0) {
        // products still in flight finish before the tensor memory is freed (bounded wait)
        umma_commit_w(bar, lead);
        mbar_wait(bar, phase & 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace gdn

namespace gdn {

namespace {

constexpr int kFwdMathWarps = 8;     // hold S (M = 64 fragment: 4 lane quarters x 2 column halves)
constexpr int kFwdThreads = 384;     // + a warpgroup: warp 8 issues the products, warp 9 the copies and stores
// registers: launched at 168 a thread; the control warpgroup gives up all but kFwdCtrlRegs, the
// math warpgroups take kFwdMathRegs (2 x 128 x 176 + 128 x 152 = 384 x 168)
constexpr int kFwdLaunchRegs = 168, kFwdMathRegs = 176, kFwdCtrlRegs = 152;
static_assert(2 * 128 * kFwdMathRegs + 128 * kFwdCtrlRegs <= kFwdThreads * kFwdLaunchRegs, "register split");

constexpr size_t kCkBox = (size_t)kL * 32 * 4;   // a [64][32] fp32 box of the checkpoint

struct SweepSmem {
    size_t wgrp, wc, tc, vb, qb, kb, pk, sop, dt, de, ysg, rsg, ckx, bar, tslot, total;
    int ck_in_w;
    __host__ __device__ SweepSmem(int DK) {
        size_t o = 0;
        // group W, two buffers (chunks alternate): -W, T diag(beta), V
        wgrp = (size_t)kL * DK * 2 + 2 * (size_t)kL * kL * 2;
        wc = o;                                // -W of the chunk                    A [64][DK]
        tc = wc + (size_t)kL * DK * 2;         // T diag(beta)                       A [64][64]
        vb = tc + (size_t)kL * kL * 2;         // V of the chunk, this block's 64 columns [64 t][64 v], 128-byte swizzle (read MN-major)
        o += 2 * wgrp;
        qb = o; o += (size_t)kL * DK * 2;      // Q of the chunk (kv head)           A [64][DK]
        kb = o; o += (size_t)kL * DK * 2;      // K of the chunk                     A [64][DK]; read MN-major as B
        pk = o; o += (size_t)2 * kL * kL * 2;  // [(Q K^T) o E_incl; (K K^T) o E_strict]   A [128][64]
        sop = o; o += (size_t)kL * DK * 2;     // S (64 value rows)                  B [64][DK]
        dt = o; o += (size_t)kL * kL * 2;      // Delta [64 t][64 v], read MN-major (B)
        de = o; o += (size_t)kL * kL * 2;      // diag(E_L) Delta [64 t][64 v], read MN-major (A, transposed)
        ysg = al(o, 1024); o = ysg + (size_t)kL * 128;       // y of a chunk, bf16 [64][64] in the 128-byte swizzle
        rsg = al(o, 1024); o = rsg + (size_t)2 * kL * 128;   // v - u of a chunk, fp32 [2][64][32] in the 128-byte swizzle
        // the fp32 checkpoint of a chunk, staged for TMA stores as DK / 32 boxes [64][32] fp32 in
        // the 128-byte swizzle (8 KB each): the first ck_in_w in the chunk's group W buffer (free
        // once Delta is formed), the rest here, two buffers (chunks alternate)
        ck_in_w = (int)(wgrp / kCkBox) < DK / 32 ? (int)(wgrp / kCkBox) : DK / 32;
        ckx = al(o, 1024); o = ckx + 2 * (size_t)(DK / 32 - ck_in_w) * kCkBox;
        bar = al(o, 8); o = bar + 16 * 8;      // see the kernel
        // (V is read in the 128-byte swizzle: its tiles start at 1024-byte boundaries, as do both
        // groups W for every DK here: the W tile is a multiple of 8 KB)
        tslot = o; o += 16;
        total = o + 1024;
        if (total < kOneCtaSmem) total = kOneCtaSmem;
    }
};

}  // namespace

// One CTA per (64-row block of the state, value head, batch row), carrying that block of the
// state through the chunks. Warps 0-7 hold the fp32 state (registers: the 16x256b fragment of
// an M = 64 accumulator, 2 rows x DK/8 columns per thread) and do the element-wise work; warp 8
// issues the products (one elected lane) and warp 9 the copies and the bf16 state's stores, so
// that no math warp stalls on an issue and no block barrier runs per chunk: every hand-off is an
// mbarrier. Per chunk the products are (fp32 accumulators in tensor memory, M = 64: row r in
// lane r % 16 + 32 (r / 16)):
//   [0, DK)               Sigma = (diag(E_L) Delta)^T K: S <- exp(Lam_L) S + Sigma
//   [DK, DK + 64)         Delta = (T diag(beta)) V + (-W) S^T (chunk row t, value column)
//   [DK + 64, + 128)      Q S^T, then K S^T
//   [DK + 192, + 256)     P Delta, then KKm Delta
// and y = diag(exp Lam) (Q S^T) + P Delta, u = diag(exp Lam) (K S^T) + KKm Delta.
// Hand-offs of chunk c (each completes once per chunk):
//   math -> control (8 warp arrivals): bS  S written as an operand;  bE  the previous chunk's
//                                      y and u read out;  bDt  Delta written as operands
//   control -> math: mD, mQ, mU, mY  the product groups (commits);  fS  the state operand's
//                    tile is free (the products that read it are done, its store has read it)
// Q and K arrive as separate [64][DK] tiles (boxes of the [Q; K] block); group W is
// double-buffered and fetched two chunks ahead. y and v - u leave by TMA stores from staging
// tiles (the copy warp, once bE says they are written).
//
// With kLite, the same sweep takes only the state through the chunks, for the sequence-parallel
// form: no checkpoints, bf16 states, y or v - u, so no Q S^T, K S^T, P Delta or KKm Delta
// products. Its first Dv / 64 CTAs of a head (the "ends") start from zero and write the end state
// to S_T; the next Dk / 64 (the "maps") take rows r0 .. r0 + 63 of the Dk x Dk identity with V
// counted as zero, so the chunks compose S <- S (exp(Lam_L) I - W^T diag(E_L) K), and write that
// map to maps_M and its transpose to maps_Mt.
template <int E, bool kLite>
__global__ void __launch_bounds__(kFwdThreads, 1) chunk_sweep_kernel(ChunkParams p, const __grid_constant__ ChunkFwdMaps maps) {
    constexpr int DK = 32 * E;
    constexpr int SC = DK / 2;                // state columns per warp half
    constexpr int NS = SC / 2;                // state values per thread (2 rows x 2 columns x SC / 8 repetitions)
    static_assert(DK + 320 <= 512, "tensor memory holds Sigma, Delta, Q S^T, K S^T, P Delta and KKm Delta");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool math = warp < kFwdMathWarps;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int T = p.T, Dv = p.Dv, Hv = p.Hv, NC = p.NC;
    const bool infer = !kLite && p.ckpt == nullptr;            // inference: nothing saved, no v - u
    const bool ends = !kLite || split < Dv / kL;               // a block of value rows (else of the identity)
    const bool maps_cta = kLite && !ends;
    const int r0 = (ends ? split : split - Dv / kL) * kL;
    const int hw = (warp >> 2) & 1;                             // warp half
    const uint32_t lane16 = (uint32_t)(32 * (warp & 3)) << 16;   // tensor-memory lane base of this warp's M = 64 rows

    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(al(reinterpret_cast<size_t>(smem_raw), 1024));
    const SweepSmem L(DK);
    unsigned char *qb = base + L.qb, *kb = base + L.kb, *pk = base + L.pk;
    unsigned char *sop = base + L.sop, *dt = base + L.dt, *de = base + L.de, *ysg = base + L.ysg, *rsg = base + L.rsg;
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + L.bar);
    uint64_t *mD = bar, *mQ = bar + 1, *mU = bar + 2, *mY = bar + 3, *cbQ = bar + 4, *cbP = bar + 5;
    uint64_t *bW = bar + 6, *cbK = bar + 8;                     // bW[2]: one per buffer
    uint64_t *bS = bar + 10, *bE = bar + 11, *bDt = bar + 12, *fS = bar + 13, *mX = bar + 14, *bK = bar + 15;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + L.tslot);
    // the buffer of chunk c's group W (-W, T diag(beta), V)
    auto wbuf = [&](int c) { return base + L.wc + (size_t)(c & 1) * L.wgrp; };
    // box q of chunk c's staged fp32 checkpoint
    auto ck_box = [&](int c, int q) {
        return q < L.ck_in_w ? wbuf(c) + q * kCkBox
                             : base + L.ckx + ((size_t)(c & 1) * (DK / 32 - L.ck_in_w) + (q - L.ck_in_w)) * kCkBox;
    };

    const size_t head = (size_t)b * Hv + h;
    const int hk = h / (Hv / p.Hk);
    const int qkblk0 = (b * p.Hk + hk) * NC;                   // [Q; K] block of chunk 0 of this kv head

    if (tid == 0) {
        for (int i = 0; i < 10; ++i) mbar_init(bar + i, 1);
        for (int i = 10; i < 13; ++i) mbar_init(bar + i, kFwdMathWarps);
        for (int i = 13; i < 15; ++i) mbar_init(bar + i, 1);
        mbar_init(bK, kFwdMathWarps);
        fence_mbar_init();
    }
    if (warp == kFwdMathWarps + 1 && lane == 0) {
        tma_prefetch_map(&maps.vb);
        tma_prefetch_map(&maps.qk);
        tma_prefetch_map(&maps.y);
        tma_prefetch_map(&maps.r);
    }
    if (warp == kFwdMathWarps) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tSg = tmem, tD = tmem + DK, tY = tmem + DK + 64, tU = tmem + DK + 128, tPy = tmem + DK + 192,
                   tPu = tmem + DK + 256;
    griddep_wait();                                           // the previous kernel's writes are visible
    griddep_launch();

    bool fail = false;
    if (!math) {
        regs_dec<kFwdCtrlRegs>();            // the whole control warpgroup, at one point of the code
        if (warp == kFwdMathWarps) {
            // ================================================================ product warp
            const uint32_t lead = elect_one_sync();
            constexpr uint32_t id64 = umma_idesc(1, kL, kL);
            // U = (T diag(beta)) V starts Delta's accumulator (the first chunk's here, each later
            // one once the previous Delta is read out)
            if (ends) {
                const bool w = mbar_wait(bW, 0);
                fail = __any_sync(kFullMask, !w);
                if (!fail) {
                    tc_fence_after();
                    unsigned char *g = wbuf(0);
                    umma_gemm_wd(tD, CmOp{g + (L.tc - L.wc), kL, 0, 0, false}, sw128_mnmajor(g + (L.vb - L.wc)), 2048 >> 4,
                                 kL, umma_idesc_t(1, kL, kL, false, true), false, lead);
                }
            }
            for (int c = 0; c < NC && !fail; ++c) {
                unsigned char *wc = wbuf(c);
                // ---- Delta += (-W) S^T once S is written (the maps: Delta = (-W) S^T)
                bool w = mbar_wait(bS, c & 1) && (!maps_cta || mbar_wait(bW + (c & 1), (c >> 1) & 1));
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                tc_fence_after();
                umma_gemm_w(tD, CmOp{wc, kL, 0, 0, false}, CmOp{sop, kL, 0, 0, false}, DK, id64, ends, lead);
                umma_commit_w(mD, lead);
                if constexpr (kLite) {
                    // ---- Sigma = (diag(E_L) Delta)^T K once Delta is written; then U of the next
                    // chunk (the ends)
                    w = mbar_wait(bDt, c & 1) && mbar_wait(cbK, c & 1);
                    if (__any_sync(kFullMask, !w)) { fail = true; break; }
                    tc_fence_after();
                    umma_gemm_w(tSg, CmOp{de, kL, 0, 0, true}, CmOp{kb, kL, 0, 0, true}, kL,
                                umma_idesc_t(1, kL, DK, true, true), false, lead);
                    umma_commit_w(mU, lead);
                    if (ends && c + 1 < NC) {
                        w = mbar_wait(bW + ((c + 1) & 1), ((c + 1) >> 1) & 1);
                        if (__any_sync(kFullMask, !w)) { fail = true; break; }
                        tc_fence_after();
                        unsigned char *g = wbuf(c + 1);
                        umma_gemm_wd(tD, CmOp{g + (L.tc - L.wc), kL, 0, 0, false}, sw128_mnmajor(g + (L.vb - L.wc)),
                                     2048 >> 4, kL, umma_idesc_t(1, kL, kL, false, true), false, lead);
                    }
                    continue;
                }
                // ---- Q S^T and K S^T once the previous chunk's are read out and Q, K landed
                w = (c == 0 || mbar_wait(bE, (c - 1) & 1)) && mbar_wait(cbQ, c & 1) && mbar_wait(cbK, c & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                tc_fence_after();
                umma_gemm_w(tY, CmOp{qb, kL, 0, 0, false}, CmOp{sop, kL, 0, 0, false}, DK, id64, false, lead);
                if (!infer) umma_gemm_w(tU, CmOp{kb, kL, 0, 0, false}, CmOp{sop, kL, 0, 0, false}, DK, id64, false, lead);
                umma_commit_w(mQ, lead);
                // ---- Sigma = (diag(E_L) Delta)^T K once Delta is written; then P Delta and KKm Delta
                w = mbar_wait(bDt, c & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                tc_fence_after();
                umma_gemm_w(tSg, CmOp{de, kL, 0, 0, true}, CmOp{kb, kL, 0, 0, true}, kL, umma_idesc_t(1, kL, DK, true, true),
                            false, lead);
                umma_commit_w(mU, lead);
                w = mbar_wait(cbP, c & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                tc_fence_after();
                umma_gemm_w(tPy, CmOp{pk, 2 * kL, 0, 0, false}, CmOp{dt, kL, 0, 0, true}, kL,
                            umma_idesc_t(1, kL, kL, false, true), false, lead);
                if (!infer)
                umma_gemm_w(tPu, CmOp{pk, 2 * kL, kL, 0, false}, CmOp{dt, kL, 0, 0, true}, kL,
                            umma_idesc_t(1, kL, kL, false, true), false, lead);
                umma_commit_w(mY, lead);
                // ---- U of the next chunk (Delta was read out before bDt)
                if (c + 1 < NC) {
                    w = mbar_wait(bW + ((c + 1) & 1), ((c + 1) >> 1) & 1);
                    if (__any_sync(kFullMask, !w)) { fail = true; break; }
                    tc_fence_after();
                    unsigned char *g = wbuf(c + 1);
                    umma_gemm_wd(tD, CmOp{g + (L.tc - L.wc), kL, 0, 0, false}, sw128_mnmajor(g + (L.vb - L.wc)), 2048 >> 4,
                                 kL, umma_idesc_t(1, kL, kL, false, true), false, lead);
                }
            }
            if (fail) {
                // products still in flight finish before the tensor memory is freed (bounded wait)
                umma_commit_w(mX, lead);
                mbar_wait(mX, 0);
            }
        } else if (warp == kFwdMathWarps + 1) {
            // ================================================================ copy warp (lane 0)
            if (lane == 0) {
                int nQ = 0, nP = 0, nK = 0, nW[2] = {0, 0};
                auto issue_w = [&](int cc) {               // group W of chunk cc: -W, T diag(beta), V of this block
                    const size_t ck = head * NC + cc;
                    unsigned char *g = wbuf(cc);
                    uint64_t *bw = bW + (cc & 1);
                    mbar_expect_tx(bw, maps_cta ? kL * DK * 2 : kL * DK * 2 + 2 * kL * kL * 2);
                    bulk_load(g, p.wm + ck * kL * DK, kL * DK * 2, bw);
                    if (ends) {
                        bulk_load(g + (L.tc - L.wc), p.tcm + ck * kL * kL, kL * kL * 2, bw);
                        tma_load_4d(g + (L.vb - L.wc), &maps.vb, bw, r0, h, cc * kL, b);
                    }
                    ++nW[cc & 1];
                };
                auto copy_Q = [&](int cc) {                // Q of chunk cc: rows 0-63 of its [Q; K] block
                    mbar_expect_tx(cbQ, kL * DK * 2);
                    tma_load_5d(qb, &maps.qk, cbQ, 0, 0, 0, 0, qkblk0 + cc);
                    ++nQ;
                };
                auto copy_K = [&](int cc) {                // K of chunk cc: rows 64-127
                    mbar_expect_tx(cbK, kL * DK * 2);
                    tma_load_5d(kb, &maps.qk, cbK, 0, 0, 1, 0, qkblk0 + cc);
                    ++nK;
                };
                // y and v - u of chunk cc leave from their staging tiles
                auto store_out = [&](int cc) {
                    tma_store_4d(&maps.y, ysg, r0, h, cc * kL, b);
                    if (!infer) tma_store_5d(&maps.r, rsg, 0, cc * kL, r0 / 32, h, b);
                    bulk_commit();
                };
                auto copy_P = [&](int cc) {                // [P; KKm] of chunk cc
                    mbar_expect_tx(cbP, 2 * kL * kL * 2);
                    bulk_load(pk, p.pkm + (head * NC + cc) * 2 * kL * kL, 2 * kL * kL * 2, cbP);
                    ++nP;
                };
                for (int cc = 0; cc < 2 && cc < NC; ++cc) issue_w(cc);
                copy_K(0);
                if constexpr (!kLite) {
                    copy_Q(0);
                    copy_P(0);
                }
                for (int c = 0; c < NC && kLite; ++c) {
                    // K and group W only. Sigma done (mU) frees K; it also means that every product
                    // issued before it is done (U and Delta of chunk c), so group W's buffer of
                    // chunk c takes chunk c + 2; and the state operand's tile is free
                    if (!mbar_wait(mU, c & 1) || !mbar_wait(bDt, c & 1)) { fail = true; break; }
                    if (c + 1 < NC) copy_K(c + 1);
                    if (c + 2 < NC) issue_w(c + 2);
                    mbar_arrive(fS);
                }
                for (int c = 0; c < NC && !kLite; ++c) {
                    const size_t chk = head * NC + c;
                    // the bf16 state leaves (the backward's operand) once written
                    if (!mbar_wait(bS, c & 1)) { fail = true; break; }
                    if (!infer) {
                        bulk_store(p.s0m + (chk * gridDim.x + split) * kL * DK, sop, kL * DK * 2);
                        bulk_commit();
                    }
                    // the previous chunk's y and v - u once staged
                    if (c > 0) {
                        if (!mbar_wait(bE, (c - 1) & 1)) { fail = true; break; }
                        store_out(c - 1);
                    }
                    // Q S^T and K S^T are done: Q is free
                    if (!mbar_wait(mQ, c & 1)) { fail = true; break; }
                    if (c + 1 < NC) copy_Q(c + 1);
                    // Sigma is done: K is free
                    if (!mbar_wait(mU, c & 1) || !mbar_wait(bDt, c & 1)) { fail = true; break; }
                    if (c + 1 < NC) copy_K(c + 1);
                    // the staged fp32 checkpoint leaves; once the stores before it have read the
                    // state operand's tile and the y, v - u staging, they are free (fS); once it
                    // has been read too, group W's buffer takes chunk c + 2
                    if (!mbar_wait(bK, c & 1)) { fail = true; break; }
                    if (!infer) {
                        for (int q = 0; q < DK / 32; ++q) tma_store_2d(&maps.ck, ck_box(c, q), 32 * q, (int)(chk * Dv + r0));
                        bulk_commit();
                        bulk_wait_read_but<1>();
                    } else {
                        bulk_wait_read();                   // no checkpoint store: the newest group is y's
                    }
                    mbar_arrive(fS);
                    bulk_wait_read();
                    if (c + 2 < NC) issue_w(c + 2);
                    // P Delta and KKm Delta are done: [P; KKm] is free
                    if (!mbar_wait(mY, c & 1)) { fail = true; break; }
                    if (c + 1 < NC) copy_P(c + 1);
                }
                if (fail) {
                    // copies still in flight land before the CTA exits (each wait bounded)
                    if (nQ > 0) mbar_wait(cbQ, (nQ - 1) & 1);
                    if (nP > 0) mbar_wait(cbP, (nP - 1) & 1);
                    if (nK > 0) mbar_wait(cbK, (nK - 1) & 1);
                    for (int i = 0; i < 2; ++i)
                        if (nW[i] > 0) mbar_wait(bW + i, (nW[i] - 1) & 1);
                } else if (kLite) {
                } else if (mbar_wait(bE, (NC - 1) & 1)) {
                    store_out(NC - 1);                      // the last chunk's y and v - u
                } else {
                    fail = true;
                }
                bulk_wait_all();                            // the bf16 states are complete
            }
            fail = __shfl_sync(kFullMask, fail, 0);
        }
    } else {
        regs_inc<kFwdMathRegs>();
        // ================================================================ math warps
        // this thread's fragment of the state (rows fs.row(k), columns fs.col(j, k)) and of the
        // 64-column accumulators (chunk rows ta, tb, value columns fd.col(j, 0), + 1)
        const M64Frag fs(warp, lane, DK), fd(warp, lane, kL);
        const int ta = fd.row(0), tb = fd.row(2);
        float S[NS];
#pragma unroll
        for (int j = 0; j < NS / 4; ++j)
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                float2 s2 = make_float2(0.f, 0.f);
                const int row = r0 + fs.row(2 * k2), col = fs.col(j, 0);
                if (maps_cta)
                    s2 = make_float2(row == col ? 1.f : 0.f, row == col + 1 ? 1.f : 0.f);
                else if (!kLite && p.S0 != nullptr)
                    s2 = *reinterpret_cast<const float2 *>(p.S0 + (head * Dv + row) * DK + col);
                S[4 * j + 2 * k2] = s2.x;
                S[4 * j + 2 * k2 + 1] = s2.y;
            }
        const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
        // Lam_L, Lam_ta, Lam_tb and v of rows ta, tb (this thread's columns) of chunk cc, loaded
        // a chunk ahead and kept raw until used (rows past T: v zeros)
        float nlL, nla, nlb;
        uint32_t nva[4], nvb[4];
        auto load_lam = [&](int cc) {
            const float *lm = p.lam + (head * NC + cc) * kL;
            nlL = lm[kL - 1];
            nla = lm[ta];
            nlb = lm[tb];
        };
        auto load_v = [&](int cc) {
            const int tt0 = cc * kL, ln = min(kL, T - tt0);
            const size_t ra = (((size_t)b * T + tt0 + ta) * Hv + h) * Dv + r0, rb = (((size_t)b * T + tt0 + tb) * Hv + h) * Dv + r0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = fd.col(j, 0);
                nva[j] = ta < ln ? *reinterpret_cast<const uint32_t *>(v + ra + col) : 0u;
                nvb[j] = tb < ln ? *reinterpret_cast<const uint32_t *>(v + rb + col) : 0u;
            }
        };
        // the state as a bf16 operand (stmatrix: 4 8x8 blocks per instruction)
        auto write_sop = [&]() {
#pragma unroll
            for (int j = 0; j < NS / 4; j += 2) {
                const uint32_t a = frag_row_addr(smem_addr(sop), kL, 16 * (warp & 3), (DK / 16) * hw + j, lane);
                stmatrix_x4(a, pack2_bf16(S[4 * j], S[4 * j + 1]), pack2_bf16(S[4 * j + 2], S[4 * j + 3]),
                            pack2_bf16(S[4 * j + 4], S[4 * j + 5]), pack2_bf16(S[4 * j + 6], S[4 * j + 7]));
            }
        };
        auto warp_done = [&](uint64_t *bar_) {
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_);
        };
        // y and v - u of chunk cc from tensor memory (its decays: ga, gb = exp(Lam) of rows ta,
        // tb; v pairs va, vb), staged in the 128-byte swizzle for the copy warp's TMA stores (rows
        // past T are clipped by them): y row t at t * 128, 16-byte chunk j (8 columns) at
        // j ^ (t % 8); v - u in two boxes of 32 columns, 16-byte chunk j (4 columns) likewise
        auto epilogue = [&](float ga, float gb, const uint32_t (&va)[4], const uint32_t (&vb)[4]) {
            {
                float q[16], pq[16];
                tmem_ld16x256_x4(tY + lane16 + 32 * hw, q);
                tmem_ld16x256_x4(tPy + lane16 + 32 * hw, pq);
                tmem_wait_ld();
                uint32_t yv[8];   // pairs (j, row ta), (j, row tb)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    yv[2 * j] = pack2_bf16(fmaf(ga, q[4 * j], pq[4 * j]), fmaf(ga, q[4 * j + 1], pq[4 * j + 1]));
                    yv[2 * j + 1] = pack2_bf16(fmaf(gb, q[4 * j + 2], pq[4 * j + 2]), fmaf(gb, q[4 * j + 3], pq[4 * j + 3]));
                }
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                    const int m = lane >> 3, t = 16 * (warp & 3) + 8 * (m & 1) + (lane & 7), cb = 4 * hw + j + (m >> 1);
                    stmatrix_x4(smem_addr(ysg) + t * 128 + ((cb ^ (t & 7)) << 4), yv[2 * j], yv[2 * j + 1], yv[2 * j + 2],
                                yv[2 * j + 3]);
                }
            }
            if (!infer) {
                float k[16], pu[16];
                tmem_ld16x256_x4(tU + lane16 + 32 * hw, k);
                tmem_ld16x256_x4(tPu + lane16 + 32 * hw, pu);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int col = fd.col(j, 0);
                    const uint32_t oc = (col >> 5) * (kL * 128) + (col & 3) * 4;
                    const float2 xa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&va[j]));
                    const float2 xb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&vb[j]));
                    *reinterpret_cast<float2 *>(rsg + oc + ta * 128 + ((((col & 31) >> 2) ^ (ta & 7)) << 4)) =
                        make_float2(xa.x - fmaf(ga, k[4 * j], pu[4 * j]), xa.y - fmaf(ga, k[4 * j + 1], pu[4 * j + 1]));
                    *reinterpret_cast<float2 *>(rsg + oc + tb * 128 + ((((col & 31) >> 2) ^ (tb & 7)) << 4)) =
                        make_float2(xb.x - fmaf(gb, k[4 * j + 2], pu[4 * j + 2]), xb.y - fmaf(gb, k[4 * j + 3], pu[4 * j + 3]));
                }
            }
        };
        load_lam(0);
        if (!kLite && !infer) load_v(0);
        float decay = 1.f, pga = 1.f, pgb = 1.f;     // exp(Lam_L), exp(Lam_ta), exp(Lam_tb) of the previous chunk
        uint32_t pva[4], pvb[4];                      // v pairs of the previous chunk
        for (int c = 0; c < NC; ++c) {
            const float lL = nlL, la = nla, lb = nlb;
            uint32_t cva[4], cvb[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                cva[j] = nva[j];
                cvb[j] = nvb[j];
            }
            if (c + 1 < NC) {
                load_lam(c + 1);
                if (!kLite && !infer) load_v(c + 1);
            }
            // ---- S <- exp(Lam_L) S + Sigma of the previous chunk; S as an operand
            if (c > 0) {
                const bool w = mbar_wait(mU, (c - 1) & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < NS / 16; ++i) {
                    float x[16];
                    tmem_ld16x256_x4(tSg + lane16 + SC * hw + 32 * i, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) S[16 * i + e] = fmaf(decay, S[16 * i + e], x[e]);
                }
                // the state operand's tile: the previous chunk's products and store are done with it
                const bool w2 = mbar_wait(fS, (c - 1) & 1);
                if (__any_sync(kFullMask, !w2)) { fail = true; break; }
            }
            write_sop();
            warp_done(bS);
            // ---- y and v - u of the previous chunk
            if (!kLite && c > 0) {
                const bool w = mbar_wait(mY, (c - 1) & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                tc_fence_after();
                epilogue(pga, pgb, pva, pvb);
                warp_done(bE);
            }
            // ---- Delta as operands: Delta (for P Delta, KKm Delta) and diag(E_L) Delta (for the
            // update); their tiles are free since the previous chunk's products are done (mY)
            {
                const bool w = mbar_wait(mD, c & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
            }
            tc_fence_after();
            {
                float x[16];
                tmem_ld16x256_x4(tD + lane16 + 32 * hw, x);
                tmem_wait_ld();
                const float ea = expf(lL - la), eb = expf(lL - lb);
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                    const uint32_t o = frag_row_addr(0, kL, 16 * (warp & 3), 4 * hw + j, lane);
                    if (!kLite)
                        stmatrix_x4(smem_addr(dt) + o, pack2_bf16(x[4 * j], x[4 * j + 1]),
                                    pack2_bf16(x[4 * j + 2], x[4 * j + 3]), pack2_bf16(x[4 * j + 4], x[4 * j + 5]),
                                    pack2_bf16(x[4 * j + 6], x[4 * j + 7]));
                    stmatrix_x4(smem_addr(de) + o, pack2_bf16(ea * x[4 * j], ea * x[4 * j + 1]),
                                pack2_bf16(eb * x[4 * j + 2], eb * x[4 * j + 3]), pack2_bf16(ea * x[4 * j + 4], ea * x[4 * j + 5]),
                                pack2_bf16(eb * x[4 * j + 6], eb * x[4 * j + 7]));
                }
            }
            warp_done(bDt);
            if (!kLite) {
                // the fp32 checkpoint while Sigma runs (off the path from S to the next chunk's
                // products), staged for the copy warp's TMA stores: box q = col / 32 holds row r,
                // 16-byte piece j = (col % 32) / 4 at r * 128 + ((j ^ (r % 8)) << 4); the group W
                // buffer of this chunk is free (Delta is formed, mD) until the copy warp refills it
                // after these stores have read it
#pragma unroll
                for (int j = 0; j < NS / 4 && !infer; ++j)
#pragma unroll
                    for (int k2 = 0; k2 < 2; ++k2) {
                        const int row = fs.row(2 * k2), col = fs.col(j, 0);
                        unsigned char *box = ck_box(c, col >> 5);
                        *reinterpret_cast<float2 *>(box + row * 128 + ((((col & 31) >> 2) ^ (row & 7)) << 4) + (col & 3) * 4) =
                            make_float2(S[4 * j + 2 * k2], S[4 * j + 2 * k2 + 1]);
                    }
                warp_done(bK);
            }
            decay = expf(lL);
            pga = expf(la);
            pgb = expf(lb);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                pva[j] = cva[j];
                pvb[j] = cvb[j];
            }
        }
        if (!fail) {
            // the last chunk: its update, S_T, and its y and v - u
            bool w = mbar_wait(mU, (NC - 1) & 1);
            fail = __any_sync(kFullMask, !w);
            if (!fail) {
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < NS / 16; ++i) {
                    float x[16];
                    tmem_ld16x256_x4(tSg + lane16 + SC * hw + 32 * i, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) S[16 * i + e] = fmaf(decay, S[16 * i + e], x[e]);
                }
                float *out = maps_cta ? p.maps_M : p.S_T;
                const int orows = maps_cta ? DK : Dv;
                if (out != nullptr)
#pragma unroll
                    for (int j = 0; j < NS / 4; ++j)
#pragma unroll
                        for (int k2 = 0; k2 < 2; ++k2)
                            *reinterpret_cast<float2 *>(out + (head * orows + r0 + fs.row(2 * k2)) * DK + fs.col(j, 0)) =
                                make_float2(S[4 * j + 2 * k2], S[4 * j + 2 * k2 + 1]);
                // the map also transposed (the reverse scan's operand)
                if (maps_cta && p.maps_Mt != nullptr)
#pragma unroll
                    for (int j = 0; j < NS / 4; ++j)
#pragma unroll
                        for (int k2 = 0; k2 < 2; ++k2) {
                            const int row = r0 + fs.row(2 * k2), col = fs.col(j, 0);
                            p.maps_Mt[(head * DK + col) * DK + row] = S[4 * j + 2 * k2];
                            p.maps_Mt[(head * DK + col + 1) * DK + row] = S[4 * j + 2 * k2 + 1];
                        }
                // (the staging tiles are free once the previous chunk's stores have read them: fS)
                w = kLite || (mbar_wait(mY, (NC - 1) & 1) && mbar_wait(fS, (NC - 1) & 1));
                fail = __any_sync(kFullMask, !w);
                if (!fail && !kLite) {
                    tc_fence_after();
                    epilogue(pga, pgb, pva, pvb);
                    warp_done(bE);
                }
            }
        }
    }
    if (fail && lane == 0) report_status(p.status, kStatusTimeout);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kFwdMathWarps) tmem_dealloc(tmem, 512);
}

size_t chunk_prep_smem(int Dk, int Dv) {
    (void)Dv;
    return PrepSmem(Dk).total;
}
size_t chunk_sweep_smem(int Dk) { return SweepSmem(Dk).total; }

template <int E, bool kLite>
static cudaError_t prepare_sweep(size_t ss) {
    // the sweep's register split waits for registers that only a launch of kFwdLaunchRegs per
    // thread provides
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, chunk_sweep_kernel<E, kLite>);
    if (err != cudaSuccess) return err;
    if (fa.numRegs < kFwdLaunchRegs || fa.maxThreadsPerBlock < kFwdThreads) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(chunk_sweep_kernel<E, kLite>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss);
}

template <int E>
static cudaError_t launch_chunk_t(const ChunkParams &p, const ChunkFwdMaps &maps, cudaStream_t s, int stages) {
    constexpr int DK = 32 * E;
    const size_t sp = PrepSmem(DK).total, ss = SweepSmem(DK).total;
    cudaError_t err = cudaSuccess;
    if (stages & kStagePrep) {
        err = cudaFuncSetAttribute(chunk_prep_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp);
        if (err != cudaSuccess) return err;
        // two prep CTAs share an SM: ask for the largest shared-memory carve-out
        err = cudaFuncSetAttribute(chunk_prep_kernel<E>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (err != cudaSuccess) return err;
        timing_mark("chunk_prep", 0, s);
        const int units = p.NC * p.Hv * p.B;
        int dev = 0, sms = 0;
        err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
        // persistent: two CTAs per SM
        err = launch_pdl(chunk_prep_kernel<E>, dim3(units < 2 * sms ? units : 2 * sms), dim3(256), sp, s, p, units, maps);
        timing_mark("chunk_prep", 1, s);
        if (err != cudaSuccess) return err;
    }
    if (stages & kStageSweep) {
        err = prepare_sweep<E, false>(ss);
        if (err != cudaSuccess) return err;
        timing_mark("chunk_sweep", 0, s);
        err = launch_pdl(chunk_sweep_kernel<E, false>, dim3(p.Dv / kL, p.Hv, p.B), dim3(kFwdThreads), ss, s, p, maps);
        timing_mark("chunk_sweep", 1, s);
        if (err != cudaSuccess) return err;
    }
    if (stages & kStageLite) {
        // the end states from zero (Dv / 64 CTAs of a head) and the maps (Dk / 64) in one launch
        err = prepare_sweep<E, true>(ss);
        if (err != cudaSuccess) return err;
        timing_mark("chunk_lite", 0, s);
        err = launch_pdl(chunk_sweep_kernel<E, true>, dim3(p.Dv / kL + DK / kL, p.Hv, p.B), dim3(kFwdThreads), ss, s, p,
                         maps);
        timing_mark("chunk_lite", 1, s);
    }
    return err;
}

cudaError_t launch_chunk_fwd(const ChunkParams &p, const ChunkFwdMaps &maps, int Dk, cudaStream_t s, int stages) {
    switch (Dk) {
        case 64: return launch_chunk_t<2>(p, maps, s, stages);
        case 128: return launch_chunk_t<4>(p, maps, s, stages);
        case 192: return launch_chunk_t<6>(p, maps, s, stages);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
