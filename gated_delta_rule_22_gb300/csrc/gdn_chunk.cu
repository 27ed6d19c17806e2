// gdn_chunk.cu -- the forward of the gated delta rule in its chunkwise (dense) form on the
// 5th-generation tensor cores, for bf16 inputs and chunks of 64 steps.
//
// The recurrence is that of mlx issue #4614 ("Recurrence used for the references"); the
// chunkwise form is derived from it (the pages do not give it). Per value head and chunk of
// L = 64 steps with start state S0 [Dv, Dk] (lam_t = log g_t, Lam its in-chunk prefix sum,
// E(s, i) = exp(Lam_s - Lam_i) <= 1, never a division by a decay):
//     A[t, i] = beta_t (k_t . k_i) E(t, i)  (i < t),   T = (I + A)^-1
//     W = T diag(beta exp Lam) K,   U = T diag(beta) V,   Delta = U - W S0^T
//     y = diag(exp Lam) Q S0^T + ((Q K^T) o E_incl) Delta
//     u = diag(exp Lam) K S0^T + ((K K^T) o E_strict) Delta      (u_t = g_t S_{t-1} k_t)
//     S_L = exp(Lam_L) S0 + (diag(E(L, .)) Delta)^T K
// chunk_prep_kernel computes what does not depend on the state, for all chunks at once;
// chunk_sweep_kernel carries the state through the chunks of one head. Products run on the
// tensor cores with bf16 operands and fp32 accumulators in tensor memory; T is formed in
// fp32 on the CUDA cores. The outputs (y, the chunk-start states, v - u) are those of the
// sequential forward, so the backward consumes them unchanged.
#include "gdn_umma.cuh"

namespace gdn {

namespace {

constexpr int kL = 64;           // chunk length of the tensor-core forward
constexpr int kP = 68;           // row of prep's fp32 64 x 64 work matrices (16-byte aligned, conflict-free float4 columns)
// Both kernels hold all 512 tensor-memory columns, so each must be alone on its SM: they ask
// for more than half of the shared memory.
constexpr size_t kOneCtaSmem = 120 * 1024;

__host__ __device__ inline size_t al(size_t x, size_t a) { return (x + a - 1) / a * a; }

// U leaves prep by TMA stores of [64][32] fp32 boxes staged in the 128-byte swizzle, in
// kUSlots slots of 8 KB that reuse T, the inversion scratch and the T operands (slots 0-3;
// the next unit writes them from its inversion on) and A (slots 4-5; written from the next
// unit's start): all are dead once the products W and U are done.
constexpr int kUSlots = 6;

struct PrepSmem {
    size_t kc, qc, kk, qk, am, ts, xs, tcw, tcu, vc, lam, bar, tslot, ustg, ustg2, total;
    __host__ __device__ PrepSmem(int DK, int Dv) {
        size_t o = 0;
        kc = o; o += (size_t)kL * DK * 2;           // K of the chunk, bf16 operand [64][DK]
        qc = o; o += (size_t)kL * DK * 2;           // Q of the chunk
        kk = o; o += (size_t)kL * kP * 4;           // K K^T, fp32
        qk = o; o += (size_t)kL * kP * 4;           // Q K^T, fp32
        am = o; o += (size_t)kL * kP * 4;           // A
        ts = o; o += (size_t)kL * kP * 4;           // T = (I + A)^-1 (blocks above the diagonal not written)
        xs = o; o += (size_t)32 * 32 * 4;           // block products of the inversion
        tcw = o; o += (size_t)kL * kL * 2;          // T diag(beta exp Lam), bf16 operand [64][64]
        tcu = o; o += (size_t)kL * kL * 2;          // T diag(beta), bf16 operand [64][64]
        ustg = al(ts, 1024);                        // U staging slots 0-3 (base 1024-aligned), up to the end of tcu
        ustg2 = al(am, 1024);                       // slots 4-5
        vc = o; o += (size_t)2 * kL * Dv * 2;       // V of the chunk, bf16 operand [64][Dv], two buffers (heads alternate)
        lam = o; o += 4 * kL * 4;                   // log g, Lam, exp Lam, beta
        bar = al(o, 8); o = bar + 3 * 8;            // MMA, copies of V, of K and Q
        tslot = o; o += 16;
        total = o + 1024;
        if (total < kOneCtaSmem) total = kOneCtaSmem;
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

__device__ __forceinline__ void unpack8_bf16(const uint4 &u, float (&x)[8]) {
    x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
    x[4] = __uint_as_float(u.z << 16); x[5] = __uint_as_float(u.z & 0xffff0000u);
    x[6] = __uint_as_float(u.w << 16); x[7] = __uint_as_float(u.w & 0xffff0000u);
}


// T = (I + A)^-1 for the strictly lower 64 x 64 A (row stride kP), in two levels of 2 x 2
// block recursion: the four diagonal 16 x 16 blocks by forward substitution (a column per
// thread); then the two 32 x 32 diagonal blocks, and then the 64 x 64, each by
//     T_21 = -T_22 (A_21 T_11)
// as two dependent products with four consecutive columns of one row per thread (a scalar
// and a float4 load per four multiply-adds). Blocks of T above the diagonal are not written,
// and the products skip them. Called by all 256 threads; xs holds 32 x 32 floats. Threads
// 64-255, idle during the diagonal blocks, run `other` meanwhile.
template <class Other>
__device__ void invert_unit_lower(const float *am, float *ts, float *xs, int tid, Other &&other) {
    if (tid >= kL) other();
    if (tid < kL) {
        const int b0 = 16 * (tid >> 4), c = tid & 15;
        float col[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float x = r == c ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < r; ++i) x = fmaf(-am[(b0 + r) * kP + b0 + i], col[i], x);
            col[r] = r < c ? 0.f : x;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) ts[(b0 + r) * kP + b0 + c] = col[r];
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

// Persistent: one CTA per SM over a contiguous range of units (batch row, chunk, kv head,
// value head), value head fastest. When a unit starts a new (batch row, chunk, kv head) group
// the CTA forms K K^T and Q K^T from K and Q (fetched by TMA while the previous group's last
// unit was read back); per unit (value head) it forms the decay-weighted matrices, T,
// W = (T diag(beta exp Lam)) K and U = (T diag(beta)) V (the row scalings folded into T's
// columns, K and V read as MN-major operands). The next unit's V, g and beta are fetched while
// the current one computes.
template <int E>
__global__ void __launch_bounds__(256, 1) chunk_prep_kernel(ChunkParams p, int units,
                                                            const __grid_constant__ ChunkFwdMaps maps) {
    constexpr int DK = 32 * E;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.T, Dv = p.Dv, Hv = p.Hv, Hk = p.Hk, NC = p.NC, rep = p.Hv / p.Hk;
    const int u_begin = (int)((long long)blockIdx.x * units / gridDim.x);
    const int u_end = (int)((long long)(blockIdx.x + 1) * units / gridDim.x);

    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(al(reinterpret_cast<size_t>(smem_raw), 1024));
    const PrepSmem L(DK, Dv);
    unsigned char *kc = base + L.kc, *qc = base + L.qc, *tcw = base + L.tcw, *tcu = base + L.tcu, *vc = base + L.vc;
    float *kk = reinterpret_cast<float *>(base + L.kk);
    float *qk = reinterpret_cast<float *>(base + L.qk);
    float *am = reinterpret_cast<float *>(base + L.am);
    float *ts = reinterpret_cast<float *>(base + L.ts);
    float *xs = reinterpret_cast<float *>(base + L.xs);
    float *lg = reinterpret_cast<float *>(base + L.lam);     // log g
    float *Lm = lg + kL;                                      // Lam (inclusive prefix)
    float *gm = Lm + kL;                                      // exp(Lam)
    float *bt = gm + kL;                                      // beta
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + L.bar), *cbV = bar + 1, *cbKQ = bar + 2;
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
        for (int j = 0; j < 3; ++j) mbar_init(bar + j, 1);
        fence_mbar_init();
        tma_prefetch_map(&maps.v);
        tma_prefetch_map(&maps.u);
    }
    if (tid == 32) {
        tma_prefetch_map(&maps.k);
        tma_prefetch_map(&maps.q);
        tma_prefetch_map(&maps.qk);
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    // V of a unit's chunk into buffer `buf` in its operand layout, as one TMA box of 1 KB
    // core-matrix columns (rows past T are zeros). Thread 0 issues it and waits for it.
    int nV = 0, wV = 0, nKQ = 0, wKQ = 0;
    auto fetch_v = [&](const Unit &x, int buf) {
        mbar_expect_tx(cbV, kL * Dv * 2);
        tma_load_5d(vc + (size_t)buf * kL * Dv * 2, &maps.v, cbV, 0, x.t0, 0, x.h, x.b);
        ++nV;
    };
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
    // K and Q of a (batch row, chunk, kv head) into kc and qc in their operand layout, a TMA
    // box each as for V, issued by thread 32 (called by all threads, which all wait for it)
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
    // A (batch row, chunk, kv head) group whose K and Q were fetched into kc and qc: K K^T and
    // Q K^T into kk and qk, and K and [Q; K] in the layouts of the sweeps and the gradient
    // kernel (bulk stores by thread 32, which waits for their reads before kc and qc are
    // refilled)
    auto stage_group = [&](const Unit &x) {
        {
            const bool w = mbar_wait(cbKQ, wKQ & 1);
            ++wKQ;
            tc_fence_before();
            ok = !__syncthreads_or(!w);
            tc_fence_after();
            if (!ok) return;
        }
        // K K^T -> columns [0, 64), Q K^T -> [64, 128) (M = 64: row m in lane m % 16 + 32 (m / 16))
        if (tid == 0) {
            constexpr uint32_t id = umma_idesc(1, kL, kL);
            umma_gemm_bf16(tmem, kc, kL, 0, kc, kL, 0, DK, id, false);
            umma_gemm_bf16(tmem + kL, qc, kL, 0, kc, kL, 0, DK, id, false);
            umma_commit(bar);
        }
        if (tid == 32) {
            // K in its operand layout (for both sweeps), and [Q; K] in the gradient kernel's
            // 128-row layout (K chunk j: the 64 rows of Q, then the 64 rows of K; a TMA store of
            // each half). A group split between two CTAs is written by both, alike.
            const size_t ckv = ((size_t)x.b * Hk + x.hk) * NC + x.c;
            bulk_store(p.ktm + ckv * kL * DK, kc, kL * DK * 2);
            tma_store_5d(&maps.qk, qc, 0, 0, 0, 0, (int)ckv);
            tma_store_5d(&maps.qk, kc, 0, 0, 0, 1, (int)ckv);
            bulk_commit();
        }
        ok = !__syncthreads_or(!mbar_wait(bar, phase & 1));
        ++phase;
        tc_fence_after();
        if (ok) {
            // warps 0-3 read K K^T, warps 4-7 Q K^T; each warp its quarter's 16 valid lanes
            const int quarter = warp & 3, row = 16 * quarter + lane;
            float *dst = warp < 4 ? kk : qk;
            const uint32_t col0 = warp < 4 ? 0u : (uint32_t)kL;
            float xv[64];
            tmem_ld32f(tmem + ((uint32_t)(32 * quarter) << 16) + col0, xv);
            tmem_ld32f(tmem + ((uint32_t)(32 * quarter) << 16) + col0 + 32, xv + 32);
            tmem_wait_ld();
            if (lane < 16)
#pragma unroll
                for (int i = 0; i < 64; i += 4)
                    *reinterpret_cast<float4 *>(dst + row * kP + i) = make_float4(xv[i], xv[i + 1], xv[i + 2], xv[i + 3]);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };
    // the first unit's g and beta go out before anything else, its V, K and Q once the
    // barriers are initialised
    if (u_begin < u_end && warp == 0) fetch_gb(unit_of(u_begin));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tmem = *tslot;
    if (u_begin < u_end) {
        const Unit x0 = unit_of(u_begin);
        if (tid == 0) fetch_v(x0, 0);
        fetch_kq(x0);
    }

    for (int u = u_begin, i = 0; u < u_end && ok; ++u, ++i) {
        const Unit x = unit_of(u);
        const int b = x.b, c = x.c, h = x.h, len = x.len;
        if (i == 0 || (u - 1) / rep != u / rep) {
            stage_group(x);
            if (!ok) break;
        }
        const size_t chk = ((size_t)b * Hv + h) * NC + c;   // (b, h, c)
        unsigned char *vch = vc + (size_t)(i & 1) * kL * Dv * 2;
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
        if (tid == 128 && Dv > 128) bulk_wait_read();   // the last unit's U boxes have left A
        __syncthreads();
        // A, and the decay-weighted Q K^T (i <= t) and K K^T (i < t) as bf16 operands stacked
        // in one 128-row core-matrix layout: columns 8 j .. + 7 of row t are 16-byte piece
        // 128 j + t (P) and 128 j + 64 + t (KKm)
        uint4 *PK = reinterpret_cast<uint4 *>(p.pkm + chk * 2 * kL * kL);
        for (int e = tid; e < kL * 8; e += 256) {
            const int t = e & (kL - 1), i0 = 8 * (e >> 6);
            float kk8[8], qk8[8], a8[8], pv[8], kv8[8];
            *reinterpret_cast<float4 *>(kk8) = *reinterpret_cast<const float4 *>(kk + t * kP + i0);
            *reinterpret_cast<float4 *>(kk8 + 4) = *reinterpret_cast<const float4 *>(kk + t * kP + i0 + 4);
            *reinterpret_cast<float4 *>(qk8) = *reinterpret_cast<const float4 *>(qk + t * kP + i0);
            *reinterpret_cast<float4 *>(qk8 + 4) = *reinterpret_cast<const float4 *>(qk + t * kP + i0 + 4);
            const float lt = Lm[t], bb = bt[t];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + j;
                const float ex = i <= t ? expf(lt - Lm[i]) : 0.f;
                a8[j] = i < t ? bb * kk8[j] * ex : 0.f;
                pv[j] = qk8[j] * ex;
                kv8[j] = i < t ? kk8[j] * ex : 0.f;
            }
            *reinterpret_cast<float4 *>(am + t * kP + i0) = *reinterpret_cast<const float4 *>(a8);
            *reinterpret_cast<float4 *>(am + t * kP + i0 + 4) = *reinterpret_cast<const float4 *>(a8 + 4);
            PK[(e >> 6) * 2 * kL + t] = pack8_bf16(pv);
            PK[(e >> 6) * 2 * kL + kL + t] = pack8_bf16(kv8);
        }
        if (tid == 128) bulk_wait_read();   // the last unit's U boxes have left T and the T operands
        __syncthreads();
        // T = (I + A)^-1; while threads 0-63 form its diagonal blocks, the others write
        // [diag(exp Lam) Q; diag(exp Lam) K] (row scaling of the staged operands), one 128-row
        // operand: piece e of Q (K chunk e / 64, row e % 64) goes to 128 (e / 64) + e % 64,
        // that of K 64 pieces later
        invert_unit_lower(am, ts, xs, tid, [&] {
            uint4 *QK = reinterpret_cast<uint4 *>(p.qksm + chk * 2 * kL * DK);
            for (int e = tid - kL; e < kL * DK / 8; e += 256 - kL) {
                const int o = (e >> 6) * 2 * kL + (e & (kL - 1));
                const float gr = gm[e & (kL - 1)];
                float a[8];
                unpack8_bf16(reinterpret_cast<const uint4 *>(qc)[e], a);
#pragma unroll
                for (int j = 0; j < 8; ++j) a[j] *= gr;
                QK[o] = pack8_bf16(a);
                unpack8_bf16(reinterpret_cast<const uint4 *>(kc)[e], a);
#pragma unroll
                for (int j = 0; j < 8; ++j) a[j] *= gr;
                QK[o + kL] = pack8_bf16(a);
            }
        });
        // T (for the backward), T diag(beta exp Lam) and T diag(beta) as bf16 operands; the
        // blocks of T above the diagonal are zero
        {
            unsigned char *Tg = reinterpret_cast<unsigned char *>(p.tm != nullptr ? p.tm + chk * kL * kL : nullptr);
            for (int e = tid; e < kL * 8; e += 256) {
                const int t = e & (kL - 1), ch = e >> 6;
                float x[8], w8[8], u8[8];
                if ((8 * ch) >> 4 <= t >> 4) {
                    const float4 a = *reinterpret_cast<const float4 *>(ts + t * kP + 8 * ch);
                    const float4 a2 = *reinterpret_cast<const float4 *>(ts + t * kP + 8 * ch + 4);
                    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = a2.x; x[5] = a2.y; x[6] = a2.z; x[7] = a2.w;
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] = 0.f;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int col = 8 * ch + i;
                    u8[i] = x[i] * bt[col];
                    w8[i] = u8[i] * gm[col];
                }
                const uint32_t o = cm_off(t, 16 * ch, kL);
                *reinterpret_cast<uint4 *>(tcw + o) = pack8_bf16(w8);
                *reinterpret_cast<uint4 *>(tcu + o) = pack8_bf16(u8);
                if (Tg != nullptr) *reinterpret_cast<uint4 *>(Tg + o) = pack8_bf16(x);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // W -> columns [256, 256 + DK), U -> [0, Dv) (once this unit's V has landed); then the
        // next unit's V goes out into the other buffer
        bool vok = true;
        if (tid == 0) {
            vok = mbar_wait(cbV, wV & 1);
            ++wV;
            if (vok) {
                umma_gemm(tmem + 256, CmOp{tcw, kL, 0, 0, false}, CmOp{kc, kL, 0, 0, true}, kL,
                          umma_idesc_t(1, kL, DK, false, true), false);
                umma_gemm(tmem, CmOp{tcu, kL, 0, 0, false}, CmOp{vch, kL, 0, 0, true}, kL,
                          umma_idesc_t(1, kL, Dv, false, true), false);
                umma_commit(bar);
                if (u + 1 < u_end) fetch_v(unit_of(u + 1), (i + 1) & 1);
            }
        }
        // when the next unit starts another group, its K and Q are fetched into kc and qc
        // (free once these products are done) while this unit's results are read back
        const bool kq_next = u + 1 < u_end && (u + 1) / rep != u / rep;
        if (tid == 32 && kq_next) bulk_wait_read();   // the stores of K and [Q; K] have read kc, qc
        ok = !__syncthreads_or(!vok || !mbar_wait(bar, phase & 1));
        ++phase;
        tc_fence_after();
        if (ok && kq_next) fetch_kq(unit_of(u + 1));
        if (ok) {
            const int quarter = warp & 3, row = 16 * quarter + lane;
            const uint32_t lo = (uint32_t)(32 * quarter) << 16;
            if (warp < 4) {
                // W in its operand layout, 96 columns per tensor-memory wait
                unsigned char *W = reinterpret_cast<unsigned char *>(p.wm + chk * kL * DK);
                for (int c0 = 0; c0 < DK; c0 += 96) {
                    const int n = DK - c0 < 96 ? DK - c0 : 96;
                    float x[96];
#pragma unroll
                    for (int j = 0; j < 3; ++j)
                        if (32 * j < n) tmem_ld32f(tmem + lo + 256 + c0 + 32 * j, x + 32 * j);
                    tmem_wait_ld();
                    if (lane < 16)
#pragma unroll
                        for (int j = 0; j < 12; ++j)
                            if (8 * j < n)
                                *reinterpret_cast<uint4 *>(W + cm_off(row, 2 * (c0 + 8 * j), kL)) =
                                    pack8_bf16(*reinterpret_cast<const float (*)[8]>(x + 8 * j));
                }
            } else {
                // U in blocks of 32 columns, [Dv / 32][64][32] (a row's 32 columns are 128
                // contiguous bytes): each block staged as a 128-byte-swizzled box (row r's
                // 16-byte piece j at r * 128 + ((j ^ (r & 7)) << 4)) and written by a TMA store
                // from thread 128; up to three boxes per pass, kUSlots slots in a ring
                const int nb = Dv / 32;
                auto slot = [&](int i) { return base + (i < 4 ? L.ustg + (size_t)i * 8192 : L.ustg2 + (size_t)(i - 4) * 8192); };
                for (int c0 = 0, pass = 0; c0 < Dv; c0 += 96, ++pass) {
                    const int n = Dv - c0 < 96 ? Dv - c0 : 96;
                    float x[96];
#pragma unroll
                    for (int j = 0; j < 3; ++j)
                        if (32 * j < n) tmem_ld32f(tmem + lo + c0 + 32 * j, x + 32 * j);
                    tmem_wait_ld();
                    if (3 * (pass + 1) > kUSlots) {
                        // the slots of two passes ago: their stores must have read them
                        if (tid == 128) bulk_wait_read_but<1>();
                        named_bar_sync(1, 128);
                    }
                    if (lane < 16)
#pragma unroll
                        for (int j = 0; j < 3; ++j)
                            if (32 * j < n) {
                                unsigned char *box = slot((c0 / 32 + j) % kUSlots) + row * 128;
#pragma unroll
                                for (int q4 = 0; q4 < 8; ++q4)
                                    *reinterpret_cast<float4 *>(box + ((q4 ^ (row & 7)) << 4)) =
                                        make_float4(x[32 * j + 4 * q4], x[32 * j + 4 * q4 + 1], x[32 * j + 4 * q4 + 2],
                                                    x[32 * j + 4 * q4 + 3]);
                            }
                    fence_proxy_async();
                    named_bar_sync(1, 128);
                    if (tid == 128) {
                        for (int j = 0; j < 3 && 32 * j < n; ++j) {
                            const int blk = c0 / 32 + j;
                            tma_store_2d(&maps.u, slot(blk % kUSlots), 0, (int)((chk * nb + blk) * kL));
                        }
                        bulk_commit();
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (!ok && tid == 0) {
        report_status(p.status, kStatusTimeout);
        // copies still in flight land before the CTA exits (each wait bounded)
        if (nV > wV) mbar_wait(cbV, (nV - 1) & 1);
        if (nKQ > wKQ) mbar_wait(cbKQ, (nKQ - 1) & 1);
    }
    if (tid == 32 || tid == 128) bulk_wait_all();   // no store still reads shared memory when the CTA exits
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace gdn

namespace gdn {

namespace {

struct SweepSmem {
    size_t wc, qks, kt, pkc, sop, dt, de, ckst, ysg, rsg, vec, bar, tslot, total;
    __host__ __device__ SweepSmem(int DK) {
        size_t o = 0;
        wc = o; o += (size_t)kL * DK * 2;     // W of the chunk        A [64][DK]
        qks = o; o += (size_t)2 * kL * DK * 2;   // [diag(exp Lam) Q; diag(exp Lam) K]   A [128][DK]
        kt = o; o += (size_t)kL * DK * 2;     // K (read MN-major)     B [64][DK]
        pkc = o; o += (size_t)2 * kL * kL * 2;   // [(Q K^T) o E_incl; (K K^T) o E_strict]   A [128][64]
        sop = o; o += (size_t)kL * DK * 2;    // S (64 value rows)     B [64][DK]
        dt = o; o += (size_t)kL * kL * 2;     // Delta [64 t][64 v], read MN-major (B)
        de = o; o += (size_t)kL * kL * 2;     // diag(E_L) Delta [64 t][64 v], read MN-major (A, transposed)
        ckst = al(o, 1024); o = ckst + (size_t)kL * DK * 4;   // chunk-start state, fp32, boxes of [64][32] in the 128-byte swizzle
        ysg = al(o, 1024); o = ysg + (size_t)kL * 128;       // y of a chunk, bf16 [64][64] in the 128-byte swizzle
        rsg = al(o, 1024); o = rsg + (size_t)2 * kL * 128;   // v - u of a chunk, fp32 [2][64][32] in the 128-byte swizzle
        vec = o; o += 3 * kL * 4;             // Lam, exp Lam, E(L, .)
        bar = al(o, 8); o = bar + 24;         // MMA completion, the two groups of operand copies
        tslot = o; o += 16;
        total = o + 1024;
        if (total < kOneCtaSmem) total = kOneCtaSmem;
    }
};

}  // namespace

// One CTA per (64-row block of the state, value head, batch row), carrying that block of the
// state through the chunks. Tensor memory (fp32 accumulators):
//   [0, DK)             the state S (M = 64: value row r in lane r % 16 + 32 (r / 16)); per
//                       chunk it is scaled by exp(Lam_L) in place and the update
//                       (diag(E_L) Delta)^T K is accumulated onto it by MMA
//   [DK, DK + 64)       [y; u] of the chunk, one M = 128 product of the stacked operands: chunk
//                       row t of y in lane t, of the prediction u in lane 64 + t
//   [DK + 64, DK + 128) W S^T (M = 64)
template <int E>
__global__ void __launch_bounds__(256, 1) chunk_sweep_kernel(ChunkParams p, const __grid_constant__ CUtensorMap tm_ck,
                                                             const __grid_constant__ CUtensorMap tm_y,
                                                             const __grid_constant__ CUtensorMap tm_r) {
    constexpr int DK = 32 * E;
    static_assert(DK + 128 <= 512, "tensor memory holds the state, [y; u] and W S^T");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int T = p.T, Dv = p.Dv, Hv = p.Hv, r0 = split * kL;
    const int quarter = warp & 3, half = warp >> 2;
    const int lrow = 16 * quarter + lane;                   // M = 64 row of this lane (lanes 0-15)
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(al(reinterpret_cast<size_t>(smem_raw), 1024));
    const SweepSmem L(DK);
    unsigned char *wc = base + L.wc, *qks = base + L.qks, *kt = base + L.kt, *pkc = base + L.pkc;
    unsigned char *sop = base + L.sop, *dt = base + L.dt, *de = base + L.de;
    unsigned char *ckst = base + L.ckst, *ysg = base + L.ysg;
    unsigned char *rsg = base + L.rsg;
    float *Lm = reinterpret_cast<float *>(base + L.vec), *gm = Lm + kL, *eL = gm + kL;
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + L.bar), *cbar = bar + 1, *rbar = bar + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + L.tslot);

    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
    const size_t head = (size_t)b * Hv + h;
    // the operand matrices of chunk cc (W, [Qs; Ks], K, [P; KKm]), prepared in their
    // shared-memory layout, by bulk copies in two groups (thread 0): W, read by the first
    // product of a chunk, goes out as soon as that product is done; the rest, read by the
    // second group, after that group
    constexpr unsigned kBig = kL * DK * 2, kSmall = kL * kL * 2;
    int ncw = 0, ncr = 0;
    auto issue_w = [&](int cc) {
        mbar_expect_tx(cbar, kBig);
        bulk_load(wc, p.wm + (head * p.NC + cc) * kL * DK, kBig, cbar);
        ++ncw;
    };
    auto issue_r = [&](int cc) {
        const size_t ck = head * p.NC + cc;
        mbar_expect_tx(rbar, 3 * kBig + 2 * kSmall);
        bulk_load(qks, p.qksm + ck * 2 * kL * DK, 2 * kBig, rbar);
        bulk_load(kt, p.ktm + (((size_t)b * p.Hk + h / (Hv / p.Hk)) * p.NC + cc) * kL * DK, kBig, rbar);
        bulk_load(pkc, p.pkm + ck * 2 * kL * kL, 2 * kSmall, rbar);
        ++ncr;
    };

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(cbar, 1);
        mbar_init(rbar, 1);
        fence_mbar_init();
        tma_prefetch_map(&tm_ck);
        tma_prefetch_map(&tm_y);
        tma_prefetch_map(&tm_r);
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tS = tmem, tYU = tmem + DK, tD = tmem + DK + 64;
    constexpr int SC = DK / 2;                              // state columns per warp half

    // the start state into tensor memory
    {
        float x[16];
        for (int cc = half * SC; cc < half * SC + SC; cc += 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                x[i] = (p.S0 != nullptr && lane < 16 && r0 + lrow < Dv)
                           ? p.S0[(head * Dv + r0 + lrow) * DK + cc + i] : 0.f;
            tmem_st16f(tS + lane_off + cc, x);
        }
        tmem_wait_st();
    }
    unsigned phase = 0, cph = 0;
    bool ok = true;
    float4 ux[8];        // U of the current chunk: this lane's row, this warp's 32 columns
    uint4 vx[4];         // v of the chunk whose epilogue is pending
    float lamn = 0.f;    // Lam of the next chunk (threads < 64)
    auto load_u = [&](int cc) {
        const float *Ug = p.um + (head * p.NC + cc) * kL * Dv + ((size_t)((r0 + half * 32) >> 5) * kL + lrow) * 32;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            ux[i] = lane < 16 ? reinterpret_cast<const float4 *>(Ug)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    // v for the threads that form v - u (warps of row quarters 2 and 3: chunk row
    // 32 (quarter - 2) + lane, this half's 32 value columns)
    auto load_v = [&](int cc) {
        const int tt0 = cc * kL, ln = min(kL, T - tt0), t = 32 * (quarter & 1) + lane;
        const size_t o = (((size_t)b * T + tt0 + t) * Hv + h) * Dv + r0 + half * 32;
        const bool mine = quarter >= 2 && t < ln;
#pragma unroll
        for (int i = 0; i < 4; ++i) vx[i] = mine ? reinterpret_cast<const uint4 *>(v + o)[i] : make_uint4(0u, 0u, 0u, 0u);
    };
    // y and v - u of chunk cc, from tensor memory (its columns are rewritten only by the next
    // chunk's second group of products), staged in the 128-byte swizzle for TMA stores: y (row
    // quarters 0-1 of [y; u]) and v - u (quarters 2-3), each in its own tile (thread 0 waits
    // for the stores' reads before the next chunk's first product). Rows past T are clipped by
    // the stores.
    auto epilogue = [&](int cc) {
        float x[32];
        tmem_ld32f(tYU + lane_off + half * 32, x);
        tmem_wait_ld();
        const int t = 32 * (quarter & 1) + lane, sw = t & 7;
        if (quarter < 2) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4 *>(ysg + t * 128 + (((half * 4 + j) ^ sw) << 4)) =
                    pack8_bf16(*reinterpret_cast<const float (*)[8]>(x + 8 * j));
        } else {
            float va[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) unpack8_bf16(vx[j], *reinterpret_cast<float (*)[8]>(va + 8 * j));
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4 *>(rsg + half * (kL * 128) + t * 128 + ((j ^ sw) << 4)) =
                    make_float4(va[4 * j] - x[4 * j], va[4 * j + 1] - x[4 * j + 1], va[4 * j + 2] - x[4 * j + 2],
                                va[4 * j + 3] - x[4 * j + 3]);
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
            const int tt0 = cc * kL;
            tma_store_4d(&tm_y, ysg, r0, h, tt0, b);
            if (p.resid != nullptr) {
                tma_store_5d(&tm_r, rsg, 0, tt0, r0 / 32, h, b);
            }
            bulk_commit();
        }
    };
    if (tid == 0) { issue_w(0); issue_r(0); }
    if (tid < kL) lamn = p.lam[head * p.NC * kL + tid];
    load_u(0);
    for (int c = 0; c < p.NC && ok; ++c) {
        const size_t chk = head * p.NC + c;
        // ---- decays of the chunk (Lam loaded one chunk ahead)
        if (tid < kL) {
            Lm[tid] = lamn;
            gm[tid] = expf(lamn);
            if (c + 1 < p.NC) lamn = p.lam[(chk + 1) * kL + tid];
        }
        // the previous chunk's state stores have read sop and ckst (from the third chunk on, the
        // y and v - u stores committed after them may still be reading ysg and rsg)
        if (tid == 0) {
            if (c >= 2) bulk_wait_read_but<1>();
            else bulk_wait_read();
        }
        __syncthreads();
        if (tid < kL) eL[tid] = expf(Lm[kL - 1] - Lm[tid]);
        // ---- the state as an operand, and the chunk-start checkpoint staged for TMA stores (all
        // of this thread's columns loaded from tensor memory before one wait). The stores of the
        // previous chunk have read both buffers (thread 0 waited before the barrier above).
        {
            float xs[SC];
#pragma unroll
            for (int j = 0; j < SC / 32; ++j) tmem_ld32f(tS + lane_off + half * SC + 32 * j, xs + 32 * j);
            tmem_wait_ld();
            if (lane < 16) {
#pragma unroll
                for (int j = 0; j < SC / 8; ++j) {
                    const uint32_t o = cm_off(lrow, 2 * (half * SC + 8 * j), kL);
                    *reinterpret_cast<uint4 *>(sop + o) = pack8_bf16(*reinterpret_cast<const float (*)[8]>(xs + 8 * j));
                }
                // box bx holds columns 32 bx .. + 31: row r at r * 128 bytes, its 16-byte chunk q
                // at chunk q ^ (r % 8) (the 128-byte swizzle)
#pragma unroll
                for (int j = 0; j < SC / 4; ++j) {
                    const int col = half * SC + 4 * j, bx = col >> 5, q = (col & 31) >> 2;
                    *reinterpret_cast<float4 *>(ckst + bx * (kL * 128) + lrow * 128 + ((q ^ (lrow & 7)) << 4)) =
                        make_float4(xs[4 * j], xs[4 * j + 1], xs[4 * j + 2], xs[4 * j + 3]);
                }
            }
            // S <- exp(Lam_L) S in place: the chunk's update (diag(E_L) Delta)^T K is accumulated
            // onto it by the second group of products
            const float decay = gm[kL - 1];
#pragma unroll
            for (int i = 0; i < SC; ++i) xs[i] *= decay;
#pragma unroll
            for (int j = 0; j < SC / 32; ++j) tmem_st32f(tS + lane_off + half * SC + 32 * j, xs + 32 * j);
            tmem_wait_st();
        }
        fence_proxy_async();
        tc_fence_before();
        if (tid == 0) bulk_wait_read();                     // the y and v - u stores have read ysg and rsg
        // W of the chunk (copied half a chunk ahead; only the MMAs read it)
        ok = !__syncthreads_or(tid == 0 && !mbar_wait(cbar, cph & 1));
        tc_fence_after();
        if (!ok) break;
        if (tid == 0) {
            // the bf16 state (the backward's operand) and the fp32 checkpoint leave by bulk stores
            if (p.s0m != nullptr) bulk_store(p.s0m + (chk * gridDim.x + split) * kL * DK, sop, kL * DK * 2);
            if (p.ckpt != nullptr) tma_store_5d(&tm_ck, ckst, 0, (int)(chk * Dv + r0), 0, 0, 0);
            bulk_commit();
        }
        // ---- W S^T
        if (tid == 0) {
            umma_gemm_bf16(tD, wc, kL, 0, sop, kL, 0, DK, umma_idesc(1, kL, kL), false);
            umma_commit(bar);
        }
        // the previous chunk's y and v - u while the product runs
        if (c > 0) epilogue(c - 1);
        tc_fence_before();
        ok = !__syncthreads_or(!mbar_wait(bar, phase & 1));
        ++phase;
        tc_fence_after();
        if (!ok) break;
        if (tid == 0 && c + 1 < p.NC) issue_w(c + 1);      // W's buffer is free again
        {
            // Delta = U - W S^T, straight into the operands Delta and diag(E_L) Delta, stored as
            // [t][v] (row t of the lane, 8 value columns per 16-byte piece) and read MN-major:
            // Delta as the B of [P; KKm] Delta, diag(E_L) Delta as the (transposed) A of the update
            float x[32];
            tmem_ld32f(tD + lane_off + half * 32, x);
            tmem_wait_ld();
            if (lane < 16) {
                const float *uf = reinterpret_cast<const float *>(ux);
                const float el = eL[lrow];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float a[8], bb[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        a[i] = uf[8 * j + i] - x[8 * j + i];
                        bb[i] = el * a[i];
                    }
                    const uint32_t o = cm_off(lrow, 2 * (half * 32 + 8 * j), kL);
                    *reinterpret_cast<uint4 *>(dt + o) = pack8_bf16(a);
                    *reinterpret_cast<uint4 *>(de + o) = pack8_bf16(bb);
                }
            }
        }
        if (c + 1 < p.NC) load_u(c + 1);                   // the next chunk's U, used one chunk later
        fence_proxy_async();
        // the rest of the chunk's operands (copied a chunk ahead)
        ok = !__syncthreads_or(tid == 0 && !mbar_wait(rbar, cph & 1));
        ++cph;
        tc_fence_after();
        if (!ok) break;
        // ---- [y; u] = [Qs; Ks] S^T + [P; KKm] Delta (M = 128);  update = (E_L Delta)^T K
        if (tid == 0) {
            constexpr uint32_t id128 = umma_idesc(1, 2 * kL, kL);
            umma_gemm(tYU, CmOp{qks, 2 * kL, 0, 0, false}, CmOp{sop, kL, 0, 0, false}, DK, id128, false);
            umma_gemm(tYU, CmOp{pkc, 2 * kL, 0, 0, false}, CmOp{dt, kL, 0, 0, true}, kL,
                      umma_idesc_t(1, 2 * kL, kL, false, true), true);
            umma_gemm(tS, CmOp{de, kL, 0, 0, true}, CmOp{kt, kL, 0, 0, true}, kL, umma_idesc_t(1, kL, DK, true, true), true);
            umma_commit(bar);
        }
        load_v(c);                                          // for this chunk's epilogue, one chunk later
        ok = !__syncthreads_or(!mbar_wait(bar, phase & 1));
        ++phase;
        tc_fence_after();
        if (!ok) break;
        // the other operand buffers are free again: bring in the next chunk's (no block barrier
        // before the next chunk: nothing after this point reads what its first section writes)
        if (tid == 0 && c + 1 < p.NC) issue_r(c + 1);
    }
    if (ok) {
        // the previous chunk's y and v - u stores were committed after this chunk's wait: they
        // must have read ysg and rsg before the last epilogue rewrites them
        if (tid == 0) bulk_wait_read();
        __syncthreads();
        epilogue(p.NC - 1);
    }
    if (tid == 0) bulk_wait_all();                          // the state stores are complete
    if (ok && p.S_T != nullptr) {
        for (int cc = half * SC; cc < half * SC + SC; cc += 16) {
            float x[16];
            tmem_ld16f(tS + lane_off + cc, x);
            tmem_wait_ld();
            if (lane < 16 && r0 + lrow < Dv)
#pragma unroll
                for (int i = 0; i < 16; i += 4)
                    *reinterpret_cast<float4 *>(p.S_T + (head * Dv + r0 + lrow) * DK + cc + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
        }
    }
    if (!ok && tid == 0) {
        report_status(p.status, kStatusTimeout);
        // copies still in flight land before the CTA exits (each wait bounded)
        if (ncw > 0) mbar_wait(cbar, (ncw - 1) & 1);
        if (ncr > 0) mbar_wait(rbar, (ncr - 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

size_t chunk_prep_smem(int Dk, int Dv) {
    const PrepSmem L(Dk, Dv);
    // the U staging slots must lie inside the regions they reuse
    const bool fits = L.ustg + (size_t)4 * 8192 <= L.tcu + (size_t)kL * kL * 2 &&
                      L.ustg2 + (size_t)(kUSlots - 4) * 8192 <= L.ts;
    return fits ? L.total : ~(size_t)0;
}
size_t chunk_sweep_smem(int Dk) { return SweepSmem(Dk).total; }

template <int E>
static cudaError_t launch_chunk_t(const ChunkParams &p, const ChunkFwdMaps &maps, cudaStream_t s) {
    constexpr int DK = 32 * E;
    const size_t sp = PrepSmem(DK, p.Dv).total, ss = SweepSmem(DK).total;
    cudaError_t err = cudaFuncSetAttribute(chunk_prep_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(chunk_sweep_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss);
    if (err != cudaSuccess) return err;
    timing_mark("chunk_prep", 0, s);
    const int units = p.NC * p.Hv * p.B;
    int dev = 0, sms = 0;
    err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    chunk_prep_kernel<E><<<units < sms ? units : sms, 256, sp, s>>>(p, units, maps);   // persistent: one CTA per SM
    timing_mark("chunk_prep", 1, s);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    timing_mark("chunk_sweep", 0, s);
    chunk_sweep_kernel<E><<<dim3(p.Dv / kL, p.Hv, p.B), 256, ss, s>>>(p, maps.ck, maps.y, maps.r);
    timing_mark("chunk_sweep", 1, s);
    return cudaGetLastError();
}

cudaError_t launch_chunk_fwd(const ChunkParams &p, const ChunkFwdMaps &maps, int Dk, cudaStream_t s) {
    switch (Dk) {
        case 64: return launch_chunk_t<2>(p, maps, s);
        case 128: return launch_chunk_t<4>(p, maps, s);
        case 192: return launch_chunk_t<6>(p, maps, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
