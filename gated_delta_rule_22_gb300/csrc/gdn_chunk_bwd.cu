// gdn_chunk_bwd.cu -- the backward (VJP) of the gated delta rule in its chunkwise form on the
// 5th-generation tensor cores, for bf16 inputs and chunks of 64 steps. It consumes the
// saved buffer of the chunkwise forward (gdn_chunk.cu).
//
// The recurrence is that of mlx issue #4614 ("Recurrence used for the references"); the
// chunkwise VJP is derived from it (the pages give neither form). Per value head and chunk of
// L = 64 steps, with the forward's quantities (Lam, E, T, P = (Q K^T) o E_incl, the chunk-start
// state S0, Delta = diag(beta) (v - u)) and the adjoint dS_L of the chunk-end state:
//     dD  = T^T (diag(E(L, .)) K dS_L^T + P^T dY)          (row t: ddelta_t = Sc_t k_t)
//     dv  = diag(beta) dD,  dU = -diag(beta) dD,  dbeta_t = ddelta_t . (v_t - u_t)
//     dS0 = exp(Lam_L) dS_L + dY^T diag(exp Lam) Q + dU^T diag(exp Lam) K
//     G = dY Delta^T,  H = dU Delta^T
//     dQ = diag(exp Lam) dY S0 + (G o E_incl) K
//     dK = diag(E(L, .)) Delta dS_L + (G o E_incl)^T Q + (H o E_strict)^T K
//          + diag(exp Lam) dU S0 + (H o E_strict) K
//     dg_t = <dA_t, S_{t-1}>, expanded over the chunk without any division by a decay:
//          E(L,t) e^{Lam_{t-1}} c0 + E(L,t) sum_{i<t} E(t-1,i) f_i
//          + sum_{s>=t} e^{Lam_{t-1}} E(s,t) (a_s + b_s) + sum_{s>=t} E(s,t) Z[s,t]
//       with c0 = <dS_L, S0>, f_i = delta_i . (dS_L k_i), a_s = dy_s . S0 q_s,
//       b_s = du_s . S0 k_s, Z = (G o (Q K^T) + H o (K K^T)) M, M[i,t] = E(t-1,i) [i < t].
//
// Two kernels:
//   chunk_dsweep_kernel  the reverse sweep over the chunks of one (b, h, block of 64 value
//                        rows), carrying dS (fp32, registers): dD, dv, dbeta and f (partials
//                        over 32 value rows), dU and dS_L for the next kernel, dS0.
//                        K dS_L^T takes dS as a bf16 high part plus a bf16 low part (exact to
//                        about 2^-16): with dS rounded once to bf16, dg under strong decay
//                        misses the bf16 parity bound.
//   chunk_grad_kernel    per (b, h, chunk), persistent over whole groups of units (the value
//                        heads of one kv head and chunk): everything else. dq, dk summed over
//                        the value heads of each kv head (ascending) in tensor memory, written
//                        as bf16 once per group; dbeta and f summed over their partials
//                        (ascending); dg.
// Operands are bf16 in the core-matrix layout of gdn_umma.cuh, read K-major or MN-major (one
// stored copy serves a matrix and its transpose); accumulators fp32 in tensor memory. No
// atomics, and every sum has a fixed order that depends on nothing but the problem: a group of
// value heads never straddles two gradient CTAs, so the grid (the SM count) and the batch size
// leave every result bit unchanged (a batch row's results are those of that row alone).
#include "gdn_umma.cuh"

namespace gdn {

namespace {

constexpr int kL = 64;           // chunk length
// Polls of one ready counter before the gradient kernel gives up (each a round trip to L2 and
// a short sleep: about a second in all, far above a chunk of the reverse sweep).
constexpr unsigned kReadyWaitLimit = 1u << 21;

__host__ __device__ inline size_t alb(size_t x, size_t a) { return (x + a - 1) / a * a; }

__device__ __forceinline__ uint4 pack8(const float *x) {
    uint4 u;
    __nv_bfloat162 h;
    h = __floats2bfloat162_rn(x[0], x[1]); u.x = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2bfloat162_rn(x[2], x[3]); u.y = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2bfloat162_rn(x[4], x[5]); u.z = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2bfloat162_rn(x[6], x[7]); u.w = *reinterpret_cast<uint32_t *>(&h);
    return u;
}

__device__ __forceinline__ void unpack8(const uint4 &u, float *x) {
    x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
    x[4] = __uint_as_float(u.z << 16); x[5] = __uint_as_float(u.z & 0xffff0000u);
    x[6] = __uint_as_float(u.w << 16); x[7] = __uint_as_float(u.w & 0xffff0000u);
}

// A kernel holding all 512 tensor-memory columns must be alone on its SM: it asks for more
// than half of the shared memory.
constexpr size_t kOneCtaSmem = 120 * 1024;

// ------------------------------------------------------------------ reverse sweep (dS)
constexpr int kSweepMathWarps = 8;      // hold dS (M = 64 fragment: 4 lane quarters x 2 column halves)
constexpr int kSweepThreads = 384;      // + a warpgroup: warp 8 issues the products, warp 9 the copies and stores
// registers: launched at 168 a thread; the control warpgroup gives up all but kSweepCtrlRegs,
// the math warpgroups take kSweepMathRegs (2 x 128 x 176 + 128 x 152 = 384 x 168)
constexpr int kSweepLaunchRegs = 168, kSweepMathRegs = 176, kSweepCtrlRegs = 152;
static_assert(2 * 128 * kSweepMathRegs + 128 * kSweepCtrlRegs <= kSweepThreads * kSweepLaunchRegs, "register split");

struct DSweepSmem {
    size_t qb, kb, tm, pb, ydu, yds, lms, shl, rhs, dls, dvs, bar, tslot, total;
    __host__ __device__ DSweepSmem(int DK) {
        size_t o = 0;
        qb = o; o += (size_t)kL * DK * 2;        // Q of the chunk (kv head) [64][DK] (read MN-major by the carry)
        kb = o; o += (size_t)2 * kL * DK * 2;    // K, two buffers [64][DK] (K-major for K dS^T, MN-major for the carry)
        tm = o; o += (size_t)kL * kL * 2;        // T [64][64] (read MN-major as T^T)
        pb = o; o += (size_t)2 * kL * kL * 2;    // P = (Q K^T) o E_incl, two buffers [64][64] (read MN-major)
        ydu = o; o += (size_t)2 * 2 * kL * kL * 2;   // [dY; dU] block [128][64 v] (rows 0-63 dY, 64-127 dU), two buffers
        yds = o; o += (size_t)2 * kL * kL * 2;       // [diag(exp Lam) dY; diag(exp Lam) dU] [128][64 v] (read MN-major)
        lms = o; o += (size_t)2 * kL * 4;        // Lam, two buffers
        shl = o; o += (size_t)2 * kL * DK * 2;   // dS as bf16 parts: high [64][DK], then low (dS - high) [64][DK]
        rhs = o; o += (size_t)kL * kL * 2;       // diag(E_L) K dS^T + P^T dY [64 t][64 v]
        dls = o; o += (size_t)kL * kL * 2;       // Delta block [64 t][64 v], for the gradient kernel
        dvs = alb(o, 1024); o = dvs + (size_t)kL * 128;   // dv block, bf16 [64][64] in the 128-byte swizzle
        bar = alb(o, 8); o = bar + 18 * 8;       // see the kernel
        tslot = o; o += 16;
        total = o + 1024;
        if (total < kOneCtaSmem) total = kOneCtaSmem;
    }
};

}  // namespace

// One CTA per (block of 64 value rows, value head, batch row), over the chunks in reverse.
// Warps 0-7 hold the adjoint dS (fp32, registers: the 16x256b fragment of an M = 64
// accumulator, 2 rows x DK/8 columns per thread) and do the element-wise work; warp 8 issues
// the products (one elected lane) and warp 9 the copies and stores, so that no math warp stalls
// on an issue and no block barrier runs per chunk: every hand-off is an mbarrier. Per chunk the
// products are (fp32 accumulators in tensor memory, M = 64 layout: row r in lane
// r % 16 + 32 (r / 16)):
//   [0, DK)              the chunk's part of the carry, (e^Lam dY)^T Q + (e^Lam dU)^T K; the
//                        next chunk's dS = exp(Lam_L) dS + this
//   [DK, DK + 64)        K dS_high^T + K dS_low^T (chunk row t, value column; the two parts
//                        accumulate in fp32); then dD
//   [DK + 128, DK + 192) P^T dY
// Hand-offs of chunk c (each completes once per chunk):
//   math -> control (8 warp arrivals): bHi the dS high part written;  bH  both dS parts written;
//                                      bR  rhs and Delta written;
//                                      bU  dU, [e^Lam dY; e^Lam dU] and dv written
//   control -> math: m1, mD, mS  the product groups (commits);  fS  the dS parts' tile is free
//                    (products done, the dS_L store has read it);  fO  the Delta and dv staging
//                    tiles are free (their stores have read them)
// Q and K arrive as separate [64][DK] tiles (boxes of the [Q; K] block), K double-buffered and
// fetched two chunks ahead. v - u is read by the math threads straight into registers, a chunk
// ahead. dbeta and f leave as one partial per 32 value columns (the two column halves).
template <int E>
__global__ void __launch_bounds__(kSweepThreads, 1) chunk_dsweep_kernel(ChunkBwdParams p,
                                                                        const __grid_constant__ CUtensorMap tm_dv,
                                                                        const __grid_constant__ CUtensorMap tm_dy,
                                                                        const __grid_constant__ CUtensorMap tm_qk,
                                                                        const __grid_constant__ CUtensorMap tm_pk) {
    constexpr int DK = 32 * E;
    constexpr int SC = DK / 2;                // dS columns per warp half
    constexpr int NS = SC / 2;                // dS values per thread
    static_assert(DK + 192 <= 512, "tensor memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool math = warp < kSweepMathWarps;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int T = p.T, Dv = p.Dv, Hv = p.Hv, NC = p.NC, r0 = split * kL, nsplit = p.nsplit;
    const int hw = (warp >> 2) & 1;                             // warp half: value columns [32 hw, 32 hw + 32)
    const uint32_t lane16 = (uint32_t)(32 * (warp & 3)) << 16;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(alb(reinterpret_cast<size_t>(smem_raw), 1024));
    const DSweepSmem L(DK);
    unsigned char *qb = base + L.qb, *kb2 = base + L.kb, *tmm = base + L.tm, *pb2 = base + L.pb, *yds = base + L.yds;
    unsigned char *ydu2 = base + L.ydu, *shl = base + L.shl, *rhs = base + L.rhs, *dls = base + L.dls;
    unsigned char *dvs = base + L.dvs;
    float *lms = reinterpret_cast<float *>(base + L.lms);
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + L.bar);
    uint64_t *m1 = bar, *mD = bar + 1, *mS = bar + 2, *cbT = bar + 3, *cbQ = bar + 4;
    uint64_t *cbP = bar + 5, *cbK = bar + 7, *cbY = bar + 9;   // [2] each: one per buffer
    uint64_t *bH = bar + 11, *bR = bar + 12, *bU = bar + 13, *fS = bar + 14, *fO = bar + 15, *mX = bar + 16;
    uint64_t *bHi = bar + 17;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + L.tslot);
    // the buffers of the chunk handled k-th (chunk NC - 1 - k): K, P, [dY; dU], Lam
    auto kbuf = [&](int k) { return kb2 + (size_t)(k & 1) * kL * DK * 2; };
    auto pbuf = [&](int k) { return pb2 + (size_t)(k & 1) * kL * kL * 2; };
    auto ybuf = [&](int k) { return ydu2 + (size_t)(k & 1) * 2 * kL * kL * 2; };

    const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(p.beta);
    const size_t head = (size_t)b * Hv + h;
    const int qkblk0 = (b * p.Hk + h / (Hv / p.Hk)) * NC;     // [Q; K] block of chunk 0 of this kv head

    if (tid == 0) {
        for (int i = 0; i < 11; ++i) mbar_init(bar + i, 1);
        for (int i = 11; i < 14; ++i) mbar_init(bar + i, kSweepMathWarps);
        for (int i = 14; i < 17; ++i) mbar_init(bar + i, 1);
        mbar_init(bHi, kSweepMathWarps);
        fence_mbar_init();
    }
    if (warp == kSweepMathWarps + 1 && lane == 0) {
        tma_prefetch_map(&tm_dy);
        tma_prefetch_map(&tm_qk);
        tma_prefetch_map(&tm_pk);
        tma_prefetch_map(&tm_dv);
    }
    if (warp == kSweepMathWarps) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tS = tmem, tX = tmem + DK, tP = tmem + DK + 128;
    griddep_wait();                                           // the previous kernel's writes are visible
    griddep_launch();

    bool fail = false;
    if (!math) {
        regs_dec<kSweepCtrlRegs>();            // the whole control warpgroup, at one point of the code
        if (warp == kSweepMathWarps) {
            // ================================================================ product warp
            const uint32_t lead = elect_one_sync();
            constexpr uint32_t idX = umma_idesc(1, kL, kL);
            constexpr uint32_t idP = umma_idesc_t(1, kL, kL, true, true);
            constexpr uint32_t idS = umma_idesc_t(1, kL, DK, true, true);
            // P^T dY needs no dS: each chunk's is issued a chunk ahead (the first one here), so that
            // only K dS^T is on the path from dS to the next chunk
            {
                const bool w = mbar_wait(cbP, 0) && mbar_wait(cbY, 0);
                fail = __any_sync(kFullMask, !w);
                if (!fail) {
                    tc_fence_after();
                    umma_gemm_w(tP, CmOp{pbuf(0), kL, 0, 0, true}, CmOp{ybuf(0), 2 * kL, 0, 0, true}, kL, idP, false, lead);
                }
            }
            for (int k = 0; k < NC && !fail; ++k) {
                unsigned char *kb = kbuf(k);
                // ---- K dS_high^T once the high part is written and K landed, then + K dS_low^T
                // once the low part is (it is formed while the first product runs)
                bool w = mbar_wait(bHi, k & 1) && mbar_wait(cbK + (k & 1), (k >> 1) & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                tc_fence_after();
                umma_gemm_w(tX, CmOp{kb, kL, 0, 0, false}, CmOp{shl, kL, 0, 0, false}, DK, idX, false, lead);
                w = mbar_wait(bH, k & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                tc_fence_after();
                umma_gemm_w(tX, CmOp{kb, kL, 0, 0, false}, CmOp{shl + kL * DK * 2, kL, 0, 0, false}, DK, idX, true, lead);
                umma_commit_w(m1, lead);
                // ---- dD = T^T rhs once rhs is written
                w = mbar_wait(bR, k & 1) && mbar_wait(cbT, k & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                tc_fence_after();
                umma_gemm_w(tX, CmOp{tmm, kL, 0, 0, true}, CmOp{rhs, kL, 0, 0, true}, kL, umma_idesc_t(1, kL, kL, true, true),
                            false, lead);
                umma_commit_w(mD, lead);
                // ---- the carry: its dY part (e^Lam dY)^T Q now (its operand rows were written before
                // bR; the math warps read the later chunk's carry before bH), its dU part
                // (e^Lam dU)^T K once dU is written
                w = mbar_wait(cbQ, k & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                umma_gemm_w(tS, CmOp{yds, 2 * kL, 0, 0, true}, CmOp{qb, kL, 0, 0, true}, kL, idS, false, lead);
                w = mbar_wait(bU, k & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                tc_fence_after();
                umma_gemm_w(tS, CmOp{yds, 2 * kL, 0, kL, true}, CmOp{kb, kL, 0, 0, true}, kL, idS, true, lead);
                umma_commit_w(mS, lead);
                // ---- P^T dY of the next chunk: its P and dY landed (copied two chunks ahead), and the
                // math warps read this chunk's (before bR)
                if (k + 1 < NC) {
                    const int k1 = k + 1;
                    w = mbar_wait(cbP + (k1 & 1), (k1 >> 1) & 1) && mbar_wait(cbY + (k1 & 1), (k1 >> 1) & 1);
                    if (__any_sync(kFullMask, !w)) { fail = true; break; }
                    tc_fence_after();
                    umma_gemm_w(tP, CmOp{pbuf(k1), kL, 0, 0, true}, CmOp{ybuf(k1), 2 * kL, 0, 0, true}, kL, idP, false, lead);
                }
            }
            if (fail) {
                // products still in flight finish before the tensor memory is freed (bounded wait)
                umma_commit_w(mX, lead);
                mbar_wait(mX, 0);
            }
        } else if (warp == kSweepMathWarps + 1) {
            // ================================================================ copy warp (lane 0)
            if (lane == 0) {
                int nT = 0, nQ = 0, nP[2] = {0, 0}, nK[2] = {0, 0}, nY[2] = {0, 0};
                auto copy_T = [&](int cc) {                      // T of chunk cc
                    mbar_expect_tx(cbT, kL * kL * 2);
                    bulk_load(tmm, p.tm + (head * NC + cc) * kL * kL, kL * kL * 2, cbT);
                    ++nT;
                };
                auto copy_Q = [&](int cc) {                      // Q of chunk cc: rows 0-63 of its [Q; K] block
                    mbar_expect_tx(cbQ, kL * DK * 2);
                    tma_load_5d(qb, &tm_qk, cbQ, 0, 0, 0, 0, qkblk0 + cc);
                    ++nQ;
                };
                // the chunk handled kk-th: K (rows 64-127 of its [Q; K] block), P (rows 0-63 of its
                // [P; KKm] block), and dY (one 128-row box in the [dY; dU] layout: rows 64-127, the
                // following steps, land in the dU rows, which the math warps rewrite before anything
                // reads them) with Lam (rows past T: zeros)
                auto copy_K = [&](int kk) {
                    mbar_expect_tx(cbK + (kk & 1), kL * DK * 2);
                    tma_load_5d(kbuf(kk), &tm_qk, cbK + (kk & 1), 0, 0, 1, 0, qkblk0 + NC - 1 - kk);
                    ++nK[kk & 1];
                };
                auto copy_P = [&](int kk) {
                    mbar_expect_tx(cbP + (kk & 1), kL * kL * 2);
                    tma_load_5d(pbuf(kk), &tm_pk, cbP + (kk & 1), 0, 0, 0, 0, (int)(head * NC) + NC - 1 - kk);
                    ++nP[kk & 1];
                };
                auto fetch = [&](int kk) {
                    const int cc = NC - 1 - kk;
                    mbar_expect_tx(cbY + (kk & 1), 2 * kL * kL * 2 + kL * 4);
                    tma_load_5d(ybuf(kk), &tm_dy, cbY + (kk & 1), 0, cc * kL, r0 / 8, h, b);
                    bulk_load(lms + (kk & 1) * kL, p.lam + (head * NC + cc) * kL, kL * 4, cbY + (kk & 1));
                    ++nY[kk & 1];
                };
                for (int kk = 0; kk < 2 && kk < NC; ++kk) {
                    copy_K(kk);
                    fetch(kk);
                    copy_P(kk);
                }
                copy_T(NC - 1);
                copy_Q(NC - 1);
                for (int k = 0; k < NC; ++k) {
                    const int c = NC - 1 - k;
                    const size_t chk = head * NC + c, blk = chk * nsplit + split;
                    // dS_L (high part) for the gradient kernel once written
                    if (!mbar_wait(bH, k & 1)) { fail = true; break; }
                    bulk_store(p.ws_dsl + blk * kL * DK, shl, kL * DK * 2);
                    bulk_commit();
                    // rhs written: the math warps saw m1, so this chunk's P buffer is free (the
                    // chunk two ahead)
                    if (!mbar_wait(bR, k & 1)) { fail = true; break; }
                    if (k + 2 < NC) copy_P(k + 2);
                    bulk_wait_read();                           // the dS_L store has read the dS parts
                    mbar_arrive(fS);
                    // dU written: the math warps saw mD, so T is free; the block's outputs leave
                    if (!mbar_wait(bU, k & 1)) { fail = true; break; }
                    if (c > 0) copy_T(c - 1);
                    bulk_store(p.ws_yu + blk * 2 * kL * kL, ybuf(k), 2 * kL * kL * 2);
                    bulk_store(p.ws_dl + blk * kL * kL, dls, kL * kL * 2);
                    tma_store_4d(&tm_dv, dvs, r0, h, c * kL, b);
                    bulk_commit();
                    // the carry is done: Q and this chunk's K buffer are free; once the stores have
                    // read them, so are the [dY; dU] buffer and the staging tiles (Lam was read
                    // before bR)
                    if (!mbar_wait(mS, k & 1)) { fail = true; break; }
                    if (c > 0) copy_Q(c - 1);
                    if (k + 2 < NC) copy_K(k + 2);
                    bulk_wait_read();
                    mbar_arrive(fO);
                    if (k + 2 < NC) fetch(k + 2);
                    // every second chunk: the two chunks handled three and two before (c + 3, c + 2)
                    // are complete for the gradient kernel -- their bulk stores (committed a chunk
                    // or more ago: every group but the last four) and the math warps' f and dbeta
                    // partials (written before they arrived at a later chunk's bU). Publishing
                    // every chunk, or with a lag of one, held the copy warp up on its chain.
                    if (p.ready != nullptr && k > 1 && (k & 1) == 1) {
                        bulk_wait_but<4>();
                        add_release_gpu(p.ready + head * NC + c + 3, 1u);
                        add_release_gpu(p.ready + head * NC + c + 2, 1u);
                    }
                }
                if (fail) {
                    // copies still in flight land before the CTA exits (each wait bounded)
                    if (nT > 0) mbar_wait(cbT, (nT - 1) & 1);
                    if (nQ > 0) mbar_wait(cbQ, (nQ - 1) & 1);
                    for (int i = 0; i < 2; ++i) {
                        if (nP[i] > 0) mbar_wait(cbP + i, (nP[i] - 1) & 1);
                        if (nK[i] > 0) mbar_wait(cbK + i, (nK[i] - 1) & 1);
                        if (nY[i] > 0) mbar_wait(cbY + i, (nY[i] - 1) & 1);
                    }
                }
                bulk_wait_all();                                // the block outputs are complete
            }
            fail = __shfl_sync(kFullMask, fail, 0);
        }
    } else {
        regs_inc<kSweepMathRegs>();
        // ================================================================ math warps
        // this thread's fragment of dS (rows fs.row(k), columns fs.col(j, k)), from dS_T
        const M64Frag fs(warp, lane, DK);
        float dS[NS];
#pragma unroll
        for (int j = 0; j < NS / 4; ++j)
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                float2 s2 = make_float2(0.f, 0.f);
                if (p.dS_T != nullptr)
                    s2 = *reinterpret_cast<const float2 *>(p.dS_T + (head * Dv + r0 + fs.row(2 * k2)) * DK + fs.col(j, 0));
                dS[4 * j + 2 * k2] = s2.x;
                dS[4 * j + 2 * k2 + 1] = s2.y;
            }
        // this thread's fragment of the 64-column accumulators (chunk rows ta, tb, value columns)
        const M64Frag fd(warp, lane, kL);
        const int ta = fd.row(0), tb = fd.row(2);
        // beta and v - u of rows ta, tb (value columns fd.col(j, 0), + 1): loaded one chunk ahead,
        // kept raw until used (rows past T: zeros)
        __nv_bfloat16 bna, bnb;
        float2 rna[4], rnb[4];
        auto load_rows = [&](int cc) {
            const int tt0 = cc * kL, ln = min(kL, T - tt0);
            const __nv_bfloat16 z = __float2bfloat16_rn(0.f);
            const size_t ra = ((size_t)b * T + tt0 + ta) * Hv + h, rb = ((size_t)b * T + tt0 + tb) * Hv + h;
            bna = ta < ln ? beta[ra] : z;
            bnb = tb < ln ? beta[rb] : z;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = r0 + fd.col(j, 0);
                rna[j] = ta < ln ? *reinterpret_cast<const float2 *>(p.resid + ra * Dv + col) : make_float2(0.f, 0.f);
                rnb[j] = tb < ln ? *reinterpret_cast<const float2 *>(p.resid + rb * Dv + col) : make_float2(0.f, 0.f);
            }
        };
        // a warp's part is written: its lanes' shared-memory writes are visible to the
        // products and copies, and its tensor-memory reads are complete
        auto warp_done = [&](uint64_t *bar_) {
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_);
        };
        load_rows(NC - 1);
        float decay_next = 1.f;                       // exp(Lam_L) of the chunk processed before (later in time)
        for (int k = 0; k < NC; ++k) {
            const int c = NC - 1 - k, buf = k & 1;
            const int t0 = c * kL, len = min(kL, T - t0);
            const size_t rowbase = (size_t)b * T + t0;          // (b, t0) row of [B, T, ...]
            unsigned char *ydu = ybuf(k);                      // [dY; dU] of this chunk
            const float *lmb = lms + buf * kL;                 // Lam of this chunk
            const float ba = __bfloat162float(bna), bb = __bfloat162float(bnb);
            float2 rsa[4], rsb[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                rsa[j] = rna[j];
                rsb[j] = rnb[j];
            }
            if (c > 0) load_rows(c - 1);
            // ---- dS of this chunk's end: exp(Lam_L) dS + the later chunk's part of the carry
            if (k > 0) {
                const bool w = mbar_wait(mS, (k - 1) & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < NS / 16; ++i) {
                    float x[16];
                    tmem_ld16x256_x4(tS + lane16 + SC * hw + 32 * i, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) dS[16 * i + e] = fmaf(decay_next, dS[16 * i + e], x[e]);
                }
                // the tile of the dS parts: the later chunk's products and dS_L store are done with it
                const bool w2 = mbar_wait(fS, (k - 1) & 1);
                if (__any_sync(kFullMask, !w2)) { fail = true; break; }
            }
            // ---- dS as operands: a bf16 high part and a bf16 low part (dS - high), each [64][DK],
            // the high part first (its product starts while the low part is formed); the high part
            // also leaves for the gradient kernel (a bulk store by the copy warp)
#pragma unroll
            for (int j = 0; j < NS / 4; j += 2) {
                uint32_t hi[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) hi[m] = pack2_bf16(dS[4 * j + 2 * m], dS[4 * j + 2 * m + 1]);
                stmatrix_x4(frag_row_addr(smem_addr(shl), kL, 16 * (warp & 3), (DK / 16) * hw + j, lane), hi[0], hi[1],
                            hi[2], hi[3]);
            }
            warp_done(bHi);
#pragma unroll
            for (int j = 0; j < NS / 4; j += 2) {
                uint32_t lo[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float x0 = dS[4 * j + 2 * m], x1 = dS[4 * j + 2 * m + 1];
                    const uint32_t hi = pack2_bf16(x0, x1);
                    lo[m] = pack2_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
                }
                stmatrix_x4(frag_row_addr(smem_addr(shl), kL, 16 * (warp & 3), (DK / 16) * hw + j, lane) + kL * DK * 2,
                            lo[0], lo[1], lo[2], lo[3]);
            }
            warp_done(bH);
            // ---- this chunk's dY and Lam
            {
                const bool w = mbar_wait(cbY + buf, (k >> 1) & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
            }
            const float ela = expf(lmb[kL - 1] - lmb[ta]), elb = expf(lmb[kL - 1] - lmb[tb]);
            const float ga = expf(lmb[ta]), gb = expf(lmb[tb]);
            decay_next = expf(lmb[kL - 1]);
            // diag(exp Lam) dY while the products run: rows 0-63 of the carry's operand (the dU
            // rows follow below); its tile is free since the later chunk's carry is done (mS)
            for (int e = tid; e < kL * kL / 8; e += kSweepMathWarps * 32) {
                const int t = e & (kL - 1);
                const uint32_t o = cm_off(t, 16 * (e >> 6), 2 * kL);
                float x8[8];
                unpack8(*reinterpret_cast<const uint4 *>(ydu + o), x8);
                const float gt = expf(lmb[t]);
#pragma unroll
                for (int i = 0; i < 8; ++i) x8[i] *= gt;
                *reinterpret_cast<uint4 *>(yds + o) = pack8(x8);
            }
            // ---- rhs = diag(E_L) K dS^T + P^T dY as an operand; Delta = beta (v - u) for the gradient
            // kernel; f partial = beta_t (v_t - u_t) . (dS k_t) over this warp's 32 value columns
            {
                bool w = mbar_wait(m1, k & 1);
                if (k > 0) w = w && mbar_wait(fO, (k - 1) & 1);   // the Delta and dv tiles are free
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
            }
            tc_fence_after();
            {
                float xh[16], pp[16];
                tmem_ld16x256_x4(tX + lane16 + 32 * hw, xh);
                tmem_ld16x256_x4(tP + lane16 + 32 * hw, pp);
                tmem_wait_ld();
                float fa = 0.f, fb = 0.f;
                uint32_t rv[8], dl[8];   // pairs (j, row ta), (j, row tb) for j = 0..3
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 ra = rsa[j], rb = rsb[j];
                    const float x0 = xh[4 * j], x1 = xh[4 * j + 1], x2 = xh[4 * j + 2], x3 = xh[4 * j + 3];
                    fa = fmaf(ra.x, x0, fmaf(ra.y, x1, fa));
                    fb = fmaf(rb.x, x2, fmaf(rb.y, x3, fb));
                    rv[2 * j] = pack2_bf16(fmaf(ela, x0, pp[4 * j]), fmaf(ela, x1, pp[4 * j + 1]));
                    rv[2 * j + 1] = pack2_bf16(fmaf(elb, x2, pp[4 * j + 2]), fmaf(elb, x3, pp[4 * j + 3]));
                    dl[2 * j] = pack2_bf16(ba * ra.x, ba * ra.y);
                    dl[2 * j + 1] = pack2_bf16(bb * rb.x, bb * rb.y);
                }
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                    const uint32_t o = frag_row_addr(0, kL, 16 * (warp & 3), 4 * hw + j, lane);
                    stmatrix_x4(smem_addr(rhs) + o, rv[2 * j], rv[2 * j + 1], rv[2 * j + 2], rv[2 * j + 3]);
                    stmatrix_x4(smem_addr(dls) + o, dl[2 * j], dl[2 * j + 1], dl[2 * j + 2], dl[2 * j + 3]);
                }
                warp_done(bR);
                // the row sums over this warp's 32 columns: the four lanes that share a row
                fa += __shfl_xor_sync(kFullMask, fa, 1);
                fa += __shfl_xor_sync(kFullMask, fa, 2);
                fb += __shfl_xor_sync(kFullMask, fb, 1);
                fb += __shfl_xor_sync(kFullMask, fb, 2);
                if ((lane & 3) == 0) {
                    float *f = p.ws_f + (rowbase * Hv + h) * 2 * nsplit + 2 * split + hw;
                    if (ta < len) f[(size_t)ta * Hv * 2 * nsplit] = ba * fa;
                    if (tb < len) f[(size_t)tb * Hv * 2 * nsplit] = bb * fb;
                }
            }
            // ---- dv = beta dD, dbeta partial, dU = -beta dD (operand rows 64-127, stored for the
            // gradient kernel) and exp(Lam) dU (the carry's operand)
            {
                const bool w = mbar_wait(mD, k & 1);
                if (__any_sync(kFullMask, !w)) { fail = true; break; }
            }
            tc_fence_after();
            {
                float x[16];
                tmem_ld16x256_x4(tX + lane16 + 32 * hw, x);
                tmem_wait_ld();
                float da = 0.f, db = 0.f;
                uint32_t du[8], us[8], dv[8];   // pairs (j, row ta), (j, row tb) for j = 0..3
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 ra = rsa[j], rb = rsb[j];
                    da = fmaf(x[4 * j], ra.x, fmaf(x[4 * j + 1], ra.y, da));
                    db = fmaf(x[4 * j + 2], rb.x, fmaf(x[4 * j + 3], rb.y, db));
                    const float va0 = ba * x[4 * j], va1 = ba * x[4 * j + 1], vb0 = bb * x[4 * j + 2], vb1 = bb * x[4 * j + 3];
                    du[2 * j] = pack2_bf16(-va0, -va1);
                    du[2 * j + 1] = pack2_bf16(-vb0, -vb1);
                    us[2 * j] = pack2_bf16(-ga * va0, -ga * va1);
                    us[2 * j + 1] = pack2_bf16(-gb * vb0, -gb * vb1);
                    dv[2 * j] = pack2_bf16(va0, va1);
                    dv[2 * j + 1] = pack2_bf16(vb0, vb1);
                }
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                    // dU: rows 64-127 of [dY; dU] (stored for the gradient kernel) and of the carry's
                    // operand (scaled by exp Lam)
                    const uint32_t o = frag_row_addr(0, 2 * kL, kL + 16 * (warp & 3), 4 * hw + j, lane);
                    stmatrix_x4(smem_addr(ydu) + o, du[2 * j], du[2 * j + 1], du[2 * j + 2], du[2 * j + 3]);
                    stmatrix_x4(smem_addr(yds) + o, us[2 * j], us[2 * j + 1], us[2 * j + 2], us[2 * j + 3]);
                    // dv staged in the 128-byte swizzle for a TMA store (rows past T are clipped by
                    // it): row t at t * 128, 16-byte chunk c (8 columns) at c ^ (t % 8)
                    const int m = lane >> 3, t = 16 * (warp & 3) + 8 * (m & 1) + (lane & 7), cc = 4 * hw + j + (m >> 1);
                    stmatrix_x4(smem_addr(dvs) + t * 128 + ((cc ^ (t & 7)) << 4), dv[2 * j], dv[2 * j + 1], dv[2 * j + 2],
                                dv[2 * j + 3]);
                }
                warp_done(bU);
                da += __shfl_xor_sync(kFullMask, da, 1);
                da += __shfl_xor_sync(kFullMask, da, 2);
                db += __shfl_xor_sync(kFullMask, db, 1);
                db += __shfl_xor_sync(kFullMask, db, 2);
                if ((lane & 3) == 0) {
                    float *d = p.ws_db + (rowbase * Hv + h) * 2 * nsplit + 2 * split + hw;
                    if (ta < len) d[(size_t)ta * Hv * 2 * nsplit] = da;
                    if (tb < len) d[(size_t)tb * Hv * 2 * nsplit] = db;
                }
            }
        }
        if (!fail && p.dS0 != nullptr) {
            // dS0 = exp(Lam_L) dS + the first chunk's part of the carry
            const bool w = mbar_wait(mS, (NC - 1) & 1);
            fail = __any_sync(kFullMask, !w);
            if (!fail) {
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < NS / 16; ++i) {
                    float x[16];
                    tmem_ld16x256_x4(tS + lane16 + SC * hw + 32 * i, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) dS[16 * i + e] = fmaf(decay_next, dS[16 * i + e], x[e]);
                }
#pragma unroll
                for (int j = 0; j < NS / 4; ++j)
#pragma unroll
                    for (int k2 = 0; k2 < 2; ++k2)
                        *reinterpret_cast<float2 *>(p.dS0 + (head * Dv + r0 + fs.row(2 * k2)) * DK + fs.col(j, 0)) =
                            make_float2(dS[4 * j + 2 * k2], dS[4 * j + 2 * k2 + 1]);
            }
        }
    }
    if (fail && lane == 0) report_status(p.status, kStatusTimeout);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the chunks the loop left (the last two or three) for the gradient kernel: the copy warp's
    // stores completed (bulk_wait_all) and the math warps' partials precede the barrier
    if (warp == kSweepMathWarps + 1 && lane == 0 && !fail && p.ready != nullptr) {
        for (int cc = ((NC - 1) & 1) == 1 ? 1 : 2; cc >= 0; --cc)   // what the loop left
            if (cc < NC) add_release_gpu(p.ready + head * NC + cc, 1u);
    }
    if (warp == kSweepMathWarps) tmem_dealloc(tmem, 512);
}

namespace {

// ------------------------------------------------------------------ per-chunk gradients
struct GradSmem {
    size_t qk, yu, dl, s0, dsl, vec, stg, bar, tslot, total;
    size_t gehe, wst, mt;     // in the S0 region once the first products are done
    __host__ __device__ GradSmem(int DK, int Dv) {
        size_t o = 0;
        qk = o; o += (size_t)2 * kL * DK * 2;                      // [Q; K] [128][DK]
        yu = o; o += (size_t)2 * kL * Dv * 2;                      // [dY; dU] [128][Dv]
        dl = o; o += (size_t)kL * Dv * 2;                          // Delta [64][Dv]
        s0 = o;
        {
            const size_t a = (size_t)Dv * DK * 2, b2 = (size_t)5 * kL * kL * 2;
            o += a > b2 ? a : b2;                                  // S0 [Dv / 64][64][DK]; later GE|HE, W1|W2 [128][64], M^T [64][64]
        }
        gehe = s0; wst = s0 + (size_t)2 * kL * kL * 2; mt = wst + (size_t)2 * kL * kL * 2;
        dsl = o; o += (size_t)Dv * DK * 2;                         // dS_L [Dv / 64][64][DK]
        vec = o; o += (6 * kL + 4 * kL + 16 + 12 * kL + 4 * kL) * 4;   // Lam, Lam_{t-1}, exp Lam, E(L,.), beta, f; ab [2][128]; c0 parts; dg parts [4][3][64]; Z column sums [4][64]
        stg = alb(o, 1024);                                        // the unit's decay table E [64][65] fp32; at the group's end
        {                                                          // dq or dk [64 rows][DK] bf16 in 64-column 128-byte-swizzled boxes
            const size_t a = (size_t)kL * DK * 2, b2 = (size_t)kL * (kL + 1) * 4;
            o = stg + (a > b2 ? a : b2);
        }
        bar = alb(o, 8); o = bar + 5 * 8;                          // MMA; copies of (dY;dU, Delta, dS_L), of S0, of [Q; K]; drain
        tslot = o; o += 16;
        total = o + 1024;
        if (total < kOneCtaSmem) total = kOneCtaSmem;
    }
};

}  // namespace

// Persistent: one CTA per SM, each taking whole groups of units (b, chunk, value heads of one kv
// head) from a counter, last chunk first, and the units of a group in ascending value head, so
// that they share [Q; K] and the value heads of a kv head are summed by one CTA, in ascending
// order, whatever the grid or the order the groups are taken in. Given ready counters, the
// kernel runs alongside the reverse sweep (it does not wait for it to finish): the sweep goes
// through the chunks from the last, publishing them (ready counters), and a group starts once
// every CTA of the sweep has published its chunk for the group's value heads, so that the SMs the
// sweep leaves free work from its first chunks on. Every operand arrives by bulk
// copy, the next unit's as soon as its buffers are free, all after the second products:
// [dY; dU], Delta (scaled in place by E_L for the second products) and dS_L, S0 (whose region
// then holds the scratch operands) and [Q; K] (when the kv head or chunk changes).
// Tensor memory:
//   [0, DK)             R1, M = 128, per unit: first [dY; dU] S0 (rows 0-63 for dQ, 64-127 for
//                       dK), then (diag(E_L) Delta) dS_L + GE^T Q + HE^T K, whose A operands are
//                       read from 64 rows before the real ones, so that row t lands in the lane
//                       of dK row t (rows 0-63 are not used)
//   [DK, 2 DK)          RS, M = 128: [dQ; dK] summed over the value heads of the kv head's
//                       group: per unit += diag(e^Lam) [dY; dU] S0 (from R1, on the
//                       CUDA cores), += [GE; HE] K (MMA), rows 64-127 += R1's second terms
//   [2 DK, 2 DK + 64)   [Q; K] K^T (M = 128), formed once per (b, chunk, kv head)
//   [2 DK + 64, + 128)  [dY; dU] Delta^T = [G; H] (M = 128), later [W1; W2] M (M = 128)
template <int E>
__global__ void __launch_bounds__(256, 1) chunk_grad_kernel(ChunkBwdParams p, int groups,
                                                            const __grid_constant__ CUtensorMap tm_dq,
                                                            const __grid_constant__ CUtensorMap tm_dk) {
    constexpr int DK = 32 * E;
    constexpr int SC = DK / 2;
    static_assert(2 * DK + 128 <= 512, "tensor memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.T, Dv = p.Dv, Hv = p.Hv, Hk = p.Hk, nsplit = p.nsplit, NC = p.NC, rep = Hv / Hk;
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    // unit u = ((b * NC + c) * Hk + hk) * rep + (h % rep): group u / rep

    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(alb(reinterpret_cast<size_t>(smem_raw), 1024));
    const GradSmem L(DK, Dv);
    unsigned char *qk = base + L.qk, *yu = base + L.yu, *dl = base + L.dl, *s0 = base + L.s0, *dsl = base + L.dsl;
    unsigned char *gehe = base + L.gehe, *wst = base + L.wst, *mt = base + L.mt;
    unsigned char *stg = base + L.stg;
    float *Et = reinterpret_cast<float *>(stg);                // E [64][65], see below
    float *Lm = reinterpret_cast<float *>(base + L.vec), *LmP = Lm + kL, *gm = LmP + kL, *eL = gm + kL;
    float *bt = eL + kL, *fv = bt + kL, *abp = fv + kL, *c0p = abp + 4 * kL, *dgp = c0p + 16, *zq = dgp + 12 * kL;
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + L.bar), *cbA = bar + 1, *cbS = bar + 2, *cbQ = bar + 3, *mX = bar + 4;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(base + L.tslot);
    const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(p.beta);

    // unit u = ((b * NC + c) * Hv + h)
    auto chunk_of = [&](int u, int &b, int &c, int &h) {
        h = u % Hv;
        const int bc = u / Hv;
        c = bc % NC;
        b = bc / NC;
    };
    constexpr unsigned kSb = kL * DK * 2, kYub = 2 * kL * kL * 2, kDlb = kL * kL * 2, kQkb = 2 * kL * DK * 2;
    int nA = 0, nS = 0, nQ = 0, wA = 0, wS = 0, wQ = 0;
    auto copy_a = [&](int u) {            // [dY; dU], Delta and dS_L of unit u
        int b, c, h;
        chunk_of(u, b, c, h);
        const size_t chk = ((size_t)b * Hv + h) * NC + c;
        // the row blocks of a unit are adjacent in the workspace and in shared memory
        mbar_expect_tx(cbA, (unsigned)nsplit * (kYub + kDlb + kSb));
        const size_t blk = chk * nsplit;
        bulk_load(yu, p.ws_yu + blk * 2 * kL * kL, (unsigned)nsplit * kYub, cbA);
        bulk_load(dl, p.ws_dl + blk * kL * kL, (unsigned)nsplit * kDlb, cbA);
        bulk_load(dsl, p.ws_dsl + blk * kL * DK, (unsigned)nsplit * kSb, cbA);
        ++nA;
    };
    auto copy_s = [&](int u) {            // S0 of unit u
        int b, c, h;
        chunk_of(u, b, c, h);
        const size_t chk = ((size_t)b * Hv + h) * NC + c;
        mbar_expect_tx(cbS, (unsigned)nsplit * kSb);
        bulk_load(s0, p.s0m + chk * nsplit * kL * DK, (unsigned)nsplit * kSb, cbS);
        ++nS;
    };
    auto copy_q = [&](int u) {            // [Q; K] of unit u's chunk and kv head
        int b, c, h;
        chunk_of(u, b, c, h);
        mbar_expect_tx(cbQ, kQkb);
        bulk_load(qk, p.qkm + (((size_t)b * Hk + h / rep) * NC + c) * 2 * kL * DK, kQkb, cbQ);
        ++nQ;
    };
    // the group taken i-th: chunks from the last (the reverse sweep's order), then batch row and
    // kv head
    auto group_of = [&](int i) {
        const int per_c = p.B * Hk, c = NC - 1 - i / per_c, r = i % per_c;
        return ((r / Hk) * NC + c) * Hk + r % Hk;
    };
    // thread 32 (which issues the copies): the group taken as index i (>= groups when none is
    // left) once every value head of it has the chunk published by all nsplit CTAs of the
    // reverse sweep (the heads' counters polled together, bounded), into next_slot for every
    // thread once a barrier has passed (-1 when the wait ran out); then what the sweep published
    // is visible to this thread's copies and, past the barrier, to every thread's loads
    int *next_slot = reinterpret_cast<int *>(tslot + 1);
    auto resolve_group = [&](int i) {
        bool okw = true;
        if (i < groups && p.ready != nullptr) {
            const int g = group_of(i), hk = g % Hk, c = (g / Hk) % NC, b = g / Hk / NC;
            const unsigned *f = p.ready + ((size_t)b * Hv + hk * rep) * NC + c;   // head hk rep + hh at + hh NC
            for (int h0 = 0; h0 < rep && okw; h0 += 4) {
                for (unsigned it = 0;; ++it) {
                    unsigned v[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = h0 + j < rep ? load_relaxed_gpu(f + (size_t)(h0 + j) * NC) : nsplit;
                    bool all = true;
#pragma unroll
                    for (int j = 0; j < 4; ++j) all = all && v[j] >= (unsigned)nsplit;
                    if (all) break;
                    if (it >= kReadyWaitLimit) { okw = false; break; }
                    __nanosleep(64);
                }
            }
            fence_acquire_gpu();
            fence_proxy_async_global();
        }
        *next_slot = okw ? i : -1;
    };
    // decays, beta and the f partials of a unit (threads < 64), loaded one unit ahead and kept
    // raw (converted and summed where they are used, so that the loads do not stall here)
    constexpr int kMaxPart = 8;                             // two per block of 64 value rows, Dv <= 256
    const int nparts = 2 * nsplit;
    float vlam = 0.f, vfp[kMaxPart], vdb[kMaxPart];
    __nv_bfloat16 vbt = __float2bfloat16_rn(0.f);
    auto load_vec = [&](int u) {
        if (tid >= kL) return;
        int b, c, h;
        chunk_of(u, b, c, h);
        const size_t chk = ((size_t)b * Hv + h) * NC + c;
        const int t0 = c * kL, len = min(kL, T - t0);
        const size_t row = ((size_t)b * T + t0 + (tid < len ? tid : 0)) * Hv + h;
        vlam = p.lam[chk * kL + tid];
        vbt = beta[row];
#pragma unroll
        for (int s = 0; s < kMaxPart; ++s) {
            vfp[s] = s < nparts ? p.ws_f[row * nparts + s] : 0.f;
            vdb[s] = s < nparts ? p.ws_db[row * nparts + s] : 0.f;
        }
    };

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(bar + i, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    const uint32_t lead = warp == 0 ? elect_one_sync() : 0u;   // the lane of warp 0 that issues products
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tR1 = tmem, tRS = tmem + DK, tS1 = tmem + 2 * DK, tS2 = tmem + 2 * DK + 64;
    // With ready counters, no wait for the previous kernel (the reverse sweep) to finish: its
    // outputs are taken chunk by chunk through them, and everything else this kernel reads was
    // written before the reverse sweep began. Without, the sweep's writes are all visible first.
    if (p.ready == nullptr) griddep_wait();
    griddep_launch();

    if (tid == 32) resolve_group(atomicAdd(p.next, 1));
    __syncthreads();
    bool ok = *next_slot >= 0;
    int un = ok && *next_slot < groups ? group_of(*next_slot) * rep : -1;   // the next unit
    if (tid == 32 && un >= 0) {
        copy_q(un);
        copy_a(un);
        copy_s(un);
    }
    if (un >= 0) load_vec(un);
    unsigned ph = 0;
    int taken = 0;      // thread 32: the index of the group after this one, taken at this group's first unit
    int nxt = 0;        // every thread: that index once resolved (in the first unit's second products)
    for (int u = un; u >= 0 && ok; u = un) {
        int b, c, h;
        chunk_of(u, b, c, h);
        const int t0 = c * kL, len = min(kL, T - t0);
        const size_t rowbase = (size_t)b * T + t0;
        const bool newq = u % rep == 0;                     // a new group: its [Q; K]
        // ---- decays, beta, f
        if (tid < kL) {
            Lm[tid] = vlam;
            gm[tid] = expf(vlam);
            const bool in = tid < len;
            bt[tid] = in ? __bfloat162float(vbt) : 0.f;
            float f = 0.f;
#pragma unroll
            for (int s = 0; s < kMaxPart; ++s) f += s < nparts ? vfp[s] : 0.f;   // partials in ascending order
            fv[tid] = in ? f : 0.f;
            // dbeta of the row: its value-row block partials, in ascending order
            float db = 0.f;
#pragma unroll
            for (int s = 0; s < kMaxPart; ++s) db += s < nparts ? vdb[s] : 0.f;
            if (in) static_cast<__nv_bfloat16 *>(p.dbeta)[(rowbase + tid) * Hv + h] = __float2bfloat16_rn(db);
        }
        if (tid == 32) bulk_wait_read();                    // the last group's dq, dk stores have read stg
        __syncthreads();
        if (tid < kL) {
            LmP[tid] = tid > 0 ? Lm[tid - 1] : 0.f;
            eL[tid] = expf(Lm[kL - 1] - Lm[tid]);
        }
        // the unit's decay weights E(s, i) = exp(Lam_s - Lam_i) <= 1 for i <= s (0 above the
        // diagonal), in the output tile (not used until this unit's dq, dk leave)
        for (int e = tid; e < kL * kL; e += 256) {
            const int s2 = e >> 6, i = e & (kL - 1);
            Et[s2 * (kL + 1) + i] = i <= s2 ? expf(Lm[s2] - Lm[i]) : 0.f;
        }
        // ---- this unit's operands (every thread reads S0 and dS_L, and [Q; K] rows in pass 1)
        {
            bool w = mbar_wait(cbA, wA & 1) && mbar_wait(cbS, wS & 1);
            if (newq) w = w && mbar_wait(cbQ, wQ & 1);
            ok = !__syncthreads_or(!w);
            ++wA;
            ++wS;
            if (newq) ++wQ;
        }
        tc_fence_after();
        if (!ok) break;
        // this unit's place in its group of value heads (one kv head, one chunk), which lies
        // wholly in this CTA's range
        const int hh = h % rep;
        const bool gfirst = hh == 0, glast = hh == rep - 1;
        // ---- first products: [Q; K] K^T (when the kv head or chunk changes), [dY; dU] Delta^T,
        // [dY; dU] S0
        if (warp == 0) {
            if (newq)
                umma_gemm_w(tS1, CmOp{qk, 2 * kL, 0, 0, false}, CmOp{qk, 2 * kL, kL, 0, false}, DK,
                            umma_idesc_t(1, 2 * kL, kL, false, false), false, lead);
            umma_gemm_w(tS2, CmOp{yu, 2 * kL, 0, 0, false}, CmOp{dl, kL, 0, 0, false}, Dv,
                        umma_idesc_t(1, 2 * kL, kL, false, false), false, lead);
            for (int s = 0; s < nsplit; ++s)
                umma_gemm_w(tR1, CmOp{yu, 2 * kL, 0, kL * s, false}, CmOp{s0 + (size_t)s * kSb, kL, 0, 0, true}, kL,
                            umma_idesc_t(1, 2 * kL, DK, false, true), s > 0, lead);
            umma_commit_w(bar, lead);
        }
        // ---- the group after this one, taken at this group's first unit (thread 32; resolved in
        // the second products)
        if (gfirst && tid == 32) taken = atomicAdd(p.next, 1);
        // ---- c0 = <dS_L, S0> (both in the same layout) while the products run, by warps 1-7 (warp
        // 0 is issuing them)
        if (warp > 0) {
            float c0s = 0.f;
            const uint4 *a4 = reinterpret_cast<const uint4 *>(s0), *d4 = reinterpret_cast<const uint4 *>(dsl);
            const int n8 = Dv * DK / 8;
#pragma unroll 4
            for (int e = tid - 32; e < n8; e += 224) {
                float x[8], d[8];
                unpack8(a4[e], x);
                unpack8(d4[e], d);
#pragma unroll
                for (int i = 0; i < 8; ++i) c0s = fmaf(x[i], d[i], c0s);
            }
            c0s = warp_sum(c0s);
            if (lane == 0) c0p[warp] = c0s;
        } else if (lane == 0) {
            c0p[0] = 0.f;
        }
        tc_fence_before();
        ok = !__syncthreads_or(!mbar_wait(bar, ph & 1));
        ++ph;
        tc_fence_after();
        if (!ok) break;
        un = u + 1;
        if (glast && !gfirst) {                            // the next group, resolved at an earlier unit
            ok = nxt >= 0;
            if (!ok) break;
            un = nxt < groups ? group_of(nxt) * rep : -1;
        }
        if (un >= 0 && !(glast && gfirst)) load_vec(un);   // used at the next unit's start
        {
            // ---- G o E_incl, H o E_strict and [W1; W2] = [G o QK^T; H o KK^T] as operands
            const int r = 32 * quarter + lane, s = r & (kL - 1);
            const bool upper = r >= kL;
            {
                float a[32], g2[32];
                tmem_ld32f(tS1 + lane_off + half * 32, a);
                tmem_ld32f(tS2 + lane_off + half * 32, g2);
                tmem_wait_ld();
                const float *Es = Et + s * (kL + 1) + half * 32;
                float ge[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int col = half * 32 + i;
                    const bool keep = upper ? col < s : col <= s;
                    ge[i] = keep ? g2[i] * Es[i] : 0.f;
                    a[i] *= g2[i];
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t o = cm_off(r, 2 * (half * 32 + 8 * j), 2 * kL);
                    *reinterpret_cast<uint4 *>(gehe + o) = pack8(ge + 8 * j);
                    *reinterpret_cast<uint4 *>(wst + o) = pack8(a + 8 * j);
                }
            }
            // ---- R1: a_s = (dY S0)_s . q_s, b_s = (dU S0)_s . k_s; the rows scaled by exp(Lam_s)
            // into the running sum
            {
                const float gs = gm[s];
                float ab = 0.f;
                float x[SC];
#pragma unroll
                for (int j = 0; j < SC / 32; ++j) tmem_ld32f(tR1 + lane_off + half * SC + 32 * j, x + 32 * j);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < SC / 8; ++j) {
                    float qv[8];
                    unpack8(*reinterpret_cast<const uint4 *>(qk + cm_off(r, 2 * (half * SC + 8 * j), 2 * kL)), qv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        ab = fmaf(x[8 * j + i], qv[i], ab);
                        x[8 * j + i] *= gs;
                    }
                }
                abp[half * 2 * kL + r] = ab;
                // 32 columns at a time (registers)
#pragma unroll
                for (int j = 0; j < SC / 32; ++j) {
                    if (!gfirst) {
                        float y[32];
                        tmem_ld32f(tRS + lane_off + half * SC + 32 * j, y);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[32 * j + i] = y[i] + x[32 * j + i];
                    }
                    tmem_st32f(tRS + lane_off + half * SC + 32 * j, x + 32 * j);
                }
            }
            // ---- diag(E_L) Delta in place (G and H are formed): rows t scaled by E(L, t)
            for (int e = tid; e < kL * Dv / 8; e += 256) {
                const int t = e & (kL - 1);
                uint4 *p4 = reinterpret_cast<uint4 *>(dl) + e;    // piece e: row e % 64 of K chunk e / 64
                float d8[8];
                unpack8(*p4, d8);
                const float sc = eL[t];
#pragma unroll
                for (int i = 0; i < 8; ++i) d8[i] *= sc;
                *p4 = pack8(d8);
            }
            // ---- M^T [t][i] = E(t-1, i) for i < t, bf16 operand
            for (int e = tid; e < kL * kL / 8; e += 256) {
                const int t = e & (kL - 1), i0 = 8 * (e >> 6);
                float m8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) m8[j] = i0 + j < t ? Et[(t - 1) * (kL + 1) + i0 + j] : 0.f;
                *reinterpret_cast<uint4 *>(mt + cm_off(t, 2 * i0, kL)) = pack8(m8);
            }
        }
        tmem_wait_st();
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- second products: RS += [GE; HE] K; R1 = (diag(E_L) Delta) dS_L + GE^T Q + HE^T K;
        // Z = [W1; W2] M
        if (warp == 0) {
            umma_gemm_w(tRS, CmOp{gehe, 2 * kL, 0, 0, false}, CmOp{qk, 2 * kL, 0, kL, true}, kL,
                        umma_idesc_t(1, 2 * kL, DK, false, true), true, lead);
            for (int s = 0; s < nsplit; ++s)
                umma_gemm_w(tR1, CmOp{dl, kL, -kL, kL * s, false}, CmOp{dsl + (size_t)s * kSb, kL, 0, 0, true}, kL,
                            umma_idesc_t(1, 2 * kL, DK, false, true), s > 0, lead);
            umma_gemm_w(tR1, CmOp{gehe, 2 * kL, -kL, 0, true}, CmOp{qk, 2 * kL, 0, 0, true}, kL,
                        umma_idesc_t(1, 2 * kL, DK, true, true), true, lead);
            umma_gemm_w(tR1, CmOp{gehe, 2 * kL, -kL, kL, true}, CmOp{qk, 2 * kL, 0, kL, true}, kL,
                        umma_idesc_t(1, 2 * kL, DK, true, true), true, lead);
            umma_gemm_w(tS2, CmOp{wst, 2 * kL, 0, 0, false}, CmOp{mt, kL, 0, 0, false}, kL,
                        umma_idesc_t(1, 2 * kL, kL, false, false), false, lead);
            umma_commit_w(bar, lead);
        }
        {
            // ---- dg_t: the sums over the chunk's steps, a quarter of the steps per thread (while
            // the second products run: they need none of them)
            // s2 = sum_{j < t} E(t-1, j) f_j, s3 = exp(Lam_{t-1}) sum_{j >= t} E(j, t) (a_j + b_j)
            const int t = tid & (kL - 1), part = tid >> 6;
            const float *Ep = Et + (t > 0 ? t - 1 : 0) * (kL + 1);
            float s2 = 0.f, s3 = 0.f;
            for (int j = 16 * part; j < 16 * part + 16; ++j) {
                if (j < t) {
                    s2 = fmaf(Ep[j], fv[j], s2);
                } else {
                    const float ab = abp[j] + abp[2 * kL + j] + abp[kL + j] + abp[3 * kL + j];
                    s3 = fmaf(Et[j * (kL + 1) + t], ab, s3);
                }
            }
            dgp[(2 * part + 0) * kL + t] = s2;
            dgp[(2 * part + 1) * kL + t] = expf(LmP[t]) * s3;
        }
        if (gfirst && tid == 32) resolve_group(taken);
        ok = !__syncthreads_or(!mbar_wait(bar, ph & 1));
        ++ph;
        tc_fence_after();
        if (!ok) break;
        // [dY; dU], Delta, dS_L, the S0 region (scratch) and, when the next unit needs another
        // [Q; K], its buffer are free: the next unit's go out now
        if (gfirst) nxt = *next_slot;
        if (glast && gfirst) {                             // one unit per group: resolved just now
            ok = nxt >= 0;
            if (!ok) break;
            un = nxt < groups ? group_of(nxt) * rep : -1;
            if (un >= 0) load_vec(un);                     // used at the next unit's start
        }
        if (tid == 32 && un >= 0) {
            copy_a(un);
            copy_s(un);
            if (glast) copy_q(un);
        }
        {
            // ---- Z weighted by E(s, t) (s >= t), summed over the rows of both halves: a
            // transpose reduction over the warp's 32 rows, then the four row quarters
            const int r = 32 * quarter + lane, s = r & (kL - 1);
            float z[32];
            tmem_ld32f(tS2 + lane_off + half * 32, z);
            tmem_wait_ld();
            const float *Es = Et + s * (kL + 1) + half * 32;
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] *= Es[i];   // E(s, t) = 0 for t > s
            zq[quarter * kL + half * 32 + lane] = transpose_reduce<32>(z, lane);
        }
        __syncthreads();
        if (tid < kL && tid < len) {
            const int t = tid;
            float c0 = 0.f;
            for (int w = 0; w < 8; ++w) c0 += c0p[w];
            float s2 = 0.f, s3 = 0.f, s4 = 0.f;
            for (int part = 0; part < 4; ++part) {
                s2 += dgp[(2 * part + 0) * kL + t];
                s3 += dgp[(2 * part + 1) * kL + t];
                s4 += zq[part * kL + t];
            }
            const float lt = Lm[t], lp = LmP[t], lL = Lm[kL - 1];
            const float dgv = expf(lL - lt + lp) * c0 + expf(lL - lt) * s2 + s3 + s4;
            static_cast<__nv_bfloat16 *>(p.dg)[(rowbase + t) * Hv + h] = __float2bfloat16_rn(dgv);
        }
        {
            // ---- rows 64-127 of R1 (the second dK terms) into the running sum
            const int r = 32 * quarter + lane;
            if (r >= kL) {
#pragma unroll
                for (int j = 0; j < SC / 32; ++j) {
                    float x[32], y[32];
                    tmem_ld32f(tR1 + lane_off + half * SC + 32 * j, x);
                    tmem_ld32f(tRS + lane_off + half * SC + 32 * j, y);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = y[i] + x[i];
                    tmem_st32f(tRS + lane_off + half * SC + 32 * j, x);
                }
                tmem_wait_st();
            }
        }
        if (glast) {
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            // ---- dq (rows 0-63) and then dk (rows 64-127) of the group, from RS, as bf16: each
            // staged in 64-column boxes in the 128-byte swizzle (row r at r * 128, 16-byte chunk j at
            // j ^ (r % 8)) and written by TMA stores (rows past T are clipped by them)
            const int hk = h / rep;
            float x[SC];
#pragma unroll
            for (int j = 0; j < SC / 32; ++j) tmem_ld32f(tRS + lane_off + half * SC + 32 * j, x + 32 * j);
            tmem_wait_ld();
            const int r = 32 * quarter + lane, t = r & (kL - 1);
            for (int pass = 0; pass < 2; ++pass) {
                if ((quarter >> 1) == pass) {
#pragma unroll
                    for (int j = 0; j < SC / 8; ++j) {
                        const int col = half * SC + 8 * j;
                        *reinterpret_cast<uint4 *>(stg + (col >> 6) * (kL * 128) + t * 128 +
                                                   ((((col & 63) >> 3) ^ (t & 7)) << 4)) = pack8(x + 8 * j);
                    }
                }
                fence_proxy_async();
                __syncthreads();
                if (tid == 32) {
                    for (int bx = 0; bx < DK / 64; ++bx)
                        tma_store_4d(pass ? &tm_dk : &tm_dq, stg + bx * (kL * 128), 64 * bx, hk, t0, b);
                    bulk_commit();
                    if (pass == 0) bulk_wait_read();        // dk reuses the tile
                }
                if (pass == 0) __syncthreads();
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (!ok && tid == 32) {
        report_status(p.status, kStatusTimeout);
        // copies still in flight land before the CTA exits (each wait bounded)
        if (nA > wA) mbar_wait(cbA, (nA - 1) & 1);
        if (nS > wS) mbar_wait(cbS, (nS - 1) & 1);
        if (nQ > wQ) mbar_wait(cbQ, (nQ - 1) & 1);
    }
    if (!ok && warp == 0) {
        // products still in flight finish before the tensor memory is freed (bounded wait)
        umma_commit_w(mX, lead);
        mbar_wait(mX, 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
    // this kernel completes after the reverse sweep, so that what follows on the stream sees both
    griddep_wait();
}

size_t chunk_dsweep_smem(int Dk) { return DSweepSmem(Dk).total; }
size_t chunk_grad_smem(int Dk, int Dv) { return GradSmem(Dk, Dv).total; }

template <int E>
static cudaError_t launch_chunk_bwd_t(const ChunkBwdParams &p, const CUtensorMap &tm_dv, const CUtensorMap &tm_dy,
                                      const CUtensorMap &tm_qk, const CUtensorMap &tm_pk, const CUtensorMap &tm_dq,
                                      const CUtensorMap &tm_dk, cudaStream_t s, int stages) {
    constexpr int DK = 32 * E;
    const size_t sd = DSweepSmem(DK).total, sg = GradSmem(DK, p.Dv).total;
    // the reverse sweep's register split waits for registers that only a launch of
    // kSweepLaunchRegs per thread provides
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, chunk_dsweep_kernel<E>);
    if (err != cudaSuccess) return err;
    if (fa.numRegs < kSweepLaunchRegs || fa.maxThreadsPerBlock < kSweepThreads) return cudaErrorInvalidConfiguration;
    err = cudaFuncSetAttribute(chunk_dsweep_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sd);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(chunk_grad_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sg);
    if (err != cudaSuccess) return err;
    const int groups = p.NC * p.Hk * p.B;                   // (b, chunk, kv head)
    int dev = 0, sms = 0;
    err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    // The gradient kernel runs alongside the reverse sweep (on the ready counters it publishes)
    // where that pays: the sweep in one wave (all its rows publish their chunks in step) and more
    // groups than SMs (a CTA that takes its next group early then keeps none from an idle CTA).
    // Elsewhere it waits for the sweep to finish.
    ChunkBwdParams q = p;
    if (!(stages & kStageGrad) || (long long)p.B * p.Hv * p.nsplit > sms || groups <= sms) q.ready = nullptr;
    if (stages & kStageDsweep) {
        timing_mark("chunk_dsweep", 0, s);
        err = launch_pdl(chunk_dsweep_kernel<E>, dim3(p.nsplit, p.Hv, p.B), dim3(kSweepThreads), sd, s, q, tm_dv, tm_dy,
                         tm_qk, tm_pk);
        timing_mark("chunk_dsweep", 1, s);
        if (err != cudaSuccess) return err;
    }
    if (!(stages & kStageGrad)) return err;
    timing_mark("chunk_grad", 0, s);
    const int grid = groups < sms ? groups : sms;           // persistent: one CTA per SM
    err = launch_pdl(chunk_grad_kernel<E>, dim3(grid), dim3(256), sg, s, q, groups, tm_dq, tm_dk);
    timing_mark("chunk_grad", 1, s);
    return err;
}

cudaError_t launch_chunk_bwd(const ChunkBwdParams &p, const CUtensorMap &tm_dv, const CUtensorMap &tm_dy,
                             const CUtensorMap &tm_qk, const CUtensorMap &tm_pk, const CUtensorMap &tm_dq,
                             const CUtensorMap &tm_dk, int Dk, cudaStream_t s, int stages) {
    switch (Dk) {
        case 64: return launch_chunk_bwd_t<2>(p, tm_dv, tm_dy, tm_qk, tm_pk, tm_dq, tm_dk, s, stages);
        case 128: return launch_chunk_bwd_t<4>(p, tm_dv, tm_dy, tm_qk, tm_pk, tm_dq, tm_dk, s, stages);
        case 192: return launch_chunk_bwd_t<6>(p, tm_dv, tm_dy, tm_qk, tm_pk, tm_dq, tm_dk, s, stages);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
