// gdn_segments.cu -- the scan over segments of chunks of the sequence-parallel form.
//
// The recurrence is that of mlx issue #4614 ("Recurrence used for the references"). Across one
// chunk the state map is affine, S -> S M_c + C_c (the chunkwise forward writes it out: see
// gdn_chunk.cu), so across a segment of chunks it is S -> S M + C, where M is the product of the
// chunks' maps (the maps sweep) and C the segment's end state from a zero start (the ordinary
// sweep with S0 = 0). The segments' start states then follow from one short scan per head,
//     X_0 = S0,   X_s = X_{s-1} M_{s-1} + C_{s-1},
// and the backward's end adjoints from the reverse scan with the transposed maps,
//     Y_{P-1} = dS_T,   Y_s = Y_{s+1} M_{s+1}^T + D_{s+1},
// D_s being segment s's start adjoint from a zero end adjoint (the reverse sweep with dS_T = 0).
// This file holds that scan: fp32 on the CUDA cores, the P - 1 steps of a block of state rows in
// one CTA.
#include "gdn_common.cuh"

namespace gdn {

namespace {

// The layout of a CTA of R state rows: warps of 8 rows x all DK columns (lane l: columns
// 2 l + 64 j), KS warps per 8 rows, each over one KS-th of the k range (their partial products
// summed through shared memory when KS > 1).
__host__ __device__ constexpr int scan_ks(int R) { return R <= 16 ? 4 : (R == 32 ? 2 : 1); }
__host__ __device__ constexpr int scan_threads(int R) { return 32 * (R / 8) * scan_ks(R); }

// Shared memory: two mbarriers, X of the block [R][DK + 4], the partial products [KS][R][DK]
// (KS > 1), then `nbuf` maps [DK][DK].
constexpr size_t scan_smem(int R, int Dk, int nbuf) {
    return 16 + (size_t)(R * (Dk + 4) + (scan_ks(R) > 1 ? scan_ks(R) * R * Dk : 0) + nbuf * Dk * Dk) * sizeof(float);
}

}  // namespace

// One CTA per (block of R state rows, head, batch row). Tensors of the segmented problem are
// indexed by view row b * P + s; X0 (zero when null) by b. The maps of the steps arrive by 1-D
// bulk copies (each map is contiguous); with two buffers the next step's map is in flight while
// this step multiplies. `Mt` is the array read: the maps, or for the reverse scan their
// transposes (written beside them by the lite sweep), so both directions run the same product
// X M with M read row by row. Per k, a warp reads one float4 of X per 4 k (the same address in
// every lane) and a row of M in float2s (distinct, contiguous): 8 x 2 multiply-adds per lane per
// element pair read.
template <int E, int R>
__global__ void __launch_bounds__(scan_threads(R), 1) segment_scan_kernel(const float *__restrict__ X0,
                                                                          const float *__restrict__ Mt,
                                                                          const float *__restrict__ C, float *__restrict__ X,
                                                                          int P, int Hv, int rows, int nbuf, int reverse,
                                                                          int *status) {
    constexpr int DK = 32 * E;
    constexpr int KS = scan_ks(R);              // k splits
    constexpr int NT = scan_threads(R);
    constexpr int C2 = DK / 64;                 // float2 column groups per lane
    constexpr int XS = DK + 4;                  // row stride of X in shared memory (16-byte rows)
    constexpr int KR = DK / KS;                 // k range of a warp
    constexpr int F4 = R * DK / 4 / NT;         // float4s of the block per thread (the sums)
    static_assert(KR % 4 == 0 && (R * DK / 4) % NT == 0, "scan layout");
    extern __shared__ __align__(16) unsigned char smraw[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smraw);
    float *xs = reinterpret_cast<float *>(smraw + 16);
    float *red = xs + R * XS;
    float *ms = red + (KS > 1 ? KS * R * DK : 0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = warp / KS, ks = warp % KS;   // rows 8 rg .. 8 rg + 7, k in [ks KR, ks KR + KR)
    const int r0 = blockIdx.x * R, h = blockIdx.y, b = blockIdx.z;
    auto slab = [&](int s) { return ((size_t)(b * P + s) * Hv + h) * rows + r0; };   // row r0 of view row s
    auto sp_of = [&](int i) { return reverse ? P - i : i - 1; };   // step i applies segment sp's map and offset
    auto so_of = [&](int i) { return reverse ? P - 1 - i : i; };   // ... and gives segment so's start (end)
    constexpr unsigned kMapBytes = DK * DK * sizeof(float);
    auto fetch = [&](int i) {                   // step i's map into buffer (i - 1) % nbuf
        uint64_t *bb = bar + (i - 1) % nbuf;
        const float *src = Mt + ((size_t)(b * P + sp_of(i)) * Hv + h) * DK * DK;
        float *dst = ms + (size_t)((i - 1) % nbuf) * DK * DK;
        mbar_expect_tx(bb, kMapBytes);
#pragma unroll
        for (int q = 0; q < 4; ++q) bulk_load(dst + q * (DK * DK / 4), src + q * (DK * DK / 4), kMapBytes / 4, bb);
    };
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);
        fence_mbar_init();
    }
    __syncthreads();
    int issued = 0;                             // steps whose map was fetched (thread 0)
    if (tid == 0)
        for (; issued < nbuf && issued < P - 1; ++issued) fetch(issued + 1);
    // the first segment's state (the last, in reverse)
    {
        const size_t o0 = ((size_t)b * Hv + h) * rows * DK + (size_t)r0 * DK;
        float *Xf = X + slab(reverse ? P - 1 : 0) * DK;
        for (int e = 4 * tid; e < R * DK; e += 4 * NT) {
            const float4 x = X0 != nullptr ? *reinterpret_cast<const float4 *>(X0 + o0 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(xs + (e / DK) * XS + e % DK) = x;
            *reinterpret_cast<float4 *>(Xf + e) = x;
        }
    }
    bool fail = false;
    for (int i = 1; i < P; ++i) {
        // this step's offset, fetched before the wait: with KS > 1 thread t sums float4s
        // t + NT f of the block; with KS = 1 each lane adds it to its own outputs
        const float *Cp = C + slab(sp_of(i)) * DK;
        float4 cv[KS > 1 ? F4 : 1];
        float2 cl[KS > 1 ? 1 : 8][C2];
        if constexpr (KS > 1) {
#pragma unroll
            for (int f = 0; f < F4; ++f) cv[f] = *reinterpret_cast<const float4 *>(Cp + 4 * (tid + NT * f));
        } else {
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int j = 0; j < C2; ++j)
                    cl[r][j] = *reinterpret_cast<const float2 *>(Cp + (8 * rg + r) * DK + 2 * lane + 64 * j);
        }
        // the map has landed (every thread's wait, one verdict for the CTA); xs is written
        const bool ok = mbar_wait(bar + (i - 1) % nbuf, ((i - 1) / nbuf) & 1);
        if (__syncthreads_or(!ok)) { fail = true; break; }
        const float *mb = ms + (size_t)((i - 1) % nbuf) * DK * DK;
        float2 acc[8][C2];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int j = 0; j < C2; ++j) acc[r][j] = make_float2(0.f, 0.f);
#pragma unroll 2
        for (int k = ks * KR; k < ks * KR + KR; k += 4) {
            float4 xq[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) xq[r] = *reinterpret_cast<const float4 *>(xs + (8 * rg + r) * XS + k);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                for (int j = 0; j < C2; ++j) {
                    const float2 m = *reinterpret_cast<const float2 *>(mb + (k + kk) * DK + 2 * lane + 64 * j);
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const float xv = kk == 0 ? xq[r].x : kk == 1 ? xq[r].y : kk == 2 ? xq[r].z : xq[r].w;
                        acc[r][j].x = fmaf(xv, m.x, acc[r][j].x);
                        acc[r][j].y = fmaf(xv, m.y, acc[r][j].y);
                    }
                }
            }
        }
        float *Xo = X + slab(so_of(i)) * DK;
        if constexpr (KS > 1) {
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int j = 0; j < C2; ++j)
                    *reinterpret_cast<float2 *>(red + (ks * R + 8 * rg + r) * DK + 2 * lane + 64 * j) = acc[r][j];
            __syncthreads();                    // every partial is written; xs and the map are read
            if (tid == 0 && issued < P - 1) fetch(++issued);
#pragma unroll
            for (int f = 0; f < F4; ++f) {
                const int e = 4 * (tid + NT * f);
                float4 x = cv[f];
#pragma unroll
                for (int q = 0; q < KS; ++q) {
                    const float4 pq = *reinterpret_cast<const float4 *>(red + q * R * DK + e);
                    x.x += pq.x;
                    x.y += pq.y;
                    x.z += pq.z;
                    x.w += pq.w;
                }
                *reinterpret_cast<float4 *>(xs + (e / DK) * XS + e % DK) = x;
                *reinterpret_cast<float4 *>(Xo + e) = x;
            }
        } else {
            __syncthreads();                    // xs and the map are read
            if (tid == 0 && issued < P - 1) fetch(++issued);
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int j = 0; j < C2; ++j) {
                    const int row = 8 * rg + r, col = 2 * lane + 64 * j;
                    const float2 x = make_float2(acc[r][j].x + cl[r][j].x, acc[r][j].y + cl[r][j].y);
                    *reinterpret_cast<float2 *>(xs + row * XS + col) = x;
                    *reinterpret_cast<float2 *>(Xo + row * DK + col) = x;
                }
        }
    }
    if (fail) {
        if (tid == 0) {
            report_status(status, kStatusTimeout);
            // copies still in flight land before the CTA exits (bounded waits)
            for (int i = issued > nbuf ? issued - nbuf + 1 : 1; i <= issued; ++i)
                mbar_wait(bar + (i - 1) % nbuf, ((i - 1) / nbuf) & 1);
        }
    }
}

template <int E, int R>
static cudaError_t launch_scan_r(const float *X0, const float *M, const float *C, float *X, int B, int P, int Hv,
                                 int rows, bool reverse, int *status, cudaStream_t s) {
    constexpr int DK = 32 * E;
    constexpr int NT = scan_threads(R);
    // two map buffers where they fit in shared memory
    const int nbuf = scan_smem(R, DK, 2) <= 227 * 1024 ? 2 : 1;
    const size_t smem = scan_smem(R, DK, nbuf);
    cudaError_t err = cudaFuncSetAttribute(segment_scan_kernel<E, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    timing_mark("segment_scan", 0, s);
    segment_scan_kernel<E, R><<<dim3(rows / R, Hv, B), NT, smem, s>>>(X0, M, C, X, P, Hv, rows, nbuf, reverse ? 1 : 0,
                                                                       status);
    err = cudaGetLastError();
    timing_mark("segment_scan", 1, s);
    return err;
}

template <int E>
static cudaError_t launch_scan_t(const float *X0, const float *M, const float *C, float *X, int B, int P, int Hv,
                                 int rows, bool reverse, int *status, cudaStream_t s) {
    // rows per CTA: the largest of 64, 32, 16, 8 that still gives every SM a CTA (the steps are
    // a dependent chain: more, smaller CTAs shorten it)
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    int R = 64;
    while (R > 8 && (long long)(rows / R) * Hv * B < sms) R /= 2;
    switch (R) {
        case 64: return launch_scan_r<E, 64>(X0, M, C, X, B, P, Hv, rows, reverse, status, s);
        case 32: return launch_scan_r<E, 32>(X0, M, C, X, B, P, Hv, rows, reverse, status, s);
        case 16: return launch_scan_r<E, 16>(X0, M, C, X, B, P, Hv, rows, reverse, status, s);
        default: return launch_scan_r<E, 8>(X0, M, C, X, B, P, Hv, rows, reverse, status, s);
    }
}

cudaError_t launch_segment_scan(const float *X0, const float *M, const float *C, float *X, int B, int P, int Hv,
                                int rows, int Dk, bool reverse, int *status, cudaStream_t s) {
    if (rows % 64 != 0 || P < 1) return cudaErrorInvalidValue;
    switch (Dk) {
        case 64: return launch_scan_t<2>(X0, M, C, X, B, P, Hv, rows, reverse, status, s);
        case 128: return launch_scan_t<4>(X0, M, C, X, B, P, Hv, rows, reverse, status, s);
        case 192: return launch_scan_t<6>(X0, M, C, X, B, P, Hv, rows, reverse, status, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
