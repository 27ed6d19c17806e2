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

constexpr int kMaxScanThreads = 256;

// Shared memory: two mbarriers, X of the block [R][DK + 4] (the padding puts a thread's rows and
// its neighbour's in different banks), then `nbuf` maps [DK][DK].
constexpr size_t scan_smem(int R, int Dk, int nbuf) {
    return 16 + (size_t)(R * (Dk + 4) + nbuf * Dk * Dk) * sizeof(float);
}

}  // namespace

// One CTA per (block of R state rows, head, batch row); 16 x (R / RPT) threads, thread (tx, ty)
// holding rows ty * RPT .. + RPT - 1 of the block and columns 4 tx + 64 i + (0 .. 3). Tensors of
// the segmented problem are indexed by view row b * P + s; X0 (zero when null) by b. The maps of
// the steps arrive by 1-D bulk copies (each map is contiguous); with two buffers the next step's
// map is in flight while this step multiplies. `Mt` is the array read: the maps, or for the
// reverse scan their transposes (written beside them by the maps sweep), so both directions run
// the same product X M with M read row by row.
template <int E, int R>
__global__ void __launch_bounds__(kMaxScanThreads, 1) segment_scan_kernel(const float *__restrict__ X0,
                                                                          const float *__restrict__ Mt,
                                                                          const float *__restrict__ C, float *__restrict__ X,
                                                                          int P, int Hv, int rows, int nbuf, int reverse,
                                                                          int *status) {
    constexpr int DK = 32 * E;
    constexpr int RPT = R <= 16 ? 1 : R / 16;   // rows per thread
    constexpr int NT = 16 * (R / RPT);          // threads
    constexpr int C4 = DK / 64;                 // float4 column groups per thread
    constexpr int XS = DK + 4;                  // row stride of X in shared memory
    extern __shared__ __align__(16) unsigned char smraw[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smraw);
    float *xs = reinterpret_cast<float *>(smraw + 16), *ms = xs + R * XS;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
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
        // this step's offset, fetched before the wait
        const float *Cp = C + slab(sp_of(i)) * DK;
        float4 cv[RPT][C4];
#pragma unroll
        for (int r = 0; r < RPT; ++r)
#pragma unroll
            for (int j = 0; j < C4; ++j)
                cv[r][j] = *reinterpret_cast<const float4 *>(Cp + (ty * RPT + r) * DK + 4 * tx + 64 * j);
        // the map has landed (every thread's wait, one verdict for the CTA); xs is written
        const bool ok = mbar_wait(bar + (i - 1) % nbuf, ((i - 1) / nbuf) & 1);
        if (__syncthreads_or(!ok)) { fail = true; break; }
        const float *mb = ms + (size_t)((i - 1) % nbuf) * DK * DK;
        float4 acc[RPT][C4];
#pragma unroll
        for (int r = 0; r < RPT; ++r)
#pragma unroll
            for (int j = 0; j < C4; ++j) acc[r][j] = cv[r][j];
#pragma unroll 4
        for (int k = 0; k < DK; ++k) {
            float xv[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) xv[r] = xs[(ty * RPT + r) * XS + k];
#pragma unroll
            for (int j = 0; j < C4; ++j) {
                const float4 m = *reinterpret_cast<const float4 *>(mb + k * DK + 4 * tx + 64 * j);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    acc[r][j].x = fmaf(xv[r], m.x, acc[r][j].x);
                    acc[r][j].y = fmaf(xv[r], m.y, acc[r][j].y);
                    acc[r][j].z = fmaf(xv[r], m.z, acc[r][j].z);
                    acc[r][j].w = fmaf(xv[r], m.w, acc[r][j].w);
                }
            }
        }
        __syncthreads();                        // every thread is done with xs and this map's buffer
        if (tid == 0 && issued < P - 1) fetch(++issued);
        float *Xo = X + slab(so_of(i)) * DK;
#pragma unroll
        for (int r = 0; r < RPT; ++r)
#pragma unroll
            for (int j = 0; j < C4; ++j) {
                const int row = ty * RPT + r, col = 4 * tx + 64 * j;
                *reinterpret_cast<float4 *>(xs + row * XS + col) = acc[r][j];
                *reinterpret_cast<float4 *>(Xo + row * DK + col) = acc[r][j];
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
    constexpr int NT = 16 * (R / (R <= 16 ? 1 : R / 16));
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
