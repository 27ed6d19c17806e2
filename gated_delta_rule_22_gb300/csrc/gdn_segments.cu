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
// This file holds that scan: fp32 on the CUDA cores, the P - 1 steps of a head in one CTA.
#include "gdn_common.cuh"

namespace gdn {

namespace {

constexpr int kRows = 64;        // state rows per CTA
constexpr int kScanThreads = 256;

}  // namespace

// One CTA per (block of 64 rows, head, batch row). Tensors of the segmented problem are indexed
// by view row b * P + s; X0 (or zero when null) is indexed by b. Shared memory: the running X
// [64][DK] and the map of the step, [DK][DK] (rows of DK + 1 when `reverse`).
template <int E>
__global__ void __launch_bounds__(kScanThreads, 1) segment_scan_kernel(const float *__restrict__ X0,
                                                                       const float *__restrict__ M,
                                                                       const float *__restrict__ C, float *__restrict__ X,
                                                                       int P, int Hv, int rows, int reverse) {
    constexpr int DK = 32 * E;
    constexpr int CW = DK / 16;                 // columns per thread (strided by 16)
    extern __shared__ float smf[];
    float *xs = smf, *ms = smf + kRows * DK;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;   // rows 4 ty .. + 3, columns tx + 16 i
    const int r0 = blockIdx.x * kRows, h = blockIdx.y, b = blockIdx.z;
    auto slab = [&](int s) { return ((size_t)(b * P + s) * Hv + h) * rows + r0; };   // first row of block r0 of view row s
    // the first segment's state (last, in reverse)
    const int s_first = reverse ? P - 1 : 0;
    for (int e = tid; e < kRows * DK; e += kScanThreads) {
        const float x = X0 != nullptr ? X0[((size_t)b * Hv + h) * rows * DK + (size_t)r0 * DK + e] : 0.f;
        xs[e] = x;
        X[slab(s_first) * DK + e] = x;
    }
    for (int i = 1; i < P; ++i) {
        const int sp = reverse ? P - i : i - 1;      // the segment whose map and offset are applied
        const int so = reverse ? P - 1 - i : i;      // the segment whose start (end) this gives
        const float *Mp = M + ((size_t)(b * P + sp) * Hv + h) * DK * DK;
        __syncthreads();                             // the previous step has read ms
        // forward: ms[k][c] = M[k][c]; reverse: ms holds M row by row with a padded stride, so
        // that M^T[k][c] = M[c][k] is read without bank conflicts
        if (reverse) {
            for (int e = tid; e < DK * DK; e += kScanThreads) ms[(e / DK) * (DK + 1) + e % DK] = Mp[e];
        } else {
            for (int e = tid; e < DK * DK; e += kScanThreads) ms[e] = Mp[e];
        }
        __syncthreads();
        float acc[4][CW];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int i2 = 0; i2 < CW; ++i2) acc[r][i2] = 0.f;
        for (int k = 0; k < DK; ++k) {
            float xv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) xv[r] = xs[(4 * ty + r) * DK + k];
#pragma unroll
            for (int i2 = 0; i2 < CW; ++i2) {
                const int c = tx + 16 * i2;
                const float mv = reverse ? ms[c * (DK + 1) + k] : ms[k * DK + c];
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[r][i2] = fmaf(xv[r], mv, acc[r][i2]);
            }
        }
        __syncthreads();                             // every thread has read xs
        const float *Cp = C + slab(sp) * DK;
        float *Xo = X + slab(so) * DK;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int i2 = 0; i2 < CW; ++i2) {
                const int e = (4 * ty + r) * DK + tx + 16 * i2;
                const float x = acc[r][i2] + Cp[e];
                xs[e] = x;
                Xo[e] = x;
            }
    }
}

size_t segment_scan_smem(int Dk) { return (size_t)(kRows * Dk + Dk * (Dk + 1)) * sizeof(float); }

template <int E>
static cudaError_t launch_scan_t(const float *X0, const float *M, const float *C, float *X, int B, int P, int Hv,
                                 int rows, bool reverse, cudaStream_t s) {
    constexpr int DK = 32 * E;
    const size_t smem = segment_scan_smem(DK);
    cudaError_t err = cudaFuncSetAttribute(segment_scan_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    timing_mark("segment_scan", 0, s);
    segment_scan_kernel<E><<<dim3(rows / kRows, Hv, B), kScanThreads, smem, s>>>(X0, M, C, X, P, Hv, rows, reverse ? 1 : 0);
    err = cudaGetLastError();
    timing_mark("segment_scan", 1, s);
    return err;
}

cudaError_t launch_segment_scan(const float *X0, const float *M, const float *C, float *X, int B, int P, int Hv,
                                int rows, int Dk, bool reverse, cudaStream_t s) {
    if (rows % kRows != 0) return cudaErrorInvalidValue;
    switch (Dk) {
        case 64: return launch_scan_t<2>(X0, M, C, X, B, P, Hv, rows, reverse, s);
        case 128: return launch_scan_t<4>(X0, M, C, X, B, P, Hv, rows, reverse, s);
        case 192: return launch_scan_t<6>(X0, M, C, X, B, P, Hv, rows, reverse, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
