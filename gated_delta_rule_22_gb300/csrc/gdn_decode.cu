// gdn_decode.cu -- one step of the gated delta rule (T = 1, the decode step of inference), no
// saved buffer.
//
// The recurrence of mlx issue #4614 ("Recurrence used for the references"), for value head h
// on kv head h / (Hv / Hk):  S <- g S;  S <- S + (beta (v - S k)) k^T;  y = S q.  A step touches
// each row r of S (Dk values) on its own: with a_r = S_r . k and b_r = S_r . q on the incoming
// state,
//     delta_r = beta (v_r - g a_r),   S'_r = g S_r + delta_r k,   y_r = g b_r + delta_r (k . q),
// so the step is one streaming pass over the state: every element read once and written once,
// two dot products per row. The state is fp32; q, k, v, g, beta and y are the input type.
//
// Layout of the work: 16 lanes per state row, lane j holding columns 4 j + 64 m (float4 pieces,
// 16 lanes cover 256 contiguous bytes per m); two rows per half-warp pair, 32 rows per CTA of
// 256 threads, CTAs over (row block, value head, batch row). Loads and stores of the state are
// streamed (read once, written once).
#include "gdn_common.cuh"

namespace gdn {

namespace {

constexpr int kDecodeRows = 32;      // state rows per CTA
constexpr int kDecodeThreads = 256;  // 16 lanes per row, 2 rows per thread

template <typename T>
__device__ __forceinline__ void load4(const T *p, float (&o)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float *p, float (&o)[4]) {
    const float4 x = *reinterpret_cast<const float4 *>(p);
    o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float (&o)[4]) {
    const uint2 x = *reinterpret_cast<const uint2 *>(p);
    o[0] = __uint_as_float(x.x << 16); o[1] = __uint_as_float(x.x & 0xffff0000u);
    o[2] = __uint_as_float(x.y << 16); o[3] = __uint_as_float(x.y & 0xffff0000u);
}

__device__ __forceinline__ float half_sum(float x) {   // over the 16 lanes of a half-warp
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) x += __shfl_xor_sync(kFullMask, x, m);
    return x;
}

}  // namespace

template <int E4, typename TIn>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(FwdParams p) {
    constexpr int DK = 64 * E4;
    constexpr int RPT = kDecodeRows / (kDecodeThreads / 16);   // rows per thread (2)
    const int tid = threadIdx.x, hl = tid & 15, slot = tid >> 4;
    const int h = blockIdx.y, b = blockIdx.z, hk = h / (p.Hv / p.Hk), Dv = p.Dv;
    const size_t head = (size_t)b * p.Hv + h;
    const TIn *q = static_cast<const TIn *>(p.q) + ((size_t)b * p.Hk + hk) * DK;
    const TIn *k = static_cast<const TIn *>(p.k) + ((size_t)b * p.Hk + hk) * DK;
    // the state rows of this thread (rows past Dv: none)
    int row[RPT];
    float s[RPT][E4][4];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        row[r] = blockIdx.x * kDecodeRows + slot + 16 * r;
#pragma unroll
        for (int m = 0; m < E4; ++m) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row[r] < Dv && p.S0 != nullptr)
                x = __ldcs(reinterpret_cast<const float4 *>(p.S0 + (head * Dv + row[r]) * DK + 4 * hl + 64 * m));
            s[r][m][0] = x.x; s[r][m][1] = x.y; s[r][m][2] = x.z; s[r][m][3] = x.w;
        }
    }
    float kk[E4][4], qq[E4][4];
#pragma unroll
    for (int m = 0; m < E4; ++m) {
        load4<TIn>(k + 4 * hl + 64 * m, kk[m]);
        load4<TIn>(q + 4 * hl + 64 * m, qq[m]);
    }
    const TIn *vp = static_cast<const TIn *>(p.v) + head * Dv;
    const float g = to_f32(static_cast<const TIn *>(p.g)[head]), beta = to_f32(static_cast<const TIn *>(p.beta)[head]);
    float v[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) v[r] = row[r] < Dv ? to_f32(vp[row[r]]) : 0.f;
    // k . q and, per row, S k and S q on the incoming state
    float kq = 0.f, a[RPT], bq[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) a[r] = bq[r] = 0.f;
#pragma unroll
    for (int m = 0; m < E4; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            kq = fmaf(kk[m][e], qq[m][e], kq);
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                a[r] = fmaf(s[r][m][e], kk[m][e], a[r]);
                bq[r] = fmaf(s[r][m][e], qq[m][e], bq[r]);
            }
        }
    kq = half_sum(kq);
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        a[r] = half_sum(a[r]);
        bq[r] = half_sum(bq[r]);
    }
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        if (row[r] >= Dv) continue;
        const float delta = beta * (v[r] - g * a[r]);
        if (hl == 0) static_cast<TIn *>(p.y)[head * Dv + row[r]] = from_f32<TIn>(fmaf(g, bq[r], delta * kq));
        if (p.S_T != nullptr)
#pragma unroll
            for (int m = 0; m < E4; ++m)
                __stcs(reinterpret_cast<float4 *>(p.S_T + (head * Dv + row[r]) * DK + 4 * hl + 64 * m),
                       make_float4(fmaf(g, s[r][m][0], delta * kk[m][0]), fmaf(g, s[r][m][1], delta * kk[m][1]),
                                   fmaf(g, s[r][m][2], delta * kk[m][2]), fmaf(g, s[r][m][3], delta * kk[m][3])));
    }
}

template <int E4, typename TIn>
static cudaError_t launch_decode_t(const FwdParams &p, cudaStream_t s) {
    timing_mark("decode", 0, s);
    decode_kernel<E4, TIn><<<dim3((p.Dv + kDecodeRows - 1) / kDecodeRows, p.Hv, p.B), kDecodeThreads, 0, s>>>(p);
    const cudaError_t err = cudaGetLastError();
    timing_mark("decode", 1, s);
    return err;
}

template <typename TIn>
static cudaError_t launch_decode_d(const FwdParams &p, int Dk, cudaStream_t s) {
    switch (Dk) {
        case 64: return launch_decode_t<1, TIn>(p, s);
        case 128: return launch_decode_t<2, TIn>(p, s);
        case 192: return launch_decode_t<3, TIn>(p, s);
        case 256: return launch_decode_t<4, TIn>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

bool decode_takes(int Dk) { return Dk == 64 || Dk == 128 || Dk == 192 || Dk == 256; }

cudaError_t launch_decode(const FwdParams &p, int Dk, int dtype, cudaStream_t s) {
    if (p.T != 1) return cudaErrorInvalidValue;
    return dtype == 0 ? launch_decode_d<float>(p, Dk, s) : launch_decode_d<__nv_bfloat16>(p, Dk, s);
}

}  // namespace gdn
