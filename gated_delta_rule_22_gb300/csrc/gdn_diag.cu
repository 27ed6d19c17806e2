// gdn_diag.cu -- diagnostics of the library (no counterpart on the pages): the timeout path of
// the bounded device-side waits, and the FP32 FMA rate that bounds the sequential kernels.
#include "gdn_common.cuh"

namespace gdn {

namespace {

// One CTA that takes the steps every kernel of the library takes around a bounded wait: it
// allocates tensor memory, arms an mbarrier for 16 bytes that no copy will ever deliver (so no
// copy is in flight at any point), waits for it at most `polls` polls, and on the timeout
// records kStatusTimeout in the status word, then frees its tensor memory and exits as a
// timed-out kernel does.
__global__ void __launch_bounds__(128, 1) wait_probe_kernel(int *status, unsigned polls) {
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_expect_tx(&bar, 16);       // the one arrival, with 16 bytes still owed
    }
    if (warp == 0) tmem_alloc(&tslot, 32);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    const bool ok = !__syncthreads_or(tid == 0 && !mbar_wait(&bar, 0, polls));
    if (!ok && tid == 0) report_status(status, kStatusTimeout);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 32);
}

// FP32 FMA rate: every thread runs 8 independent chains x <- x * a + b (a, b shared by all
// chains, so that only x is a distinct register operand) for `iters` rounds; scalar FFMA or
// the packed f32x2 form that the sequential kernels use. 2 flops per FMA and lane.
__device__ float g_fma_sink;   // written only if the chains reach a value they cannot reach

template <bool kPacked>
__global__ void __launch_bounds__(256) fma_rate_kernel(int iters, float a, float b) {
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (float)(threadIdx.x + i);
    if (kPacked) {
        const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                float2 v = make_float2(x[i], x[i + 1]);
                v = __ffma2_rn(v, a2, b2);
                x[i] = v.x;
                x[i + 1] = v.y;
            }
        }
    } else {
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = fmaf(x[i], a, b);
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += x[i];
    if (s == 1234.5f) g_fma_sink = s;   // never true: the chains converge to 1 (x -> 0.999 x + 0.001)
}

}  // namespace

cudaError_t launch_wait_probe(int *status, unsigned polls, cudaStream_t s) {
    wait_probe_kernel<<<1, 128, 0, s>>>(status, polls);
    return cudaGetLastError();
}

cudaError_t measure_fma_rate(int packed, double *tflops) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int blocks = sms * 8, threads = 256, iters = 1 << 14;
    cudaStream_t st = nullptr;
    cudaEvent_t t0 = nullptr, t1 = nullptr;
    e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreate(&t0);
    if (e == cudaSuccess) e = cudaEventCreate(&t1);
    float best = 1e30f;
    for (int rep = 0; rep < 4 && e == cudaSuccess; ++rep) {   // the first is a warm-up
        e = cudaEventRecord(t0, st);
        if (packed)
            fma_rate_kernel<true><<<blocks, threads, 0, st>>>(iters, 0.999f, 0.001f);
        else
            fma_rate_kernel<false><<<blocks, threads, 0, st>>>(iters, 0.999f, 0.001f);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e == cudaSuccess) e = cudaEventRecord(t1, st);
        if (e == cudaSuccess) e = cudaEventSynchronize(t1);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t0, t1);
        if (e == cudaSuccess && rep > 0 && ms < best) best = ms;
    }
    if (t0) cudaEventDestroy(t0);
    if (t1) cudaEventDestroy(t1);
    if (st) cudaStreamDestroy(st);
    if (e != cudaSuccess) return e;
    const double flops = 2.0 * 16.0 * iters * (double)blocks * threads;
    *tflops = flops / (best * 1e-3) / 1e12;
    return cudaSuccess;
}

}  // namespace gdn
