// gdn_gates.cu -- the decay g and write strength beta from the layer's raw gate inputs,
// and the VJP back to them.
//
// mlx-lm PR #1217 ("Correctness") trains through eight inputs: q, k, v, a, b, A_log,
// dt_bias and the state. The pages do not print how g and beta follow from a, b, A_log and
// dt_bias; the map taken is the public mlx-lm Qwen3-Next / Qwen3.5 linear-attention
// layer's, per batch row, step and value head h:
//     log g = -exp(A_log[h]) * softplus(a + dt_bias[h]),   g = exp(log g)
//     beta  = sigmoid(b)
// The VJP goes through log g, as mlx issue #4614 says a log_g parameterisation trains:
//     d(log g) = g dg,  da = -exp(A_log) sigmoid(a + dt_bias) d(log g),
//     ddt_bias[h] = sum over rows of da,  dA_log[h] = sum over rows of log g d(log g),
//     db = dbeta beta (1 - beta).
// Arithmetic is fp32 (the parameter sums in fp64), elementwise and memory-bound.
#include "gdn_common.cuh"

#include <cooperative_groups.h>

namespace cg = cooperative_groups;

namespace gdn {

namespace {

__device__ __forceinline__ float softplus_f(float x) {
    return x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}

__device__ __forceinline__ float sigmoid_f(float x) {
    if (x >= 0.f) return 1.f / (1.f + expf(-x));
    const float e = expf(x);
    return e / (1.f + e);
}

}  // namespace

template <typename T>
__global__ void __launch_bounds__(256) gates_fwd_kernel(GatesParams p) {
    const T *a = static_cast<const T *>(p.a);
    const T *b = static_cast<const T *>(p.b);
    T *g = static_cast<T *>(p.g);
    T *beta = static_cast<T *>(p.beta);
    const size_t n = (size_t)p.rows * p.Hv;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int h = (int)(i % p.Hv);
        const float log_g = -expf(p.A_log[h]) * softplus_f(to_f32(a[i]) + p.dt_bias[h]);
        g[i] = from_f32<T>(expf(log_g));
        beta[i] = from_f32<T>(sigmoid_f(to_f32(b[i])));
    }
}

// A cluster of kGateSplit CTAs per group of 32 value heads (lane = head): CTA y of the cluster
// and warp w walk rows y * 32 + w, then every kGateSplit * 32 rows further (a fixed interleaved
// order). The per-head parameter sums are added over a CTA's warps in ascending order, then
// over the cluster's CTAs in ascending order by its first CTA, which reads the others' partials
// from their shared memory: the result does not depend on scheduling.
constexpr int kGateSplit = 8;

template <typename T>
__global__ void __cluster_dims__(1, kGateSplit, 1) __launch_bounds__(1024) gates_bwd_kernel(GatesParams p) {
    __shared__ double part[2][32][33];
    __shared__ double cta_sum[2][32];
    const T *a = static_cast<const T *>(p.a);
    const T *b = static_cast<const T *>(p.b);
    const T *dg = static_cast<const T *>(p.dg);
    const T *dbeta = static_cast<const T *>(p.dbeta);
    T *da = static_cast<T *>(p.da);
    T *db = static_cast<T *>(p.db);
    cg::cluster_group cluster = cg::this_cluster();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int h = blockIdx.x * 32 + lane;
    const size_t stride = (size_t)gridDim.y * nw;
    double sA = 0.0, sdt = 0.0;
    if (h < p.Hv) {
        const float A = expf(p.A_log[h]), dt = p.dt_bias[h];
        for (size_t r = (size_t)blockIdx.y * nw + warp; r < (size_t)p.rows; r += stride) {
            const size_t i = r * p.Hv + h;
            const float x = to_f32(a[i]) + dt;
            const float log_g = -A * softplus_f(x);
            const float dlog_g = expf(log_g) * to_f32(dg[i]);
            const float dx = dlog_g * (-A) * sigmoid_f(x);
            da[i] = from_f32<T>(dx);
            sdt += (double)dx;
            sA += (double)dlog_g * (double)log_g;
            const float bt = sigmoid_f(to_f32(b[i]));
            db[i] = from_f32<T>(to_f32(dbeta[i]) * bt * (1.f - bt));
        }
    }
    part[0][warp][lane] = sA;
    part[1][warp][lane] = sdt;
    __syncthreads();
    if (warp == 0) {
        double tA = 0.0, tdt = 0.0;
        for (int w = 0; w < nw; ++w) {
            tA += part[0][w][lane];
            tdt += part[1][w][lane];
        }
        cta_sum[0][lane] = tA;
        cta_sum[1][lane] = tdt;
    }
    cluster.sync();                      // every CTA's sums are in its shared memory
    if (cluster.block_rank() == 0 && warp == 0 && h < p.Hv) {
        double tA = 0.0, tdt = 0.0;
        for (unsigned r = 0; r < cluster.num_blocks(); ++r) {
            const double *o = cluster.map_shared_rank(&cta_sum[0][0], r);
            tA += o[lane];
            tdt += o[32 + lane];
        }
        p.dA_log[h] = (float)tA;
        p.ddt_bias[h] = (float)tdt;
    }
    cluster.sync();                      // no CTA leaves while the first still reads its sums
}

cudaError_t launch_gates_fwd(const GatesParams &p, int dtype, cudaStream_t s) {
    const size_t n = (size_t)p.rows * p.Hv;
    const size_t want = (n + 255) / 256;
    const int blocks = (int)(want < 152 * 8 ? want : 152 * 8);
    timing_mark("gates_fwd", 0, s);
    if (dtype == 0) gates_fwd_kernel<float><<<blocks, 256, 0, s>>>(p);
    else gates_fwd_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(p);
    timing_mark("gates_fwd", 1, s);
    return cudaGetLastError();
}

cudaError_t launch_gates_bwd(const GatesParams &p, int dtype, cudaStream_t s) {
    const dim3 grid((p.Hv + 31) / 32, kGateSplit);          // one cluster per 32 value heads
    timing_mark("gates_bwd", 0, s);
    if (dtype == 0) gates_bwd_kernel<float><<<grid, 1024, 0, s>>>(p);
    else gates_bwd_kernel<__nv_bfloat16><<<grid, 1024, 0, s>>>(p);
    timing_mark("gates_bwd", 1, s);
    return cudaGetLastError();
}

}  // namespace gdn
