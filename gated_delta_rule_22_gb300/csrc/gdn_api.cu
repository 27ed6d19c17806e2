// gdn_api.cu -- the C ABI declared in include/gdn.h: argument checks (all on the host,
// before anything is enqueued), scratch layout, and dispatch to the kernels.
#include "gdn.h"
#include "gdn_common.cuh"

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <vector>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

namespace {

thread_local char g_last_error[256] = "";

struct Plan {
    int B, T, Hk, Hv, Dk, Dv, C, NC, dtype;
    int warps;     // forward warps per CTA
    int RB;        // backward: rows of a state per CTA
    int nsplit;    // backward: CTAs per (b, h)
    int sub;       // backward sub-block length
    int nsub_max;  // sub-blocks per chunk
    int slots;     // backward partial-sum ring depth (steps)
    bool tc;       // forward in the chunkwise tensor-core form (bf16, C = 64, supported sizes)
    bool tcb;      // backward in the chunkwise form too (its shared memory fits)
};

constexpr size_t kMaxSmem = 232448;   // opt-in shared memory per block on sm_103

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int make_plan(const gdn_shape *s, Plan *p) {
    if (s == nullptr) return GDN_ERR_INVALID_ARG;
    if (s->B <= 0 || s->T <= 0 || s->Hk <= 0 || s->Hv <= 0 || s->Dk <= 0 || s->Dv <= 0 || s->chunk < 0)
        return GDN_ERR_INVALID_ARG;
    if (s->dtype != GDN_F32 && s->dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (s->Hv % s->Hk != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (s->Dk % 32 != 0 || s->Dk > 256) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (s->Dv % 4 != 0 || s->Dv > gdn::kMaxDv) return GDN_ERR_UNSUPPORTED_SHAPE;
    const int C = s->chunk == 0 ? 64 : s->chunk;
    if (C > gdn::kMaxChunk) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (s->Hv > 65535 || s->B > 65535) return GDN_ERR_UNSUPPORTED_SHAPE;
    // every tensor and scratch region must be indexable with 62-bit offsets
    const double rows = (double)s->B * s->Hv * s->Dv;
    const double big = (double)s->T * rows * (s->Dk + 8.0) * 8.0;
    if (big > 4.0e18) return GDN_ERR_UNSUPPORTED_SHAPE;
    p->B = s->B; p->T = s->T; p->Hk = s->Hk; p->Hv = s->Hv; p->Dk = s->Dk; p->Dv = s->Dv;
    p->C = C;
    p->NC = (s->T + C - 1) / C;
    p->dtype = s->dtype;
    int warps = (s->Dv + gdn::kRowsPerWarp - 1) / gdn::kRowsPerWarp;
    if (warps > 8) warps = 8;
    p->warps = warps;
    p->RB = gdn::kBwdRows;
    p->nsplit = (s->Dv + p->RB - 1) / p->RB;
    p->sub = gdn::bwd_sub(s->Dk);
    p->nsub_max = (C + p->sub - 1) / p->sub;
    p->slots = gdn::bwd_slots(s->Dk, C, s->dtype, kMaxSmem);
    if (p->slots == 0) return GDN_ERR_UNSUPPORTED_SHAPE;
    p->tc = s->dtype == GDN_BF16 && C == 64 && (s->Dk == 64 || s->Dk == 128 || s->Dk == 192) &&
            s->Dv % 64 == 0 && s->Dv <= 256 && gdn::chunk_prep_smem(s->Dk, s->Dv) <= kMaxSmem &&
            gdn::chunk_sweep_smem(s->Dk) <= kMaxSmem;
    p->tcb = p->tc && gdn::chunk_dsweep_smem(s->Dk) <= kMaxSmem && gdn::chunk_grad_smem(s->Dk, s->Dv) <= kMaxSmem;
    return GDN_OK;
}

// The saved-for-backward buffer `ckpt`: the chunk-start states [B,Hv,NC,Dv,Dk], then (from a
// 256-byte boundary) the residuals v_t - u_t [B,T,Hv,Dv], all fp32.
size_t ckpt_state_bytes(const Plan &p) { return round_up((size_t)p.B * p.Hv * p.NC * p.Dv * p.Dk * sizeof(float)); }
size_t ckpt_resid_bytes(const Plan &p) { return (size_t)p.B * p.T * p.Hv * p.Dv * sizeof(float); }

// With the chunkwise forward the buffer continues (each part from a 256-byte boundary) with
// the per-chunk data of every (b, h, chunk): Lam [64] fp32 and bf16 matrices in their
// core-matrix layout ([(Q K^T) o E; (K K^T) o E] [128][64], -W [64][Dk], T [64][64],
// T diag(beta) [64][64], the bf16 chunk-start state [Dv][Dk]), and per (b, kv head, chunk)
// [Q; K] [128][Dk].
struct ChunkLayout {
    size_t lam, pkm, wm, tm, tcm, s0m, qkm, end;
};
ChunkLayout chunk_layout(const Plan &p) {
    const size_t n = (size_t)p.B * p.Hv * p.NC * 64;   // chunk rows
    ChunkLayout c;
    size_t o = ckpt_state_bytes(p) + round_up(ckpt_resid_bytes(p));
    c.lam = o; o += round_up(n * 4);
    c.pkm = o; o += round_up(n * 2 * 64 * 2);
    c.wm = o; o += round_up(n * p.Dk * 2);
    c.tm = o; o += round_up(n * 64 * 2);
    c.tcm = o; o += round_up(n * 64 * 2);
    c.s0m = o; o += round_up((size_t)p.B * p.Hv * p.NC * p.Dv * p.Dk * 2);
    c.qkm = o; o += round_up((size_t)p.B * p.Hk * p.NC * 128 * p.Dk * 2);
    c.end = o;
    return c;
}

struct Workspace {
    size_t dq, dk, dg, db, state, total;  // byte offsets and total
};

Workspace workspace_layout(const Plan &p) {
    Workspace w;
    const size_t nqk = (size_t)p.B * p.T * p.Hv * p.nsplit * p.Dk;
    const size_t ngate = (size_t)p.B * p.T * p.Hv * p.nsplit;
    const size_t nstate = (size_t)p.B * p.Hv * p.nsplit * p.nsub_max * p.RB * gdn::bwd_pairs(p.Dk) * 64;
    size_t off = 0;
    w.dq = off; off += round_up(nqk * 4);
    w.dk = off; off += round_up(nqk * 4);
    w.dg = off; off += round_up(ngate * 4);
    w.db = off; off += round_up(ngate * 4);
    w.state = off; off += round_up(nstate * 4);
    w.total = off;
    return w;
}

// Scratch of the chunkwise backward: dbeta and f partials per 32 value rows
// [B,T,Hv,nsplit,2] fp32; [dY; dU] [B,Hv,NC,nsplit][128 x 64], Delta [B,Hv,NC,nsplit][64 x 64] and
// dS at each chunk end [B,Hv,NC,nsplit][64 x Dk], bf16 in their operand layout. (dq, dk are
// summed over value heads in the gradient kernel's tensor memory and need no scratch.)
struct TcWorkspace {
    size_t db, f, yu, dl, dsl, sync, total;
};

TcWorkspace tc_workspace_layout(const Plan &p) {
    TcWorkspace w;
    const size_t ngate = (size_t)p.B * p.T * p.Hv * p.nsplit * 2;   // a partial per 32 value rows
    const size_t nblk = (size_t)p.B * p.Hv * p.NC * p.nsplit;
    size_t off = 0;
    w.db = off; off += round_up(ngate * 4);
    w.f = off; off += round_up(ngate * 4);
    w.yu = off; off += round_up(nblk * 128 * 64 * 2);
    w.dl = off; off += round_up(nblk * 64 * 64 * 2);
    w.dsl = off; off += round_up(nblk * 64 * p.Dk * 2);
    w.sync = off; off += round_up(((size_t)p.B * p.Hv * p.NC + 1) * 4);   // ready counters, group counter
    w.total = off;
    return w;
}

size_t ckpt_total(const Plan &p) { return p.tc ? chunk_layout(p).end : ckpt_state_bytes(p) + ckpt_resid_bytes(p); }

// The chunkwise form's per-chunk products (Lam onwards) of a saved buffer, and their size.
char *chunk_products(const Plan &p, const float *ckpt) {
    return const_cast<char *>(reinterpret_cast<const char *>(ckpt)) + chunk_layout(p).lam;
}
size_t chunk_products_bytes(const Plan &p) {
    const ChunkLayout cl = chunk_layout(p);
    return cl.end - cl.lam;
}

size_t bwd_workspace_total(const Plan &p) { return p.tcb ? tc_workspace_layout(p).total : workspace_layout(p).total; }

bool aligned(const void *ptr) { return ((uintptr_t)ptr & 15u) == 0; }

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GDN_OK;
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return GDN_ERR_CUDA;
}

// ---- per-device status word: kernels record GDN_ERR_TIMEOUT there when a bounded wait
// runs out. Its device address is looked up once per device.
static __device__ int g_device_status;
constexpr int kMaxDevs = 256;
std::mutex g_status_mutex;
int *g_status_addr[kMaxDevs];

int device_status_address(int **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevs) return cuda_status(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (g_status_addr[dev] == nullptr) {
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_device_status);
        if (e != cudaSuccess) return cuda_status(e);
        g_status_addr[dev] = static_cast<int *>(addr);
    }
    *out = g_status_addr[dev];
    return GDN_OK;
}

// ---- TMA tensor maps of q and k: 4-D [B, T, Hk, Dk], box {Dk, 1, box_t, 1}
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

int make_qk_map(CUtensorMap *map, const void *ptr, const Plan &p, int box_t) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled is not available from the driver");
        return GDN_ERR_CUDA;
    }
    const cuuint64_t e = p.dtype == GDN_F32 ? 4 : 2;
    const cuuint64_t dims[4] = {(cuuint64_t)p.Dk, (cuuint64_t)p.Hk, (cuuint64_t)p.T, (cuuint64_t)p.B};
    const cuuint64_t strides[3] = {p.Dk * e, (cuuint64_t)p.Hk * p.Dk * e, (cuuint64_t)p.T * p.Hk * p.Dk * e};
    const cuuint32_t box[4] = {(cuuint32_t)p.Dk, 1, (cuuint32_t)box_t, 1};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    const CUresult r = enc(map, p.dtype == GDN_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           4, const_cast<void *>(ptr), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed with CUresult %d", (int)r);
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

// ---- per-kernel timing (gdn_timing_enable / gdn_timing_read)
struct TimedLaunch {
    const char *name;
    cudaEvent_t start, stop;
};
std::atomic<bool> g_timing_on{false};
std::mutex g_timing_mutex;
std::vector<TimedLaunch> g_timed;          // launches recorded since the last read
std::vector<cudaEvent_t> g_event_pool;     // events free for reuse

cudaEvent_t pooled_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

void release_timed() {
    for (const TimedLaunch &t : g_timed) {
        if (t.start) g_event_pool.push_back(t.start);
        if (t.stop) g_event_pool.push_back(t.stop);
    }
    g_timed.clear();
}

// 4-D tensor map of a row-major [B][T][H][D] tensor (bf16 or fp32), box {box_d, 1, box_t, 1},
// 128-byte swizzle (box_d * element size must then be 128 bytes) or none.
int make_btd_map(CUtensorMap *map, const void *ptr, bool bf16, int B, int T, int H, int D, int box_d, int box_t,
                 bool swizzle = true) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled is not available from the driver");
        return GDN_ERR_CUDA;
    }
    const cuuint64_t e = bf16 ? 2 : 4;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {D * e, (cuuint64_t)H * D * e, (cuuint64_t)T * H * D * e};
    const cuuint32_t box[4] = {(cuuint32_t)box_d, 1, (cuuint32_t)box_t, 1};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    const CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                           const_cast<void *>(ptr), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed with CUresult %d", (int)r);
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

// 2-D tensor map of a row-major fp32 [rows][cols] array, box {32, box_rows}, 128-byte swizzle.
int make_rows_map(CUtensorMap *map, void *ptr, size_t rows, int cols, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled is not available from the driver");
        return GDN_ERR_CUDA;
    }
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
    const cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estride,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed with CUresult %d", (int)r);
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

// 5-D tensor map of a row-major [B][T][H][D] tensor (bf16 or fp32) whose box lands in shared
// memory column block by column block: dimensions {inner, T, D / inner, H, B}, box
// {inner, box_t, box_c, 1, 1}, so that one box holds box_c blocks of `inner` columns, each
// box_t rows x inner columns contiguous. With bf16 and inner = 8 (no swizzle) that is the
// core-matrix operand layout of box_t rows; with fp32 and inner = 32 (128-byte swizzle), box_c
// swizzled [box_t][32] tiles.
int make_colblock_map(CUtensorMap *map, const void *ptr, bool bf16, int B, int T, int H, int D, int inner, int box_t,
                      int box_c, bool swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled is not available from the driver");
        return GDN_ERR_CUDA;
    }
    const cuuint64_t e = bf16 ? 2 : 4;
    const cuuint64_t dims[5] = {(cuuint64_t)inner, (cuuint64_t)T, (cuuint64_t)(D / inner), (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[4] = {(cuuint64_t)H * D * e, inner * e, D * e, (cuuint64_t)T * H * D * e};
    const cuuint32_t box[5] = {(cuuint32_t)inner, (cuuint32_t)box_t, (cuuint32_t)box_c, 1, 1};
    const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    const CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5,
                           const_cast<void *>(ptr), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed with CUresult %d", (int)r);
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

// 5-D tensor map of a buffer of stacked operand blocks of the chunkwise forward (nblk blocks of
// [128][Dk] bf16 in the core-matrix layout, K chunk j holding 64 rows of the top half, then 64
// of the bottom half: [Q; K] with Dk columns, [P; KKm] with 64): dimensions
// {256, 2, 2 halves, Dk / 8 chunks, nblk} (a half's rows of a K chunk are 1 KB contiguous, two
// runs of 256 elements), box {256, 2, 1, Dk / 8, 1}, so that one box, at coordinates
// (0, 0, half, 0, block), is a [64][Dk] operand tile of one half (Q or K; P or KKm).
int make_qkm_map(CUtensorMap *map, void *ptr, size_t nblk, int Dk) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled is not available from the driver");
        return GDN_ERR_CUDA;
    }
    // a half's 64 rows of one K chunk are 1 KB contiguous: two runs of 256 elements
    const cuuint64_t dims[5] = {256, 2, 2, (cuuint64_t)(Dk / 8), (cuuint64_t)nblk};
    const cuuint64_t strides[4] = {512, 1024, 2048, (cuuint64_t)256 * Dk};
    const cuuint32_t box[5] = {256, 2, 1, (cuuint32_t)(Dk / 8), 1};
    const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, ptr, dims, strides, box, estride,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed with CUresult %d", (int)r);
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

}  // namespace

namespace gdn {
void timing_mark(const char *kernel, int phase, cudaStream_t s) {
    if (!g_timing_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    if (phase == 0) {
        TimedLaunch t{kernel, pooled_event(), nullptr};
        if (t.start == nullptr) return;
        cudaEventRecord(t.start, s);
        g_timed.push_back(t);
    } else {
        for (size_t i = g_timed.size(); i-- > 0;) {
            TimedLaunch &t = g_timed[i];
            if (t.stop == nullptr && strcmp(t.name, kernel) == 0) {
                t.stop = pooled_event();
                if (t.stop != nullptr) cudaEventRecord(t.stop, s);
                break;
            }
        }
    }
}
}  // namespace gdn

extern "C" {

int gdn_timing_enable(int on) {
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    g_timing_on.store(on != 0);
    if (!on) release_timed();
    return GDN_OK;
}

int gdn_timing_read(gdn_kernel_time *out, int max_entries) {
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    std::vector<gdn_kernel_time> agg;
    int rc = GDN_OK;
    for (const TimedLaunch &t : g_timed) {
        if (t.stop == nullptr) continue;
        float ms = 0.f;
        cudaError_t e = cudaEventSynchronize(t.stop);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.start, t.stop);
        if (e != cudaSuccess) {
            rc = cuda_status(e);
            break;
        }
        size_t j = 0;
        while (j < agg.size() && strcmp(agg[j].name, t.name) != 0) ++j;
        if (j == agg.size()) {
            gdn_kernel_time k;
            memset(&k, 0, sizeof k);
            snprintf(k.name, sizeof k.name, "%s", t.name);
            agg.push_back(k);
        }
        agg[j].launches += 1;
        agg[j].ms += ms;
    }
    release_timed();
    if (rc != GDN_OK) return rc;
    for (int i = 0; i < (int)agg.size() && i < max_entries; ++i)
        if (out != nullptr) out[i] = agg[(size_t)i];
    return (int)agg.size();
}

size_t gdn_ckpt_bytes(const gdn_shape *shape) {
    Plan p;
    if (make_plan(shape, &p) != GDN_OK) return 0;
    return ckpt_total(p);
}

size_t gdn_bwd_workspace_bytes(const gdn_shape *shape) {
    Plan p;
    if (make_plan(shape, &p) != GDN_OK) return 0;
    return bwd_workspace_total(p);
}

// The chunkwise forward on the tensor cores for plan p (a segmented call passes its view): the
// stages of launch_chunk_fwd; maps_out receives the lite stage's maps ([B][Hv][Dk][Dk], then the
// same transposed) and S_T its end states.
static int tc_fwd(const Plan &p, const void *q, const void *k, const void *v, const void *g, const void *beta,
                  const float *S0, void *y, float *S_T, float *ckpt, char *prod, float *maps_out, int stages,
                  cudaStream_t stream, const float *conv = nullptr) {
    const ChunkLayout cl = chunk_layout(p);
    gdn::ChunkParams cp;
    cp.q = q; cp.k = k; cp.v = v; cp.g = g; cp.beta = beta; cp.S0 = S0; cp.y = y; cp.S_T = S_T;
    cp.ckpt = ckpt; cp.resid = ckpt != nullptr ? ckpt + ckpt_state_bytes(p) / sizeof(float) : nullptr;
    cp.maps_M = maps_out;
    cp.conv = conv;
    cp.maps_Mt = maps_out != nullptr ? maps_out + (size_t)p.B * p.Hv * p.Dk * p.Dk : nullptr;
    cp.lam = reinterpret_cast<float *>(prod);
    cp.pkm = reinterpret_cast<__nv_bfloat16 *>(prod + (cl.pkm - cl.lam));
    cp.wm = reinterpret_cast<__nv_bfloat16 *>(prod + (cl.wm - cl.lam));
    cp.tm = reinterpret_cast<__nv_bfloat16 *>(prod + (cl.tm - cl.lam));
    cp.tcm = reinterpret_cast<__nv_bfloat16 *>(prod + (cl.tcm - cl.lam));
    cp.s0m = reinterpret_cast<__nv_bfloat16 *>(prod + (cl.s0m - cl.lam));
    cp.qkm = reinterpret_cast<__nv_bfloat16 *>(prod + (cl.qkm - cl.lam));
    cp.B = p.B; cp.T = p.T; cp.Hk = p.Hk; cp.Hv = p.Hv; cp.Dv = p.Dv; cp.NC = p.NC;
    g_last_error[0] = '\0';
    int rc = device_status_address(&cp.status);
    if (rc != GDN_OK) return rc;
    gdn::ChunkFwdMaps maps = {};
    if ((rc = make_colblock_map(&maps.k, k, true, p.B, p.T, p.Hk, p.Dk, 8, 64, p.Dk / 8, false)) != GDN_OK ||
        (rc = make_colblock_map(&maps.q, q, true, p.B, p.T, p.Hk, p.Dk, 8, 64, p.Dk / 8, false)) != GDN_OK ||
        (rc = make_qkm_map(&maps.qk, cp.qkm, (size_t)p.B * p.Hk * p.NC, p.Dk)) != GDN_OK)
        return rc;
    // the sweeps' maps (prep alone reads K and Q and writes [Q; K]); without a saved buffer (an
    // inference forward) nothing goes to the residual or checkpoint maps
    if ((stages & (gdn::kStageSweep | gdn::kStageLite)) &&
        ((rc = make_btd_map(&maps.vb, v, true, p.B, p.T, p.Hv, p.Dv, 64, 64, true)) != GDN_OK ||
         (rc = make_btd_map(&maps.y, y, true, p.B, p.T, p.Hv, p.Dv, 64, 64)) != GDN_OK))
        return rc;
    if ((stages & (gdn::kStageSweep | gdn::kStageLite)) && ckpt != nullptr &&
        ((rc = make_colblock_map(&maps.r, cp.resid, false, p.B, p.T, p.Hv, p.Dv, 32, 64, 2, true)) != GDN_OK ||
         (rc = make_rows_map(&maps.ck, ckpt, (size_t)p.B * p.Hv * p.NC * p.Dv, p.Dk, 64)) != GDN_OK))
        return rc;
    if ((size_t)p.B * p.Hv * p.NC * p.Dv > 0x7fffffffu) return GDN_ERR_UNSUPPORTED_SHAPE;   // TMA row coordinates
    return cuda_status(gdn::launch_chunk_fwd(cp, maps, p.Dk, stream, stages));
}

// The chunkwise backward on the tensor cores for plan p: the stages of launch_chunk_bwd.
static int tc_bwd(const Plan &p, const void *beta, const float *ckpt, const char *prod, const void *dy,
                  const float *dS_T, void *dq, void *dk, void *dv, void *dg, void *dbeta, float *dS0, char *ws,
                  int stages, cudaStream_t stream) {
    const ChunkLayout cl = chunk_layout(p);
    const TcWorkspace tw = tc_workspace_layout(p);
    gdn::ChunkBwdParams cp;
    cp.dy = dy; cp.beta = beta;
    cp.resid = ckpt + ckpt_state_bytes(p) / sizeof(float);
    cp.lam = reinterpret_cast<const float *>(prod);
    cp.tm = reinterpret_cast<const __nv_bfloat16 *>(prod + (cl.tm - cl.lam));
    cp.pkm = reinterpret_cast<const __nv_bfloat16 *>(prod + (cl.pkm - cl.lam));
    cp.s0m = reinterpret_cast<const __nv_bfloat16 *>(prod + (cl.s0m - cl.lam));
    cp.qkm = reinterpret_cast<const __nv_bfloat16 *>(prod + (cl.qkm - cl.lam));
    cp.dS_T = dS_T; cp.dS0 = dS0;
    cp.dv = dv; cp.dg = dg; cp.dq = dq; cp.dk = dk; cp.dbeta = dbeta;
    cp.ws_db = reinterpret_cast<float *>(ws + tw.db);
    cp.ws_f = reinterpret_cast<float *>(ws + tw.f);
    cp.ws_yu = reinterpret_cast<__nv_bfloat16 *>(ws + tw.yu);
    cp.ws_dl = reinterpret_cast<__nv_bfloat16 *>(ws + tw.dl);
    cp.ws_dsl = reinterpret_cast<__nv_bfloat16 *>(ws + tw.dsl);
    cp.ready = nullptr;
    cp.next = nullptr;
    cp.B = p.B; cp.T = p.T; cp.Hk = p.Hk; cp.Hv = p.Hv; cp.Dv = p.Dv; cp.NC = p.NC; cp.nsplit = p.nsplit;
    g_last_error[0] = '\0';
    int rc = device_status_address(&cp.status);
    if (rc != GDN_OK) return rc;
    CUtensorMap tm_dv, tm_dy, tm_qk, tm_pk, tm_dq, tm_dk;
    if ((rc = make_btd_map(&tm_dv, dv, true, p.B, p.T, p.Hv, p.Dv, 64, 64)) != GDN_OK ||
        (rc = make_colblock_map(&tm_dy, dy, true, p.B, p.T, p.Hv, p.Dv, 8, 128, 8, false)) != GDN_OK ||
        (rc = make_qkm_map(&tm_qk, const_cast<__nv_bfloat16 *>(cp.qkm), (size_t)p.B * p.Hk * p.NC, p.Dk)) != GDN_OK ||
        (rc = make_qkm_map(&tm_pk, const_cast<__nv_bfloat16 *>(cp.pkm), (size_t)p.B * p.Hv * p.NC, 64)) != GDN_OK ||
        (rc = make_btd_map(&tm_dq, dq, true, p.B, p.T, p.Hk, p.Dk, 64, 64)) != GDN_OK ||
        (rc = make_btd_map(&tm_dk, dk, true, p.B, p.T, p.Hk, p.Dk, 64, 64)) != GDN_OK)
        return rc;
    if (stages & gdn::kStageGrad) {
        // the gradient kernel runs alongside the reverse sweep of the same call, on the counters
        // it publishes: both start from zero
        if (!(stages & gdn::kStageDsweep)) return GDN_ERR_INVALID_ARG;
        const size_t n = (size_t)p.B * p.Hv * p.NC;
        cp.ready = reinterpret_cast<unsigned *>(ws + tw.sync);
        cp.next = reinterpret_cast<int *>(cp.ready + n);
        if ((rc = cuda_status(cudaMemsetAsync(cp.ready, 0, (n + 1) * 4, stream))) != GDN_OK) return rc;
    }
    return cuda_status(gdn::launch_chunk_bwd(cp, tm_dv, tm_dy, tm_qk, tm_pk, tm_dq, tm_dk, p.Dk, stream, stages));
}

int gdn_fwd(const gdn_shape *shape, const void *q, const void *k, const void *v, const void *g,
            const void *beta, const float *S0, void *y, float *S_T, float *ckpt, size_t ckpt_bytes,
            void *stream) {
    Plan p;
    int rc = make_plan(shape, &p);
    if (rc != GDN_OK) return rc;
    if (!q || !k || !v || !g || !beta || !y) return GDN_ERR_INVALID_ARG;
    const void *all[] = {q, k, v, g, beta, S0, y, S_T, ckpt};
    for (const void *ptr : all)
        if (ptr && !aligned(ptr)) return GDN_ERR_MISALIGNED;
    if (ckpt != nullptr && ckpt_bytes < ckpt_total(p)) return GDN_ERR_BUFFER_TOO_SMALL;
    g_last_error[0] = '\0';
    gdn::FwdParams fp;
    fp.q = q; fp.k = k; fp.v = v; fp.g = g; fp.beta = beta; fp.S0 = S0;
    fp.y = y; fp.S_T = S_T; fp.ckpt = ckpt;
    fp.resid = ckpt != nullptr ? ckpt + ckpt_state_bytes(p) / sizeof(float) : nullptr;
    fp.B = p.B; fp.T = p.T; fp.Hk = p.Hk; fp.Hv = p.Hv; fp.Dv = p.Dv; fp.C = p.C; fp.NC = p.NC;
    rc = device_status_address(&fp.status);
    if (rc != GDN_OK) return rc;
    if (p.tc && ckpt != nullptr)       // chunkwise form on the tensor cores
        return tc_fwd(p, q, k, v, g, beta, S0, y, S_T, ckpt, chunk_products(p, ckpt), nullptr,
                      gdn::kStagePrep | gdn::kStageSweep,
                      (cudaStream_t)stream);
    if (p.T == 1 && ckpt == nullptr && gdn::decode_takes(p.Dk))   // a decode step: one streaming pass
        return cuda_status(gdn::launch_decode(fp, p.Dk, p.dtype, (cudaStream_t)stream));
    CUtensorMap tm_q, tm_k;
    if ((rc = make_qk_map(&tm_q, q, p, gdn::kFwdTile)) != GDN_OK) return rc;
    if ((rc = make_qk_map(&tm_k, k, p, gdn::kFwdTile)) != GDN_OK) return rc;
    return cuda_status(gdn::launch_fwd(fp, tm_q, tm_k, p.Dk, p.dtype, p.warps, (cudaStream_t)stream));
}

int gdn_bwd(const gdn_shape *shape, const void *q, const void *k, const void *v, const void *g,
            const void *beta, const float *ckpt, size_t ckpt_bytes, const void *dy, const float *dS_T,
            void *dq, void *dk, void *dv, void *dg, void *dbeta, float *dS0, void *workspace,
            size_t workspace_bytes, void *stream) {
    Plan p;
    int rc = make_plan(shape, &p);
    if (rc != GDN_OK) return rc;
    if (!q || !k || !v || !g || !beta || !ckpt || !dy || !dq || !dk || !dv || !dg || !dbeta || !workspace)
        return GDN_ERR_INVALID_ARG;
    const void *all[] = {q, k, v, g, beta, ckpt, dy, dS_T, dq, dk, dv, dg, dbeta, dS0, workspace};
    for (const void *ptr : all)
        if (ptr && !aligned(ptr)) return GDN_ERR_MISALIGNED;
    if (ckpt_bytes < ckpt_total(p) || workspace_bytes < bwd_workspace_total(p)) return GDN_ERR_BUFFER_TOO_SMALL;
    char *ws = static_cast<char *>(workspace);
    if (p.tcb)                         // chunkwise form on the tensor cores, reading the chunkwise forward's saved buffer
        return tc_bwd(p, beta, ckpt, chunk_products(p, ckpt), dy, dS_T, dq, dk, dv, dg, dbeta, dS0, ws,
                      gdn::kStageDsweep | gdn::kStageGrad,
                      (cudaStream_t)stream);
    const Workspace w = workspace_layout(p);

    gdn::BwdParams bp;
    bp.q = q; bp.k = k; bp.v = v; bp.g = g; bp.beta = beta; bp.ckpt = ckpt; bp.dy = dy;
    bp.resid = ckpt + ckpt_state_bytes(p) / sizeof(float);
    bp.dS_T = dS_T; bp.dS0 = dS0; bp.dv = dv;
    bp.ws_dq = reinterpret_cast<float *>(ws + w.dq);
    bp.ws_dk = reinterpret_cast<float *>(ws + w.dk);
    bp.ws_dg = reinterpret_cast<float *>(ws + w.dg);
    bp.ws_db = reinterpret_cast<float *>(ws + w.db);
    bp.ws_state = reinterpret_cast<float *>(ws + w.state);
    bp.B = p.B; bp.T = p.T; bp.Hk = p.Hk; bp.Hv = p.Hv; bp.Dv = p.Dv; bp.C = p.C; bp.NC = p.NC;
    bp.nsplit = p.nsplit; bp.nsub_max = p.nsub_max; bp.slots = p.slots;

    gdn::ReduceParams rp;
    rp.ws_dq = bp.ws_dq; rp.ws_dk = bp.ws_dk; rp.ws_dg = bp.ws_dg; rp.ws_db = bp.ws_db;
    rp.dq = dq; rp.dk = dk; rp.dg = dg; rp.dbeta = dbeta;
    rp.B = p.B; rp.T = p.T; rp.Hk = p.Hk; rp.Hv = p.Hv; rp.Dk = p.Dk; rp.nsplit = p.nsplit;

    g_last_error[0] = '\0';
    rc = device_status_address(&bp.status);
    if (rc != GDN_OK) return rc;
    CUtensorMap tm_q, tm_k;
    if ((rc = make_qk_map(&tm_q, q, p, p.sub + 1)) != GDN_OK) return rc;
    if ((rc = make_qk_map(&tm_k, k, p, p.sub + 1)) != GDN_OK) return rc;
    rc = cuda_status(gdn::launch_bwd(bp, tm_q, tm_k, p.Dk, p.dtype, (cudaStream_t)stream));
    if (rc != GDN_OK) return rc;
    return cuda_status(gdn::launch_reduce(rp, p.dtype, (cudaStream_t)stream));
}

// ---- sequence-parallel form: the problem seen as B * P rows of T / P steps (segments of whole
// chunks are contiguous in [B][T][...], so every tensor keeps its address)
static int seg_plans(const gdn_shape *shape, int segments, Plan *p, Plan *pv) {
    int rc = make_plan(shape, p);
    if (rc != GDN_OK) return rc;
    if (segments < 1 || !p->tc || !p->tcb || p->T % (64 * segments) != 0 ||
        (long long)p->B * segments > (1LL << 30))
        return GDN_ERR_UNSUPPORTED_SHAPE;
    gdn_shape v = *shape;
    v.B = shape->B * segments;
    v.T = shape->T / segments;
    rc = make_plan(&v, pv);
    if (rc != GDN_OK) return rc;
    return pv->tc && pv->tcb ? GDN_OK : GDN_ERR_UNSUPPORTED_SHAPE;
}

static size_t seg_maps_offset(const Plan &pv) { return round_up(ckpt_total(pv)); }
static size_t seg_state_bytes(const Plan &pv) { return round_up((size_t)pv.B * pv.Hv * pv.Dv * pv.Dk * 4); }

size_t gdn_seg_ckpt_bytes(const gdn_shape *shape, int segments) {
    Plan p, pv;
    if (shape == nullptr || seg_plans(shape, segments, &p, &pv) != GDN_OK) return 0;
    return seg_maps_offset(pv) + round_up(2 * (size_t)pv.B * pv.Hv * pv.Dk * pv.Dk * 4);
}

size_t gdn_seg_workspace_bytes(const gdn_shape *shape, int segments) {
    Plan p, pv;
    if (shape == nullptr || seg_plans(shape, segments, &p, &pv) != GDN_OK) return 0;
    return 2 * seg_state_bytes(pv) + bwd_workspace_total(pv);
}

int gdn_seg_choose(const gdn_shape *shape, int sm_count) {
    Plan p;
    if (shape == nullptr || make_plan(shape, &p) != GDN_OK || !p.tc || !p.tcb || sm_count < 1) return 1;
    // the sweep's grid for P segments: (Dv / 64) * Hv * B * P CTAs, one per SM
    const long long base = (long long)(p.Dv / 64) * p.Hv * p.B;
    int P = 1;
    while (base * 2 * P <= sm_count && p.T % (64 * 2 * P) == 0 && P < (1 << 20)) P *= 2;
    return P;
}

// dst[b] = src[b * P + s] for every b: blocks of `blk` bytes, one copy per batch row
static int seg_pick(void *dst, const void *src, size_t blk, int B, int P, int s, cudaStream_t stream) {
    for (int b = 0; b < B; ++b) {
        const int rc = cuda_status(cudaMemcpyAsync(static_cast<char *>(dst) + (size_t)b * blk,
                                                   static_cast<const char *>(src) + ((size_t)b * P + s) * blk, blk,
                                                   cudaMemcpyDeviceToDevice, stream));
        if (rc != GDN_OK) return rc;
    }
    return GDN_OK;
}

int gdn_fwd_seg(const gdn_shape *shape, int segments, const void *q, const void *k, const void *v, const void *g,
                const void *beta, const float *S0, void *y, float *S_T, float *ckpt, size_t ckpt_bytes,
                void *workspace, size_t workspace_bytes, void *stream) {
    if (shape == nullptr) return GDN_ERR_INVALID_ARG;
    Plan p, pv;
    int rc = seg_plans(shape, segments, &p, &pv);
    if (rc != GDN_OK) return rc;
    if (!q || !k || !v || !g || !beta || !y || !ckpt || !workspace) return GDN_ERR_INVALID_ARG;
    const void *all[] = {q, k, v, g, beta, S0, y, S_T, ckpt, workspace};
    for (const void *ptr : all)
        if (ptr && !aligned(ptr)) return GDN_ERR_MISALIGNED;
    if (ckpt_bytes < gdn_seg_ckpt_bytes(shape, segments) || workspace_bytes < gdn_seg_workspace_bytes(shape, segments))
        return GDN_ERR_BUFFER_TOO_SMALL;
    const cudaStream_t st = (cudaStream_t)stream;
    float *maps = reinterpret_cast<float *>(reinterpret_cast<char *>(ckpt) + seg_maps_offset(pv));
    float *C = static_cast<float *>(workspace);
    float *X = reinterpret_cast<float *>(static_cast<char *>(workspace) + seg_state_bytes(pv));
    // every segment from a zero state (its end state: C) and as maps (the lite sweep), then the
    // scan of the start states, then every segment again from its start state
    rc = tc_fwd(pv, q, k, v, g, beta, nullptr, y, C, ckpt, chunk_products(pv, ckpt), maps, gdn::kStagePrep | gdn::kStageLite,
                st);
    if (rc != GDN_OK) return rc;
    int *status = nullptr;
    if ((rc = device_status_address(&status)) != GDN_OK) return rc;
    rc = cuda_status(gdn::launch_segment_scan(S0, maps, C, X, p.B, segments, p.Hv, p.Dv, p.Dk, false, status, st));
    if (rc != GDN_OK) return rc;
    rc = tc_fwd(pv, q, k, v, g, beta, X, y, C, ckpt, chunk_products(pv, ckpt), nullptr, gdn::kStageSweep, st);
    if (rc != GDN_OK || S_T == nullptr) return rc;
    return seg_pick(S_T, C, (size_t)p.Hv * p.Dv * p.Dk * 4, p.B, segments, segments - 1, st);
}

int gdn_bwd_seg(const gdn_shape *shape, int segments, const void *q, const void *k, const void *v, const void *g,
                const void *beta, const float *ckpt, size_t ckpt_bytes, const void *dy, const float *dS_T, void *dq,
                void *dk, void *dv, void *dg, void *dbeta, float *dS0, void *workspace, size_t workspace_bytes,
                void *stream) {
    if (shape == nullptr) return GDN_ERR_INVALID_ARG;
    Plan p, pv;
    int rc = seg_plans(shape, segments, &p, &pv);
    if (rc != GDN_OK) return rc;
    if (!q || !k || !v || !g || !beta || !ckpt || !dy || !dq || !dk || !dv || !dg || !dbeta || !workspace)
        return GDN_ERR_INVALID_ARG;
    const void *all[] = {q, k, v, g, beta, ckpt, dy, dS_T, dq, dk, dv, dg, dbeta, dS0, workspace};
    for (const void *ptr : all)
        if (ptr && !aligned(ptr)) return GDN_ERR_MISALIGNED;
    if (ckpt_bytes < gdn_seg_ckpt_bytes(shape, segments) || workspace_bytes < gdn_seg_workspace_bytes(shape, segments))
        return GDN_ERR_BUFFER_TOO_SMALL;
    const cudaStream_t st = (cudaStream_t)stream;
    const float *maps = reinterpret_cast<const float *>(reinterpret_cast<const char *>(ckpt) + seg_maps_offset(pv));
    float *D = static_cast<float *>(workspace);
    float *Y = reinterpret_cast<float *>(static_cast<char *>(workspace) + seg_state_bytes(pv));
    char *ws = static_cast<char *>(workspace) + 2 * seg_state_bytes(pv);
    // every segment's reverse sweep from a zero end adjoint (its start adjoint: D), the reverse
    // scan of the end adjoints, then the backward proper from them
    rc = tc_bwd(pv, beta, ckpt, chunk_products(pv, ckpt), dy, nullptr, dq, dk, dv, dg, dbeta, D, ws, gdn::kStageDsweep, st);
    if (rc != GDN_OK) return rc;
    int *status = nullptr;
    if ((rc = device_status_address(&status)) != GDN_OK) return rc;
    const float *maps_t = maps + (size_t)pv.B * pv.Hv * pv.Dk * pv.Dk;
    rc = cuda_status(gdn::launch_segment_scan(dS_T, maps_t, D, Y, p.B, segments, p.Hv, p.Dv, p.Dk, true, status, st));
    if (rc != GDN_OK) return rc;
    rc = tc_bwd(pv, beta, ckpt, chunk_products(pv, ckpt), dy, Y, dq, dk, dv, dg, dbeta, D, ws,
                gdn::kStageDsweep | gdn::kStageGrad, st);
    if (rc != GDN_OK || dS0 == nullptr) return rc;
    return seg_pick(dS0, D, (size_t)p.Hv * p.Dv * p.Dk * 4, p.B, segments, 0, st);
}

// ---- inference forward on the tensor cores: the per-chunk products in a workspace, nothing saved
size_t gdn_infer_workspace_bytes(const gdn_shape *shape) {
    Plan p;
    if (shape == nullptr || make_plan(shape, &p) != GDN_OK || !p.tc) return 0;
    return round_up(chunk_products_bytes(p));
}

int gdn_fwd_infer(const gdn_shape *shape, const void *q, const void *k, const void *v, const void *g,
                  const void *beta, const float *S0, void *y, float *S_T, void *workspace, size_t workspace_bytes,
                  void *stream) {
    if (shape == nullptr) return GDN_ERR_INVALID_ARG;
    Plan p;
    int rc = make_plan(shape, &p);
    if (rc != GDN_OK) return rc;
    if (!p.tc) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!q || !k || !v || !g || !beta || !y || !workspace) return GDN_ERR_INVALID_ARG;
    const void *all[] = {q, k, v, g, beta, S0, y, S_T, workspace};
    for (const void *ptr : all)
        if (ptr && !aligned(ptr)) return GDN_ERR_MISALIGNED;
    if (workspace_bytes < gdn_infer_workspace_bytes(shape)) return GDN_ERR_BUFFER_TOO_SMALL;
    return tc_fwd(p, q, k, v, g, beta, S0, y, S_T, nullptr, static_cast<char *>(workspace), nullptr,
                  gdn::kStagePrep | gdn::kStageSweep, (cudaStream_t)stream);
}

// ---- re-computation mode: the saved buffer holds only the checkpoints and the residuals
static int rc_plan(const gdn_shape *shape, Plan *p) {
    if (shape == nullptr) return GDN_ERR_INVALID_ARG;
    const int rc = make_plan(shape, p);
    if (rc != GDN_OK) return rc;
    return p->tc && p->tcb ? GDN_OK : GDN_ERR_UNSUPPORTED_SHAPE;
}

size_t gdn_rc_ckpt_bytes(const gdn_shape *shape) {
    Plan p;
    if (rc_plan(shape, &p) != GDN_OK) return 0;
    return ckpt_state_bytes(p) + round_up(ckpt_resid_bytes(p));
}

size_t gdn_rc_fwd_workspace_bytes(const gdn_shape *shape) {
    Plan p;
    if (rc_plan(shape, &p) != GDN_OK) return 0;
    return round_up(chunk_products_bytes(p));
}

size_t gdn_rc_bwd_workspace_bytes(const gdn_shape *shape) {
    Plan p;
    if (rc_plan(shape, &p) != GDN_OK) return 0;
    return round_up(chunk_products_bytes(p)) + bwd_workspace_total(p);
}

int gdn_fwd_rc(const gdn_shape *shape, const void *q, const void *k, const void *v, const void *g, const void *beta,
               const float *S0, void *y, float *S_T, float *ckpt, size_t ckpt_bytes, void *workspace,
               size_t workspace_bytes, void *stream) {
    Plan p;
    int rc = rc_plan(shape, &p);
    if (rc != GDN_OK) return rc;
    if (!q || !k || !v || !g || !beta || !y || !ckpt || !workspace) return GDN_ERR_INVALID_ARG;
    const void *all[] = {q, k, v, g, beta, S0, y, S_T, ckpt, workspace};
    for (const void *ptr : all)
        if (ptr && !aligned(ptr)) return GDN_ERR_MISALIGNED;
    if (ckpt_bytes < gdn_rc_ckpt_bytes(shape) || workspace_bytes < gdn_rc_fwd_workspace_bytes(shape))
        return GDN_ERR_BUFFER_TOO_SMALL;
    // the chunkwise forward with its per-chunk products in the workspace (dropped afterwards)
    return tc_fwd(p, q, k, v, g, beta, S0, y, S_T, ckpt, static_cast<char *>(workspace), nullptr,
                  gdn::kStagePrep | gdn::kStageSweep, (cudaStream_t)stream);
}

int gdn_bwd_rc(const gdn_shape *shape, const void *q, const void *k, const void *v, const void *g, const void *beta,
               const float *ckpt, size_t ckpt_bytes, const void *dy, const float *dS_T, void *dq, void *dk, void *dv,
               void *dg, void *dbeta, float *dS0, void *workspace, size_t workspace_bytes, void *stream) {
    Plan p;
    int rc = rc_plan(shape, &p);
    if (rc != GDN_OK) return rc;
    if (!q || !k || !v || !g || !beta || !ckpt || !dy || !dq || !dk || !dv || !dg || !dbeta || !workspace)
        return GDN_ERR_INVALID_ARG;
    const void *all[] = {q, k, v, g, beta, ckpt, dy, dS_T, dq, dk, dv, dg, dbeta, dS0, workspace};
    for (const void *ptr : all)
        if (ptr && !aligned(ptr)) return GDN_ERR_MISALIGNED;
    if (ckpt_bytes < gdn_rc_ckpt_bytes(shape) || workspace_bytes < gdn_rc_bwd_workspace_bytes(shape))
        return GDN_ERR_BUFFER_TOO_SMALL;
    const cudaStream_t st = (cudaStream_t)stream;
    char *prod = static_cast<char *>(workspace);
    char *ws = prod + round_up(chunk_products_bytes(p));
    // every chunk's forward products again (prep, which also turns the checkpoints into the
    // gradient kernel's bf16 operand tiles), then the backward proper
    rc = tc_fwd(p, q, k, v, g, beta, nullptr, nullptr, nullptr, const_cast<float *>(ckpt), prod, nullptr,
                gdn::kStagePrep, st, ckpt);
    if (rc != GDN_OK) return rc;
    return tc_bwd(p, beta, ckpt, prod, dy, dS_T, dq, dk, dv, dg, dbeta, dS0, ws, gdn::kStageDsweep | gdn::kStageGrad,
                  st);
}

int gdn_gates_fwd(const gdn_shape *shape, const void *a, const void *b, const float *A_log,
                  const float *dt_bias, void *g, void *beta, void *stream) {
    Plan p;
    int rc = make_plan(shape, &p);
    if (rc != GDN_OK) return rc;
    if ((long long)p.B * p.T > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!a || !b || !A_log || !dt_bias || !g || !beta) return GDN_ERR_INVALID_ARG;
    const void *all[] = {a, b, A_log, dt_bias, g, beta};
    for (const void *ptr : all)
        if (!aligned(ptr)) return GDN_ERR_MISALIGNED;
    g_last_error[0] = '\0';
    gdn::GatesParams gp = {};
    gp.a = a; gp.b = b; gp.A_log = A_log; gp.dt_bias = dt_bias; gp.g = g; gp.beta = beta;
    gp.rows = p.B * p.T; gp.Hv = p.Hv;
    return cuda_status(gdn::launch_gates_fwd(gp, p.dtype, (cudaStream_t)stream));
}

int gdn_gates_bwd(const gdn_shape *shape, const void *a, const void *b, const float *A_log,
                  const float *dt_bias, const void *dg, const void *dbeta, void *da, void *db,
                  float *dA_log, float *ddt_bias, void *stream) {
    Plan p;
    int rc = make_plan(shape, &p);
    if (rc != GDN_OK) return rc;
    if ((long long)p.B * p.T > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!a || !b || !A_log || !dt_bias || !dg || !dbeta || !da || !db || !dA_log || !ddt_bias)
        return GDN_ERR_INVALID_ARG;
    const void *all[] = {a, b, A_log, dt_bias, dg, dbeta, da, db, dA_log, ddt_bias};
    for (const void *ptr : all)
        if (!aligned(ptr)) return GDN_ERR_MISALIGNED;
    g_last_error[0] = '\0';
    gdn::GatesParams gp = {};
    gp.a = a; gp.b = b; gp.A_log = A_log; gp.dt_bias = dt_bias; gp.dg = dg; gp.dbeta = dbeta;
    gp.da = da; gp.db = db; gp.dA_log = dA_log; gp.ddt_bias = ddt_bias;
    gp.rows = p.B * p.T; gp.Hv = p.Hv;
    return cuda_status(gdn::launch_gates_bwd(gp, p.dtype, (cudaStream_t)stream));
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// gdn_bwd_noalloc: gdn_bwd with its scratch in a fixed device array instead of a caller
// workspace, for callers that cannot allocate device memory.
namespace {

// The scratch itself: one copy per device, allocated by the CUDA runtime when this
// library's device code is loaded on that device, kept until the process exits.
static __device__ __align__(256) unsigned char g_bwd_static_scratch[GDN_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices];  // device address of g_bwd_static_scratch, per device

// Host code cannot use g_bwd_static_scratch's name as a device address (on the host it
// names a stand-in). Look the address up once per device, with that device current.
int static_scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_status(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_bwd_static_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        g_scratch_addr[dev] = addr;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_bwd_noalloc(const gdn_shape *shape, const void *q, const void *k, const void *v,
                    const void *g, const void *beta, const float *ckpt, size_t ckpt_bytes,
                    const void *dy, const float *dS_T, void *dq, void *dk, void *dv, void *dg,
                    void *dbeta, float *dS0, void *stream) {
    Plan p;
    int rc = make_plan(shape, &p);
    if (rc != GDN_OK) return rc;
    const size_t need = bwd_workspace_total(p);
    if (need > GDN_BWD_NOALLOC_SCRATCH_BYTES) return GDN_ERR_SCRATCH_LIMIT;
    if (!q || !k || !v || !g || !beta || !ckpt || !dy || !dq || !dk || !dv || !dg || !dbeta)
        return GDN_ERR_INVALID_ARG;
    const void *all[] = {q, k, v, g, beta, ckpt, dy, dS_T, dq, dk, dv, dg, dbeta, dS0};
    for (const void *ptr : all)
        if (ptr && !aligned(ptr)) return GDN_ERR_MISALIGNED;
    if (ckpt_bytes < ckpt_total(p)) return GDN_ERR_BUFFER_TOO_SMALL;
    g_last_error[0] = '\0';
    void *scratch = nullptr;
    rc = static_scratch_address(&scratch);
    if (rc != GDN_OK) return rc;
    return gdn_bwd(shape, q, k, v, g, beta, ckpt, ckpt_bytes, dy, dS_T, dq, dk, dv, dg, dbeta, dS0, scratch,
                   GDN_BWD_NOALLOC_SCRATCH_BYTES, stream);
}

const char *gdn_strerror(int code) {
    switch (code) {
        case GDN_OK: return "success";
        case GDN_ERR_INVALID_ARG: return "invalid argument (NULL shape or required pointer, size <= 0, or bad dtype)";
        case GDN_ERR_MISALIGNED: return "a pointer is not 16-byte aligned";
        case GDN_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (Hv % Hk, Dk, Dv, chunk or tensor size)";
        case GDN_ERR_BUFFER_TOO_SMALL:
            return "a caller buffer is too small (ckpt_bytes < gdn_ckpt_bytes() or workspace_bytes < "
                   "gdn_bwd_workspace_bytes())";
        case GDN_ERR_CUDA: return "CUDA runtime error (see gdn_last_error)";
        case GDN_ERR_TIMEOUT: return "a bounded device-side wait timed out";
        case GDN_ERR_SCRATCH_LIMIT:
            return "problem needs more scratch than gdn_bwd_noalloc's fixed GDN_BWD_NOALLOC_SCRATCH_BYTES "
                   "(compare gdn_bwd_workspace_bytes; use gdn_bwd with a workspace instead)";
        default: return "unknown gdn error code";
    }
}

const char *gdn_last_error(void) { return g_last_error; }

int gdn_device_status(void) {
    int *addr = nullptr;
    int rc = device_status_address(&addr);
    if (rc != GDN_OK) return rc;
    int value = 0;
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&value, g_device_status, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_status(e);
    return value;
}

int gdn_version(void) { return GDN_VERSION; }

int gdn_debug_wait_probe(unsigned polls, void *stream) {
    if (polls < 1 || polls > gdn::kWaitLimit) return GDN_ERR_INVALID_ARG;
    int *status = nullptr;
    int rc = device_status_address(&status);
    if (rc != GDN_OK) return rc;
    g_last_error[0] = '\0';
    return cuda_status(gdn::launch_wait_probe(status, polls, (cudaStream_t)stream));
}

int gdn_diag_fma_tflops(int packed, double *tflops) {
    if (tflops == nullptr) return GDN_ERR_INVALID_ARG;
    g_last_error[0] = '\0';
    return cuda_status(gdn::measure_fma_rate(packed != 0, tflops));
}

}  // extern "C"
