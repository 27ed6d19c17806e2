// gdn_umma.cuh -- 5th-generation tensor-core (tcgen05) helpers for the chunkwise kernels
// (internal; not part of the C ABI).
//
// Operands live in shared memory in the canonical no-swizzle K-major layout: "core
// matrices" of 8 rows x 16 bytes (128 contiguous bytes, rows of 16 bytes), stored K-chunk
// major: the core matrix of row group i and 16-byte K chunk j sits at (j * RG + i) * 128,
// RG = rows / 8. In a matrix descriptor the leading byte offset is then the distance
// between K-adjacent core matrices (RG * 128) and the stride byte offset the distance
// between row-adjacent ones (128). One MMA consumes 32 bytes of K (16 bf16 or 8 tf32
// elements): two core matrices; the next one starts 2 * RG * 128 bytes further.
//
// The same bytes also serve as the transposed operand: read "MN-major", the array's rows
// become the operand's K index and its K index the operand's M (or N) index. A core
// matrix is then 8 K rows x 16 bytes of M/N, and the descriptor's leading byte offset is
// still the distance between K-adjacent core matrices (here the row-group stride, 128)
// and the stride byte offset the distance between M/N-adjacent ones (RG * 128); the
// instruction descriptor marks the operand as transposed (bit 15 for A, 16 for B).
//
// Accumulators live in tensor memory (fp32). For M = 128 row m is lane m; for M = 64
// row m is lane (m % 16) + 32 * (m / 16), i.e. lanes 0-15 of each warp quarter.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Byte offset of element (r, kb) (kb = byte offset along K) of a K-major operand with
// `rows` rows (a multiple of 8), in the layout above.
__host__ __device__ __forceinline__ uint32_t cm_off(int r, int kb, int rows) {
    return (uint32_t)(((kb >> 4) * (rows >> 3) + (r >> 3)) * 128 + (r & 7) * 16 + (kb & 15));
}

// Shared-memory matrix descriptor (no swizzle) of a K-major operand with `rows` rows whose
// K range starts at byte `kb0` (a multiple of 32).
__device__ __forceinline__ uint64_t umma_desc(const void *base, int rows, int kb0) {
    const uint32_t start = smem_addr(base) + (uint32_t)((kb0 >> 4) * (rows >> 3) * 128);
    const uint32_t lbo = (uint32_t)((rows >> 3) * 128), sbo = 128;
    uint64_t d = 0;
    d |= (uint64_t)((start >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version of this generation
    return d;                 // base offset 0, no swizzle
}

// Descriptor from a shared-memory byte address and the two strides (no swizzle).
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t start, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((start >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// MN-major operand in the 128-byte swizzle (what a TMA box of 64 bf16 columns x rows with
// CU_TENSOR_MAP_SWIZZLE_128B writes at a 1024-byte aligned address): K index = tile row (128
// bytes, the 16-byte chunks of row r permuted by r % 8), MN index = column (64 of them, one
// swizzle atom wide). Atoms of 8 rows follow each other at 1024 bytes along K (the stride
// field); along MN there is one atom (the leading field is not used). A step of 16 along K
// moves the start by 2048 bytes.
__device__ __forceinline__ uint64_t sw128_mnmajor(const void *tile) {
    uint64_t d = umma_sdesc(smem_addr(tile), 1024u, 1024u);
    d |= (uint64_t)2 << 61;   // layout: 128-byte swizzle
    return d;
}

// K-major view of an array with R rows: operand rows from array row r0, K from byte kb0.
__device__ __forceinline__ uint64_t cm_kmajor(const void *base, int R, int r0, int kb0) {
    return umma_sdesc(smem_addr(base) + (uint32_t)(((kb0 >> 4) * (R >> 3) + (r0 >> 3)) * 128), (uint32_t)(R * 16),
                      128u);
}

// MN-major view of a bf16 array with R rows: operand K index = array row (from k0, a
// multiple of 8), operand M/N index = array column (from mn0, a multiple of 8).
__device__ __forceinline__ uint64_t cm_mnmajor(const void *base, int R, int k0, int mn0) {
    return umma_sdesc(smem_addr(base) + (uint32_t)(((mn0 >> 3) * (R >> 3) + (k0 >> 3)) * 128), 128u,
                      (uint32_t)(R * 16));
}

// Instruction descriptor: fp32 accumulator, A and B of format `fmt` (1 = bf16 with
// kind::f16, 2 = tf32 with kind::tf32), both K-major, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc(int fmt, int M, int N) {
    return (1u << 4) | ((uint32_t)fmt << 7) | ((uint32_t)fmt << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// The same with either operand transposed (read MN-major).
__host__ __device__ constexpr uint32_t umma_idesc_t(int fmt, int M, int N, bool a_mn, bool b_mn) {
    return umma_idesc(fmt, M, N) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16);
}

// D (tensor memory) = A B (+ D if accumulate), bf16 operands, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// The same with tf32 operands (fp32 in shared memory, mantissa cut to 10 bits).
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// Completion of this thread's earlier MMAs arrives once on `bar`.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// All K steps of one bf16 GEMM: D[M x N] (+)= A[M x K] B[N x K]^T, K in elements (a multiple
// of 16), operands at their K offsets (bytes) ka0 / kb0.
__device__ __forceinline__ void umma_gemm_bf16(uint32_t d_tmem, const void *A, int arows, int ka0, const void *B,
                                               int brows, int kb0, int K, uint32_t idesc, bool accumulate) {
    // each step of 16 columns moves a descriptor's start address by two K chunks (rows * 32
    // bytes; the start field counts 16-byte units): the descriptors are built once and advanced
    uint64_t a = umma_desc(A, arows, ka0), b = umma_desc(B, brows, kb0);
    const uint64_t da = (uint64_t)(2 * arows), db = (uint64_t)(2 * brows);
    for (int k = 0; k < K; k += 16) {
        umma_bf16(d_tmem, a, b, idesc, accumulate || k > 0);
        a += da;
        b += db;
    }
}

// One bf16 operand of a GEMM: an array in the layout above with R rows, read K-major
// (operand rows = array rows from `mn0`, K = array columns from `k0`) or MN-major (operand
// rows = array columns from `mn0`, K = array rows from `k0`). Offsets in elements.
struct CmOp {
    const void *base;
    int R, mn0, k0;
    bool mn;
    __device__ __forceinline__ uint64_t desc(int k) const {
        return mn ? cm_mnmajor(base, R, k0 + k, mn0) : cm_kmajor(base, R, mn0, 2 * (k0 + k));
    }
};

// D[M x N] (+)= A B over K elements (a multiple of 16), bf16 operands in either orientation;
// the instruction descriptor must carry the same orientations.
__device__ __forceinline__ void umma_gemm(uint32_t d_tmem, const CmOp &A, const CmOp &B, int K, uint32_t idesc,
                                          bool accumulate) {
    // a step of 16 along K advances a K-major operand by two K chunks (R * 32 bytes) and an
    // MN-major one by two row groups (256 bytes); in the 16-byte units of the start field
    uint64_t a = A.desc(0), b = B.desc(0);
    const uint64_t da = A.mn ? 16u : (uint64_t)(2 * A.R), db = B.mn ? 16u : (uint64_t)(2 * B.R);
    for (int k = 0; k < K; k += 16) {
        umma_bf16(d_tmem, a, b, idesc, accumulate || k > 0);
        a += da;
        b += db;
    }
}

// One lane of a converged warp, chosen by elect.sync: true in that lane only. The warp issues
// tensor-core products through it (a product issued from a lone thread under `tid == 0` costs
// about 50-60 cycles of issue on this GPU, from an elected lane of a converged warp about 30).
__device__ __forceinline__ uint32_t elect_one_sync() {
    uint32_t p;
    asm volatile("{\n .reg .pred q;\n elect.sync _|q, 0xffffffff;\n selp.u32 %0, 1, 0, q;\n}" : "=r"(p));
    return p;
}

// D (tensor memory) = A B (+ D if accumulate), bf16 operands: executed by a whole converged warp
// (the descriptors are then warp-uniform), issued by the lane whose `lead` is nonzero.
__device__ __forceinline__ void umma_bf16_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            bool accumulate, uint32_t lead) {
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
        " @q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate), "r"(lead)
        : "memory");
}

// Completion of the `lead` lane's earlier products arrives once on `bar` (whole warp executes).
__device__ __forceinline__ void umma_commit_w(uint64_t *bar, uint32_t lead) {
    asm volatile(
        "{\n .reg .pred q;\n setp.ne.b32 q, %1, 0;\n"
        " @q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(smem_addr(bar)),
        "r"(lead)
        : "memory");
}

// umma_gemm for a whole converged warp, issued by its `lead` lane.
__device__ __forceinline__ void umma_gemm_w(uint32_t d_tmem, const CmOp &A, const CmOp &B, int K, uint32_t idesc,
                                            bool accumulate, uint32_t lead) {
    uint64_t a = A.desc(0), b = B.desc(0);
    const uint64_t da = A.mn ? 16u : (uint64_t)(2 * A.R), db = B.mn ? 16u : (uint64_t)(2 * B.R);
    for (int k = 0; k < K; k += 16) {
        umma_bf16_w(d_tmem, a, b, idesc, accumulate || k > 0, lead);
        a += da;
        b += db;
    }
}

// The same with B given by a descriptor and its step per 16 along K (in the start field's
// 16-byte units), e.g. a swizzled operand.
__device__ __forceinline__ void umma_gemm_wd(uint32_t d_tmem, const CmOp &A, uint64_t b, uint64_t db, int K,
                                             uint32_t idesc, bool accumulate, uint32_t lead) {
    uint64_t a = A.desc(0);
    const uint64_t da = A.mn ? 16u : (uint64_t)(2 * A.R);
    for (int k = 0; k < K; k += 16) {
        umma_bf16_w(d_tmem, a, b, idesc, accumulate || k > 0, lead);
        a += da;
        b += db;
    }
}

// 16x256b tensor-memory load, four repetitions (32 columns) from lane base `taddr` (a multiple of
// 16 within the warp's 32 lanes): thread t gets, for repetition j, v[4j], v[4j+1] = lane
// base + t/4, columns 8j + 2 (t % 4) and + 1, and v[4j+2], v[4j+3] = the same columns of lane
// base + 8 + t/4. Every thread of the warp holds data (a 32x32b load of an M = 64 accumulator
// leaves half of the threads idle).
__device__ __forceinline__ void tmem_ld16x256_x4(uint32_t taddr, float *v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]),
          "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15])
        : "r"(taddr)
        : "memory");
}

// Where a thread's values of an M = 64 accumulator of N columns lie when the 8 warps of a
// 256-thread CTA read it with 16x256b loads: warp w reads rows 16 (w % 4) .. + 15 (tensor-memory
// lanes 32 (w % 4) .. + 15) and columns [N/2 (w / 4), N/2 (w / 4 + 1)); value e = 4 j + k of the
// thread (j the 8-column repetition, k = 0..3) is row row(k) and column col(j, k).
struct M64Frag {
    int row0, colbase;
    __device__ __forceinline__ M64Frag(int warp, int lane, int N) {
        row0 = 16 * (warp & 3) + (lane >> 2);
        colbase = (N / 2) * (warp >> 2) + 2 * (lane & 3);
    }
    __device__ __forceinline__ int row(int k) const { return row0 + 8 * (k >> 1); }
    __device__ __forceinline__ int col(int j, int k) const { return colbase + 8 * j + (k & 1); }
};

// Two values as a bf16 pair (round to nearest even), the first in the low half.
__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// stmatrix m8n8.x4 (whole warp): four 8x8 matrices of 16-bit values to shared memory. Lane l
// gives the address of row l % 8 of matrix l / 8 (16 contiguous bytes) and holds, in r0..r3,
// row l / 4, columns 2 (l % 4) and + 1 of matrices 0..3: the layout in which an M64Frag holds
// a pair of values, so a fragment goes to any tile whose 8x8 blocks have 16-byte rows.
__device__ __forceinline__ void stmatrix_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0), "r"(r1),
                 "r"(r2), "r"(r3)
                 : "memory");
}

// The row address that `lane` gives to stmatrix_x4 for the M64Frag values of column blocks cb
// and cb + 1 (8 columns each) in an R-row core-matrix tile (shared-memory address `tile`), the
// warp's 16 rows starting at row16: matrices (cb, rows row16..+7), (cb, row16+8..+15),
// (cb + 1, row16..), (cb + 1, row16+8..) -- r0..r3 = the value pairs 4j, 4j+2, 4j+4, 4j+6.
__device__ __forceinline__ uint32_t frag_row_addr(uint32_t tile, int R, int row16, int cb, int lane) {
    const int m = lane >> 3;
    return tile + cm_off(row16 + 8 * (m & 1) + (lane & 7), 16 * (cb + (m >> 1)), R);
}

// 32x32b tensor-memory load of 16 consecutive columns.
__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]),
          "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st16f(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
        "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15])
        : "memory");
}

// 32x32b tensor-memory load/store of 32 consecutive columns (no wait: the caller issues
// several loads, then one tmem_wait_ld).
__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float *v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]),
          "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]),
          "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]),
          "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st32f(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
        "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]),
        "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]),
        "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
}

// Store bf16 value x at element (r, k) of a K-major bf16 operand with `rows` rows.
__device__ __forceinline__ void cm_put_bf16(unsigned char *base, int r, int k, int rows, float x) {
    *reinterpret_cast<__nv_bfloat16 *>(base + cm_off(r, 2 * k, rows)) = __float2bfloat16_rn(x);
}

}  // namespace gdn
