// libgdnspec: chunked prefill of the Gated DeltaNet layer on the sm_103a
// tensor cores (tcgen05).  The C entry point gdn_prefill_chunked (gdnspec.cu,
// declared in include/gdnspec.h) computes what gdn_prefill computes, in the
// chunked form whose bulk is dense products.
//
// Chunked form (C = 64 tokens; S the K x V state at the chunk start; G_t the
// running sum of the log-decays g inside the chunk; k^, q^ normalised rows):
//   A_ts = beta_t e^(G_t - G_s) (k^_t . k^_s)   for s < t       (C x C)
//   B_t  = beta_t (v_t - e^(G_t) S^T k^_t)
//   V'   = (I + A)^-1 B
//   o_t  = e^(G_t) S^T q^_t + sum_{s<=t} e^(G_t - G_s) (q^_t . k^_s) v'_s
//   S   <- e^(G_last) S + K~^T V',   K~_s = e^(G_last - G_s) k^_s
// This is the token recurrence S_t = e^(g_t) S_{t-1} + k^_t v'_t^T with
// v'_t = beta_t (v_t - (e^(g_t) S_{t-1})^T k^_t) and o_t = S_t^T q^_t, unrolled
// over the chunk: the same quantities in exact arithmetic.  All decay factors
// are e^(non-positive), so nothing overflows however strong the decay.
//
// Kernel (one CTA of 8 warps per (sequence, v-head) unit, or two, one CTA per SM):
//  * Products run on the tensor cores as 128-row tcgen05.mma (kind::f16: bf16
//    operands, FP32 accumulators) issued by one thread, at FP32 accuracy: every
//    operand x is carried as two bf16 terms, hi = bf16(x) and lo = bf16(x - hi)
//    (|x - hi - lo| <= 2^-18 |x|), and a product accumulates the hi.hi, lo.hi
//    and hi.lo terms in FP32 (the lo.lo term is below 2^-18).  Token tiles store
//    hi and lo side by side along K, so the tensor cores add the terms inside
//    the accumulator.
//  * The value column v is the row (tensor-memory lane) of every product that
//    involves the state: X^T = S^T K^^T, Y^T = S^T Q^^T, V'^T = B^T T^T (with
//    T = (I + A)^-1), S^T += V'^T K~ and O^T += V'^T R~^T.  Their 128 rows are
//    all live, and the per-column work after each product (B, the rescales,
//    the images) is spread over the four lane quadrants, that is over all four
//    SM sub-partitions.  The two token products P = K^ K^^T and R = Q^ K^^T
//    form one 128-row product [K^; Q^] K^^T: lanes 0-63 hold P, lanes 64-127 R.
//    Tensor-memory columns:
//      0- 63 [P; R]     64-127 X^T     128-191 Y^T, then O^T     192-255 V'^T
//      256-383 S^T (FP32, carried over the whole prompt)
//  * T = (I + A)^-1 is formed on CUDA cores in FP32 by blocks: the four 16 x 16
//    diagonal blocks by substitution, one thread per column, then the
//    off-diagonal blocks by doubling (T_10 = -T_11 A_10 T_00 at 16 and then at
//    32 rows), each a small dense product spread over the threads.
//  * With fewer (sequence, v-head) units than half the SMs, a unit's 128 value
//    columns are split over a 2-CTA cluster (64 each): the recurrence of a
//    value column involves no other column, and the RMSNorm's sums of squares
//    are exchanged through distributed shared memory once per chunk.
//  * Every wait on the tensor cores is bounded.  On a timeout the CTA sets
//    GDN_FLAG_TIMEOUT, writes no final state, waits (bounded) for the MMAs in
//    flight and releases its tensor memory; a lone CTA stops at once, a
//    2-CTA unit runs its remaining chunks (their outputs are not valid) so
//    that both CTAs meet at every cluster barrier.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "gdn_internal.h"
#include "gdnspec.h"

namespace cg = cooperative_groups;

namespace {

using gdn_internal::Params;

constexpr int kK = 128;
constexpr int kV = 128;
constexpr int kC = 64;                          // tokens per chunk
constexpr int kThreads = 256;
constexpr float kQkEps = 1e-6f;                 // inside the L2-norm square root
constexpr float kSoftplusThreshold = 20.0f;     // softplus(x) = x above this
constexpr uint32_t kSpinLimit = 1u << 24;       // try_wait polls before giving up (well over 1 s)

// ---- shared memory (offsets from a 1024-byte aligned base) ----------------------
// 128-byte-swizzled K-major bf16 tiles (the canonical SWIZZLE_128B layout):
// a tile of R rows is stored in atom columns of 64 elements; element (r, c)
// sits at (c / 64) * R * 128 + r * 128 + (((c % 64) / 8) ^ (r % 8)) * 16 + (c % 8) * 2.
// A CTA owns VC of the unit's 128 value columns (128, or 64 with the unit over
// a 2-CTA cluster).  Regions are reused once the products that read them have
// completed:
//   region 1  S^T hi | lo   [VC v][128 kd] each         (read by the first products)
//             then B^T hi | lo [VC v][64 s] at its start, V'^T hi | lo in their place,
//             and K~^T hi | lo [128 kd][64 t] in its second half
//   region 2  [K^; Q^]      [128 rows][hi 128 | lo 128 kd]
//             then the chunk's outputs, FP32 [64 t][VC + 4]
//   kVT       v^T FP32 [VC v][65], then T FP32 [64][68] and T hi | lo [64 t][64 s]
//   kA        A^T FP32 [64 s][68 t]
//   kRt       R~ [64 t][hi 64 | lo 64 s]
//   kM        FP32 products of the doubling steps (2 x [16][16], then [32][32])
//   kZ        raw z, bf16 quads [64 t][VC / 4 + 1]
// A 128-row product over a 64-row A tile (VC = 64) reads 8 KB past each atom
// column; every such read stays inside region 1 and lands in unread lanes.
template <int VC>
struct Layout {
    static constexpr int kImg = VC * kK * 2;                   // one state image
    static constexpr int kSHi = 0, kSLo = kImg;
    static constexpr int kBHi = 0, kBLo = VC * 128;            // B^T, then V'^T: one atom column each
    static constexpr int kKtHi = 32768, kKtLo = 49152;         // K~^T
    static constexpr int kKQ = 65536;                          // [K^; Q^], atom columns of 16 KB
    static constexpr int kKQLo = kKQ + 32768;                  // its lo half (columns 128-255)
    static constexpr int kStage = kKQ;
    static constexpr int kStagePitch = VC + 4;
    static constexpr int kVT = 131072;
    static constexpr int kVTPitch = kC + 1;                    // odd pitch: column walks are conflict-free
    static constexpr int kT = kVT;
    static constexpr int kTPitch = 68;
    static constexpr int kTHi = kVT + 17408, kTLo = kTHi + 8192;
    static constexpr int kA = kVT + 33792;
    static constexpr int kAPitch = 68;
    static constexpr int kRt = kA + 17408;
    static constexpr int kM = kRt + 16384;
    static constexpr int kZ = kM + 4096;
    static constexpr int kZStride = VC / 4 + 1;                // uint2 per padded z row
    static constexpr int kMisc = (kZ + kC * kZStride * 8 + 15) / 16 * 16;
    static_assert(2 * kImg <= 65536 && kKtHi >= 2 * VC * 128, "region 1");
    static_assert(kC * kStagePitch * 4 <= 65536, "the output rows fit region 2");
    static_assert(VC * kVTPitch * 4 <= 33792 && kTLo + 8192 <= kVT + 33792, "v^T and T share a region");
    static_assert(64 * kTPitch * 4 <= 17408 && kTHi % 1024 == 0, "T");
    static_assert(kRt % 1024 == 0, "R~ tile alignment");
};

struct Misc {
    float G[kC], g[kC], beta[kC], eG[kC], kfac[kC];            // G 16-byte aligned (float4 reads)
    float ssq_cta[2][kC];                       // with a 2-CTA unit: this CTA's sums of squares, read
                                                // by its peer (indexed by chunk parity)
    float wn[kV];                               // norm_w of this CTA's columns
    int row[kC];
    unsigned long long bar;                     // MMA completion barrier
    unsigned long long drain;                   // completion of every MMA issued, after a timeout
    uint32_t tmem;                              // tensor-memory base column
    float gamma;                                // e^(G_last) of the current chunk
};
template <int VC>
constexpr int smem_bytes() { return Layout<VC>::kMisc + static_cast<int>(sizeof(Misc)) + 1024; }   // + alignment
static_assert(smem_bytes<128>() <= 227 * 1024 && smem_bytes<64>() <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ uint32_t swz(int r, int c, int R) {
    return static_cast<uint32_t>((c >> 6) * R * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}
// the 16-byte chunk holding elements 8j .. 8j+7 of row r
__device__ __forceinline__ uint32_t swz_chunk(int r, int j, int R) {
    return static_cast<uint32_t>((j >> 3) * R * 128 + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// (a, b) -> bf16 hi pair and the bf16 pair of the remainders x - hi (the
// remainder of a round-to-nearest bf16 is exact in FP32)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}
// 8 values -> the 16-byte chunks of their hi and lo parts
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
    split2(x[0], x[1], hi.x, lo.x);
    split2(x[2], x[3], hi.y, lo.y);
    split2(x[4], x[5], hi.z, lo.z);
    split2(x[6], x[7], hi.w, lo.w);
}

// ---- tcgen05 / mbarrier ---------------------------------------------------------------
__device__ __forceinline__ uint32_t saddr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// shared-memory matrix descriptor: SWIZZLE_128B, K-major, 8-row groups 1024 B apart
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
    return static_cast<uint64_t>((addr & 0x3FFFF) >> 4) | (static_cast<uint64_t>(16 >> 4) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// kind::f16 instruction descriptor: FP32 D, bf16 A and B, both K-major
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// D[128][N] (+)= A[128][K] B[N][K]^T over K = 16-element steps; A and B are
// swizzled K-major tiles of a_rows / b_rows rows
__device__ __forceinline__ void gemm(uint32_t d, uint32_t a_tile, int a_rows, uint32_t b_tile, int b_rows, int N,
                                     int K, bool accumulate) {
    const uint32_t idesc = idesc_bf16(128, N);
    for (int ks = 0; ks < K / 16; ++ks) {
        const uint32_t oa = (ks >> 2) * a_rows * 128 + (ks & 3) * 32;
        const uint32_t ob = (ks >> 2) * b_rows * 128 + (ks & 3) * 32;
        mma_bf16(d, desc_sw128(a_tile + oa), desc_sw128(b_tile + ob), idesc, (accumulate || ks > 0) ? 1u : 0u);
    }
}

// D[128][N] (+)= A B^T at FP32 accuracy from hi / lo parts: the hi.hi, lo.hi
// and hi.lo terms over K.  a_hi / a_lo and b_hi / b_lo are the tiles (or the
// column halves of one tile) holding the parts; a_rows / b_rows their row
// counts (the stride between atom columns).
__device__ __forceinline__ void gemm_split(uint32_t d, uint32_t a_hi, uint32_t a_lo, int a_rows, uint32_t b_hi,
                                           uint32_t b_lo, int b_rows, int N, int K, bool accumulate) {
    gemm(d, a_hi, a_rows, b_hi, b_rows, N, K, accumulate);
    gemm(d, a_lo, a_rows, b_hi, b_rows, N, K, true);
    gemm(d, a_hi, a_rows, b_lo, b_rows, N, K, true);
}

__device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ bool wait_parity(uint32_t bar, uint32_t parity, uint32_t limit) {
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred P;\n\tmbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, P;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// the same wait with non-blocking polls (mbarrier.test_wait): a bound set by
// gdn_set_wait_limit counts these, so that a small bound runs out for certain
__device__ __forceinline__ bool test_parity(uint32_t bar, uint32_t parity, uint32_t limit) {
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred P;\n\tmbarrier.test_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, P;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// a wait on the MMA barrier: blocking polls up to the default bound, or
// non-blocking ones up to a bound set by gdn_set_wait_limit
__device__ __forceinline__ bool wait_mma(uint32_t bar, uint32_t parity, uint32_t limit) {
    return limit == 0 ? wait_parity(bar, parity, kSpinLimit) : test_parity(bar, parity, limit);
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes become visible to the tensor cores
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// all threads: shared-memory operands written, tensor-memory accesses done
__device__ __forceinline__ void sync_for_mma() {
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
}

// 32 consecutive FP32 columns of this thread's TMEM lane
__device__ __forceinline__ void tm_ld32(uint32_t taddr, float (&x)[32]) {
    uint32_t r[32];
    __syncwarp();
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tm_st32(uint32_t taddr, const float (&x)[32]) {
    __syncwarp();
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(x[0])), "r"(__float_as_uint(x[1])), "r"(__float_as_uint(x[2])),
        "r"(__float_as_uint(x[3])), "r"(__float_as_uint(x[4])), "r"(__float_as_uint(x[5])),
        "r"(__float_as_uint(x[6])), "r"(__float_as_uint(x[7])), "r"(__float_as_uint(x[8])),
        "r"(__float_as_uint(x[9])), "r"(__float_as_uint(x[10])), "r"(__float_as_uint(x[11])),
        "r"(__float_as_uint(x[12])), "r"(__float_as_uint(x[13])), "r"(__float_as_uint(x[14])),
        "r"(__float_as_uint(x[15])), "r"(__float_as_uint(x[16])), "r"(__float_as_uint(x[17])),
        "r"(__float_as_uint(x[18])), "r"(__float_as_uint(x[19])), "r"(__float_as_uint(x[20])),
        "r"(__float_as_uint(x[21])), "r"(__float_as_uint(x[22])), "r"(__float_as_uint(x[23])),
        "r"(__float_as_uint(x[24])), "r"(__float_as_uint(x[25])), "r"(__float_as_uint(x[26])),
        "r"(__float_as_uint(x[27])), "r"(__float_as_uint(x[28])), "r"(__float_as_uint(x[29])),
        "r"(__float_as_uint(x[30])), "r"(__float_as_uint(x[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- element helpers --------------------------------------------------------------------
__device__ __forceinline__ void unpack4(uint2 raw, float (&x)[4]) {
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    x[0] = lo.x;
    x[1] = lo.y;
    x[2] = hi.x;
    x[3] = hi.y;
}

// one state element <-> FP32 (the slot may be read and written by the same
// CTA, so no read-only loads); stores round to nearest even
__device__ __forceinline__ float load_elem(const float* p) { return __ldcs(p); }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load_elem(const __half* p) { return __half2float(*p); }
__device__ __forceinline__ void store_elem(float* p, float x) { __stcs(p, x); }
__device__ __forceinline__ void store_elem(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void store_elem(__half* p, float x) { *p = __float2half_rn(x); }

// d[u] = e^(Gt - G[u]) for 32 consecutive entries of G (16-byte aligned)
__device__ __forceinline__ void load_decays(const float* G, float Gt, float (&d)[32]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 g4 = reinterpret_cast<const float4*>(G)[j];
        d[4 * j] = __expf(Gt - g4.x);
        d[4 * j + 1] = __expf(Gt - g4.y);
        d[4 * j + 2] = __expf(Gt - g4.z);
        d[4 * j + 3] = __expf(Gt - g4.w);
    }
}

// silu(z) = z sigmoid(z); for very negative z the denominator overflows and
// the fast division returns zero
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// C[r][c0 .. c0+3] = sum_{q < Q} X(r, q) Y[q][c0 .. c0+3]: X read one element at
// a time through xat(q), Y a row-major FP32 block read as float4
template <int Q, typename XAt>
__device__ __forceinline__ float4 rowdot4(XAt xat, const float* y, int y_pitch) {
    float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const float x = xat(q);
        const float4 b = *reinterpret_cast<const float4*>(y + q * y_pitch);
        c.x = fmaf(x, b.x, c.x);
        c.y = fmaf(x, b.y, c.y);
        c.z = fmaf(x, b.z, c.z);
        c.w = fmaf(x, b.w, c.w);
    }
    return c;
}

// ---- the kernel -------------------------------------------------------------------------
//
// Per chunk (quadrant q = warp % 4 reaches TMEM lanes 32q .. 32q + 31; the two
// warps of a quadrant, hh = warp / 4, split the columns of each row; "column
// lanes" are the lanes v < VC):
//   phase 1  all warps      k^, q^ (hi | lo) into [K^; Q^], v^T, raw z, gates
//   MMA 1                   [P; R] = [K^; Q^] K^^T,  X^T = S^T K^^T,  Y^T = S^T Q^^T
//                           (meanwhile warp 0: the running sum G and its exponentials)
//   phase 2  lanes 0-63     A^T from P              lanes 64-127   R~ (hi | lo) from R
//            column lanes   B^T (hi | lo) = beta (v^T - e^G X^T);  O^T = e^G Y^T;  S^T <- e^(G_last) S^T
//   phase 3  T = (I + A)^-1 by blocks; K~^T (hi | lo) meanwhile; T (hi | lo)
//   MMA 2                   V'^T = B^T T^T
//   phase 4  column lanes   V'^T (hi | lo)
//   MMA 3                   S^T += V'^T K~,  O^T += V'^T R~^T  (meanwhile the next chunk's loads)
//   phase 5  column lanes   O^T into the output rows (FP32); the state images
//            all warps      the gated RMSNorm of 8 rows each, the rows to memory
template <typename StateT, int VC>
__global__ void __launch_bounds__(kThreads, 1) gdn_prefill_chunked_kernel(const Params p) {
    using Lay = Layout<VC>;
    constexpr int CL = kV / VC;                                 // CTAs per unit
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
    Misc& ms = *reinterpret_cast<Misc*>(sm + Lay::kMisc);
    float* VT = reinterpret_cast<float*>(sm + Lay::kVT);
    float* Tm = reinterpret_cast<float*>(sm + Lay::kT);
    float* At = reinterpret_cast<float*>(sm + Lay::kA);
    float* Mb = reinterpret_cast<float*>(sm + Lay::kM);
    float* Stage = reinterpret_cast<float*>(sm + Lay::kStage);
    uint2* Zq = reinterpret_cast<uint2*>(sm + Lay::kZ);
    const uint32_t sbase = saddr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3;                                  // TMEM lane quadrant of this warp
    const int hh = warp >> 2;                                   // which half of a row's columns
    const uint32_t lanes = static_cast<uint32_t>(quad * 32) << 16;
    const int row = quad * 32 + lane;                           // this thread's TMEM lane
    const bool col_lane = quad * 32 < VC;                       // lane v holds value column v
    const int rank = CL > 1 ? static_cast<int>(blockIdx.x % CL) : 0;
    const int unit = static_cast<int>(blockIdx.x / CL);
    const int cb = rank * VC;                                   // this CTA's first value column
    const int i = unit / p.H_v;
    const int h = unit - i * p.H_v;
    const int kh = h / p.group;
    const bool gated = p.z != nullptr;

    const int bos = __ldg(p.cu + i);
    const int L = __ldg(p.cu + i + 1) - bos;
    const long long rs = __ldg(p.read_slots + i);
    const long long wsl = __ldg(p.write_slots + i);
    // (every CTA of a unit takes the same exits)
    if (L <= 0) return;
    if (bos < 0 || bos + L > p.num_tokens) {
        if (tid == 0 && rank == 0 && p.status) atomicOr(p.status, GDN_FLAG_TOKEN_ROW);
        return;
    }
    if (rs >= p.num_slots || wsl >= p.num_slots) {
        if (tid == 0 && rank == 0 && p.status) atomicOr(p.status, GDN_FLAG_SLOT_RANGE);
        return;
    }

    // ---- set-up: all 512 TMEM columns, the barriers, the norm weight ----
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(saddr(&ms.tmem)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&ms.bar)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&ms.drain)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (gated && tid < VC) ms.wn[tid] = __bfloat162float(p.norm_w[cb + tid]);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tm = ms.tmem;
    const uint32_t tPR = tm, tX = tm + 64, tO = tm + 128, tVp = tm + 192, tS = tm + 256;
    const uint32_t bar = saddr(&ms.bar);
    uint32_t phase = 0;
    bool ok = true;
    const uint32_t limit = p.wait_limit;                       // 0: the default bound

    // hi and lo images of 32 FP32 state values (kd0 .. kd0 + 31 of row v)
    auto put_images = [&](int v, int kd0, const float (&x)[32]) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 hi, lo;
            split8(x + 8 * j, hi, lo);
            *reinterpret_cast<uint4*>(sm + Lay::kSHi + swz_chunk(v, (kd0 >> 3) + j, VC)) = hi;
            *reinterpret_cast<uint4*>(sm + Lay::kSLo + swz_chunk(v, (kd0 >> 3) + j, VC)) = lo;
        }
    };
    // 32 FP32 values of a [rows][64] operand row r, columns c0 .. c0 + 31, as
    // its hi and lo tiles
    auto put_row64 = [&](uint32_t hi_off, uint32_t lo_off, int r, int rows, int c0, const float (&x)[32]) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 hi, lo;
            split8(x + 8 * j, hi, lo);
            *reinterpret_cast<uint4*>(sm + hi_off + swz_chunk(r, (c0 >> 3) + j, rows)) = hi;
            *reinterpret_cast<uint4*>(sm + lo_off + swz_chunk(r, (c0 >> 3) + j, rows)) = lo;
        }
    };
    // bounded wait on the MMA barrier; a lone CTA stops at a timeout, a 2-CTA
    // unit records it and goes on (its CTAs meet at a cluster barrier every chunk)
    auto wait_products = [&]() -> bool {
        const bool done = wait_mma(bar, phase, limit);
        const bool late = __syncthreads_or(!done);
        phase ^= 1;
        if (late) ok = false;
        fence_after();
        return CL == 1 && late;
    };

    // ---- initial state: S^T (FP32) into TMEM lane v, its images into region 1.
    //      Thread (v, hh) covers kd in [64 hh, 64 hh + 64); a warp reads 32
    //      consecutive v of one kd row per load. ----
    if (col_lane) {
        const StateT* src = rs >= 0 ? static_cast<const StateT*>(p.pool) +
                                          (rs * p.H_v + h) * static_cast<int64_t>(kK * kV) + cb + row
                                    : nullptr;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int kd0 = 64 * hh + 32 * c;
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = src ? load_elem(src + (kd0 + j) * kV) : 0.f;
            tm_st32(tS + lanes + kd0, x);
            put_images(row, kd0, x);
        }
    }

    // Raw inputs of a chunk, 8 tokens per warp: q, k rows as bf16 quads, z quads
    // of this CTA's columns, v one element per lane per load (v = cb + lane +
    // 32 e, so that its transposed store hits 32 distinct banks), a / b bits in
    // lanes 0-15 (converted only in phase 1, so that nothing waits on the loads
    // before then).  The next chunk's loads are issued while the last products
    // of the current one run.
    constexpr int VE = VC / 32;                                  // v elements per lane
    uint2 qraw[8], kraw[8], zraw[8];
    __nv_bfloat16 vraw[8][VE];
    unsigned short ab_raw;                                      // lane j: a of token j, lane 8 + j: its b
    auto load_chunk = [&](int cs) {
        const int nn = min(kC, L - cs);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int t = warp + 8 * j;
            qraw[j] = kraw[j] = zraw[j] = make_uint2(0, 0);
#pragma unroll
            for (int e = 0; e < VE; ++e) vraw[j][e] = __float2bfloat16_rn(0.f);
            if (t < nn) {
                const int64_t r = bos + cs + t;
                qraw[j] = __ldg(reinterpret_cast<const uint2*>(p.q + r * p.q_stride + kh * kK) + lane);
                kraw[j] = __ldg(reinterpret_cast<const uint2*>(p.k + r * p.k_stride + kh * kK) + lane);
#pragma unroll
                for (int e = 0; e < VE; ++e) vraw[j][e] = p.v[r * p.v_stride + h * kV + cb + lane + 32 * e];
                if (gated && lane < VC / 4)
                    zraw[j] = __ldg(reinterpret_cast<const uint2*>(p.z + r * p.z_stride + h * kV + cb) + lane);
            }
        }
        ab_raw = 0;
        if (lane < 16 && warp + 8 * (lane & 7) < nn) {
            const int64_t r = bos + cs + warp + 8 * (lane & 7);
            ab_raw = __bfloat16_as_ushort(lane < 8 ? p.a[r * p.a_stride + h] : p.b[r * p.b_stride + h]);
        }
    };
    load_chunk(0);

    for (int c0 = 0; c0 < L; c0 += kC) {
        const int n = min(kC, L - c0);
        const int cpar = (c0 / kC) & 1;                          // chunk parity
        const bool more = c0 + kC < L;

        // ---- phase 1: per token (8 per warp) k^ and q^ (hi | lo) into [K^; Q^],
        //      v into v^T, raw z, gates ----
        {
            const float ab = __uint_as_float(static_cast<uint32_t>(ab_raw) << 16);
            const float b_in = __shfl_down_sync(0xffffffffu, ab, 8);
            const int t = warp + 8 * lane;
            if (lane < 8) {
                float g = 0.f, beta = 0.f;
                if (t < n) {
                    const float x = ab + __bfloat162float(p.dt_bias[h]);
                    const float sp = x > kSoftplusThreshold ? x : log1pf(expf(x));
                    g = -expf(__ldg(p.A_log + h)) * sp;
                    beta = 1.0f / (1.0f + expf(-b_in));
                    ms.row[t] = bos + c0 + t;
                }
                ms.g[t] = g;
                ms.beta[t] = beta;
            }
        }
        {
            // squared norms of the 8 q and 8 k rows, reduced together
            float sums[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float qv[4], kv[4];
                unpack4(qraw[j], qv);
                unpack4(kraw[j], kv);
                sums[j] = qv[0] * qv[0] + qv[1] * qv[1] + qv[2] * qv[2] + qv[3] * qv[3];
                sums[8 + j] = kv[0] * kv[0] + kv[1] * kv[1] + kv[2] * kv[2] + kv[3] * kv[3];
            }
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
                for (int j = 0; j < 16; ++j) sums[j] += __shfl_xor_sync(0xffffffffu, sums[j], m);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = warp + 8 * j;
                uint2 khi = make_uint2(0, 0), klo = khi, qhi = khi, qlo = khi;
                if (t < n) {
                    float qv[4], kv[4];
                    unpack4(qraw[j], qv);
                    unpack4(kraw[j], kv);
                    if (gated && lane < VC / 4) Zq[t * Lay::kZStride + lane] = zraw[j];   // the gate's input, exact
                    const float rq = rsqrtf(sums[j] + kQkEps) * p.scale;
                    const float rk = rsqrtf(sums[8 + j] + kQkEps);
                    split2(kv[0] * rk, kv[1] * rk, khi.x, klo.x);
                    split2(kv[2] * rk, kv[3] * rk, khi.y, klo.y);
                    split2(qv[0] * rq, qv[1] * rq, qhi.x, qlo.x);
                    split2(qv[2] * rq, qv[3] * rq, qhi.y, qlo.y);
#pragma unroll
                    for (int e = 0; e < VE; ++e) VT[(lane + 32 * e) * Lay::kVTPitch + t] = __bfloat162float(vraw[j][e]);
                }
                *reinterpret_cast<uint2*>(sm + Lay::kKQ + swz(t, lane * 4, 128)) = khi;
                *reinterpret_cast<uint2*>(sm + Lay::kKQ + swz(t, kK + lane * 4, 128)) = klo;
                *reinterpret_cast<uint2*>(sm + Lay::kKQ + swz(64 + t, lane * 4, 128)) = qhi;
                *reinterpret_cast<uint2*>(sm + Lay::kKQ + swz(64 + t, kK + lane * 4, 128)) = qlo;
            }
        }
        sync_for_mma();

        // ---- MMA 1: [P; R] = [K^; Q^] K^^T and [X^T | Y^T] = S^T [K^; Q^]^T
        //      (hi.hi + lo.hi + hi.lo each) ----
        if (tid == 0) {
            const uint32_t kqH = sbase + Lay::kKQ, kqL = sbase + Lay::kKQLo;
            const uint32_t sH = sbase + Lay::kSHi, sL = sbase + Lay::kSLo;
            gemm_split(tPR, kqH, kqL, 128, kqH, kqL, 128, 64, kK, false);
            gemm_split(tX, sH, sL, VC, kqH, kqL, 128, 128, kK, false);              // [X^T | Y^T]
            commit(bar);
        }
        if (warp == 0) {
            // while the products run: G = inclusive running sum of g; e^(G_t),
            // e^(G_last - G_t), e^(G_last)
            const float g0 = ms.g[2 * lane], g1 = ms.g[2 * lane + 1];
            float s = g0 + g1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            ms.G[2 * lane] = s - g1;
            ms.G[2 * lane + 1] = s;
            __syncwarp();
            const float G_last = ms.G[n - 1];
            if (lane == 0) ms.gamma = expf(G_last);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = lane + 32 * e;
                ms.eG[t] = expf(ms.G[t]);
                ms.kfac[t] = t < n ? expf(G_last - ms.G[t]) : 0.f;
            }
        }
        if (wait_products()) break;

        // ---- phase 2 ----
        {
            // K~^T [kd][t] = k^_t[kd] e^(G_last - G_t) (k^ = hi + lo): thread
            // (j = warp, kd4 = 4 lane) forms the 16-byte chunk j (8 tokens) of rows
            // kd4 .. kd4 + 3, hi and lo
            const int kd4 = 4 * lane, j = warp;
            float x[4][8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = 8 * j + u;
                float hv[4], lv[4];
                unpack4(*reinterpret_cast<const uint2*>(sm + Lay::kKQ + swz(t, kd4, 128)), hv);
                unpack4(*reinterpret_cast<const uint2*>(sm + Lay::kKQ + swz(t, kK + kd4, 128)), lv);
                const float f = ms.kfac[t];
#pragma unroll
                for (int c = 0; c < 4; ++c) x[c][u] = (hv[c] + lv[c]) * f;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint4 hi, lo;
                split8(x[c], hi, lo);
                *reinterpret_cast<uint4*>(sm + Lay::kKtHi + swz_chunk(kd4 + c, j, 128)) = hi;
                *reinterpret_cast<uint4*>(sm + Lay::kKtLo + swz_chunk(kd4 + c, j, 128)) = lo;
            }
        }
        {
            // token rows of [P; R]: this warp's 32 columns s0 .. s0 + 31
            const int t = row & 63;
            const int s0 = 32 * hh;
            const float Gt = ms.G[t];
            const bool live = t < n;
            float x[32], d[32];
            load_decays(ms.G + s0, Gt, d);
            tm_ld32(tPR + lanes + s0, x);
            if (quad < 2) {
                // A (s < t), stored transposed: A^T[s][t]
                const float bt = ms.beta[t];
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int s = s0 + u;
                    At[s * Lay::kAPitch + t] = (live && s < t) ? bt * d[u] * x[u] : 0.f;
                }
            } else {
                // R~ (s <= t), hi | lo
#pragma unroll
                for (int u = 0; u < 32; ++u) x[u] = (live && s0 + u <= t) ? d[u] * x[u] : 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 hi, lo;
                    split8(x + 8 * j, hi, lo);
                    *reinterpret_cast<uint4*>(sm + Lay::kRt + swz_chunk(t, (s0 >> 3) + j, kC)) = hi;
                    *reinterpret_cast<uint4*>(sm + Lay::kRt + swz_chunk(t, 8 + (s0 >> 3) + j, kC)) = lo;
                }
            }
        }
        if (col_lane) {
            // value column v = row: tokens t0 .. t0 + 31
            const int v = row;
            const int t0 = 32 * hh;
            float x[32];
            // B^T = beta (v^T - e^G X^T), hi | lo
            tm_ld32(tX + lanes + t0, x);
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4) {
                const float4 b4 = *reinterpret_cast<const float4*>(ms.beta + t0 + 4 * u4);
                const float4 e4 = *reinterpret_cast<const float4*>(ms.eG + t0 + 4 * u4);
                const float bb[4] = {b4.x, b4.y, b4.z, b4.w}, ee[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int u = 4 * u4 + e;
                    x[u] = (t0 + u < n) ? bb[e] * (VT[v * Lay::kVTPitch + t0 + u] - ee[e] * x[u]) : 0.f;
                }
            }
            put_row64(Lay::kBHi, Lay::kBLo, v, VC, t0, x);
            // O^T <- e^G Y^T
            tm_ld32(tO + lanes + t0, x);
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4) {
                const float4 e4 = *reinterpret_cast<const float4*>(ms.eG + t0 + 4 * u4);
                x[4 * u4] *= e4.x;
                x[4 * u4 + 1] *= e4.y;
                x[4 * u4 + 2] *= e4.z;
                x[4 * u4 + 3] *= e4.w;
            }
            tm_st32(tO + lanes + t0, x);
            // S^T <- e^(G_last) S^T, this half of the kd columns
            const float gamma = ms.gamma;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint32_t col = tS + lanes + 64 * hh + 32 * c;
                tm_ld32(col, x);
#pragma unroll
                for (int u = 0; u < 32; ++u) x[u] *= gamma;
                tm_st32(col, x);
            }
        }
        fence_before();
        __syncthreads();
        fence_after();

        // ---- phase 3: T = (I + A)^-1.  (a) the diagonal 16 x 16 blocks, thread
        //      (b, c) of warps 0-1 substituting column c of block b; meanwhile the
        //      other warps zero T's upper blocks ----
        if (tid < 64) {
            const int b = tid >> 4, c = tid & 15;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = r == c ? 1.f : 0.f;
            const float* arow = At + (16 * b) * Lay::kAPitch + 16 * b;
#pragma unroll
            for (int k = 0; k < 15; ++k) {
                // x_r -= A[r][k] x_k for r > k (A^T[k][r] is zero for r <= k)
                const float nxk = -x[k];
#pragma unroll
                for (int r4 = k / 4; r4 < 4; ++r4) {
                    const float4 a4 = *reinterpret_cast<const float4*>(arow + k * Lay::kAPitch + 4 * r4);
                    x[4 * r4 + 0] = fmaf(a4.x, nxk, x[4 * r4 + 0]);
                    x[4 * r4 + 1] = fmaf(a4.y, nxk, x[4 * r4 + 1]);
                    x[4 * r4 + 2] = fmaf(a4.z, nxk, x[4 * r4 + 2]);
                    x[4 * r4 + 3] = fmaf(a4.w, nxk, x[4 * r4 + 3]);
                }
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Tm[(16 * b + r) * Lay::kTPitch + 16 * b + c] = x[r];
        } else {
            const int w = tid - 64;                             // 0 .. 191
            // the six 16 x 16 blocks above the diagonal
            for (int e = w; e < 6 * 256; e += 192) {
                const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
                const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
                const int bj = blk < 3 ? 1 + blk : (blk < 5 ? blk - 1 : 3);
                Tm[(16 * bi + r) * Lay::kTPitch + 16 * bj + c] = 0.f;
            }
        }
        __syncthreads();
        // (b) 16-row doubling: for J = 0, 1 (blocks b0 = 2J, b1 = 2J + 1)
        //     M_J = A_{b1 b0} T_{b0 b0}, then T_{b1 b0} = -T_{b1 b1} M_J
        if (tid < 128) {
            const int J = tid >> 6, r = (tid >> 2) & 15, c4 = 4 * (tid & 3);
            const int b0 = 16 * (2 * J), b1 = b0 + 16;
            const float4 m = rowdot4<16>([&](int q) { return At[(b0 + q) * Lay::kAPitch + b1 + r]; },
                                         Tm + b0 * Lay::kTPitch + b0 + c4, Lay::kTPitch);
            *reinterpret_cast<float4*>(Mb + J * 256 + r * 16 + c4) = m;
        }
        __syncthreads();
        if (tid < 128) {
            const int J = tid >> 6, r = (tid >> 2) & 15, c4 = 4 * (tid & 3);
            const int b0 = 16 * (2 * J), b1 = b0 + 16;
            const float4 m = rowdot4<16>([&](int q) { return Tm[(b1 + r) * Lay::kTPitch + b1 + q]; },
                                         Mb + J * 256 + c4, 16);
            *reinterpret_cast<float4*>(Tm + (b1 + r) * Lay::kTPitch + b0 + c4) = make_float4(-m.x, -m.y, -m.z, -m.w);
        }
        __syncthreads();
        // (c) 32-row doubling: M = A[32..63][0..31] T[0..31][0..31], then
        //     T[32..63][0..31] = -T[32..63][32..63] M.  Thread (r2, c4, hq): rows
        //     2 r2 and 2 r2 + 1, columns c4 .. c4 + 3, over q in [16 hq, 16 hq + 16);
        //     the two halves of q are added across neighbouring lanes.
        {
            const int hq = tid & 1, r2 = 2 * (tid >> 4), c4 = 4 * ((tid >> 1) & 7);
            float acc[2][4] = {};
#pragma unroll
            for (int qq = 0; qq < 16; ++qq) {
                const int q = 16 * hq + qq;
                const float2 a = *reinterpret_cast<const float2*>(At + q * Lay::kAPitch + 32 + r2);
                const float4 b = *reinterpret_cast<const float4*>(Tm + q * Lay::kTPitch + c4);
                const float av[2] = {a.x, a.y}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int i2 = 0; i2 < 2; ++i2)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[i2][c] = fmaf(av[i2], bv[c], acc[i2][c]);
            }
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[i2][c] += __shfl_xor_sync(0xffffffffu, acc[i2][c], 1);
            float m[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) m[c] = hq ? acc[1][c] : acc[0][c];
            *reinterpret_cast<float4*>(Mb + (r2 + hq) * 32 + c4) = make_float4(m[0], m[1], m[2], m[3]);
        }
        __syncthreads();
        {
            const int hq = tid & 1, r2 = 2 * (tid >> 4), c4 = 4 * ((tid >> 1) & 7);
            float acc[2][4] = {};
#pragma unroll
            for (int qq = 0; qq < 16; ++qq) {
                const int q = 16 * hq + qq;
                const float a0 = Tm[(32 + r2) * Lay::kTPitch + 32 + q];
                const float a1 = Tm[(33 + r2) * Lay::kTPitch + 32 + q];
                const float4 b = *reinterpret_cast<const float4*>(Mb + q * 32 + c4);
                const float av[2] = {a0, a1}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int i2 = 0; i2 < 2; ++i2)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[i2][c] = fmaf(av[i2], bv[c], acc[i2][c]);
            }
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[i2][c] += __shfl_xor_sync(0xffffffffu, acc[i2][c], 1);
            float m[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) m[c] = hq ? acc[1][c] : acc[0][c];
            *reinterpret_cast<float4*>(Tm + (32 + r2 + hq) * Lay::kTPitch + c4) =
                make_float4(-m[0], -m[1], -m[2], -m[3]);
        }
        __syncthreads();
        // (d) T hi | lo tiles [64 t][64 s]
#pragma unroll
        for (int e = tid; e < kC * 8; e += kThreads) {
            const int t = e >> 3, j = e & 7;
            const float4 a = *reinterpret_cast<const float4*>(Tm + t * Lay::kTPitch + 8 * j);
            const float4 b = *reinterpret_cast<const float4*>(Tm + t * Lay::kTPitch + 8 * j + 4);
            const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint4 hi, lo;
            split8(x, hi, lo);
            *reinterpret_cast<uint4*>(sm + Lay::kTHi + swz_chunk(t, j, kC)) = hi;
            *reinterpret_cast<uint4*>(sm + Lay::kTLo + swz_chunk(t, j, kC)) = lo;
        }
        sync_for_mma();

        // ---- MMA 2: V'^T = B^T T^T ----
        if (tid == 0) {
            gemm_split(tVp, sbase + Lay::kBHi, sbase + Lay::kBLo, VC, sbase + Lay::kTHi, sbase + Lay::kTLo, kC, 64,
                       kC, false);
            commit(bar);
        }
        if (wait_products()) break;

        // ---- phase 4: V'^T hi | lo (in place of B^T) ----
        if (col_lane) {
            float x[32];
            tm_ld32(tVp + lanes + 32 * hh, x);
            put_row64(Lay::kBHi, Lay::kBLo, row, VC, 32 * hh, x);
        }
        sync_for_mma();

        // ---- MMA 3: S^T += V'^T K~, O^T += V'^T R~^T; meanwhile the next chunk's loads ----
        if (tid == 0) {
            const uint32_t vH = sbase + Lay::kBHi, vL = sbase + Lay::kBLo;
            gemm_split(tS, vH, vL, VC, sbase + Lay::kKtHi, sbase + Lay::kKtLo, 128, 128, kC, true);
            gemm_split(tO, vH, vL, VC, sbase + Lay::kRt, sbase + Lay::kRt + kC * 128, kC, 64, kC, true);
            commit(bar);
        }
        if (more) load_chunk(c0 + kC);
        if (wait_products()) break;

        // ---- phase 5: O^T into the output rows (FP32 [t][v]); the state images
        //      for the next chunk ----
        if (col_lane) {
            float x[32];
            tm_ld32(tO + lanes + 32 * hh, x);
#pragma unroll
            for (int u = 0; u < 32; ++u) Stage[(32 * hh + u) * Lay::kStagePitch + row] = x[u];
            if (more) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int kd0 = 64 * hh + 32 * c;
                    tm_ld32(tS + lanes + kd0, x);
                    put_images(row, kd0, x);
                }
            }
        }
        __syncthreads();
        {
            // the gated RMSNorm of rows t = warp + 8 j; lane holds VC / 32
            // consecutive columns of a row
            constexpr int PL = VC / 32;
            float o[8][PL];
            float ss[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float* src = Stage + (warp + 8 * j) * Lay::kStagePitch + PL * lane;
                if constexpr (PL == 4) {
                    const float4 f = *reinterpret_cast<const float4*>(src);
                    o[j][0] = f.x; o[j][1] = f.y; o[j][2] = f.z; o[j][3] = f.w;
                } else {
                    const float2 f = *reinterpret_cast<const float2*>(src);
                    o[j][0] = f.x; o[j][1] = f.y;
                }
                ss[j] = 0.f;
#pragma unroll
                for (int e = 0; e < PL; ++e) ss[j] = fmaf(o[j][e], o[j][e], ss[j]);
            }
            if (gated) {
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
                    for (int j = 0; j < 8; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], m);
            }
            if constexpr (CL > 1) {
                // the other CTA's half of each row's sum of squares (distributed
                // shared memory; the buffer alternates with the chunk parity, so the
                // peer's next write to it comes after the next chunk's barrier)
                if (gated && lane < 8) {
                    float mine = ss[0];
#pragma unroll
                    for (int j = 1; j < 8; ++j) mine = lane == j ? ss[j] : mine;
                    ms.ssq_cta[cpar][warp + 8 * lane] = mine;
                }
                cg::cluster_group cl = cg::this_cluster();
                cl.sync();
                if (gated) {
                    const float* peer = cl.map_shared_rank(&ms.ssq_cta[cpar][0], rank ^ 1);
#pragma unroll
                    for (int j = 0; j < 8; ++j) ss[j] += peer[warp + 8 * j];
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = warp + 8 * j;
                if (t >= n) continue;
                float y[PL];
                if (gated) {
                    const float rinv = rsqrtf(ss[j] * (1.0f / kV) + p.eps);
                    float zz[4];
                    unpack4(Zq[t * Lay::kZStride + (PL * lane) / 4], zz);
#pragma unroll
                    for (int e = 0; e < PL; ++e) {
                        const int v = PL * lane + e;
                        const float zv = PL == 4 ? zz[e] : ((lane & 1) ? zz[2 + e] : zz[e]);
                        y[e] = o[j][e] * rinv * ms.wn[v] * silu(zv);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < PL; ++e) y[e] = o[j][e];
                }
                __nv_bfloat16* dst = p.out + ms.row[t] * p.out_stride + h * kV + cb + PL * lane;
                if constexpr (PL == 4) {
                    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
                } else {
                    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(y[0], y[1]);
                }
            }
        }
        fence_before();
        __syncthreads();
        fence_after();
    }

    // ---- the final state to its slot (rounded once), then release TMEM ----
    if (ok && wsl >= 0 && col_lane) {
        StateT* dst =
            static_cast<StateT*>(p.pool) + (wsl * p.H_v + h) * static_cast<int64_t>(kK * kV) + cb + row;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int kd0 = 64 * hh + 32 * c;
            float x[32];
            tm_ld32(tS + lanes + kd0, x);
#pragma unroll
            for (int j = 0; j < 32; ++j) store_elem(dst + (kd0 + j) * kV, x[j]);
        }
    }
    if (!ok) {
        // the MMAs still in flight, with the default bound: one more commit, on
        // a barrier of its own, tracks every MMA the issuing thread has started,
        // and tensor memory is released only once they have finished writing it
        // (a drain that runs out is reported and the memory released regardless)
        if (tid == 0) commit(saddr(&ms.drain));
        const bool drained = wait_parity(saddr(&ms.drain), 0u, kSpinLimit);
        if (tid == 0 && p.status) atomicOr(p.status, GDN_FLAG_TIMEOUT | (drained ? 0 : GDN_FLAG_DRAIN));
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tm));
    // a CTA's shared memory stays until its peer has read the last sums
    if constexpr (CL > 1) cg::this_cluster().sync();
}

template <typename StateT, int VC>
cudaError_t launch(const Params& p, int64_t units, cudaStream_t stream) {
    auto kernel = gdn_prefill_chunked_kernel<StateT, VC>;
    constexpr int kSmem = smem_bytes<VC>();
    static bool done[64] = {false};                             // smem opt-in, once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !done[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) done[dev] = true;
    }
    constexpr int CL = kV / VC;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units * CL), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CL > 1 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Units fewer than half the SMs: each unit's value columns over a 2-CTA
// cluster, so that twice the SMs run the chunks; otherwise one CTA per unit.
template <typename StateT>
cudaError_t launch_any(const Params& p, int64_t units, cudaStream_t stream) {
    static int sms[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && sms[dev] == 0) {
        e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const int n_sm = (dev >= 0 && dev < 64) ? sms[dev] : 0;
    if (2 * units <= n_sm) return launch<StateT, 64>(p, units, stream);
    return launch<StateT, 128>(p, units, stream);
}

}  // namespace


namespace gdn_internal {

uint32_t g_wait_limit = 0;

cudaError_t launch_prefill_chunked(const Params& p0, int64_t units, gdn_dtype state_dtype, cudaStream_t stream) {
    Params p = p0;
    p.wait_limit = __atomic_load_n(&g_wait_limit, __ATOMIC_RELAXED);
    switch (state_dtype) {
    case GDN_F32: return launch_any<float>(p, units, stream);
    case GDN_BF16: return launch_any<__nv_bfloat16>(p, units, stream);
    default: return launch_any<__half>(p, units, stream);
    }
}

}  // namespace gdn_internal
