// libgdnspec: chunked prefill of the Gated DeltaNet layer on the sm_103a
// tensor cores (tcgen05).  The C entry point gdn_prefill_chunked (gdnspec.cu,
// declared in include/gdnspec.h) computes what gdn_prefill computes, in the
// chunked form whose bulk is dense products.
//
// Chunked form (C = 64 tokens; S the K x V state at the chunk start; G_t the
// running sum of the log-decays g inside the chunk; k^, q^ normalised rows):
//   X = K^ S,  Y = Q^ S                                        (C x V)
//   A_ts = beta_t e^(G_t - G_s) (k^_t . k^_s)   for s < t       (C x C)
//   B_t  = beta_t (v_t - e^(G_t) X_t)
//   (I + A) V' = B                                  (forward substitution)
//   O_t  = e^(G_t) Y_t + sum_{s<=t} e^(G_t - G_s) (q^_t . k^_s) V'_s
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
//    and hi.lo terms in FP32 (the lo.lo term is below 2^-18).  A token operand
//    (64 rows) stores hi and lo side by side along K, so the tensor cores add
//    the terms inside the accumulator: its products land in lanes 0-63, and
//    lanes 64-127 (the MMA's rows past the tile) are never read.  Operands are
//    128-byte-swizzled K-major tiles in shared memory; accumulators live in
//    tensor memory:
//      columns   0- 63 P = K^ K^^T         columns  64-127 R = Q^ K^^T
//      columns 128-255 X = K^ S            columns 256-383 O = Q^ S, then
//                                          e^G O + R~ V' (the chunk's output)
//      columns 384-511 S^T (FP32, carried over the whole prompt)
//  * The FP32 state stays in tensor memory from the first chunk to the last.
//    Per chunk it is rescaled by e^(G_last) (tcgen05.ld / st) and V'^T K~ is
//    accumulated into it; its hi and lo bf16 images are the B operands of X
//    and O for the next chunk.
//  * The unit lower-triangular solve runs on CUDA cores in FP32, two (or
//    four) threads per value column with the column in registers,
//    right-looking so that each step is a batch of independent FMAs.
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
// Token tiles have 64 rows and carry hi in columns 0 .. K-1, lo in K .. 2K-1.
// A CTA owns VC of the unit's 128 value columns (128, or 64 with the unit
// over a 2-CTA cluster).  Regions are reused once the products that read
// them have completed:
//   kTileK   [64 t][hi 128 | lo 128 kd]   K^        after phase 2: the FP32 gate w silu(z) [64 t][VC]
//   kTileQ   [64 t][hi 128 | lo 128 kd]   Q^        after MMA 1: K~^T hi | lo  [128 kd][64 t] each
//   kTileS   [VC v][128 kd]               S^T hi
//   kTileS2  [VC v][128 kd]               S^T lo    after MMA 1: V'^T hi | lo  [VC v][64 t] each
//   kTileR   [64 t][hi 64 | lo 64 s]      R~
// A 128-row MMA over a 64-row tile reads 8 KB past each atom column; every
// such read stays inside the shared-memory block and lands in unread lanes.
template <int VC>
struct Layout {
    static constexpr int kTPC = kThreads / VC;                 // solve threads per value column: 2 or 4
    static constexpr int kRowsPT = kC / kTPC;                  // rows per solve thread: 32 or 16
    static constexpr int kTileK = 0;
    static constexpr int kTileQ = kTileK + 32768;
    static constexpr int kTileS = kTileQ + 32768;
    static constexpr int kImg = VC * kK * 2;                   // one state image
    static constexpr int kTileS2 = kTileS + kImg;
    static constexpr int kTileR = kTileS2 + kImg;
    static constexpr int kTileKdHi = kTileQ, kTileKdLo = kTileQ + 16384;
    static constexpr int kTileVHi = kTileS2, kTileVLo = kTileS2 + VC * kC * 2;
    static constexpr int kGate = kTileK;                       // FP32 [64 t][VC], column v stored at v ^ (t % 32)
    static constexpr int kA2Part = kRowsPT + 4;                // floats per residue part of an A row (the pad
                                                               // puts the parts on different banks)
    static constexpr int kA2Row = kTPC * kA2Part;
    static constexpr int kA2 = kTileR + 16384;                 // A     fp32 [64 s][kTPC residue][kA2Part (t / kTPC)]
    static constexpr int kBStride = kC + 1;                    // odd row pitch: column walks are conflict-free
    static constexpr int kBT = kA2 + kC * kA2Row * 4;          // B^T   fp32 [VC v][65]
    static constexpr int kStagePitch = VC / 4 + 1;             // uint2 per padded output-staging row (aliases B^T)
    static constexpr int kZStride = VC / 4 + 1;                // uint2 per padded gate row
    static constexpr int kZ = kBT + VC * kBStride * 4;         // raw z, bf16 quads [64 t][VC / 4 + 1]
    static constexpr int kMisc = (kZ + kC * kZStride * 8 + 15) / 16 * 16;
    static_assert(kC * kStagePitch * 8 <= VC * kBStride * 4, "staging fits the B^T region");
    static_assert(kC * VC * 4 <= 32768, "the gate fits the K^ region");
    static_assert(2 * VC * kC * 2 <= kImg, "V'^T hi and lo fit the S^T lo region");
    static_assert(kTileR + 16384 + 8192 <= kMisc, "the R~ tile's unread rows stay inside the block");
};

struct Misc {
    unsigned long long bar;                     // MMA completion barrier
    uint32_t tmem;                              // tensor-memory base column
    float gamma;                                // e^(G_last) of the current chunk
    float g[kC], G[kC], beta[kC], eG[kC], kfac[kC];   // G 16-byte aligned (float4 reads)
    float ssq[2][kC];                           // per-row sums of squares of this CTA's two column halves
    float ssq_cta[2][kC];                       // with a 2-CTA unit: this CTA's sums, read by its peer
                                                // (indexed by chunk parity)
    float wn[kV];                               // norm_w of this CTA's columns
    int row[kC];
    unsigned long long drain;                   // completion of every MMA issued, after a timeout
};
static_assert(offsetof(Misc, G) % 16 == 0, "float4 reads of G");
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

// (x0, x1) <- (a0, a1) * c + (x0, x1), one paired FP32 FMA (each lane an
// ordinary round-to-nearest FMA)
__device__ __forceinline__ void fma2(float& x0, float& x1, float a0, float a1, float c) {
    uint64_t xv = (static_cast<uint64_t>(__float_as_uint(x1)) << 32) | __float_as_uint(x0);
    const uint64_t av = (static_cast<uint64_t>(__float_as_uint(a1)) << 32) | __float_as_uint(a0);
    const uint64_t cv = (static_cast<uint64_t>(__float_as_uint(c)) << 32) | __float_as_uint(c);
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(xv) : "l"(av), "l"(cv));
    x0 = __uint_as_float(static_cast<uint32_t>(xv));
    x1 = __uint_as_float(static_cast<uint32_t>(xv >> 32));
}

// silu(z) = z sigmoid(z); for very negative z the denominator overflows and
// the fast division returns zero
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// ---- the kernel -------------------------------------------------------------------------
//
// Per chunk, with the warps' TMEM quadrants q = warp % 4 (tcgen05.ld / st reach
// only lanes 32q .. 32q + 31: token rows 0-63 of P, R, X and O from warps 0, 1,
// 4, 5, the "row warps"; state rows v from the warps of their quadrant):
//   phase 1  all warps        k^, q^ (hi | lo), v, z, gates of the chunk's 64
//                             tokens; the running sum G
//   MMA 1                     P = K^ K^^T, R = Q^ K^^T, X = K^ S, O = Q^ S
//   phase 2  row warps 0,1    A from P            row warps 4,5   R~ (hi | lo) from R
//            row warps        B = beta (v - e^G X) and O <- e^G O (each half of v)
//            warps 2,3,6,7    K~^T hi and lo, then the FP32 output gate w silu(z)
//            state warps      S^T <- e^(G_last) S^T (their state rows)
//   phase 3  all warps        (I + A) V' = B: 256 / VC threads per value column,
//                             rows split by residue; V'^T hi and lo tiles
//   MMA 2                     O += R~ V',  S^T += V'^T K~
//   phase 4  row warps        the gated RMSNorm of the chunk's rows (each warp
//                             half of the columns; a 2-CTA unit adds its
//                             peer's sums of squares); state images
//            then all warps store the output rows
//
// VC: value columns of this CTA.  128: one CTA per (prompt, v-head); the
// state warps are all 8.  64: the unit's columns over a 2-CTA cluster (a
// column's recurrence needs no other column; only the RMSNorm adds over
// them); state rows v < 64 live in lanes 0-63, so the row warps are the state
// warps.  The state lives transposed in tensor memory (lane v, column kd), so
// its images, the K-major [v][kd] operands, are written row by row.
template <typename StateT, int VC>
__global__ void __launch_bounds__(kThreads, 1) gdn_prefill_chunked_kernel(const Params p) {
    using Lay = Layout<VC>;
    constexpr int CL = kV / VC;                                 // CTAs per unit
    constexpr int TPC = Lay::kTPC;
    constexpr int RPT = Lay::kRowsPT;
    constexpr int HC = VC / 2;                                  // columns per half
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
    Misc& ms = *reinterpret_cast<Misc*>(sm + Lay::kMisc);
    float* A2 = reinterpret_cast<float*>(sm + Lay::kA2);
    float* BT = reinterpret_cast<float*>(sm + Lay::kBT);
    float* Gate = reinterpret_cast<float*>(sm + Lay::kGate);
    uint2* Zq = reinterpret_cast<uint2*>(sm + Lay::kZ);
    uint2* Stage = reinterpret_cast<uint2*>(sm + Lay::kBT);     // output rows, after the solve
    const uint32_t sbase = saddr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3;                                  // TMEM lane quadrant of this warp
    const int half = warp >> 2;                                 // which half of the columns
    const bool row_warp = quad < 2;                             // reaches the token rows 0-63
    const bool state_warp = quad * 32 < VC;                     // holds state rows v
    const uint32_t lanes = static_cast<uint32_t>(quad * 32) << 16;
    const int row = quad * 32 + lane;                           // this thread's TMEM lane
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

    // ---- set-up: all 512 TMEM columns, the MMA barrier, the norm weight ----
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
    const uint32_t tP = tm, tR = tm + 64, tX = tm + 128, tO = tm + 128 + VC, tS = tm + 384;
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
            *reinterpret_cast<uint4*>(sm + Lay::kTileS + swz_chunk(v, (kd0 >> 3) + j, VC)) = hi;
            *reinterpret_cast<uint4*>(sm + Lay::kTileS2 + swz_chunk(v, (kd0 >> 3) + j, VC)) = lo;
        }
    };

    // ---- initial state: S^T (FP32) into TMEM lane v, its images into the S^T tiles.
    //      Thread (v, half) covers kd in [64 half, 64 half + 64); a warp reads 32
    //      consecutive v of one kd row per load. ----
    if (state_warp) {
        const StateT* src = rs >= 0 ? static_cast<const StateT*>(p.pool) +
                                          (rs * p.H_v + h) * static_cast<int64_t>(kK * kV) + cb + row
                                    : nullptr;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int kd0 = 64 * half + 32 * c;
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = src ? load_elem(src + (kd0 + j) * kV) : 0.f;
            tm_st32(tS + lanes + kd0, x);
            put_images(row, kd0, x);
        }
    }

    // Raw inputs of a chunk, 8 tokens per warp: q, k rows as bf16 quads, z quads
    // of this CTA's columns, v one element per lane per load (v = cb + lane +
    // 32 e, so that its transposed store into B^T hits 32 distinct banks), a / b
    // in lanes 0-15.  The next chunk's loads are issued as soon as the current
    // chunk's solve has finished, so their latency overlaps the epilogue.
    constexpr int VE = VC / 32;                                  // v elements per lane
    uint2 qraw[8], kraw[8], zraw[8];
    __nv_bfloat16 vraw[8][VE];
    float ab;                                                   // lane j: a of token j, lane 8 + j: its b
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
        ab = 0.f;
        if (lane < 16 && warp + 8 * (lane & 7) < nn) {
            const int64_t r = bos + cs + warp + 8 * (lane & 7);
            ab = __bfloat162float(lane < 8 ? p.a[r * p.a_stride + h] : p.b[r * p.b_stride + h]);
        }
    };
    load_chunk(0);

    for (int c0 = 0; c0 < L; c0 += kC) {
        const int n = min(kC, L - c0);
        const int cpar = (c0 / kC) & 1;                          // chunk parity

        // ---- phase 1: per token (8 per warp) k^, q^ (hi | lo), v (B^T), raw z,
        //      gates, from the raw rows loaded while the previous chunk finished ----
        {
            // gates of the warp's 8 tokens, one per lane
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
                for (int e = 0; e < VE; ++e) BT[(lane + 32 * e) * Lay::kBStride + t] = __bfloat162float(vraw[j][e]);
            }
            *reinterpret_cast<uint2*>(sm + Lay::kTileK + swz(t, lane * 4, kC)) = khi;
            *reinterpret_cast<uint2*>(sm + Lay::kTileK + swz(t, kK + lane * 4, kC)) = klo;
            *reinterpret_cast<uint2*>(sm + Lay::kTileQ + swz(t, lane * 4, kC)) = qhi;
            *reinterpret_cast<uint2*>(sm + Lay::kTileQ + swz(t, kK + lane * 4, kC)) = qlo;
        }
        __syncthreads();
        if (warp == 0) {
            // G = inclusive running sum of g; e^(G_t), e^(G_last - G_t), e^(G_last)
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
        sync_for_mma();

        // ---- MMA 1: P = K^ K^^T, R = Q^ K^^T, X = K^ S, O = Q^ S (hi.hi + lo.hi +
        //      hi.lo each) ----
        if (tid == 0) {
            const uint32_t kH = sbase + Lay::kTileK, kL = kH + 2 * kC * 128;     // K^ hi | lo atom columns
            const uint32_t qH = sbase + Lay::kTileQ, qL = qH + 2 * kC * 128;
            const uint32_t sH = sbase + Lay::kTileS, sL = sbase + Lay::kTileS2;
            gemm_split(tP, kH, kL, kC, kH, kL, kC, 64, kK, false);
            gemm_split(tX, kH, kL, kC, sH, sL, VC, VC, kK, false);
            gemm_split(tO, qH, qL, kC, sH, sL, VC, VC, kK, false);
            gemm_split(tR, qH, qL, kC, kH, kL, kC, 64, kK, false);
            commit(bar);
        }
        {
            // a 2-CTA unit never leaves the loop early (its CTAs meet at a cluster
            // barrier every chunk): a wait that runs out is recorded and the chunk
            // goes on
            const bool done = wait_mma(bar, phase, limit);
            const bool late = __syncthreads_or(!done);
            phase ^= 1;
            if (late) ok = false;
            if (CL == 1 && late) break;
        }
        fence_after();

        // ---- phase 2 ----
        if (row_warp) {
            const int t = row;                                  // token row of this lane
            const float Gt = ms.G[t], bt = ms.beta[t], eG = ms.eG[t];
            const bool live = t < n;
            if (half == 0) {
                // A (s < t) from P, stored as A2[s][t % TPC][t / TPC]; the decay
                // factors are formed before any store, so no shared load waits
                // behind a store
                float* dst = A2 + (t % TPC) * Lay::kA2Part + (t / TPC);
#pragma unroll
                for (int s0 = 0; s0 < kC; s0 += 32) {
                    float x[32], d[32];
                    load_decays(ms.G + s0, Gt, d);
                    tm_ld32(tP + lanes + s0, x);
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        const int s = s0 + u;
                        dst[s * Lay::kA2Row] = (live && s < t) ? bt * d[u] * x[u] : 0.f;
                    }
                }
            } else {
                // R~ (s <= t) from R, hi | lo
#pragma unroll
                for (int s0 = 0; s0 < kC; s0 += 32) {
                    float x[32], d[32];
                    load_decays(ms.G + s0, Gt, d);
                    tm_ld32(tR + lanes + s0, x);
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        const int s = s0 + u;
                        x[u] = (live && s <= t) ? d[u] * x[u] : 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint4 hi, lo;
                        split8(x + 8 * j, hi, lo);
                        *reinterpret_cast<uint4*>(sm + Lay::kTileR + swz_chunk(t, (s0 >> 3) + j, kC)) = hi;
                        *reinterpret_cast<uint4*>(sm + Lay::kTileR + swz_chunk(t, 8 + (s0 >> 3) + j, kC)) = lo;
                    }
                }
            }
            // B = beta (v - e^(G_t) X) and O <- e^(G_t) O for this half of the value columns
#pragma unroll
            for (int c = 0; c < HC / 32; ++c) {
                const int v0 = HC * half + 32 * c;
                float x[32];
                tm_ld32(tX + lanes + v0, x);
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    float* bp = &BT[(v0 + u) * Lay::kBStride + t];
                    *bp = live ? bt * (*bp - eG * x[u]) : 0.f;
                }
                tm_ld32(tO + lanes + v0, x);
#pragma unroll
                for (int u = 0; u < 32; ++u) x[u] *= eG;
                tm_st32(tO + lanes + v0, x);
            }
        } else {
            // K~^T [kd][t] = k^_t[kd] e^(G_last - G_t) (k^ = hi + lo), split again:
            // one 16-byte chunk (8 tokens) of each part per item (the Q^ region,
            // free since MMA 1)
            const int wt = tid - 64 * (1 + half);              // 0..127 over warps 2, 3, 6, 7
            for (int e = wt; e < kK * (kC / 8); e += 128) {
                const int kd = e & (kK - 1), j = e >> 7;
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int t = 8 * j + u;
                    const float kv =
                        __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + Lay::kTileK + swz(t, kd, kC))) +
                        __bfloat162float(
                            *reinterpret_cast<const __nv_bfloat16*>(sm + Lay::kTileK + swz(t, kK + kd, kC)));
                    x[u] = kv * ms.kfac[t];
                }
                uint4 hi, lo;
                split8(x, hi, lo);
                *reinterpret_cast<uint4*>(sm + Lay::kTileKdHi + swz_chunk(kd, j, 128)) = hi;
                *reinterpret_cast<uint4*>(sm + Lay::kTileKdLo + swz_chunk(kd, j, 128)) = lo;
            }
            // every K^ read above is done before the gate overwrites the region
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (gated) {
                // the output gate w silu(z) in FP32, [t][v ^ (t % 32)]
                for (int e = wt; e < kC * (VC / 4); e += 128) {
                    const int t = e / (VC / 4), q4 = e % (VC / 4);
                    float zz[4];
                    unpack4(Zq[t * Lay::kZStride + q4], zz);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int v = 4 * q4 + c;
                        Gate[t * VC + (v ^ (t & 31))] = ms.wn[v] * silu(zz[c]);
                    }
                }
            }
        }
        if (state_warp) {
            // S^T <- e^(G_last) S^T: lane v of this quadrant, this half of the kd columns
            const float gamma = ms.gamma;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint32_t col = tS + lanes + 64 * half + 32 * c;
                float x[32];
                tm_ld32(col, x);
#pragma unroll
                for (int u = 0; u < 32; ++u) x[u] *= gamma;
                tm_st32(col, x);
            }
        }
        fence_before();
        __syncthreads();
        fence_after();

        // ---- phase 3: (I + A) V' = B.  TPC threads per value column vc; member r
        //      owns rows t = TPC i + r in x[i].  Right-looking: once x_s is final
        //      its owner broadcasts it and all remove its part from their later
        //      rows (A2[s][.][i] is zero for rows t <= s, so the float4 groups
        //      may start below). ----
        {
            const int vc = tid / TPC, r = tid % TPC;
            float x[RPT];
#pragma unroll
            for (int i2 = 0; i2 < RPT; ++i2) x[i2] = BT[vc * Lay::kBStride + TPC * i2 + r];
            const float* arow = A2 + r * Lay::kA2Part;
#pragma unroll
            for (int s = 0; s < kC - 1; ++s) {
                const float mine = (r == (s % TPC)) ? x[s / TPC] : 0.f;
                const float nxs = -__shfl_sync(0xffffffffu, mine, (lane & ~(TPC - 1)) | (s % TPC));
#pragma unroll
                for (int i4 = (s / (4 * TPC)); i4 < RPT / 4; ++i4) {
                    const float4 a4 = *reinterpret_cast<const float4*>(arow + s * Lay::kA2Row + 4 * i4);
                    fma2(x[4 * i4 + 0], x[4 * i4 + 1], a4.x, a4.y, nxs);
                    fma2(x[4 * i4 + 2], x[4 * i4 + 3], a4.z, a4.w, nxs);
                }
            }
            // V'^T tile rows vc, hi and lo: this thread's tokens TPC i + r
#pragma unroll
            for (int i2 = 0; i2 < RPT; ++i2) {
                const __nv_bfloat16 hi = __float2bfloat16_rn(x[i2]);
                const __nv_bfloat16 lo = __float2bfloat16_rn(x[i2] - __bfloat162float(hi));
                *reinterpret_cast<__nv_bfloat16*>(sm + Lay::kTileVHi + swz(vc, TPC * i2 + r, VC)) = hi;
                *reinterpret_cast<__nv_bfloat16*>(sm + Lay::kTileVLo + swz(vc, TPC * i2 + r, VC)) = lo;
            }
        }
        sync_for_mma();

        // ---- MMA 2: O += R~ V',  S^T += V'^T K~; meanwhile the next chunk's loads ----
        if (tid == 0) {
            const uint32_t rH = sbase + Lay::kTileR, rL = rH + kC * 128;     // R~ hi | lo atom columns
            const uint32_t vH = sbase + Lay::kTileVHi, vL = sbase + Lay::kTileVLo;
            gemm_split(tO, rH, rL, kC, vH, vL, VC, VC, kC, true);
            gemm_split(tS, vH, vL, VC, sbase + Lay::kTileKdHi, sbase + Lay::kTileKdLo, 128, 128, kC, true);
            commit(bar);
        }
        if (c0 + kC < L) load_chunk(c0 + kC);
        {
            const bool done = wait_mma(bar, phase, limit);
            const bool late = __syncthreads_or(!done);
            phase ^= 1;
            if (late) ok = false;
            if (CL == 1 && late) break;
        }
        fence_after();

        // ---- phase 4: outputs (rows t < 64 on the row warps; each warp half of
        //      the columns), then the state images for the next chunk ----
        const bool more = c0 + kC < L;
        if (row_warp && gated) {
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < HC / 32; ++c) {
                float x[32];
                tm_ld32(tO + lanes + HC * half + 32 * c, x);
#pragma unroll
                for (int u = 0; u < 32; ++u) ss = fmaf(x[u], x[u], ss);
            }
            ms.ssq[half][row] = ss;
        }
        if (more && state_warp && !row_warp) {
            // images of rows v = 64..127 while the others wait for the norms
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int kd0 = 64 * half + 32 * c;
                float x[32];
                tm_ld32(tS + lanes + kd0, x);
                put_images(row, kd0, x);
            }
        }
        __syncthreads();
        if constexpr (CL > 1) {
            // the other CTA's half of each token's sum of squares (distributed
            // shared memory; the buffer alternates with the chunk parity, so the
            // peer's next write to it comes after the next chunk's barrier)
            if (gated && tid < kC) ms.ssq_cta[cpar][tid] = ms.ssq[0][tid] + ms.ssq[1][tid];
            cg::cluster_group cl = cg::this_cluster();
            cl.sync();
            if (gated && tid < kC)
                ms.ssq[0][tid] += *cl.map_shared_rank(&ms.ssq_cta[cpar][tid], rank ^ 1);
            __syncthreads();
        }
        if (row_warp) {
            // normalised, gated rows into the staging buffer (the B^T region,
            // free until the next chunk), then the images of rows v = 0..63
            const int t = row;
            const float rinv = gated ? rsqrtf((ms.ssq[0][t] + ms.ssq[1][t]) * (1.0f / kV) + p.eps) : 1.0f;
            uint2* srow = Stage + t * Lay::kStagePitch + (HC / 4) * half;
#pragma unroll
            for (int c = 0; c < HC / 32; ++c) {
                float x[32];
                tm_ld32(tO + lanes + HC * half + 32 * c, x);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    float y[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int v = HC * half + 32 * c + 4 * j4 + e;
                        y[e] = gated ? x[4 * j4 + e] * rinv * Gate[t * VC + (v ^ (t & 31))] : x[4 * j4 + e];
                    }
                    srow[8 * c + j4] = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
                }
            }
            if (more) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int kd0 = 64 * half + 32 * c;
                    float x[32];
                    tm_ld32(tS + lanes + kd0, x);
                    put_images(row, kd0, x);
                }
            }
        }
        __syncthreads();
        // the chunk's output rows, this CTA's columns
#pragma unroll
        for (int e = tid; e < kC * (VC / 4); e += kThreads) {
            const int t = e / (VC / 4), q4 = e % (VC / 4);
            if (t < n)
                *reinterpret_cast<uint2*>(p.out + ms.row[t] * p.out_stride + h * kV + cb + 4 * q4) =
                    Stage[t * Lay::kStagePitch + q4];
        }
        fence_before();
        __syncthreads();
        fence_after();
    }

    // ---- the final state to its slot (rounded once), then release TMEM ----
    if (ok && wsl >= 0 && state_warp) {
        StateT* dst =
            static_cast<StateT*>(p.pool) + (wsl * p.H_v + h) * static_cast<int64_t>(kK * kV) + cb + row;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int kd0 = 64 * half + 32 * c;
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
