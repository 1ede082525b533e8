// libgdnspec: the Gated DeltaNet speculative / MTP decode step for sm_103a.
//
// What each call computes is stated in include/gdnspec.h, with the report
// pages it follows.  This file holds the decode kernel (and its variant with
// the short causal convolution fused in front), the per-token prefill kernel,
// and every C entry point with its host-side checks; the tensor-core chunked
// prefill kernel is in gdnprefill_chunked.cu.
//
// Design (GB300):
//  * The step is HBM-bound: one 128x128 state tile read and up to 8 tile writes
//    per (sequence, v-head), against ~4 FP32 ops per state element per token.
//    No tensor cores: per token it is a rank-1 update and two K-reductions.
//  * Work unit = (sequence i, v-head h).  A warp owns 16 full V columns of the
//    tile (all 128 K rows): lane = cg + 4*rg holds rows rg, rg+8, .., rg+120 of
//    columns 16*wg + 4cg .. +3 in 64 registers, FP32, for all draft tokens.
//    Because each V column evolves on its own, the two K-reductions are
//    warp-local shuffles and the token loop needs no block barrier for the
//    math.  One CTA per unit: the block scheduler starts the next CTA on an
//    SM as soon as one ends (a grid of resident CTAs walking the units, with
//    the next unit's tile prefetched into L2, was measured slower).
//  * Latency: every load that does not depend on another is issued up front.
//    The tile is read straight into registers with 16-byte (FP32) / 8-byte
//    (BF16, FP16) streaming loads before the per-token prologue, and the
//    prologue fetches q, k, v, z, a, b and the parameters of all draft tokens
//    at once, so the epilogue touches no global input.
//  * Both reductions use the state BEFORE the token (the "pair" reduction of
//    the PR #51674 report, implementation step 1): with d = e^g,
//        u = d (S^T k^),   v' = beta (v - u),   o = d (S^T q^) + (k^.q^) v'
//    which equals o = S_new^T q^ exactly in real arithmetic.
//  * Each token's state is rounded once to the pool dtype (RNE) while the
//    carried state stays FP32 (PR #52191 report, implementation step 4).  Each
//    warp writes its 128 x 16 block to its own staging buffer in shared memory
//    and one lane hands it to the tensor-memory-access unit as one 2-D store
//    into the slot; a warp-level barrier is all it needs (a CTA-wide tile and
//    barrier per token was measured slower).
//  * Small batches may split the 8 column blocks of a unit over SPLIT CTAs of
//    one thread-block cluster (SPLIT = 2, 4, 8); the gated RMSNorm's
//    mean-square over V is then combined through distributed shared memory.
//    The narrow layout (NCW = 8) gives each warp 8 columns instead of 16: a
//    unit's 16 warps run over a 2- or 4-CTA cluster with half the state per
//    lane and one more butterfly step.  The half-K layout (KS = 2) keeps 16
//    columns per warp but gives each warp half of their K rows; the two warps
//    of a column block add their partial products through shared memory once
//    per token, and a unit's 16 warps run in one CTA or over a 2-CTA cluster.
//    It is the automatic choice for an FP32 state with at most 128 units.
//  * No device-side waits on flags, no traps: bad device data is skipped and
//    reported through an optional status word.
//  * Fused convolution (CONV = true, SPLIT = 1): each lane convolves its 12
//    channels (4 of q, 4 of k, 4 of v) for its warp's draft token from the
//    rewound history rows and the step's rows, all loads first, in FP32; the
//    result enters the same per-token prologue.  The new conv slot is written
//    once the sequence is known not to be skipped.
//  * Prefill (per token): the same token step over whole prompts, 8 tokens
//    per round of prologue / tokens / epilogue, the state in registers from
//    the first token to the last and stored once.

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include <cudaTypedefs.h>

#include "gdn_internal.h"
#include "gdnspec.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kK = 128;
constexpr int kV = 128;
constexpr int kMaxT = 8;
constexpr int kColsPerWarp = 16;             // the default (wide) warp: 16 V columns ...
constexpr int kRowsPerLane = 16;             // ... 16 K rows per lane
constexpr float kQkEps = 1e-6f;              // inside the L2-norm square root
constexpr float kSoftplusThreshold = 20.0f;  // softplus(x) = x above this
constexpr unsigned kFull = 0xffffffffu;
constexpr int64_t kTile = static_cast<int64_t>(kK) * kV;
// Lane layout of a warp's block of the state tile.  NCW = V columns per warp:
// 16 (the default) or 8 (the narrow variant for small batches, where a unit's
// 16 warps spread over a 2- or 4-CTA cluster).  Lane = cg + (NCW/4) rg holds
// the 4 consecutive columns of column group cg in the K rows rg + G j, j = 0
// .. R-1 (G row groups, R = 128 / G rows per lane).  The lane bits above the
// column group are the row group in both layouts, so the reduce-scatter over
// lane bits 4, 3, 2 means the same in both.
//
// With KS = 2 (the half-K layout, 16 columns per warp) a warp owns half of
// the K rows of its columns: warps w and w + W/2 of a CTA hold rows 0-63 and
// 64-127, lane rows kq 64 + rg + 8 j (kq the half), 8 rows per lane, and
// the two warps add their partial dot products through shared memory.
template <int NCW, int KS = 1>
struct Lanes {
    static_assert(NCW == 16 || NCW == 8, "16 or 8 columns per warp");
    static_assert(KS == 1 || (KS == 2 && NCW == 16), "the half-K layout has 16 columns per warp");
    static constexpr int kColGroups = NCW / 4;            // 4 or 2
    static constexpr int kRowGroups = 32 / kColGroups;    // 8 or 16
    static constexpr int kSpan = kK / KS;                 // K rows of one warp
    static constexpr int kRows = kSpan / kRowGroups;      // 16, 8 (narrow) or 8 (half-K)
    // k^ / q^ sit in shared memory permuted so that a lane's rows are
    // contiguous (row -> R (row % G) + row / G), with 4 floats of padding after
    // every 16 (NCW = 16) or 32 (NCW = 8) positions: the row groups' 16-byte
    // chunks then spread evenly over the banks (one wavefront for 8 groups,
    // two for 16).
    static constexpr int kPadEvery = (NCW == 16 && KS == 1) ? 16 : 32;
    __host__ __device__ static constexpr int pos(int p) { return p + (p / kPadEvery) * 4; }
    __host__ __device__ static constexpr int perm(int row) {
        return pos((row / kSpan) * kSpan + (row % kRowGroups) * kRows + (row % kSpan) / kRowGroups);
    }
};
constexpr int kKPad = kK + kK / 4;           // room for either padding

using gdn_internal::Params;

// per-CTA shared memory
struct alignas(16) Smem {
    float k[kMaxT][kKPad];       // k^ per token (padded rows)
    float q[kMaxT][kKPad];       // q^ * scale per token
    float v[kMaxT][kV];
    float o[kMaxT][kV];          // readout per token, for the epilogue
    uint2 z[kMaxT][kV / 4];      // raw bf16 quads of the output gate
    uint2 w[kV / 4];             // raw bf16 quads of norm_w
    float decay[kMaxT], beta[kMaxT], kq[kMaxT], red[kMaxT];
    int row[kMaxT];
    long long ws[kMaxT];
    float xch[2][8][2][32];      // half-K layout: the warp pairs' partial dots, by token parity
};

template <typename StateT, int SPLIT, int NCW = kColsPerWarp, int KS = 1>
struct Config {
    static constexpr int kWarps = kV / NCW / SPLIT * KS;
    static constexpr int kThreads = 32 * kWarps;
    // each warp stages its (128 / KS) x NCW block of a token's state for the tensor store
    static constexpr size_t kStageOffset = (sizeof(Smem) + 127) / 128 * 128;
    static constexpr size_t kStageElems = static_cast<size_t>(kK / KS) * NCW;
    // + 128 bytes so that the staging buffers can start on a 128-byte boundary
    static constexpr size_t kSmem = kStageOffset + kWarps * kStageElems * sizeof(StateT) + 128;
};

// ---- element I/O ---------------------------------------------------------------

__device__ __forceinline__ void unpack_bf16x4(uint2 raw, float (&x)[4]) {
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    x[0] = lo.x; x[1] = lo.y; x[2] = hi.x; x[3] = hi.y;
}

__device__ __forceinline__ uint2 pack_bf16x4(const float (&x)[4]) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(x[2], x[3]);
    uint2 raw;
    raw.x = *reinterpret_cast<const uint32_t*>(&lo);
    raw.y = *reinterpret_cast<const uint32_t*>(&hi);
    return raw;
}

// read-only inputs (never written by the kernel)
__device__ __forceinline__ uint2 ldg_quad(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const uint2*>(p));
}

// state tile: 4 consecutive V columns of one K row, streaming (read once /
// written once per step)
template <typename T>
struct StateIO;

template <>
struct StateIO<float> {
    static __device__ __forceinline__ void load4(const float* p, float (&x)[4]) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(p));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    static __device__ __forceinline__ void store4(float* p, const float (&x)[4]) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
    }
    static __device__ __forceinline__ void stage4(float* p, const float (&x)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};

template <>
struct StateIO<__nv_bfloat16> {
    static __device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&x)[4]) {
        unpack_bf16x4(__ldcs(reinterpret_cast<const uint2*>(p)), x);
    }
    static __device__ __forceinline__ uint2 pack(const float (&x)[4]) { return pack_bf16x4(x); }
    static __device__ __forceinline__ void store4(__nv_bfloat16* p, const float (&x)[4]) {
        __stcs(reinterpret_cast<uint2*>(p), pack(x));
    }
    static __device__ __forceinline__ void stage4(__nv_bfloat16* p, const float (&x)[4]) {
        *reinterpret_cast<uint2*>(p) = pack(x);
    }
};

template <>
struct StateIO<__half> {
    static __device__ __forceinline__ void load4(const __half* p, float (&x)[4]) {
        const uint2 raw = __ldcs(reinterpret_cast<const uint2*>(p));
        const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        x[0] = lo.x; x[1] = lo.y; x[2] = hi.x; x[3] = hi.y;
    }
    static __device__ __forceinline__ uint2 pack(const float (&x)[4]) {
        const __half2 lo = __floats2half2_rn(x[0], x[1]);
        const __half2 hi = __floats2half2_rn(x[2], x[3]);
        uint2 raw;
        raw.x = *reinterpret_cast<const uint32_t*>(&lo);
        raw.y = *reinterpret_cast<const uint32_t*>(&hi);
        return raw;
    }
    static __device__ __forceinline__ void store4(__half* p, const float (&x)[4]) {
        __stcs(reinterpret_cast<uint2*>(p), pack(x));
    }
    static __device__ __forceinline__ void stage4(__half* p, const float (&x)[4]) {
        *reinterpret_cast<uint2*>(p) = pack(x);
    }
};

// ---- tensor (TMA) stores of a warp's staged block ------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// store the 128 x 16 box at smem `src` to global columns x.., rows y.. of the pool map
__device__ __forceinline__ void tma_store_box(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(src)), "r"(x), "r"(y) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// this thread's earlier tensor stores have finished reading shared memory
__device__ __forceinline__ void tma_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and have completed
__device__ __forceinline__ void tma_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(kFull, x, m);
    return x;
}

__device__ __forceinline__ void raise_flag(const Params& p, int rank, int flag) {
    if (p.status != nullptr && threadIdx.x == 0 && rank == 0) atomicOr(p.status, flag);
}

// Paired FP32 arithmetic (fma.rn.f32x2 / mul.rn.f32x2): each lane of the pair
// rounds exactly as fmaf / a plain multiply would, at half the instructions.
__device__ __forceinline__ uint64_t pk2(float a, float b) {
    return (static_cast<uint64_t>(__float_as_uint(b)) << 32) | __float_as_uint(a);
}
__device__ __forceinline__ void upk2(uint64_t v, float& a, float& b) {
    a = __uint_as_float(static_cast<uint32_t>(v));
    b = __uint_as_float(static_cast<uint32_t>(v >> 32));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ---- the pieces of one unit ------------------------------------------------------

// Per-token prologue arithmetic for token t of unit (i, h), one warp: the raw
// quads are this lane's 4 elements of q, k (key head), v and z (v-head);
// `ws` is the slot that receives the state after this token (-1: none).
template <int NCW = kColsPerWarp, int KS = 1>
__device__ __forceinline__ void prologue_token_f(Smem& s, const Params& p, int h, int t, int r, int lane,
                                                 float (&qv)[4], float (&kv)[4], const float (&vv)[4], uint2 zraw,
                                                 long long ws) {
    float a_in = 0.f, b_in = 0.f, dtb = 0.f, alog = 0.f;
    if (lane == 0) {
        a_in = __bfloat162float(p.a[r * p.a_stride + h]);
        b_in = __bfloat162float(p.b[r * p.b_stride + h]);
        dtb = __bfloat162float(p.dt_bias[h]);
        alog = __ldg(p.A_log + h);
    }
    // |q|^2, |k|^2 and q.k in one butterfly: k^.q^ = (q.k) rq rk needs no
    // second reduction after the normalisation
    float sq = 0.f, sk = 0.f, qk = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) { sq += qv[e] * qv[e]; sk += kv[e] * kv[e]; qk += qv[e] * kv[e]; }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        sq += __shfl_xor_sync(kFull, sq, m);
        sk += __shfl_xor_sync(kFull, sk, m);
        qk += __shfl_xor_sync(kFull, qk, m);
    }
    const float rq = rsqrtf(sq + kQkEps) * p.scale;
    const float rk = rsqrtf(sk + kQkEps);
    const float kq = qk * rq * rk;
#pragma unroll
    for (int e = 0; e < 4; ++e) { qv[e] *= rq; kv[e] *= rk; }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        s.q[t][Lanes<NCW, KS>::perm(lane * 4 + e)] = qv[e];
        s.k[t][Lanes<NCW, KS>::perm(lane * 4 + e)] = kv[e];
    }
    *reinterpret_cast<float4*>(&s.v[t][lane * 4]) = make_float4(vv[0], vv[1], vv[2], vv[3]);
    s.z[t][lane] = zraw;
    if (lane == 0) {
        const float x = a_in + dtb;
        const float sp = x > kSoftplusThreshold ? x : log1pf(expf(x));
        s.decay[t] = expf(-expf(alog) * sp);
        s.beta[t] = 1.0f / (1.0f + expf(-b_in));
        s.kq[t] = kq;
        s.row[t] = r;
        s.ws[t] = ws;
    }
}

template <int NCW = kColsPerWarp, int KS = 1>
__device__ __forceinline__ void prologue_token(Smem& s, const Params& p, int h, int t, int r, int lane,
                                               uint2 qraw, uint2 kraw, uint2 vraw, uint2 zraw, long long ws) {
    float qv[4], kv[4], vv[4];
    unpack_bf16x4(qraw, qv);
    unpack_bf16x4(kraw, kv);
    unpack_bf16x4(vraw, vv);
    prologue_token_f<NCW, KS>(s, p, h, t, r, lane, qv, kv, vv, zraw, ws);
}

// The state in this lane's block to slot ws (skip -1).  With a staging
// buffer the warp writes its 128 x NCW block to shared memory (8 lanes of a
// row group fill 8 consecutive 32 / 64-byte rows: no bank conflicts) and one
// lane hands it to the tensor-memory-access unit, which writes the strided
// block to the slot; the buffer is reused once that store has read it.
// Without one, every lane stores its rows itself.
template <typename StateT, int NCW, int KS = 1>
__device__ __forceinline__ void write_slot(const float (&S)[Lanes<NCW, KS>::kRows][4], const Params& p, long long ws,
                                           int h, int lane, int col0, int rank, StateT* stage, int kq = 0) {
    using L = Lanes<NCW, KS>;
    const int cgi = lane % L::kColGroups;
    const int rg = lane / L::kColGroups;
    if (ws >= p.num_slots) raise_flag(p, rank, GDN_FLAG_SLOT_RANGE);
    if (ws >= 0 && ws < p.num_slots) {
        if (stage != nullptr) {
            if (lane == 0) tma_wait_read();
            __syncwarp();
#pragma unroll
            for (int r = 0; r < L::kRows; ++r)
                StateIO<StateT>::stage4(stage + (rg + L::kRowGroups * r) * NCW + 4 * cgi, S[r]);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0)
                tma_store_box(&p.pool_map, stage, col0 - 4 * cgi,
                              static_cast<int>((ws * p.H_v + h) * kK + kq * L::kSpan));
        } else {
            StateT* d = static_cast<StateT*>(p.pool) + (ws * p.H_v + h) * kTile + col0;
#pragma unroll
            for (int r = 0; r < L::kRows; ++r)
                StateIO<StateT>::store4(d + static_cast<int64_t>(kq * L::kSpan + rg + L::kRowGroups * r) * kV, S[r]);
        }
    }
}

// One draft token for this lane's 16x4 block: both reductions, the delta rule,
// the readout into s.o, the state update and (when s.ws[t] names a slot) the
// slot write.  With PIPE the state after token t - 1 is staged for its slot
// write while token t's partial products are formed (both only read S), and
// the state after token t is left for the next call (or write_slot after the
// last token): one CTA per SM waits on nothing between the two.
template <typename StateT, int NCW = kColsPerWarp, bool PIPE = false, int KS = 1>
__device__ __forceinline__ void token_step(float (&S)[Lanes<NCW, KS>::kRows][4], Smem& s, const Params& p, int t,
                                           int h, int lane, int col0, int row0, int rank, StateT* stage,
                                           int kq = 0, int pair = 0) {
    using L = Lanes<NCW, KS>;
    const int cgi = lane % L::kColGroups;
    const int rg = lane / L::kColGroups;
    long long pws = -1;                  // PIPE: the previous token's slot, staged below
    if constexpr (PIPE) {
        if (t > 0) pws = s.ws[t - 1];
        if (pws >= p.num_slots) {
            raise_flag(p, rank, GDN_FLAG_SLOT_RANGE);
            pws = -1;
        }
        if (pws >= 0) {
            if (lane == 0) tma_wait_read();
            __syncwarp();
        }
    }
    const int c_own = (lane >> 2) & 3; // after the reduce-scatter: my column ...
    const int d_own = (lane >> 4) & 1; // ... and which dot product (0: k, 1: q)
    const float decay = s.decay[t];
    const float beta = s.beta[t];
    const float kq_dot = s.kq[t];

    // partial S^T k^ and S^T q^ over this lane's 16 rows, 4 columns each
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = 0.f;
#pragma unroll
    for (int r4 = 0; r4 < L::kRows / 4; ++r4) {
        const float4 kk = *reinterpret_cast<const float4*>(&s.k[t][L::pos(row0 + 4 * r4)]);
        const float4 qq = *reinterpret_cast<const float4*>(&s.q[t][L::pos(row0 + 4 * r4)]);
        const float kr[4] = {kk.x, kk.y, kk.z, kk.w};
        const float qr[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int c = 0; c < 4; c += 2) {                   // column pairs
                const uint64_t s2 = pk2(S[4 * r4 + rr][c], S[4 * r4 + rr][c + 1]);
                uint64_t xk = pk2(x[c], x[c + 1]), xq = pk2(x[4 + c], x[5 + c]);
                xk = ffma2(s2, pk2(kr[rr], kr[rr]), xk);
                xq = ffma2(s2, pk2(qr[rr], qr[rr]), xq);
                upk2(xk, x[c], x[c + 1]);
                upk2(xq, x[4 + c], x[5 + c]);
            }
        if constexpr (PIPE) {
            if (pws >= 0) {
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
                    StateIO<StateT>::stage4(stage + (rg + L::kRowGroups * (4 * r4 + rr)) * NCW + 4 * cgi,
                                            S[4 * r4 + rr]);
            }
        }
    }
    if constexpr (PIPE) {
        if (pws >= 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0)
                tma_store_box(&p.pool_map, stage, col0 - 4 * cgi,
                              static_cast<int>((pws * p.H_v + h) * kK + kq * L::kSpan));
        }
    }
    // reduce-scatter over the row groups on lane bits 4, 3, 2: afterwards the
    // lane holds the sum of value index 4 d + c = (lane >> 2) & 7 (d = 0: k,
    // 1: q; c: column within its group) over those groups; with 16 row groups
    // (NCW = 8) lane bit 1 is a row-group bit too and one more step completes
    // the sum on both lanes of the pair
    float y[4];
    {
        const bool hi = (lane >> 4) & 1;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float send = hi ? x[e] : x[4 + e];
            const float keep = hi ? x[4 + e] : x[e];
            y[e] = keep + __shfl_xor_sync(kFull, send, 16);
        }
    }
    float z2[2];
    {
        const bool hi = (lane >> 3) & 1;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float send = hi ? y[e] : y[2 + e];
            const float keep = hi ? y[2 + e] : y[e];
            z2[e] = keep + __shfl_xor_sync(kFull, send, 8);
        }
    }
    float dot;
    {
        const bool hi = (lane >> 2) & 1;
        const float send = hi ? z2[0] : z2[1];
        const float keep = hi ? z2[1] : z2[0];
        dot = keep + __shfl_xor_sync(kFull, send, 4);
    }
    if constexpr (NCW == 8) dot += __shfl_xor_sync(kFull, dot, 2);
    if constexpr (KS == 2) {
        // the other half of K: the partner warp's partial sums, through shared
        // memory (by token parity, so that a warp's next write never meets a
        // read of the partner's that is still pending), one named barrier per
        // warp pair
        float* xch = &s.xch[t & 1][pair][0][0];
        xch[kq * 32 + lane] = dot;
        asm volatile("bar.sync %0, 64;" ::"r"(1 + pair) : "memory");
        dot += xch[(kq ^ 1) * 32 + lane];
    }
    // delta rule on the k lanes; readout on the q lanes
    const float vp = beta * (s.v[t][col0 + c_own] - decay * dot);   // valid where d_own == 0
    const float vp_pair = __shfl_xor_sync(kFull, vp, 16);
    if (d_own == 1 && kq == 0) s.o[t][col0 + c_own] = fmaf(decay, dot, kq_dot * vp_pair);
    float vpc[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) vpc[c] = __shfl_sync(kFull, vp, cgi + 4 * c);

    // S <- e^g S + k^ v'^T
#pragma unroll
    for (int r4 = 0; r4 < L::kRows / 4; ++r4) {
        const float4 kk = *reinterpret_cast<const float4*>(&s.k[t][L::pos(row0 + 4 * r4)]);
        const float kr[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int c = 0; c < 4; c += 2) {                   // S = fmaf(S, decay, k v'), by pairs
                const uint64_t t2 = fmul2(pk2(kr[rr], kr[rr]), pk2(vpc[c], vpc[c + 1]));
                const uint64_t s2 = ffma2(pk2(S[4 * r4 + rr][c], S[4 * r4 + rr][c + 1]), pk2(decay, decay), t2);
                upk2(s2, S[4 * r4 + rr][c], S[4 * r4 + rr][c + 1]);
            }
    }

    // the state after token t goes to slot s.ws[t] (skip -1); with PIPE, during
    // the next token
    if constexpr (!PIPE) write_slot<StateT, NCW, KS>(S, p, s.ws[t], h, lane, col0, rank, stage, kq);
}

// Gated RMSNorm epilogue over tokens 0 .. n-1 in shared memory: out = o *
// rsqrt(mean(o^2) + eps) * w * silu(z), written at the rows in s.row.  With
// SPLIT > 1 the mean-square is combined across the cluster through
// distributed shared memory.
template <int SPLIT, int W = 8 / SPLIT>
__device__ __forceinline__ void epilogue(Smem& s, const Params& p, int h, int n, int warp, int lane, int rank) {
    constexpr int CW = kV / SPLIT;  // V columns of this CTA
    const bool gated = p.z != nullptr;
    if (SPLIT > 1 && gated) {
        for (int t = warp; t < n; t += W) {
            float ss = 0.f;
            for (int c = lane; c < CW; c += 32) {
                const float o = s.o[t][rank * CW + c];
                ss += o * o;
            }
            ss = warp_sum(ss);
            if (lane == 0) s.red[t] = ss;
        }
        cg::this_cluster().sync();
    }
    for (int t = warp; t < n; t += W) {
        float rinv = 1.0f;
        if (gated) {
            float ss = 0.f;
            if (SPLIT > 1) {
                cg::cluster_group cl = cg::this_cluster();
#pragma unroll
                for (int rr = 0; rr < SPLIT; ++rr) ss += cl.map_shared_rank(&s.red[0], rr)[t];
            } else {
#pragma unroll
                for (int c = 0; c < kV / 32; ++c) {
                    const float o = s.o[t][lane + 32 * c];
                    ss += o * o;
                }
                ss = warp_sum(ss);
            }
            rinv = rsqrtf(ss * (1.0f / kV) + p.eps);
        }
        if (lane < CW / 4) {
            const int quad = rank * (CW / 4) + lane;
            const int col = quad * 4;
            const int r = s.row[t];
            const float4 o4 = *reinterpret_cast<const float4*>(&s.o[t][col]);
            float y[4] = {o4.x, o4.y, o4.z, o4.w};
            if (gated) {
                float zz[4], ww[4];
                unpack_bf16x4(s.z[t][quad], zz);
                unpack_bf16x4(s.w[quad], ww);
#pragma unroll
                for (int e = 0; e < 4; ++e) y[e] = y[e] * rinv * ww[e] * (zz[e] / (1.0f + expf(-zz[e])));
            }
            *reinterpret_cast<uint2*>(p.out + r * p.out_stride + static_cast<int64_t>(h) * kV + col) =
                pack_bf16x4(y);
        }
    }
    if (SPLIT > 1 && gated) cg::this_cluster().sync();         // peers may still read s.red
}

// this lane's 4 elements of token row r: q, k (key head kh), v, z (v-head h)
__device__ __forceinline__ void load_token_quads(const Params& p, int r, int kh, int h, int lane, uint2& qraw,
                                                 uint2& kraw, uint2& vraw, uint2& zraw) {
    qraw = ldg_quad(p.q + r * p.q_stride + kh * kK + lane * 4);
    kraw = ldg_quad(p.k + r * p.k_stride + kh * kK + lane * 4);
    vraw = ldg_quad(p.v + r * p.v_stride + static_cast<int64_t>(h) * kV + lane * 4);
    zraw = p.z != nullptr ? ldg_quad(p.z + r * p.z_stride + static_cast<int64_t>(h) * kV + lane * 4)
                          : make_uint2(0, 0);
}

// ---- the short causal convolution in front of the step ------------------------------

// The three 4-channel groups of this lane in a projection row: q and k of key
// head kh, v of v-head h (channels in the order q | k | v).
__device__ __forceinline__ void conv_channels(const Params& p, int kh, int h, int lane, int (&ch)[3]) {
    const int qk = p.H_k * kK;
    ch[0] = kh * kK + lane * 4;
    ch[1] = qk + kh * kK + lane * 4;
    ch[2] = 2 * qk + h * kV + lane * 4;
}

// The W-1 rewound history rows in conv slot ci (rows a .. a+W-2, a =
// max(num_accepted, 1)), or null for zero history (ci < 0).
__device__ __forceinline__ const __nv_bfloat16* conv_history(const Params& p, long long ci, int acc) {
    return ci < 0 ? nullptr
                  : p.conv_pool + (ci * p.conv_state_len + max(acc, 1)) * static_cast<int64_t>(p.conv_dim);
}

// Row of the step's token tau of the sequence starting at bos (gathered
// through spec_token_indx when given); -1 when out of range.
__device__ __forceinline__ int conv_row(const Params& p, int bos, int tau) {
    const int n = bos + tau;
    const int r = p.sti != nullptr ? __ldg(p.sti + n) : n;
    return (r < 0 || r >= p.num_tokens) ? -1 : r;
}

// q, k, v of draft token t for this lane's channels: y = silu(bias + sum_w
// weight[w] x_{t-W+1+w}) over (the W-1 history rows at `hist`, null for zero
// history; then the step's rows), FP32.  Every load of the token is issued
// before the arithmetic.  Sets `bad` for an out-of-range row.
__device__ __forceinline__ void conv_token(const Params& p, int bos, int t, const int (&ch)[3],
                                           const __nv_bfloat16* hist, float (&y)[3][4], int& bad) {
    const int W = p.conv_width;
    uint2 raw[4][3];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const int tau = t - (W - 1) + w;
        const __nv_bfloat16* src = nullptr;
        if (w < W) {
            if (tau < 0) {
                if (hist != nullptr) src = hist + static_cast<int64_t>(W - 1 + tau) * p.conv_dim;
            } else {
                const int r = conv_row(p, bos, tau);
                if (r < 0) bad = 1;
                else src = p.x + r * p.x_stride;
            }
        }
#pragma unroll
        for (int g = 0; g < 3; ++g) raw[w][g] = src != nullptr ? ldg_quad(src + ch[g]) : make_uint2(0, 0);
    }
    // per group: bias, weights ([channel][W]: one 32-byte run per 4 channels
    // when W = 4; these stay in L1 across tokens), then the taps
#pragma unroll
    for (int g = 0; g < 3; ++g) {
        float wt[4][4];
        if (W == 4) {
            const uint4* wp = reinterpret_cast<const uint4*>(p.conv_w + static_cast<int64_t>(ch[g]) * 4);
            const uint4 w0 = __ldg(wp), w1 = __ldg(wp + 1);
            const uint32_t ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ww[j]));
                wt[j >> 1][(2 * j) & 3] = f.x;
                wt[j >> 1][(2 * j + 1) & 3] = f.y;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    wt[e][w] = w < W ? __bfloat162float(p.conv_w[static_cast<int64_t>(ch[g] + e) * W + w]) : 0.f;
        }
        float b4[4] = {0.f, 0.f, 0.f, 0.f};
        if (p.conv_b != nullptr) unpack_bf16x4(ldg_quad(p.conv_b + ch[g]), b4);
#pragma unroll
        for (int e = 0; e < 4; ++e) y[g][e] = b4[e];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            float u[4];
            unpack_bf16x4(raw[w][g], u);
#pragma unroll
            for (int e = 0; e < 4; ++e) y[g][e] = fmaf(wt[e][w], u[e], y[g][e]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) y[g][e] = __fdividef(y[g][e], 1.0f + __expf(-y[g][e]));   // SiLU
    }
}

// ---- the speculative decode kernel -------------------------------------------------
//
// Grid: one CTA per (unit, column slice); SPLIT CTAs of a unit form one cluster.
// Block: 128 / NCW / SPLIT warps, each owning NCW of the unit's 128 V columns.
template <typename StateT, int SPLIT, bool CONV = false, int NCW = kColsPerWarp, bool PIPE = false, int KS = 1>
__global__ void __launch_bounds__(Config<StateT, SPLIT, NCW, KS>::kThreads, 512 / Config<StateT, SPLIT, NCW, KS>::kThreads)
gdn_spec_decode_kernel(const __grid_constant__ Params p) {
    using C = Config<StateT, SPLIT, NCW, KS>;
    using L = Lanes<NCW, KS>;
    constexpr int W = C::kWarps;
    constexpr int WC = W / KS;                                  // warps per K half: column blocks of the CTA
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem& s = *reinterpret_cast<Smem*>(smem_raw);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = SPLIT > 1 ? static_cast<int>(blockIdx.x % SPLIT) : 0;
    const int unit = static_cast<int>(blockIdx.x / SPLIT);
    const int i = unit / p.H_v;
    const int h = unit - i * p.H_v;
    const int cgi = lane % L::kColGroups;  // column group: 4 consecutive columns
    const int rg = lane / L::kColGroups;   // row group: K rows kq 64 + rg + G j
    const int kq = warp / WC;              // this warp's half of K (0 unless KS = 2)
    const int wg = rank * WC + warp % WC;  // this warp's NCW-column block
    const int col0 = wg * NCW + cgi * 4;
    const int krow0 = kq * L::kSpan + rg;  // this lane's first K row
    const int row0 = kq * L::kSpan + rg * L::kRows;   // where its rows sit in the permuted k^ / q^

    // Launched with programmatic stream serialization: this CTA may become
    // resident while the previous kernel in the stream is still running.  It
    // waits (dep_wait) until that grid has completed and its writes are
    // visible before it touches memory the grid may have written, then lets
    // the next kernel's CTAs be scheduled.  By default the wait comes before
    // the first global access; GDN_PRE_INDEX moves it after the index reads,
    // GDN_PRE_TOKENS (with it) after the token prologue as well and
    // GDN_PRE_STATE (with it) after the state tile's load, so that those reads
    // overlap the previous grid's tail.  Every write (slots, out, the conv
    // slots, the status word) comes after the wait; every exit waits first, so
    // that no successor is released before this grid's predecessor has
    // completed.
    // (the fused convolution reads its history rows, conv slots, in the token
    // prologue: it runs the prologue early only when both the token rows and
    // the recurrent slots, state and conv, are declared)
    const bool pre_index = (p.flags & GDN_PRE_INDEX) != 0;
    const bool pre_both = (p.flags & (GDN_PRE_TOKENS | GDN_PRE_STATE)) == (GDN_PRE_TOKENS | GDN_PRE_STATE);
    const bool pre_tokens = pre_index && (CONV ? pre_both : (p.flags & GDN_PRE_TOKENS) != 0);
    const bool pre_state = pre_index && (CONV ? pre_both : (p.flags & GDN_PRE_STATE) != 0);
    bool waited = false;
    auto dep_wait = [&]() {
        if (!waited) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            waited = true;
        }
    };
    if (!pre_index) dep_wait();

    // ---- resolve the work item (every thread computes the same answer) ----
    // The sequence's slot row is read in the same round trip as its length and
    // acceptance, so the read slot costs no extra dependent load; so are the
    // total token count and, with the convolution, the sequence's conv slots.
    const int32_t* slot_row = p.idx + static_cast<int64_t>(i) * p.stride;
    int slots[kMaxT];
#pragma unroll
    for (int j = 0; j < kMaxT; ++j) slots[j] = j < p.stride ? __ldg(slot_row + j) : -1;
    const int bos = __ldg(p.cu + i);
    const int q_len = __ldg(p.cu + i + 1) - bos;
    const int acc = __ldg(p.num_acc + i);
    const int cu_total = __ldg(p.cu + p.batch);
    long long conv_in = -1, conv_out = -1;                     // this sequence's conv slots
    if constexpr (CONV) {
        conv_in = __ldg(p.conv_in + i);
        conv_out = __ldg(p.conv_out + i);
    }
    if (q_len <= 0) { dep_wait(); return; }                    // nothing to do
    // token positions must lie inside [0, cu_seqlens[batch]), the length of
    // spec_token_indx (rows themselves are range-checked below)
    if (bos < 0 || bos + q_len > cu_total) { dep_wait(); raise_flag(p, rank, GDN_FLAG_TOKEN_ROW); return; }
    if (acc > p.stride) { dep_wait(); raise_flag(p, rank, GDN_FLAG_ACCEPTED); return; }
    if (q_len > p.max_T || q_len > p.stride) { dep_wait(); raise_flag(p, rank, GDN_FLAG_QLEN); return; }
    // rewind: the state after the last accepted token; acc-1 clamped at 0
    const int rj = max(acc - 1, 0);
    long long rs = 0;
#pragma unroll
    for (int j = 0; j < kMaxT; ++j)
        if (j == rj) rs = slots[j];
    if (rj >= kMaxT) rs = __ldg(slot_row + rj);                // acceptance beyond the first 8 columns
    if (rs < 0) { dep_wait(); return; }                        // padded sequence
    if (rs >= p.num_slots) { dep_wait(); raise_flag(p, rank, GDN_FLAG_SLOT_RANGE); return; }
    if constexpr (CONV) {
        if (conv_in >= p.num_conv_slots || conv_out >= p.num_conv_slots) {
            dep_wait();
            raise_flag(p, rank, GDN_FLAG_SLOT_RANGE);
            return;
        }
    }
    // ---- load this lane's R x 4 block of the state tile (FP32 in registers):
    //      rows rg + G r, columns col0 .. col0 + 3; issued before the token
    //      prologue (ahead of the wait with GDN_PRE_STATE), or after the
    //      prologue when only the prologue runs ahead of the wait ----
    const StateT* src = static_cast<const StateT*>(p.pool) + (rs * p.H_v + h) * kTile;
    float S[L::kRows][4];
    if (!pre_state && !pre_tokens) dep_wait();
    if (pre_state || !pre_tokens) {
#pragma unroll
        for (int r = 0; r < L::kRows; ++r)
            StateIO<StateT>::load4(src + static_cast<int64_t>(krow0 + L::kRowGroups * r) * kV + col0, S[r]);
    }
    if (pre_state && !pre_tokens) dep_wait();

    // ---- per-token prologue: gather rows, gates, normalised q / k, v, z ----
    const int kh = h / p.group;
    if (p.z != nullptr && warp == 0) s.w[lane] = ldg_quad(p.norm_w + lane * 4);
    int bad = 0;

#pragma unroll
    for (int j = 0; j < (kMaxT + W - 1) / W; ++j) {            // warp w: tokens w, w + W, ...
        const int t = warp + j * W;
        if (t < q_len) {
            const int n = bos + t;
            const int r = p.sti != nullptr ? __ldg(p.sti + n) : n;
            if (r < 0 || r >= p.num_tokens) {
                bad = 1;
            } else {
                long long ws = 0;
#pragma unroll
                for (int jj = 0; jj < kMaxT; ++jj)
                    if (jj == t) ws = slots[jj];                   // t < q_len <= 8
                if constexpr (CONV) {
                    int conv_ch[3];
                    conv_channels(p, kh, h, lane, conv_ch);
                    float y[3][4];
                    conv_token(p, bos, t, conv_ch, conv_history(p, conv_in, acc), y, bad);
                    const uint2 zraw = p.z != nullptr
                                           ? ldg_quad(p.z + r * p.z_stride + static_cast<int64_t>(h) * kV + lane * 4)
                                           : make_uint2(0, 0);
                    prologue_token_f<NCW, KS>(s, p, h, t, r, lane, y[0], y[1], y[2], zraw, ws);
                } else {
                    uint2 qraw, kraw, vraw, zraw;
                    load_token_quads(p, r, kh, h, lane, qraw, kraw, vraw, zraw);
                    prologue_token<NCW, KS>(s, p, h, t, r, lane, qraw, kraw, vraw, zraw, ws);
                }
            }
        }
    }
    if (pre_tokens) {
        dep_wait();
        if (!pre_state) {
#pragma unroll
            for (int r = 0; r < L::kRows; ++r)
                StateIO<StateT>::load4(src + static_cast<int64_t>(krow0 + L::kRowGroups * r) * kV + col0, S[r]);
        }
    }
    // publishes the prologue; every CTA of the cluster checks every token row,
    // so the skip decision below is the same in all of them
    if (__syncthreads_or(bad)) { raise_flag(p, rank, GDN_FLAG_TOKEN_ROW); return; }

    // ---- the new conv slot: the history, then this step's rows.  Channels of
    //      v-head h by this unit; q / k channels of the key head by its first
    //      v-head only.  (Only with SPLIT = 1.) ----
    if constexpr (CONV) {
        if (conv_out >= 0) {
            int conv_ch[3];
            conv_channels(p, kh, h, lane, conv_ch);
            const __nv_bfloat16* hist = conv_history(p, conv_in, acc);
            __nv_bfloat16* dst = p.conv_pool + conv_out * p.conv_state_len * static_cast<int64_t>(p.conv_dim);
            const int g0 = (h % p.group) == 0 ? 0 : 2;
            const int Wc = p.conv_width;
            if (warp < q_len) {
                const int r = conv_row(p, bos, warp);
                const __nv_bfloat16* src = p.x + r * p.x_stride;
                for (int g = g0; g < 3; ++g)
                    *reinterpret_cast<uint2*>(dst + static_cast<int64_t>(Wc - 1 + warp) * p.conv_dim + conv_ch[g]) =
                        ldg_quad(src + conv_ch[g]);
            }
            if (warp == 0) {
                for (int m = 0; m < Wc - 1; ++m)
                    for (int g = g0; g < 3; ++g)
                        *reinterpret_cast<uint2*>(dst + static_cast<int64_t>(m) * p.conv_dim + conv_ch[g]) =
                            hist != nullptr ? ldg_quad(hist + static_cast<int64_t>(m) * p.conv_dim + conv_ch[g])
                                            : make_uint2(0, 0);
            }
        }
    }

    // ---- the draft tokens, in order ----
    // this warp's staging buffer for the tensor stores (128-byte aligned)
    StateT* stage = reinterpret_cast<StateT*>(smem_raw + C::kStageOffset +
                                              ((128u - (smem_addr(smem_raw) & 127u)) & 127u)) +
                    warp * C::kStageElems;
    for (int t = 0; t < q_len; ++t)
        token_step<StateT, NCW, PIPE, KS>(S, s, p, t, h, lane, col0, row0, rank, stage, kq, warp % WC);
    if constexpr (PIPE) write_slot<StateT, NCW, KS>(S, p, s.ws[q_len - 1], h, lane, col0, rank, stage, kq);

    // ---- gated RMSNorm epilogue ----
    __syncthreads();                                           // s.o of this CTA complete
    epilogue<SPLIT, W>(s, p, h, q_len, warp, lane, rank);
    if (lane == 0) tma_wait_all();                              // the slot writes have landed
}

// ---- the prefill kernel (recurrent form) -------------------------------------------
//
// One CTA of 8 warps per (sequence, v-head): the prompt runs through the same
// per-token step as the decode path, 8 tokens per round of prologue / tokens /
// epilogue, with the FP32 state in registers from the first token to the
// last; only the final state is stored.
template <typename StateT>
__global__ void __launch_bounds__(256, 2) gdn_prefill_kernel(const Params p) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem& s = *reinterpret_cast<Smem*>(smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int unit = static_cast<int>(blockIdx.x);
    const int i = unit / p.H_v;
    const int h = unit - i * p.H_v;
    const int cgi = lane & 3;
    const int rg = lane >> 2;
    const int col0 = warp * kColsPerWarp + cgi * 4;
    const int row0 = rg * kRowsPerLane;

    const int bos = __ldg(p.cu + i);
    const int L = __ldg(p.cu + i + 1) - bos;
    const long long rs = __ldg(p.read_slots + i);
    const long long wsl = __ldg(p.write_slots + i);
    if (L <= 0) return;
    if (bos < 0 || bos + L > p.num_tokens) { raise_flag(p, 0, GDN_FLAG_TOKEN_ROW); return; }
    if (rs >= p.num_slots || wsl >= p.num_slots) { raise_flag(p, 0, GDN_FLAG_SLOT_RANGE); return; }

    float S[kRowsPerLane][4];
    if (rs >= 0) {
        const StateT* src = static_cast<const StateT*>(p.pool) + (rs * p.H_v + h) * kTile;
#pragma unroll
        for (int r = 0; r < kRowsPerLane; ++r)
            StateIO<StateT>::load4(src + static_cast<int64_t>(rg + 8 * r) * kV + col0, S[r]);
    } else {
#pragma unroll
        for (int r = 0; r < kRowsPerLane; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) S[r][c] = 0.f;         // no initial state
    }
    const int kh = h / p.group;
    if (p.z != nullptr && warp == 0) s.w[lane] = ldg_quad(p.norm_w + lane * 4);
    for (int c0 = 0; c0 < L; c0 += kMaxT) {
        const int n = min(kMaxT, L - c0);
        if (warp < n) {
            const int r = bos + c0 + warp;
            uint2 qraw, kraw, vraw, zraw;
            load_token_quads(p, r, kh, h, lane, qraw, kraw, vraw, zraw);
            prologue_token(s, p, h, warp, r, lane, qraw, kraw, vraw, zraw, -1);
        }
        __syncthreads();                                       // prologue published
        for (int t = 0; t < n; ++t) token_step<StateT>(S, s, p, t, h, lane, col0, row0, 0, nullptr);
        __syncthreads();                                       // s.o complete
        epilogue<1>(s, p, h, n, warp, lane, 0);
        __syncthreads();                                       // before the next round overwrites s
    }
    if (wsl >= 0) {
        StateT* d = static_cast<StateT*>(p.pool) + (wsl * p.H_v + h) * kTile + col0;
#pragma unroll
        for (int r = 0; r < kRowsPerLane; ++r) StateIO<StateT>::store4(d + static_cast<int64_t>(rg + 8 * r) * kV, S[r]);
    }
}

// ---- host side ----------------------------------------------------------------

template <typename StateT, int SPLIT, bool CONV = false, int NCW = kColsPerWarp, bool PIPE = false, int KS = 1>
cudaError_t launch(const Params& p, int64_t units, cudaStream_t stream) {
    using C = Config<StateT, SPLIT, NCW, KS>;
    auto kernel = gdn_spec_decode_kernel<StateT, SPLIT, CONV, NCW, PIPE, KS>;
    if (C::kSmem > 48 * 1024) {
        // opt in to more than 48 KB of dynamic shared memory, once per device
        static bool done[64] = {false};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64 || !done[dev]) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(C::kSmem));
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) done[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units * SPLIT), 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (SPLIT > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = SPLIT;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Pipelined slot writes (token_step's PIPE) when every CTA of the launch has
// an SM to itself: there a CTA's token chain is latency-bound and staging one
// token's state while the next token's products form shortens it (BS=4 bf16
// 7.78 -> 7.63 us, BS=8 8.93 -> 8.70 us); with two CTAs per SM the longer
// live ranges cost more than the overlap saves (BS=32 28.89 -> 29.29 us), and
// the narrow layout loses too (BS=4 fp32 9.41 -> 9.57 us).
bool pipelined(int64_t ctas) {
    static int sms[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    return ctas <= sms[dev];
}

template <typename StateT>
cudaError_t launch_split(const Params& p, int64_t units, int split, cudaStream_t stream) {
    switch (split) {
    case 1:
        return pipelined(units) ? launch<StateT, 1, false, kColsPerWarp, true>(p, units, stream)
                                : launch<StateT, 1>(p, units, stream);
    case 2: return launch<StateT, 2>(p, units, stream);
    case 4: return launch<StateT, 4>(p, units, stream);
    case GDN_SPLIT_NARROW | 2: return launch<StateT, 2, false, 8>(p, units, stream);
    case GDN_SPLIT_NARROW | 4: return launch<StateT, 4, false, 8>(p, units, stream);
    case GDN_SPLIT_HALFK | 1:
        return pipelined(units) ? launch<StateT, 1, false, kColsPerWarp, true, 2>(p, units, stream)
                                : launch<StateT, 1, false, kColsPerWarp, false, 2>(p, units, stream);
    case GDN_SPLIT_HALFK | 2:
        return pipelined(2 * units) ? launch<StateT, 2, false, kColsPerWarp, true, 2>(p, units, stream)
                                    : launch<StateT, 2, false, kColsPerWarp, false, 2>(p, units, stream);
    default: return launch<StateT, 8>(p, units, stream);
    }
}

template <typename StateT>
cudaError_t launch_prefill(const Params& p, int64_t units, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = sizeof(Smem);
    cfg.stream = stream;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, gdn_prefill_kernel<StateT>, p);
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// The state pool as a 2-D tensor for the decode kernel's per-warp tensor
// stores: rows = slots * H_v * K, columns = V, box = 128 rows x `cols` columns
// (the columns a warp owns: 16, or 8 in the narrow layout).
// cuTensorMapEncodeTiled is reached through the runtime's driver entry point
// (no link against the driver library); maps are cached per host thread for
// the last few pools, so a steady stream of calls encodes nothing.
gdn_status make_pool_map(Params& p, void* pool, int64_t num_slots, int32_t H_v, gdn_dtype dt, int cols,
                         int box_rows = kK) {
    using Encode = PFN_cuTensorMapEncodeTiled_v12000;
    static const Encode encode = [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            fn = nullptr;
        return reinterpret_cast<Encode>(fn);
    }();
    const int64_t rows = num_slots * H_v * kK;
    if (rows > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;      // row coordinates are 32-bit
    if (encode == nullptr) return GDN_ERR_CUDA;
    struct Entry {
        const void* pool;
        int64_t rows;
        int dt, cols, box_rows;
        CUtensorMap map;
    };
    thread_local Entry cache[4] = {};
    thread_local int next = 0;
    for (const Entry& e : cache)
        if (e.pool == pool && e.rows == rows && e.dt == dt && e.cols == cols && e.box_rows == box_rows) {
            p.pool_map = e.map;
            return GDN_OK;
        }
    const size_t elem = dt == GDN_F32 ? 4 : 2;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kV), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kV * elem)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType type = dt == GDN_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : dt == GDN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap map;
    if (encode(&map, type, 2, pool, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return GDN_ERR_CUDA;
    cache[next] = Entry{pool, rows, static_cast<int>(dt), cols, box_rows, map};
    next = (next + 1) % 4;
    p.pool_map = map;
    return GDN_OK;
}

// One CTA per unit, each warp owning 16 V columns, at every batch size
// measured (4 to 256 sequences of 16 v-heads) but two: an FP32 state with at
// most 64 units (4 sequences of 16 v-heads) runs the half-K layout over 2-CTA
// clusters (BS=4: 9.40 us with the narrow layout, 9.08 us), and with at most
// 128 units the half-K layout in one 16-warp CTA (BS=8: 13.52 -> 13.06 us).
// Splitting the 16-column warps over a cluster shortens no per-token chain and
// adds cluster barriers; with 16-bit states neither half-K form nor the narrow
// layout beats one 8-warp CTA per unit (BS=4 bf16: 7.64 us; half-K 7.98 /
// 8.31 us; narrow 9.47 us).
int choose_split(int64_t units, gdn_dtype dt) {
    if (dt == GDN_F32 && units <= 64) return GDN_SPLIT_HALFK | 2;
    if (dt == GDN_F32 && units <= 128) return GDN_SPLIT_HALFK | 1;
    return 1;
}

gdn_status check_dims(const gdn_dims* d) {
    if (d == nullptr) return GDN_ERR_NULL_ARG;
    if (d->batch < 0 || d->num_tokens < 0 || d->H_k <= 0 || d->H_v <= 0 || d->spec_stride < 1 ||
        d->num_slots < 1 || d->H_v % d->H_k != 0 ||
        (d->flags & ~(GDN_PRE_INDEX | GDN_PRE_TOKENS | GDN_PRE_STATE)) != 0)
        return GDN_ERR_BAD_SHAPE;
    if (d->max_T < 1 || d->max_T > kMaxT) return GDN_ERR_BAD_SHAPE;
    if (d->q_stride < 0 || d->k_stride < 0 || d->v_stride < 0 || d->a_stride < 0 || d->b_stride < 0 ||
        d->z_stride < 0 || d->out_stride < 0)
        return GDN_ERR_BAD_SHAPE;
    if (d->K != kK || d->V != kV) return GDN_ERR_UNSUPPORTED;
    if (!(d->split == 0 || d->split == 1 || d->split == 2 || d->split == 4 || d->split == 8 ||
          d->split == (GDN_SPLIT_NARROW | 2) || d->split == (GDN_SPLIT_NARROW | 4) ||
          d->split == (GDN_SPLIT_HALFK | 1) || d->split == (GDN_SPLIT_HALFK | 2)))
        return GDN_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(d->batch) * d->H_v * 8 > 0x7fffffffLL) return GDN_ERR_BAD_SHAPE;
    return GDN_OK;
}

// Sizes shared by both entry points (decode-only fields are not checked here).
gdn_status check_common_dims(const gdn_dims* d) {
    if (d == nullptr) return GDN_ERR_NULL_ARG;
    if (d->batch < 0 || d->num_tokens < 0 || d->H_k <= 0 || d->H_v <= 0 || d->num_slots < 1 ||
        d->H_v % d->H_k != 0 || d->flags != 0)
        return GDN_ERR_BAD_SHAPE;
    if (d->q_stride < 0 || d->k_stride < 0 || d->v_stride < 0 || d->a_stride < 0 || d->b_stride < 0 ||
        d->z_stride < 0 || d->out_stride < 0)
        return GDN_ERR_BAD_SHAPE;
    if (d->K != kK || d->V != kV) return GDN_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(d->batch) * d->H_v * 8 > 0x7fffffffLL) return GDN_ERR_BAD_SHAPE;
    return GDN_OK;
}

// Fill the kernel parameters from the call and check pointers and alignment.
gdn_status make_params(Params& p, const void* q, const void* k, const void* v, const void* a, const void* b,
                       const void* z, const float* A_log, const void* dt_bias, const void* norm_w, void* state_pool,
                       const int32_t* cu_seqlens, void* out, const gdn_dims* dims, float scale, float eps,
                       int32_t* status_word) {
    if (!q || !k || !v || !a || !b || !A_log || !dt_bias || !state_pool || !cu_seqlens || !out)
        return GDN_ERR_NULL_ARG;
    if ((z == nullptr) != (norm_w == nullptr)) return GDN_ERR_NULL_ARG;
    const int64_t qk_row = static_cast<int64_t>(dims->H_k) * kK;
    const int64_t v_row = static_cast<int64_t>(dims->H_v) * kV;
    p = Params{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.a = static_cast<const __nv_bfloat16*>(a);
    p.b = static_cast<const __nv_bfloat16*>(b);
    p.z = static_cast<const __nv_bfloat16*>(z);
    p.A_log = A_log;
    p.dt_bias = static_cast<const __nv_bfloat16*>(dt_bias);
    p.norm_w = static_cast<const __nv_bfloat16*>(norm_w);
    p.pool = state_pool;
    p.cu = cu_seqlens;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.status = status_word;
    p.q_stride = dims->q_stride ? dims->q_stride : qk_row;
    p.k_stride = dims->k_stride ? dims->k_stride : qk_row;
    p.v_stride = dims->v_stride ? dims->v_stride : v_row;
    p.a_stride = dims->a_stride ? dims->a_stride : dims->H_v;
    p.b_stride = dims->b_stride ? dims->b_stride : dims->H_v;
    p.z_stride = dims->z_stride ? dims->z_stride : v_row;
    p.out_stride = dims->out_stride ? dims->out_stride : v_row;
    p.num_slots = dims->num_slots;
    p.batch = dims->batch;
    p.num_tokens = dims->num_tokens;
    p.H_k = dims->H_k;
    p.H_v = dims->H_v;
    p.stride = dims->spec_stride;
    p.max_T = dims->max_T;
    p.group = dims->H_v / dims->H_k;
    p.flags = dims->flags;
    p.scale = scale;
    p.eps = eps;
    // vector accesses: 16 B state rows, 8 B bf16 quads
    if (!aligned(state_pool, 16) || !aligned(q, 8) || !aligned(k, 8) || !aligned(v, 8) || !aligned(out, 8) ||
        (z && !aligned(z, 8)) || (norm_w && !aligned(norm_w, 8)) || !aligned(a, 2) || !aligned(b, 2) ||
        !aligned(dt_bias, 2) || !aligned(A_log, 4) || !aligned(cu_seqlens, 4) ||
        (status_word && !aligned(status_word, 4)))
        return GDN_ERR_MISALIGNED;
    if (p.q_stride % 4 || p.k_stride % 4 || p.v_stride % 4 || p.z_stride % 4 || p.out_stride % 4)
        return GDN_ERR_MISALIGNED;
    return GDN_OK;
}

template <template <typename> class Launcher, typename... Args>
cudaError_t by_state_dtype(gdn_dtype dt, Args... args) {
    switch (dt) {
    case GDN_F32: return Launcher<float>::run(args...);
    case GDN_BF16: return Launcher<__nv_bfloat16>::run(args...);
    default: return Launcher<__half>::run(args...);
    }
}

template <typename StateT>
struct DecodeLauncher {
    static cudaError_t run(const Params& p, int64_t units, int split, cudaStream_t s) {
        return launch_split<StateT>(p, units, split, s);
    }
};

template <typename StateT>
struct ConvDecodeLauncher {
    static cudaError_t run(const Params& p, int64_t units, cudaStream_t s) { return launch<StateT, 1, true>(p, units, s); }
};

template <typename StateT>
struct PrefillLauncher {
    static cudaError_t run(const Params& p, int64_t units, cudaStream_t s) { return launch_prefill<StateT>(p, units, s); }
};

}  // namespace

extern "C" {

gdn_status gdn_spec_decode(const void* q, const void* k, const void* v, const void* a, const void* b,
                           const void* z, const float* A_log, const void* dt_bias, const void* norm_w,
                           void* state_pool, const int32_t* state_indices, const int32_t* num_accepted,
                           const int32_t* cu_seqlens, const int32_t* spec_token_indx, void* out,
                           const gdn_dims* dims, float scale, float eps, gdn_dtype state_dtype,
                           int32_t* status_word, gdn_stream_t stream) {
    const gdn_status ds = check_dims(dims);
    if (ds != GDN_OK) return ds;
    if (state_dtype != GDN_F32 && state_dtype != GDN_BF16 && state_dtype != GDN_F16) return GDN_ERR_UNSUPPORTED;
    if (dims->batch == 0) return GDN_OK;
    if (!state_indices || !num_accepted) return GDN_ERR_NULL_ARG;
    Params p;
    const gdn_status ps = make_params(p, q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, cu_seqlens, out,
                                      dims, scale, eps, status_word);
    if (ps != GDN_OK) return ps;
    if (!aligned(state_indices, 4) || !aligned(num_accepted, 4) || (spec_token_indx && !aligned(spec_token_indx, 4)))
        return GDN_ERR_MISALIGNED;
    p.idx = state_indices;
    p.num_acc = num_accepted;
    p.sti = spec_token_indx;
    const int64_t units = static_cast<int64_t>(dims->batch) * dims->H_v;
    const int split = dims->split ? dims->split : choose_split(units, state_dtype);
    const gdn_status ms = make_pool_map(p, state_pool, dims->num_slots, dims->H_v, state_dtype,
                                        (split & GDN_SPLIT_NARROW) ? 8 : kColsPerWarp,
                                        (split & GDN_SPLIT_HALFK) ? kK / 2 : kK);
    if (ms != GDN_OK) return ms;
    const cudaError_t err =
        by_state_dtype<DecodeLauncher>(state_dtype, p, units, split, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_spec_decode_conv(const void* x, const void* conv_weight, const void* conv_bias, void* conv_pool,
                                const int32_t* conv_in, const int32_t* conv_out, const gdn_conv_dims* cdims,
                                const void* a, const void* b, const void* z, const float* A_log, const void* dt_bias,
                                const void* norm_w, void* state_pool, const int32_t* state_indices,
                                const int32_t* num_accepted, const int32_t* cu_seqlens,
                                const int32_t* spec_token_indx, void* out, const gdn_dims* dims, float scale,
                                float eps, gdn_dtype state_dtype, int32_t* status_word, gdn_stream_t stream) {
    const gdn_status ds = check_dims(dims);
    if (ds != GDN_OK) return ds;
    if (cdims == nullptr) return GDN_ERR_NULL_ARG;
    if (cdims->width < 1 || cdims->width > 4 || cdims->num_conv_slots < 1 || cdims->x_stride < 0 ||
        cdims->reserved[0] != 0 || cdims->reserved[1] != 0 ||
        static_cast<int64_t>(cdims->state_len) < cdims->width - 1 + static_cast<int64_t>(dims->spec_stride))
        return GDN_ERR_BAD_SHAPE;
    if (state_dtype != GDN_F32 && state_dtype != GDN_BF16 && state_dtype != GDN_F16) return GDN_ERR_UNSUPPORTED;
    if (dims->split > 1) return GDN_ERR_UNSUPPORTED;
    if (dims->batch == 0) return GDN_OK;
    if (!state_indices || !num_accepted || !x || !conv_weight || !conv_pool || !conv_in || !conv_out)
        return GDN_ERR_NULL_ARG;
    Params p;
    // q, k and v are not read on this path: x stands in for the null checks
    const gdn_status ps = make_params(p, x, x, x, a, b, z, A_log, dt_bias, norm_w, state_pool, cu_seqlens, out,
                                      dims, scale, eps, status_word);
    if (ps != GDN_OK) return ps;
    if (!aligned(state_indices, 4) || !aligned(num_accepted, 4) || (spec_token_indx && !aligned(spec_token_indx, 4)) ||
        !aligned(conv_pool, 8) || (conv_bias && !aligned(conv_bias, 8)) ||
        !aligned(conv_weight, cdims->width == 4 ? 16 : 2) ||
        !aligned(conv_in, 4) || !aligned(conv_out, 4) || cdims->x_stride % 4 != 0)
        return GDN_ERR_MISALIGNED;
    p.idx = state_indices;
    p.num_acc = num_accepted;
    p.sti = spec_token_indx;
    const gdn_status ms = make_pool_map(p, state_pool, dims->num_slots, dims->H_v, state_dtype, kColsPerWarp);
    if (ms != GDN_OK) return ms;
    p.conv_dim = 2 * dims->H_k * kK + dims->H_v * kV;
    p.x = static_cast<const __nv_bfloat16*>(x);
    p.x_stride = cdims->x_stride ? cdims->x_stride : p.conv_dim;
    p.conv_w = static_cast<const __nv_bfloat16*>(conv_weight);
    p.conv_b = static_cast<const __nv_bfloat16*>(conv_bias);
    p.conv_pool = static_cast<__nv_bfloat16*>(conv_pool);
    p.conv_in = conv_in;
    p.conv_out = conv_out;
    p.num_conv_slots = cdims->num_conv_slots;
    p.conv_width = cdims->width;
    p.conv_state_len = cdims->state_len;
    const int64_t units = static_cast<int64_t>(dims->batch) * dims->H_v;
    const cudaError_t err =
        by_state_dtype<ConvDecodeLauncher>(state_dtype, p, units, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_prefill(const void* q, const void* k, const void* v, const void* a, const void* b, const void* z,
                       const float* A_log, const void* dt_bias, const void* norm_w, void* state_pool,
                       const int32_t* read_slots, const int32_t* write_slots, const int32_t* cu_seqlens, void* out,
                       const gdn_dims* dims, float scale, float eps, gdn_dtype state_dtype, int32_t* status_word,
                       gdn_stream_t stream) {
    const gdn_status ds = check_common_dims(dims);
    if (ds != GDN_OK) return ds;
    if (state_dtype != GDN_F32 && state_dtype != GDN_BF16 && state_dtype != GDN_F16) return GDN_ERR_UNSUPPORTED;
    if (dims->batch == 0) return GDN_OK;
    if (!read_slots || !write_slots) return GDN_ERR_NULL_ARG;
    Params p;
    const gdn_status ps = make_params(p, q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, cu_seqlens, out,
                                      dims, scale, eps, status_word);
    if (ps != GDN_OK) return ps;
    if (!aligned(read_slots, 4) || !aligned(write_slots, 4)) return GDN_ERR_MISALIGNED;
    p.read_slots = read_slots;
    p.write_slots = write_slots;
    const int64_t units = static_cast<int64_t>(dims->batch) * dims->H_v;
    const cudaError_t err =
        by_state_dtype<PrefillLauncher>(state_dtype, p, units, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_prefill_chunked(const void* q, const void* k, const void* v, const void* a, const void* b,
                               const void* z, const float* A_log, const void* dt_bias, const void* norm_w,
                               void* state_pool, const int32_t* read_slots, const int32_t* write_slots,
                               const int32_t* cu_seqlens, void* out, const gdn_dims* dims, float scale, float eps,
                               gdn_dtype state_dtype, int32_t* status_word, gdn_stream_t stream) {
    const gdn_status ds = check_common_dims(dims);
    if (ds != GDN_OK) return ds;
    if (state_dtype != GDN_F32 && state_dtype != GDN_BF16 && state_dtype != GDN_F16) return GDN_ERR_UNSUPPORTED;
    if (dims->batch == 0) return GDN_OK;
    if (!read_slots || !write_slots) return GDN_ERR_NULL_ARG;
    Params p;
    const gdn_status ps = make_params(p, q, k, v, a, b, z, A_log, dt_bias, norm_w, state_pool, cu_seqlens, out,
                                      dims, scale, eps, status_word);
    if (ps != GDN_OK) return ps;
    if (!aligned(read_slots, 4) || !aligned(write_slots, 4)) return GDN_ERR_MISALIGNED;
    p.read_slots = read_slots;
    p.write_slots = write_slots;
    const int64_t units = static_cast<int64_t>(dims->batch) * dims->H_v;
    const cudaError_t err =
        gdn_internal::launch_prefill_chunked(p, units, state_dtype, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int32_t gdn_spec_decode_split(const gdn_dims* dims, gdn_dtype state_dtype) {
    if (check_dims(dims) != GDN_OK) return 0;
    if (state_dtype != GDN_F32 && state_dtype != GDN_BF16 && state_dtype != GDN_F16) return 0;
    if (dims->split) return dims->split;
    return choose_split(static_cast<int64_t>(dims->batch) * dims->H_v, state_dtype);
}

const char* gdn_status_str(gdn_status status) {
    switch (status) {
    case GDN_OK: return "ok";
    case GDN_ERR_NULL_ARG: return "a required pointer is NULL (or z / norm_w not both set)";
    case GDN_ERR_BAD_SHAPE: return "bad sizes";
    case GDN_ERR_UNSUPPORTED: return "unsupported head dims, state dtype or split";
    case GDN_ERR_MISALIGNED: return "a pointer or row stride is misaligned";
    case GDN_ERR_CUDA: return "CUDA launch failed";
    }
    return "unknown status";
}

void gdn_set_wait_limit(uint32_t polls) { __atomic_store_n(&gdn_internal::g_wait_limit, polls, __ATOMIC_RELAXED); }

int32_t gdn_version(void) { return GDNSPEC_VERSION; }

}  // extern "C"
