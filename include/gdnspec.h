/*
 * libgdnspec -- the speculative / MTP decode step of a Gated DeltaNet (GDN)
 * linear-attention layer, as hand-written CUDA for sm_103a (GB300), behind a
 * plain C ABI.
 *
 * The operation follows these vLLM pull-request report pages:
 *   "PR #51674 report -- [Kernel][Perf] Add fused CUDA post-conv MTP decode
 *    kernel for Qwen3.5 GDN", implementation steps 1-3 and the
 *    _custom_ops.py listing (one fused step per (request, v-head): rewind to
 *    the last accepted state slot, up to 8 draft tokens through the gated
 *    delta rule in order, gated RMSNorm epilogue; scale = 128^-0.5,
 *    norm_eps = 1e-5; K = V = 128; the state is updated in place);
 *   "PR #46090 report -- [CPU][Spec Decode] Support DFlash speculative
 *    decoding for GDN models on CPU", implementation step 3 and the fla.cpp
 *    listing (initial slot spec_indices[i, max(num_accepted-1, 0)], the
 *    state after every token written to its own slot, q_len <= 0 skipped,
 *    v-head h uses key head h / (H_v / H_k));
 *   "PR #52191 report -- [CPU] Support FP16/BF16 persisted GDN state on
 *    AMX", implementation steps 3-4 (arithmetic in FP32, the state stored as
 *    FP32 / BF16 / FP16 with one rounding per slot write);
 *   "PR #51812 report -- [Bugfix] Align Qwen GDN gates with speculative
 *    tokens", implementation steps 1-3 (q/k/v and the a/b gates gathered with
 *    one shared spec_token_indx in a mixed batch).
 *
 * Per (sequence i, v-head h), with S the K x V state (V contiguous) and
 * r(t) the token row of draft token t:
 *     S <- state_pool[state_indices[i, max(num_accepted[i]-1, 0)], h]
 *     for t in 0 .. q_len-1:
 *         g = -exp(A_log[h]) * softplus(a[r,h] + dt_bias[h]);  beta = sigmoid(b[r,h])
 *         k^ = k[r,kh] / |k[r,kh]|;  q^ = q[r,kh] / |q[r,kh]| * scale
 *         S <- S e^g;  v' = beta (v[r,h] - S^T k^);  S <- S + k^ v'^T;  o = S^T q^
 *         if state_indices[i, t] >= 0: state_pool[state_indices[i, t], h] <- round(S)
 *         out[r,h] = round_bf16( o * rsqrt(mean(o^2) + eps) * norm_w * silu(z[r,h]) )
 * (softplus(x) = x above 20; |x| = sqrt(sum x^2 + 1e-6).)
 *
 * Everything here is asynchronous on the caller's stream: the library never
 * synchronises, never reads device data on the host and allocates nothing, so
 * a call can be captured in a CUDA graph.  All tensor pointers are
 * caller-owned DEVICE memory (for example PyTorch tensors); the library keeps
 * no pointer after the call returns.
 */
#ifndef GDNSPEC_H
#define GDNSPEC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 2: gdn_spec_decode_split takes the state dtype; dims->split accepts GDN_SPLIT_NARROW
   3: dims->flags (formerly reserved): GDN_PRE_INDEX, GDN_PRE_TOKENS, GDN_PRE_STATE
   4: dims->split accepts GDN_SPLIT_HALFK | 1 and | 2, the automatic choice for small
      FP32 batches */
#define GDNSPEC_VERSION 4

#if defined(__GNUC__)
#define GDNSPEC_API __attribute__((visibility("default")))
#else
#define GDNSPEC_API
#endif

/* Host-side result of a call.  Nothing is launched unless GDN_OK. */
typedef enum {
    GDN_OK = 0,
    GDN_ERR_NULL_ARG = 1,    /* a required pointer is NULL, or z / norm_w not both set */
    GDN_ERR_BAD_SHAPE = 2,   /* negative sizes, H_v % H_k != 0, spec_stride < 1, max_T outside 1..8, ... */
    GDN_ERR_UNSUPPORTED = 3, /* K != 128, V != 128, unknown state dtype, bad split */
    GDN_ERR_MISALIGNED = 4,  /* a pointer or row stride breaks the alignment rules below */
    GDN_ERR_CUDA = 5         /* the launch failed (the CUDA error is left for the caller to query) */
} gdn_status;

/* Element type of the recurrent-state pool. */
typedef enum { GDN_F32 = 0, GDN_BF16 = 1, GDN_F16 = 2 } gdn_dtype;

/*
 * Bits the kernel ORs into *status_word (when given) for bad DEVICE data.
 * The offending sequence (or, for a bad write slot, just that slot write) is
 * skipped; nothing traps and nothing waits.
 */
#define GDN_FLAG_SLOT_RANGE 1  /* a read or write slot >= num_slots (read: sequence skipped; write: that write skipped) */
#define GDN_FLAG_ACCEPTED   2  /* num_accepted[i] > spec_stride: sequence skipped */
#define GDN_FLAG_QLEN       4  /* q_len > max_T or q_len > spec_stride: sequence skipped */
#define GDN_FLAG_TOKEN_ROW  8  /* a token row outside [0, num_tokens), or cu_seqlens[i] < 0 or
                                  cu_seqlens[i+1] > cu_seqlens[batch]: sequence skipped */
#define GDN_FLAG_TIMEOUT    16 /* gdn_prefill_chunked only: a wait on the tensor cores ran past its
                                  bound (gdn_set_wait_limit); that sequence's outputs and final
                                  state are incomplete */
#define GDN_FLAG_DRAIN      32 /* gdn_prefill_chunked only: after such a timeout, the wait (with the
                                  default bound) for the products still in flight ran out too; the
                                  CTA released its tensor memory regardless, since holding it would
                                  block every later kernel on that SM */

/*
 * dims->split flag: each warp of the decode step owns 8 of a unit's 128 V
 * columns instead of 16, so a unit runs on 16 warps with half the state per
 * lane and half the work per token.  Meant for small batches, where most SMs
 * would otherwise idle: the unit's warps spread over a 2- or 4-CTA cluster.
 * Same results up to FP32 rounding order.
 */
#define GDN_SPLIT_NARROW 0x100

/*
 * dims->split flag (GDN_SPLIT_HALFK | 1 or | 2): each warp keeps 16 V columns
 * but only half of their 128 K rows, the two warps of a column block adding
 * their partial products through shared memory once per token, so its
 * tensor stores keep the 16-column rows.  A unit's 16 warps run in one CTA
 * (| 1) or over a 2-CTA cluster (| 2, half of a unit's work per SM).  Meant
 * for small batches.  Same results up to FP32 rounding order.
 */
#define GDN_SPLIT_HALFK 0x200

/*
 * dims->flags: what the caller promises about the kernel launched on the
 * stream immediately before this call.  Each decode launch lets the next
 * launch on the stream start its CTAs while it finishes (programmatic
 * dependent launch); a CTA then waits for its predecessor to complete before
 * it touches memory that the predecessor may have written.  With these flags
 * it reads some inputs before that wait, which hides their latency behind the
 * predecessor's tail:
 *   GDN_PRE_INDEX   state_indices, num_accepted, cu_seqlens and
 *                   spec_token_indx were not written by the preceding kernel
 *                   (for example: they were filled at the start of the step);
 *   GDN_PRE_TOKENS  with GDN_PRE_INDEX: neither were q, k, v, a, b, z, A_log,
 *                   dt_bias and norm_w (for example: the batch's inputs are
 *                   resident and the preceding kernel is another decode step);
 *   GDN_PRE_STATE   with GDN_PRE_INDEX: nor were the state slots this call
 *                   reads (the rewound slots).  True in a model's forward
 *                   pass, where the kernel before a layer's step is never that
 *                   layer's own step; false for two steps of one layer in a
 *                   row where the second rewinds into the first's slots.
 * out, status_word and every slot write are accessed after the wait; without
 * GDN_PRE_STATE so is the state read, so back-to-back steps that rewind into
 * each other's slots stay ordered.  A
 * decode launch signals its successor only after its own wait, so when the
 * preceding kernel is one of this library's decode launches, or a kernel that
 * does not use programmatic dependent launch, every kernel before it has
 * completed when the early reads happen.
 * For gdn_spec_decode_conv, GDN_PRE_STATE also covers the conv slots the call
 * reads (its conv history), and the token prologue, which convolves that
 * history, runs early only with both GDN_PRE_TOKENS and GDN_PRE_STATE set.
 * The prefill entry points take no flags.
 */
#define GDN_PRE_INDEX  0x1
#define GDN_PRE_TOKENS 0x2
#define GDN_PRE_STATE  0x4

/* Opaque CUDA stream handle; the same type as cudaStream_t (NULL = legacy default stream). */
typedef struct CUstream_st* gdn_stream_t;

/* Sizes.  All host-side integers: the launch shape never depends on device data. */
typedef struct {
    int32_t batch;        /* number of speculative sequences (rows of state_indices) */
    int32_t num_tokens;   /* rows of q, k, v, a, b, z and out */
    int32_t H_k, H_v;     /* key heads and value heads; H_v % H_k == 0 (the tuned case is H_v = 8 H_k) */
    int32_t K, V;         /* head dims; both must be 128 */
    int32_t spec_stride;  /* columns of state_indices (>= every q_len) */
    int32_t max_T;        /* host-known bound on every q_len, 1..8 */
    int64_t num_slots;    /* slots in state_pool */
    /* Row strides between consecutive tokens, in ELEMENTS; 0 selects the dense
       default (q, k: H_k*K; v, z, out: H_v*V; a, b: H_v).  Within a row the
       heads are contiguous.  A packed mixed_qkv tensor [N, 2*H_k*K + H_v*V]
       is passed as three pointers into it with q_stride = k_stride =
       v_stride = 2*H_k*K + H_v*V. */
    int64_t q_stride, k_stride, v_stride, a_stride, b_stride, z_stride, out_stride;
    int32_t split;        /* CTAs per (sequence, v-head), one thread-block cluster:
                             0 = chosen from the batch size; else 1, 2, 4 or 8
                             (each warp owns 16 V columns), GDN_SPLIT_NARROW
                             | 2 or | 4 (each warp owns 8 V columns: 16 warps
                             per unit over 2 or 4 CTAs), or GDN_SPLIT_HALFK | 1
                             or | 2 (16 columns and half the K rows per warp:
                             16 warps per unit in 1 or 2 CTAs) */
    int32_t flags;        /* 0, or GDN_PRE_INDEX [| GDN_PRE_TOKENS] [| GDN_PRE_STATE] (above); 0 for prefill */
} gdn_dims;

/*
 * gdn_spec_decode -- one speculative decode step over a batch.
 *
 * Arguments (device pointers unless stated; element types fixed):
 *   q, k            bf16 [num_tokens, H_k, K]  (row stride q_stride / k_stride)
 *   v               bf16 [num_tokens, H_v, V]  (row stride v_stride)
 *   a, b            bf16 [num_tokens, H_v]     (row strides a_stride, b_stride)
 *   z               bf16 [num_tokens, H_v, V] output gate, or NULL
 *   A_log           fp32 [H_v]
 *   dt_bias         bf16 [H_v]
 *   norm_w          bf16 [V] gated-RMSNorm weight, or NULL.  z and norm_w are
 *                   both NULL or both set; with both NULL no epilogue runs
 *                   and out holds the raw readout o.
 *   state_pool      state_dtype [num_slots, H_v, K, V], V contiguous; read
 *                   and written in place
 *   state_indices   int32 [batch, spec_stride]; -1 marks a padded slot
 *   num_accepted    int32 [batch]; values < 1 read position 0
 *   cu_seqlens      int32 [batch + 1]; q_len_i = cu_seqlens[i+1] - cu_seqlens[i]
 *   spec_token_indx int32 [cu_seqlens[batch]] token row of every spec token,
 *                   or NULL when the spec tokens are rows cu_seqlens[i] + t
 *   out             bf16 [num_tokens, H_v, V] (row stride out_stride);
 *                   written only at the rows of active spec tokens, other
 *                   rows keep the caller's contents (zero-fill them first if
 *                   padded rows flow onward, as under CUDA graphs)
 *   dims            HOST pointer, read during the call only
 *   scale           query scale (128^-0.5 in the pages' default)
 *   eps             RMSNorm epsilon (1e-5 in the pages' default)
 *   state_dtype     GDN_F32, GDN_BF16 or GDN_F16
 *   status_word     device int32 that receives GDN_FLAG_* bits, or NULL
 *   stream          CUDA stream to launch on
 *
 * Skips: q_len <= 0, or a read slot < 0 (a padded sequence), write nothing
 * for that sequence.  A write slot < 0 skips only that write.
 *
 * Caller contract (not checked on the device): non-negative write slots are
 * distinct across the batch; no sequence reads a slot that another sequence
 * writes; token rows are used by at most one spec token.
 *
 * Alignment: state_pool 16 bytes; q, k, v, z, out, norm_w 8 bytes with
 * q/k/v/z/out row strides multiples of 4 elements; int32 tables 4 bytes.
 * Size limit: num_slots * H_v * K < 2^31 (the slot writes address the pool
 * as one 2-D tensor with 32-bit row coordinates); beyond it the call returns
 * GDN_ERR_UNSUPPORTED.  The call encodes that tensor's description on the
 * host the first time it sees a pool (cached per host thread for the last 4
 * pools); no device memory is allocated.
 */
GDNSPEC_API gdn_status gdn_spec_decode(
    const void* q, const void* k, const void* v,
    const void* a, const void* b, const void* z,
    const float* A_log, const void* dt_bias, const void* norm_w,
    void* state_pool,
    const int32_t* state_indices, const int32_t* num_accepted,
    const int32_t* cu_seqlens, const int32_t* spec_token_indx,
    void* out,
    const gdn_dims* dims, float scale, float eps, gdn_dtype state_dtype,
    int32_t* status_word, gdn_stream_t stream);

/*
 * gdn_prefill -- the same gated delta rule over whole prompts: the prefill
 * path whose state is carried across the prompt and written back to its slot
 * ("PR #52191 report -- [CPU] Support FP16/BF16 persisted GDN state on AMX",
 * implementation steps 3-4: arithmetic in FP32, the slot written in the pool
 * dtype, rounded once).
 *
 * Sequence i is token rows cu_seqlens[i] .. cu_seqlens[i+1]-1, in order (no
 * gather).  It starts from slot read_slots[i], or from the zero state when
 * read_slots[i] < 0; every token writes its output row (with the gated RMSNorm
 * epilogue when z / norm_w are given); the state after its last token goes to
 * slot write_slots[i] (no write when negative).  read_slots[i] ==
 * write_slots[i] updates a slot in place.
 *
 *   read_slots, write_slots   int32 [batch] (device)
 *   every other argument       as for gdn_spec_decode; dims->spec_stride,
 *                              max_T and split are not used
 *
 * Caller contract: non-negative write slots are distinct; no sequence reads a
 * slot that another sequence writes.  Bad device data skips the sequence:
 * a slot >= num_slots sets GDN_FLAG_SLOT_RANGE, rows outside [0, num_tokens)
 * set GDN_FLAG_TOKEN_ROW.  Asynchronous on `stream`, allocates nothing.
 */
GDNSPEC_API gdn_status gdn_prefill(
    const void* q, const void* k, const void* v,
    const void* a, const void* b, const void* z,
    const float* A_log, const void* dt_bias, const void* norm_w,
    void* state_pool,
    const int32_t* read_slots, const int32_t* write_slots,
    const int32_t* cu_seqlens,
    void* out,
    const gdn_dims* dims, float scale, float eps, gdn_dtype state_dtype,
    int32_t* status_word, gdn_stream_t stream);

/*
 * gdn_prefill_chunked -- what gdn_prefill computes, in the chunked form that
 * runs on the tensor cores: the prompt is cut into chunks of 64 tokens and the
 * per-token recurrence inside a chunk is unrolled into dense products
 * ("PR #52191 report", implementation steps 3-4: the inter-chunk recurrence
 * kernel with all products and the exp(g_last) rescale in FP32 buffers).
 * With G_t the running sum of the log-decays g inside the chunk, S the state
 * at its start and k^, q^ the normalised rows:
 *     (I + A) V' = B,  A_ts = beta_t e^(G_t - G_s) k^_t.k^_s (s < t),
 *                      B_t  = beta_t (v_t - e^(G_t) S^T k^_t)
 *     o_t = e^(G_t) S^T q^_t + sum_{s <= t} e^(G_t - G_s) (q^_t.k^_s) v'_s
 *     S  <- e^(G_last) S + sum_s e^(G_last - G_s) k^_s v'_s^T
 * which is the same quantity as the token recurrence, in exact arithmetic.
 * The products run on the tensor cores at FP32 accuracy: each operand is
 * carried as a bf16 hi part and a bf16 lo part (hi + lo within 2^-18 of the
 * FP32 value) and the hi.hi, lo.hi and hi.lo products accumulate in FP32; the
 * carried state, the triangular solve and the epilogue are FP32.  The state
 * is rounded to the pool dtype once, when it is stored at the end of the
 * prompt.
 *
 * Arguments, layouts, the caller contract and the status bits are those of
 * gdn_prefill; in addition GDN_FLAG_TIMEOUT reports a tensor-core wait that
 * ran past its bound.  One CTA per (sequence, v-head) unit, holding the
 * whole 512-column tensor memory of its SM (~218 KiB of shared memory); with
 * fewer units than half the device's SMs, two CTAs per unit as a cluster,
 * each with 64 of the value columns (~210 KiB of shared memory each).  The
 * results do not depend on which form runs beyond FP32 rounding order.
 * Asynchronous on `stream`, allocates nothing.
 */
GDNSPEC_API gdn_status gdn_prefill_chunked(
    const void* q, const void* k, const void* v,
    const void* a, const void* b, const void* z,
    const float* A_log, const void* dt_bias, const void* norm_w,
    void* state_pool,
    const int32_t* read_slots, const int32_t* write_slots,
    const int32_t* cu_seqlens,
    void* out,
    const gdn_dims* dims, float scale, float eps, gdn_dtype state_dtype,
    int32_t* status_word, gdn_stream_t stream);

/* Sizes of the short causal convolution in front of the step (gdn_spec_decode_conv). */
typedef struct {
    int32_t width;          /* taps W, 1..4 */
    int32_t state_len;      /* rows per conv slot; >= W - 1 + spec_stride */
    int64_t num_conv_slots; /* slots in conv_pool */
    int64_t x_stride;       /* elements between rows of x; 0 = conv_dim (dense); multiple of 4 */
    int32_t reserved[2];    /* must be 0 */
} gdn_conv_dims;

/*
 * gdn_spec_decode_conv -- gdn_spec_decode with the depthwise causal
 * convolution that produces q, k and v fused in front of it ("PR #46090
 * report", implementation step 2: the speculative conv state is a wide
 * rolling buffer sliced per token, convolved and written back; "PR #51674
 * report", implementation step 3: the speculative path runs
 * causal_conv1d_update with rewind before the post-conv decode kernel).
 *
 * Instead of q, k, v the call takes the projection rows x
 * [num_tokens, conv_dim] (bf16, conv_dim = 2 H_k K + H_v V, channels in the
 * order q | k | v; row r of token t is gathered like every other input).  For
 * a processed sequence i (one that gdn_spec_decode would not skip), with
 * a = max(num_accepted[i], 1):
 *   history   the W-1 rows a .. a+W-2 of conv slot conv_in[i] (zeros when
 *             conv_in[i] < 0): the inputs up to the previous step's last
 *             accepted token;
 *   conv      y_t[c] = silu(bias[c] + sum_{w<W} weight[c][w] x_{t-W+1+w}[c])
 *             over (history, this step's rows) in time order, in FP32; y
 *             feeds the step as q | k | v (never rounded to bf16);
 *   new slot  conv slot conv_out[i] (skipped when < 0): rows 0 .. W-2 = the
 *             history, rows W-1 .. W-2+q_len = this step's rows, bit for bit;
 *             later rows are left as they were.
 * After a prefill the caller seeds a slot with the prompt's last W inputs in
 * rows 0 .. W-1 and passes num_accepted = 1.
 *
 *   x             bf16 [num_tokens, conv_dim], row stride cdims->x_stride
 *   conv_weight   bf16 [conv_dim, W]
 *   conv_bias     bf16 [conv_dim], or NULL (no bias)
 *   conv_pool     bf16 [num_conv_slots, state_len, conv_dim], caller-owned
 *   conv_in, conv_out  int32 [batch] (device)
 *   every other argument as for gdn_spec_decode; dims->q_stride, k_stride and
 *   v_stride are not used, dims->split must be 0 or 1.
 *
 * Caller contract (in addition to gdn_spec_decode's): no conv_out[j] >= 0
 * equals any conv_in[i] of the call (a slot is never read and written by one
 * step: the CTAs of a sequence share its q / k channels), and the
 * non-negative conv_out are distinct.  A conv slot >= num_conv_slots sets
 * GDN_FLAG_SLOT_RANGE and skips the sequence.  Host errors: width outside
 * 1..4, state_len too small or non-zero reserved -> GDN_ERR_BAD_SHAPE; x /
 * conv_pool / conv_bias not 8-byte aligned, conv_weight not 16-byte aligned
 * when W = 4, or x_stride not a multiple of 4 -> GDN_ERR_MISALIGNED.  Asynchronous on `stream`, allocates nothing.
 */
GDNSPEC_API gdn_status gdn_spec_decode_conv(
    const void* x, const void* conv_weight, const void* conv_bias, void* conv_pool,
    const int32_t* conv_in, const int32_t* conv_out, const gdn_conv_dims* cdims,
    const void* a, const void* b, const void* z,
    const float* A_log, const void* dt_bias, const void* norm_w,
    void* state_pool,
    const int32_t* state_indices, const int32_t* num_accepted,
    const int32_t* cu_seqlens, const int32_t* spec_token_indx,
    void* out,
    const gdn_dims* dims, float scale, float eps, gdn_dtype state_dtype,
    int32_t* status_word, gdn_stream_t stream);

/*
 * The split code that gdn_spec_decode would use for these sizes and state
 * dtype (dims->split itself when it is not 0; else, for an FP32 state,
 * GDN_SPLIT_HALFK | 2 with batch * H_v <= 64 and GDN_SPLIT_HALFK | 1 with
 * batch * H_v <= 128; else 1), or 0 for invalid dims or dtype.
 * Host only; reads no device state.
 */
GDNSPEC_API int32_t gdn_spec_decode_split(const gdn_dims* dims, gdn_dtype state_dtype);

/*
 * Bound on each wait of gdn_prefill_chunked for its tensor-core products:
 * 0 (the default) waits with blocking polls of the completion barrier, 2^24
 * of them (well over a second); a non-zero bound counts non-blocking polls
 * instead, so that a small one runs out for certain.  A wait that runs out
 * sets GDN_FLAG_TIMEOUT; the unit writes no final state and its CTAs end
 * after waiting, with the default bound, for the products still in flight
 * (a 2-CTA unit first runs its remaining chunks, whose outputs are invalid).  Process-wide, read at every
 * launch; meant for exercising that path in tests.  No counterpart on the
 * report pages.
 */
GDNSPEC_API void gdn_set_wait_limit(uint32_t polls);

/* Static English text for a status code (never NULL). */
GDNSPEC_API const char* gdn_status_str(gdn_status status);

/* GDNSPEC_VERSION of the loaded library. */
GDNSPEC_API int32_t gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDNSPEC_H */
