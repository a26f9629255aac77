/*
 * sa.h -- C ABI of the GB300 (sm_103a) SageAttention3-style attention library.
 *
 * What it computes (source pages, by title and section):
 *  - "FlashAttention kernels", sections 0-1: exact softmax attention computed
 *    tile by tile with online softmax, never materialising the L x L scores.
 *  - "GPU kernel porting with AI agents", section "Sage Attention 3": Q, K, V
 *    in NVFP4 (e2m1 values, 1x16 groups, FP8 e4m3 scales); P quantised in two
 *    levels (per-row rescale to [0, 448 x 6], then FP4 microscaling).
 *  - "kernel overview", SageAttention technique chain: smooth-K (subtract the
 *    per-channel mean of K over tokens before quantising K).
 *  - "cuda kernel pretrain", section 3: GQA -- query head h uses KV head
 *    h / (H / Hkv).
 *
 * Conventions for every entry point:
 *  - Tensors are device pointers, row-major, BHLD: Q and O are [B, H, L, d],
 *    K and V are [B, Hkv, L, d], all bfloat16 (or BLHD, [B, L, heads, d],
 *    with the SA_LAYOUT_BLHD flag where an entry point takes it).  The softmax scale is
 *    1/sqrt(d); causal means key j is visible to query i iff j <= i.
 *  - Ownership: the caller allocates and owns every buffer.  The library
 *    allocates no device memory and keeps no state between calls other than
 *    a device error word (see sa_last_device_error) and, once
 *    sa_attn_fwd_host has been called, its copy streams and events.
 *  - Asynchrony: work is enqueued on `stream` (NULL = legacy default stream)
 *    and the call returns before it finishes.
 *  - Sizes: any L >= 1 (a ragged last 128-token tile is masked: keys past L
 *    get no weight, rows past L are not written); d in {64, 128}; H a
 *    multiple of Hkv.  An empty problem (B == 0 or L == 0) is valid: the call
 *    returns SA_OK without enqueueing anything or reading any pointer.
 *  - Errors: arguments are validated before anything is enqueued; on any
 *    argument error nothing is launched.  SA_ERR_INVALID_ARG: null or
 *    misaligned pointer (all pointers must be 16-byte aligned), negative B or
 *    L, H or Hkv < 1, H % Hkv != 0.  SA_ERR_UNSUPPORTED: d not in {64, 128},
 *    or B * H * Lp >= 2^31 (Lp = L rounded up to 128).  SA_ERR_CUDA: a launch
 *    or driver call failed (the CUDA error is not cleared).
 *  - Inputs are assumed finite; NaN/Inf inputs give unspecified results.
 */
#ifndef SA_H_
#define SA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sa_stream_t;   /* same handle as cudaStream_t */

typedef enum {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = 1,
  SA_ERR_UNSUPPORTED = 2,
  SA_ERR_CUDA = 3,
  SA_ERR_TIMEOUT = 4
} sa_status;

/* SA_MODE_NVFP4_SQ: the NVFP4 path with SageAttention2's smooth-Q added (a
 * labelled variant; see sa_quantize_smooth_q).  SA_MODE_NVFP4_FQ: the NVFP4
 * path with Q quantised inside the attention kernel (see sa_quantize_kv_s). */
typedef enum { SA_MODE_BF16 = 0, SA_MODE_NVFP4 = 1, SA_MODE_NVFP4_SQ = 2, SA_MODE_NVFP4_FQ = 3 } sa_mode;

/* Output-format flag OR-ed into the `mode` argument of sa_attn_fwd: with it,
 * o is float32 [B, H, L, d] (the FP32 accumulator divided by the row sum,
 * without the final bf16 rounding); without it o is bfloat16. */
#define SA_OUT_FP32 16

/* Layout flag, OR-ed into `mode` (sa_attn_fwd, sa_attn_fwd_ws) or `flags`
 * (sa_quantize_ex): the bf16 tensors q, k, v (and o, bf16 or float32) are
 * [B, L, heads, d] ("BLHD", d contiguous) instead of [B, heads, L, d].  The
 * quantised operands keep the one layout documented below whatever the
 * inputs' layout, and the results are bit-identical to the BHLD calls on the
 * same values.  Not accepted by sa_attn_fwd_host and
 * sa_quantize_static_scratch. */
#define SA_LAYOUT_BLHD 32

/* Scheduling flag of sa_attn_fwd_host, OR-ed into `mode`: the host inputs q,
 * k, v already hold their final values when the call is made (no work
 * enqueued on `stream` before the call writes them), so the call's
 * host -> device copies may start before that work completes; each waits only
 * until the previous sa_attn_fwd_host call on this device has finished
 * computing on the workspace slot it refills (and its compute until that
 * call's copy-out from the slot is done).  This applies when the previous
 * call used the same workspace pointer and sizes that give the same slots;
 * otherwise the call waits for the work before it, as without the flag.
 * The call's compute (on `stream`) also waits until the previous call's last
 * compute has finished, whichever stream that call used: the split-KV region
 * of the workspace is shared by all slots, so no chunk of this call may use
 * it while a chunk of the previous call still does.
 * Back-to-back calls on one workspace then overlap one call's first copy-ins
 * with the previous call's last compute and copy-out.  Results are
 * unchanged.  Accepted by
 * sa_attn_fwd_host (and its workspace-size query) only. */
#define SA_HOST_OVERLAP 64

/*
 * Quantised operands produced by sa_quantize (device pointers, caller-owned).
 * Every layout holds Lp = L rounded up to a multiple of 128 tokens per head;
 * tokens past L have zero codes and zero scales, and a V group that straddles
 * L is quantised with zeros for its missing tokens.
 *
 * Codes: two e2m1 nibbles per byte, element 2i in the low nibble.
 *   q_codes [B, H, Lp, d/2]    Q, groups of 16 along d
 *   k_codes [B, Hkv, Lp, d/2]  K' = K - mean_tokens(K), groups along d
 *   v_codes [B, Hkv, d, Lp/2]  V transposed (channel rows), groups of 16
 *                              consecutive tokens
 * Scale factors (e4m3 bytes) in 512-byte blocks of 128 rows x 4 groups; the
 * byte at m0*16 + j*4 + k of a block is the scale of row 32*j + m0, group k:
 *   q_sf [B, H, Lp/128, d/64, 512]   rows = tokens, groups = d/16 along d
 *   k_sf [B, Hkv, Lp/128, d/64, 512]
 *   v_sf [B, Hkv, Lp/64, 512]        rows = channels (rows >= d are 0),
 *                                    groups = 16-token groups of a 64-token chunk
 * k_mean [B, Hkv, d] float32: the smooth-K mean, computed as the float32 sum
 *   over 128-token chunks (token order inside a chunk, then chunk order; the
 *   last chunk holds the L % 128 remaining tokens) divided by L.
 * workspace: scratch for sa_quantize (float32 [B, Hkv, Lp/128, d] partial sums).
 * This is the layout the tcgen05 block-scaled MMA consumes (scale blocks are
 * copied to tensor memory unchanged).
 */
typedef struct {
  void* q_codes;
  void* q_sf;
  void* k_codes;
  void* k_sf;
  void* v_codes;
  void* v_sf;
  float* k_mean;
  void* workspace;
} sa_fp4_qkv;

/*
 * Sizes of a problem whose query length differs from its key length: Q (and
 * O) [B, H, Lq, d], K and V [B, Hkv, Lkv, d] -- a chunk of queries against a
 * longer key/value sequence (chunked prefill, decode).  Under the causal mask
 * the queries are the last Lq positions of the sequence: key j is visible to
 * query i iff j <= i + Lkv - Lq (causal calls need Lkv >= Lq).  The `_s`
 * entry points take this struct; the others are the special case Lq = Lkv =
 * L.  With Lq != Lkv the quantised layouts below have Lq rows for Q and Lkv
 * rows (or token columns) for K and V, each rounded up to 128.
 * Decode with grouped heads: a one-token query (Lq = 1) sees every key, so
 * the G = H / Hkv query heads of a kv head differ only in their query
 * vectors; in BHLD, Q [B, H, 1, d] is the same memory as [B, Hkv, G, d], and
 * calling with {B, Hkv, Hkv, G, Lkv, d}, non-causal, gives the same O with G
 * query rows per 128-row tile instead of one (G times fewer tiles).
 */
typedef struct {
  int B, H, Hkv;   /* batch, query heads, key/value heads (H % Hkv == 0) */
  int Lq, Lkv;     /* query tokens, key/value tokens */
  int d;           /* head dimension, 64 or 128 */
} sa_shape;

/*
 * Bytes of one device blob holding every sa_fp4_qkv buffer, each at a
 * 256-byte aligned offset.  offsets_out (may be NULL) receives 8 offsets in
 * struct order (q_codes, q_sf, k_codes, k_sf, v_codes, v_sf, k_mean,
 * workspace).  Returns 0 for unsupported sizes and for an empty problem
 * (which needs no blob).
 */
size_t sa_fp4_qkv_bytes(int B, int H, int Hkv, int L, int d, size_t offsets_out[8]);

/* Fill `out` with pointers into `blob` (device memory of sa_fp4_qkv_bytes). */
sa_status sa_fp4_qkv_from_blob(void* blob, int B, int H, int Hkv, int L, int d,
                               sa_fp4_qkv* out);
/* The same two for an sa_shape (0 / an error for empty or invalid sizes). */
size_t sa_fp4_qkv_bytes_s(const sa_shape* shape, size_t offsets_out[8]);
sa_status sa_fp4_qkv_from_blob_s(void* blob, const sa_shape* shape, sa_fp4_qkv* out);

/*
 * sa_quantize -- smooth-K mean, then NVFP4 quantisation of Q, K' and V
 * ("Sage Attention 3" section of "GPU kernel porting with AI agents";
 * smooth-K from "kernel overview").  For every 1x16 group x (float32):
 *   s8 = e4m3_rne_satfinite(max|x| / 6)      (IEEE float32 division)
 *   code_i = e2m1_rne_satfinite(x_i / decode(s8)); all codes +0 if s8 == 0
 * with K' = float32(k) - k_mean[c].  Results are bit-exact functions of the
 * inputs.  q, k, v: bf16 BHLD device tensors; out: buffers as documented
 * above (all eight pointers required).  Enqueues 2 kernels on `stream`, the
 * second a programmatic dependent launch of the first (it starts while the
 * first drains and waits for it before it reads the K means); the second
 * also lets a programmatic dependent launch behind it (sa_attn_fwd's) start
 * early.  Ordering on `stream` is unchanged: work enqueued after the call
 * that is not itself such a launch starts after both kernels complete, and
 * such a launch reads nothing before they have.
 */
sa_status sa_quantize(const void* q, const void* k, const void* v,
                      int B, int H, int Hkv, int L, int d,
                      const sa_fp4_qkv* out, sa_stream_t stream);

/* sa_quantize_ex -- sa_quantize with `flags`: 0 or SA_LAYOUT_BLHD (q, k, v
 * given as [B, L, heads, d]); the outputs are the same bytes as sa_quantize
 * on the BHLD tensors with the same values. */
sa_status sa_quantize_ex(const void* q, const void* k, const void* v,
                         int B, int H, int Hkv, int L, int d, int flags,
                         const sa_fp4_qkv* out, sa_stream_t stream);
/* sa_quantize_ex for an sa_shape: Q with Lq tokens, K and V with Lkv (the
 * smooth-K mean runs over the Lkv key tokens).  Lq == 0 with Lkv > 0 is
 * SA_ERR_INVALID_ARG. */
sa_status sa_quantize_s(const void* q, const void* k, const void* v, const sa_shape* shape,
                        int flags, const sa_fp4_qkv* out, sa_stream_t stream);

/*
 * sa_quantize_static_scratch -- sa_quantize for callers that cannot allocate
 * device memory.  (The pages describe no such call; it is part of this
 * library's interface only.)
 *
 * sa_quantize needs a scratch buffer for the K-mean partial sums, which the
 * caller normally provides inside the sa_fp4_qkv blob.  Some callers have no
 * way to obtain one: host code embedded in a runtime that plans all device
 * memory ahead of time and forbids cudaMalloc once it is running, plugin or
 * custom-operator interfaces that hand over only the input and output
 * buffers, and code that must not risk the implicit device synchronisation an
 * allocation can cause.  This entry point does the same work, bit for bit,
 * with the partial sums kept in a fixed array compiled into the library
 * (SA_STATIC_SCRATCH_FLOATS floats = 4 MiB, held by every GPU that loads the
 * library until the process exits).  It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *  - Arguments as for sa_quantize; out->workspace is ignored and may be NULL.
 *  - Sizes with B * Hkv * (Lp/128) * d > SA_STATIC_SCRATCH_FLOATS return
 *    SA_ERR_UNSUPPORTED before anything is launched.
 *  - The first call on each device, made with that device current, looks up
 *    the array's device address (cudaGetSymbolAddress); make that first call
 *    before any stream capture.
 *  - Every call on a device uses the same array.  Each call writes every
 *    partial sum it reads before reading it, so leftovers from an earlier
 *    call never reach the outputs and nothing needs clearing; but calls whose
 *    kernels overlap on the GPU (other streams, other host threads) race on
 *    the array and must be serialised by the caller.
 */
#define SA_STATIC_SCRATCH_FLOATS 1048576
sa_status sa_quantize_static_scratch(const void* q, const void* k, const void* v,
                                     int B, int H, int Hkv, int L, int d,
                                     const sa_fp4_qkv* out, sa_stream_t stream);

/*
 * Q quantised inside the attention kernel ("GPU kernel porting with AI
 * agents", section "Sage Attention 3": the same 1x16 NVFP4 quantisation of
 * Q, fused into the attention's load stage instead of a separate pass).
 * sa_quantize_kv_s: sa_quantize_s for K and V only -- smooth-K mean, K' and V
 *   codes and scales, bit-identical to sa_quantize_s's; out->q_codes and
 *   out->q_sf are neither read nor written (may be NULL).  Arguments and
 *   errors as sa_quantize_s without q.  Two kernels on `stream`.
 * sa_attn_fwd(_ws, _s) with mode SA_MODE_NVFP4_FQ: q is the bf16 Q device
 *   tensor (BHLD, or BLHD with SA_LAYOUT_BLHD; 16-byte aligned, else
 *   SA_ERR_INVALID_ARG), k points to a host `const sa_fp4_qkv*` from
 *   sa_quantize_kv_s for the same sizes, v must be NULL.  The attention
 *   kernel copies each unit's bf16 Q tiles by TMA into shared memory and its
 *   softmax threads quantise their own rows with sa_quantize's arithmetic,
 *   so O is bit-identical to sa_quantize + SA_MODE_NVFP4 on the same work
 *   split (the few-row decode kernel is not used: such shapes run on the
 *   prefill kernel).  sa_attn_fwd_host does not take it (SA_ERR_UNSUPPORTED).
 */
sa_status sa_quantize_kv_s(const void* k, const void* v, const sa_shape* shape, int flags, const sa_fp4_qkv* out,
                           sa_stream_t stream);

/*
 * Smooth-Q variant ("kernel overview", SageAttention evolution chain: "Smooth-K
 * -> Smooth-Q+K"; the SageAttention2 step, kept beside the SA3 path as a
 * labelled variant).  Q is quantised as Q' = Q - qbar_i, qbar_i the mean of
 * its 128-token block i (the attention kernel's query tile of one head:
 * float32 sum of the block's valid rows, row by row from 0, divided by their
 * count; Q' = RN(q - qbar_i), then 1x16 NVFP4 as sa_quantize does), and the
 * attention kernel adds the block mean's share of the scores back:
 *   S = Q^' K^'^T + dS,  dS[i, j] = qbar_i . K^'_j  (= (Q^' + qbar_i) K^'^T)
 * with K^' the dequantised smoothed keys.  dS is float32: per 1x16 group an
 * FMA chain over its channels, then the group sums times the group scales in
 * group order; the rest is the NVFP4 path unchanged.
 *
 * sa_fp4_sq: the sa_fp4_qkv buffers plus q_mean [B, H, Lqp/128, d] and ds
 *   [B, H, Lqp/128, Lkvp] (float32; Lqp, Lkvp the lengths rounded up to 128).
 * sa_smooth_q_bytes_s: device bytes of one blob holding q_mean and ds at
 *   256-byte aligned offsets (offsets_out, may be NULL, receives 2); 0 for
 *   invalid or empty sizes.  sa_smooth_q_from_blob_s sets out->q_mean and
 *   out->ds into such a blob (out->fp4 is left as it is).
 * sa_quantize_smooth_q: run after sa_quantize(_s) of the same q, k, v into
 *   x->fp4 (it reads the K codes and scales): overwrites x->fp4.q_codes and
 *   q_sf with those of Q', writes q_mean and ds.  flags: 0 or SA_LAYOUT_BLHD
 *   (the layout of q).  Two kernels on `stream` (plain launches); bit-exact
 *   codes, scales and means.
 * sa_attn_fwd(_ws, _s) with mode SA_MODE_NVFP4_SQ: q points to a host
 *   `const sa_fp4_sq*`; otherwise as SA_MODE_NVFP4 (the few-row decode kernel
 *   is not used: such shapes run on the prefill kernel).  sa_attn_fwd_host
 *   does not take it (SA_ERR_UNSUPPORTED).
 */
typedef struct {
  sa_fp4_qkv fp4;
  float* q_mean;
  float* ds;
} sa_fp4_sq;
size_t sa_smooth_q_bytes_s(const sa_shape* shape, size_t offsets_out[2]);
sa_status sa_smooth_q_from_blob_s(void* blob, const sa_shape* shape, sa_fp4_sq* out);
sa_status sa_quantize_smooth_q(const void* q, const sa_shape* shape, int flags, const sa_fp4_sq* x,
                               sa_stream_t stream);

/*
 * sa_attn_fwd -- fused attention forward, O = softmax(Q K^T / sqrt(d)) V,
 * tile by tile with online softmax ("FlashAttention kernels" sections 0-1).
 *  mode SA_MODE_BF16:  q, k, v are bf16 BHLD device tensors; tcgen05 BF16
 *    MMAs with FP32 accumulation; P rounded to bf16 for the P.V product.
 *  mode SA_MODE_NVFP4: q points to a host `const sa_fp4_qkv*` produced by
 *    sa_quantize for the same sizes; k and v must be NULL.  QK^T and P.V are
 *    tcgen05 block-scaled FP4 MMAs (FP32 accumulation); P is quantised in
 *    two levels in the kernel ("Sage Attention 3"): per row and 128-key
 *    tile, P2 = p~ * 2688 / rowmax_tile(p~), then 1x16 e2m1 groups along the
 *    keys with e4m3 scales; the tile's P.V is weighted by rowmax/2688.
 *  o: bf16 [B, H, L, d] device output (float32 if mode has SA_OUT_FP32).
 *  causal: 0 or 1 (top-left aligned).
 *  Heads map as GQA: head h reads KV head h / (H / Hkv).
 */
sa_status sa_attn_fwd(const void* q, const void* k, const void* v, void* o,
                      int B, int H, int Hkv, int L, int d, int causal,
                      int mode, sa_stream_t stream);

/*
 * Split-KV ("FlashAttention kernels": the online-softmax rescaling that merges
 * tiles also merges independent shares of the key range).  When the (batch,
 * head, pair of query tiles) units alone cannot fill the GPU, each unit's key
 * tiles are cut into nsplit contiguous shares computed by separate CTAs, and
 * a combine kernel merges the shares' partial results (unnormalised O, row
 * maximum, row sum) into O.  Shares are whole 128-key tiles, so the P
 * quantisation is unchanged and only the float32 summation order differs
 * from the unsplit call.
 *
 * Stream-K (NVFP4 path): persistent CTAs, one per SM, each over an equal
 * range of (query-tile pair, key tile) items; a pair cut by a range
 * boundary is computed in segments and merged the same way.
 *
 * Decode (NVFP4 path, at most 16 query rows per kv head: (H / Hkv) * Lq <=
 * 16): a kernel laid out for few rows ("FlashAttention kernels" section 3,
 * Flash-Decoding) takes the query rows of the G heads of a kv head together.
 * Split-KV there cuts each (batch, kv head) pair's key range into shares;
 * stream-K (-1) means equal ranges of all (pair, key tile) items, the pairs
 * that ranges cut merged by a combine kernel.  The library's choice (0) is
 * as many shares as let the pairs fill one wave of resident CTAs.
 *
 * sa_attn_fwd_workspace_bytes: device workspace bytes sa_attn_fwd_ws needs
 *   for the given sizes and `nsplit`: 0 = the library's choice (NVFP4,
 *   non-causal: stream-K once the pairs fill the SMs; split-KV while the units leave at
 *   least half of the SMs idle and every share keeps 16 key tiles or more, at
 *   most 16 shares; else neither; decode shapes: shares as above); 1 = one
 *   unit per CTA; n > 1 = n shares, at most one per key tile; -1 = stream-K
 *   (NVFP4 only).  0 when neither would be used, or for invalid or empty
 *   sizes.
 * sa_attn_fwd_ws: sa_attn_fwd with split-KV or stream-K.  Arguments as
 *   sa_attn_fwd, plus nsplit as above and a caller-owned, 16-byte aligned
 *   device workspace of workspace_bytes.  With nsplit 0 a missing or short
 *   workspace means one unit per CTA; with nsplit > 1 or -1 it is
 *   SA_ERR_INVALID_ARG; -1 with the BF16 path is SA_ERR_UNSUPPORTED.
 *   Enqueues the attention kernel and, when work is split, the combine
 *   kernel, on `stream`; both are programmatic dependent launches (each may
 *   start its set-up while the kernel before it finishes and reads its
 *   inputs only after that kernel has completed), so stream order holds.
 */
size_t sa_attn_fwd_workspace_bytes(int B, int H, int Hkv, int L, int d, int causal, int mode, int nsplit);
sa_status sa_attn_fwd_ws(const void* q, const void* k, const void* v, void* o,
                         int B, int H, int Hkv, int L, int d, int causal, int mode, int nsplit,
                         void* workspace, size_t workspace_bytes, sa_stream_t stream);
/* The same two for an sa_shape (o is [B, H, Lq, d]; split shares and stream-K
 * items run over the Lkv key tiles; a causal call with Lkv < Lq is
 * SA_ERR_INVALID_ARG, and so is Lkv == 0 with Lq > 0). */
size_t sa_attn_fwd_workspace_bytes_s(const sa_shape* shape, int causal, int mode, int nsplit);
sa_status sa_attn_fwd_s(const void* q, const void* k, const void* v, void* o, const sa_shape* shape,
                        int causal, int mode, int nsplit, void* workspace, size_t workspace_bytes,
                        sa_stream_t stream);

/*
 * sa_attn_fwd_host -- the path of sa_attn_fwd (mode SA_MODE_NVFP4:
 * sa_quantize then the FP4 attention; SA_MODE_BF16: the BF16 attention) on
 * bf16 BHLD Q, K, V in pinned HOST memory, writing O to pinned host memory.
 * (A library entry point for callers whose tensors live on the host; the
 * pages describe the computation only.)
 *  q, k, v, o: host pointers inside page-locked allocations (cudaHostAlloc or
 *    cudaHostRegister; anything else is SA_ERR_INVALID_ARG), laid out as for
 *    sa_attn_fwd; o is bf16, or float32 with SA_OUT_FP32 in `mode`.
 *  workspace: device buffer of at least
 *    sa_attn_fwd_host_workspace_bytes(B, H, Hkv, L, d, mode, chunk_pairs)
 *    bytes, 256-byte aligned; must not be used by anything else until the
 *    call's work on `stream` has completed.
 *  chunk_pairs: (batch, kv head) pairs per chunk, the last chunk ragged;
 *    0 = the library's chunking: chunks of n pairs (the most whose attention
 *    CTAs fit in one wave on the SMs, and at least two chunks); for
 *    SA_MODE_NVFP4 the last ones shrink by halves (..., n, 8, 4, 2 pairs)
 *    and a chunk whose CTAs would leave half of the SMs idle runs with
 *    split-KV (shares of 8 key tiles or more).
 * The problem is cut into chunks of consecutive (batch, kv head) pairs with
 * all their query heads.  Each chunk's inputs are copied host -> device on a
 * copy stream, computed on `stream` (the same kernels as the device-buffer
 * calls) and its O copied back on a second copy stream; three workspace
 * slots rotate between chunks, so the copies of one chunk overlap the compute
 * of its neighbours, and the shrinking last chunks shorten the part of the
 * call that no copy-in overlaps.  The results are bit-identical to
 * sa_quantize + sa_attn_fwd on device buffers, except that a split NVFP4
 * chunk (chunk_pairs 0) differs from them in float32 summation order (its P
 * is quantised per key tile, so split-KV changes nothing else).  The copies start after the work already enqueued on
 * `stream`, and `stream` reaches the end of the call's work only after O is
 * in host memory (synchronise on `stream` before reading o).  The two copy
 * streams and thirteen events are created on the first call on each device
 * and kept until the process exits; calls on one device must not be made
 * concurrently from several host threads.  Errors as for sa_attn_fwd; a
 * failure after the first copy was enqueued leaves o partly written, and
 * `stream` still waits for every copy the call enqueued (after synchronising
 * it, no copy of the failed call touches q, k, v, o or the workspace).
 */
size_t sa_attn_fwd_host_workspace_bytes(int B, int H, int Hkv, int L, int d, int mode, int chunk_pairs);
sa_status sa_attn_fwd_host(const void* q, const void* k, const void* v, void* o,
                           int B, int H, int Hkv, int L, int d, int causal, int mode,
                           void* workspace, size_t workspace_bytes, int chunk_pairs,
                           sa_stream_t stream);

/* Static string for a status code. */
const char* sa_status_string(sa_status s);

/*
 * Reads and clears the device error word on the current device
 * (synchronises the device).  Kernels bound every wait on a barrier; a wait
 * that gives up records SA_ERR_TIMEOUT here and the kernel returns early, so
 * its output is then invalid.  Returns SA_OK if no kernel recorded an error,
 * SA_ERR_CUDA if the word could not be read.
 */
sa_status sa_last_device_error(void);

/*
 * Self-test of the bounded-wait path used by every kernel: launches one CTA
 * that waits, with the given limit (nanoseconds, 1..10^10), on a
 * shared-memory barrier that nothing completes.  The wait gives up, records
 * SA_ERR_TIMEOUT in the device error word and the kernel returns normally,
 * leaving the context usable.  Read the result with sa_last_device_error().
 */
sa_status sa_selftest_wait_timeout(uint64_t limit_ns, sa_stream_t stream);

/*
 * Self-test of the score step of the NVFP4 attention kernel (test support; the
 * pages describe no such call): S = Q^ K^'^T for query tile qt (rows
 * 128*qt .. 128*qt + 127, padded) of head (b, h) and key tile kt (keys
 * 128*kt .. 128*kt + 127) of its kv head h / (H / Hkv), computed with the
 * kernel's own block-scaled FP4 MMAs ("GPU kernel porting with AI agents",
 * section "Sage Attention 3": Q and K' in 1x16 NVFP4 groups) and written as
 * float32 [128][128] (row = query, column = key, unscaled: no 1/sqrt(d)) to
 * the device buffer s_out.  x: operands from sa_quantize for `shape`
 * (Lq and Lkv as there).  Lets a test measure how far the tensor core's
 * float32 scores lie from the exact products of the dequantised operands.
 * SA_ERR_INVALID_ARG for indices outside the padded tiles, null or
 * misaligned pointers, or an empty problem.  Asynchronous on `stream`.
 */
sa_status sa_selftest_nvfp4_score_tile(const sa_fp4_qkv* x, const sa_shape* shape, int b, int h, int qt, int kt,
                                       float* s_out, sa_stream_t stream);

/*
 * Self-test of the exponent path of the attention kernels' softmax (test
 * support; the pages describe no such call): ex2_out[i] = 2^x[i] and
 * lg2_out[i] = log2(y[i]) computed with the same approximate hardware
 * instructions the softmax uses for P and for the e4m3 group-scale fold, so
 * that a test can measure their error.  x, y, ex2_out, lg2_out: device
 * buffers of n floats.  Asynchronous on `stream`.
 */
sa_status sa_selftest_exp_path(const float* x, const float* y, int n, float* ex2_out, float* lg2_out,
                                sa_stream_t stream);

/* Library version string. */
const char* sa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SA_H_ */
