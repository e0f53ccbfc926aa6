/*
 * kv_attn.h — C ABI of the GB300 KV-cache GQA attention step.
 *
 * Four compute entry points, one per step of the decoder's attention hot path:
 *   kv_cache_append_rope_qknorm  QK-Norm + RoPE fused into the K/V cache write
 *   kv_attn_prefill              parallel prefill attention over the cache
 *   kv_attn_decode               single-token split-KV decode attention
 *   lmhead_argmax                tied lm_head GEMV + greedy argmax
 * and the ones that extend them:
 *   kv_attn_decode_step          the new token's append and its decode in one launch
 *   kv_attn_decode_static        kv_attn_decode without a caller workspace (allocates nothing)
 *   kv_attn_verify, kv_verify_commit   speculative-decoding verify block and its commit
 *   lmhead_topk                  final RMSNorm + lm_head + the k best ids
 * plus workspace sizers (kva_workspace_size and the per-call ones), error strings, the
 * version, and the counter of in-kernel waits that gave up (kva_wait_timeouts).
 *
 * Conventions shared by every call
 *  - Ownership: every buffer belongs to the caller.  The library never allocates or
 *    frees memory; pointers are borrowed for the duration of the stream work the call
 *    enqueues (inputs are referenced, not copied: HunyuanOCR v1.0 ncnn port, section
 *    five item 10).  Device pointers must stay valid until that work completes.
 *  - Streams: every call is asynchronous on the caller's stream `stream` (a
 *    cudaStream_t; NULL = legacy default stream).
 *  - Errors: arguments are validated on the host before anything is launched; a
 *    call that returns a status other than KVA_OK has enqueued nothing, so the cache
 *    keeps its committed contents (the cache is only replaced after success:
 *    HunyuanOCR v1.5 ncnn port, section 3.7).  Context overflow is rejected, never
 *    wrapped (Youtu-VL-4B ncnn port, known limitations: sequences beyond the window
 *    are refused).  Kernels also guard every index they write, so a host mirror that
 *    disagrees with its device copy can drop a write but never corrupt memory.
 *  - Layouts are row-major with the last dimension contiguous.  D = head_dim.
 *    Token-major activations: q [.., T, Hq, D], k/v [.., T, Hkv, D], as a projection
 *    emits them.  Cache instance: K [Hkv, capacity, D], V [Hkv, capacity, D]
 *    (fixed-window cache of static shape: Youtu-VL-4B ncnn port, step 7).
 *  - Asymmetric caches: K rows of Dk = head_dim and V rows of Dv = head_dim_v elements (an
 *    MLA layer expanded to per-head K = 192, V = 128: Youtu-VL-4B ncnn port, section 6).
 *    Then q, k and q_out rows are Dk wide, v rows and attention outputs Dv wide.
 *  - GQA: query head h reads KV head h / (Hq / Hkv) (repeat-interleave grouping:
 *    Penguin-VL ncnn port, section 3 item 2).
 *  - Alignment: every device pointer must be 16-byte aligned, and D must be a
 *    multiple of 8 (vectorised 16-byte accesses); violations return KVA_EALIGN.
 */
#ifndef KV_ATTN_H_
#define KV_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kva_stream; /* identical to cudaStream_t */

typedef enum {
  KVA_OK = 0,
  KVA_EINVAL = 1,       /* bad shape, null pointer, unknown enum */
  KVA_ECAPACITY = 2,    /* slot or length beyond the cache window */
  KVA_EUNSUPPORTED = 3, /* valid request this build does not implement */
  KVA_ECUDA = 4,        /* a CUDA launch or driver call failed */
  KVA_EALIGN = 5,       /* pointer or stride not 16-byte aligned, D % 8 != 0 */
  KVA_EWORKSPACE = 6    /* workspace missing or smaller than required */
} kva_status;

typedef enum { KVA_F32 = 0, KVA_BF16 = 1 } kva_dtype;

typedef enum {
  KVA_MASK_CAUSAL = 0,  /* key slot j visible to query slot i iff j <= i */
  KVA_MASK_FULL = 1,    /* all S keys visible (bidirectional vision layers) */
  KVA_MASK_SEGMENT = 2, /* block diagonal: j visible iff segment[j] == segment[i] */
  KVA_MASK_CAUSAL_SEGMENT = 3  /* j <= i or segment[j] == segment[i]: causal, with each segment
                                  (an image span; a text token is its own segment) fully visible
                                  to its own rows (MNN llm_demo walkthrough, section 3.3) */
} kva_mask;

typedef enum {
  KVA_ROPE_NONE = 0,
  KVA_ROPE_1D = 1,       /* rotate-half over D, every frequency uses position axis 0 */
  KVA_ROPE_SECTIONS = 2, /* xdRoPE: frequency j uses the axis whose section holds j */
  KVA_ROPE_2D = 3,       /* two halves of D/2, each rotate-half; half b uses axis b */
  KVA_ROPE_INTERLEAVED = 4  /* de-interleave x to [x0,x2,..,x1,x3,..] then 1D rotate-half; the
                               output (q_out, cache K) stays in that order (rope_interleave:
                               Youtu-VL-4B ncnn port, implementation difficulty 2) */
} kva_rope_kind;

/* One cache: N instances (layers and/or sequences) of K [n_kv_heads, capacity, head_dim] and
 * V [n_kv_heads, capacity, head_dim_v] of `dtype`, K instance i starting at
 * k + i * inst_stride elements and V instance i at v + i * inst_stride_v elements.
 * inst_stride >= n_kv_heads*capacity*head_dim, inst_stride_v >= n_kv_heads*capacity*head_dim_v.
 * head_dim_v = 0 means head_dim and inst_stride_v = 0 means inst_stride (a symmetric cache,
 * where the two strides must agree). */
typedef struct {
  void* k;
  void* v;
  kva_dtype dtype;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t capacity;
  int64_t inst_stride;
  int32_t head_dim_v;
  int64_t inst_stride_v;
} kva_cache;

/* Rotary embedding (rotate-half pairs (j, j + W/2) inside each rotated block of width W):
 *   angle_j = pos[axis(j)] * base^(-2j/W),  y_j = x_j cos - x_{j+W/2} sin,
 *   y_{j+W/2} = x_{j+W/2} cos + x_j sin.
 *  1D (theta 1e6: Penguin-VL ncnn port, section 2.1), xdRoPE sections [16,16,16,16]
 *  with effective base 1.11588e7 (HunyuanOCR v1.0 ncnn port, section five items 1, 3),
 *  2D vision halves (Penguin-VL ncnn port, section 2.3).
 *  n_axes: position ids per token (1 for 1D, number of sections, 2 for 2D).
 *  rot_offset, rot_dim: the rotation covers head dims [rot_offset, rot_offset + rot_dim) and
 *  W above is rot_dim; the other dims pass through (the rotary 64 of a 192-wide MLA head:
 *  Youtu-VL-4B ncnn port, implementation difficulty 2).  rot_dim = 0: the whole head
 *  (rot_offset must then be 0). */
typedef struct {
  kva_rope_kind kind;
  int32_t n_axes;
  int32_t sections[4];
  double base;
  int32_t rot_offset;
  int32_t rot_dim;
} kva_rope;

/* Per-head RMSNorm y = x / sqrt(mean(x^2) + eps) * w with w [D] float32 on the device
 * (Penguin-VL ncnn port, sections 2.1, 4.2).  q_w == NULL and k_w == NULL: no norm.
 * inst_stride: floats between the weights of consecutive instances (0 = shared).
 * after_rope: 0 = norm then RoPE (Qwen3); 1 = RoPE then norm, the cache holding the
 * normalised K (HunyuanOCR v1.0 ncnn port, section five item 2). */
typedef struct {
  const float* q_w;
  const float* k_w;
  int64_t inst_stride;
  float eps;
  int32_t after_rope;
} kva_qknorm;

/* ---------------------------------------------------------------------------------
 * kv_cache_append_rope_qknorm
 *   For each instance n < N and token t < T:
 *     q_out[n,t,h,:] = f_q(q[n,t,h,:])                      h < Hq
 *     K_n[g, slot[n,t], :] = store(f_k(k[n,t,g,:]))          g < Hkv
 *     V_n[g, slot[n,t], :] = store(v[n,t,g,:])
 *   f = QK-Norm and RoPE in the order `norm.after_rope` gives; store rounds to the cache
 *   dtype (bf16: round to nearest even).  The runtime writes the new token's k/v into its
 *   cache slot between the qkv and the attention step (Youtu-VL-4B ncnn port, step 6).
 *  q       [N,T,Hq,D] of in_dtype (device);  k, v [N,T,Hkv,D] of in_dtype (device)
 *  pos     [.., T, rope.n_axes] int32 (device); instance n reads pos + n*pos_inst_stride
 *  slot    [.., T] int32 destination slot (device); instance n reads slot + n*slot_inst_stride
 *  slot_host  host mirror of the slot values actually read (same strides), used to reject
 *          slots outside [0, capacity) with KVA_ECAPACITY before launching
 *  q_out   [N,T,Hq,D] of q_out_dtype (device), token order
 *  Asymmetric caches take q, k [.., Dk] and v [.., Dv]; QK-Norm weights are Dk wide.
 *  Errors: KVA_EINVAL (N,T < 0, Hq % Hkv, sections not summing to W/2, W/2 odd for 2D, a
 *          rotary range outside the head), KVA_ECAPACITY, KVA_EALIGN,
 *          KVA_EUNSUPPORTED (Dk or Dv > 256), KVA_ECUDA.
 *  N == 0 or T == 0 is a no-op returning KVA_OK. */
kva_status kv_cache_append_rope_qknorm(
    const void* q, const void* k, const void* v, kva_dtype in_dtype,
    int32_t N, int32_t T, int32_t n_q_heads,
    const int32_t* pos, int64_t pos_inst_stride,
    const int32_t* slot, int64_t slot_inst_stride, const int32_t* slot_host,
    kva_qknorm norm, kva_rope rope,
    void* q_out, kva_dtype q_out_dtype,
    kva_cache cache, kva_stream stream);

/* ---------------------------------------------------------------------------------
 * kv_attn_prefill
 *   Parallel prefill over cache slots 0..S-1 of each instance (Youtu-VL-4B ncnn port,
 *   step 7; the fused flash-style form of MNN llm_demo walkthrough, section 5.1):
 *     o_i = softmax_j( q_i . K[g, j] * scale, j visible to i ) . V[g, j]
 *   softmax taken as max -> subtract -> exp -> sum -> divide (Youtu-VL-4B ncnn port,
 *   implementation difficulty 3), accumulated in fp32.
 *  q       [N,S,Hq,D] of q_dtype (device), token order.  The query of cache slot i is
 *          q row r(i) = row_of_slot[i] (or i when row_of_slot == NULL), and its output
 *          goes to out row r(i): this undoes a window permutation (the vision tower's
 *          window_index grouping: Youtu-VL-4B ncnn port, step 3).
 *  segment [S] int32 (device), non-decreasing segment id per slot, for KVA_MASK_SEGMENT
 *          and KVA_MASK_CAUSAL_SEGMENT (else NULL); segment_host: its host mirror
 *          (validated: non-decreasing).
 *  scale   softmax scale; <= 0 selects 1/sqrt(Dk).
 *  out     [N,S,Hq,Dv] float32 (device).
 *  Errors: KVA_EINVAL, KVA_ECAPACITY (S > capacity), KVA_EALIGN, KVA_EUNSUPPORTED
 *          (D > 256), KVA_ECUDA.  q_dtype must equal cache.dtype. */
kva_status kv_attn_prefill(
    const void* q, kva_dtype q_dtype, kva_cache cache,
    int32_t N, int32_t S, int32_t n_q_heads, kva_mask mask,
    const int32_t* segment, const int32_t* segment_host,
    const int32_t* row_of_slot,
    float scale, float* out, kva_stream stream);

/* ---------------------------------------------------------------------------------
 * kv_attn_decode
 *   One query token per instance b against its first L_b cache slots (the new token's
 *   slot included): o = softmax(q K[:L]^T * scale) V[:L] (Youtu-VL-4B ncnn port,
 *   step 8; dattn consumes the whole cache window plus the mask).  Split-KV: the
 *   L_b keys are cut into chunks processed by separate CTAs whose partial
 *   (max, sum, acc) triples are merged by the last CTA of each (b, kv head).
 *  q          [B,Hq,D] of q_dtype (device)
 *  lengths    [B] int32 valid slots per instance (device); lengths_host: host mirror,
 *             required (validation 1 <= L_b <= capacity, and chunk planning)
 *  out        [B,Hq,D] float32 (device)
 *  workspace  device scratch of at least kva_decode_workspace_size(...) bytes whose
 *             first kva_decode_workspace_zero_bytes(B, Hkv) bytes are zero before the first
 *             call; every call leaves them zero again.  Calls sharing one workspace must
 *             not overlap on the GPU.
 *  Built for (Dk, Dv) = (128, 128) and the asymmetric (192, 128); q is [B,Hq,Dk], out
 *  [B,Hq,Dv]; kva_decode_workspace_size takes Dv as its head_dim.
 *  Errors: KVA_EINVAL, KVA_ECAPACITY, KVA_EALIGN, KVA_EWORKSPACE,
 *          KVA_EUNSUPPORTED (other head dims), KVA_ECUDA.  B == 0 is a no-op. */
kva_status kv_attn_decode(
    const void* q, kva_dtype q_dtype, kva_cache cache,
    const int32_t* lengths, const int32_t* lengths_host, int32_t B, int32_t n_q_heads,
    float scale, float* out, void* workspace, size_t workspace_bytes, kva_stream stream);

/* ---------------------------------------------------------------------------------
 * kv_attn_decode_step
 *   One decode step in one launch: the append of the new token followed by decode
 *   attention, i.e. exactly
 *     kv_cache_append_rope_qknorm(q, k, v, T = 1, slot = L_b - 1, ...)   then
 *     kv_attn_decode(q_out, lengths, ...)
 *   (the runtime writes the new k/v into the cache between the qkv and the attention step:
 *   Youtu-VL-4B ncnn port, step 6; each step attends to the whole prefix: step 8).  Every
 *   CTA derives the normalised, rotated query rows of its group itself; the CTA that owns the
 *   last chunk of an instance also writes the new K/V row into slot L_b - 1.
 *  q        [B,Hq,Dk], k [B,Hkv,Dk], v [B,Hkv,Dv] of in_dtype: the new token's projections (device)
 *  pos      [.., n_axes] int32 position ids (device); instance b reads pos + b*pos_inst_stride
 *  lengths  [B] valid slots including the new token (device) + lengths_host (host mirror)
 *  q_out    nullable [B,Hq,Dk] of q_out_dtype: the transformed queries, if wanted
 *  out      [B,Hq,Dv] float32;  workspace as for kv_attn_decode
 *  Built for (Dk, Dv) = (128, 128) bf16 or fp32 caches and the asymmetric (192, 128) cache,
 *  any RoPE kind over the whole head or a sub-range (rope.rot_offset, rope.rot_dim), and
 *  Hq/Hkv in {1, 2, 4} (else KVA_EUNSUPPORTED: call the two entry points).  A symmetric bf16
 *  cache with whole-head RoPE runs on the tensor-core decode kernel, the other forms on the
 *  CUDA-core one.  workspace: kva_decode_workspace_size with head_dim = Dv.  Errors as the two
 *  calls it replaces. */
kva_status kv_attn_decode_step(
    const void* q, const void* k, const void* v, kva_dtype in_dtype,
    const int32_t* pos, int64_t pos_inst_stride,
    kva_qknorm norm, kva_rope rope, kva_cache cache,
    const int32_t* lengths, const int32_t* lengths_host, int32_t B, int32_t n_q_heads,
    float scale, void* q_out, kva_dtype q_out_dtype, float* out,
    void* workspace, size_t workspace_bytes, kva_stream stream);

/* ---------------------------------------------------------------------------------
 * kv_attn_verify  (speculative-decoding verify block)
 *   The target-verification forward of a draft block (HunyuanOCR v1.5 ncnn port, section 3.8):
 *   the block's k tokens (the current token and k-1 draft candidates) already sit in the last
 *   k valid slots, L-k .. L-1, of each instance (appended like any tokens), and block row i
 *   attends to slots 0 .. L-k+i with the same GQA grouping and softmax as kv_attn_decode.
 *  q        [B,k,Hq,D] of q_dtype: the block's transformed queries (device)
 *  lengths  [B] valid slots L including the block (device); lengths_host: host copy or an
 *           upper bound of it (used for validation and work planning; L >= k required)
 *  out      [B,k,Hq,D] float32
 *  workspace as for kv_attn_decode, sized by kva_verify_workspace_size; merge counters are
 *  left at zero.  Requires a symmetric bf16 cache with head_dim 128 (else KVA_EUNSUPPORTED) and
 *  1 <= k <= KVA_VERIFY_MAX_BLOCK. */
#define KVA_VERIFY_MAX_BLOCK 64
kva_status kv_attn_verify(
    const void* q, kva_dtype q_dtype, kva_cache cache,
    const int32_t* lengths, const int32_t* lengths_host, int32_t B, int32_t k, int32_t n_q_heads,
    float scale, float* out, void* workspace, size_t workspace_bytes, kva_stream stream);
size_t kva_verify_workspace_size(int32_t B, int32_t n_kv_heads, int32_t n_q_heads, int32_t k,
                                 int32_t max_len, int32_t head_dim);

/* ---------------------------------------------------------------------------------
 * kv_verify_commit
 *   Acceptance and commit of a verify block (HunyuanOCR v1.5 ncnn port, section 3.8), on the
 *   device so no host round trip is needed: for instance b, block_tokens[b,0..k) are the block's
 *   tokens and posterior[b,0..k) the target's greedy id after each of them (lmhead_argmax over
 *   the block's rows).  Candidate i+1 is accepted while posterior[b,i] == block_tokens[b,i+1];
 *   accepted[b] = the accepted count a, next_token[b] = posterior[b,a] (the target's correction,
 *   or its next token when every candidate matched), and lengths[b] is cut from L to
 *   L - k + a + 1 (the current token and the accepted candidates keep their K/V; the slots
 *   after them are free for the next block).  All pointers are device int32 arrays. */
kva_status kv_verify_commit(const int32_t* posterior, const int32_t* block_tokens, int32_t B, int32_t k,
                            int32_t* lengths, int32_t* accepted, int32_t* next_token, kva_stream stream);

size_t kva_decode_workspace_size(int32_t B, int32_t n_kv_heads, int32_t n_q_heads,
                                 int32_t max_len, int32_t head_dim);
size_t kva_decode_workspace_zero_bytes(int32_t B, int32_t n_kv_heads);

/* ---------------------------------------------------------------------------------
 * kv_attn_decode_static
 *   The same decode as kv_attn_decode for callers that cannot allocate device memory
 *   (a host framework that owns every allocation, code that must not touch an allocator
 *   in its hot loop): there is no workspace argument.  The split-KV scratch lives in a
 *   fixed 4 MiB array inside this library's device image; every GPU that loads the
 *   library holds it until the process exits.  The reference pages have no counterpart
 *   of this call.
 *  Arguments and errors: as kv_attn_decode, for symmetric caches.  A batch whose partials cannot fit the fixed
 *   scratch even as one chunk per instance (B * n_q_heads * (head_dim + 2) * 4 bytes plus
 *   the counters above 4 MiB) returns KVA_EWORKSPACE; otherwise larger chunks are chosen
 *   until the partials fit.
 *  The call allocates nothing (no cudaMalloc, no cudaFree).  The first call on a device
 *   looks up the array's device address (cudaGetSymbolAddress); make that first call
 *   before any stream capture.  The address is kept for the life of the process, so do not
 *   use the library across a cudaDeviceReset.  Every call clears the merge counters it needs
 *   on `stream`.
 *  All calls share the one array, which keeps the last call's contents: calls that
 *   overlap on the GPU (different streams, or concurrent graphs) race on it and must be
 *   serialised by the caller. */
kva_status kv_attn_decode_static(
    const void* q, kva_dtype q_dtype, kva_cache cache,
    const int32_t* lengths, const int32_t* lengths_host, int32_t B, int32_t n_q_heads,
    float scale, float* out, kva_stream stream);

/* ---------------------------------------------------------------------------------
 * lmhead_argmax
 *   Greedy tied lm_head: z[b, v] = sum_k W[v, k] h[b, k] for v < V, ids[b] = argmax_v z[b, v]
 *   (Youtu-VL-4B ncnn port, step 6: final-norm hidden dotted with every vocab row,
 *   argmax only; HunyuanOCR v1.5 ncnn port, section 3.4: one [vocab, hidden] copy).
 *   Ties go to the lowest id.  Only rows v < V are candidates; V > V_rows is rejected
 *   (the vocab is clamped to the logits length: Penguin-VL ncnn port, section 4.1).
 *   Logits accumulate in float32.  NaN inputs are outside the contract.
 *  h          [B,H] float32 (device);  W [V_rows, H] of w_dtype (device)
 *  out_ids    [B] int32 (device);  out_max [B] float32 max logit (device, nullable)
 *  logits     [B,V] float32 (device, nullable): every logit, for inspection
 *  workspace  device scratch of at least kva_lmhead_workspace_size(B, H) bytes whose first
 *             kva_lmhead_workspace_zero_bytes(B) bytes are zero before the first call; every
 *             call leaves them zero again.  Calls sharing one workspace must not overlap on
 *             the GPU.
 *  B == 1 streams the table with CUDA-core dot products; 2 <= B <= 128 (bf16 table, H a
 *  multiple of 64) runs on the tensor cores with h split into two bf16 halves (h_hi + h_lo
 *  carries ~16 significant bits), fp32 accumulation.
 *  Errors: KVA_EINVAL, KVA_EALIGN (H % 8), KVA_EWORKSPACE, KVA_ECUDA.  B == 0 is a no-op. */
kva_status lmhead_argmax(
    const float* h, const void* W, kva_dtype w_dtype,
    int32_t B, int32_t H, int32_t V, int32_t V_rows,
    int32_t* out_ids, float* out_max, float* logits,
    void* workspace, size_t workspace_bytes, kva_stream stream);

/* ---------------------------------------------------------------------------------
 * lmhead_topk  (final RMSNorm + lm_head, k best ids)
 *   Every decode step ends with the final RMSNorm, the tied lm_head over the whole vocabulary
 *   and the pick of the best token (Youtu-VL-4B ncnn port, "decoding and sampling"; step 8);
 *   top_k is one of the runtime's generation options (HunyuanOCR v1.5 ncnn port, section 3.6).
 *   h_b' = h_b / sqrt(mean(h_b^2) + eps) * norm_w (skipped when norm_w is NULL), logits
 *   z_b[v] = W[v] . h_b' for v < V, then the top_k best (id, logit) pairs per row ordered by
 *   logit descending, equal logits toward the lower id.  The norm is applied inside the lm_head
 *   kernels as they load h (no separate pass).  top_k = 1 is the greedy id through the fused
 *   argmax; top_k > 1 writes the logits to the workspace and ranks each row in a second kernel.
 *  h        [B,H] float32;  norm_w  [H] float32 or NULL;  W [V_rows,H] of w_dtype
 *  out_ids  [B,top_k] int32;  out_vals [B,top_k] float32 or NULL
 *  workspace: kva_lmhead_topk_workspace_size(B, H, V, top_k) bytes, counters zeroed once
 *  (the calls leave them at zero).  1 <= top_k <= 32 and top_k <= V, else KVA_EINVAL. */
kva_status lmhead_topk(
    const float* h, const float* norm_w, float eps, const void* W, kva_dtype w_dtype,
    int32_t B, int32_t H, int32_t V, int32_t V_rows, int32_t top_k,
    int32_t* out_ids, float* out_vals, void* workspace, size_t workspace_bytes, kva_stream stream);
size_t kva_lmhead_topk_workspace_size(int32_t B, int32_t H, int32_t V, int32_t top_k);

size_t kva_lmhead_workspace_size(int32_t B, int32_t H);
size_t kva_lmhead_workspace_zero_bytes(int32_t B);

/* ---------------------------------------------------------------------------------
 * kva_workspace_size
 *   One sizer for every call that takes a workspace (the boundary lists a single
 *   kva_workspace_size(which, ...)); it returns what the per-call sizer above returns for
 *   the same dimensions.  `which` names the call; the fields of `dims` it reads:
 *     KVA_WS_DECODE        kv_attn_decode, kv_attn_decode_step:
 *                          B, n_kv_heads, n_q_heads, max_len, head_dim (Dv)
 *     KVA_WS_VERIFY        kv_attn_verify: the same plus block (k)
 *     KVA_WS_LMHEAD        lmhead_argmax: B, hidden
 *     KVA_WS_LMHEAD_TOPK   lmhead_topk: B, hidden, vocab, block (top_k)
 *   Fields a kind does not read are ignored.  Returns 0 for an unknown kind, a NULL `dims` or
 *   a dimension that is not positive. */
typedef enum {
  KVA_WS_DECODE = 0,
  KVA_WS_VERIFY = 1,
  KVA_WS_LMHEAD = 2,
  KVA_WS_LMHEAD_TOPK = 3
} kva_workspace_kind;

typedef struct {
  int32_t B;
  int32_t n_kv_heads;
  int32_t n_q_heads;
  int32_t max_len;   /* largest valid length L any call will pass */
  int32_t head_dim;  /* value head width Dv of the attention output */
  int32_t hidden;    /* lm_head hidden size H */
  int32_t vocab;     /* lm_head candidate rows V */
  int32_t block;     /* verify block length k, or top_k */
} kva_workspace_dims;

size_t kva_workspace_size(int32_t which, const kva_workspace_dims* dims);

/* ---------------------------------------------------------------------------------
 * Introspection */
const char* kva_strerror(kva_status s);
/* Message describing the last non-OK status returned on the calling host thread. */
const char* kva_last_error(void);
/* Number of kernels this library has launched in this process (all threads). */
uint64_t kva_launch_count(void);
/* Library ABI version: major * 10000 + minor * 100 + patch. */
int32_t kva_version(void);

/* ---------------------------------------------------------------------------------
 * Failure detection (no counterpart on the pages).  Every wait of a kernel on an mbarrier (a
 * copy landing, another warp's hand-off) gives up after about 2 s of GPU time instead of
 * hanging; the kernel then abandons its work and writes NaN into the outputs it owns (-1 into
 * the lm_head's ids), and the device stays usable.
 * kva_wait_timeouts: how many thread-level waits have given up on the current device since the
 *   last reset (0 in normal operation; one abandoned kernel usually counts many), or -1 if the
 *   count could not be read.  reset != 0 clears it.  Synchronise the streams that ran the
 *   kernels before reading; the call is synchronous and must not be made during stream capture.
 * kva_selftest_wait_timeout: launches one kernel whose wait nothing satisfies, so that it gives
 *   up after the limit: a test of the timeout path that neither hangs nor faults the GPU. */
int64_t kva_wait_timeouts(int32_t reset);
kva_status kva_selftest_wait_timeout(kva_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* KV_ATTN_H_ */
