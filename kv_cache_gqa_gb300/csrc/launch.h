// Internal interface between the host entry points (kv_attn_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "kv_attn.h"

namespace kva {

// Set-up that a launcher does once per device, such as raising a kernel's shared-memory
// limit: function attributes belong to each device's context, so a process that drives
// several GPUs sets them on each.  done() tells whether the current device is set up and
// mark() records it (devices past 63 are set up on every call; repeating it is harmless).
// Per-device state lives for the whole process: the library is not meant to be used across
// a cudaDeviceReset.
struct DeviceOnce {
  std::atomic<unsigned long long> mask{0};
  static int current() {
    int d = 0;
    return cudaGetDevice(&d) == cudaSuccess ? d : 64;
  }
  bool done() const {
    const int d = current();
    return d < 64 && ((mask.load(std::memory_order_acquire) >> d) & 1ull);
  }
  void mark() {
    const int d = current();
    if (d < 64) mask.fetch_or(1ull << d, std::memory_order_release);
  }
};

constexpr int MAX_ROPE_FREQ = 128;  // D/2 for D <= 256

// Rotary table description: angle slot j (0 <= j < D/2) uses position axis axis[j] and
// inverse frequency inv[j] (float64, computed on the host).
struct RopeTable {
  int kind;
  int n_axes;
  double inv[MAX_ROPE_FREQ];
  float inv_hi[MAX_ROPE_FREQ];   // float(inv[j]) and float(inv[j] - inv_hi[j]): inv as a float pair
  float inv_lo[MAX_ROPE_FREQ];
  unsigned char axis[MAX_ROPE_FREQ];
};

struct AppendArgs {
  const void* q;
  const void* k;
  const void* v;
  void* q_out;
  void* kc;
  void* vc;
  const int32_t* pos;
  int64_t pos_stride;
  const int32_t* slot;
  int64_t slot_stride;
  const float* q_w;
  const float* k_w;
  int64_t w_stride;
  float eps;
  int after_rope;
  int N, T, Hq, Hkv, D, capacity;
  int64_t inst_stride;
  int Dv;                  // V row width (= D unless the cache is asymmetric)
  int64_t inst_stride_v;   // elements between V instances
  int rot_offset, rot_dim; // rotated dims [rot_offset, rot_offset + rot_dim); the table is rot_dim wide
  RopeTable rope;
};

bool append_supports_head_dim(int D);
// Any layout the fast forms do not take: an asymmetric cache, a rotary sub-range, other head dims.
bool append_general_supports(int Dk, int Dv);
cudaError_t launch_append_general(const AppendArgs& a, kva_dtype in_dtype, kva_dtype q_out_dtype,
                                  kva_dtype cache_dtype, cudaStream_t s);
cudaError_t launch_append(const AppendArgs& a, kva_dtype in_dtype, kva_dtype q_out_dtype,
                          kva_dtype cache_dtype, cudaStream_t s);

// ---------------------------------------------------------------------------------
struct DecodeArgs {
  const void* q;          // [B, Hq, D]
  const void* kc;
  const void* vc;
  const int32_t* lengths; // [B]
  float* out;             // [B, Hq, D]
  unsigned int* counters; // [B * Hkv] zero on entry, zero on exit
  float* part_acc;        // [B, Hq, max_chunks, D]
  float* part_ml;         // [B, Hq, max_chunks, 2]
  int B, Hq, Hkv, capacity, chunk, max_chunks;
  int64_t inst_stride;
  int64_t inst_stride_v;  // V instances (= inst_stride for symmetric caches)
  float scale_log2;       // softmax scale * log2(e)
};

// Multi-query verify block (kv_attn_verify): k query rows per instance, row i attending to
// slots [0, L - k + i].  Rows are (block position i, head j of the group) -> r = i * G + j,
// 16 per CTA; RT = ceil(G * k / 16) row tiles per (instance, KV head).
struct VerifyArgs {
  const void* q;          // [B, k, Hq, D]
  const void* kc;
  const void* vc;
  const int32_t* lengths; // [B] valid slots, the block's k tokens included
  float* out;             // [B, k, Hq, D]
  unsigned int* counters; // [B, Hkv, RT] zero on entry, zero on exit
  float* part_acc;        // [B, Hkv, RT, 16, max_chunks, D]
  float* part_ml;         // [B, Hkv, RT, 16, max_chunks, 2]
  int B, k, Hq, Hkv, RT, capacity, chunk, max_chunks;
  int64_t inst_stride;
  float scale_log2;
};
cudaError_t launch_verify(const VerifyArgs& a, kva_dtype q_dtype, cudaStream_t s);
// tcgen05 form (a group of G*k <= 128 rows on one 128-row MMA tile): persistent CTAs over
// (chunk, KV head, instance) units.  `chunk` is planned by verify_tc_plan_chunk.
bool verify_tc_supports(int G, int k);
int verify_tc_plan_chunk(const int32_t* lengths_host, int B, int Hkv, int max_len);
cudaError_t launch_verify_tc(const VerifyArgs& a, kva_dtype q_dtype, cudaStream_t s);
// (D=128 bf16 cache) 4-D TMA map over a cache with boxes of [16 slots x 64 dims].
cudaError_t decode_cache_map(CUtensorMap* map, const void* base, int capacity, int Hkv, int B, int64_t inst_stride);
// Acceptance and commit of verify blocks (one thread per instance).
cudaError_t launch_verify_commit(const int32_t* posterior, const int32_t* block_tokens, int B, int k,
                                 int32_t* lengths, int32_t* accepted, int32_t* next_token, cudaStream_t s);

// Raw inputs of the new token for the fused append + decode step (kv_attn_decode_step).
struct StepArgs {
  const void* q;          // [B, Hq, D] projections of the new token
  const void* k;          // [B, Hkv, D]
  const void* v;          // [B, Hkv, D]
  int in_dtype;           // kva_dtype of q, k, v
  const int32_t* pos;     // instance b reads pos + b * pos_stride (n_axes ids)
  int64_t pos_stride;
  const float* q_w;       // QK-Norm weights or null
  const float* k_w;
  int64_t w_stride;
  float eps;
  int after_rope;
  void* q_out;            // optional [B, Hq, D] transformed queries
  int q_out_dtype;
  int rot_offset, rot_dim;  // rotated dims [rot_offset, rot_offset + rot_dim) of a q/k row
  RopeTable rope;           // frequencies of a rot_dim-wide block
};

constexpr int DECODE_HEAD_DIM = 128;
int decode_subtile(kva_dtype cache_dtype);   // keys per pipeline stage
// The fused decode step on the CUDA-core kernel (fp32 caches, the 192/128 cache, rotary
// sub-ranges); the tensor-core form is launch_decode_step.
bool decode_step_simt_supported(int Dk, int Dv, int G);
cudaError_t launch_decode_step_simt(const DecodeArgs& a, const StepArgs& st, int Dk, kva_dtype cache_dtype,
                                    cudaStream_t s);
int decode_num_sms();
// Split-KV plan: `chunk` = target keys per CTA (instance b is cut into ceil(L_b / chunk)
// nearly equal chunks), a multiple of 64, with at most 64 chunks per instance.
// row_bytes: K plus V bytes per key and KV head; ctas_per_sm: resident decode CTAs per SM.
int decode_plan_chunk(const int32_t* lengths_host, int B, int Hkv, int max_len, double row_bytes = 512.0,
                      int ctas_per_sm = 2);
cudaError_t launch_decode(const DecodeArgs& a, kva_dtype q_dtype, kva_dtype cache_dtype,
                          cudaStream_t s);
// CUDA-core decode for (Dk, Dv) = (192, 128) caches (G in {1, 2, 4}).
bool decode_asym_supported(int Dk, int Dv);
cudaError_t launch_decode_asym(const DecodeArgs& a, int Dk, int Dv, kva_dtype q_dtype, kva_dtype cache_dtype,
                               cudaStream_t s);
// Fused append + decode (bf16 cache, D = 128, G in {1, 2, 4}); false if this build cannot.
bool decode_step_supported(int G);
bool decode_mma_supported();
cudaError_t launch_decode_step(const DecodeArgs& a, const StepArgs& st, cudaStream_t s);

// ---------------------------------------------------------------------------------
struct LmheadArgs {
  const float* h;            // [B, H]
  const void* W;             // [V_rows, H]
  int32_t* out_ids;          // [B]
  float* out_max;            // [B] or null
  float* logits;             // [B, V] or null
  unsigned long long* best;  // [B] zero on entry, zero on exit
  unsigned int* counter;     // [1] zero on entry, zero on exit
  const float* norm_w;       // [H] final RMSNorm weight applied to h first, or null
  float eps;
  int B, H, V;
};
size_t lmhead_workspace_bytes(int B, int H);
size_t lmhead_zero_bytes(int B);
// Launches the lm_head for `a`; *n_launches receives the number of kernels enqueued.
cudaError_t launch_lmhead(const LmheadArgs& a, kva_dtype w_dtype, void* hb_scratch, cudaStream_t s,
                          unsigned* n_launches);
// Top-k of each row of logits [B, V] (k <= 32): ids and values ordered by value descending,
// ties toward the lower id.
constexpr int LMHEAD_TOPK_MAX = 32;
// workspace: topk_rows_workspace_bytes(B, V), its first round_up(4 B, 256) bytes (per-row
// tickets) zero on entry and left at zero.
size_t topk_rows_workspace_bytes(int B, int V);
cudaError_t launch_topk_rows(const float* logits, int B, int V, int k, void* workspace, int32_t* out_ids,
                             float* out_vals, cudaStream_t s);

// ---------------------------------------------------------------------------------
constexpr int PREFILL_SEG_TABLE = 64;   // segment ids with bounds passed in the arguments
struct PrefillArgs {
  const void* q;              // [N, S, Hq, D]
  const void* kc;
  const void* vc;
  const int32_t* segment;     // [S] or null
  const int32_t* row_of_slot; // [S] or null
  float* out;                 // [N, S, Hq, Dv]
  int N, S, Hq, Hkv, D, capacity, mask;
  int64_t inst_stride;
  int Dv;                     // V row width (= D unless asymmetric)
  int64_t inst_stride_v;
  float scale_log2;
  int single_slot;            // tcgen05 form: one query tile per work unit (set by its launcher)
  // Segment masks: slots [seg_lo[g], seg_hi[g]) hold segment id g, for ids g < seg_table
  // (filled on the host from the segment ids' host mirror; 0 = no table).  A row whose id is
  // in the table reads its window bounds here instead of bisecting the ids.
  int seg_table;
  int seg_lo[PREFILL_SEG_TABLE], seg_hi[PREFILL_SEG_TABLE];
};
int lmhead_max_hidden();
cudaError_t launch_prefill(const PrefillArgs& a, kva_dtype dtype, cudaStream_t s);

// Launch `kern` with programmatic stream serialization: its set-up overlaps the tail of the
// kernel before it on the stream.  The kernel must call griddep_wait() before its first global
// memory access.  A kernel that allocates tensor memory must do so before it calls
// griddep_launch_dependents(): a dependent CTA may allocate during its own set-up, so every CTA
// of the earlier grid must already hold its columns by then.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Launch bookkeeping (kernel launches issued by this library).
void count_launches(unsigned n);
// Record the message kva_last_error() returns on this host thread.
void set_last_error(const char* msg);

}  // namespace kva
