// Host side of the C ABI declared in include/kv_attn.h: argument validation, launch
// planning and dispatch to the kernels.  Nothing here allocates device memory.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <vector>

#include "common.cuh"
#include "kv_attn.h"
#include "launch.h"

namespace kva {

static std::atomic<unsigned long long> g_launches{0};

// Readers of the per-translation-unit wait give-up counters (registered at library load).
static std::vector<cudaError_t (*)(unsigned*, bool)>& wait_counters() {
  static std::vector<cudaError_t (*)(unsigned*, bool)> v;
  return v;
}
void register_wait_counter(cudaError_t (*read)(unsigned*, bool)) { wait_counters().push_back(read); }

// One thread waits on a barrier that nothing arrives on: the wait gives up after its limit.
__global__ void selftest_wait_kernel() {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0u);
}
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int lmhead_max_hidden();
bool prefill_simt_supports(int Dk, int Dv);
cudaError_t launch_prefill_simt(const PrefillArgs& a, kva_dtype dt, cudaStream_t s);
bool prefill_tc_supports(int D, int Dv, kva_dtype dt);
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s);

namespace {

thread_local char g_msg[512] = "";

kva_status fail(kva_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

kva_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return KVA_OK;
  return fail(KVA_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int elem_size(kva_dtype d) { return d == KVA_BF16 ? 2 : 4; }
bool valid_dtype(kva_dtype d) { return d == KVA_F32 || d == KVA_BF16; }

// Checks the cache and resolves its defaults in place (head_dim_v, inst_stride_v).
kva_status check_cache(kva_cache& c, int n_instances) {
  if (!valid_dtype(c.dtype)) return fail(KVA_EINVAL, "cache dtype %d unknown", (int)c.dtype);
  if (!c.k || !c.v) return fail(KVA_EINVAL, "cache k/v pointer is NULL");
  if (c.head_dim_v < 0 || c.inst_stride_v < 0) return fail(KVA_EINVAL, "negative head_dim_v or inst_stride_v");
  if (c.head_dim_v == 0) c.head_dim_v = c.head_dim;
  if (c.inst_stride_v == 0) c.inst_stride_v = c.inst_stride;
  if (c.n_kv_heads <= 0 || c.head_dim <= 0 || c.capacity <= 0)
    return fail(KVA_EINVAL, "cache shape must be positive (Hkv=%d D=%d capacity=%d)",
                c.n_kv_heads, c.head_dim, c.capacity);
  if (c.head_dim_v == c.head_dim && c.inst_stride_v != c.inst_stride)
    return fail(KVA_EINVAL, "a symmetric cache has one instance stride (inst_stride_v %lld != %lld)",
                (long long)c.inst_stride_v, (long long)c.inst_stride);
  const int64_t inst = (int64_t)c.n_kv_heads * c.capacity * c.head_dim;
  const int64_t inst_v = (int64_t)c.n_kv_heads * c.capacity * c.head_dim_v;
  if (n_instances > 1 && c.inst_stride < inst)
    return fail(KVA_EINVAL, "cache inst_stride %lld < Hkv*capacity*D = %lld",
                (long long)c.inst_stride, (long long)inst);
  if (n_instances > 1 && c.inst_stride_v < inst_v)
    return fail(KVA_EINVAL, "cache inst_stride_v %lld < Hkv*capacity*Dv = %lld",
                (long long)c.inst_stride_v, (long long)inst_v);
  if (c.head_dim % 8 != 0 || c.head_dim_v % 8 != 0)
    return fail(KVA_EALIGN, "head_dim %d / head_dim_v %d not a multiple of 8", c.head_dim, c.head_dim_v);
  if (!aligned16(c.k) || !aligned16(c.v)) return fail(KVA_EALIGN, "cache k/v not 16-byte aligned");
  if ((c.inst_stride * elem_size(c.dtype)) % 16 != 0 || (c.inst_stride_v * elem_size(c.dtype)) % 16 != 0)
    return fail(KVA_EALIGN, "cache instance strides are not multiples of 16 bytes");
  return KVA_OK;
}

bool asymmetric(const kva_cache& c) { return c.head_dim_v != c.head_dim; }

// Resolves the rotated range of a head of width Dk: [*off, *off + *width).
kva_status rope_range(const kva_rope& r, int Dk, int* off, int* width) {
  if (r.rot_dim == 0) {
    if (r.rot_offset != 0) return fail(KVA_EINVAL, "rot_offset %d needs a rot_dim", r.rot_offset);
    *off = 0; *width = Dk;
    return KVA_OK;
  }
  if (r.rot_offset < 0 || r.rot_dim < 0 || (int64_t)r.rot_offset + r.rot_dim > Dk)
    return fail(KVA_EINVAL, "rotary range [%d, %d + %d) outside the head of %d dims", r.rot_offset,
                r.rot_offset, r.rot_dim, Dk);
  if (r.rot_dim % 2 != 0) return fail(KVA_EINVAL, "rot_dim %d must be even", r.rot_dim);
  *off = r.rot_offset; *width = r.rot_dim;
  return KVA_OK;
}

// Table of a rotated block of width D (the head, or the rotary sub-range of it).
kva_status build_rope(const kva_rope& r, int D, RopeTable* t) {
  std::memset(t, 0, sizeof(*t));
  t->kind = (int)r.kind;
  t->n_axes = r.n_axes;
  if (r.kind == KVA_ROPE_NONE) return KVA_OK;
  if (!(r.base > 0.0) || !std::isfinite(r.base)) return fail(KVA_EINVAL, "rope base must be > 0");
  if (D / 2 > MAX_ROPE_FREQ) return fail(KVA_EUNSUPPORTED, "head_dim %d too large for RoPE", D);
  switch (r.kind) {
    case KVA_ROPE_1D:
    case KVA_ROPE_INTERLEAVED:
      if (r.n_axes < 1) return fail(KVA_EINVAL, "1D RoPE needs n_axes >= 1");
      for (int j = 0; j < D / 2; ++j) { t->inv[j] = std::pow(r.base, -2.0 * j / D); t->axis[j] = 0; }
      return KVA_OK;
    case KVA_ROPE_SECTIONS: {
      if (r.n_axes < 1 || r.n_axes > 4) return fail(KVA_EINVAL, "section RoPE needs 1..4 axes");
      int j = 0;
      for (int ax = 0; ax < r.n_axes; ++ax) {
        if (r.sections[ax] < 0) return fail(KVA_EINVAL, "negative RoPE section");
        for (int u = 0; u < r.sections[ax]; ++u, ++j) {
          if (j >= D / 2) return fail(KVA_EINVAL, "RoPE sections exceed D/2 = %d", D / 2);
          t->inv[j] = std::pow(r.base, -2.0 * j / D);
          t->axis[j] = (unsigned char)ax;
        }
      }
      if (j != D / 2) return fail(KVA_EINVAL, "RoPE sections sum to %d, expected D/2 = %d", j, D / 2);
      return KVA_OK;
    }
    case KVA_ROPE_2D: {
      if (r.n_axes != 2) return fail(KVA_EINVAL, "2D RoPE needs n_axes == 2");
      if (D % 4 != 0) return fail(KVA_EINVAL, "2D RoPE needs a rotated width %% 4 == 0");
      const int Q = D / 4;
      for (int b = 0; b < 2; ++b)
        for (int j = 0; j < Q; ++j) {
          t->inv[b * Q + j] = std::pow(r.base, -2.0 * j / (D / 2));
          t->axis[b * Q + j] = (unsigned char)b;
        }
      return KVA_OK;
    }
    default:
      return fail(KVA_EINVAL, "rope kind %d unknown", (int)r.kind);
  }
}

kva_status build_rope_table(const kva_rope& r, int D, RopeTable* t) {
  // A decode loop passes the same rotary layout on every call: the last table built on this
  // host thread is reused when the layout and width match (the D/2 pow() calls cost microseconds).
  thread_local kva_rope last_r{};
  thread_local int last_D = -1;
  thread_local RopeTable last_t;
  if (last_D == D && std::memcmp(&last_r, &r, sizeof(r)) == 0) {
    *t = last_t;
    return KVA_OK;
  }
  const kva_status st = build_rope(r, D, t);
  if (st != KVA_OK) return st;
  for (int j = 0; j < MAX_ROPE_FREQ; ++j) {
    t->inv_hi[j] = (float)t->inv[j];
    t->inv_lo[j] = (float)(t->inv[j] - (double)t->inv_hi[j]);
  }
  last_r = r; last_D = D; last_t = *t;
  return KVA_OK;
}

constexpr int DECODE_MAX_CHUNKS = 64;
constexpr int DECODE_CHUNK_ALIGN = 64;

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

size_t decode_zero_bytes(int B, int Hkv) { return round_up(sizeof(unsigned) * (size_t)B * Hkv, 256); }

size_t decode_ws_bytes(int B, int Hkv, int Hq, int max_chunks, int D) {
  return decode_zero_bytes(B, Hkv) + round_up(sizeof(float) * (size_t)B * Hq * max_chunks * 2, 256) +
         sizeof(float) * (size_t)B * Hq * max_chunks * D;
}

int decode_max_chunks_bound(int max_len) {
  return std::max(1, std::min(DECODE_MAX_CHUNKS, (max_len + DECODE_CHUNK_ALIGN - 1) / DECODE_CHUNK_ALIGN));
}

}  // namespace

void set_last_error(const char* msg) { std::snprintf(g_msg, sizeof(g_msg), "%s", msg); }

// Split-KV plan.  Instance b is cut into ceil(L_b / chunk) chunks, one CTA each.  Candidate
// chunk sizes are ceil(max_len / k) (k = 1..64, rounded up to 64 keys); each is scored with a
// simple cost model and the cheapest wins:
//   one wave:   fixed cost + max(all bytes / HBM bandwidth, one chunk / one CTA's share)
//   more waves: waves x fixed cost + all bytes / HBM bandwidth + one chunk / share (the tail)
//   plus, when instances are split, the merge (partials written, the counter, the last CTA's
//   reads): a 65..80-key fp32 decode step is one chunk per head instead of 64 + 1..16 keys
//   (6.0 instead of 7.7 us); a larger merge cost would also keep the 512-slot MLA step whole,
//   which measured 35% slower
// (fixed cost = a CTA's first DRAM round trip and its warps' merge; a CTA's share of the bandwidth is
// at most what its ~100 KB of copies in flight sustain, so a small batch still spreads its keys)
// Short contexts thus get one wave of whole-instance CTAs (no partials to merge); long, ragged
// contexts get a few waves of equal chunks so that no CTA runs long past the others.
int decode_plan_chunk(const int32_t* lengths, int B, int Hkv, int max_len, double row_bytes, int ctas_per_sm) {
  constexpr double T_FIX_US = 3.0;           // per-wave fixed cost
  constexpr double T_MERGE_US = 1.5;         // a split instance's partial write, counter and merge
  constexpr double BW = 6.5e6;               // bytes per microsecond (HBM)
  constexpr double CTA_BW = 1.0e5;           // bytes per microsecond one CTA sustains
  const double ROW = row_bytes;              // bytes per key and KV head (512: bf16 K + V, D = 128)
  const double slots = (double)ctas_per_sm * decode_num_sms();
  long long total = 0;
  for (int b = 0; b < B; ++b) total += lengths[b];
  const double total_bytes = (double)total * Hkv * ROW;
  int best_chunk = 0;
  double best_t = 1e300;
  int prev = -1;
  const int k_max = B > 4096 ? 1 : DECODE_MAX_CHUNKS;       // keep host planning cheap
  for (int k = 1; k <= k_max; ++k) {
    int chunk = (max_len + k - 1) / k;
    chunk = std::max(DECODE_CHUNK_ALIGN, (int)round_up((size_t)chunk, DECODE_CHUNK_ALIGN));
    if (chunk == prev) continue;
    prev = chunk;
    long long ctas = 0;
    for (int b = 0; b < B; ++b) ctas += (lengths[b] + chunk - 1) / chunk;
    ctas *= Hkv;
    const double waves = std::ceil((double)ctas / slots);
    const double share = std::min(CTA_BW, BW / std::min((double)ctas, slots));
    const double chunk_t = (double)chunk * ROW / share;  // one CTA's chunk at its bandwidth share
    double t = waves <= 1.0 ? T_FIX_US + std::max(total_bytes / BW, chunk_t)
                            : waves * T_FIX_US + total_bytes / BW + chunk_t;   // + tail of the last wave
    if (chunk < max_len) t += T_MERGE_US;      // partials written, counted and merged
    if (t < best_t - 1e-9) { best_t = t; best_chunk = chunk; }
  }
  const int floor_chunk = (max_len + DECODE_MAX_CHUNKS - 1) / DECODE_MAX_CHUNKS;
  return std::max(best_chunk, (int)round_up((size_t)std::max(floor_chunk, 1), DECODE_CHUNK_ALIGN));
}

}  // namespace kva

using namespace kva;

extern "C" {

const char* kva_strerror(kva_status s) {
  switch (s) {
    case KVA_OK: return "ok";
    case KVA_EINVAL: return "invalid argument";
    case KVA_ECAPACITY: return "slot or length beyond the cache capacity";
    case KVA_EUNSUPPORTED: return "unsupported configuration";
    case KVA_ECUDA: return "CUDA error";
    case KVA_EALIGN: return "misaligned pointer, stride or head_dim";
    case KVA_EWORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char* kva_last_error(void) { return g_msg; }

int64_t kva_wait_timeouts(int32_t reset) {
  int64_t total = 0;
  for (auto read : wait_counters()) {
    unsigned v = 0;
    if (read(&v, reset != 0) != cudaSuccess) return -1;
    total += v;
  }
  return total;
}

kva_status kva_selftest_wait_timeout(kva_stream stream) {
  selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>();
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return cuda_status(e, "self-test launch");
}
uint64_t kva_launch_count(void) { return g_launches.load(); }
int32_t kva_version(void) { return 100; }

size_t kva_decode_workspace_size(int32_t B, int32_t n_kv_heads, int32_t n_q_heads, int32_t max_len,
                                 int32_t head_dim) {
  if (B <= 0 || n_kv_heads <= 0 || n_q_heads <= 0 || max_len <= 0 || head_dim <= 0) return 0;
  return decode_ws_bytes(B, n_kv_heads, n_q_heads, decode_max_chunks_bound(max_len), head_dim);
}

size_t kva_decode_workspace_zero_bytes(int32_t B, int32_t n_kv_heads) {
  if (B <= 0 || n_kv_heads <= 0) return 0;
  return decode_zero_bytes(B, n_kv_heads);
}

size_t kva_lmhead_workspace_size(int32_t B, int32_t H) {
  if (B <= 0 || H <= 0) return 0;
  return lmhead_workspace_bytes(B, H);
}

size_t kva_lmhead_workspace_zero_bytes(int32_t B) {
  if (B <= 0) return 0;
  return lmhead_zero_bytes(B);
}

size_t kva_workspace_size(int32_t which, const kva_workspace_dims* d) {
  if (!d) return 0;
  switch (which) {
    case KVA_WS_DECODE: return kva_decode_workspace_size(d->B, d->n_kv_heads, d->n_q_heads, d->max_len, d->head_dim);
    case KVA_WS_VERIFY:
      return kva_verify_workspace_size(d->B, d->n_kv_heads, d->n_q_heads, d->block, d->max_len, d->head_dim);
    case KVA_WS_LMHEAD: return kva_lmhead_workspace_size(d->B, d->hidden);
    case KVA_WS_LMHEAD_TOPK: return kva_lmhead_topk_workspace_size(d->B, d->hidden, d->vocab, d->block);
  }
  return 0;
}

kva_status kv_cache_append_rope_qknorm(
    const void* q, const void* k, const void* v, kva_dtype in_dtype,
    int32_t N, int32_t T, int32_t n_q_heads,
    const int32_t* pos, int64_t pos_inst_stride,
    const int32_t* slot, int64_t slot_inst_stride, const int32_t* slot_host,
    kva_qknorm norm, kva_rope rope,
    void* q_out, kva_dtype q_out_dtype,
    kva_cache cache, kva_stream stream) {
  if (N < 0 || T < 0) return fail(KVA_EINVAL, "N=%d T=%d must be >= 0", N, T);
  if (N == 0 || T == 0) return KVA_OK;
  if (!valid_dtype(in_dtype) || !valid_dtype(q_out_dtype)) return fail(KVA_EINVAL, "unknown dtype");
  kva_status st = check_cache(cache, N);
  if (st != KVA_OK) return st;
  const int D = cache.head_dim, Hkv = cache.n_kv_heads;
  if (n_q_heads <= 0 || n_q_heads % Hkv != 0)
    return fail(KVA_EINVAL, "n_q_heads %d must be a positive multiple of n_kv_heads %d", n_q_heads, Hkv);
  if (!q || !k || !v || !q_out || !slot || !slot_host) return fail(KVA_EINVAL, "NULL q/k/v/q_out/slot");
  if (rope.kind != KVA_ROPE_NONE && !pos) return fail(KVA_EINVAL, "RoPE needs positions");
  if (pos_inst_stride < 0 || slot_inst_stride < 0) return fail(KVA_EINVAL, "negative instance stride");
  if ((norm.q_w == nullptr) != (norm.k_w == nullptr))
    return fail(KVA_EINVAL, "q and k norm weights must both be given or both be NULL");
  if (norm.q_w && (!(norm.eps >= 0.f) || norm.inst_stride < 0))
    return fail(KVA_EINVAL, "QK-Norm eps must be >= 0 and inst_stride >= 0");
  int rot_off = 0, rot_w = D;
  if (rope.kind != KVA_ROPE_NONE) {
    st = rope_range(rope, D, &rot_off, &rot_w);
    if (st != KVA_OK) return st;
  }
  // the fast forms take symmetric heads they tile, with RoPE over the whole head
  const bool fast = !asymmetric(cache) && rot_off == 0 && rot_w == D && append_supports_head_dim(D) &&
                    !(rope.kind == KVA_ROPE_INTERLEAVED && D % 16 != 0);
  if (!fast && !append_general_supports(D, cache.head_dim_v))
    return fail(KVA_EUNSUPPORTED, "append: head dims %d/%d not built (multiples of 8 up to 256)", D,
                cache.head_dim_v);
  if (N > 65535) return fail(KVA_EUNSUPPORTED, "append: N=%d > 65535", N);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_out))
    return fail(KVA_EALIGN, "q/k/v/q_out must be 16-byte aligned");
  if (norm.q_w && (!aligned16(norm.q_w) || !aligned16(norm.k_w) || (norm.inst_stride * 4) % 16 != 0))
    return fail(KVA_EALIGN, "norm weights must be 16-byte aligned with a 16-byte instance stride");

  AppendArgs a{};
  st = build_rope_table(rope, rot_w, &a.rope);
  if (st != KVA_OK) return st;
  for (int n = 0; n < N; ++n)
    for (int t = 0; t < T; ++t) {
      const int32_t s = slot_host[(int64_t)n * slot_inst_stride + t];
      if (s < 0 || s >= cache.capacity)
        return fail(KVA_ECAPACITY, "slot %d of instance %d token %d outside [0, %d)", s, n, t,
                    cache.capacity);
    }
  a.q = q; a.k = k; a.v = v; a.q_out = q_out; a.kc = cache.k; a.vc = cache.v;
  a.pos = pos; a.pos_stride = pos_inst_stride; a.slot = slot; a.slot_stride = slot_inst_stride;
  a.q_w = norm.q_w; a.k_w = norm.k_w; a.w_stride = norm.inst_stride; a.eps = norm.eps;
  a.after_rope = norm.after_rope ? 1 : 0;
  a.N = N; a.T = T; a.Hq = n_q_heads; a.Hkv = Hkv; a.D = D; a.capacity = cache.capacity;
  a.inst_stride = cache.inst_stride;
  a.Dv = cache.head_dim_v; a.inst_stride_v = cache.inst_stride_v;
  a.rot_offset = rot_off; a.rot_dim = rot_w;
  cudaError_t e = fast ? launch_append(a, in_dtype, q_out_dtype, cache.dtype, (cudaStream_t)stream)
                       : launch_append_general(a, in_dtype, q_out_dtype, cache.dtype, (cudaStream_t)stream);
  if (e == cudaSuccess) count_launches(1);
  return cuda_status(e, "append launch");
}

kva_status kv_attn_prefill(
    const void* q, kva_dtype q_dtype, kva_cache cache,
    int32_t N, int32_t S, int32_t n_q_heads, kva_mask mask,
    const int32_t* segment, const int32_t* segment_host,
    const int32_t* row_of_slot,
    float scale, float* out, kva_stream stream) {
  if (N < 0 || S < 0) return fail(KVA_EINVAL, "N=%d S=%d must be >= 0", N, S);
  if (N == 0 || S == 0) return KVA_OK;
  kva_status st = check_cache(cache, N);
  if (st != KVA_OK) return st;
  if (q_dtype != cache.dtype) return fail(KVA_EINVAL, "prefill: q dtype must equal the cache dtype");
  const int D = cache.head_dim, Hkv = cache.n_kv_heads;
  if (n_q_heads <= 0 || n_q_heads % Hkv != 0)
    return fail(KVA_EINVAL, "n_q_heads %d must be a positive multiple of n_kv_heads %d", n_q_heads, Hkv);
  if (!q || !out) return fail(KVA_EINVAL, "NULL q/out");
  if (S > cache.capacity) return fail(KVA_ECAPACITY, "prefill S=%d > capacity %d", S, cache.capacity);
  if (mask != KVA_MASK_CAUSAL && mask != KVA_MASK_FULL && mask != KVA_MASK_SEGMENT && mask != KVA_MASK_CAUSAL_SEGMENT)
    return fail(KVA_EINVAL, "mask %d unknown", (int)mask);
  if (mask == KVA_MASK_SEGMENT || mask == KVA_MASK_CAUSAL_SEGMENT) {
    if (!segment || !segment_host) return fail(KVA_EINVAL, "segment mask needs segment ids");
    for (int i = 1; i < S; ++i)
      if (segment_host[i] < segment_host[i - 1])
        return fail(KVA_EINVAL, "segment ids must be non-decreasing (slot %d)", i);
  }
  if (!aligned16(q) || !aligned16(out)) return fail(KVA_EALIGN, "q/out must be 16-byte aligned");
  if (N > 65535 || n_q_heads > 65535) return fail(KVA_EUNSUPPORTED, "prefill: N or Hq > 65535");
  PrefillArgs a{};
  a.q = q; a.kc = cache.k; a.vc = cache.v;
  a.segment = (mask == KVA_MASK_SEGMENT || mask == KVA_MASK_CAUSAL_SEGMENT) ? segment : nullptr;
  a.row_of_slot = row_of_slot; a.out = out;
  a.N = N; a.S = S; a.Hq = n_q_heads; a.Hkv = Hkv; a.D = D; a.capacity = cache.capacity;
  a.mask = (int)mask; a.inst_stride = cache.inst_stride;
  a.Dv = cache.head_dim_v; a.inst_stride_v = cache.inst_stride_v;
  a.seg_table = 0;
  if (a.segment && segment_host[0] >= 0 && segment_host[S - 1] < PREFILL_SEG_TABLE) {
    // ids are non-decreasing (checked above): each id's slots are one contiguous run
    for (int g = 0; g <= segment_host[S - 1]; ++g) a.seg_lo[g] = a.seg_hi[g] = 0;
    for (int i = 0; i < S; ++i) {
      const int g = segment_host[i];
      if (i == 0 || segment_host[i - 1] != g) a.seg_lo[g] = i;
      a.seg_hi[g] = i + 1;
    }
    a.seg_table = segment_host[S - 1] + 1;
  }
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
  a.scale_log2 = sc * 1.4426950408889634f;
  cudaError_t e;
  if (prefill_tc_supports(D, cache.head_dim_v, cache.dtype)) {
    e = launch_prefill_tc(a, (cudaStream_t)stream);
  } else if (prefill_simt_supports(D, cache.head_dim_v)) {
    e = launch_prefill_simt(a, cache.dtype, (cudaStream_t)stream);
  } else {
    return fail(KVA_EUNSUPPORTED, "prefill: head dims %d/%d not built", D, cache.head_dim_v);
  }
  if (e == cudaSuccess) count_launches(1);
  return cuda_status(e, "prefill launch");
}

kva_status kv_attn_decode(
    const void* q, kva_dtype q_dtype, kva_cache cache,
    const int32_t* lengths, const int32_t* lengths_host, int32_t B, int32_t n_q_heads,
    float scale, float* out, void* workspace, size_t workspace_bytes, kva_stream stream) {
  if (B < 0) return fail(KVA_EINVAL, "B=%d must be >= 0", B);
  if (B == 0) return KVA_OK;
  if (!valid_dtype(q_dtype)) return fail(KVA_EINVAL, "unknown q dtype");
  kva_status st = check_cache(cache, B);
  if (st != KVA_OK) return st;
  const int D = cache.head_dim, Hkv = cache.n_kv_heads;
  if (n_q_heads <= 0 || n_q_heads % Hkv != 0)
    return fail(KVA_EINVAL, "n_q_heads %d must be a positive multiple of n_kv_heads %d", n_q_heads, Hkv);
  const int Dv = cache.head_dim_v;
  const bool asym = asymmetric(cache);
  if (asym ? !decode_asym_supported(D, Dv) : D != DECODE_HEAD_DIM)
    return fail(KVA_EUNSUPPORTED, "decode: head dims %d/%d (built: 128/128, 192/128)", D, Dv);
  const int G = n_q_heads / Hkv;
  if (G != 1 && G != 2 && G != 4) return fail(KVA_EUNSUPPORTED, "decode: group size %d", G);
  if (!q || !out || !lengths || !lengths_host) return fail(KVA_EINVAL, "NULL q/out/lengths");
  if (!workspace) return fail(KVA_EWORKSPACE, "decode: workspace is NULL");
  if (!aligned16(workspace)) return fail(KVA_EALIGN, "workspace must be 16-byte aligned");
  if (B > 65535 || Hkv > 65535) return fail(KVA_EUNSUPPORTED, "decode: B or Hkv > 65535");
  int max_len = 0;
  for (int b = 0; b < B; ++b) {
    const int L = lengths_host[b];
    if (L < 1 || L > cache.capacity)
      return fail(KVA_ECAPACITY, "length %d of instance %d outside [1, %d]", L, b, cache.capacity);
    max_len = std::max(max_len, L);
  }
  const int chunk = decode_plan_chunk(lengths_host, B, Hkv, max_len, (double)(D + Dv) * elem_size(cache.dtype),
                                      asym ? 1 : 2);
  const int max_chunks = (max_len + chunk - 1) / chunk;
  const size_t need = decode_ws_bytes(B, Hkv, n_q_heads, max_chunks, Dv);
  if (workspace_bytes < need)
    return fail(KVA_EWORKSPACE, "decode workspace %zu bytes < %zu needed", workspace_bytes, need);

  DecodeArgs a{};
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.counters = reinterpret_cast<unsigned*>(ws);
  a.part_ml = reinterpret_cast<float*>(ws + decode_zero_bytes(B, Hkv));
  a.part_acc = reinterpret_cast<float*>(ws + decode_zero_bytes(B, Hkv) +
                                        round_up(sizeof(float) * (size_t)B * n_q_heads * max_chunks * 2, 256));
  a.q = q; a.kc = cache.k; a.vc = cache.v; a.lengths = lengths; a.out = out;
  a.B = B; a.Hq = n_q_heads; a.Hkv = Hkv; a.capacity = cache.capacity;
  a.chunk = chunk; a.max_chunks = max_chunks; a.inst_stride = cache.inst_stride;
  a.inst_stride_v = cache.inst_stride_v;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
  a.scale_log2 = sc * 1.4426950408889634f;
  cudaError_t e = asym ? launch_decode_asym(a, D, Dv, q_dtype, cache.dtype, (cudaStream_t)stream)
                       : launch_decode(a, q_dtype, cache.dtype, (cudaStream_t)stream);
  if (e == cudaSuccess) count_launches(1);
  return cuda_status(e, "decode launch");
}

kva_status kv_attn_decode_step(
    const void* q, const void* k, const void* v, kva_dtype in_dtype,
    const int32_t* pos, int64_t pos_inst_stride,
    kva_qknorm norm, kva_rope rope, kva_cache cache,
    const int32_t* lengths, const int32_t* lengths_host, int32_t B, int32_t n_q_heads,
    float scale, void* q_out, kva_dtype q_out_dtype, float* out,
    void* workspace, size_t workspace_bytes, kva_stream stream) {
  if (B < 0) return fail(KVA_EINVAL, "B=%d must be >= 0", B);
  if (B == 0) return KVA_OK;
  if (!valid_dtype(in_dtype) || (q_out && !valid_dtype(q_out_dtype))) return fail(KVA_EINVAL, "unknown dtype");
  kva_status st = check_cache(cache, B);
  if (st != KVA_OK) return st;
  const int D = cache.head_dim, Hkv = cache.n_kv_heads;
  if (n_q_heads <= 0 || n_q_heads % Hkv != 0)
    return fail(KVA_EINVAL, "n_q_heads %d must be a positive multiple of n_kv_heads %d", n_q_heads, Hkv);
  if (!q || !k || !v || !out || !lengths || !lengths_host) return fail(KVA_EINVAL, "NULL q/k/v/out/lengths");
  if (rope.kind != KVA_ROPE_NONE && !pos) return fail(KVA_EINVAL, "RoPE needs positions");
  if (pos_inst_stride < 0) return fail(KVA_EINVAL, "negative position stride");
  if ((norm.q_w == nullptr) != (norm.k_w == nullptr))
    return fail(KVA_EINVAL, "q and k norm weights must both be given or both be NULL");
  if (norm.q_w && (!(norm.eps >= 0.f) || norm.inst_stride < 0)) return fail(KVA_EINVAL, "bad QK-Norm eps/stride");
  const int G = n_q_heads / Hkv;
  const int Dv = cache.head_dim_v;
  int rot_off = 0, rot_w = D;
  st = rope_range(rope, D, &rot_off, &rot_w);
  if (st != KVA_OK) return st;
  const bool whole_head = rope.kind == KVA_ROPE_NONE || (rot_off == 0 && rot_w == D);
  // tensor-core form: bf16 symmetric D = 128 with whole-head RoPE; CUDA-core form: fp32 caches,
  // the asymmetric 192/128 cache and rotary sub-ranges
  const bool mma_form = cache.dtype == KVA_BF16 && D == DECODE_HEAD_DIM && !asymmetric(cache) &&
                        decode_step_supported(G) && whole_head && decode_mma_supported();
  if (!mma_form && !decode_step_simt_supported(D, Dv, G))
    return fail(KVA_EUNSUPPORTED, "fused step: head dims %d/%d with Hq/Hkv %d (built: 128/128 and 192/128, "
                "Hq/Hkv in {1,2,4})", D, Dv, G);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (q_out && !aligned16(q_out)))
    return fail(KVA_EALIGN, "q/k/v/out/q_out must be 16-byte aligned");
  if (norm.q_w && (!aligned16(norm.q_w) || !aligned16(norm.k_w) || (norm.inst_stride * 4) % 16 != 0))
    return fail(KVA_EALIGN, "norm weights must be 16-byte aligned with a 16-byte instance stride");
  if (!workspace) return fail(KVA_EWORKSPACE, "decode step: workspace is NULL");
  if (!aligned16(workspace)) return fail(KVA_EALIGN, "workspace must be 16-byte aligned");
  if (B > 65535) return fail(KVA_EUNSUPPORTED, "decode step: B > 65535");
  StepArgs sa{};
  st = build_rope_table(rope, rot_w, &sa.rope);
  if (st != KVA_OK) return st;
  sa.rot_offset = rot_off;
  sa.rot_dim = rot_w;
  int max_len = 0;
  for (int b = 0; b < B; ++b) {
    const int L = lengths_host[b];
    if (L < 1 || L > cache.capacity)
      return fail(KVA_ECAPACITY, "length %d of instance %d outside [1, %d]", L, b, cache.capacity);
    max_len = std::max(max_len, L);
  }
  const int chunk = mma_form ? decode_plan_chunk(lengths_host, B, Hkv, max_len)
                             : decode_plan_chunk(lengths_host, B, Hkv, max_len, (double)(D + Dv) * elem_size(cache.dtype),
                                                 asymmetric(cache) ? 1 : 2);
  const int max_chunks = (max_len + chunk - 1) / chunk;
  const size_t need = decode_ws_bytes(B, Hkv, n_q_heads, max_chunks, Dv);
  if (workspace_bytes < need)
    return fail(KVA_EWORKSPACE, "decode step workspace %zu bytes < %zu needed", workspace_bytes, need);
  DecodeArgs a{};
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.counters = reinterpret_cast<unsigned*>(ws);
  a.part_ml = reinterpret_cast<float*>(ws + decode_zero_bytes(B, Hkv));
  a.part_acc = reinterpret_cast<float*>(ws + decode_zero_bytes(B, Hkv) +
                                        round_up(sizeof(float) * (size_t)B * n_q_heads * max_chunks * 2, 256));
  a.q = nullptr; a.kc = cache.k; a.vc = cache.v; a.lengths = lengths; a.out = out;
  a.B = B; a.Hq = n_q_heads; a.Hkv = Hkv; a.capacity = cache.capacity;
  a.chunk = chunk; a.max_chunks = max_chunks; a.inst_stride = cache.inst_stride;
  a.inst_stride_v = cache.inst_stride_v;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
  a.scale_log2 = sc * 1.4426950408889634f;
  sa.q = q; sa.k = k; sa.v = v; sa.in_dtype = (int)in_dtype;
  sa.pos = pos; sa.pos_stride = pos_inst_stride;
  sa.q_w = norm.q_w; sa.k_w = norm.k_w; sa.w_stride = norm.inst_stride; sa.eps = norm.eps;
  sa.after_rope = norm.after_rope ? 1 : 0;
  sa.q_out = q_out; sa.q_out_dtype = (int)q_out_dtype;
  cudaError_t e = mma_form ? launch_decode_step(a, sa, (cudaStream_t)stream)
                           : launch_decode_step_simt(a, sa, D, cache.dtype, (cudaStream_t)stream);
  if (e == cudaSuccess) count_launches(1);
  return cuda_status(e, "decode step launch");
}

static int verify_row_tiles(int G, int k) { return (G * k + 15) / 16; }

size_t kva_verify_workspace_size(int32_t B, int32_t n_kv_heads, int32_t n_q_heads, int32_t k, int32_t max_len,
                                 int32_t head_dim) {
  if (B <= 0 || n_kv_heads <= 0 || n_q_heads <= 0 || k <= 0 || max_len <= 0 || head_dim <= 0 ||
      n_q_heads % n_kv_heads != 0)
    return 0;
  const int RT = verify_row_tiles(n_q_heads / n_kv_heads, k);
  return decode_ws_bytes(B, n_kv_heads * RT, n_kv_heads * RT * 16, decode_max_chunks_bound(max_len), head_dim);
}

kva_status kv_attn_verify(
    const void* q, kva_dtype q_dtype, kva_cache cache,
    const int32_t* lengths, const int32_t* lengths_host, int32_t B, int32_t k, int32_t n_q_heads,
    float scale, float* out, void* workspace, size_t workspace_bytes, kva_stream stream) {
  if (B < 0) return fail(KVA_EINVAL, "B=%d must be >= 0", B);
  if (B == 0) return KVA_OK;
  if (k < 1 || k > KVA_VERIFY_MAX_BLOCK) return fail(KVA_EINVAL, "block size k=%d outside [1, %d]", k, KVA_VERIFY_MAX_BLOCK);
  if (!valid_dtype(q_dtype)) return fail(KVA_EINVAL, "unknown q dtype");
  kva_status st = check_cache(cache, B);
  if (st != KVA_OK) return st;
  const int D = cache.head_dim, Hkv = cache.n_kv_heads;
  if (n_q_heads <= 0 || n_q_heads % Hkv != 0)
    return fail(KVA_EINVAL, "n_q_heads %d must be a positive multiple of n_kv_heads %d", n_q_heads, Hkv);
  if (!q || !out || !lengths || !lengths_host) return fail(KVA_EINVAL, "NULL q/out/lengths");
  if (cache.dtype != KVA_BF16 || D != DECODE_HEAD_DIM || asymmetric(cache))
    return fail(KVA_EUNSUPPORTED, "verify: needs a symmetric bf16 cache with head_dim 128");
  if (!workspace) return fail(KVA_EWORKSPACE, "verify: workspace is NULL");
  if (!aligned16(workspace)) return fail(KVA_EALIGN, "workspace must be 16-byte aligned");
  const int G = n_q_heads / Hkv, RT = verify_row_tiles(G, k);
  if (B > 65535 || Hkv * RT > 65535) return fail(KVA_EUNSUPPORTED, "verify: B or Hkv * row tiles > 65535");
  int max_len = 0;
  for (int b = 0; b < B; ++b) {
    const int L = lengths_host[b];
    if (L < k || L > cache.capacity)
      return fail(KVA_ECAPACITY, "length %d of instance %d outside [k=%d, %d]", L, b, k, cache.capacity);
    max_len = std::max(max_len, L);
  }
  // the tcgen05 form reads q and writes out with 16-byte accesses
  const bool tc_form = verify_tc_supports(G, k) && aligned16(q) && aligned16(out);
  const int chunk = tc_form ? verify_tc_plan_chunk(lengths_host, B, Hkv, max_len)
                            : decode_plan_chunk(lengths_host, B, Hkv * RT, max_len);
  const int max_chunks = (max_len + chunk - 1) / chunk;
  const size_t need = decode_ws_bytes(B, Hkv * RT, Hkv * RT * 16, max_chunks, D);
  if (workspace_bytes < need)
    return fail(KVA_EWORKSPACE, "verify workspace %zu bytes < %zu needed", workspace_bytes, need);
  VerifyArgs a{};
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const size_t zero = decode_zero_bytes(B, Hkv * RT);
  a.counters = reinterpret_cast<unsigned*>(ws);
  a.part_ml = reinterpret_cast<float*>(ws + zero);
  a.part_acc = reinterpret_cast<float*>(ws + zero + round_up(sizeof(float) * (size_t)B * Hkv * RT * 16 * max_chunks * 2, 256));
  a.q = q; a.kc = cache.k; a.vc = cache.v; a.lengths = lengths; a.out = out;
  a.B = B; a.k = k; a.Hq = n_q_heads; a.Hkv = Hkv; a.RT = RT; a.capacity = cache.capacity;
  a.chunk = chunk; a.max_chunks = max_chunks; a.inst_stride = cache.inst_stride;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
  a.scale_log2 = sc * 1.4426950408889634f;
  cudaError_t e = tc_form ? launch_verify_tc(a, q_dtype, (cudaStream_t)stream)
                          : launch_verify(a, q_dtype, (cudaStream_t)stream);
  if (e == cudaSuccess) count_launches(1);
  return cuda_status(e, "verify launch");
}

kva_status kv_verify_commit(const int32_t* posterior, const int32_t* block_tokens, int32_t B, int32_t k,
                            int32_t* lengths, int32_t* accepted, int32_t* next_token, kva_stream stream) {
  if (B < 0 || k < 1) return fail(KVA_EINVAL, "B=%d must be >= 0 and k=%d >= 1", B, k);
  if (B == 0) return KVA_OK;
  if (!posterior || !block_tokens || !lengths || !accepted || !next_token)
    return fail(KVA_EINVAL, "NULL posterior/block_tokens/lengths/accepted/next_token");
  cudaError_t e = launch_verify_commit(posterior, block_tokens, B, k, lengths, accepted, next_token, (cudaStream_t)stream);
  if (e == cudaSuccess) count_launches(1);
  return cuda_status(e, "verify commit launch");
}

kva_status lmhead_argmax(
    const float* h, const void* W, kva_dtype w_dtype,
    int32_t B, int32_t H, int32_t V, int32_t V_rows,
    int32_t* out_ids, float* out_max, float* logits,
    void* workspace, size_t workspace_bytes, kva_stream stream) {
  if (B < 0) return fail(KVA_EINVAL, "B=%d must be >= 0", B);
  if (B == 0) return KVA_OK;
  if (!valid_dtype(w_dtype)) return fail(KVA_EINVAL, "unknown weight dtype");
  if (H <= 0 || V <= 0 || V_rows <= 0) return fail(KVA_EINVAL, "H, V, V_rows must be positive");
  if (V > V_rows) return fail(KVA_EINVAL, "vocab V=%d exceeds the table's %d rows", V, V_rows);
  if (H % 8 != 0) return fail(KVA_EALIGN, "hidden %d is not a multiple of 8", H);
  if (H > lmhead_max_hidden()) return fail(KVA_EUNSUPPORTED, "hidden %d > %d", H, lmhead_max_hidden());
  if (!h || !W || !out_ids) return fail(KVA_EINVAL, "NULL h/W/out_ids");
  if (!aligned16(h) || !aligned16(W)) return fail(KVA_EALIGN, "h and W must be 16-byte aligned");
  if (!workspace) return fail(KVA_EWORKSPACE, "lm_head: workspace is NULL");
  if (!aligned16(workspace)) return fail(KVA_EALIGN, "workspace must be 16-byte aligned");
  if (workspace_bytes < lmhead_workspace_bytes(B, H))
    return fail(KVA_EWORKSPACE, "lm_head workspace %zu bytes < %zu needed", workspace_bytes,
                lmhead_workspace_bytes(B, H));
  if (B > 65535 * 8) return fail(KVA_EUNSUPPORTED, "lm_head: batch too large");
  LmheadArgs a{};
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.counter = reinterpret_cast<unsigned*>(ws);
  a.best = reinterpret_cast<unsigned long long*>(ws + 256);   // see lmhead_zero_bytes
  a.h = h; a.W = W; a.out_ids = out_ids; a.out_max = out_max; a.logits = logits;
  a.B = B; a.H = H; a.V = V;
  unsigned n_launch = 0;
  cudaError_t e = launch_lmhead(a, w_dtype, ws + lmhead_zero_bytes(B), (cudaStream_t)stream, &n_launch);
  if (e == cudaSuccess) count_launches(n_launch);
  return cuda_status(e, "lm_head launch");
}

size_t kva_lmhead_topk_workspace_size(int32_t B, int32_t H, int32_t V, int32_t top_k) {
  if (B <= 0 || H <= 0 || V <= 0 || top_k <= 0) return 0;
  size_t n = lmhead_workspace_bytes(B, H);
  if (top_k > 1)
    n += round_up(sizeof(float) * (size_t)B * V, 256) + round_up(sizeof(int32_t) * (size_t)B, 256) +
         round_up(topk_rows_workspace_bytes(B, V), 256);
  return n;
}

kva_status lmhead_topk(
    const float* h, const float* norm_w, float eps, const void* W, kva_dtype w_dtype,
    int32_t B, int32_t H, int32_t V, int32_t V_rows, int32_t top_k,
    int32_t* out_ids, float* out_vals, void* workspace, size_t workspace_bytes, kva_stream stream) {
  if (B < 0) return fail(KVA_EINVAL, "B=%d must be >= 0", B);
  if (B == 0) return KVA_OK;
  if (top_k < 1 || top_k > LMHEAD_TOPK_MAX) return fail(KVA_EINVAL, "top_k=%d outside [1, %d]", top_k, LMHEAD_TOPK_MAX);
  if (!valid_dtype(w_dtype)) return fail(KVA_EINVAL, "unknown weight dtype");
  if (H <= 0 || V <= 0 || V_rows <= 0) return fail(KVA_EINVAL, "H, V, V_rows must be positive");
  if (V > V_rows) return fail(KVA_EINVAL, "vocab V=%d exceeds the table's %d rows", V, V_rows);
  if (top_k > V) return fail(KVA_EINVAL, "top_k=%d exceeds the vocab %d", top_k, V);
  if (norm_w && !(eps >= 0.f)) return fail(KVA_EINVAL, "final-norm eps must be >= 0");
  if (H % 8 != 0) return fail(KVA_EALIGN, "hidden %d is not a multiple of 8", H);
  if (H > lmhead_max_hidden()) return fail(KVA_EUNSUPPORTED, "hidden %d > %d", H, lmhead_max_hidden());
  if (!h || !W || !out_ids) return fail(KVA_EINVAL, "NULL h/W/out_ids");
  if (!aligned16(h) || !aligned16(W) || (norm_w && !aligned16(norm_w)))
    return fail(KVA_EALIGN, "h, W and norm_w must be 16-byte aligned");
  if (!workspace) return fail(KVA_EWORKSPACE, "lm_head: workspace is NULL");
  if (!aligned16(workspace)) return fail(KVA_EALIGN, "workspace must be 16-byte aligned");
  const size_t need = kva_lmhead_topk_workspace_size(B, H, V, top_k);
  if (workspace_bytes < need) return fail(KVA_EWORKSPACE, "lm_head top-k workspace %zu bytes < %zu needed", workspace_bytes, need);
  if (B > 65535) return fail(KVA_EUNSUPPORTED, "lm_head top-k: batch too large");
  LmheadArgs a{};
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.counter = reinterpret_cast<unsigned*>(ws);
  a.best = reinterpret_cast<unsigned long long*>(ws + 256);   // see lmhead_zero_bytes
  a.h = h; a.W = W; a.B = B; a.H = H; a.V = V;
  a.norm_w = norm_w; a.eps = eps;
  float* logits = nullptr;
  if (top_k == 1) {                                   // the greedy id: the fused argmax
    a.out_ids = out_ids; a.out_max = out_vals;
  } else {                                            // logits to the workspace, then a row top-k
    unsigned char* extra = ws + lmhead_workspace_bytes(B, H);
    logits = reinterpret_cast<float*>(extra);
    a.logits = logits;
    a.out_ids = reinterpret_cast<int32_t*>(extra + round_up(sizeof(float) * (size_t)B * V, 256));
  }
  unsigned n_launch = 0;
  cudaError_t e = launch_lmhead(a, w_dtype, ws + lmhead_zero_bytes(B), (cudaStream_t)stream, &n_launch);
  if (e == cudaSuccess && top_k > 1) {
    unsigned char* rank_ws = ws + lmhead_workspace_bytes(B, H) + round_up(sizeof(float) * (size_t)B * V, 256) +
                             round_up(sizeof(int32_t) * (size_t)B, 256);
    e = launch_topk_rows(logits, B, V, top_k, rank_ws, out_ids, out_vals, (cudaStream_t)stream);
    ++n_launch;
  }
  if (e == cudaSuccess) count_launches(n_launch);
  return cuda_status(e, "lm_head top-k launch");
}

}  // extern "C"
