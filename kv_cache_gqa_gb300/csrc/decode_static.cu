// Decode attention for callers that cannot allocate device memory.
//
// kv_attn_decode needs a caller-provided workspace for its split-KV partials and merge
// counters.  Some callers have no way to obtain one: code running where cudaMalloc is
// forbidden or unavailable (a plugin whose host framework owns every device allocation, or
// a latency-critical loop that must never touch the allocator).  kv_attn_decode_static serves them: it runs the same decode kernel
// with its scratch taken from a fixed-size array that lives in this library's device image,
// so the call itself allocates nothing.
//
// The array below lives in device memory, one copy per GPU that loads the library.  Host
// code can name it only through its host-side shadow symbol, which is not a device address:
// the device address is looked up once per device with cudaGetSymbolAddress (the first call
// on that device does it, with that device current) and that address is what the kernel
// receives.  The looked-up addresses are kept for the life of the process, so the library
// must not be used across a cudaDeviceReset.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "kv_attn.h"
#include "launch.h"

namespace kva {

constexpr size_t STATIC_SCRATCH_BYTES = 4u << 20;   // 4 MiB, held by every GPU that loads the library

static __device__ __align__(256) unsigned char g_decode_scratch[STATIC_SCRATCH_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[MAX_DEVICES] = {};

kva_status static_fail(kva_status st, const char* msg) {
  set_last_error(msg);   // readable through kva_last_error()
  return st;
}

// Device address of the scratch array on the current device (set up on first use).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

size_t round_up_s(size_t x, size_t m) { return (x + m - 1) / m * m; }

}  // namespace

}  // namespace kva

using namespace kva;

extern "C" {

kva_status kv_attn_decode_static(
    const void* q, kva_dtype q_dtype, kva_cache cache,
    const int32_t* lengths, const int32_t* lengths_host, int32_t B, int32_t n_q_heads,
    float scale, float* out, kva_stream stream) {
  if (B < 0) return static_fail(KVA_EINVAL, "B must be >= 0");
  if (B == 0) return KVA_OK;
  if (q_dtype != KVA_F32 && q_dtype != KVA_BF16) return static_fail(KVA_EINVAL, "unknown q dtype");
  if (cache.dtype != KVA_F32 && cache.dtype != KVA_BF16) return static_fail(KVA_EINVAL, "unknown cache dtype");
  if (!cache.k || !cache.v || !q || !out || !lengths || !lengths_host)
    return static_fail(KVA_EINVAL, "NULL q/out/lengths/cache pointer");
  const int D = cache.head_dim, Hkv = cache.n_kv_heads;
  if (Hkv <= 0 || cache.capacity <= 0 || n_q_heads <= 0 || n_q_heads % Hkv != 0)
    return static_fail(KVA_EINVAL, "bad head counts or capacity");
  const int64_t inst = (int64_t)Hkv * cache.capacity * D;
  if (B > 1 && cache.inst_stride < inst) return static_fail(KVA_EINVAL, "cache inst_stride too small");
  if (D != DECODE_HEAD_DIM) return static_fail(KVA_EUNSUPPORTED, "decode is built for head_dim 128");
  if ((cache.head_dim_v != 0 && cache.head_dim_v != D) || (cache.inst_stride_v != 0 && cache.inst_stride_v != cache.inst_stride))
    return static_fail(KVA_EUNSUPPORTED, "the static decode takes symmetric caches only");
  const int G = n_q_heads / Hkv;
  if (G != 1 && G != 2 && G != 4) return static_fail(KVA_EUNSUPPORTED, "decode group size must be 1, 2 or 4");
  const int es = cache.dtype == KVA_BF16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(cache.k) | reinterpret_cast<uintptr_t>(cache.v) |
       reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15u ||
      (cache.inst_stride * es) % 16 != 0)
    return static_fail(KVA_EALIGN, "pointers and the instance stride must be 16-byte aligned");
  if (B > 65535) return static_fail(KVA_EUNSUPPORTED, "B > 65535");
  int max_len = 0;
  for (int b = 0; b < B; ++b) {
    const int L = lengths_host[b];
    if (L < 1 || L > cache.capacity) return static_fail(KVA_ECAPACITY, "a length is outside [1, capacity]");
    max_len = std::max(max_len, L);
  }

  // Scratch layout: merge counters (cleared by every call), then (max, sum) and acc partials.
  const size_t zero_bytes = round_up_s(sizeof(unsigned) * (size_t)B * Hkv, 256);
  const size_t per_chunk = (size_t)B * n_q_heads * (2 + D) * sizeof(float);
  if (zero_bytes + 256 + per_chunk > STATIC_SCRATCH_BYTES)
    return static_fail(KVA_EWORKSPACE, "B * n_q_heads too large for the fixed 4 MiB decode scratch");
  const int fit_chunks = (int)std::min<size_t>(64, (STATIC_SCRATCH_BYTES - zero_bytes - 256) / per_chunk);
  // Same split rule as kv_attn_decode, then widened until the partials fit in the fixed scratch.
  long long chunk = decode_plan_chunk(lengths_host, B, Hkv, max_len, (double)(2 * D) * es, 2);
  chunk = std::max<long long>(chunk, (max_len + fit_chunks - 1) / fit_chunks);
  chunk = std::max<long long>(64, (chunk + 63) / 64 * 64);
  const int max_chunks = (int)((max_len + chunk - 1) / chunk);

  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return static_fail(KVA_ECUDA, "cudaGetSymbolAddress of the decode scratch failed");
  unsigned char* ws = static_cast<unsigned char*>(base);
  e = cudaMemsetAsync(ws, 0, zero_bytes, (cudaStream_t)stream);   // counters start at zero
  if (e != cudaSuccess) return static_fail(KVA_ECUDA, "clearing the decode scratch counters failed");

  DecodeArgs a{};
  a.counters = reinterpret_cast<unsigned*>(ws);
  a.part_ml = reinterpret_cast<float*>(ws + zero_bytes);
  a.part_acc = reinterpret_cast<float*>(
      ws + zero_bytes + round_up_s(sizeof(float) * (size_t)B * n_q_heads * max_chunks * 2, 256));
  a.q = q; a.kc = cache.k; a.vc = cache.v; a.lengths = lengths; a.out = out;
  a.B = B; a.Hq = n_q_heads; a.Hkv = Hkv; a.capacity = cache.capacity;
  a.chunk = (int)chunk; a.max_chunks = max_chunks; a.inst_stride = cache.inst_stride;
  a.inst_stride_v = cache.inst_stride;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt((float)D);
  a.scale_log2 = sc * 1.4426950408889634f;
  e = launch_decode(a, q_dtype, cache.dtype, (cudaStream_t)stream);
  if (e != cudaSuccess) return static_fail(KVA_ECUDA, cudaGetErrorString(e));
  count_launches(1);
  return KVA_OK;
}

}  // extern "C"
