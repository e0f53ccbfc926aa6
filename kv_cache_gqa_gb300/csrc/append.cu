// Kernel (a): QK-Norm + RoPE fused into the K/V cache write.
//
// One CTA per (token t, instance n).  The CTA first evaluates the token's D/2 rotary
// angles once (shared by its Hq + Hkv rotated rows), then its warps stream the
// Hq q rows, Hkv k rows and Hkv v rows: each row is split over D/8 lanes that own
// 8 consecutive elements, so every global load and store is a 128-bit access and a
// row is one contiguous, coalesced segment.
//
// Method: per-head RMSNorm over head_dim (Penguin-VL ncnn port, sections 2.1 and 4.2);
// rotate-half RoPE x*cos + rotate_half(x)*sin (Youtu-VL-4B ncnn port, implementation
// difficulty 2) in 1D, xdRoPE-section (HunyuanOCR v1.0 ncnn port, section five) or
// 2D-halves form (Penguin-VL ncnn port, section 2.3); k/v written into the new token's
// cache slot by the runtime (Youtu-VL-4B ncnn port, step 6), k normalised before the
// write when the norm follows RoPE (HunyuanOCR v1.0 ncnn port, section five item 2).
#include "common.cuh"
#include "launch.h"

namespace kva {

namespace {

constexpr int APPEND_THREADS = 256;
constexpr int APPEND_WARPS = APPEND_THREADS / 32;

// Reduce a per-lane partial over the LPR lanes of one row (rows are aligned groups).
template <int LPR>
__device__ __forceinline__ float row_sum(float part, int lane) {
  if constexpr ((LPR & (LPR - 1)) == 0) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) part += __shfl_xor_sync(FULL_MASK, part, o);
    return part;
  } else {
    const int base = (lane / LPR) * LPR;
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < LPR; ++i) tot += __shfl_sync(FULL_MASK, part, (base + i) & 31);
    return tot;
  }
}

// Reduce the angle a = pos * inv_freq (float64) into [-pi, pi] before the float32 sin/cos:
// positions reach 3.3e4 and a float32 product would lose ~1e-3 rad.
__device__ __forceinline__ void rope_cos_sin(int32_t p, double inv, float* c, float* s) {
  const double a = (double)p * inv;
  const double k = rint(a * 0.15915494309189535);          // a / (2 pi)
  const double r = fma(-k, 6.283185307179586, a);
  sincosf((float)r, s, c);
}

template <int D, typename InT, typename QOutT, typename CacheT>
__global__ void __launch_bounds__(APPEND_THREADS)
append_kernel(const __grid_constant__ AppendArgs a) {
  constexpr int LPR = D / 8;            // lanes per row
  constexpr int RPW = 32 / LPR;         // rows per warp
  constexpr int HALF = D / 2;
  constexpr int QUARTER = D / 4;

  __shared__ float s_cos[D / 2];
  __shared__ float s_sin[D / 2];
  __shared__ float s_row[APPEND_WARPS][RPW * D];

  const int t = blockIdx.x;
  const int n = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // ---- rotary angles of this token ----
  if (a.rope.kind != KVA_ROPE_NONE) {
    const int32_t* pos = a.pos + (int64_t)n * a.pos_stride + (int64_t)t * a.rope.n_axes;
    for (int j = tid; j < D / 2; j += APPEND_THREADS)
      rope_cos_sin(pos[a.rope.axis[j]], a.rope.inv[j], &s_cos[j], &s_sin[j]);
  }
  __syncthreads();

  const int32_t slot = a.slot[(int64_t)n * a.slot_stride + t];
  const bool slot_ok = slot >= 0 && slot < a.capacity;

  const int sub = lane / LPR;            // row within the warp's group
  const int e0 = (lane % LPR) * 8;       // first element owned by this lane
  const bool lane_on = sub < RPW;
  const int n_rows = a.Hq + 2 * a.Hkv;
  const float* qw = a.q_w ? a.q_w + (int64_t)n * a.w_stride : nullptr;
  const float* kw = a.k_w ? a.k_w + (int64_t)n * a.w_stride : nullptr;
  float* rowbuf = &s_row[warp][sub < RPW ? sub * D : 0];

  for (int r0 = warp * RPW; r0 < n_rows; r0 += APPEND_WARPS * RPW) {
    const int r = r0 + sub;
    const bool active = lane_on && r < n_rows;
    const int kind = !active ? 3 : (r < a.Hq ? 0 : (r < a.Hq + a.Hkv ? 1 : 2));  // q, k, v, idle
    const int head = kind == 0 ? r : (kind == 1 ? r - a.Hq : r - a.Hq - a.Hkv);

    float x[8];
    if (kind == 0) {
      load8(reinterpret_cast<const InT*>(a.q) + (((int64_t)n * a.T + t) * a.Hq + head) * D + e0, x);
    } else if (kind == 1) {
      load8(reinterpret_cast<const InT*>(a.k) + (((int64_t)n * a.T + t) * a.Hkv + head) * D + e0, x);
    } else if (kind == 2) {
      load8(reinterpret_cast<const InT*>(a.v) + (((int64_t)n * a.T + t) * a.Hkv + head) * D + e0, x);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = 0.f;
    }
    const float* w = kind == 0 ? qw : (kind == 1 ? kw : nullptr);
    const bool norm = w != nullptr;

    // ---- QK-Norm before RoPE (Qwen3 order) ----
    if (!a.after_rope) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += x[i] * x[i];
      ss = row_sum<LPR>(ss, lane);
      if (norm) {
        const float rinv = 1.0f / sqrtf(ss / (float)D + a.eps);
        float wv[8];
        load8(w + e0, wv);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = x[i] * rinv * wv[i];
      }
    }

    // ---- RoPE: partner elements exchanged through the warp's row buffer ----
    if (a.rope.kind != KVA_ROPE_NONE) {
      if (lane_on) {
#pragma unroll
        for (int i = 0; i < 8; ++i) rowbuf[e0 + i] = x[i];
      }
      __syncwarp();
      if (kind <= 1) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int d = e0 + i;
          int j, partner;
          float sgn;
          if (a.rope.kind == KVA_ROPE_2D) {
            const int b = d / HALF, dd = d - b * HALF;
            if (dd < QUARTER) { j = b * QUARTER + dd; partner = d + QUARTER; sgn = -1.f; }
            else { j = b * QUARTER + dd - QUARTER; partner = d - QUARTER; sgn = 1.f; }
          } else {
            if (d < HALF) { j = d; partner = d + HALF; sgn = -1.f; }
            else { j = d - HALF; partner = d - HALF; sgn = 1.f; }
          }
          y[i] = x[i] * s_cos[j] + sgn * rowbuf[partner] * s_sin[j];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = y[i];
      }
      __syncwarp();
    }

    // ---- QK-Norm after RoPE (HunyuanOCR order) ----
    if (a.after_rope) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += x[i] * x[i];
      ss = row_sum<LPR>(ss, lane);
      if (norm) {
        const float rinv = 1.0f / sqrtf(ss / (float)D + a.eps);
        float wv[8];
        load8(w + e0, wv);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = x[i] * rinv * wv[i];
      }
    }

    // ---- stores ----
    if (kind == 0) {
      store8(reinterpret_cast<QOutT*>(a.q_out) + (((int64_t)n * a.T + t) * a.Hq + head) * D + e0, x);
    } else if ((kind == 1 || kind == 2) && slot_ok) {
      CacheT* base = reinterpret_cast<CacheT*>(kind == 1 ? a.kc : a.vc);
      store8(base + (int64_t)n * a.inst_stride + ((int64_t)head * a.capacity + slot) * D + e0, x);
    }
  }
}

template <int D, typename InT, typename QOutT>
cudaError_t launch_cache(const AppendArgs& a, kva_dtype cache_dtype, cudaStream_t s) {
  dim3 grid(a.T, a.N);
  if (cache_dtype == KVA_BF16)
    append_kernel<D, InT, QOutT, bf16_t><<<grid, APPEND_THREADS, 0, s>>>(a);
  else
    append_kernel<D, InT, QOutT, float><<<grid, APPEND_THREADS, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D, typename InT>
cudaError_t launch_qout(const AppendArgs& a, kva_dtype q_out_dtype, kva_dtype cache_dtype,
                        cudaStream_t s) {
  if (q_out_dtype == KVA_BF16) return launch_cache<D, InT, bf16_t>(a, cache_dtype, s);
  return launch_cache<D, InT, float>(a, cache_dtype, s);
}

template <int D>
cudaError_t launch_d(const AppendArgs& a, kva_dtype in_dtype, kva_dtype q_out_dtype,
                     kva_dtype cache_dtype, cudaStream_t s) {
  if (in_dtype == KVA_BF16) return launch_qout<D, bf16_t>(a, q_out_dtype, cache_dtype, s);
  return launch_qout<D, float>(a, q_out_dtype, cache_dtype, s);
}

}  // namespace

bool append_supports_head_dim(int D) { return D == 64 || D == 72 || D == 128 || D == 256; }

cudaError_t launch_append(const AppendArgs& a, kva_dtype in_dtype, kva_dtype q_out_dtype,
                          kva_dtype cache_dtype, cudaStream_t s) {
  switch (a.D) {
    case 64: return launch_d<64>(a, in_dtype, q_out_dtype, cache_dtype, s);
    case 72: return launch_d<72>(a, in_dtype, q_out_dtype, cache_dtype, s);
    case 128: return launch_d<128>(a, in_dtype, q_out_dtype, cache_dtype, s);
    case 256: return launch_d<256>(a, in_dtype, q_out_dtype, cache_dtype, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kva
