// Kernel (a), general-layout form: QK-Norm + RoPE fused into the K/V cache write for the
// layouts the fast forms in append.cu do not tile.
//
//  - Asymmetric caches: q and k rows Dk wide, v rows Dv wide (an MLA layer expanded to
//    per-head K = 192 and V = 128 before it reaches the cache, Youtu-VL-4B ncnn port,
//    section 6).
//  - RoPE over a sub-range of the head: only dims [rot_offset, rot_offset + rot_dim) rotate,
//    with the frequencies of a rot_dim-wide head (the 64 rotary dims of that 192-wide head,
//    interleaved: implementation difficulty 2); the rest passes through.
//  - Any head width that is a multiple of 8 up to 256.
//
// One CTA per (token t, instance n, row group), one warp per row; short appends (a decode
// token) split a token's rows over several CTAs so that its row loads run in parallel, and a
// warp loads four of its rows before transforming them (long appends).  Each
// CTA evaluates the token's rot_dim/2 angles once into shared memory.  A lane holds 8 consecutive elements of its row in
// registers (a 16- or 32-byte access); the row is mirrored into a per-warp shared buffer so
// that each element can read its rotation partner wherever it sits (rotate-half partner,
// 2D-halves partner, or the interleaved pair).  The norm's sum of squares is a warp
// reduction over the whole head width.
//
// Method: per-head RMSNorm (Penguin-VL ncnn port, sections 2.1 and 4.2); rotate-half RoPE
// in 1D, xdRoPE-section, 2D-halves or de-interleaved form (Youtu-VL-4B ncnn port,
// implementation difficulty 2; HunyuanOCR v1.0 ncnn port, section five; Penguin-VL ncnn
// port, section 2.3); k/v written into the token's cache slot (Youtu-VL-4B ncnn port, step 6).
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace kva {

namespace {

constexpr int GEN_THREADS = 256;
constexpr int GEN_WARPS = GEN_THREADS / 32;
constexpr int GEN_MAX_D = 256;   // 32 lanes x 8 elements
constexpr int RB = 4;            // rows a warp loads before transforming them

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  return v;
}

template <typename InT, typename QOutT, typename CacheT>
__global__ void __launch_bounds__(GEN_THREADS, 4)
append_general_kernel(const __grid_constant__ AppendArgs a) {
  __shared__ float s_cos[MAX_ROPE_FREQ];
  __shared__ float s_sin[MAX_ROPE_FREQ];
  __shared__ __align__(16) float s_row[GEN_WARPS][GEN_MAX_D];

  const int t = blockIdx.x, n = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Dk = a.D, Dv = a.Dv;
  const int ro = a.rot_offset, rw = a.rot_dim, half = rw / 2, quarter = rw / 4;
  const int kind_r = a.rope.kind;
  const int n_rows = a.Hq + 2 * a.Hkv;
  const float* qw = a.q_w ? a.q_w + (int64_t)n * a.w_stride : nullptr;
  const float* kw = a.k_w ? a.k_w + (int64_t)n * a.w_stride : nullptr;
  griddep_wait();                               // inputs of this launch are complete from here on
  const int32_t slot = a.slot[(int64_t)n * a.slot_stride + t];
  const int64_t tok = (int64_t)n * a.T + t;

  if (kind_r != KVA_ROPE_NONE) {
    for (int j = tid; j < half; j += GEN_THREADS) {
      const int32_t p = a.pos[(int64_t)n * a.pos_stride + (int64_t)t * a.rope.n_axes + a.rope.axis[j]];
      rope_cos_sin(p, a.rope.inv_hi[j], a.rope.inv_lo[j], a.rope.inv[j], &s_cos[j], &s_sin[j]);
    }
  }
  __syncthreads();

  float* rowbuf = s_row[warp];
  const int e0 = lane * 8;
  // A warp takes RB rows per pass and issues all their loads before transforming any of them:
  // with one row at a time a warp had a single 16-byte load per lane in flight, too few bytes
  // per SM for HBM when a token's rows all sit in one CTA (long appends).
  const int stride = GEN_WARPS * gridDim.z;
  for (int r0 = blockIdx.z * GEN_WARPS + warp; r0 < n_rows; r0 += RB * stride) {
    float xs[RB][8];
#pragma unroll
    for (int k = 0; k < RB; ++k) {
      const int r = r0 + k * stride;
      const int kind = r < a.Hq ? 0 : (r < a.Hq + a.Hkv ? 1 : 2);     // q, k, v (warp-uniform)
      const int head = kind == 0 ? r : (kind == 1 ? r - a.Hq : r - a.Hq - a.Hkv);
      const int width = kind == 2 ? Dv : Dk;
      if (r < n_rows && e0 < width) {
        if (kind == 0) load8(reinterpret_cast<const InT*>(a.q) + (tok * a.Hq + head) * Dk + e0, xs[k]);
        else if (kind == 1) load8(reinterpret_cast<const InT*>(a.k) + (tok * a.Hkv + head) * Dk + e0, xs[k]);
        else load8(reinterpret_cast<const InT*>(a.v) + (tok * a.Hkv + head) * Dv + e0, xs[k]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) xs[k][i] = 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < RB; ++k) {
    const int r = r0 + k * stride;
    if (r >= n_rows) break;                     // warp-uniform
    const int kind = r < a.Hq ? 0 : (r < a.Hq + a.Hkv ? 1 : 2);
    const int head = kind == 0 ? r : (kind == 1 ? r - a.Hq : r - a.Hq - a.Hkv);
    const int width = kind == 2 ? Dv : Dk;
    const bool on = e0 < width;
    float (&x)[8] = xs[k];

    if (kind <= 1) {
      const float* w = kind == 0 ? qw : kw;
      auto apply_norm = [&]() {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss += x[i] * x[i];
        ss = warp_sum(ss);
        if (w != nullptr && on) {
          float wv[8];
          load8(w + e0, wv);
          const float rinv = 1.0f / sqrtf(ss / (float)Dk + a.eps);
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = x[i] * rinv * wv[i];
        }
      };
      if (!a.after_rope) apply_norm();
      if (kind_r != KVA_ROPE_NONE) {
        if (on) {
#pragma unroll
          for (int i = 0; i < 8; ++i) rowbuf[e0 + i] = x[i];
        }
        __syncwarp();
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int dd = e0 + i - ro;                    // index inside the rotated range
          y[i] = x[i];
          if (on && dd >= 0 && dd < rw) {
            const float* xr = rowbuf + ro;
            if (kind_r == KVA_ROPE_INTERLEAVED) {
              // output dd < W/2 pairs (x[2j], x[2j+1]) as x[2j] c - x[2j+1] s; dd >= W/2 as
              // x[2j+1] c + x[2j] s, j = dd mod W/2
              const int j = dd < half ? dd : dd - half;
              const float ev = xr[2 * j], od = xr[2 * j + 1];
              y[i] = dd < half ? ev * s_cos[j] - od * s_sin[j] : od * s_cos[j] + ev * s_sin[j];
            } else if (kind_r == KVA_ROPE_2D) {
              const int b = dd / half, e2 = dd - b * half;
              const bool lo = e2 < quarter;
              const int j = b * quarter + (lo ? e2 : e2 - quarter);
              const float pv = xr[lo ? dd + quarter : dd - quarter];
              y[i] = x[i] * s_cos[j] + (lo ? -pv : pv) * s_sin[j];
            } else {                                     // 1D and sections: rotate-half over W
              const bool lo = dd < half;
              const int j = lo ? dd : dd - half;
              const float pv = xr[lo ? dd + half : dd - half];
              y[i] = x[i] * s_cos[j] + (lo ? -pv : pv) * s_sin[j];
            }
          }
        }
        __syncwarp();                                    // buffer reads done before the next row
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = y[i];
      }
      if (a.after_rope) apply_norm();
    }

    if (!on) continue;
    if (kind == 0) {
      store8(reinterpret_cast<QOutT*>(a.q_out) + (tok * a.Hq + head) * Dk + e0, x);
    } else if (slot >= 0 && slot < a.capacity) {
      if (kind == 1)
        store8(reinterpret_cast<CacheT*>(a.kc) + (int64_t)n * a.inst_stride + ((int64_t)head * a.capacity + slot) * Dk + e0, x);
      else
        store8(reinterpret_cast<CacheT*>(a.vc) + (int64_t)n * a.inst_stride_v + ((int64_t)head * a.capacity + slot) * Dv + e0, x);
    }
    }
  }
  // the next kernel may start its set-up only as this CTA finishes: a long (many-wave) append
  // must not have its SMs taken by a waiting persistent kernel
  griddep_launch_dependents();
}

int gen_num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 148;
  }
  return n;
}

template <typename InT, typename QOutT>
cudaError_t launch_c(const AppendArgs& a, kva_dtype cache_dtype, cudaStream_t s) {
  // row groups per token: enough CTAs for about two per SM, at most one warp per row
  const int64_t tokens = (int64_t)a.T * a.N;
  const int n_rows = a.Hq + 2 * a.Hkv;
  const int max_groups = (n_rows + GEN_WARPS - 1) / GEN_WARPS;
  const int groups = (int)std::max<int64_t>(1, std::min<int64_t>(max_groups, 2 * gen_num_sms() / std::max<int64_t>(1, tokens)));
  dim3 grid(a.T, a.N, std::min(groups, 65535));
  if (cache_dtype == KVA_BF16) return launch_pdl(append_general_kernel<InT, QOutT, bf16_t>, grid, dim3(GEN_THREADS), 0, s, a);
  return launch_pdl(append_general_kernel<InT, QOutT, float>, grid, dim3(GEN_THREADS), 0, s, a);
}

template <typename InT>
cudaError_t launch_q(const AppendArgs& a, kva_dtype q_out_dtype, kva_dtype cache_dtype, cudaStream_t s) {
  if (q_out_dtype == KVA_BF16) return launch_c<InT, bf16_t>(a, cache_dtype, s);
  return launch_c<InT, float>(a, cache_dtype, s);
}

}  // namespace

bool append_general_supports(int Dk, int Dv) {
  return Dk > 0 && Dv > 0 && Dk % 8 == 0 && Dv % 8 == 0 && Dk <= GEN_MAX_D && Dv <= GEN_MAX_D;
}

cudaError_t launch_append_general(const AppendArgs& a, kva_dtype in_dtype, kva_dtype q_out_dtype,
                                  kva_dtype cache_dtype, cudaStream_t s) {
  if (!append_general_supports(a.D, a.Dv) || a.rot_dim / 2 > MAX_ROPE_FREQ || a.N > 65535)
    return cudaErrorInvalidValue;
  if (in_dtype == KVA_BF16) return launch_q<bf16_t>(a, q_out_dtype, cache_dtype, s);
  return launch_q<float>(a, q_out_dtype, cache_dtype, s);
}

}  // namespace kva
