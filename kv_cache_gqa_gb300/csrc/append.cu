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
__global__ void __launch_bounds__(APPEND_THREADS, 3)
append_kernel(const __grid_constant__ AppendArgs a) {
  constexpr int LPR = D / 8;            // lanes per row
  constexpr int RPW = 32 / LPR;         // rows per warp
  constexpr int HALF = D / 2;
  constexpr int QUARTER = D / 4;
  constexpr int ROWS_PER_PASS = APPEND_WARPS * RPW;
  constexpr bool POW2 = (LPR & (LPR - 1)) == 0;
  constexpr bool SHFL_1D = POW2 && HALF % 8 == 0;      // partner lane = lane ^ X1D
  constexpr int X1D = HALF / 8;
  constexpr bool SHFL_2D = POW2 && QUARTER % 8 == 0;   // partner lane = lane ^ X2D
  constexpr int X2D = QUARTER > 8 ? QUARTER / 8 : 1;
  constexpr int MAXP = 2;               // passes whose loads are in flight together

  __shared__ float s_cos[D / 2];
  __shared__ float s_sin[D / 2];
  __shared__ float s_row[APPEND_WARPS][RPW * D];

  const int t = blockIdx.x;
  const int n = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int sub = lane / LPR;            // row within the warp's group
  const int e0 = (lane % LPR) * 8;       // first element owned by this lane
  const bool lane_on = sub < RPW;
  const int n_rows = a.Hq + 2 * a.Hkv;
  const float* qw = a.q_w ? a.q_w + (int64_t)n * a.w_stride : nullptr;
  const float* kw = a.k_w ? a.k_w + (int64_t)n * a.w_stride : nullptr;
  float* rowbuf = &s_row[warp][sub < RPW ? sub * D : 0];

  // ---- independent loads first: slot, this token's position ids, weights ----
  const int32_t slot = a.slot[(int64_t)n * a.slot_stride + t];
  int32_t p_ang = 0;
  if (a.rope.kind != KVA_ROPE_NONE && tid < D / 2)
    p_ang = a.pos[(int64_t)n * a.pos_stride + (int64_t)t * a.rope.n_axes + a.rope.axis[tid]];
  float wq[8], wk[8];
  if (qw && lane_on) { load8(qw + e0, wq); load8(kw + e0, wk); }

  for (int pg = 0; pg < n_rows; pg += MAXP * ROWS_PER_PASS) {
    // ---- row loads of up to MAXP passes, all in flight together ----
    float x[MAXP][8];
    int kind[MAXP], head[MAXP];
#pragma unroll
    for (int p = 0; p < MAXP; ++p) {
      const int r = pg + p * ROWS_PER_PASS + warp * RPW + sub;
      const bool active = lane_on && r < n_rows;
      kind[p] = !active ? 3 : (r < a.Hq ? 0 : (r < a.Hq + a.Hkv ? 1 : 2));   // q, k, v, idle
      head[p] = kind[p] == 0 ? r : (kind[p] == 1 ? r - a.Hq : r - a.Hq - a.Hkv);
      if (kind[p] == 0) {
        load8(reinterpret_cast<const InT*>(a.q) + (((int64_t)n * a.T + t) * a.Hq + head[p]) * D + e0, x[p]);
      } else if (kind[p] == 1) {
        load8(reinterpret_cast<const InT*>(a.k) + (((int64_t)n * a.T + t) * a.Hkv + head[p]) * D + e0, x[p]);
      } else if (kind[p] == 2) {
        load8(reinterpret_cast<const InT*>(a.v) + (((int64_t)n * a.T + t) * a.Hkv + head[p]) * D + e0, x[p]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[p][i] = 0.f;
      }
    }

    // ---- rotary angles of this token (once; shared by every rotated row) ----
    if (pg == 0) {
      if (a.rope.kind != KVA_ROPE_NONE && tid < D / 2) rope_cos_sin(p_ang, a.rope.inv[tid], &s_cos[tid], &s_sin[tid]);
      __syncthreads();
    }

#pragma unroll
    for (int p = 0; p < MAXP; ++p) {
      if (pg + p * ROWS_PER_PASS >= n_rows) break;       // uniform across the CTA
      const bool norm = qw != nullptr && kind[p] <= 1;

      // ---- QK-Norm before RoPE (Qwen3 order) ----
      if (!a.after_rope) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss += x[p][i] * x[p][i];
        ss = row_sum<LPR>(ss, lane);
        if (norm) {
          const float rinv = 1.0f / sqrtf(ss / (float)D + a.eps);
#pragma unroll
          for (int i = 0; i < 8; ++i) x[p][i] = x[p][i] * rinv * (kind[p] == 0 ? wq[i] : wk[i]);
        }
      }

      // ---- RoPE ----
      // Partner of element d is d +- W/2 inside its rotated block of width W.  When W/2 is a
      // multiple of 8 it sits in lane ^ (W/16) at the same register index (rows are aligned
      // groups of a power-of-two lane count): one shuffle per element.  Otherwise (D = 72)
      // the partner goes through the warp's row buffer.
      const bool two_d = a.rope.kind == KVA_ROPE_2D;
      if (a.rope.kind != KVA_ROPE_NONE && ((!two_d && SHFL_1D) || (two_d && SHFL_2D))) {
        const int xm = two_d ? X2D : X1D;
        const int wh = two_d ? QUARTER : HALF;      // half width of the rotated block
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float pv = __shfl_xor_sync(FULL_MASK, x[p][i], xm);
          const int d = e0 + i;
          const int blk = two_d ? d / HALF : 0;
          const int dd = d - blk * HALF;
          const bool lo_half = dd < wh;
          const int j = blk * QUARTER + (lo_half ? dd : dd - wh);   // 1D: blk = 0, j = d mod HALF
          y[i] = x[p][i] * s_cos[j] + (lo_half ? -pv : pv) * s_sin[j];
        }
        if (kind[p] <= 1) {
#pragma unroll
          for (int i = 0; i < 8; ++i) x[p][i] = y[i];
        }
      } else if (a.rope.kind != KVA_ROPE_NONE) {
        if (lane_on) {
#pragma unroll
          for (int i = 0; i < 8; ++i) rowbuf[e0 + i] = x[p][i];
        }
        __syncwarp();
        if (kind[p] <= 1) {
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
            y[i] = x[p][i] * s_cos[j] + sgn * rowbuf[partner] * s_sin[j];
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) x[p][i] = y[i];
        }
        __syncwarp();
      }

      // ---- QK-Norm after RoPE (HunyuanOCR order) ----
      if (a.after_rope) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss += x[p][i] * x[p][i];
        ss = row_sum<LPR>(ss, lane);
        if (norm) {
          const float rinv = 1.0f / sqrtf(ss / (float)D + a.eps);
#pragma unroll
          for (int i = 0; i < 8; ++i) x[p][i] = x[p][i] * rinv * (kind[p] == 0 ? wq[i] : wk[i]);
        }
      }

      // ---- stores ----
      if (kind[p] == 0) {
        store8(reinterpret_cast<QOutT*>(a.q_out) + (((int64_t)n * a.T + t) * a.Hq + head[p]) * D + e0, x[p]);
      } else if ((kind[p] == 1 || kind[p] == 2) && slot >= 0 && slot < a.capacity) {
        CacheT* base = reinterpret_cast<CacheT*>(kind[p] == 1 ? a.kc : a.vc);
        store8(base + (int64_t)n * a.inst_stride + ((int64_t)head[p] * a.capacity + slot) * D + e0, x[p]);
      }
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
