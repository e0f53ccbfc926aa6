// Kernel (a): QK-Norm + RoPE fused into the K/V cache write.
//
// Warp-per-token form (head_dim 64, 128, 256).  Each warp owns one (token t, instance n):
// it evaluates the token's D/2 rotary angles once (two per lane for D = 128), keeps the
// cos/sin of its own eight elements in registers, and then streams the token's Hq q rows,
// Hkv k rows and Hkv v rows.  A row is split over D/8 lanes that own 8 consecutive
// elements, so every global load and store is a 128-bit access and each row is one
// contiguous, coalesced segment; the loads of four row groups are in flight together.  The
// rotate-half partner of an element sits D/16 (1D, sections) or D/32 (2D) lanes away at the
// same register index: one shuffle per element.  A CTA holds 1, 2, 4 or 8 tokens (8, 4, 2
// or 1 warps per token) so that short appends (one decode token) still spread over 8 warps.
// Head_dim 72 (rows of 9 lanes) keeps the CTA-per-token form with a shared row buffer.
//
// Method: per-head RMSNorm over head_dim (Penguin-VL ncnn port, sections 2.1 and 4.2);
// rotate-half RoPE x*cos + rotate_half(x)*sin (Youtu-VL-4B ncnn port, implementation
// difficulty 2) in 1D, xdRoPE-section (HunyuanOCR v1.0 ncnn port, section five) or
// 2D-halves form (Penguin-VL ncnn port, section 2.3); k/v written into the new token's
// cache slot by the runtime (Youtu-VL-4B ncnn port, step 6), k normalised before the
// write when the norm follows RoPE (HunyuanOCR v1.0 ncnn port, section five item 2).
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace kva {

namespace {

constexpr int APPEND_THREADS = 256;
constexpr int APPEND_WARPS = APPEND_THREADS / 32;

int append_num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 148;
  }
  return n;
}

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

// CTA-per-token form, used for head_dim 72 (a row is 9 lanes, so the rotate-half partner
// goes through a shared row buffer).
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
      if (a.rope.kind != KVA_ROPE_NONE && tid < D / 2)
        rope_cos_sin(p_ang, a.rope.inv_hi[tid], a.rope.inv_lo[tid], a.rope.inv[tid], &s_cos[tid], &s_sin[tid]);
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


__device__ __forceinline__ void load4_smem(const float* p, float (&x)[4]) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
}
__device__ __forceinline__ void load4_smem(const bf16_t* p, float (&x)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
}
__device__ __forceinline__ void store4(float* p, const float (&y)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(y[0], y[1], y[2], y[3]);
}
__device__ __forceinline__ void store4(bf16_t* p, const float (&y)[4]) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
}

__device__ __forceinline__ void load8_smem(const float* p, float (&x)[8]) {
  const float4 u = reinterpret_cast<const float4*>(p)[0], w = reinterpret_cast<const float4*>(p)[1];
  x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w; x[4] = w.x; x[5] = w.y; x[6] = w.z; x[7] = w.w;
}
__device__ __forceinline__ void load8_smem(const bf16_t* p, float (&x)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
  x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}

// Warp-per-token form.  tpc = tokens per CTA (1, 2, 4 or 8); the 8 / tpc warps of a token
// take its row groups round-robin.
template <int D, typename InT, typename QOutT, typename CacheT>
__global__ void __launch_bounds__(APPEND_THREADS, 2)
append_warp_kernel(const __grid_constant__ AppendArgs a, int tpc) {
  constexpr int LPR = D / 8;            // lanes per row
  constexpr int RPW = 32 / LPR;         // rows per warp and row group
  constexpr int HALF = D / 2, QUARTER = D / 4;
  constexpr int U = 4;                  // row groups whose loads are in flight together
  static_assert(LPR == 8 || LPR == 16 || LPR == 32, "power-of-two lanes per row");
  __shared__ __align__(16) float s_cs[APPEND_WARPS][2][HALF];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpt = APPEND_WARPS / tpc;
  const int t = blockIdx.x * tpc + warp / wpt;
  const int wt = warp % wpt;
  const int n = blockIdx.y;
  constexpr int JPL = (HALF + 31) / 32;  // angle slots per lane
  float r_ih[JPL], r_il[JPL];
  double r_inv[JPL];
  int r_axis[JPL];
#pragma unroll
  for (int i = 0; i < JPL; ++i) {        // parameter-table reads before the wait (see rope_cos_sin)
    const int j = min(lane + 32 * i, HALF - 1);
    r_ih[i] = a.rope.inv_hi[j]; r_il[i] = a.rope.inv_lo[j]; r_inv[i] = a.rope.inv[j]; r_axis[i] = a.rope.axis[j];
  }
  griddep_wait();
  griddep_launch_dependents();
  if (t >= a.T) return;                 // warp-uniform, and no CTA-wide barrier follows

  const int sub = lane / LPR;           // row within the group
  const int e0 = (lane % LPR) * 8;      // first element owned by this lane
  const int n_rows = a.Hq + 2 * a.Hkv;
  const int64_t tok = (int64_t)n * a.T + t;
  const int32_t slot = a.slot[(int64_t)n * a.slot_stride + t];
  const bool rotate = a.rope.kind != KVA_ROPE_NONE;
  const bool two_d = a.rope.kind == KVA_ROPE_2D;
  // interleaved RoPE: the lane's 8 inputs are the pairs j = e0/2 .. e0/2 + 3, whose rotated
  // values land at outputs j (x[0..3] after the rotation) and D/2 + j (x[4..7])
  const bool inter = a.rope.kind == KVA_ROPE_INTERLEAVED;

  // ---- this token's angles: slot j in [0, D/2) ----
  float* cs = &s_cs[warp][0][0];
  if (rotate) {
#pragma unroll
    for (int i = 0; i < JPL; ++i) {
      const int j = lane + 32 * i;
      if (j < HALF) {
        const int32_t p = a.pos[(int64_t)n * a.pos_stride + (int64_t)t * a.rope.n_axes + r_axis[i]];
        rope_cos_sin(p, r_ih[i], r_il[i], r_inv[i], &cs[j], &cs[HALF + j]);
      }
    }
  }
  float wq[8], wk[8];
  const bool norm = a.q_w != nullptr;
  if (norm && inter && a.after_rope) {            // the norm sees the outputs' order
    const float* qwp = a.q_w + (int64_t)n * a.w_stride;
    const float* kwp = a.k_w + (int64_t)n * a.w_stride;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      wq[i] = qwp[e0 / 2 + i]; wq[4 + i] = qwp[HALF + e0 / 2 + i];
      wk[i] = kwp[e0 / 2 + i]; wk[4 + i] = kwp[HALF + e0 / 2 + i];
    }
  } else if (norm) {
    load8(a.q_w + (int64_t)n * a.w_stride + e0, wq);
    load8(a.k_w + (int64_t)n * a.w_stride + e0, wk);
  }
  __syncwarp();
  // element e0 + i uses slot j0 + i; the rotate-half partner is d +- W/2 (W = D, or D/2 per
  // half in 2D), which the sign folded into sn[] accounts for
  float c[8], sn[8];
  if (inter) {                                      // angles of the lane's pairs e0/2 .. e0/2 + 3
    const float4 c0 = *reinterpret_cast<const float4*>(&cs[e0 / 2]);
    const float4 s0 = *reinterpret_cast<const float4*>(&cs[HALF + e0 / 2]);
    c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
    sn[0] = s0.x; sn[1] = s0.y; sn[2] = s0.z; sn[3] = s0.w;
#pragma unroll
    for (int i = 4; i < 8; ++i) c[i] = sn[i] = 0.f;
  } else if (rotate) {
    const int blk = two_d ? e0 / HALF : 0;
    const int dd = e0 - blk * HALF;
    const int wh = two_d ? QUARTER : HALF;
    const bool lo = dd < wh;
    const int j0 = blk * QUARTER + (lo ? dd : dd - wh);
    const float4 c0 = *reinterpret_cast<const float4*>(&cs[j0]);
    const float4 c1 = *reinterpret_cast<const float4*>(&cs[j0 + 4]);
    const float4 s0 = *reinterpret_cast<const float4*>(&cs[HALF + j0]);
    const float4 s1 = *reinterpret_cast<const float4*>(&cs[HALF + j0 + 4]);
    const float sg = lo ? -1.f : 1.f;
    c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w; c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
    sn[0] = sg * s0.x; sn[1] = sg * s0.y; sn[2] = sg * s0.z; sn[3] = sg * s0.w;
    sn[4] = sg * s1.x; sn[5] = sg * s1.y; sn[6] = sg * s1.z; sn[7] = sg * s1.w;
  }
  const int xm = two_d ? QUARTER / 8 : HALF / 8;     // partner lane distance (xor)

  const int n_groups = (n_rows + RPW - 1) / RPW;
  for (int g0 = wt; g0 < n_groups; g0 += U * wpt) {
    float x[U][8];
    int kind[U], head[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int grp = g0 + u * wpt;
      const int r = grp * RPW + sub;
      kind[u] = (grp >= n_groups || r >= n_rows) ? 3 : (r < a.Hq ? 0 : (r < a.Hq + a.Hkv ? 1 : 2));
      head[u] = kind[u] == 0 ? r : (kind[u] == 1 ? r - a.Hq : r - a.Hq - a.Hkv);
      if (kind[u] == 0) load8(reinterpret_cast<const InT*>(a.q) + (tok * a.Hq + head[u]) * D + e0, x[u]);
      else if (kind[u] == 1) load8(reinterpret_cast<const InT*>(a.k) + (tok * a.Hkv + head[u]) * D + e0, x[u]);
      else if (kind[u] == 2) load8(reinterpret_cast<const InT*>(a.v) + (tok * a.Hkv + head[u]) * D + e0, x[u]);
      else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[u][i] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (g0 + u * wpt >= n_groups) break;           // uniform across the warp
      const bool qk = kind[u] <= 1;
      auto apply_norm = [&]() {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(x[u][i], x[u][i], ss);
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
        if (norm && qk) {
          const float rinv = rsqrtf(ss * (1.0f / (float)D) + a.eps);
#pragma unroll
          for (int i = 0; i < 8; ++i) x[u][i] *= rinv * (kind[u] == 0 ? wq[i] : wk[i]);
        }
      };
      if (!a.after_rope) apply_norm();
      if (inter) {
        if (qk) {
          float y[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            y[i] = fmaf(-x[u][2 * i + 1], sn[i], x[u][2 * i] * c[i]);
            y[4 + i] = fmaf(x[u][2 * i], sn[i], x[u][2 * i + 1] * c[i]);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) x[u][i] = y[i];
        }
      } else if (rotate) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float pv = __shfl_xor_sync(FULL_MASK, x[u][i], xm);
          y[i] = fmaf(pv, sn[i], x[u][i] * c[i]);
        }
        if (qk) {
#pragma unroll
          for (int i = 0; i < 8; ++i) x[u][i] = y[i];
        }
      }
      if (a.after_rope) apply_norm();
      auto put = [&](auto* dst) {                     // q/k rows of interleaved RoPE: two halves
        if (inter && qk) {
          float lo[4] = {x[u][0], x[u][1], x[u][2], x[u][3]}, hi[4] = {x[u][4], x[u][5], x[u][6], x[u][7]};
          store4(dst + e0 / 2, lo);
          store4(dst + HALF + e0 / 2, hi);
        } else {
          store8(dst + e0, x[u]);
        }
      };
      if (kind[u] == 0) {
        put(reinterpret_cast<QOutT*>(a.q_out) + (tok * a.Hq + head[u]) * D);
      } else if ((kind[u] == 1 || kind[u] == 2) && slot >= 0 && slot < a.capacity) {
        CacheT* base = reinterpret_cast<CacheT*>(kind[u] == 1 ? a.kc : a.vc);
        put(base + (int64_t)n * a.inst_stride + ((int64_t)head[u] * a.capacity + slot) * D);
      }
    }
  }
}

// Streaming form for long appends (prefill): a persistent CTA per SM walks work items
// (instance n, block of tb tokens).  One producer lane copies an item's q, k and v rows (three
// contiguous segments, since the inputs are token-major) and the instance's norm weights into
// a 3-stage shared-memory ring with bulk async copies, so ~3 items (~190 KB) are in flight per
// SM; sixteen consumer warps transform the rows out of shared memory and store them.  In this
// form the D/8 lanes of a row each own two 4-element chunks, at o1 and o1 + W/2 (W the width of
// the rotated block), so an element and its rotate-half partner sit in the same lane and every
// shared-memory read is a conflict-free 16-byte access.  The positions and slots of the next
// item are loaded while the current one is processed; its angles go to a per-stage table.
constexpr int STREAM_STAGES = 3;
constexpr int STREAM_CONSUMERS = 16;                      // consumer warps
constexpr int STREAM_THREADS = (STREAM_CONSUMERS + 1) * 32;
constexpr int STREAM_ANGLES = 512;                        // tb * D/2 per item, at most
constexpr int STREAM_STAGE_MAX = 64 * 1024;

// Barrier over the consumer warps (named barrier 1) that also ANDs a predicate across them.
__device__ __forceinline__ bool consumers_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 1, %2, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r) : "r"((uint32_t)v), "r"(STREAM_CONSUMERS * 32) : "memory");
  return r != 0;
}

template <int D, typename InT, typename QOutT, typename CacheT>
__global__ void __launch_bounds__(STREAM_THREADS, 1)
append_stream_kernel(const __grid_constant__ AppendArgs a, int tb, int stage_bytes) {
  constexpr int LPR = D / 8, RPW = 32 / LPR, HALF = D / 2, QUARTER = D / 4;
  constexpr int NC = STREAM_CONSUMERS;
  constexpr int APT = (STREAM_ANGLES + NC * 32 - 1) / (NC * 32);   // angles per consumer thread
  static_assert((NC * 32) % HALF == 0, "a thread keeps one angle slot across its angles");
  constexpr int U = 2;                                  // row groups in flight per warp
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[STREAM_STAGES], empty[STREAM_STAGES];
  __shared__ __align__(16) float s_cs[STREAM_STAGES][2][STREAM_ANGLES];   // [stage][cos|sin][tt * HALF + j]
  __shared__ int32_t s_slot[STREAM_STAGES][STREAM_ANGLES / 32];            // destination slot per token

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tb = (a.T + tb - 1) / tb;
  const int items = a.N * n_tb;
  const int64_t tok_q = (int64_t)a.Hq * D, tok_kv = (int64_t)a.Hkv * D;      // elements per token
  if (threadIdx.x == 0) {
    for (int st = 0; st < STREAM_STAGES; ++st) { mbar_init(&full[st], 1); mbar_init(&empty[st], NC); }
    fence_mbar_init();
  }
  // this consumer thread's angle slot (the same for every item) and its table entries: read
  // once here, since per-lane different indices into the parameter table serialise
  const int ct = threadIdx.x;
  const int my_j = ct % HALF;
  const float my_ih = a.rope.inv_hi[my_j], my_il = a.rope.inv_lo[my_j];
  const double my_inv = a.rope.inv[my_j];
  const int my_axis = a.rope.axis[my_j];
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();

  if (warp == NC) {                                     // ---- producer ----
    if (lane == 0) {
      int k = 0;
      for (int it = blockIdx.x; it < items; it += gridDim.x, ++k) {
        const int st = k % STREAM_STAGES;
        if (k >= STREAM_STAGES && !mbar_wait_bounded(&empty[st], (uint32_t)((k / STREAM_STAGES - 1) & 1))) break;
        const int n = it / n_tb, t0 = (it % n_tb) * tb, nt = min(tb, a.T - t0);
        const int64_t tok = (int64_t)n * a.T + t0;
        const uint32_t bq = (uint32_t)(nt * tok_q * sizeof(InT)), bkv = (uint32_t)(nt * tok_kv * sizeof(InT));
        const uint32_t bw = a.q_w ? 2u * D * (uint32_t)sizeof(float) : 0u;
        unsigned char* dst = ring + (size_t)st * stage_bytes;
        mbar_arrive_expect_tx(&full[st], bq + 2 * bkv + bw);
        bulk_g2s(dst, reinterpret_cast<const InT*>(a.q) + tok * tok_q, bq, &full[st]);
        bulk_g2s(dst + (size_t)tb * tok_q * sizeof(InT), reinterpret_cast<const InT*>(a.k) + tok * tok_kv, bkv, &full[st]);
        bulk_g2s(dst + (size_t)tb * (tok_q + tok_kv) * sizeof(InT), reinterpret_cast<const InT*>(a.v) + tok * tok_kv,
                 bkv, &full[st]);
        if (bw) {                                         // this instance's norm weights ride along
          unsigned char* wdst = dst + (size_t)tb * (tok_q + 2 * tok_kv) * sizeof(InT);
          bulk_g2s(wdst, a.q_w + (int64_t)n * a.w_stride, D * sizeof(float), &full[st]);
          bulk_g2s(wdst + D * sizeof(float), a.k_w + (int64_t)n * a.w_stride, D * sizeof(float), &full[st]);
        }
      }
      // copies this CTA issued have normally been consumed; never leave one in flight
      for (int j = max(0, k - STREAM_STAGES); j < k; ++j)
        mbar_wait_bounded(&full[j % STREAM_STAGES], (uint32_t)((j / STREAM_STAGES) & 1));
    }
    return;
  }

  // ---- consumers ----
  const int sub = lane / LPR, rl = lane % LPR;
  const int n_rows = a.Hq + 2 * a.Hkv;
  const int gpt = (n_rows + RPW - 1) / RPW;             // row groups per token
  const bool rotate = a.rope.kind != KVA_ROPE_NONE;
  const bool two_d = a.rope.kind == KVA_ROPE_2D;
  const bool inter = a.rope.kind == KVA_ROPE_INTERLEAVED;   // q/k inputs in (x_2j, x_2j+1) pairs
  const bool norm = a.q_w != nullptr;
  // this lane's chunks: o1 (low half of its rotated block) and o2 = o1 + W/2; angle slot j0.
  // With interleaved RoPE the outputs o1.. and o2.. come from the input pairs at 2 * o1 ..
  int o1, j0;
  if (two_d) {
    const int per_blk = LPR / 2, blk = rl / per_blk, ll = rl % per_blk;
    o1 = blk * HALF + 4 * ll;
    j0 = blk * QUARTER + 4 * ll;
  } else {
    o1 = 4 * rl;
    j0 = o1;
  }
  const int o2 = o1 + (two_d ? QUARTER : HALF);

  // positions and destination slots of an item, loaded one item ahead
  auto load_meta = [&](int it, int32_t (&p)[APT], int32_t& slot) {
    if (it >= items) return;
    const int n = it / n_tb, t0 = (it % n_tb) * tb, nt = min(tb, a.T - t0);
    if (ct < nt) slot = a.slot[(int64_t)n * a.slot_stride + t0 + ct];
    if (!rotate) return;
#pragma unroll
    for (int i = 0; i < APT; ++i) {
      const int tt = (ct + i * NC * 32) / HALF;
      if (tt < nt) p[i] = a.pos[(int64_t)n * a.pos_stride + (int64_t)(t0 + tt) * a.rope.n_axes + my_axis];
    }
  };
  int32_t p_next[APT], slot_next = 0;
#pragma unroll
  for (int i = 0; i < APT; ++i) p_next[i] = 0;
  load_meta(blockIdx.x, p_next, slot_next);
  int k = 0;
  for (int it = blockIdx.x; it < items; it += gridDim.x, ++k) {
    const int st = k % STREAM_STAGES;
    const int n = it / n_tb, t0 = (it % n_tb) * tb, nt = min(tb, a.T - t0);
    int32_t p_cur[APT];
#pragma unroll
    for (int i = 0; i < APT; ++i) p_cur[i] = p_next[i];
    if (ct < nt) s_slot[st][ct] = slot_next;
    load_meta(it + gridDim.x, p_next, slot_next);       // in flight during this item
    if (rotate) {
#pragma unroll
      for (int i = 0; i < APT; ++i) {
        const int idx = ct + i * NC * 32;                 // slot my_j of token idx / HALF
        if (idx / HALF < nt) rope_cos_sin(p_cur[i], my_ih, my_il, my_inv, &s_cs[st][0][idx], &s_cs[st][1][idx]);
      }
    }
    // the item's rows have landed and its angles are in the table, for every consumer warp (the
    // outcome of the bounded wait is reduced over all of them, so they leave the loop together)
    const bool landed = mbar_wait_bounded(&full[st], (uint32_t)((k / STREAM_STAGES) & 1));
    if (!consumers_all(landed)) break;
    const unsigned char* stage = ring + (size_t)st * stage_bytes;
    const InT* sq = reinterpret_cast<const InT*>(stage);
    const InT* sk = sq + (size_t)tb * tok_q;
    const InT* sv = sk + (size_t)tb * tok_kv;
    const float* swq = reinterpret_cast<const float*>(sv + (size_t)tb * tok_kv);
    const float* swk = swq + D;

    // row groups g = warp, warp + NC, ... of the item (group gg of token tt), U at a time
    int tt = 0, gg = warp;
    while (gg >= gpt && tt < nt) { gg -= gpt; ++tt; }
    while (tt < nt) {
      float xl[U][4], xh[U][4];
      int kind[U], head[U], tok_of[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int r = gg * RPW + sub;
        const bool live = tt < nt;
        kind[u] = (!live || r >= n_rows) ? 3 : (r < a.Hq ? 0 : (r < a.Hq + a.Hkv ? 1 : 2));
        head[u] = kind[u] == 0 ? r : (kind[u] == 1 ? r - a.Hq : r - a.Hq - a.Hkv);
        tok_of[u] = tt;
        const InT* src = kind[u] == 0 ? sq + (tt * a.Hq + head[u]) * D
                       : kind[u] == 1 ? sk + (tt * a.Hkv + head[u]) * D
                       : kind[u] == 2 ? sv + (tt * a.Hkv + head[u]) * D : nullptr;
        if (src && inter && kind[u] <= 1) {             // evens -> low output half, odds -> high
          float t8[8];
          load8_smem(src + 2 * o1, t8);
#pragma unroll
          for (int i = 0; i < 4; ++i) { xl[u][i] = t8[2 * i]; xh[u][i] = t8[2 * i + 1]; }
        } else if (src) {
          load4_smem(src + o1, xl[u]);
          load4_smem(src + o2, xh[u]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) xl[u][i] = xh[u][i] = 0.f;
        }
        gg += NC;                                       // next group of this warp
        while (gg >= gpt && tt < nt) { gg -= gpt; ++tt; }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool qk = kind[u] <= 1;
        auto apply_norm = [&]() {
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) { s0 = fmaf(xl[u][i], xl[u][i], s0); s1 = fmaf(xh[u][i], xh[u][i], s1); }
          float ss = s0 + s1;
#pragma unroll
          for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
          if (norm && qk) {
            const float rinv = rsqrtf(ss * (1.0f / (float)D) + a.eps);
            const float* w = kind[u] == 0 ? swq : swk;
            float wl[4], wh[4];
            if (inter && !a.after_rope) {               // before RoPE the weights follow the inputs
              float w8[8];
              load8_smem(w + 2 * o1, w8);
#pragma unroll
              for (int i = 0; i < 4; ++i) { wl[i] = w8[2 * i]; wh[i] = w8[2 * i + 1]; }
            } else {
              load4_smem(w + o1, wl);
              load4_smem(w + o2, wh);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) { xl[u][i] *= rinv * wl[i]; xh[u][i] *= rinv * wh[i]; }
          }
        };
        if (!a.after_rope) apply_norm();
        if (rotate && qk) {
          float c[4], sn[4];
          load4_smem(&s_cs[st][0][tok_of[u] * HALF + j0], c);
          load4_smem(&s_cs[st][1][tok_of[u] * HALF + j0], sn);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lo = xl[u][i], hi = xh[u][i];
            xl[u][i] = fmaf(-hi, sn[i], lo * c[i]);
            xh[u][i] = fmaf(lo, sn[i], hi * c[i]);
          }
        }
        if (a.after_rope) apply_norm();
        const int64_t tok = (int64_t)n * a.T + t0 + tok_of[u];
        if (kind[u] == 0) {
          QOutT* dst = reinterpret_cast<QOutT*>(a.q_out) + (tok * a.Hq + head[u]) * D;
          store4(dst + o1, xl[u]);
          store4(dst + o2, xh[u]);
        } else if (kind[u] <= 2) {
          const int32_t slot = s_slot[st][tok_of[u]];
          if (slot >= 0 && slot < a.capacity) {
            CacheT* dst = reinterpret_cast<CacheT*>(kind[u] == 1 ? a.kc : a.vc) + (int64_t)n * a.inst_stride +
                          ((int64_t)head[u] * a.capacity + slot) * D;
            store4(dst + o1, xl[u]);
            store4(dst + o2, xh[u]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
}

// Lean streaming form for the common prefill layout: head_dim 128, float32 inputs, rotate-half
// RoPE over the whole head (1D or xdRoPE sections, or none) and QK-Norm before, after or
// absent, all fixed at compile time.  The producer and the per-item angle table are those of the
// general streaming form.  The consumer work is cut to what the method needs: a token's rows are
// taken in pairs (both q, both k or both v, since Hq and Hkv are even), half a warp per row and
// 8 elements per lane (lane chunk at o and o + 64, so the rotate-half partner is in the same
// lane), norm weights held in registers for the item, and no per-row mode branches.
template <int NORM, bool ROT, typename QOutT, typename CacheT>
__global__ void __launch_bounds__(STREAM_THREADS, 1)
append_lean_kernel(const __grid_constant__ AppendArgs a, int tb, int stage_bytes) {
  constexpr int D = 128, HALF = 64;
  constexpr int NC = STREAM_CONSUMERS;
  constexpr int APT = (STREAM_ANGLES + NC * 32 - 1) / (NC * 32);
  static_assert((NC * 32) % HALF == 0, "a thread keeps one angle slot across its angles");
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[STREAM_STAGES], empty[STREAM_STAGES];
  __shared__ __align__(16) float s_cs[STREAM_STAGES][2][STREAM_ANGLES];
  __shared__ int32_t s_slot[STREAM_STAGES][STREAM_ANGLES / 32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tb = (a.T + tb - 1) / tb;
  const int items = a.N * n_tb;
  const int64_t tok_q = (int64_t)a.Hq * D, tok_kv = (int64_t)a.Hkv * D;
  if (threadIdx.x == 0) {
    for (int st = 0; st < STREAM_STAGES; ++st) { mbar_init(&full[st], 1); mbar_init(&empty[st], NC); }
    fence_mbar_init();
  }
  const int ct = threadIdx.x;
  const int my_j = ct % HALF;
  const float my_ih = a.rope.inv_hi[my_j], my_il = a.rope.inv_lo[my_j];
  const double my_inv = a.rope.inv[my_j];
  const int my_axis = a.rope.axis[my_j];
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();

  if (warp == NC) {                                     // ---- producer (as the general form) ----
    if (lane == 0) {
      int k = 0;
      for (int it = blockIdx.x; it < items; it += gridDim.x, ++k) {
        const int st = k % STREAM_STAGES;
        if (k >= STREAM_STAGES && !mbar_wait_bounded(&empty[st], (uint32_t)((k / STREAM_STAGES - 1) & 1))) break;
        const int n = it / n_tb, t0 = (it % n_tb) * tb, nt = min(tb, a.T - t0);
        const int64_t tok = (int64_t)n * a.T + t0;
        const uint32_t bq = (uint32_t)(nt * tok_q * 4), bkv = (uint32_t)(nt * tok_kv * 4);
        const uint32_t bw = NORM ? 2u * D * 4u : 0u;
        unsigned char* dst = ring + (size_t)st * stage_bytes;
        mbar_arrive_expect_tx(&full[st], bq + 2 * bkv + bw);
        bulk_g2s(dst, reinterpret_cast<const float*>(a.q) + tok * tok_q, bq, &full[st]);
        bulk_g2s(dst + (size_t)tb * tok_q * 4, reinterpret_cast<const float*>(a.k) + tok * tok_kv, bkv, &full[st]);
        bulk_g2s(dst + (size_t)tb * (tok_q + tok_kv) * 4, reinterpret_cast<const float*>(a.v) + tok * tok_kv, bkv,
                 &full[st]);
        if (NORM) {
          unsigned char* wdst = dst + (size_t)tb * (tok_q + 2 * tok_kv) * 4;
          bulk_g2s(wdst, a.q_w + (int64_t)n * a.w_stride, D * 4, &full[st]);
          bulk_g2s(wdst + D * 4, a.k_w + (int64_t)n * a.w_stride, D * 4, &full[st]);
        }
      }
      for (int j = max(0, k - STREAM_STAGES); j < k; ++j)
        mbar_wait_bounded(&full[j % STREAM_STAGES], (uint32_t)((j / STREAM_STAGES) & 1));
    }
    return;
  }

  // ---- consumers ----
  const int hw = lane >> 4;                             // row of the pair
  const int o1 = 4 * (lane & 15), o2 = o1 + HALF;
  const int pq = a.Hq / 2, pk = a.Hkv / 2, ppt = pq + 2 * pk;   // row pairs per token
  auto load_meta = [&](int it, int32_t (&p)[APT], int32_t& slot) {
    if (it >= items) return;
    const int n = it / n_tb, t0 = (it % n_tb) * tb, nt = min(tb, a.T - t0);
    if (ct < nt) slot = a.slot[(int64_t)n * a.slot_stride + t0 + ct];
    if constexpr (ROT) {
#pragma unroll
      for (int i = 0; i < APT; ++i) {
        const int tt = (ct + i * NC * 32) / HALF;
        if (tt < nt) p[i] = a.pos[(int64_t)n * a.pos_stride + (int64_t)(t0 + tt) * a.rope.n_axes + my_axis];
      }
    }
  };
  int32_t p_next[APT], slot_next = 0;
#pragma unroll
  for (int i = 0; i < APT; ++i) p_next[i] = 0;
  load_meta(blockIdx.x, p_next, slot_next);
  int k = 0;
  for (int it = blockIdx.x; it < items; it += gridDim.x, ++k) {
    const int st = k % STREAM_STAGES;
    const int n = it / n_tb, t0 = (it % n_tb) * tb, nt = min(tb, a.T - t0);
    int32_t p_cur[APT];
#pragma unroll
    for (int i = 0; i < APT; ++i) p_cur[i] = p_next[i];
    if (ct < nt) s_slot[st][ct] = slot_next;
    load_meta(it + gridDim.x, p_next, slot_next);
    if constexpr (ROT) {
#pragma unroll
      for (int i = 0; i < APT; ++i) {
        const int idx = ct + i * NC * 32;
        if (idx / HALF < nt) rope_cos_sin(p_cur[i], my_ih, my_il, my_inv, &s_cs[st][0][idx], &s_cs[st][1][idx]);
      }
    }
    const bool landed = mbar_wait_bounded(&full[st], (uint32_t)((k / STREAM_STAGES) & 1));
    if (!consumers_all(landed)) break;
    const float* sq = reinterpret_cast<const float*>(ring + (size_t)st * stage_bytes);
    const float* sk = sq + (size_t)tb * tok_q;
    const float* sv = sk + (size_t)tb * tok_kv;
    float4 wql = make_float4(1.f, 1.f, 1.f, 1.f), wqh = wql, wkl = wql, wkh = wql;
    if (NORM) {
      const float* swq = sv + (size_t)tb * tok_kv;
      wql = *reinterpret_cast<const float4*>(swq + o1); wqh = *reinterpret_cast<const float4*>(swq + o2);
      wkl = *reinterpret_cast<const float4*>(swq + D + o1); wkh = *reinterpret_cast<const float4*>(swq + D + o2);
    }
    const int64_t tok0 = (int64_t)n * a.T + t0;
    int tt = 0, pi = warp;
    while (pi >= ppt) { pi -= ppt; ++tt; }
    for (; tt < nt;) {
      const int kind = pi < pq ? 0 : (pi < pq + pk ? 1 : 2);
      const int head = 2 * (kind == 0 ? pi : (kind == 1 ? pi - pq : pi - pq - pk)) + hw;
      const float* src = kind == 0 ? sq + ((int64_t)tt * a.Hq + head) * D
                       : (kind == 1 ? sk : sv) + ((int64_t)tt * a.Hkv + head) * D;
      float4 lo = *reinterpret_cast<const float4*>(src + o1);
      float4 hi = *reinterpret_cast<const float4*>(src + o2);
      if (kind < 2) {
        const float4 wl = kind == 0 ? wql : wkl, wh = kind == 0 ? wqh : wkh;
        auto norm = [&]() {
          float ss = lo.x * lo.x;
          ss = fmaf(lo.y, lo.y, ss); ss = fmaf(lo.z, lo.z, ss); ss = fmaf(lo.w, lo.w, ss);
          float s2 = hi.x * hi.x;
          s2 = fmaf(hi.y, hi.y, s2); s2 = fmaf(hi.z, hi.z, s2); s2 = fmaf(hi.w, hi.w, s2);
          ss += s2;
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
          const float r = rsqrtf(ss * (1.0f / (float)D) + a.eps);
          lo.x *= r * wl.x; lo.y *= r * wl.y; lo.z *= r * wl.z; lo.w *= r * wl.w;
          hi.x *= r * wh.x; hi.y *= r * wh.y; hi.z *= r * wh.z; hi.w *= r * wh.w;
        };
        if (NORM == 1) norm();
        if constexpr (ROT) {
          const float4 c = *reinterpret_cast<const float4*>(&s_cs[st][0][tt * HALF + o1]);
          const float4 sn = *reinterpret_cast<const float4*>(&s_cs[st][1][tt * HALF + o1]);
          float l0 = lo.x, h0 = hi.x;
          lo.x = fmaf(-h0, sn.x, l0 * c.x); hi.x = fmaf(l0, sn.x, h0 * c.x);
          l0 = lo.y; h0 = hi.y;
          lo.y = fmaf(-h0, sn.y, l0 * c.y); hi.y = fmaf(l0, sn.y, h0 * c.y);
          l0 = lo.z; h0 = hi.z;
          lo.z = fmaf(-h0, sn.z, l0 * c.z); hi.z = fmaf(l0, sn.z, h0 * c.z);
          l0 = lo.w; h0 = hi.w;
          lo.w = fmaf(-h0, sn.w, l0 * c.w); hi.w = fmaf(l0, sn.w, h0 * c.w);
        }
        if (NORM == 2) norm();
      }
      const float yl[4] = {lo.x, lo.y, lo.z, lo.w}, yh[4] = {hi.x, hi.y, hi.z, hi.w};
      if (kind == 0) {
        QOutT* dst = reinterpret_cast<QOutT*>(a.q_out) + ((tok0 + tt) * a.Hq + head) * D;
        store4(dst + o1, yl);
        store4(dst + o2, yh);
      } else {
        const int32_t slot = s_slot[st][tt];
        if (slot >= 0 && slot < a.capacity) {
          CacheT* dst = reinterpret_cast<CacheT*>(kind == 1 ? a.kc : a.vc) + (int64_t)n * a.inst_stride +
                        ((int64_t)head * a.capacity + slot) * D;
          store4(dst + o1, yl);
          store4(dst + o2, yh);
        }
      }
      pi += NC;
      while (pi >= ppt) { pi -= ppt; ++tt; }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
}

template <int NORM, bool ROT, typename QOutT, typename CacheT>
cudaError_t launch_lean(const AppendArgs& a, int tb, int stage, cudaStream_t s) {
  static DeviceOnce configured;
  if (!configured.done()) {
    const cudaError_t e = cudaFuncSetAttribute(append_lean_kernel<NORM, ROT, QOutT, CacheT>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(STREAM_STAGES * (STREAM_STAGE_MAX + 2 * 128 * sizeof(float))));
    if (e != cudaSuccess) return e;
    configured.mark();
  }
  const int64_t items = (int64_t)a.N * ((a.T + tb - 1) / tb);
  const int grid = (int)std::min<int64_t>(items, append_num_sms());
  return launch_pdl(append_lean_kernel<NORM, ROT, QOutT, CacheT>, dim3(grid), dim3(STREAM_THREADS),
                    (size_t)STREAM_STAGES * stage, s, a, tb, stage);
}

template <typename QOutT, typename CacheT>
cudaError_t launch_lean_modes(const AppendArgs& a, int tb, int stage, cudaStream_t s) {
  const bool rot = a.rope.kind == KVA_ROPE_1D || a.rope.kind == KVA_ROPE_SECTIONS;
  const int norm = a.q_w == nullptr ? 0 : (a.after_rope ? 2 : 1);
  if (rot) {
    if (norm == 1) return launch_lean<1, true, QOutT, CacheT>(a, tb, stage, s);
    if (norm == 2) return launch_lean<2, true, QOutT, CacheT>(a, tb, stage, s);
    return launch_lean<0, true, QOutT, CacheT>(a, tb, stage, s);
  }
  if (norm == 1) return launch_lean<1, false, QOutT, CacheT>(a, tb, stage, s);
  if (norm == 2) return launch_lean<2, false, QOutT, CacheT>(a, tb, stage, s);
  return launch_lean<0, false, QOutT, CacheT>(a, tb, stage, s);
}

template <int D, typename InT, typename QOutT, typename CacheT>
cudaError_t launch_tokens(const AppendArgs& a, cudaStream_t s) {
  if constexpr (D == 72) {
    dim3 grid(a.T, a.N);
    append_kernel<D, InT, QOutT, CacheT><<<grid, APPEND_THREADS, 0, s>>>(a);
    return cudaGetLastError();
  } else {
    const int64_t per_tok = (int64_t)(a.Hq + 2 * a.Hkv) * D * sizeof(InT);
    const int tb_max = STREAM_ANGLES / (D / 2);
    const int64_t w_bytes = 2 * D * sizeof(float);            // q and k norm weights
    const int tb = (int)std::min<int64_t>(tb_max, std::max<int64_t>(1, STREAM_STAGE_MAX / per_tok));
    const int64_t items = (int64_t)a.N * ((a.T + tb - 1) / tb);
    if (a.T >= tb && items >= 2 * append_num_sms() && tb * per_tok <= STREAM_STAGE_MAX) {
      const int stage = (int)(tb * per_tok + w_bytes);
      if constexpr (D == 128 && sizeof(InT) == 4) {
        // the lean form: rotate-half over the whole head (or none) and even head counts
        const bool lean_rope = a.rope.kind == KVA_ROPE_1D || a.rope.kind == KVA_ROPE_SECTIONS ||
                               a.rope.kind == KVA_ROPE_NONE;
        if (lean_rope && a.Hq % 2 == 0 && a.Hkv % 2 == 0) return launch_lean_modes<QOutT, CacheT>(a, tb, stage, s);
      }
      const size_t smem = (size_t)STREAM_STAGES * stage;
      static DeviceOnce configured;                 // one attribute per template instance
      if (!configured.done()) {
        const cudaError_t e = cudaFuncSetAttribute(append_stream_kernel<D, InT, QOutT, CacheT>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)(STREAM_STAGES * (STREAM_STAGE_MAX + w_bytes)));
        if (e != cudaSuccess) return e;
        configured.mark();
      }
      const int grid = (int)std::min<int64_t>(items, append_num_sms());
      return launch_pdl(append_stream_kernel<D, InT, QOutT, CacheT>, dim3(grid), dim3(STREAM_THREADS), smem, s, a,
                        tb, stage);
    }
    // the most tokens per CTA that still leaves about four CTAs per SM
    int tpc = 8;
    while (tpc > 1 && (int64_t)((a.T + tpc - 1) / tpc) * a.N < 4 * append_num_sms()) tpc >>= 1;
    dim3 grid((a.T + tpc - 1) / tpc, a.N);
    return launch_pdl(append_warp_kernel<D, InT, QOutT, CacheT>, grid, dim3(APPEND_THREADS), 0, s, a, tpc);
  }
}

template <int D, typename InT, typename QOutT>
cudaError_t launch_cache(const AppendArgs& a, kva_dtype cache_dtype, cudaStream_t s) {
  if (cache_dtype == KVA_BF16) return launch_tokens<D, InT, QOutT, bf16_t>(a, s);
  return launch_tokens<D, InT, QOutT, float>(a, s);
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
