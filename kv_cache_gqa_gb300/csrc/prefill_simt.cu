// Kernel (b), FFMA form: flash-style prefill attention in fp32 on the CUDA cores.
//
// This is the path for fp32 caches (where the contract asks for 1e-5 relative error, which
// bf16 tensor-core operands cannot give) and for head dims the tensor-core kernel does not
// tile, including asymmetric caches (K rows Dk = 192 wide, V rows Dv = 128: an MLA layer
// expanded per head, Youtu-VL-4B ncnn port, section 6).  One CTA per (64- or 48-query tile, query
// head, instance): Q, K and V tiles are widened
// to fp32 in shared memory; each warp owns 8 query rows, computes their 8x64 score block
// as a register tile, applies the mask, runs the online softmax (max -> subtract -> exp
// -> sum, final divide) and accumulates P.V with each lane owning head-dim columns.
// Key tiles that the mask hides entirely (causal future, other windows) are skipped.
//
// Method: QK^T*scale + mask, softmax, times V (Youtu-VL-4B ncnn port, implementation
// difficulty 3), parallel causal prefill over the fixed window (step 7), block-diagonal
// window mask or full attention of the vision layers (step 3), fused in one kernel with
// intermediates kept on chip (MNN llm_demo walkthrough, section 5.1).
#include "common.cuh"
#include "launch.h"

namespace kva {

namespace {

// A CTA of W warps owns BQ = 8 W query slots (8 rows per warp); W is 8 (64 rows) or 6 (48 rows,
// chosen on the host when it spreads a one-wave grid more evenly over the SMs).
constexpr int BK = 64;                 // keys per tile
constexpr int RPW = 8;                 // query rows per warp

template <typename T>
__device__ __forceinline__ void load_row_f32(const T* src, float* dst, int D, int tid0, int nthr) {
  for (int e = tid0 * 4; e < D; e += nthr * 4) {
    float4 v;
    v.x = load1(src + e); v.y = load1(src + e + 1); v.z = load1(src + e + 2); v.w = load1(src + e + 3);
    *reinterpret_cast<float4*>(dst + e) = v;
  }
}

// First slot in [0, S) whose segment id equals seg[i] (segments are non-decreasing).
__device__ int seg_lower(const int32_t* seg, int S, int key) {
  int lo = 0, hi = S;
  while (lo < hi) { const int mid = (lo + hi) >> 1; if (seg[mid] < key) lo = mid + 1; else hi = mid; }
  return lo;
}
__device__ int seg_upper(const int32_t* seg, int S, int key) {
  int lo = 0, hi = S;
  while (lo < hi) { const int mid = (lo + hi) >> 1; if (seg[mid] <= key) lo = mid + 1; else hi = mid; }
  return lo;
}

template <int D, int DV, typename T, int WARPS>
// Resident CTAs per SM: one for wide heads (shared memory); three for heads up to 80 wide (the
// 1288-patch vision pass then fits its tiles in one wave: 437 instead of 538 us), two between.
__global__ void __launch_bounds__(WARPS * 32, (D + DV > 256) ? 1 : (D + DV > 160 ? 2 : 3))
prefill_simt_kernel(const __grid_constant__ PrefillArgs a) {
  constexpr int BQ = WARPS * RPW;                    // query slots per CTA
  constexpr int DP = D + 4;                          // padded K row (conflict-free float4)
  constexpr int DPL = (DV + 31) / 32;                // output column groups per lane
  // Value widths of 32 k + 8 (72): each lane owns k full column groups for all 8 rows of its
  // warp and two outputs of the 8-column tail (rows tr0 and tr0 + 1, column 32 k + lane % 8),
  // instead of a (k+1)-th group that only 8 lanes use.
  constexpr bool TAIL8 = (DV % 32 == 8);
  constexpr int NC = TAIL8 ? DV / 32 : DPL;          // column groups per lane
  extern __shared__ __align__(16) float sm[];
  float* sQ = sm;                                    // [BQ][D]
  float* sK = sQ + BQ * D;                           // [BK][DP]
  float* sV = sK + BK * DP;                          // [BK][DV]
  float* sP = sV + BK * DV;                          // [WARPS][BK][RPW]
  __shared__ int s_range[2];
  __shared__ int s_qseg[BQ];

  const int qt = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.Hq / a.Hkv;
  const int g = h / G;
  const int i0 = qt * BQ;
  const int i1 = min(a.S, i0 + BQ);

  const T* Kc = reinterpret_cast<const T*>(a.kc) + (int64_t)n * a.inst_stride + (int64_t)g * a.capacity * D;
  const T* Vc = reinterpret_cast<const T*>(a.vc) + (int64_t)n * a.inst_stride_v + (int64_t)g * a.capacity * DV;
  const T* Qn = reinterpret_cast<const T*>(a.q) + (int64_t)n * a.S * a.Hq * D;

  // ---- key range visible to this tile ----
  if (tid == 0) {
    int lo = 0, hi = a.S;
    if (a.mask == KVA_MASK_CAUSAL) hi = i1;
    else if (a.mask == KVA_MASK_SEGMENT) {
      const int g0 = a.segment[i0], g1 = a.segment[i1 - 1];   // bounds from the launch's table if there
      lo = (unsigned)g0 < (unsigned)a.seg_table ? a.seg_lo[g0] : seg_lower(a.segment, a.S, g0);
      hi = (unsigned)g1 < (unsigned)a.seg_table ? a.seg_hi[g1] : seg_upper(a.segment, a.S, g1);
    } else if (a.mask == KVA_MASK_CAUSAL_SEGMENT) {
      const int g1 = a.segment[i1 - 1];                        // the last row's segment end
      hi = (unsigned)g1 < (unsigned)a.seg_table ? a.seg_hi[g1] : seg_upper(a.segment, a.S, g1);
    }
    s_range[0] = lo; s_range[1] = hi;
  }
  // ---- Q tile (row r(i) of the token-order q holds the query of slot i) ----
  for (int r = warp; r < BQ; r += WARPS) {
    const int i = i0 + r;
    const int row = (i < i1 && a.row_of_slot) ? a.row_of_slot[i] : i;
    if (i < i1 && row >= 0 && row < a.S) {   // a malformed permutation entry reads nothing
      load_row_f32(Qn + ((int64_t)row * a.Hq + h) * D, sQ + r * D, D, lane, 32);
      if (lane == 0) s_qseg[r] = a.segment ? a.segment[i] : 0;
    } else {
      for (int e = lane; e < D; e += 32) sQ[r * D + e] = 0.f;
      if (lane == 0) s_qseg[r] = -1;
    }
  }
  __syncthreads();
  const int k_lo = s_range[0], k_hi = s_range[1];

  float m_run[RPW], l_run[RPW], acc[RPW][NC];
  float acc_t[2] = {0.f, 0.f};              // the tail outputs (TAIL8 only)
  const int tr0 = 2 * (lane >> 3);          // the tail rows of this lane: tr0, tr0 + 1
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    m_run[r] = -INFINITY; l_run[r] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[r][c] = 0.f;
  }
  const int rbase = warp * RPW;            // this warp's first query row in the tile
  float* myP = sP + warp * BK * RPW;

  for (int kt = k_lo - (k_lo % BK); kt < k_hi; kt += BK) {
    __syncthreads();   // previous tile fully consumed
    for (int r = warp; r < BK; r += WARPS) {
      const int j = kt + r;
      if (j < k_hi && j >= 0) {
        load_row_f32(Kc + (int64_t)j * D, sK + r * DP, D, lane, 32);
        load_row_f32(Vc + (int64_t)j * DV, sV + r * DV, DV, lane, 32);
      } else {
        for (int e = lane; e < D; e += 32) sK[r * DP + e] = 0.f;
        for (int e = lane; e < DV; e += 32) sV[r * DV + e] = 0.f;
      }
    }
    __syncthreads();

    // ---- scores: lane owns keys lane and lane+32 for the warp's 8 rows ----
    float s[RPW][2];
#pragma unroll
    for (int r = 0; r < RPW; ++r) { s[r][0] = 0.f; s[r][1] = 0.f; }
#pragma unroll 2
    for (int d = 0; d < D; d += 4) {
      const float4 k0 = *reinterpret_cast<const float4*>(sK + lane * DP + d);
      const float4 k1 = *reinterpret_cast<const float4*>(sK + (lane + 32) * DP + d);
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        const float4 q = *reinterpret_cast<const float4*>(sQ + (rbase + r) * D + d);
        s[r][0] = fmaf(q.x, k0.x, fmaf(q.y, k0.y, fmaf(q.z, k0.z, fmaf(q.w, k0.w, s[r][0]))));
        s[r][1] = fmaf(q.x, k1.x, fmaf(q.y, k1.y, fmaf(q.z, k1.z, fmaf(q.w, k1.w, s[r][1]))));
      }
    }

    // ---- mask + online softmax per row ----
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const int ir = rbase + r;
      const int i = i0 + ir;
      const int qs = s_qseg[ir];
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int j = kt + lane + 32 * u;
        bool ok = (i < i1) && j >= k_lo && j < k_hi;
        if (a.mask == KVA_MASK_CAUSAL) ok = ok && j <= i;
        else if (a.mask == KVA_MASK_SEGMENT) ok = ok && a.segment[j] == qs;
        else if (a.mask == KVA_MASK_CAUSAL_SEGMENT) ok = ok && (j <= i || a.segment[j] == qs);
        s[r][u] = ok ? s[r][u] * a.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[r][u]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, o));
      const float m_new = fmaxf(m_run[r], mx);
      // rows with nothing visible yet keep m = -inf; use 0 as the offset so exp2 stays 0
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(m_run[r] - m_use);
      float sum = 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float p = exp2f(s[r][u] - m_use);
        myP[(lane + 32 * u) * RPW + r] = p;
        sum += p;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL_MASK, sum, o);
      l_run[r] = l_run[r] * alpha + sum;
      m_run[r] = m_new;
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[r][c] *= alpha;
      if (TAIL8 && (r >> 1) == (lane >> 3)) acc_t[r & 1] *= alpha;
    }
    __syncwarp();

    // ---- acc += P V ----
    for (int j = 0; j < BK; ++j) {
      float p[RPW];
#pragma unroll
      for (int r = 0; r < RPW; r += 4) {
        const float4 pv = *reinterpret_cast<const float4*>(myP + j * RPW + r);
        p[r] = pv.x; p[r + 1] = pv.y; p[r + 2] = pv.z; p[r + 3] = pv.w;
      }
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int d = lane + 32 * c;
        const float v = (TAIL8 || d < DV) ? sV[j * DV + d] : 0.f;
#pragma unroll
        for (int r = 0; r < RPW; ++r) acc[r][c] = fmaf(p[r], v, acc[r][c]);
      }
      if (TAIL8) {
        const float2 pt = *reinterpret_cast<const float2*>(myP + j * RPW + tr0);
        const float vt = sV[j * DV + 32 * NC + (lane & 7)];
        acc_t[0] = fmaf(pt.x, vt, acc_t[0]);
        acc_t[1] = fmaf(pt.y, vt, acc_t[1]);
      }
    }
    __syncwarp();
  }

  // ---- normalise and store to the token-order output row ----
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int i = i0 + rbase + r;
    if (i >= i1) continue;
    const int row = a.row_of_slot ? a.row_of_slot[i] : i;
    if (row < 0 || row >= a.S) continue;
    float* o = a.out + (((int64_t)n * a.S + row) * a.Hq + h) * DV;
    const float inv = 1.0f / l_run[r];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int d = lane + 32 * c;
      if (TAIL8 || d < DV) o[d] = acc[r][c] * inv;
    }
    if (TAIL8 && (r >> 1) == (lane >> 3)) o[32 * NC + (lane & 7)] = acc_t[r & 1] * inv;
  }
}

template <int D, int DV, int WARPS>
size_t simt_smem() {
  return sizeof(float) * ((size_t)WARPS * RPW * D + BK * (D + 4) + BK * DV + WARPS * BK * RPW);
}

template <int D, int DV, typename T, int WARPS>
cudaError_t launch_w(const PrefillArgs& a, cudaStream_t s) {
  constexpr int BQ = WARPS * RPW;
  const size_t smem = simt_smem<D, DV, WARPS>();
  static DeviceOnce configured;
  if (!configured.done()) {
    cudaError_t e = cudaFuncSetAttribute(prefill_simt_kernel<D, DV, T, WARPS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured.mark();
  }
  dim3 grid((a.S + BQ - 1) / BQ, a.Hq, a.N);
  prefill_simt_kernel<D, DV, T, WARPS><<<grid, WARPS * 32, smem, s>>>(a);
  return cudaGetLastError();
}

// 48-row CTAs when they lower the rows the busiest SM carries by at least 5% (the 1288-patch
// vision pass: 336 CTAs of 64 rows put 192 rows on some SMs, 432 of 48 rows at most 144; full
// pass 437 -> 389 us), else 64-row CTAs (more warps per CTA, one K/V tile load per 64 rows).
int simt_warps(const PrefillArgs& a) {
  const long long heads = (long long)a.Hq * a.N, sms = decode_num_sms();   // the device's SM count
  const long long rows64 = ((heads * ((a.S + 63) / 64) + sms - 1) / sms) * 64;
  const long long rows48 = ((heads * ((a.S + 47) / 48) + sms - 1) / sms) * 48;
  return rows48 * 100 < rows64 * 95 ? 6 : 8;
}

template <int D, int DV, typename T>
cudaError_t launch_dt(const PrefillArgs& a, cudaStream_t s) {
  return simt_warps(a) == 6 ? launch_w<D, DV, T, 6>(a, s) : launch_w<D, DV, T, 8>(a, s);
}

template <int D, int DV>
cudaError_t launch_d(const PrefillArgs& a, kva_dtype dt, cudaStream_t s) {
  if (dt == KVA_BF16) return launch_dt<D, DV, bf16_t>(a, s);
  return launch_dt<D, DV, float>(a, s);
}

}  // namespace

bool prefill_simt_supports(int Dk, int Dv) {
  return (Dk == Dv && (Dk == 64 || Dk == 72 || Dk == 128)) || (Dk == 192 && Dv == 128);
}

cudaError_t launch_prefill_simt(const PrefillArgs& a, kva_dtype dt, cudaStream_t s) {
  if (a.D == 192 && a.Dv == 128) return launch_d<192, 128>(a, dt, s);
  if (a.D != a.Dv) return cudaErrorInvalidValue;
  switch (a.D) {
    case 64: return launch_d<64, 64>(a, dt, s);
    case 72: return launch_d<72, 72>(a, dt, s);
    case 128: return launch_d<128, 128>(a, dt, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kva
