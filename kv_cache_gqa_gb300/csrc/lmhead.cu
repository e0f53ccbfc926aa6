// Kernel (d): tied lm_head GEMV + greedy argmax with ties toward the lowest id.
//
// Streaming form for small batches: each warp owns a run of vocabulary rows, reads each
// row once with 128-bit loads, dots it with the batch's hidden vectors (staged in shared
// memory), and keeps a running (logit, id) best per batch row.  The CTA folds its warps'
// bests into one 64-bit key per batch row (order-preserving logit bits above ~id) and
// publishes it with atomicMax; the last CTA to finish turns the keys into ids and clears
// the workspace for the next call.
//
// Method: greedy decoding takes the argmax of final-norm hidden . vocab row over the whole
// tied table (Youtu-VL-4B ncnn port, step 6 and "decoding and sampling"; one
// [vocab, hidden] copy: HunyuanOCR v1.5 ncnn port, section 3.4); the vocab is clamped to
// the logits length (Penguin-VL ncnn port, section 4.1).
#include "common.cuh"
#include "launch.h"

namespace kva {

namespace {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int ROWS_PER_WARP = 4;
constexpr int ROWS_PER_CTA = WARPS * ROWS_PER_WARP;
constexpr int BG = 8;                 // batch rows staged per CTA
constexpr int MAX_H = 4096;

template <typename WT>
__global__ void __launch_bounds__(THREADS)
lmhead_kernel(const __grid_constant__ LmheadArgs a) {
  constexpr int ES = ElemSize<WT>::value;
  constexpr int CH = 16 / ES;                    // elements per 16-byte chunk
  extern __shared__ __align__(16) float sh[];    // [nb][H]
  __shared__ unsigned long long s_best[WARPS][BG];
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b0 = blockIdx.y * BG;
  const int nb = min(BG, a.B - b0);
  const int H = a.H;

  for (int i = tid; i < nb * H; i += THREADS) sh[i] = a.h[(int64_t)b0 * H + i];
  __syncthreads();

  float best_v[BG];
  int best_i[BG];
#pragma unroll
  for (int b = 0; b < BG; ++b) { best_v[b] = -INFINITY; best_i[b] = 0x7fffffff; }

  const int row0 = blockIdx.x * ROWS_PER_CTA + warp * ROWS_PER_WARP;
  const int n_chunks = H / CH;
  for (int r = 0; r < ROWS_PER_WARP; ++r) {
    const int row = row0 + r;
    if (row >= a.V) break;
    const WT* wrow = reinterpret_cast<const WT*>(a.W) + (int64_t)row * H;
    float part[BG];
#pragma unroll
    for (int b = 0; b < BG; ++b) part[b] = 0.f;
    for (int c = lane; c < n_chunks; c += 32) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(wrow) + c);
      float x[8];
      int nx;
      if constexpr (ES == 2) {
        x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
        x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
        nx = 8;
      } else {
        x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
        nx = 4;
      }
#pragma unroll
      for (int b = 0; b < BG; ++b) {
        if (b < nb) {
          const float* hb = sh + b * H + c * CH;
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e < nx) part[b] = fmaf(x[e], hb[e], part[b]);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < BG; ++b) {
      float v = part[b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
      if (b < nb) {
        if (v > best_v[b]) { best_v[b] = v; best_i[b] = row; }   // rows ascend: keeps lowest id on ties
        if (a.logits && lane == 0) a.logits[(int64_t)(b0 + b) * a.V + row] = v;
      }
    }
  }

  if (lane == 0) {
#pragma unroll
    for (int b = 0; b < BG; ++b)
      s_best[warp][b] = best_i[b] == 0x7fffffff ? 0ull : argmax_key(best_v[b], (uint32_t)best_i[b]);
  }
  __syncthreads();
  if (tid < nb) {
    unsigned long long k = 0ull;
    for (int w = 0; w < WARPS; ++w) k = max(k, s_best[w][tid]);
    if (k) atomicMax(&a.best[b0 + tid], k);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned total = gridDim.x * gridDim.y;
    s_last = atomicAdd(a.counter, 1u) == total - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int b = tid; b < a.B; b += THREADS) {
    const unsigned long long k = atomicExch(&a.best[b], 0ull);
    a.out_ids[b] = (int32_t)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
    if (a.out_max) a.out_max[b] = float_from_order_bits((uint32_t)(k >> 32));
  }
  if (tid == 0) *a.counter = 0u;
}

template <typename WT>
cudaError_t launch_t(const LmheadArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(float) * (size_t)BG * a.H;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(lmhead_kernel<WT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(float) * BG * MAX_H));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid((a.V + ROWS_PER_CTA - 1) / ROWS_PER_CTA, (a.B + BG - 1) / BG);
  lmhead_kernel<WT><<<grid, THREADS, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t lmhead_workspace_bytes(int B) {
  return 256 + sizeof(unsigned long long) * (size_t)(B > 0 ? B : 0);
}

int lmhead_max_hidden() { return MAX_H; }

cudaError_t launch_lmhead(const LmheadArgs& a, kva_dtype w_dtype, cudaStream_t s) {
  if (w_dtype == KVA_BF16) return launch_t<bf16_t>(a, s);
  return launch_t<float>(a, s);
}

}  // namespace kva
