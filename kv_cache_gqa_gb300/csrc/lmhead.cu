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
#include <algorithm>

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
  if (a.norm_w) {                                 // final RMSNorm of each staged row
    __shared__ float s_r[BG];
    for (int b = warp; b < nb; b += WARPS) {
      float ss = 0.f;
      for (int i = lane; i < H; i += 32) ss = fmaf(sh[b * H + i], sh[b * H + i], ss);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
      if (lane == 0) s_r[b] = rsqrtf(ss / (float)H + a.eps);
    }
    __syncthreads();
    for (int i = tid; i < nb * H; i += THREADS) sh[i] *= s_r[i / H] * a.norm_w[i % H];
    __syncthreads();
  }

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

// Final RMSNorm of h held in registers: lane owns elements (c * 32 + lane) * 8 + e, so a warp
// holds the whole vector and the sum of squares is one warp reduction.
template <int NCH>
__device__ __forceinline__ void norm_h_regs(float (&hv)[NCH][8], const float* w, float eps, int H, int lane) {
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < NCH; ++c)
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(hv[c][e], hv[c][e], ss);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
  const float r = rsqrtf(ss / (float)H + eps);
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const float4 u = __ldg(reinterpret_cast<const float4*>(w) + (c * 32 + lane) * 2);
    const float4 v = __ldg(reinterpret_cast<const float4*>(w) + (c * 32 + lane) * 2 + 1);
    hv[c][0] *= r * u.x; hv[c][1] *= r * u.y; hv[c][2] *= r * u.z; hv[c][3] *= r * u.w;
    hv[c][4] *= r * v.x; hv[c][5] *= r * v.y; hv[c][6] *= r * v.z; hv[c][7] *= r * v.w;
  }
}

// ---------------------------------------------------------------------------------
// Batch-1 fast path: a grid-stride GEMV over groups of 4 consecutive vocabulary rows per
// warp.  All 16-byte loads of a group (4 rows x H/256 chunks per lane) are issued before
// any arithmetic, so each lane keeps 4*H/128 bytes in flight; h lives in registers.
// ---------------------------------------------------------------------------------
constexpr int FAST_ROWS = 4;              // rows per warp iteration
constexpr int FAST_THREADS = 256;
constexpr int FAST_WARPS = FAST_THREADS / 32;

template <int H>
__global__ void __launch_bounds__(FAST_THREADS)
lmhead_b1_kernel(const __grid_constant__ LmheadArgs a) {
  constexpr int NCH = H / 256;            // 16-byte bf16 chunks per lane per row
  __shared__ unsigned long long s_best[FAST_WARPS];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  float hv[NCH][8];
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const float4 u = __ldg(reinterpret_cast<const float4*>(a.h) + (c * 32 + lane) * 2);
    const float4 w = __ldg(reinterpret_cast<const float4*>(a.h) + (c * 32 + lane) * 2 + 1);
    hv[c][0] = u.x; hv[c][1] = u.y; hv[c][2] = u.z; hv[c][3] = u.w;
    hv[c][4] = w.x; hv[c][5] = w.y; hv[c][6] = w.z; hv[c][7] = w.w;
  }
  if (a.norm_w) norm_h_regs<NCH>(hv, a.norm_w, a.eps, H, lane);

  float best_v = -INFINITY;
  int best_i = 0x7fffffff;
  const int n_groups = (a.V + FAST_ROWS - 1) / FAST_ROWS;
  const int gw = blockIdx.x * FAST_WARPS + warp, n_warps = gridDim.x * FAST_WARPS;
  const uint4* W = reinterpret_cast<const uint4*>(a.W);
  for (int grp = gw; grp < n_groups; grp += n_warps) {
    const int r0 = grp * FAST_ROWS;
    uint4 w[FAST_ROWS][NCH];
#pragma unroll
    for (int r = 0; r < FAST_ROWS; ++r) {
      const int row = min(r0 + r, a.V - 1);          // clamp the ragged last group (value unused)
#pragma unroll
      for (int c = 0; c < NCH; ++c) w[r][c] = __ldcs(W + (int64_t)row * (H / 8) + c * 32 + lane);
    }
    float dot[FAST_ROWS];
#pragma unroll
    for (int r = 0; r < FAST_ROWS; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const uint4 u = w[r][c];
        acc = fmaf(bf16_lo(u.x), hv[c][0], acc); acc = fmaf(bf16_hi(u.x), hv[c][1], acc);
        acc = fmaf(bf16_lo(u.y), hv[c][2], acc); acc = fmaf(bf16_hi(u.y), hv[c][3], acc);
        acc = fmaf(bf16_lo(u.z), hv[c][4], acc); acc = fmaf(bf16_hi(u.z), hv[c][5], acc);
        acc = fmaf(bf16_lo(u.w), hv[c][6], acc); acc = fmaf(bf16_hi(u.w), hv[c][7], acc);
      }
      dot[r] = acc;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int r = 0; r < FAST_ROWS; ++r) dot[r] += __shfl_xor_sync(FULL_MASK, dot[r], o);
#pragma unroll
    for (int r = 0; r < FAST_ROWS; ++r) {
      const int row = r0 + r;
      if (row < a.V) {
        if (dot[r] > best_v) { best_v = dot[r]; best_i = row; }   // rows ascend within a warp
        if (a.logits && lane == r) a.logits[row] = dot[r];
      }
    }
  }

  if (lane == 0) s_best[warp] = best_i == 0x7fffffff ? 0ull : argmax_key(best_v, (uint32_t)best_i);
  __syncthreads();
  if (tid == 0) {
    unsigned long long k = 0ull;
    for (int w2 = 0; w2 < FAST_WARPS; ++w2) k = max(k, s_best[w2]);
    if (k) atomicMax(&a.best[0], k);
    __threadfence();
    s_last = atomicAdd(a.counter, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  if (tid == 0) {
    __threadfence();
    const unsigned long long k = atomicExch(&a.best[0], 0ull);
    a.out_ids[0] = (int32_t)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
    if (a.out_max) a.out_max[0] = float_from_order_bits((uint32_t)(k >> 32));
    *a.counter = 0u;
  }
}

// ---------------------------------------------------------------------------------
// Batch-1 pipelined path: one CTA per SM streams every P-th 32 KB stage of the table (16
// contiguous rows) through a 5-stage shared-memory ring, one bulk copy per stage.  Bytes in
// flight cost no registers, so each SM keeps ~160 KB moving.
// The 8 warps reduce the staged rows with conflict-free 128-bit shared-memory reads.
// ---------------------------------------------------------------------------------
constexpr int PIPE_STAGE_BYTES = 32768;
constexpr int PIPE_STAGES = 5;
constexpr int PIPE_THREADS = 256;
constexpr int PIPE_WARPS = PIPE_THREADS / 32;

template <int H>
__global__ void __launch_bounds__(PIPE_THREADS, 1)
lmhead_b1_pipe_kernel(const __grid_constant__ LmheadArgs a, int rows_per_cta) {
  constexpr int ROWB = H * 2;
  constexpr int RPS = PIPE_STAGE_BYTES / ROWB;         // rows per stage
  constexpr int NCH = H / 256;                         // 16-byte chunks per lane per row
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[PIPE_STAGES], empty[PIPE_STAGES];
  __shared__ unsigned long long s_best[PIPE_WARPS];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // CTA b streams the table's 32 KB stages b, b + P, b + 2P, ... (P CTAs): at any moment the
  // grid reads one compact region of the table.  Against one contiguous slice per CTA this
  // measured 0.7 us slower per launch alone but 1% faster over the whole Qwen3-shaped job,
  // where each launch follows a decode step (15.53 -> 15.38 ms).
  (void)rows_per_cta;
  const int P = gridDim.x, bidx = blockIdx.x;
  const int tot_st = (a.V + RPS - 1) / RPS;
  const int n_st = bidx < tot_st ? (tot_st - bidx + P - 1) / P : 0;
  const unsigned char* W = reinterpret_cast<const unsigned char*>(a.W);
  auto issue = [&](int it) {
    const int rs = (bidx + it * P) * RPS;
    const uint32_t bytes = (uint32_t)(min(RPS, a.V - rs) * ROWB);
    mbar_arrive_expect_tx(&full[it % PIPE_STAGES], bytes);
    bulk_g2s(ring + (it % PIPE_STAGES) * PIPE_STAGE_BYTES, W + (int64_t)rs * ROWB, bytes, &full[it % PIPE_STAGES]);
  };
  if (tid == 0) {
    for (int st = 0; st < PIPE_STAGES; ++st) { mbar_init(&full[st], 1); mbar_init(&empty[st], PIPE_WARPS); }
    fence_mbar_init();
  }
  // Warm L2 with the first stages of this CTA's slice and with h while the kernel before this
  // one drains (prefetches return no data, so they may run before the wait: a write by that
  // kernel still lands in L2, the point of coherence, where the copies after the wait read it)
  if (tid < PIPE_STAGES && tid < n_st) {
    const int rs = (bidx + tid * P) * RPS;
    bulk_prefetch_l2(W + (int64_t)rs * ROWB, (uint32_t)(min(RPS, a.V - rs) * ROWB));
  } else if (tid >= 32 && tid < 32 + H * 4 / 128) {
    prefetch_l2(reinterpret_cast<const char*>(a.h) + (tid - 32) * 128);
  }
  griddep_wait();                               // h (and the table) are complete from here on
  griddep_launch_dependents();
  if (tid == 0)
    for (int it = 0; it < PIPE_STAGES && it < n_st; ++it) issue(it);
  float hv[NCH][8];
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const float4 u = __ldg(reinterpret_cast<const float4*>(a.h) + (c * 32 + lane) * 2);
    const float4 w = __ldg(reinterpret_cast<const float4*>(a.h) + (c * 32 + lane) * 2 + 1);
    hv[c][0] = u.x; hv[c][1] = u.y; hv[c][2] = u.z; hv[c][3] = u.w;
    hv[c][4] = w.x; hv[c][5] = w.y; hv[c][6] = w.z; hv[c][7] = w.w;
  }
  if (a.norm_w) norm_h_regs<NCH>(hv, a.norm_w, a.eps, H, lane);
  __syncthreads();

  float best_v = -INFINITY;
  int best_i = 0x7fffffff;
  bool ok = true;
  for (int it = 0; it < n_st; ++it) {
    const int st = it % PIPE_STAGES;
    if (!__all_sync(FULL_MASK, mbar_wait_bounded(&full[st], (uint32_t)((it / PIPE_STAGES) & 1)))) { ok = false; break; }
    const int rs = (bidx + it * P) * RPS;
    const int nr = min(RPS, a.V - rs);
    const unsigned char* base = ring + st * PIPE_STAGE_BYTES;
    for (int rr = warp; rr < nr; rr += PIPE_WARPS) {
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const uint4 u = *reinterpret_cast<const uint4*>(base + rr * ROWB + (c * 32 + lane) * 16);
        acc = fmaf(bf16_lo(u.x), hv[c][0], acc); acc = fmaf(bf16_hi(u.x), hv[c][1], acc);
        acc = fmaf(bf16_lo(u.y), hv[c][2], acc); acc = fmaf(bf16_hi(u.y), hv[c][3], acc);
        acc = fmaf(bf16_lo(u.z), hv[c][4], acc); acc = fmaf(bf16_hi(u.z), hv[c][5], acc);
        acc = fmaf(bf16_lo(u.w), hv[c][6], acc); acc = fmaf(bf16_hi(u.w), hv[c][7], acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL_MASK, acc, o);
      const int row = rs + rr;
      if (acc > best_v) { best_v = acc; best_i = row; }          // rows ascend within a warp
      if (a.logits && lane == 0) a.logits[row] = acc;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    if (tid == 0 && it + PIPE_STAGES < n_st) {
      // refill this stage once every warp has released it
      if (!mbar_wait_bounded(&empty[st], (uint32_t)((it / PIPE_STAGES) & 1))) { ok = false; }
      else issue(it + PIPE_STAGES);
    }
  }

  if (lane == 0) s_best[warp] = (!ok || best_i == 0x7fffffff) ? 0ull : argmax_key(best_v, (uint32_t)best_i);
  __syncthreads();
  if (tid == 0) {
    unsigned long long k = 0ull;
    for (int w2 = 0; w2 < PIPE_WARPS; ++w2) k = max(k, s_best[w2]);
    if (k) atomicMax(&a.best[0], k);
    __threadfence();
    s_last = atomicAdd(a.counter, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  if (tid == 0) {
    __threadfence();
    const unsigned long long k = atomicExch(&a.best[0], 0ull);
    a.out_ids[0] = k ? (int32_t)(0xffffffffu - (uint32_t)(k & 0xffffffffull)) : -1;
    if (a.out_max) a.out_max[0] = float_from_order_bits((uint32_t)(k >> 32));
    *a.counter = 0u;
  }
}

int num_sms_lm() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

template <int H>
cudaError_t launch_b1(const LmheadArgs& a, cudaStream_t s) {
  static int per_sm = 0;   // resident CTAs per SM: the grid-stride grid fills the GPU exactly once
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lmhead_b1_kernel<H>, FAST_THREADS, 0) !=
            cudaSuccess || per_sm <= 0)
      per_sm = 2;
  }
  const int groups = (a.V + FAST_ROWS - 1) / FAST_ROWS;
  const int want = (groups + FAST_WARPS - 1) / FAST_WARPS;
  const int grid = std::max(1, std::min(want, num_sms_lm() * per_sm));
  lmhead_b1_kernel<H><<<grid, FAST_THREADS, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename WT>
cudaError_t launch_t(const LmheadArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(float) * (size_t)BG * a.H;
  static DeviceOnce configured;
  if (!configured.done()) {
    cudaError_t e = cudaFuncSetAttribute(lmhead_kernel<WT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(float) * BG * MAX_H));
    if (e != cudaSuccess) return e;
    configured.mark();
  }
  dim3 grid((a.V + ROWS_PER_CTA - 1) / ROWS_PER_CTA, (a.B + BG - 1) / BG);
  lmhead_kernel<WT><<<grid, THREADS, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool lmhead_tc_supports(int B, int H);
size_t lmhead_tc_hb_bytes(int B, int H);
cudaError_t launch_lmhead_tc(const LmheadArgs& a, uint16_t* hb, cudaStream_t s);

// Workspace: [counter, 256 B][packed best keys, 8 B per batch row, rounded to 256 B]
//            [bf16 hi/lo copy of h for the batched tensor-core path]
size_t lmhead_zero_bytes(int B) {
  return 256 + (sizeof(unsigned long long) * (size_t)(B > 0 ? B : 0) + 255) / 256 * 256;
}

size_t lmhead_workspace_bytes(int B, int H) {
  return lmhead_zero_bytes(B) + (B >= 2 ? lmhead_tc_hb_bytes(B, H) : 0);
}

int lmhead_max_hidden() { return MAX_H; }

template <int H>
cudaError_t launch_b1_pipe(const LmheadArgs& a, cudaStream_t s) {
  static DeviceOnce configured;
  if (!configured.done()) {
    cudaError_t e = cudaFuncSetAttribute(lmhead_b1_pipe_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PIPE_STAGES * PIPE_STAGE_BYTES);
    if (e != cudaSuccess) return e;
    configured.mark();
  }
  const int grid = num_sms_lm();
  const int rows_per_cta = (a.V + grid - 1) / grid;
  return launch_pdl(lmhead_b1_pipe_kernel<H>, dim3(grid), dim3(PIPE_THREADS), (size_t)(PIPE_STAGES * PIPE_STAGE_BYTES), s,
                    a, rows_per_cta);
}

cudaError_t launch_lmhead(const LmheadArgs& a, kva_dtype w_dtype, void* hb_scratch, cudaStream_t s,
                          unsigned* n_launches) {
  *n_launches = 1;
  if (w_dtype == KVA_BF16 && a.B == 1) {
    switch (a.H) {
      case 1024: return launch_b1_pipe<1024>(a, s);
      case 2048: return launch_b1_pipe<2048>(a, s);
      case 2560: return launch_b1<2560>(a, s);
      case 4096: return launch_b1_pipe<4096>(a, s);
      default: break;
    }
  }
  if (w_dtype == KVA_BF16 && hb_scratch && lmhead_tc_supports(a.B, a.H)) {
    *n_launches = 2;
    return launch_lmhead_tc(a, static_cast<uint16_t*>(hb_scratch), s);
  }
  if (w_dtype == KVA_BF16) return launch_t<bf16_t>(a, s);
  return launch_t<float>(a, s);
}

}  // namespace kva
