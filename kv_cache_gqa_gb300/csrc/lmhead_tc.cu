// Kernel (d), batched form on tcgen05: logits = W . h^T for 2..128 hidden vectors, argmax
// fused into the epilogue.
//
// The table W is exact in bf16; h is fp32.  h is split once into two bf16 halves,
// h = h_hi + h_lo (h_lo = bf16(h - h_hi)), which represent it to ~16 significant bits, and the
// two halves are stacked as the N dimension of one MMA operand B = [h_hi ; h_lo] (2*Bp rows,
// K-major).  One tcgen05.mma (M = 128 vocabulary rows, N = 2*Bp, K = 16) therefore reads each W
// element from shared memory once for both halves; the epilogue adds column b and column Bp+b.
//
// Persistent CTAs walk vocabulary tiles of 128 rows (ascending within a CTA).  Warp roles:
//   warp 0  TMA producer: W tile chunks [128 rows x 64] and B chunks [2*Bp rows x 64], 128-byte
//           swizzled, into a ring of as many stages as fit (W rows past the vocabulary read as zeros)
//   warp 1  MMA issuer: 4 MMAs per 64-wide K chunk into one of two TMEM accumulators
//   warps 2-5 epilogue: row r = TMEM lane r; logits go through a padded shared tile so that
//           thread b scans the 128 rows of column b in order, keeping (max, lowest row)
// The CTA's best per batch row is published as a packed (logit, ~id) key with atomicMax and
// the last CTA turns the keys into ids.  All waits are bounded.
//
// Method: greedy argmax of the tied lm_head over the whole vocabulary (Youtu-VL-4B ncnn port,
// step 6; HunyuanOCR v1.5 ncnn port, section 3.4), vocab clamped to the logits length
// (Penguin-VL ncnn port, section 4.1).
#include <algorithm>
#include <mutex>

#include "launch.h"
#include "tc.cuh"

namespace kva {

namespace {

constexpr int TM = 128;                 // vocabulary rows per tile
constexpr int KC = 64;                  // K elements per chunk (one 128-byte swizzle row)
constexpr int THREADS = 192;
constexpr int A_BYTES = TM * 128;       // 16 KB
constexpr int MAX_N = 256;              // 2 * Bp
constexpr int BAR_BYTES = 256;          // barriers (2 per stage + 4) and the TMEM address
// Shared memory beside the ring: the padded logits tile, 64 bytes of gap, the barriers and the
// slack that aligns the base to 1024.
template <int BP> struct Fixed { static constexpr int value = TM * (BP + 1) * 4 + 64 + BAR_BYTES + 1024; };
// Ring stages: as many [128 x 64] W chunks (with their h chunks) as fit in 227 KB, at most 8.
// The table bytes in flight per SM set the kernel's rate (HBM-bound): at B = 64, 6 stages
// instead of 4 took a launch from 56.4 to 54.5 us.
template <int BP> struct Stages {
  static constexpr int fit = (232448 - Fixed<BP>::value) / (A_BYTES + 2 * BP * 128);
  static constexpr int value = fit < 8 ? fit : 8;
  static_assert(fit >= 2, "ring stages");
};

// One CTA per padded batch row b: the row's final RMSNorm (when norm_w is given), then its
// bf16 high half into row b and the residual's bf16 into row Bp + b (rows >= B are zeros).
__global__ void __launch_bounds__(256)
lmhead_split_kernel(const float* __restrict__ h, const float* __restrict__ norm_w, float eps, uint16_t* __restrict__ hb,
                    int B, int Bp, int H) {
  const int b = blockIdx.x, tid = threadIdx.x;
  __shared__ float s_part[8];
  griddep_wait();                               // h is complete from here on
  griddep_launch_dependents();
  float r = 1.f;
  if (norm_w && b < B) {
    float ss = 0.f;
    for (int k = tid; k < H; k += 256) { const float x = h[(int64_t)b * H + k]; ss = fmaf(x, x, ss); }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
    if ((tid & 31) == 0) s_part[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += s_part[w];
    r = rsqrtf(tot / (float)H + eps);
  }
  for (int k = tid; k < H; k += 256) {
    float x = b < B ? h[(int64_t)b * H + k] : 0.f;
    if (norm_w && b < B) x *= r * norm_w[k];
    const uint32_t hi = f32_to_bf16_rne(x);
    hb[(int64_t)b * H + k] = (uint16_t)hi;
    hb[(int64_t)(Bp + b) * H + k] = (uint16_t)f32_to_bf16_rne(x - __uint_as_float(hi << 16));   // residual
  }
}

template <int BP>   // batch rows padded to BP (a multiple of 16); N = 2*BP
__global__ void __launch_bounds__(THREADS, 1)
lmhead_tc_kernel(const __grid_constant__ LmheadArgs a, const __grid_constant__ CUtensorMap tmW,
                 const __grid_constant__ CUtensorMap tmH) {
  constexpr int N = 2 * BP;
  constexpr int NSTAGE = Stages<BP>::value;
  constexpr int B_BYTES = N * 128;
  constexpr int STAGE = A_BYTES + B_BYTES;
  constexpr uint32_t IDESC = tc::idesc_bf16(TM, N, 0, 0);
  constexpr uint64_t DESC = tc::desc_template(16, 1024, tc::SWIZZLE_128B);
  constexpr int LOG_LD = BP + 1;        // padded row of the logits tile
  static_assert(BP % 16 == 0 && N <= MAX_N, "batch bucket");
  constexpr uint32_t TMEM_COLS = (2 * N <= 32) ? 32 : (2 * N <= 64 ? 64 : (2 * N <= 128 ? 128 : (2 * N <= 256 ? 256 : 512)));

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sLog = reinterpret_cast<float*>(sm + NSTAGE * STAGE);                  // [TM][LOG_LD]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + NSTAGE * STAGE + TM * LOG_LD * 4 + 64);
  uint64_t* full = bars;                 // [NSTAGE]
  uint64_t* empty = bars + NSTAGE;       // [NSTAGE]
  uint64_t* acc_full = bars + 2 * NSTAGE;      // [2]
  uint64_t* acc_empty = bars + 2 * NSTAGE + 2; // [2]
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(bars + 2 * NSTAGE + 4);
  __shared__ unsigned long long s_key[BP];
  __shared__ int s_last, s_err;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (a.V + TM - 1) / TM;
  const int kchunks = a.H / KC;
  const int my_tiles = blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (warp == 1) tc::tmem_alloc(s_taddr, TMEM_COLS);
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], 4); }
    fence_mbar_init();
    s_err = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_taddr;
  // Warm L2 with this CTA's first W stages while the kernels before drain (prefetches return no
  // data, so they may run before the wait), then wait for the split rows of h
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tmW);
    tc::tma_prefetch_desc(&tmH);
    for (int it = 0; it < NSTAGE && it < my_tiles * kchunks; ++it)
      tc::tma_prefetch_l2_4d(&tmW, (it % kchunks) * KC, (blockIdx.x + (it / kchunks) * gridDim.x) * TM, 0, 0);
  }
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      for (int lt = 0; lt < my_tiles; ++lt) {
        const int tile = blockIdx.x + lt * gridDim.x;
        for (int c = 0; c < kchunks; ++c, ++it) {
          const int s = it % NSTAGE;
          if (it >= NSTAGE && !mbar_wait_bounded(&empty[s], ((it / NSTAGE) + 1) & 1)) { s_err = 1; goto producer_done; }
          mbar_arrive_expect_tx(&full[s], STAGE);
          tc::tma_load_4d(sm + s * STAGE, &tmW, c * KC, tile * TM, 0, 0, &full[s]);
          tc::tma_load_4d(sm + s * STAGE + A_BYTES, &tmH, c * KC, 0, 0, 0, &full[s]);
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0;
      for (int lt = 0; lt < my_tiles; ++lt) {
        const int ab = lt & 1;
        if (lt >= 2 && !mbar_wait_bounded(&acc_empty[ab], ((lt >> 1) + 1) & 1)) { s_err = 1; break; }
        tc::fence_after_sync();
        bool ok = true;
        for (int c = 0; c < kchunks; ++c, ++it) {
          const int s = it % NSTAGE;
          if (!mbar_wait_bounded(&full[s], (it / NSTAGE) & 1)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t a_addr = smem_u32(sm + s * STAGE), b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int k = 0; k < KC / 16; ++k)
            tc::mma_ss(tmem + ab * N, tc::desc_at(DESC, a_addr + k * 32), tc::desc_at(DESC, b_addr + k * 32), IDESC,
                       (c > 0 || k > 0));
          tc::mma_commit(&empty[s]);
        }
        if (!ok) { s_err = 1; break; }
        tc::mma_commit(&acc_full[ab]);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue warps 2..5
    const int q = warp & 3;                       // TMEM lane quarter of this warp
    const int row = q * 32 + lane;                // tile row = TMEM lane
    const int et = tid - 64;                      // 0..127 among the epilogue threads
    float best_v = -INFINITY;
    int best_i = 0x7fffffff;
    bool ok = true;
    for (int lt = 0; lt < my_tiles; ++lt) {
      const int tile = blockIdx.x + lt * gridDim.x;
      const int ab = lt & 1;
      if (!__all_sync(FULL_MASK, mbar_wait_bounded(&acc_full[ab], (lt >> 1) & 1))) ok = false;   // warp-uniform
      tc::fence_after_sync();
      const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + ab * N;
#pragma unroll
      for (int c0 = 0; c0 < BP; c0 += 16) {
        uint32_t hi[16], lo[16];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(hi[0]), "=r"(hi[1]), "=r"(hi[2]), "=r"(hi[3]), "=r"(hi[4]), "=r"(hi[5]), "=r"(hi[6]), "=r"(hi[7]),
              "=r"(hi[8]), "=r"(hi[9]), "=r"(hi[10]), "=r"(hi[11]), "=r"(hi[12]), "=r"(hi[13]), "=r"(hi[14]), "=r"(hi[15])
            : "r"(base + c0));
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(lo[0]), "=r"(lo[1]), "=r"(lo[2]), "=r"(lo[3]), "=r"(lo[4]), "=r"(lo[5]), "=r"(lo[6]), "=r"(lo[7]),
              "=r"(lo[8]), "=r"(lo[9]), "=r"(lo[10]), "=r"(lo[11]), "=r"(lo[12]), "=r"(lo[13]), "=r"(lo[14]), "=r"(lo[15])
            : "r"(base + BP + c0));
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e)
          sLog[row * LOG_LD + c0 + e] = __uint_as_float(hi[e]) + __uint_as_float(lo[e]);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);        // accumulator may be overwritten
      asm volatile("bar.sync 1, 128;" ::: "memory");    // logits tile complete
      const int v0 = tile * TM;
      if (a.logits) {
        for (int i = et; i < TM * a.B; i += 128) {
          const int b = i / TM, r = i % TM;
          if (v0 + r < a.V) a.logits[(int64_t)b * a.V + v0 + r] = sLog[r * LOG_LD + b];
        }
      }
      if (et < a.B) {
        const int rmax = min(TM, a.V - v0);
        for (int r = 0; r < rmax; ++r) {
          const float v = sLog[r * LOG_LD + et];
          if (v > best_v) { best_v = v; best_i = v0 + r; }   // rows and tiles ascend: lowest id on ties
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");    // tile consumed before the next overwrite
    }
    if (!ok) s_err = 1;
    if (et < a.B) s_key[et] = best_i == 0x7fffffff ? 0ull : argmax_key(best_v, (uint32_t)best_i);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (tid < a.B && my_tiles > 0 && s_key[tid]) atomicMax(&a.best[tid], s_key[tid]);
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int b = tid; b < a.B; b += THREADS) {
      const unsigned long long k = atomicExch(&a.best[b], 0ull);
      a.out_ids[b] = s_err ? -1 : (int32_t)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
      if (a.out_max) a.out_max[b] = float_from_order_bits((uint32_t)(k >> 32));
    }
    if (tid == 0) *a.counter = 0u;
  }
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn_lm() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 map [rows, H] (dims as 4-D with unit outer dims), box [box_rows x 64].
cudaError_t make_map(CUtensorMap* m, const void* base, int H, int rows, int box_rows) {
  EncodeTiledFn fn = encode_fn_lm();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {(cuuint64_t)H, (cuuint64_t)rows, 1, 1};
  const cuuint64_t strides[3] = {(cuuint64_t)H * 2, (cuuint64_t)H * 2 * rows, (cuuint64_t)H * 2 * rows};
  const cuuint32_t box[4] = {KC, (cuuint32_t)box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int num_sms_tc() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

template <int BP>
cudaError_t launch_bp(const LmheadArgs& a, uint16_t* hb, cudaStream_t s) {
  constexpr int N = 2 * BP;
  constexpr int smem = Stages<BP>::value * (A_BYTES + N * 128) + Fixed<BP>::value;
  static_assert(smem <= 232448, "shared memory per CTA");
  static_assert((2 * Stages<BP>::value + 4) * 8 + 4 <= BAR_BYTES, "barrier area");
  static DeviceOnce configured;
  if (!configured.done()) {
    cudaError_t e = cudaFuncSetAttribute(lmhead_tc_kernel<BP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.mark();
  }
  cudaError_t e = launch_pdl(lmhead_split_kernel, dim3(BP), dim3(256), 0, s, a.h, a.norm_w, a.eps, hb, a.B, BP, a.H);
  if (e != cudaSuccess) return e;
  CUtensorMap mw, mh;
  if ((e = make_map(&mw, a.W, a.H, a.V, TM)) != cudaSuccess) return e;
  if ((e = make_map(&mh, hb, a.H, N, N)) != cudaSuccess) return e;
  const int n_tiles = (a.V + TM - 1) / TM;
  const int grid = std::min(n_tiles, num_sms_tc());
  return launch_pdl(lmhead_tc_kernel<BP>, dim3(grid), dim3(THREADS), (size_t)smem, s, a, mw, mh);
}

}  // namespace

bool lmhead_tc_supports(int B, int H) {
  return B >= 2 && B <= MAX_N / 2 && H % KC == 0 && encode_fn_lm() != nullptr;
}

// Bytes of the bf16 hi/lo copy of h the batched path keeps in the workspace.
size_t lmhead_tc_hb_bytes(int B, int H) {
  const int bp = B <= 16 ? 16 : (B <= 32 ? 32 : (B <= 64 ? 64 : 128));
  return (size_t)2 * bp * H * sizeof(uint16_t);
}

// Two launches: the hi/lo split of h, then the persistent GEMM + argmax.
cudaError_t launch_lmhead_tc(const LmheadArgs& a, uint16_t* hb, cudaStream_t s) {
  if (a.B <= 16) return launch_bp<16>(a, hb, s);
  if (a.B <= 32) return launch_bp<32>(a, hb, s);
  if (a.B <= 64) return launch_bp<64>(a, hb, s);
  return launch_bp<128>(a, hb, s);
}

}  // namespace kva
