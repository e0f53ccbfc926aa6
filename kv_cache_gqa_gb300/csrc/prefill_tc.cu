// Kernel (b), tensor-core form: flash-style prefill attention on tcgen05 (bf16 operands,
// fp32 accumulation in tensor memory).
//
// One CTA per (128-query tile, query head, instance), six warps with fixed roles:
//   warps 0-3  softmax: thread t owns query row t = TMEM lane t.  It stages its Q row in
//              shared memory (128-byte swizzled, K-major), then per key tile reads the
//              128 fp32 scores S from TMEM, applies the row's visible-key range (causal,
//              window segment or full), keeps the running max/sum, writes P = exp2(S - m)
//              back into the same TMEM columns as packed bf16 pairs, and at the end divides
//              O by the row sum.  O is only rescaled when the row max grows by more than
//              2^8 (the stale max keeps every P <= 256, so the result is unchanged).
//   warp 4     TMA producer: K and V tiles of the KV head (two 64-column, 128-byte swizzled
//              boxes each) into a 2-stage ring; rows past the valid prefix read as zeros.
//   warp 5     MMA issuer (one thread): S_j = Q K_j^T into TMEM buffer j%2 (both operands
//              K-major in shared memory), then O += P_{j-1} V_{j-1} with P read from TMEM
//              and V as an MN-major shared-memory operand.  Issue order S_0, S_1, PV_0,
//              S_2, PV_1, ... lets the tensor core run S_{j+1} while the softmax warps work
//              on S_j; commits to mbarriers signal S ready / K,V stage free.
// Every mbarrier wait is bounded; a timeout marks the output rows NaN instead of hanging.
//
// Method: QK^T*scale + mask, softmax, times V (Youtu-VL-4B ncnn port, implementation
// difficulty 3; parallel causal prefill, step 7; block-diagonal window mask, step 3) fused
// in one kernel with intermediates on chip (MNN llm_demo walkthrough, section 5.1), bf16
// storage with fp32 accumulation (HunyuanOCR v1.5 ncnn port, section 3.7).
#include <cstring>
#include <mutex>

#include "launch.h"
#include "tc.cuh"

namespace kva {

namespace {

constexpr int BM = 128;                   // query rows per CTA = TMEM lanes
constexpr int BN = 128;                   // keys per tile
constexpr int THREADS = 192;
constexpr int SUB = BM * 128;             // bytes of one [128 rows x 64 bf16] swizzled box
constexpr int Q_OFF = 0;
constexpr int K_OFF = Q_OFF + 2 * SUB;
constexpr int V_OFF = K_OFF + 4 * SUB;
constexpr int BAR_OFF = V_OFF + 4 * SUB;
constexpr int SMEM_BYTES = BAR_OFF + 128 + 1024;   // + slack to align the base to 1024
constexpr uint32_t TMEM_COLS = 512;       // S0 [0,128)  S1 [128,256)  O [256, 256+DN)
constexpr uint32_t O_COL = 256;
constexpr float RESCALE_LOG2 = 8.0f;

constexpr uint64_t DESC_KMAJ = tc::desc_template(16, 1024, tc::SWIZZLE_128B);
constexpr uint64_t DESC_VMN = tc::desc_template(SUB, 1024, tc::SWIZZLE_128B);

__device__ int seg_lower_tc(const int32_t* seg, int S, int key) {
  int lo = 0, hi = S;
  while (lo < hi) { const int mid = (lo + hi) >> 1; if (seg[mid] < key) lo = mid + 1; else hi = mid; }
  return lo;
}
__device__ int seg_upper_tc(const int32_t* seg, int S, int key) {
  int lo = 0, hi = S;
  while (lo < hi) { const int mid = (lo + hi) >> 1; if (seg[mid] <= key) lo = mid + 1; else hi = mid; }
  return lo;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
         "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
prefill_tc_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  constexpr int DK = (D + 15) / 16 * 16;      // MMA K extent of Q K^T (zero padded)
  constexpr int DN = DK;                      // MMA N extent of P V
  constexpr int KSTEPS = DK / 16;
  constexpr int NSUB = (D + 63) / 64;         // 64-column boxes per K / V tile
  constexpr uint32_t IDESC_S = tc::idesc_bf16(BM, BN, 0, 0);
  constexpr uint32_t IDESC_PV = tc::idesc_bf16(BM, DN, 0, 1);
  static_assert(DN % 16 == 0 && DN <= 256 - 0, "N extent");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + BAR_OFF);
  uint64_t* kv_full = bars + 0;    // [2] K,V tile landed
  uint64_t* pv_done = bars + 2;    // [2] P V of the tile finished: O updated, K/V stage free
  uint64_t* s_full = bars + 4;     // [2] S ready in TMEM
  uint64_t* p_full = bars + 6;     // [2] P written to TMEM by the 4 softmax warps
  uint64_t* q_full = bars + 8;     // Q staged by the 4 softmax warps
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(bars + 9);
  __shared__ int s_err;

  const int qt = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.Hq / a.Hkv, g = h / G;
  const int i0 = qt * BM;
  const int i_last = min(a.S, i0 + BM) - 1;

  // keys any row of this tile may see -> key tiles [j0, j1)
  int lo = 0, hi = a.S;
  if (a.mask == KVA_MASK_CAUSAL) {
    hi = i_last + 1;
  } else if (a.mask == KVA_MASK_SEGMENT) {
    lo = seg_lower_tc(a.segment, a.S, a.segment[i0]);
    hi = seg_upper_tc(a.segment, a.S, a.segment[i_last]);
  }
  const int j0 = lo / BN, j1 = (hi + BN - 1) / BN;
  const int nt = j1 - j0;

  if (warp == 5) tc::tmem_alloc(s_taddr, TMEM_COLS);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1); mbar_init(&pv_done[i], 1); mbar_init(&s_full[i], 1); mbar_init(&p_full[i], 4);
    }
    mbar_init(q_full, 4);
    fence_mbar_init();
    s_err = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_taddr;

  uint8_t* sQ = sm + Q_OFF;
  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmK);
      tc::tma_prefetch_desc(&tmV);
      for (int it = 0; it < nt; ++it) {
        const int st = it & 1;
        if (it >= 2 && !mbar_wait_bounded(&pv_done[st], ((it >> 1) + 1) & 1)) { s_err = 1; break; }
        mbar_arrive_expect_tx(&kv_full[st], 2 * NSUB * SUB);
        const int key0 = (j0 + it) * BN;
        for (int s = 0; s < NSUB; ++s) {
          tc::tma_load_4d(sm + K_OFF + (st * 2 + s) * SUB, &tmK, s * 64, key0, g, n, &kv_full[st]);
          tc::tma_load_4d(sm + V_OFF + (st * 2 + s) * SUB, &tmV, s * 64, key0, g, n, &kv_full[st]);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait_bounded(q_full, 0);
      tc::fence_after_sync();
      const uint32_t q_addr = smem_u32(sQ);
      for (int it = 0; ok && it <= nt; ++it) {
        if (it < nt) {
          const int st = it & 1;
          if (!mbar_wait_bounded(&kv_full[st], (it >> 1) & 1)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t k_addr = smem_u32(sm + K_OFF + st * 2 * SUB);
#pragma unroll
          for (int k = 0; k < KSTEPS; ++k) {
            const uint32_t off = (k >> 2) * SUB + (k & 3) * 32;
            tc::mma_ss(tmem + st * BN, tc::desc_at(DESC_KMAJ, q_addr + off), tc::desc_at(DESC_KMAJ, k_addr + off),
                       IDESC_S, k > 0);
          }
          tc::mma_commit(&s_full[st]);
        }
        if (it >= 1) {
          const int pj = it - 1, pst = pj & 1;
          if (!mbar_wait_bounded(&p_full[pst], (pj >> 1) & 1)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t v_addr = smem_u32(sm + V_OFF + pst * 2 * SUB);
#pragma unroll
          for (int k = 0; k < BN / 16; ++k)
            tc::mma_ts(tmem + O_COL, tmem + pst * BN + k * 8, tc::desc_at(DESC_VMN, v_addr + k * 2048),
                       IDESC_PV, (pj > 0 || k > 0));
          tc::mma_commit(&pv_done[pst]);
        }
      }
      if (!ok) s_err = 1;
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int t = tid;                                  // query row within the tile
    const int i = i0 + t;
    const bool row_ok = i < a.S;
    int row = i;
    if (row_ok && a.row_of_slot) row = a.row_of_slot[i];
    const bool row_valid = row_ok && row >= 0 && row < a.S;
    // stage the Q row: chunk c (8 bf16) -> box c/8, swizzled position (c%8) ^ (t%8)
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          reinterpret_cast<const uint16_t*>(a.q) + (((int64_t)n * a.S + row) * a.Hq + h) * D);
#pragma unroll
      for (int c = 0; c < DK / 8; ++c) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row_valid && c < D / 8) v = __ldg(src + c);
        uint8_t* dst = sQ + (c >> 3) * SUB + (t >> 3) * 1024 + (t & 7) * 128 + (((c & 7) ^ (t & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = v;
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(q_full);

    // visible keys of this row
    int rlo = 0, rhi = 0;
    if (row_ok) {
      if (a.mask == KVA_MASK_CAUSAL) { rlo = 0; rhi = i + 1; }
      else if (a.mask == KVA_MASK_FULL) { rlo = 0; rhi = a.S; }
      else { const int sg = a.segment[i]; rlo = seg_lower_tc(a.segment, a.S, sg); rhi = seg_upper_tc(a.segment, a.S, sg); }
    }
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int it = 0; it < nt; ++it) {
      const int st = it & 1;
      const int kv0 = (j0 + it) * BN;
      // every lane waits; the vote keeps the warp converged for the .aligned TMEM accesses
      if (!__all_sync(FULL_MASK, mbar_wait_bounded(&s_full[st], (it >> 1) & 1))) { ok = false; break; }
      tc::fence_after_sync();
      float x[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(lane_base + st * BN + c * 32, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(r[e]) * a.scale_log2;
      }
      if (!(kv0 >= rlo && kv0 + BN <= rhi)) {          // tile straddles this row's range
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int key = kv0 + c;
          if (key < rlo || key >= rhi) x[c] = -INFINITY;
        }
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN; ++c) mt = fmaxf(mt, x[c]);
      const float m_new = fmaxf(m, mt);
      const bool first = (m == -INFINITY);            // first visible keys: O holds zeros
      const bool grow = !first && m_new > m + RESCALE_LOG2;
      if (first) m = m_new;
      if (__any_sync(FULL_MASK, grow)) {
        // some row's max grew by > 2^8: rescale those rows of O once P V of the previous tile
        // has landed.  The whole warp takes part (TMEM loads/stores are warp-collective);
        // rows that need no rescale use alpha = 1.
        if (!__all_sync(FULL_MASK, mbar_wait_bounded(&pv_done[(it - 1) & 1], ((it - 1) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const float alpha = grow ? exp2f(m - m_new) : 1.0f;
#pragma unroll
        for (int c = 0; c < DN / 16; ++c) {
          uint32_t r[16];
          tmem_ld16(lane_base + O_COL + c * 16, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tmem_st16(lane_base + O_COL + c * 16, r);
        }
        tc::tmem_wait_st();
        if (grow) { l *= alpha; m = m_new; }
      }
      const float mref = (m == -INFINITY) ? 0.f : m;
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p0 = exp2f(x[c * 64 + 2 * e] - mref);
          const float p1 = exp2f(x[c * 64 + 2 * e + 1] - mref);
          const uint32_t pk = pack_bf16x2(p0, p1);
          l += bf16_lo(pk) + bf16_hi(pk);
          w[e] = pk;
        }
        tc::tmem_st32(lane_base + st * BN + c * 32, w);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[st]);
    }
    // epilogue: O / l -> token-order output row.  The TMEM loads are warp-collective, so every
    // lane loads; only rows inside the sequence store.
    if (ok) ok = __all_sync(FULL_MASK, mbar_wait_bounded(&pv_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1));
    tc::fence_after_sync();
    {
      float* o = a.out + (((int64_t)n * a.S + (row_valid ? row : 0)) * a.Hq + h) * D;
      const float inv = (ok && l > 0.f) ? 1.0f / l : NAN;
#pragma unroll
      for (int c = 0; c < DN / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(lane_base + O_COL + c * 16, r);
        tc::tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const int d = c * 16 + e;
            if (d < D)
              *reinterpret_cast<float4*>(o + d) = make_float4(__uint_as_float(r[e]) * inv, __uint_as_float(r[e + 1]) * inv,
                                                              __uint_as_float(r[e + 2]) * inv, __uint_as_float(r[e + 3]) * inv);
          }
        }
      }
    }
    if (!ok) s_err = 1;
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 5) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------------------------
// Host: tensor maps over the cache (4-D: head_dim, slot, kv head, instance)
// ---------------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// Cache view for TMA: dims (D, S valid slots, Hkv, N); rows >= S read as zeros.
cudaError_t make_cache_map(CUtensorMap* map, const void* base, const PrefillArgs& a) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {(cuuint64_t)a.D, (cuuint64_t)a.S, (cuuint64_t)a.Hkv, (cuuint64_t)a.N};
  const cuuint64_t strides[3] = {(cuuint64_t)a.D * 2, (cuuint64_t)a.capacity * a.D * 2, (cuuint64_t)a.inst_stride * 2};
  const cuuint32_t box[4] = {64, BN, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_d(const PrefillArgs& a, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  CUtensorMap mk, mv;
  cudaError_t e = make_cache_map(&mk, a.kc, a);
  if (e != cudaSuccess) return e;
  e = make_cache_map(&mv, a.vc, a);
  if (e != cudaSuccess) return e;
  dim3 grid((a.S + BM - 1) / BM, a.Hq, a.N);
  prefill_tc_kernel<D><<<grid, THREADS, SMEM_BYTES, s>>>(a, mk, mv);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supports(int D, kva_dtype dt) {
  return dt == KVA_BF16 && (D == 64 || D == 72 || D == 128) && encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s) {
  switch (a.D) {
    case 64: return launch_d<64>(a, s);
    case 72: return launch_d<72>(a, s);
    case 128: return launch_d<128>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kva
