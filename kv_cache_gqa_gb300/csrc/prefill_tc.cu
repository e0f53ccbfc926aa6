// Kernel (b), tensor-core form: flash-style prefill attention on tcgen05 (bf16 operands,
// fp32 accumulation in tensor memory).
//
// One CTA serves two 128-row query tiles ("slots") that read the same KV head: the two query
// heads of a GQA group at the same rows when the group size is even (each K/V tile is loaded
// once for both), otherwise two row tiles of one head paired so that causal work is balanced
// (tiles t and n-1-t).  Ten warps with fixed roles:
//   warps 0-3, 4-7  softmax of slot 0 and slot 1: thread t of a group owns row t = TMEM lane
//              t.  It stages its Q row in shared memory (128-byte swizzled, K-major), then per
//              key tile reads the 128 fp32 scores from TMEM, applies the row's visible-key
//              range (causal, window segment or full), keeps the running max and sum, writes
//              P = exp2(S - m) back into the same TMEM columns as packed bf16 pairs, and at
//              the end divides O by the row sum.  O is rescaled only when the row max grows
//              by more than 2^8 (the stale max keeps every P <= 256).
//   warp 8     TMA producer: K and V tiles (64-column, 128-byte swizzled boxes) into a
//              2-stage ring; rows past the valid keys read as zeros.
//   warp 9     MMA issuer (one thread).  TMEM: S of slot s at columns [128 s, 128 s + 128),
//              O of slot s at [256 + 128 s, ...).  Per key tile j it issues, for s = 0, 1:
//              O_s += P_s(j) V_j once slot s's softmax has written P_s(j), then
//              S_s(j+1) = Q_s K_{j+1}^T into the same columns (tensor-core operations of one
//              thread run in issue order, so the P V read precedes the overwrite).  While
//              one slot's warps run the softmax of tile j, the tensor core works on the
//              other slot's P V and next S: the two slots ping-pong.
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

constexpr int BM = 128;                   // query rows per slot = TMEM lanes
constexpr int BN = 128;                   // keys per tile
constexpr int SOFTMAX_WARPS = 16;         // per slot: 4 lane quarters x 2 column halves
constexpr int TMA_WARP = 16, MMA_WARP = 17;
constexpr int THREADS = 576;
constexpr int SUB = BM * 128;             // bytes of one [128 rows x 64 bf16] swizzled box
constexpr int NSTAGE = 2;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;

template <int D>
struct Layout {
  static constexpr int NSUB = (D + 63) / 64;                 // 64-column boxes per row tile
  static constexpr int Q_OFF = 0;                            // [2 slots][NSUB boxes]
  static constexpr int K_OFF = Q_OFF + 2 * NSUB * SUB;       // [NSTAGE][NSUB]
  static constexpr int V_OFF = K_OFF + NSTAGE * NSUB * SUB;  // [NSTAGE][NSUB]
  static constexpr int BAR_OFF = V_OFF + NSTAGE * NSUB * SUB;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;          // + slack to align the base to 1024
};

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
// Paired fp32 arithmetic (two lanes of a 64-bit register pair per instruction) and a
// three-input max.
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2split(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The two slots of a CTA: (query head, row tile) each, or an empty slot (qt < 0).
struct Slots {
  int h[2], qt[2];
};
__device__ __forceinline__ Slots cta_slots(const PrefillArgs& a, int nq) {
  Slots sl;
  const int G = a.Hq / a.Hkv;
  if (G % 2 == 0) {            // grid (Hq/2, N, nq): the two heads of a pair, heaviest row tiles first
    sl.h[0] = 2 * blockIdx.x; sl.h[1] = 2 * blockIdx.x + 1;
    sl.qt[0] = sl.qt[1] = nq - 1 - (int)blockIdx.z;
  } else {                     // grid (Hq, N, ceil(nq/2)): row tiles t and nq-1-t of one head
    sl.h[0] = sl.h[1] = blockIdx.x;
    sl.qt[0] = blockIdx.z;
    sl.qt[1] = nq - 1 - (int)blockIdx.z;
    if (sl.qt[1] == sl.qt[0]) sl.qt[1] = -1;
  }
  return sl;
}

// Key range [lo, hi) that rows [i0, i_last] of a tile may see.
__device__ __forceinline__ void tile_keys(const PrefillArgs& a, int i0, int i_last, int& lo, int& hi) {
  lo = 0; hi = a.S;
  if (a.mask == KVA_MASK_CAUSAL) {
    hi = i_last + 1;
  } else if (a.mask == KVA_MASK_SEGMENT) {
    lo = seg_lower_tc(a.segment, a.S, a.segment[i0]);
    hi = seg_upper_tc(a.segment, a.S, a.segment[i_last]);
  } else if (a.mask == KVA_MASK_CAUSAL_SEGMENT) {
    hi = seg_upper_tc(a.segment, a.S, a.segment[i_last]);    // the last row's segment end
  }
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
prefill_tc_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmO) {
  using LY = Layout<D>;
  constexpr int DK = (D + 15) / 16 * 16;      // MMA K extent of Q K^T (zero padded)
  constexpr int DN = DK;                      // MMA N extent of P V
  constexpr int KSTEPS = DK / 16;
  constexpr int NSUB = LY::NSUB;
  constexpr uint32_t IDESC_S = tc::idesc_bf16(BM, BN, 0, 0);
  constexpr uint32_t IDESC_PV = tc::idesc_bf16(BM, DN, 0, 1);
  static_assert(DN % 16 == 0 && DN <= 128, "N extent");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + LY::BAR_OFF);
  uint64_t* kv_full = bars + 0;    // [NSTAGE] K, V tile landed
  uint64_t* kv_free = bars + 2;    // [NSTAGE] both slots' P V of the tile done: stage free
  uint64_t* s_full = bars + 4;     // [slot] S ready in TMEM
  uint64_t* p_full = bars + 6;     // [slot] P written to TMEM by the slot's 4 warps
  uint64_t* pv_done = bars + 8;    // [slot] P V of the slot's tile finished
  uint64_t* q_full = bars + 10;    // [slot] Q tile landed (TMA) or staged by the slot's 4 warps
  uint64_t* mma_done = bars + 12;  // every MMA of the CTA completed
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(bars + 13);
  const bool gather = a.row_of_slot != nullptr;   // permuted rows: threads stage Q and store O

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.y;
  const int nq = (a.S + BM - 1) / BM;
  const Slots sl = cta_slots(a, nq);
  const int g = sl.h[0] / (a.Hq / a.Hkv);

  if (warp == MMA_WARP) tc::tmem_alloc(s_taddr, TMEM_COLS);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1); mbar_init(&kv_free[i], 1); mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], SOFTMAX_WARPS / 2); mbar_init(&pv_done[i], 1);
      mbar_init(&q_full[i], gather ? SOFTMAX_WARPS / 2 : 1);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == TMA_WARP && lane == 0) {
    tc::tma_prefetch_desc(&tmK); tc::tma_prefetch_desc(&tmV); tc::tma_prefetch_desc(&tmQ); tc::tma_prefetch_desc(&tmO);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_taddr;
  griddep_wait();                              // inputs of this launch are complete from here on
  griddep_launch_dependents();

  // key tiles of each slot, [js0, js1), and their union [j0, j1)
  int js0[2], js1[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    if (sl.qt[s] < 0) { js0[s] = js1[s] = 0; continue; }
    const int i0 = sl.qt[s] * BM, i_last = min(a.S, i0 + BM) - 1;
    int lo, hi;
    tile_keys(a, i0, i_last, lo, hi);
    js0[s] = lo / BN; js1[s] = (hi + BN - 1) / BN;
  }
  const bool act1 = sl.qt[1] >= 0;
  const int j0 = act1 ? min(js0[0], js0[1]) : js0[0];
  const int j1 = act1 ? max(js1[0], js1[1]) : js1[0];
  auto active = [&](int s, int j) { return (s == 0 || act1) && j >= js0[s] && j < js1[s]; };
  // Key tiles the CTA loads: those some slot needs, in increasing order (the two slots' ranges
  // may be disjoint under a window mask).  Producer and MMA walk the same list, numbering its
  // entries it = 0, 1, ... for the ring stage and barrier phases.
  auto next_tile = [&](int j) {
    ++j;
    while (j < j1 && !active(0, j) && !active(1, j)) ++j;
    return j;
  };


  if (warp == TMA_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      if (!gather) {
        for (int s = 0; s < 2; ++s) {
          if (s == 1 && !act1) break;
          mbar_arrive_expect_tx(&q_full[s], NSUB * SUB);
          for (int b = 0; b < NSUB; ++b)
            tc::tma_load_4d(sm + LY::Q_OFF + (s * NSUB + b) * SUB, &tmQ, b * 64, sl.h[s], sl.qt[s] * BM, n, &q_full[s]);
        }
      }
      int issued = 0;
      for (int j = j0, it = 0; j < j1; j = next_tile(j), ++it) {
        const int st = it % NSTAGE;
        if (it >= NSTAGE && !mbar_wait_bounded(&kv_free[st], (uint32_t)((it / NSTAGE - 1) & 1))) break;
        mbar_arrive_expect_tx(&kv_full[st], 2 * NSUB * SUB);
        const int key0 = j * BN;
        for (int b = 0; b < NSUB; ++b) {
          tc::tma_load_4d(sm + LY::K_OFF + (st * NSUB + b) * SUB, &tmK, b * 64, key0, g, n, &kv_full[st]);
          tc::tma_load_4d(sm + LY::V_OFF + (st * NSUB + b) * SUB, &tmV, b * 64, key0, g, n, &kv_full[st]);
        }
        issued = it + 1;
      }
      // the copies this CTA issued have normally landed long ago; never leave one in flight
      for (int it = max(0, issued - NSTAGE); it < issued; ++it)
        mbar_wait_bounded(&kv_full[it % NSTAGE], (uint32_t)((it / NSTAGE) & 1));
      if (!gather) {
        mbar_wait_bounded(&q_full[0], 0);
        if (act1) mbar_wait_bounded(&q_full[1], 0);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait_bounded(&q_full[0], 0) && (!act1 || mbar_wait_bounded(&q_full[1], 0));
      tc::fence_after_sync();
      auto issue_s = [&](int s, int it) {
        const int st = it % NSTAGE;
        const uint32_t q_addr = smem_u32(sm + LY::Q_OFF + s * NSUB * SUB);
        const uint32_t k_addr = smem_u32(sm + LY::K_OFF + st * NSUB * SUB);
#pragma unroll
        for (int k = 0; k < KSTEPS; ++k) {
          const uint32_t off = (k >> 2) * SUB + (k & 3) * 32;
          tc::mma_ss(tmem + s * BN, tc::desc_at(DESC_KMAJ, q_addr + off), tc::desc_at(DESC_KMAJ, k_addr + off),
                     IDESC_S, k > 0);
        }
        tc::mma_commit(&s_full[s]);
      };
      if (ok) {
        ok = mbar_wait_bounded(&kv_full[0], 0);
        tc::fence_after_sync();
        for (int s = 0; ok && s < 2; ++s)
          if (active(s, j0)) issue_s(s, 0);
      }
      for (int j = j0, it = 0; ok && j < j1; ++it) {
        const int st = it % NSTAGE;
        const int jn = next_tile(j);                  // the tile loaded after j (entry it + 1)
        bool next_landed = false;
        for (int s = 0; ok && s < 2; ++s) {
          if (active(s, j)) {
            const int k = j - js0[s];
            if (!mbar_wait_bounded(&p_full[s], (uint32_t)(k & 1))) { ok = false; break; }
            tc::fence_after_sync();
            const uint32_t v_addr = smem_u32(sm + LY::V_OFF + st * NSUB * SUB);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              tc::mma_ts(tmem + 256 + s * 128, tmem + s * BN + kk * 8, tc::desc_at(DESC_VMN, v_addr + kk * 2048),
                         IDESC_PV, (k > 0 || kk > 0));
            tc::mma_commit(&pv_done[s]);
          }
          if (jn < j1 && active(s, jn)) {
            if (!next_landed) {
              if (!mbar_wait_bounded(&kv_full[(it + 1) % NSTAGE], (uint32_t)(((it + 1) / NSTAGE) & 1))) { ok = false; break; }
              tc::fence_after_sync();
              next_landed = true;
            }
            issue_s(s, it + 1);
          }
        }
        tc::mma_commit(&kv_free[st]);             // the stage is free once this tile's MMAs are done
        j = jn;
      }
      tc::mma_commit(mma_done);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    // warp w: slot s = w / 8, column half ch = (w / 4) % 2, TMEM lane quarter w % 4.  Thread
    // (ch, t) owns columns [64 ch, 64 ch + 64) of row t; the two threads of a row trade their
    // partial maxima (and at the end their partial sums) through shared memory.
    const int s = warp >> 3;
    const int ch = (warp >> 2) & 1;
    const int t = (warp & 3) * 32 + lane;        // row within the tile = TMEM lane
    __shared__ float s_pmax[2][2][2][BM];        // [tile parity][slot][half][row]
    const int pair_bar = 1 + s * 4 + (warp & 3); // named barrier of warps w and w ^ 4 (64 threads)
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" :: "r"(pair_bar) : "memory"); };
    if (s == 0 || act1) {
      const int h = sl.h[s];
      const int i = sl.qt[s] * BM + t;
      const bool row_ok = i < a.S;
      int row = i;
      if (row_ok && a.row_of_slot) row = a.row_of_slot[i];
      const bool row_valid = row_ok && row >= 0 && row < a.S;
      // permuted rows: stage the Q row (this thread's half of the 16-byte chunks): chunk c
      // (8 bf16) -> box c/8, swizzled position (c%8) ^ (t%8)
      uint8_t* sQ = sm + LY::Q_OFF + s * NSUB * SUB;
      if (gather) {
        const uint4* src = reinterpret_cast<const uint4*>(
            reinterpret_cast<const uint16_t*>(a.q) + (((int64_t)n * a.S + row) * a.Hq + h) * D);
#pragma unroll
        for (int c = ch; c < DK / 8; c += 2) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (row_valid && c < D / 8) v = __ldg(src + c);
          uint8_t* dst = sQ + (c >> 3) * SUB + (t >> 3) * 1024 + (t & 7) * 128 + (((c & 7) ^ (t & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[s]);
      }

      // visible keys of this row
      int rlo = 0, rhi = 0;
      if (row_ok) {
        if (a.mask == KVA_MASK_CAUSAL) { rlo = 0; rhi = i + 1; }
        else if (a.mask == KVA_MASK_FULL) { rlo = 0; rhi = a.S; }
        else if (a.mask == KVA_MASK_CAUSAL_SEGMENT) { rlo = 0; rhi = seg_upper_tc(a.segment, a.S, a.segment[i]); }
        else { const int sg = a.segment[i]; rlo = seg_lower_tc(a.segment, a.S, sg); rhi = seg_upper_tc(a.segment, a.S, sg); }
      }
      const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      const uint32_t s_col = s * BN, o_col = 256 + s * 128;
      const int nk = js1[s] - js0[s];
      float m = -INFINITY, l = 0.f;             // l: this thread's half of the row sum
      bool ok = true;
      for (int k = 0; k < nk; ++k) {
        const int kv0 = (js0[s] + k) * BN + ch * 64;     // first key of this thread's columns
        // every lane waits; the vote keeps the warp converged for the .aligned TMEM accesses
        if (!__all_sync(FULL_MASK, mbar_wait_bounded(&s_full[s], (uint32_t)(k & 1)))) { ok = false; break; }
        tc::fence_after_sync();
        float x[64];
        {
          uint32_t r0[32], r1[32];
          tc::tmem_ld32(lane_base + s_col + ch * 64, r0);
          tc::tmem_ld32(lane_base + s_col + ch * 64 + 32, r1);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) { x[e] = __uint_as_float(r0[e]); x[32 + e] = __uint_as_float(r1[e]); }
        }
        // visible columns of this thread's 64 for this row: [clo, chi)
        const int clo = rlo - kv0, chi = rhi - kv0;
        if (clo > 0 || chi < 64) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e < clo || e >= chi) x[e] = -INFINITY;
        }
        float mr = -INFINITY;
#pragma unroll
        for (int e = 0; e < 64; e += 2) mr = fmax3(mr, x[e], x[e + 1]);
        // the row max over both halves (the barrier also means both threads hold their S, so
        // P may now overwrite it: half 1's P columns [32, 64) hold half 0's scores)
        s_pmax[k & 1][s][ch][t] = mr;
        pair_sync();
        mr = fmaxf(mr, s_pmax[k & 1][s][ch ^ 1][t]);
        const float m_tile = mr == -INFINITY ? -INFINITY : mr * a.scale_log2;
        const float m_new = fmaxf(m, m_tile);
        const bool first = (m == -INFINITY);            // first visible keys: O holds nothing yet
        const bool grow = !first && m_new > m + RESCALE_LOG2;
        if (first) m = m_new;
        if (__any_sync(FULL_MASK, grow)) {
          // some row's max grew by > 2^8: rescale those rows of O (this thread's 16-column
          // chunks of it) once P V of the previous tile has landed.  The whole warp takes part
          // (TMEM accesses are warp-collective); rows that need no rescale use alpha = 1.
          if (!__all_sync(FULL_MASK, mbar_wait_bounded(&pv_done[s], (uint32_t)((k - 1) & 1)))) { ok = false; break; }
          tc::fence_after_sync();
          const float alpha = grow ? ex2(m - m_new) : 1.0f;
#pragma unroll
          for (int c = ch; c < DN / 16; c += 2) {
            uint32_t r[16];
            tmem_ld16(lane_base + o_col + c * 16, r);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st16(lane_base + o_col + c * 16, r);
          }
          tc::tmem_wait_st();
          if (grow) { l *= alpha; m = m_new; }
        }
        // P = exp2(S * scale - m) as packed bf16 into columns [32 ch, 32 ch + 32) of the slot
        const float mref = (m == -INFINITY) ? 0.f : m;
        const uint64_t sc2 = f2(a.scale_log2, a.scale_log2), nm2 = f2(-mref, -mref);
        uint64_t lsum = f2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float x0, x1;
            f2split(ffma2(f2(x[32 * c + 2 * e], x[32 * c + 2 * e + 1]), sc2, nm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);         // hidden keys hold -inf: exp2 -> 0
            lsum = fadd2(lsum, f2(p0, p1));
            w[e] = pack_bf16x2(p0, p1);
          }
          tmem_st16(lane_base + s_col + ch * 32 + c * 16, w);
        }
        float l0, l1;
        f2split(lsum, l0, l1);
        l += l0 + l1;
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[s]);
      }
      // the row sum over both halves
      s_pmax[nk & 1][s][ch][t] = l;
      pair_sync();
      const float l_row = l + s_pmax[nk & 1][s][ch ^ 1][t];
      if (!gather) {
        // epilogue: once every MMA of the CTA is done, the rings and Q tiles are free: O / l goes
        // through shared memory (per 32-column box: 128 rows of 128 bytes, 128-byte swizzled)
        // and out with TMA stores, which also clip rows past the sequence.  Thread half ch
        // stages boxes ch, ch + 2, ...
        constexpr int NBOX = (D + 31) / 32;
        if (ok) ok = __all_sync(FULL_MASK, mbar_wait_bounded(mma_done, 0));
        tc::fence_after_sync();
        const float inv = (ok && l_row > 0.f) ? 1.0f / l_row : NAN;
        uint8_t* stage = sm + s * NBOX * (BM * 128);
#pragma unroll
        for (int b = ch; b < NBOX; b += 2) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t r[16];
            tmem_ld16(lane_base + o_col + b * 32 + hf * 16, r);
            tc::tmem_wait_ld();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int chunk = hf * 4 + q4;
              *reinterpret_cast<float4*>(stage + b * (BM * 128) + t * 128 + ((chunk ^ (t & 7)) << 4)) =
                  make_float4(__uint_as_float(r[4 * q4]) * inv, __uint_as_float(r[4 * q4 + 1]) * inv,
                              __uint_as_float(r[4 * q4 + 2]) * inv, __uint_as_float(r[4 * q4 + 3]) * inv);
            }
          }
        }
        fence_proxy_async_smem();
        asm volatile("bar.sync %0, 256;" :: "r"(9 + s) : "memory");        // the slot's 8 warps
        if (ch == 0 && t == 0) {
          for (int b = 0; b < NBOX; ++b) tc::tma_store_4d(&tmO, stage + b * (BM * 128), b * 32, h, sl.qt[s] * BM, n);
          tc::bulk_commit_group();
          tc::bulk_wait_read_all();
        }
      } else {
        // epilogue, permuted rows: O / l -> token-order output row from each thread (its 16-column
        // chunks).  The TMEM loads are warp-collective, so every lane loads; only rows inside the
        // sequence store.
        if (ok && nk > 0) ok = __all_sync(FULL_MASK, mbar_wait_bounded(&pv_done[s], (uint32_t)((nk - 1) & 1)));
        tc::fence_after_sync();
        float* o = a.out + (((int64_t)n * a.S + (row_valid ? row : 0)) * a.Hq + h) * D;
        const float inv = (ok && l_row > 0.f) ? 1.0f / l_row : NAN;
#pragma unroll
        for (int c = ch; c < DN / 16; c += 2) {
          uint32_t r[16];
          tmem_ld16(lane_base + o_col + c * 16, r);
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
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == MMA_WARP) tc::tmem_dealloc(tmem, TMEM_COLS);
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

// q [N, S, Hq, D] bf16 as (D, Hq, S, N): boxes of [128 rows x 64 columns] of one head.
cudaError_t make_q_map(CUtensorMap* map, const PrefillArgs& a) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {(cuuint64_t)a.D, (cuuint64_t)a.Hq, (cuuint64_t)a.S, (cuuint64_t)a.N};
  const cuuint64_t strides[3] = {(cuuint64_t)a.D * 2, (cuuint64_t)a.Hq * a.D * 2, (cuuint64_t)a.S * a.Hq * a.D * 2};
  const cuuint32_t box[4] = {64, 1, BM, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.q), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// out [N, S, Hq, D] fp32 as (D, Hq, S, N): stores of [128 rows x 32 columns] boxes.
cudaError_t make_out_map(CUtensorMap* map, const PrefillArgs& a) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {(cuuint64_t)a.D, (cuuint64_t)a.Hq, (cuuint64_t)a.S, (cuuint64_t)a.N};
  const cuuint64_t strides[3] = {(cuuint64_t)a.D * 4, (cuuint64_t)a.Hq * a.D * 4, (cuuint64_t)a.S * a.Hq * a.D * 4};
  const cuuint32_t box[4] = {32, 1, BM, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.out, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
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
  constexpr int SMEM = Layout<D>::SMEM;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  CUtensorMap mk, mv, mq, mo;
  cudaError_t e = make_cache_map(&mk, a.kc, a);
  if (e != cudaSuccess) return e;
  if ((e = make_cache_map(&mv, a.vc, a)) != cudaSuccess) return e;
  if ((e = make_q_map(&mq, a)) != cudaSuccess) return e;
  if ((e = make_out_map(&mo, a)) != cudaSuccess) return e;
  const int nq = (a.S + BM - 1) / BM;
  const int G = a.Hq / a.Hkv;
  // slots: the two heads of a GQA pair (heaviest row tiles launched first), else two row tiles
  const dim3 grid = (G % 2 == 0) ? dim3(a.Hq / 2, a.N, nq) : dim3(a.Hq, a.N, (nq + 1) / 2);
  return launch_pdl(prefill_tc_kernel<D>, grid, dim3(THREADS), (size_t)SMEM, s, a, mk, mv, mq, mo);
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
