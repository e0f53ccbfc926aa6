// Kernel (b), tensor-core form: flash-style prefill attention on tcgen05 (bf16 operands,
// fp32 accumulation in tensor memory), persistent.
//
// Work unit: two 128-row query tiles ("slots") that read the same KV head: the two query
// heads of a GQA group at the same rows when the group size is even (each K/V tile is loaded
// once for both), otherwise two row tiles of one head: tiles t and n-1-t so that causal work is
// balanced, or neighbouring tiles 2t and 2t+1 under a window mask (their key ranges overlap,
// where t and n-1-t would see disjoint windows one after the other).  One CTA per SM walks units b, 2P-1-b, 2P+b, ... (a snake over the P
// CTAs, which evens out the causal cost), so a unit's epilogue overlaps the next unit's Q load
// and first Q K^T.
//
// Twelve warps (three warpgroups) with fixed roles:
//   warps 0-3, 4-7  softmax of slot 0 and slot 1: thread t of a group owns row t = TMEM lane
//              t.  Per key tile it reads the row's 128 fp32 scores from TMEM, applies the
//              row's visible-key range (causal, window segment or full), keeps the running
//              max and sum, and writes P = exp2(S - m) back over the same columns as packed
//              bf16 pairs; 32-key chunks hidden from every row of the warp (most of a causal
//              diagonal tile) are skipped and get P = 0.  O is rescaled only when the row max
//              grows by more than 2^8 (the stale max keeps every P <= 256).  At the end of a
//              unit it copies O out of TMEM (which frees it for the next unit's P V), divides
//              by the row sum and sends the rows out in 16-column chunks through two 32 x 16
//              staging tiles per warp: TMA tensor stores for token-order rows (the warp moves
//              on while they drain), plain stores to each row's destination when the rows are
//              permuted.
//   warp 8     TMA producer: per unit the slots' Q tiles (once the previous unit's last
//              Q K^T has read its Q), then K and V tiles (64-column, 128-byte swizzled boxes)
//              into 2-stage K and V rings that run on across units (a K stage frees as soon
//              as its Q K^T is done, a V stage after its P V); rows past the valid keys read
//              as zeros.
//   warp 9     MMA issuer (one thread).  TMEM: S of slot s at columns [128 s, 128 s + 128),
//              O of slot s at [256 + 128 s, ...).  Per key tile j it issues, for s = 0, 1:
//              O_s += P_s(j) V_j once slot s's softmax has written P_s(j), then
//              S_s(j+1) = Q_s K_{j+1}^T into the same columns (tensor-core operations of one
//              thread run in issue order, so the P V read precedes the overwrite).  While one
//              slot's warps run the softmax of tile j, the tensor core works on the other
//              slot's P V and next S: the two slots ping-pong.
// Every mbarrier wait is bounded; a timeout stops the CTA and marks its remaining output rows
// NaN instead of hanging.
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
constexpr int SOFTMAX_WARPS = 8;          // 4 per slot, one row per thread
constexpr int TMA_WARP = 8, MMA_WARP = 9;  // warps 10, 11 complete their warpgroup and idle
constexpr int THREADS = 384;
// Registers per thread: 168 at launch (65536 / 384, rounded down to a multiple of 8); the
// producer/MMA warpgroup gives up 48 per thread, which the two softmax warpgroups take:
// 128 * (192 + 192 + 120) = 384 * 168, so the increase never waits on registers nobody frees.
constexpr int REGS_LAUNCH = 168, REGS_SOFTMAX = 192, REGS_CONTROL = 120;
static_assert(2 * REGS_SOFTMAX + REGS_CONTROL <= 3 * REGS_LAUNCH, "register split exceeds the launch total");
static_assert(REGS_LAUNCH * THREADS <= 65536, "launch registers");
constexpr int SUB = BM * 128;             // bytes of one [128 rows x 64 bf16] swizzled box
constexpr int ST_BYTES = 32 * 64;         // one staging tile: 32 rows x 16 fp32 (64-byte swizzle)
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;

// D: q and key width, DV: value width, NST: stages of the K and of the V ring.
template <int D, int DV, int NST>
struct Layout {
  static constexpr int NSUB = (D + 63) / 64;                 // 64-column boxes of a q / key row
  static constexpr int NSUBV = (DV + 63) / 64;               // 64-column boxes of a value row
  static constexpr int Q_OFF = 0;                            // [2 slots][NSUB boxes]
  static constexpr int K_OFF = Q_OFF + 2 * NSUB * SUB;       // [NST][NSUB]
  static constexpr int V_OFF = K_OFF + NST * NSUB * SUB;     // [NST][NSUBV]
  static constexpr int ST_OFF = V_OFF + NST * NSUBV * SUB;   // [softmax warp][2]
  static constexpr int BAR_OFF = ST_OFF + SOFTMAX_WARPS * 2 * ST_BYTES;
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
// First slot and one past the last slot of segment id g: from the launch's table when g is in
// it, else by bisecting the ids (11 dependent loads for 1288 slots, on every unit's start).
__device__ __forceinline__ int seg_first(const PrefillArgs& a, int g) {
  return (unsigned)g < (unsigned)a.seg_table ? a.seg_lo[g] : seg_lower_tc(a.segment, a.S, g);
}
__device__ __forceinline__ int seg_end(const PrefillArgs& a, int g) {
  return (unsigned)g < (unsigned)a.seg_table ? a.seg_hi[g] : seg_upper_tc(a.segment, a.S, g);
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
// 16 consecutive TMEM columns of this thread's lane, into x[0..16) as floats.
__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float* x) {
  uint32_t r[16];
  tmem_ld16(taddr, r);
#pragma unroll
  for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(r[e]);
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
// Two floats to packed bf16 (round to nearest even) in one instruction: lo in bits 0..15.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Unit geometry: units are numbered x fastest (KV-head pair or head), then instance, then
// the row-tile index z, with z = 0 the heaviest causal tiles.  When even one tile per unit
// leaves SMs idle (a short prompt of one layer), every unit holds a single query tile (slot 1
// empty), so twice as many SMs share the work.
struct Units {
  int X, Z, total;
};
__host__ __device__ __forceinline__ Units unit_geometry_of(int N, int S, int Hq, int Hkv, bool single) {
  const int nq = (S + BM - 1) / BM;
  const bool pair_heads = (Hq / Hkv) % 2 == 0;
  Units g;
  g.X = (single || !pair_heads) ? Hq : Hq / 2;
  g.Z = (single || pair_heads) ? nq : (nq + 1) / 2;
  g.total = g.X * N * g.Z;
  return g;
}
__device__ __forceinline__ Units unit_geometry(const PrefillArgs& a) {
  return unit_geometry_of(a.N, a.S, a.Hq, a.Hkv, a.single_slot != 0);
}
// The r-th unit of CTA b out of P (snake order), or -1 past the end.
__device__ __forceinline__ int unit_of(int r, int b, int P, int total) {
  const int u = r * P + ((r & 1) ? (P - 1 - b) : b);
  return u < total ? u : -1;
}

// The two slots of a unit: (query head, row tile) each, or an empty slot (qt < 0).
struct Slots {
  int h[2], qt[2], n;
};
__device__ __forceinline__ Slots unit_slots(const PrefillArgs& a, const Units& g, int u) {
  Slots sl;
  const int nq = (a.S + BM - 1) / BM;
  const int x = u % g.X, n = (u / g.X) % a.N, z = u / (g.X * a.N);
  sl.n = n;
  if (a.single_slot) {             // one query tile, heaviest row tiles first
    sl.h[0] = sl.h[1] = x;
    sl.qt[0] = nq - 1 - z;
    sl.qt[1] = -1;
  } else if ((a.Hq / a.Hkv) % 2 == 0) {   // the two heads of a pair, heaviest row tiles first
    sl.h[0] = 2 * x; sl.h[1] = 2 * x + 1;
    sl.qt[0] = sl.qt[1] = nq - 1 - z;
  } else if (a.mask == KVA_MASK_SEGMENT) {   // row tiles 2z and 2z+1 of one head: their windows
    sl.h[0] = sl.h[1] = x;                    // overlap, so the two slots share key tiles
    sl.qt[0] = 2 * z;
    sl.qt[1] = 2 * z + 1 < nq ? 2 * z + 1 : -1;
  } else {                         // row tiles z and nq-1-z of one head (balanced causal work)
    sl.h[0] = sl.h[1] = x;
    sl.qt[0] = z;
    sl.qt[1] = nq - 1 - z;
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
    lo = seg_first(a, a.segment[i0]);
    hi = seg_end(a, a.segment[i_last]);
  } else if (a.mask == KVA_MASK_CAUSAL_SEGMENT) {
    hi = seg_end(a, a.segment[i_last]);    // the last row's segment end
  }
}

// Key tiles of each slot of a unit, [js0, js1), their union [j0, j1) and the tile walk.
struct TileRanges {
  int js0[2], js1[2], j0, j1;
  bool act1;
  __device__ __forceinline__ bool active(int s, int j) const {
    return (s == 0 || act1) && j >= js0[s] && j < js1[s];
  }
  // Key tiles the CTA loads: those some slot needs, in increasing order (the two slots' ranges
  // may be disjoint under a window mask).  Producer and MMA walk the same list; its entries
  // number the ring stages and barrier phases.
  __device__ __forceinline__ int next_tile(int j) const {
    ++j;
    while (j < j1 && !active(0, j) && !active(1, j)) ++j;
    return j;
  }
  __device__ __forceinline__ int ntiles(int s) const { return (s == 0 || act1) ? js1[s] - js0[s] : 0; }
};
__device__ __forceinline__ TileRanges tile_ranges(const PrefillArgs& a, const Slots& sl) {
  TileRanges tr;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    if (sl.qt[s] < 0) { tr.js0[s] = tr.js1[s] = 0; continue; }
    const int i0 = sl.qt[s] * BM, i_last = min(a.S, i0 + BM) - 1;
    int lo, hi;
    tile_keys(a, i0, i_last, lo, hi);
    tr.js0[s] = lo / BN; tr.js1[s] = (hi + BN - 1) / BN;
  }
  tr.act1 = sl.qt[1] >= 0;
  tr.j0 = tr.act1 ? min(tr.js0[0], tr.js0[1]) : tr.js0[0];
  tr.j1 = tr.act1 ? max(tr.js1[0], tr.js1[1]) : tr.js1[0];
  return tr;
}

// A wait gave up: the CTA's unfinished rows of slot s (from its r-th unit on) become NaN, by
// plain stores.  Out of line: it never runs in a healthy launch.
template <int DV, bool GATHER>
__device__ __noinline__ void nan_rows(const PrefillArgs& a, const Units& ug, int r, int b, int P, int s, int t) {
  for (;; ++r) {
    const int u = unit_of(r, b, P, ug.total);
    if (u < 0) break;
    const Slots sl = unit_slots(a, ug, u);
    if (sl.qt[s] < 0) continue;
    const int i = sl.qt[s] * BM + t;
    if (i >= a.S) continue;
    const int row = GATHER ? a.row_of_slot[i] : i;
    if (row < 0 || row >= a.S) continue;
    float* o = a.out + (((int64_t)sl.n * a.S + row) * a.Hq + sl.h[s]) * DV;
    for (int d = 0; d < DV; ++d) o[d] = NAN;
  }
}

template <int D, int DV, int NST, bool GATHER>
__global__ void __launch_bounds__(THREADS, 1)
prefill_tc_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmO) {
  using LY = Layout<D, DV, NST>;
  constexpr int DK = (D + 15) / 16 * 16;      // MMA K extent of Q K^T (zero padded)
  constexpr int DN = (DV + 15) / 16 * 16;     // MMA N extent of P V
  constexpr int KSTEPS = DK / 16;
  constexpr int NSUB = LY::NSUB, NSUBV = LY::NSUBV;
  constexpr int NCH = (DV + 15) / 16;         // 16-column output chunks
  constexpr uint32_t IDESC_S = tc::idesc_bf16(BM, BN, 0, 0);
  constexpr uint32_t IDESC_PV = tc::idesc_bf16(BM, DN, 0, 1);
  static_assert(DN % 16 == 0 && DN <= 128, "N extent");
  static_assert(NST == 1 || NST == 2, "ring stages (two barrier slots each)");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + LY::BAR_OFF);
  uint64_t* k_full = bars + 0;     // [NST] K tile landed
  uint64_t* k_free = bars + 2;     // [NST] both slots' Q K^T of the tile done: K stage free
  uint64_t* v_full = bars + 4;     // [NST] V tile landed
  uint64_t* v_free = bars + 6;     // [NST] both slots' P V of the tile done: V stage free
  uint64_t* s_full = bars + 8;     // [slot] S ready in TMEM
  uint64_t* p_full = bars + 10;    // [slot] P written to TMEM by the slot's 4 warps
  uint64_t* pv_done = bars + 12;   // [slot] P V of the slot's tile finished
  uint64_t* q_full = bars + 14;    // [slot] Q tile landed (TMA) or staged by the slot's 4 warps
  uint64_t* o_full = bars + 16;    // [slot] the unit's last P V done: O final in TMEM
  uint64_t* o_free = bars + 18;    // [slot] O copied out of TMEM by the slot's 4 warps
  uint64_t* q_free = bars + 20;    // the unit's last Q K^T done: both Q tiles may be replaced
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(bars + 21);
  volatile int* s_abort = reinterpret_cast<volatile int*>(bars + 22);
  constexpr bool gather = GATHER;               // permuted rows: threads stage Q and store O

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Units ug = unit_geometry(a);
  const int P = gridDim.x, b = blockIdx.x;

  if (warp == MMA_WARP) tc::tmem_alloc(s_taddr, TMEM_COLS);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1); mbar_init(&k_free[i], 1); mbar_init(&v_full[i], 1); mbar_init(&v_free[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], SOFTMAX_WARPS / 2); mbar_init(&pv_done[i], 1);
      mbar_init(&q_full[i], gather ? SOFTMAX_WARPS / 2 : 1);
      mbar_init(&o_full[i], 1); mbar_init(&o_free[i], SOFTMAX_WARPS / 2);
    }
    mbar_init(q_free, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == TMA_WARP && lane == 0) {
    tc::tma_prefetch_desc(&tmK); tc::tma_prefetch_desc(&tmV); tc::tma_prefetch_desc(&tmQ);
    if (!gather) tc::tma_prefetch_desc(&tmO);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_taddr;
  // Registers move from the control warpgroup to the softmax warpgroups (warpgroup-wide; each
  // role's code follows its own setmaxnreg so the compiler budgets it with that count).
  if (warp >= SOFTMAX_WARPS) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(REGS_CONTROL));
    griddep_wait();                            // inputs of this launch are complete from here on
    griddep_launch_dependents();
  if (warp == TMA_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      int it = 0;                               // ring entries issued so far (all units)
      int nu = 0;                               // units begun so far
      for (int r = 0; ok; ++r, ++nu) {
        const int u = unit_of(r, b, P, ug.total);
        if (u < 0) break;
        const Slots sl = unit_slots(a, ug, u);
        const TileRanges tr = tile_ranges(a, sl);
        const int g = sl.h[0] / (a.Hq / a.Hkv);
        if (!gather) {
          // the previous unit's last Q K^T has read both Q tiles
          if (nu > 0 && !mbar_wait_bounded(q_free, (uint32_t)((nu - 1) & 1))) { ok = false; break; }
          for (int s = 0; s < 2; ++s) {
            if (s == 1 && !tr.act1) break;
            mbar_arrive_expect_tx(&q_full[s], NSUB * SUB);
            for (int c = 0; c < NSUB; ++c)
              tc::tma_load_4d(sm + LY::Q_OFF + (s * NSUB + c) * SUB, &tmQ, c * 64, sl.h[s], sl.qt[s] * BM, sl.n,
                              &q_full[s]);
          }
        }
        for (int j = tr.j0; j < tr.j1; j = tr.next_tile(j), ++it) {
          // K and V of a tile use separate stages: K is free again once both slots' Q K^T have
          // run (early in the tile), V only after both P V
          const int st = it % NST;
          const uint32_t ph = (uint32_t)((it / NST - 1) & 1);
          const int key0 = j * BN;
          if (it >= NST && !mbar_wait_bounded(&k_free[st], ph)) { ok = false; break; }
          mbar_arrive_expect_tx(&k_full[st], NSUB * SUB);
          for (int c = 0; c < NSUB; ++c)
            tc::tma_load_4d(sm + LY::K_OFF + (st * NSUB + c) * SUB, &tmK, c * 64, key0, g, sl.n, &k_full[st]);
          if (it >= NST && !mbar_wait_bounded(&v_free[st], ph)) { ok = false; break; }
          mbar_arrive_expect_tx(&v_full[st], NSUBV * SUB);
          for (int c = 0; c < NSUBV; ++c)
            tc::tma_load_4d(sm + LY::V_OFF + (st * NSUBV + c) * SUB, &tmV, c * 64, key0, g, sl.n, &v_full[st]);
        }
        if (*s_abort) ok = false;
      }
      if (!ok) *s_abort = 1;
      // the copies this CTA issued have normally landed long ago; never leave one in flight
      for (int e = max(0, it - NST); e < it; ++e) {
        mbar_wait_bounded(&k_full[e % NST], (uint32_t)((e / NST) & 1));
        mbar_wait_bounded(&v_full[e % NST], (uint32_t)((e / NST) & 1));
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      const uint64_t q_desc0 = tc::desc_at(DESC_KMAJ, smem_u32(sm + LY::Q_OFF));
      const uint64_t q_desc1 = tc::desc_at(DESC_KMAJ, smem_u32(sm + LY::Q_OFF + NSUB * SUB));
      const uint64_t k_desc0 = tc::desc_at(DESC_KMAJ, smem_u32(sm + LY::K_OFF));
      const uint64_t v_desc0 = tc::desc_at(DESC_VMN, smem_u32(sm + LY::V_OFF));
      // descriptor start addresses advance by constant offsets (addresses stay below 2^18)
      constexpr uint64_t K_STAGE = (uint64_t)(NSUB * SUB) >> 4, V_STAGE = (uint64_t)(NSUBV * SUB) >> 4;
      int it = 0;                               // ring entries consumed so far
      int ks[2] = {0, 0};                       // key tiles of each slot so far
      int nus[2] = {0, 0};                      // units in which each slot was active so far
      for (int r = 0; ok; ++r) {
        const int u = unit_of(r, b, P, ug.total);
        if (u < 0) break;
        const Slots sl = unit_slots(a, ug, u);
        const TileRanges tr = tile_ranges(a, sl);
        const int s_total = tr.ntiles(0) + tr.ntiles(1);
        int s_issued = 0;
        ok = mbar_wait_bounded(&q_full[0], (uint32_t)(nus[0] & 1)) &&
             (!tr.act1 || mbar_wait_bounded(&q_full[1], (uint32_t)(nus[1] & 1)));
        tc::fence_after_sync();
        auto issue_s = [&](int s, int e) {
          const uint64_t qd = s ? q_desc1 : q_desc0;
          const uint64_t kd = k_desc0 + (uint64_t)(e % NST) * K_STAGE;
#pragma unroll
          for (int k = 0; k < KSTEPS; ++k) {
            // descriptor start addresses advance by constant offsets (addresses stay below 2^18)
            const uint64_t off = (uint64_t)((((k >> 2) * SUB) + (k & 3) * 32) >> 4);
            tc::mma_ss(tmem + s * BN, qd + off, kd + off, IDESC_S, k > 0);
          }
          tc::mma_commit(&s_full[s]);
          if (++s_issued == s_total) tc::mma_commit(q_free);   // the unit's last Q K^T
        };
        if (ok) {
          ok = mbar_wait_bounded(&k_full[it % NST], (uint32_t)((it / NST) & 1));
          tc::fence_after_sync();
#pragma unroll
          for (int s = 0; s < 2; ++s)
            if (ok && tr.active(s, tr.j0)) issue_s(s, it);
          tc::mma_commit(&k_free[it % NST]);            // this K stage is free once those finish
        }
        for (int j = tr.j0; ok && j < tr.j1; ++it) {
          const int st = it % NST;
          const int jn = tr.next_tile(j);              // the tile loaded after j (entry it + 1)
          bool next_landed = false, v_landed = false;
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            if (!ok) continue;
            if (tr.active(s, j)) {
              const int k = j - tr.js0[s];
              if (!mbar_wait_bounded(&p_full[s], (uint32_t)((ks[s] + k) & 1))) { ok = false; continue; }
              if (!v_landed) {
                if (!mbar_wait_bounded(&v_full[st], (uint32_t)((it / NST) & 1))) { ok = false; continue; }
                v_landed = true;
              }
              // the first P V of a unit overwrites O: the previous unit's O must have been read
              if (k == 0 && nus[s] > 0 && !mbar_wait_bounded(&o_free[s], (uint32_t)((nus[s] - 1) & 1))) { ok = false; continue; }
              tc::fence_after_sync();
              const uint64_t vd = v_desc0 + (uint64_t)st * V_STAGE;
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk)
                tc::mma_ts(tmem + 256 + s * 128, tmem + s * BN + kk * 8, vd + (uint64_t)(kk * 2048 >> 4),
                           IDESC_PV, (k > 0 || kk > 0));
              tc::mma_commit(&pv_done[s]);
              if (j == tr.js1[s] - 1) tc::mma_commit(&o_full[s]);
            }
            if (jn < tr.j1 && tr.active(s, jn)) {
              if (!next_landed) {
                if (!mbar_wait_bounded(&k_full[(it + 1) % NST], (uint32_t)(((it + 1) / NST) & 1))) { ok = false; continue; }
                tc::fence_after_sync();
                next_landed = true;
              }
              issue_s(s, it + 1);
            }
          }
          if (!ok) break;
          tc::mma_commit(&v_free[st]);              // V of this tile: free once both P V are done
          if (jn < tr.j1) tc::mma_commit(&k_free[(it + 1) % NST]);   // K of the next: after its Q K^T
          j = jn;
        }
#pragma unroll
        for (int s = 0; s < 2; ++s)
          if (s == 0 || tr.act1) { ks[s] += tr.ntiles(s); ++nus[s]; }
        if (*s_abort) ok = false;
      }
      if (!ok) *s_abort = 1;
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(REGS_SOFTMAX));
    griddep_wait();
    griddep_launch_dependents();
    // ------------------------------------------------------------ softmax warps
    const int s = warp >> 2;                    // slot
    const int quarter = warp & 3;               // TMEM lane quarter of this warp
    const int t = quarter * 32 + lane;          // row within the tile = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_col = s * BN, o_col = 256 + s * 128;
    uint8_t* stage = sm + LY::ST_OFF + warp * 2 * ST_BYTES;
    uint8_t* sQ = sm + LY::Q_OFF + s * NSUB * SUB;
    bool ok = true;
    int ks = 0, nus = 0, nu = 0;                // tiles and active units of this slot, units begun
    int r = 0;
    for (; ok; ++r, ++nu) {
      const int u = unit_of(r, b, P, ug.total);
      if (u < 0) break;
      const Slots sl = unit_slots(a, ug, u);
      const TileRanges tr = tile_ranges(a, sl);
      if (s == 1 && !tr.act1) continue;         // the slot is empty in this unit
      const int h = sl.h[s], n = sl.n;
      const int i = sl.qt[s] * BM + t;
      const bool row_ok = i < a.S;
      int row = i;
      if (row_ok && gather) row = a.row_of_slot[i];
      const bool row_valid = row_ok && row >= 0 && row < a.S;
      if (gather) {
        // permuted rows: stage this thread's Q row once the previous unit's last Q K^T is done.
        // Chunk c (8 bf16) -> box c/8, swizzled position (c%8) ^ (t%8)
        if (nu > 0 && !__all_sync(FULL_MASK, mbar_wait_bounded(q_free, (uint32_t)((nu - 1) & 1)))) { ok = false; break; }
        const uint4* src = reinterpret_cast<const uint4*>(
            reinterpret_cast<const uint16_t*>(a.q) + (((int64_t)n * a.S + row) * a.Hq + h) * D);
#pragma unroll
        for (int c = 0; c < DK / 8; ++c) {
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
        else if (a.mask == KVA_MASK_CAUSAL_SEGMENT) { rlo = 0; rhi = seg_end(a, a.segment[i]); }
        else { const int sg = a.segment[i]; rlo = seg_first(a, sg); rhi = seg_end(a, sg); }
      }
      const int nk = tr.ntiles(s);
      float m = -INFINITY, l = 0.f;
      float x[128];
      for (int k = 0; k < nk; ++k) {
        const int kk = ks + k;
        const int kv0 = (tr.js0[s] + k) * BN;          // first key of the tile
        // every lane waits; the vote keeps the warp converged for the .aligned TMEM accesses
        if (!__all_sync(FULL_MASK, mbar_wait_bounded(&s_full[s], (uint32_t)(kk & 1)))) { ok = false; break; }
        tc::fence_after_sync();
        // visible columns of this row in the tile: [clo, chi).  A 32-column chunk that no row
        // of the warp sees is not exponentiated (its P is zero).
        const int clo = rlo - kv0, chi = rhi - kv0;
        unsigned live = 0u;
        {
          const int lo_min = __reduce_min_sync(FULL_MASK, clo), hi_max = __reduce_max_sync(FULL_MASK, chi);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            if (32 * cc < hi_max && 32 * cc + 32 > lo_min) live |= 1u << cc;
        }
        {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tc::tmem_ld32(lane_base + s_col, r0);
          tc::tmem_ld32(lane_base + s_col + 32, r1);
          tc::tmem_ld32(lane_base + s_col + 64, r2);
          tc::tmem_ld32(lane_base + s_col + 96, r3);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = __uint_as_float(r0[e]); x[32 + e] = __uint_as_float(r1[e]);
            x[64 + e] = __uint_as_float(r2[e]); x[96 + e] = __uint_as_float(r3[e]);
          }
        }
        if (clo > 0 || chi < BN) {
#pragma unroll
          for (int e = 0; e < BN; ++e)
            if (e < clo || e >= chi) x[e] = -INFINITY;
        }
        // row max: four independent chains, then combined (a single chain would serialise 64
        // dependent max instructions)
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < BN; e += 8) {
#pragma unroll
          for (int c = 0; c < 4; ++c) mq[c] = fmax3(mq[c], x[e + 2 * c], x[e + 2 * c + 1]);
        }
        const float mr = fmaxf(fmax3(mq[0], mq[1], mq[2]), mq[3]);
        const float m_tile = mr == -INFINITY ? -INFINITY : mr * a.scale_log2;
        const float m_new = fmaxf(m, m_tile);
        const bool first = (m == -INFINITY);            // first visible keys: O holds nothing yet
        const bool grow = !first && m_new > m + RESCALE_LOG2;
        if (first) m = m_new;
        if (__any_sync(FULL_MASK, grow)) {
          // some row's max grew by > 2^8: rescale those rows of O once P V of the previous tile
          // has landed.  The whole warp takes part (TMEM accesses are warp-collective); rows
          // that need no rescale use alpha = 1.
          if (!__all_sync(FULL_MASK, mbar_wait_bounded(&pv_done[s], (uint32_t)((kk - 1) & 1)))) { ok = false; break; }
          tc::fence_after_sync();
          const float alpha = grow ? ex2(m - m_new) : 1.0f;
#pragma unroll
          for (int c = 0; c < DN / 16; ++c) {
            uint32_t rr[16];
            tmem_ld16(lane_base + o_col + c * 16, rr);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
            tmem_st16(lane_base + o_col + c * 16, rr);
          }
          tc::tmem_wait_st();
          if (grow) { l *= alpha; m = m_new; }
        }
        // P = exp2(S * scale - m) as packed bf16 into columns [0, 64) of the slot
        const float mref = (m == -INFINITY) ? 0.f : m;
        const uint64_t sc2 = f2(a.scale_log2, a.scale_log2), nm2 = f2(-mref, -mref);
        uint64_t lsum = f2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w[16];
          if ((live >> c) & 1u) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float x0, x1;
              f2split(ffma2(f2(x[32 * c + 2 * e], x[32 * c + 2 * e + 1]), sc2, nm2), x0, x1);
              const float p0 = ex2(x0), p1 = ex2(x1);       // hidden keys hold -inf: exp2 -> 0
              lsum = fadd2(lsum, f2(p0, p1));
              w[e] = cvt_bf16x2(p0, p1);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = 0u;
          }
          tmem_st16(lane_base + s_col + c * 16, w);
        }
        float l0, l1;
        f2split(lsum, l0, l1);
        l += l0 + l1;
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[s]);
      }
      if (!ok) break;
      // epilogue: copy O out of TMEM (freeing it for the next unit's first P V), then O / l
      if (!__all_sync(FULL_MASK, mbar_wait_bounded(&o_full[s], (uint32_t)(nus & 1)))) { ok = false; break; }
      tc::fence_after_sync();
#pragma unroll
      for (int c = 0; c < DN / 16; ++c) tmem_ld16f(lane_base + o_col + c * 16, x + 16 * c);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[s]);
      const float inv = l > 0.f ? 1.0f / l : NAN;
      // O / l goes out in 16-column chunks through this warp's two staging tiles (32 rows x
      // 64 bytes, 16-byte piece k of row r at position k ^ ((r >> 1) & 3): the tensor map's
      // 64-byte swizzle, and conflict-free for the row-per-lane writes).
      if (!gather) {
        // token-order rows: one TMA store per chunk (rows past the sequence and columns past
        // the value width are clipped by the tensor map).  A staging tile is rewritten only
        // once the store issued from it two chunks earlier has read it.
        const int row0 = sl.qt[s] * BM + quarter * 32;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          uint8_t* buf = stage + (c & 1) * ST_BYTES;
          if (lane == 0) tc::bulk_wait_read_1();
          __syncwarp();
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float* xs = x + 16 * c + 4 * k4;
            *reinterpret_cast<float4*>(buf + lane * 64 + ((k4 ^ ((lane >> 1) & 3)) << 4)) =
                make_float4(xs[0] * inv, xs[1] * inv, xs[2] * inv, xs[3] * inv);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tc::tma_store_4d(&tmO, buf, c * 16, h, row0, n);
            tc::bulk_commit_group();
          }
        }
      } else {
        // permuted rows: transposed through the staging tile so that every store instruction
        // writes 8 rows x 64 contiguous bytes (lane 4 j + q stores piece q of rows j, j + 8,
        // j + 16, j + 24); each row's token-order destination is resolved per row.
        const int my_row = row_valid ? row : -1;
        float* orow[4];
#pragma unroll
        for (int p4 = 0; p4 < 4; ++p4) {
          const int rr = __shfl_sync(FULL_MASK, my_row, (lane >> 2) + 8 * p4);
          orow[p4] = rr < 0 ? nullptr : a.out + (((int64_t)n * a.S + rr) * a.Hq + h) * DV + (lane & 3) * 4;
        }
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          uint8_t* buf = stage + (c & 1) * ST_BYTES;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float* xs = x + 16 * c + 4 * k4;
            *reinterpret_cast<float4*>(buf + lane * 64 + ((k4 ^ ((lane >> 1) & 3)) << 4)) =
                make_float4(xs[0] * inv, xs[1] * inv, xs[2] * inv, xs[3] * inv);
          }
          __syncwarp();
#pragma unroll
          for (int p4 = 0; p4 < 4; ++p4) {
            const int rr = (lane >> 2) + 8 * p4, q = lane & 3;
            const float4 v = *reinterpret_cast<const float4*>(buf + rr * 64 + ((q ^ ((rr >> 1) & 3)) << 4));
            if (orow[p4] != nullptr && c * 16 + q * 4 < DV) *reinterpret_cast<float4*>(orow[p4] + c * 16) = v;
          }
        }
      }
      ks += nk;
      ++nus;
      if (*s_abort) { ok = false; break; }
    }
    if (!ok) {
      *s_abort = 1;
      nan_rows<DV, GATHER>(a, ug, r, b, P, s, t);
    }
  }

  if (warp < SOFTMAX_WARPS && lane == 0) tc::bulk_wait_all();   // this warp's output stores are done
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

// Cache view for TMA: dims (width, S valid slots, Hkv, N); rows >= S read as zeros.
cudaError_t make_cache_map(CUtensorMap* map, const void* base, const PrefillArgs& a, int width, int64_t inst_stride) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {(cuuint64_t)width, (cuuint64_t)a.S, (cuuint64_t)a.Hkv, (cuuint64_t)a.N};
  const cuuint64_t strides[3] = {(cuuint64_t)width * 2, (cuuint64_t)a.capacity * width * 2, (cuuint64_t)inst_stride * 2};
  const cuuint32_t box[4] = {64, BN, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// out [N, S, Hq, Dv] fp32 as (Dv, Hq, S, N): boxes of [32 rows x 16 columns] of one head, with
// 64-byte swizzle (the layout of the softmax warps' staging tiles).
cudaError_t make_out_map(CUtensorMap* map, const PrefillArgs& a) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {(cuuint64_t)a.Dv, (cuuint64_t)a.Hq, (cuuint64_t)a.S, (cuuint64_t)a.N};
  const cuuint64_t strides[3] = {(cuuint64_t)a.Dv * 4, (cuuint64_t)a.Hq * a.Dv * 4,
                                 (cuuint64_t)a.S * a.Hq * a.Dv * 4};
  const cuuint32_t box[4] = {16, 1, 32, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.out, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int prefill_num_sms() {
  static int n[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (n[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    n[dev] = v;
  }
  return n[dev];
}

template <int D, int DV, int NST, bool GATHER>
cudaError_t launch_g(const PrefillArgs& a, cudaStream_t s) {
  constexpr int SMEM = Layout<D, DV, NST>::SMEM;
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static DeviceOnce configured;
  if (!configured.done()) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D, DV, NST, GATHER>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    // the register split assumes the launch holds exactly REGS_LAUNCH per thread: with fewer,
    // the softmax warpgroups' setmaxnreg.inc could never be satisfied
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, prefill_tc_kernel<D, DV, NST, GATHER>)) != cudaSuccess) return e;
    if (fa.numRegs != REGS_LAUNCH) return cudaErrorInvalidDeviceFunction;
    configured.mark();
  }
  CUtensorMap mk, mv, mq;
  cudaError_t e = make_cache_map(&mk, a.kc, a, D, a.inst_stride);
  if (e != cudaSuccess) return e;
  if ((e = make_cache_map(&mv, a.vc, a, DV, a.inst_stride_v)) != cudaSuccess) return e;
  if ((e = make_q_map(&mq, a)) != cudaSuccess) return e;
  CUtensorMap mo;
  std::memset(&mo, 0, sizeof(mo));           // unused when rows are permuted
  if (a.row_of_slot == nullptr && (e = make_out_map(&mo, a)) != cudaSuccess) return e;
  // units: the two heads of a GQA pair at one row tile, else two row tiles of one head; one
  // query tile per unit when even that many units would fill at most one wave
  const long long nq = (a.S + BM - 1) / BM;
  const int G = a.Hq / a.Hkv;
  const long long paired = (G % 2 == 0) ? (long long)(a.Hq / 2) * a.N * nq : (long long)a.Hq * a.N * ((nq + 1) / 2);
  if (paired <= 0) return cudaSuccess;
  const long long singles = (long long)a.Hq * a.N * nq;
  PrefillArgs b = a;
  b.single_slot = singles <= prefill_num_sms() ? 1 : 0;
  const long long units = b.single_slot ? singles : paired;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int grid = (int)std::min<long long>(units, prefill_num_sms());
  return launch_pdl(prefill_tc_kernel<D, DV, NST, GATHER>, dim3(grid), dim3(THREADS), (size_t)SMEM, s, b, mk, mv, mq, mo);
}

}  // namespace

bool prefill_tc_supports(int D, int Dv, kva_dtype dt) {
  const bool shapes = (Dv == D && (D == 64 || D == 72 || D == 128)) || (D == 192 && Dv == 128);
  return dt == KVA_BF16 && shapes && encode_fn() != nullptr;
}

// Permuted rows (row_of_slot) and token-order rows are separate instantiations, so that neither
// kernel carries the other's Q staging and output path.
template <int D, int DV, int NST>
cudaError_t launch_d(const PrefillArgs& a, cudaStream_t s) {
  return a.row_of_slot != nullptr ? launch_g<D, DV, NST, true>(a, s) : launch_g<D, DV, NST, false>(a, s);
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s) {
  if (a.D == 192 && a.Dv == 128) return launch_d<192, 128, 1>(a, s);   // one K and one V stage fit
  if (a.Dv != a.D) return cudaErrorInvalidValue;
  switch (a.D) {
    case 64: return launch_d<64, 64, 2>(a, s);
    case 72: return launch_d<72, 72, 2>(a, s);
    case 128: return launch_d<128, 128, 2>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kva
