// Multi-query verify block on tcgen05 (bf16 cache, head_dim 128, a group of at most 128 rows).
//
// The G*k rows of a KV head's group (row r = (block position i = r / G, query head
// g*G + r % G); row i sees slots [0, L - k + i]) are the M rows of one 128-row tile; rows past
// the group are zero.  Work unit = (chunk c, KV head g, instance b): a run of 128-key tiles of
// instance b.  One CTA per SM walks units; inside a unit the tiles alternate between two slots
// (tile e belongs to slot e & 1), each with its own S and O in tensor memory, so while one
// slot's softmax runs the tensor core works on the other slot:
//   warps 0-3, 4-7  softmax of slot 0 and slot 1, thread t of a group owning row t (TMEM lane
//              t); only the warps holding group rows take part.  Per tile: the row's scores,
//              its visible-key limit inside the chunk, a lazily moved reference max (O is
//              rescaled only when a score exceeds it by more than 2^8), P = exp2(S - m) written
//              back over S as packed bf16.  A tile that runs past the chunk has its V rows past
//              the chunk zeroed in shared memory first (they may hold the next chunk's keys or
//              anything else), so 0 * V stays 0.  At the unit's end slot 1 publishes its row
//              max and sum, slot 0 combines both O accumulators from tensor memory and writes
//              the rows (the final output when the instance is a single chunk, else a partial
//              that the last unit of (b, g) to finish merges).  Query rows live in two buffers
//              (units alternate); fp32 rows are rounded to bf16 and staged by slot 1 for the
//              next unit as soon as it has published its statistics.
//   warp 10    TMA producer: bf16 query rows of each unit (one [64 dims x G heads x k
//              positions] box per half row, landing in (position, head) row order), K and V
//              tiles ([128 keys x 64 dims] boxes, 128-byte swizzle) of every unit in walk order
//              into a 2-stage K ring and a 3-stage V ring (a K stage frees at its Q K^T, early;
//              a V stage only at its P V, after the softmax).
//   warp 9     MMA issuer (one thread): S_s = Q K^T into slot s's columns [128 s, 128 s + 128),
//              O_s += P_s V into [256 + 128 s, ...); tensor-core operations of one thread run in
//              issue order, so a slot's next Q K^T is issued right behind its P V.
// Every mbarrier wait is bounded; a timeout stops the CTA and marks its unfinished rows NaN.
//
// Method: the target-verification forward of a draft block with a multi-token causal mask
// over the existing cache (HunyuanOCR v1.5 ncnn port, section 3.8), GQA by repeat-interleave
// grouping (Penguin-VL ncnn port, section 3), bf16 storage with fp32 accumulation
// (HunyuanOCR v1.5 ncnn port, section 3.7), softmax kept online in the flash form (MNN
// llm_demo walkthrough, section 5.1).
#include <cstring>
#include <mutex>

#include "launch.h"
#include "tc.cuh"

namespace kva {

namespace {

constexpr int D = DECODE_HEAD_DIM;        // 128
constexpr int BM = 128;                   // rows of the tile = TMEM lanes
constexpr int BN = 128;                   // keys per tile
// 8 softmax warps; warps 8-11: MMA (9) and TMA (10) issuers, two idle.  With a group of at
// most 32 rows only warps 0 and 4 (both on sub-partition 0, the only ones that reach TMEM
// lanes 0-31) do softmax work, so the issuers sit on sub-partitions 1 and 2.
constexpr int THREADS = 384;
constexpr int TMA_WARP = 10, MMA_WARP = 9;
// Registers per thread: 168 at launch (three warps per SM sub-partition); the control
// warpgroup gives up 48 per thread, which the two softmax warpgroups take:
// 128 * (192 + 192 + 120) = 384 * 168, so the increase never waits on registers nobody frees.
constexpr int REGS_LAUNCH = 168, REGS_SOFTMAX = 192, REGS_CONTROL = 120;
static_assert(2 * REGS_SOFTMAX + REGS_CONTROL <= 3 * REGS_LAUNCH, "register split exceeds the launch total");
constexpr int NK = 2, NV = 3;             // K and V ring stages
constexpr int SUB = BM * 128;             // one [128 rows x 64 bf16] swizzled box, 16 KB
constexpr int Q_OFF = 0;                  // 2 buffers x 2 boxes (units alternate)
constexpr int K_OFF = Q_OFF + 4 * SUB;    // NK x 2 boxes
constexpr int V_OFF = K_OFF + NK * 2 * SUB;
constexpr int ML_OFF = V_OFF + NV * 2 * SUB;   // slot 1's row max and sum: [2][BM] floats
constexpr int BAR_OFF = ML_OFF + 2 * BM * 4;
constexpr int SMEM = BAR_OFF + 256 + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;
static_assert(SMEM <= 232448, "shared memory per CTA");

constexpr uint64_t DESC_KMAJ = tc::desc_template(16, 1024, tc::SWIZZLE_128B);
constexpr uint64_t DESC_VMN = tc::desc_template(SUB, 1024, tc::SWIZZLE_128B);

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
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Work unit u -> (instance b, KV head g, chunk c) and its key range [k0, k1) (n tiles); an
// empty unit (c past the instance's chunks) has n = 0 and is skipped by every role alike.
struct Unit {
  int b, g, c, n_chunks, L, k0, k1, n;
};
__device__ __forceinline__ Unit unit_at(const VerifyArgs& a, int u) {
  Unit t;
  t.c = u % a.max_chunks;
  t.g = (u / a.max_chunks) % a.Hkv;
  t.b = u / (a.max_chunks * a.Hkv);
  t.L = a.lengths[t.b];
  t.n_chunks = min(a.max_chunks, (t.L + a.chunk - 1) / a.chunk);
  if (t.c >= t.n_chunks) { t.k0 = t.k1 = 0; t.n = 0; return t; }
  t.k0 = (int)(((int64_t)t.L * t.c) / t.n_chunks);
  t.k1 = (int)(((int64_t)t.L * (t.c + 1)) / t.n_chunks);
  t.n = (t.k1 - t.k0 + BN - 1) / BN;
  return t;
}
// Tiles of slot s in a unit of n tiles (tile e belongs to slot e & 1).
__device__ __forceinline__ int slot_tiles(int n, int s) { return (n - s + 1) / 2; }

__global__ void __launch_bounds__(THREADS, 1)
verify_tc_kernel(const __grid_constant__ VerifyArgs a, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQ,
                 kva_dtype q_dtype) {
  constexpr uint32_t IDESC_S = tc::idesc_bf16(BM, BN, 0, 0);
  constexpr uint32_t IDESC_PV = tc::idesc_bf16(BM, D, 0, 1);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + BAR_OFF);
  uint64_t* k_full = bars;                     // [NK] K tile landed
  uint64_t* k_free = k_full + NK;              // [NK] its Q K^T done
  uint64_t* v_full = k_free + NK;              // [NV] V tile landed
  uint64_t* v_free = v_full + NV;              // [NV] its P V done
  uint64_t* s_full = v_free + NV;              // [slot] S in tensor memory
  uint64_t* p_full = s_full + 2;               // [slot] P written by the slot's row-holding warps
  uint64_t* pv_done = p_full + 2;              // [slot] the slot's last P V finished
  uint64_t* o_full = pv_done + 2;              // [slot] the unit's last P V of the slot finished
  uint64_t* o_free = o_full + 2;               // [slot] O read out by slot 0's warps
  uint64_t* q_full = o_free + 2;               // [buffer] the unit's query rows staged
  uint64_t* q_free = q_full + 2;               // [buffer] the unit's last Q K^T done: the rows may be replaced
  uint64_t* ml_ready = q_free + 2;             // slot 1's row max and sum published
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(ml_ready + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(ml_ready + 2);
  static_assert((2 * (NK + NV) + 17) * 8 <= 256, "barrier area");
  const bool tma_q = q_dtype == KVA_BF16;   // bf16 rows come by TMA, fp32 rows are staged by slot 1
  float* ml = reinterpret_cast<float*>(sm + ML_OFF);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.Hq / a.Hkv, R = G * a.k;
  const int nvw = (R + 31) / 32;              // softmax warps per slot that hold group rows
  const int P = gridDim.x, cta = blockIdx.x;
  const int n_units = a.B * a.Hkv * a.max_chunks;

  if (warp == MMA_WARP) tc::tmem_alloc(s_taddr, TMEM_COLS);
  for (int i = tid; i < 4 * SUB / 16; i += THREADS)   // query rows past the group stay zero
    reinterpret_cast<uint4*>(sm + Q_OFF)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();                   // read by the tensor core
  if (tid == 0) {
    for (int i = 0; i < NK; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_free[i], 1); }
    for (int i = 0; i < NV; ++i) { mbar_init(&v_full[i], 1); mbar_init(&v_free[i], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1); mbar_init(&p_full[s], nvw); mbar_init(&pv_done[s], 1);
      mbar_init(&o_full[s], 1); mbar_init(&o_free[s], nvw);
    }
    for (int j = 0; j < 2; ++j) { mbar_init(&q_full[j], tma_q ? 1 : nvw); mbar_init(&q_free[j], 1); }
    mbar_init(ml_ready, nvw);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == TMA_WARP && lane == 0) {
    tc::tma_prefetch_desc(&tmK); tc::tma_prefetch_desc(&tmV);
    if (tma_q) tc::tma_prefetch_desc(&tmQ);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_taddr;
  // registers move from the control warpgroup to the softmax warpgroups (warpgroup-wide; each
  // role's code follows its own setmaxnreg so the compiler budgets it with that count)
  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(REGS_CONTROL));
    griddep_wait();                           // inputs of this launch are complete from here on
    griddep_launch_dependents();
  if (warp == TMA_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      int kn = 0, vn = 0;                     // K and V tiles issued so far (all units)
      int qn = 0;                             // query tiles issued (non-empty units)
      const uint32_t q_bytes = 2u * (uint32_t)R * 128u;
      for (int u = cta; ok && u < n_units; u += P) {
        const Unit t = unit_at(a, u);
        if (t.n > 0 && tma_q) {
          // the unit's rows into buffer qn & 1 once the unit two back has run its last Q K^T:
          // one [64 columns x G heads x k positions] box per half row, rows in (i, head) order
          const int j = qn & 1;
          if (qn >= 2 && !mbar_wait_bounded(&q_free[j], (uint32_t)(((qn - 2) >> 1) & 1))) { ok = false; break; }
          mbar_arrive_expect_tx(&q_full[j], q_bytes);
          for (int c = 0; c < 2; ++c)
            tc::tma_load_4d(sm + Q_OFF + (2 * j + c) * SUB, &tmQ, c * 64, t.g * G, 0, t.b, &q_full[j]);
          ++qn;
        }
        for (int e = 0; e < t.n; ++e) {
          const int key0 = t.k0 + e * BN;
          if (kn >= NK && !mbar_wait_bounded(&k_free[kn % NK], (uint32_t)((kn / NK - 1) & 1))) { ok = false; break; }
          mbar_arrive_expect_tx(&k_full[kn % NK], 2 * SUB);
          for (int c = 0; c < 2; ++c)
            tc::tma_load_4d(sm + K_OFF + ((kn % NK) * 2 + c) * SUB, &tmK, c * 64, key0, t.g, t.b, &k_full[kn % NK]);
          ++kn;
          if (vn >= NV && !mbar_wait_bounded(&v_free[vn % NV], (uint32_t)((vn / NV - 1) & 1))) { ok = false; break; }
          mbar_arrive_expect_tx(&v_full[vn % NV], 2 * SUB);
          for (int c = 0; c < 2; ++c)
            tc::tma_load_4d(sm + V_OFF + ((vn % NV) * 2 + c) * SUB, &tmV, c * 64, key0, t.g, t.b, &v_full[vn % NV]);
          ++vn;
        }
        if (*s_abort) ok = false;
      }
      if (!ok) *s_abort = 1;
      // never leave a copy in flight (the last copies of each ring may not have been waited on)
      for (int e = max(0, kn - NK); e < kn; ++e) mbar_wait_bounded(&k_full[e % NK], (uint32_t)((e / NK) & 1));
      for (int e = max(0, vn - NV); e < vn; ++e) mbar_wait_bounded(&v_full[e % NV], (uint32_t)((e / NV) & 1));
      for (int e = max(0, qn - 2); e < qn; ++e) mbar_wait_bounded(&q_full[e & 1], (uint32_t)((e >> 1) & 1));
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      const uint64_t q_desc0 = tc::desc_at(DESC_KMAJ, smem_u32(sm + Q_OFF));
      const uint64_t k_desc0 = tc::desc_at(DESC_KMAJ, smem_u32(sm + K_OFF));
      const uint64_t v_desc0 = tc::desc_at(DESC_VMN, smem_u32(sm + V_OFF));
      constexpr uint64_t STAGE16 = (uint64_t)(2 * SUB) >> 4;
      int it = 0;                             // tiles consumed so far (all units)
      int ks[2] = {0, 0};                     // tiles of each slot so far
      int nus1 = 0;                           // units in which slot 1 had tiles
      int nu = 0;                             // non-empty units so far
      for (int u = cta; ok && u < n_units; u += P) {
        const Unit t = unit_at(a, u);
        if (t.n == 0) continue;
        const int n = t.n;
        const int qb = nu & 1;                // query buffer of this unit
        const uint64_t q_desc = q_desc0 + (uint64_t)((2 * qb * SUB) >> 4);
        ok = mbar_wait_bounded(&q_full[qb], (uint32_t)((nu >> 1) & 1));
        tc::fence_after_sync();
        auto issue_s = [&](int e) {           // Q K^T of tile e of the unit into slot e & 1
          const int st = (it + e) % NK;
          if (!mbar_wait_bounded(&k_full[st], (uint32_t)(((it + e) / NK) & 1))) return false;
          tc::fence_after_sync();
          const uint64_t kd = k_desc0 + (uint64_t)st * STAGE16;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t off = (uint64_t)((((k >> 2) * SUB) + (k & 3) * 32) >> 4);
            tc::mma_ss(tmem + (e & 1) * BN, q_desc + off, kd + off, IDESC_S, k > 0);
          }
          tc::mma_commit(&s_full[e & 1]);
          tc::mma_commit(&k_free[st]);
          if (e == n - 1) tc::mma_commit(&q_free[qb]);   // the unit's last Q K^T
          return true;
        };
        if (ok) ok = issue_s(0);
        if (ok && n > 1) ok = issue_s(1);
        for (int e = 0; ok && e < n; ++e) {
          const int s = e & 1, j = e >> 1;
          const int sv = (it + e) % NV;
          if (!mbar_wait_bounded(&p_full[s], (uint32_t)((ks[s] + j) & 1))) { ok = false; break; }
          if (!mbar_wait_bounded(&v_full[sv], (uint32_t)(((it + e) / NV) & 1))) { ok = false; break; }
          // the first P V of a slot in a unit overwrites O: the previous unit's O must be read
          if (j == 0 && nu > 0 && !mbar_wait_bounded(&o_free[s], (uint32_t)((nu - 1) & 1))) { ok = false; break; }
          tc::fence_after_sync();
          const uint64_t vd = v_desc0 + (uint64_t)sv * STAGE16;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            tc::mma_ts(tmem + 256 + s * 128, tmem + s * BN + kk * 8, vd + (uint64_t)(kk * 2048 >> 4), IDESC_PV,
                       (j > 0 || kk > 0));
          tc::mma_commit(&pv_done[s]);
          tc::mma_commit(&v_free[sv]);
          if (e + 2 >= n) tc::mma_commit(&o_full[s]);   // the slot's last tile of the unit
          if (e + 2 < n && !issue_s(e + 2)) { ok = false; break; }
        }
        it += n;
        ks[0] += slot_tiles(n, 0);
        ks[1] += slot_tiles(n, 1);
        if (slot_tiles(n, 1) > 0) ++nus1;
        ++nu;
        if (*s_abort) ok = false;
      }
      (void)nus1;
      if (!ok) *s_abort = 1;
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(REGS_SOFTMAX));
    griddep_wait();
    griddep_launch_dependents();
  if ((warp & 3) < nvw) {
    // ------------------------------------------------------------ softmax warps holding rows
    const int s = warp >> 2;                  // slot
    const int quarter = warp & 3;             // TMEM lane quarter of this warp
    const int t = quarter * 32 + lane;        // row of the group = TMEM lane
    const bool row_ok = t < R;
    const int iblk = row_ok ? t / G : 0;      // block position of the row
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_col = s * BN, o_col = 256 + s * 128;
    bool ok = true;
    int it = 0, ks = 0, nus = 0, nus1 = 0, nu = 0;   // tiles, slot tiles, slot units, slot-1 units, units
    int u = cta;
    float x[BN];
    // Slot 1 stages each unit's query rows: the first unit's here, the next one's right after it
    // has published the unit's row statistics (the old rows are free once the unit's last Q K^T
    // has run), so the next unit's first products overlap slot 0's read-out of O.
    // Chunk c (8 values) of row t -> box c / 8, swizzled position (c % 8) ^ (t % 8).
    auto stage_q = [&](const Unit& T, int j) {
      if (row_ok) {
        const int64_t qr = (((int64_t)T.b * a.k + iblk) * a.Hq + T.g * G + t % G) * D;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          uint4 v;
          if (q_dtype == KVA_BF16) {
            v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + qr + c * 8));
          } else {
            const float4 f0 = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.q) + qr + c * 8));
            const float4 f1 = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.q) + qr + c * 8 + 4));
            v = make_uint4(cvt_bf16x2(f0.x, f0.y), cvt_bf16x2(f0.z, f0.w), cvt_bf16x2(f1.x, f1.y), cvt_bf16x2(f1.z, f1.w));
          }
          *reinterpret_cast<uint4*>(sm + Q_OFF + (2 * j + (c >> 3)) * SUB + (t >> 3) * 1024 + (t & 7) * 128 +
                                    (((c & 7) ^ (t & 7)) << 4)) = v;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[j]);
    };
    // the first non-empty unit at or after u (n_units if none)
    auto next_unit = [&](int from) {
      for (; from < n_units; from += P)
        if (unit_at(a, from).n > 0) break;
      return from;
    };
    u = next_unit(u);
    if (s == 1 && !tma_q && u < n_units) stage_q(unit_at(a, u), 0);
    for (; ok && u < n_units; u = next_unit(u + P)) {
      const Unit T = unit_at(a, u);
      const int n = T.n, ns = slot_tiles(n, s);
      const int64_t q_row = row_ok ? (((int64_t)T.b * a.k + iblk) * a.Hq + T.g * G + t % G) * D : 0;
      // visible keys of the row inside the chunk: [k0, lim)
      const int lim = row_ok ? min(T.k1, T.L - a.k + iblk + 1) : T.k0;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < ns; ++j) {
        const int e = 2 * j + s, kk = ks + j;
        const int key0 = T.k0 + e * BN;
        if (!__all_sync(FULL_MASK, mbar_wait_bounded(&s_full[s], (uint32_t)(kk & 1)))) { ok = false; break; }
        tc::fence_after_sync();
        if (key0 + BN > T.k1) {
          // the tile runs past the chunk: zero its V rows from k1 on (both 64-column boxes) before
          // P is published, once the V copy has landed
          const int ve = it + e;
          if (!__all_sync(FULL_MASK, mbar_wait_bounded(&v_full[ve % NV], (uint32_t)((ve / NV) & 1)))) { ok = false; break; }
          const int r0 = T.k1 - key0;
          uint8_t* vs = sm + V_OFF + (ve % NV) * 2 * SUB;
          for (int i = quarter * 32 + lane; i < (BN - r0) * 16; i += nvw * 32) {
            const int r = r0 + i / 16, half = (i >> 3) & 1, ch = i & 7;
            *reinterpret_cast<uint4*>(vs + half * SUB + (r >> 3) * 1024 + (r & 7) * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tc::tmem_ld32(lane_base + s_col, r0);
          tc::tmem_ld32(lane_base + s_col + 32, r1);
          tc::tmem_ld32(lane_base + s_col + 64, r2);
          tc::tmem_ld32(lane_base + s_col + 96, r3);
          tc::tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            x[q] = __uint_as_float(r0[q]); x[32 + q] = __uint_as_float(r1[q]);
            x[64 + q] = __uint_as_float(r2[q]); x[96 + q] = __uint_as_float(r3[q]);
          }
        }
        const int chi = lim - key0;           // visible columns of the tile: [0, chi)
        if (chi < BN) {
#pragma unroll
          for (int q = 0; q < BN; ++q)
            if (q >= chi) x[q] = -INFINITY;
        }
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < BN; q += 8) {
#pragma unroll
          for (int c = 0; c < 4; ++c) mq[c] = fmax3(mq[c], x[q + 2 * c], x[q + 2 * c + 1]);
        }
        const float mr = fmaxf(fmax3(mq[0], mq[1], mq[2]), mq[3]);
        const float m_tile = mr == -INFINITY ? -INFINITY : mr * a.scale_log2;
        const float m_new = fmaxf(m, m_tile);
        const bool first = (m == -INFINITY);  // first visible keys: O holds nothing yet
        const bool grow = !first && m_new > m + RESCALE_LOG2;
        if (first) m = m_new;
        if (__any_sync(FULL_MASK, grow)) {
          // some row's max grew by > 2^8: rescale those rows of O once the previous P V landed
          if (!__all_sync(FULL_MASK, mbar_wait_bounded(&pv_done[s], (uint32_t)((kk - 1) & 1)))) { ok = false; break; }
          tc::fence_after_sync();
          const float alpha = grow ? ex2(m - m_new) : 1.0f;
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            uint32_t rr[16];
            tmem_ld16(lane_base + o_col + c * 16, rr);
            tc::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 16; ++q) rr[q] = __float_as_uint(__uint_as_float(rr[q]) * alpha);
            tmem_st16(lane_base + o_col + c * 16, rr);
          }
          tc::tmem_wait_st();
          if (grow) { l *= alpha; m = m_new; }
        }
        // P = exp2(S * scale - m) as packed bf16 into columns [0, 64) of the slot
        const float mref = (m == -INFINITY) ? 0.f : m;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float p0 = ex2(fmaf(x[32 * c + 2 * q], a.scale_log2, -mref));   // hidden: -inf -> 0
            const float p1 = ex2(fmaf(x[32 * c + 2 * q + 1], a.scale_log2, -mref));
            l += p0 + p1;
            w[q] = cvt_bf16x2(p0, p1);
          }
          tmem_st16(lane_base + s_col + c * 16, w);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[s]);
      }
      if (!ok) break;
      const bool has1 = slot_tiles(n, 1) > 0;
      if (s == 1) {
        // publish the row max and sum (O stays in tensor memory for slot 0) once slot 0 has read
        // the previous unit's, then stage the next unit's query rows
        if (nu > 0 && !__all_sync(FULL_MASK, mbar_wait_bounded(&o_free[1], (uint32_t)((nu - 1) & 1)))) { ok = false; break; }
        ml[t] = row_ok ? m : -INFINITY;
        ml[BM + t] = row_ok ? l : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(ml_ready);
        const int un = tma_q ? n_units : next_unit(u + P);
        if (un < n_units) {
          // the other buffer was last read by the unit before this one
          const int j = (nu + 1) & 1;
          if (nu >= 1 && !__all_sync(FULL_MASK, mbar_wait_bounded(&q_free[j], (uint32_t)(((nu - 1) >> 1) & 1)))) { ok = false; break; }
          stage_q(unit_at(a, un), j);
        }
      } else {
        // combine both slots' O (slot 1 may have had no tile), then the final rows or a partial
        if (!__all_sync(FULL_MASK, mbar_wait_bounded(&o_full[0], (uint32_t)(nus & 1)) &&
                                       mbar_wait_bounded(ml_ready, (uint32_t)(nu & 1)) &&
                                       (!has1 || mbar_wait_bounded(&o_full[1], (uint32_t)(nus1 & 1))))) { ok = false; break; }
        tc::fence_after_sync();
        const float m1 = has1 ? ml[t] : -INFINITY, l1 = has1 ? ml[BM + t] : 0.f;
        const float M = fmaxf(m, m1);
        const float e0 = m == -INFINITY ? 0.f : ex2(m - M), e1 = m1 == -INFINITY ? 0.f : ex2(m1 - M);
        const float Ls = e0 * l + e1 * l1;
        const bool single = T.n_chunks == 1;
        const float sc = single ? (Ls > 0.f ? 1.0f / Ls : NAN) : 1.0f;
        const int64_t pidx = (((int64_t)T.b * a.Hkv + T.g) * a.RT * 16 + t) * a.max_chunks + T.c;
        float* dst = single ? a.out + q_row : a.part_acc + pidx * D;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint32_t o0[16], o1[16];
          tmem_ld16(lane_base + 256 + c * 16, o0);
          if (has1) tmem_ld16(lane_base + 384 + c * 16, o1);
          tc::tmem_wait_ld();
          float y[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) y[q] = e0 * __uint_as_float(o0[q]) + (has1 ? e1 * __uint_as_float(o1[q]) : 0.f);
          if (row_ok) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<float4*>(dst + c * 16 + 4 * q4) =
                  make_float4(y[4 * q4] * sc, y[4 * q4 + 1] * sc, y[4 * q4 + 2] * sc, y[4 * q4 + 3] * sc);
          }
        }
        if (!single && row_ok) { a.part_ml[2 * pidx] = M; a.part_ml[2 * pidx + 1] = Ls; }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) { mbar_arrive(&o_free[0]); mbar_arrive(&o_free[1]); }
        if (!single) {
          // the last unit of (b, g) to finish merges this warp's 32 rows over the chunks
          __threadfence();
          __syncwarp();
          unsigned last = 0;
          unsigned* cnt = a.counters + ((int64_t)T.b * a.Hkv + T.g) * a.RT + quarter;
          if (lane == 0) last = atomicAdd(cnt, 1u) == (unsigned)(T.n_chunks - 1) ? 1u : 0u;
          last = __shfl_sync(FULL_MASK, last, 0);
          if (last) {
            __threadfence();
            if (row_ok) {
              // the chunks' weights first (independent loads), then each 32-column block with all
              // of its loads in flight before its stores
              const float* __restrict__ pml = a.part_ml;
              const float* __restrict__ pacc = a.part_acc;
              float* __restrict__ po = a.out + q_row;
              const int64_t p0 = (((int64_t)T.b * a.Hkv + T.g) * a.RT * 16 + t) * a.max_chunks;
              float Mx = -INFINITY;
              for (int cc = 0; cc < T.n_chunks; ++cc) Mx = fmaxf(Mx, __ldcg(&pml[2 * (p0 + cc)]));
              float den = 0.f;
              for (int cc = 0; cc < T.n_chunks; ++cc) {
                const float mc = __ldcg(&pml[2 * (p0 + cc)]);
                if (mc != -INFINITY) den = fmaf(ex2(mc - Mx), __ldcg(&pml[2 * (p0 + cc) + 1]), den);
              }
              const float inv = den > 0.f ? 1.0f / den : NAN;
#pragma unroll 1
              for (int blk = 0; blk < D / 32; ++blk) {
                float4 acc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int cc = 0; cc < T.n_chunks; ++cc) {
                  const float mc = __ldcg(&pml[2 * (p0 + cc)]);
                  const float w = mc == -INFINITY ? 0.f : ex2(mc - Mx);   // a chunk wholly past the row's limit: 0
                  const float4* src = reinterpret_cast<const float4*>(pacc + (p0 + cc) * D + blk * 32);
#pragma unroll
                  for (int q = 0; q < 8; ++q) {
                    const float4 v = __ldcg(src + q);
                    acc[q].x = fmaf(w, v.x, acc[q].x); acc[q].y = fmaf(w, v.y, acc[q].y);
                    acc[q].z = fmaf(w, v.z, acc[q].z); acc[q].w = fmaf(w, v.w, acc[q].w);
                  }
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  reinterpret_cast<float4*>(po + blk * 32)[q] =
                      make_float4(acc[q].x * inv, acc[q].y * inv, acc[q].z * inv, acc[q].w * inv);
              }
            }
            if (lane == 0) *cnt = 0u;
          }
        }
      }
      it += n;
      ks += ns;
      if (ns > 0) ++nus;
      if (has1) ++nus1;
      ++nu;
      if (*s_abort) { ok = false; break; }
    }
    if (!ok) {
      *s_abort = 1;
      // a wait gave up: this CTA's unfinished rows become NaN (plain stores)
      if (s == 0 && row_ok) {
        for (; u < n_units; u += P) {
          const Unit T = unit_at(a, u);
          if (T.n == 0) continue;
          float* o = a.out + (((int64_t)T.b * a.k + iblk) * a.Hq + T.g * G + t % G) * D;
          for (int d = 0; d < D; ++d) o[d] = NAN;
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

// Cache view for TMA: dims (head_dim, capacity slots, Hkv, B), boxes of [128 slots x 64 dims].
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn_vtc() {
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
cudaError_t make_map_vtc(CUtensorMap* map, const void* base, const VerifyArgs& a) {
  EncodeTiledFn fn = encode_fn_vtc();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)a.capacity, (cuuint64_t)a.Hkv, (cuuint64_t)a.B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)a.capacity * D * 2, (cuuint64_t)a.inst_stride * 2};
  const cuuint32_t box[4] = {64, BN, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// q [B, k, Hq, 128] bf16 as (dims, Hq, k, B); boxes of [64 dims x G heads x k positions].
cudaError_t make_qmap_vtc(CUtensorMap* map, const VerifyArgs& a) {
  EncodeTiledFn fn = encode_fn_vtc();
  if (!fn) return cudaErrorNotSupported;
  const int G = a.Hq / a.Hkv;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)a.Hq, (cuuint64_t)a.k, (cuuint64_t)a.B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)a.Hq * D * 2, (cuuint64_t)a.k * a.Hq * D * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)a.k, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.q), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int vtc_num_sms() {
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

}  // namespace

bool verify_tc_supports(int G, int k) { return G * k <= BM && encode_fn_vtc() != nullptr; }

// Chunk size (a multiple of 128 keys, at most 64 chunks per instance) minimising a simple cost:
// rounds of units over the persistent CTAs times the longest unit, counted in 128-key tiles plus
// the per-unit work (O read-out; partials and their merge when instances are split).
int verify_tc_plan_chunk(const int32_t* lengths_host, int B, int Hkv, int max_len) {
  const long long P = vtc_num_sms();
  const int min_chunk = std::max(BN, (max_len + 63) / 64);
  int best = ((max_len + BN - 1) / BN) * BN;
  double best_cost = 1e300;
  for (int chunk = ((min_chunk + BN - 1) / BN) * BN; chunk < max_len + BN; chunk += BN) {
    long long units = 0;
    int unit_tiles = 0;
    for (int b = 0; b < B; ++b) {
      const int nch = (lengths_host[b] + chunk - 1) / chunk;
      units += nch;
      unit_tiles = std::max(unit_tiles, ((lengths_host[b] + nch - 1) / nch + BN - 1) / BN);
    }
    units *= Hkv;
    // a split instance also writes and merges partials: measured at about twelve tiles' worth
    // per unit (64 instances x 2048 slots: 114 us whole, 202 / 346 / 384 us in 2 / 3 / 4 chunks)
    const bool split = units > (long long)B * Hkv;
    const double cost = (double)((units + P - 1) / P) * (unit_tiles + 3 + (split ? 12 : 0));
    if (cost < best_cost - 1e-9) { best_cost = cost; best = chunk; }
  }
  return best;
}

cudaError_t launch_verify_tc(const VerifyArgs& a, kva_dtype q_dtype, cudaStream_t s) {
  static DeviceOnce configured;
  if (!configured.done()) {
    cudaError_t e = cudaFuncSetAttribute(verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    // the register split assumes the launch holds exactly REGS_LAUNCH per thread
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, verify_tc_kernel)) != cudaSuccess) return e;
    if (fa.numRegs != REGS_LAUNCH) return cudaErrorInvalidDeviceFunction;
    configured.mark();
  }
  CUtensorMap mk, mv;
  cudaError_t e = make_map_vtc(&mk, a.kc, a);
  if (e != cudaSuccess) return e;
  if ((e = make_map_vtc(&mv, a.vc, a)) != cudaSuccess) return e;
  CUtensorMap mq;
  std::memset(&mq, 0, sizeof(mq));            // unused for fp32 queries (staged by threads)
  if (q_dtype == KVA_BF16 && (e = make_qmap_vtc(&mq, a)) != cudaSuccess) return e;
  const long long units = (long long)a.B * a.Hkv * a.max_chunks;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int grid = (int)std::min<long long>(units, vtc_num_sms());
  return launch_pdl(verify_tc_kernel, dim3(grid), dim3(THREADS), (size_t)SMEM, s, a, mk, mv, mq, q_dtype);
}

}  // namespace kva
