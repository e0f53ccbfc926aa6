// Kernel (c), bf16-cache form: split-KV decode with the two per-tile contractions on tensor
// cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).
//
// Work unit = (chunk c, KV head g, instance b): instance b's L_b keys are cut into
// ceil(L_b / chunk) nearly equal chunks (at most max_chunks), one CTA each.  The CTA's four
// warps are independent: warp w takes the 16-key tiles w, w+4, ... of the chunk and streams
// them through a private 3-stage shared-memory ring.  Lane 0 issues the TMA copies (each
// tile = K and V as two [16 keys x 64 dims] boxes with 128-byte swizzle, so ldmatrix reads
// are bank-conflict free) and the warp waits on its own mbarriers.  Per tile:
//   S = q K^T      16 rows (the G query heads of the group, rest zero) x 16 keys, 16 MMAs
//   online softmax per row in registers against a reference max that moves only when a
//   score exceeds it by more than 2^8 (then two xor-shuffles across the row's 4 lanes and an
//   O rescale; after the first tiles this is rare)
//   O += P V       P reused from the S accumulator as the A fragment, 16 MMAs
// About 6 instructions per key and KV head instead of ~40 for CUDA-core dot products, so the
// kernel is limited by HBM, not by issue.  The warps merge (max, sum, O) in shared memory;
// with several chunks the CTA writes a partial and the last CTA of (b, g) merges them.
//
// Method: one query against the valid prefix of the cache window (Youtu-VL-4B ncnn port,
// step 8), GQA by repeat-interleave grouping (Penguin-VL ncnn port, section 3), softmax as
// max/subtract/exp/sum/divide (Youtu-VL-4B ncnn port, implementation difficulty 3), bf16
// storage with fp32 accumulation (HunyuanOCR v1.5 ncnn port, section 3.7).
#include <mutex>

#include "launch.h"
#include "tc.cuh"

namespace kva {

namespace {

constexpr int D = DECODE_HEAD_DIM;
constexpr int WARPS = 4;
constexpr int THREADS = WARPS * 32;
constexpr int KT = 16;                          // keys per warp tile
constexpr int NS = 3;                           // ring stages per warp
constexpr int BOX = KT * 128;                   // one [16 keys x 64 dims] swizzled box, 2 KB
constexpr int STAGE = 4 * BOX;                  // K lo, K hi, V lo, V hi
constexpr int RING = NS * STAGE;                // per warp
constexpr float RESCALE_LOG2 = 8.0f;            // a row's reference max lags its true max by <= 2^8

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
// D = A B + D, A rows g and g+8 (a1 = a3 = 0: only rows < 8 carry query heads)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
// byte offset of 16-byte chunk `ch` of key row `key` inside a 128-byte-swizzled box
__device__ __forceinline__ uint32_t swz(int key, int ch) { return key * 128 + ((ch ^ (key & 7)) << 4); }

// One 128-wide row of the new token (lane owns dims 4*lane .. 4*lane+3): QK-Norm and RoPE in
// the configured order for q/k rows (w != null or rope), untouched for v rows.
__device__ __forceinline__ void step_row(float (&x)[4], const float (&w)[4], bool has_w, bool rotate,
                                         const StepArgs& st, const float* s_cos, const float* s_sin, int lane) {
  auto rms = [&](void) {
    float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
    return 1.0f / sqrtf(ss / (float)D + st.eps);
  };
  if (has_w && !st.after_rope) {
    const float r = rms();
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = x[i] * r * w[i];
  }
  if (rotate && st.rope.kind == KVA_ROPE_INTERLEAVED) {
    // inputs 4 lane .. 4 lane + 3 are the pairs j = 2 lane, 2 lane + 1; their rotated values
    // belong at outputs j and 64 + j, so after rotating, lanes exchange values until lane m
    // holds outputs 4m .. 4m + 3 again (low outputs from lanes 2m, 2m + 1 for m < 16, high
    // outputs from lanes 2(m - 16), 2(m - 16) + 1 otherwise)
    float lo[2], hi[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int j = 2 * lane + t;
      lo[t] = x[2 * t] * s_cos[j] - x[2 * t + 1] * s_sin[j];
      hi[t] = x[2 * t + 1] * s_cos[j] + x[2 * t] * s_sin[j];
    }
    const int src = lane < 16 ? 2 * lane : 2 * (lane - 16);
    const float a0 = __shfl_sync(FULL_MASK, lo[0], src), a1 = __shfl_sync(FULL_MASK, lo[1], src);
    const float b0 = __shfl_sync(FULL_MASK, lo[0], src + 1), b1 = __shfl_sync(FULL_MASK, lo[1], src + 1);
    const float c0 = __shfl_sync(FULL_MASK, hi[0], src), c1 = __shfl_sync(FULL_MASK, hi[1], src);
    const float d0 = __shfl_sync(FULL_MASK, hi[0], src + 1), d1 = __shfl_sync(FULL_MASK, hi[1], src + 1);
    if (lane < 16) { x[0] = a0; x[1] = a1; x[2] = b0; x[3] = b1; }
    else { x[0] = c0; x[1] = c1; x[2] = d0; x[3] = d1; }
  } else if (rotate) {
    // partner of dim d: d +- 64 (lane ^ 16) for 1D / sections, d +- 32 inside a half (lane ^ 8) for 2D
    const bool two_d = st.rope.kind == KVA_ROPE_2D;
    float y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float pv = __shfl_xor_sync(FULL_MASK, x[i], two_d ? 8 : 16);
      const int d = 4 * lane + i;
      const int blk = two_d ? d / 64 : 0, dd = two_d ? d % 64 : d, wh = two_d ? 32 : 64;
      const bool lo = dd < wh;
      const int j = blk * 32 + (lo ? dd : dd - wh);
      y[i] = x[i] * s_cos[j] + (lo ? -pv : pv) * s_sin[j];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = y[i];
  }
  if (has_w && st.after_rope) {
    const float r = rms();
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = x[i] * r * w[i];
  }
}

__device__ __forceinline__ void load4(const void* p, int dt, int64_t i, float (&x)[4]) {
  if (dt == KVA_BF16) {
    const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p) + i);
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
  } else {
    const float4 u = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i);
    x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
  }
}

template <int G, bool FUSED>
__global__ void __launch_bounds__(THREADS, 2)
decode_mma_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, kva_dtype q_dtype,
                  const __grid_constant__ StepArgs st) {
  static_assert(G >= 1 && G <= 8, "query heads per KV head");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* ring = smem + warp * RING;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + WARPS * RING) + warp * NS;
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
    if (warp == 0) { tc::tma_prefetch_desc(&tmK); tc::tma_prefetch_desc(&tmV); }
  }
  // rotary table entry of angle slot tid (fused step): parameter reads with per-thread indices
  // serialise, so they are issued before the wait, overlapping the previous kernel
  float r_ih = 0.f, r_il = 0.f;
  double r_inv = 0.0;
  int r_axis = 0;
  if (FUSED && tid < D / 2) {
    r_ih = st.rope.inv_hi[tid]; r_il = st.rope.inv_lo[tid]; r_inv = st.rope.inv[tid]; r_axis = st.rope.axis[tid];
  }
  // Warm L2 with what the first steps after the wait read: the length, the new token's rows
  // and (chunk 0 starts at key 0 whatever the length) the warps' first K/V tiles.  Prefetches
  // return no data, so they may run before the wait: a write by the kernel before this one
  // still lands in L2, the point of coherence, where the loads after the wait read it.
  if (tid == 0) prefetch_l2(a.lengths + b);
  if constexpr (FUSED) {
    const int eb = st.in_dtype == KVA_BF16 ? 2 : 4;
    const int qlines = G * D * eb / 128, kvlines = D * eb / 128;   // 128-byte lines
    const char* qrows = reinterpret_cast<const char*>(st.q) + ((int64_t)b * a.Hq + g * G) * D * eb;
    const int64_t kvoff = ((int64_t)b * a.Hkv + g) * D * eb;
    if (tid < qlines) prefetch_l2(qrows + tid * 128);
    else if (tid < qlines + kvlines) prefetch_l2(reinterpret_cast<const char*>(st.k) + kvoff + (tid - qlines) * 128);
    else if (tid < qlines + 2 * kvlines)
      prefetch_l2(reinterpret_cast<const char*>(st.v) + kvoff + (tid - qlines - kvlines) * 128);
  }
  // Prefetch depth: each warp's first 2 x NS tiles.  Over the whole Qwen3-shaped job (28 layers,
  // L = 513..768, each step after an lm_head launch) 0 / 1 / 3 / 6 / 8 / 12 / 16 tiles gave
  // 15.72 / 15.55 / 15.39 / 15.29 / 15.29 / 15.65 / 16.02 ms: deeper, and the prefetches
  // compete with the lm_head launch still draining.  Around the optimum, 5 / 6 / 7 tiles gave
  // the step alone (back to back over rotating caches) 13.65 / 13.73 / 13.90 us and the job
  // 15.31 / 15.26 / 15.25 ms.
  if (c == 0 && lane == 0)
    for (int u = 0; u < 2 * NS; ++u) {
      const int ks = (warp + u * WARPS) * KT;
      if (ks >= a.capacity) break;
      tc::tma_prefetch_l2_4d(&tmK, 0, ks, g, b); tc::tma_prefetch_l2_4d(&tmK, 64, ks, g, b);
      tc::tma_prefetch_l2_4d(&tmV, 0, ks, g, b); tc::tma_prefetch_l2_4d(&tmV, 64, ks, g, b);
    }
  griddep_wait();                               // inputs of this launch are complete from here on
  griddep_launch_dependents();
  const int L = a.lengths[b];
  // fused step: the new token's rows (G queries, then k, then v; warp w takes rows w and w + 4)
  // and position are loaded here, so their latency overlaps that of the lengths load
  constexpr int ROWS = FUSED ? (G + 2 + WARPS - 1) / WARPS : 1;
  float xr[ROWS][4], wr[ROWS][4];
  int32_t pj = 0;
  if constexpr (FUSED) {
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      const int rr = warp + i * WARPS;
      wr[i][0] = wr[i][1] = wr[i][2] = wr[i][3] = 1.f;
      if (rr < G) {
        load4(st.q, st.in_dtype, ((int64_t)b * a.Hq + g * G + rr) * D + 4 * lane, xr[i]);
        if (st.q_w) load4(st.q_w + (int64_t)b * st.w_stride, KVA_F32, 4 * lane, wr[i]);
      } else if (rr < G + 2) {
        load4(rr == G ? st.k : st.v, st.in_dtype, ((int64_t)b * a.Hkv + g) * D + 4 * lane, xr[i]);
        if (rr == G && st.k_w) load4(st.k_w + (int64_t)b * st.w_stride, KVA_F32, 4 * lane, wr[i]);
      }
    }
    if (st.rope.kind != KVA_ROPE_NONE && tid < D / 2) pj = st.pos[(int64_t)b * st.pos_stride + r_axis];
  }
  const int n_chunks = min(a.max_chunks, (L + a.chunk - 1) / a.chunk);
  if (c >= n_chunks) return;
  const int k0 = (int)(((int64_t)L * c) / n_chunks);
  const int k1 = (int)(((int64_t)L * (c + 1)) / n_chunks);
  const int n_tiles = (k1 - k0 + KT - 1) / KT;

  const int n_mine = n_tiles > warp ? (n_tiles - 1 - warp) / WARPS + 1 : 0;
  auto issue = [&](int u) {                    // lane 0: tile t = warp + u*WARPS
    const int ks = k0 + (warp + u * WARPS) * KT;
    unsigned char* dst = ring + (u % NS) * STAGE;
    mbar_arrive_expect_tx(&bar[u % NS], STAGE);
    tc::tma_load_4d(dst, &tmK, 0, ks, g, b, &bar[u % NS]);
    tc::tma_load_4d(dst + BOX, &tmK, 64, ks, g, b, &bar[u % NS]);
    tc::tma_load_4d(dst + 2 * BOX, &tmV, 0, ks, g, b, &bar[u % NS]);
    tc::tma_load_4d(dst + 3 * BOX, &tmV, 64, ks, g, b, &bar[u % NS]);
  };
  if (lane == 0)
    for (int u = 0; u < NS && u < n_mine; ++u) issue(u);
  __syncwarp();

  // ---- fused step: transform the new token's rows (q of the G heads; k, v in the last chunk) ----
  __shared__ float s_cos[D / 2], s_sin[D / 2];
  __shared__ __align__(16) uint16_t s_q[G][D], s_kv[2][D];
  const bool last_chunk = (c == n_chunks - 1);
  if constexpr (FUSED) {
    const bool rotate = st.rope.kind != KVA_ROPE_NONE;
    if (rotate && tid < D / 2) rope_cos_sin(pj, r_ih, r_il, r_inv, &s_cos[tid], &s_sin[tid]);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
      const int rr = warp + i * WARPS;
      if (rr >= G + 2 || (rr >= G && !last_chunk)) continue;   // only the last chunk owns the new key
      float (&x)[4] = xr[i];
      const bool has_w = rr < G ? st.q_w != nullptr : (rr == G && st.k_w != nullptr);
      step_row(x, wr[i], has_w, rotate && rr <= G, st, s_cos, s_sin, lane);
      const uint32_t p01 = pack_bf16x2(x[0], x[1]), p23 = pack_bf16x2(x[2], x[3]);
      if (rr < G) {
        *reinterpret_cast<uint2*>(&s_q[rr][4 * lane]) = make_uint2(p01, p23);
        if (st.q_out && c == 0) {
          const int64_t qo = ((int64_t)b * a.Hq + g * G + rr) * D + 4 * lane;
          if (st.q_out_dtype == KVA_BF16) *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(st.q_out) + qo) = make_uint2(p01, p23);
          else *reinterpret_cast<float4*>(reinterpret_cast<float*>(st.q_out) + qo) = make_float4(x[0], x[1], x[2], x[3]);
        }
      } else {
        *reinterpret_cast<uint2*>(&s_kv[rr - G][4 * lane]) = make_uint2(p01, p23);
        // the cache keeps the new row for later steps (slot L-1 of this instance and head)
        unsigned char* dst = reinterpret_cast<unsigned char*>(rr == G ? const_cast<void*>(a.kc) : const_cast<void*>(a.vc)) +
                             ((int64_t)b * a.inst_stride + ((int64_t)g * a.capacity + (L - 1)) * D + 4 * lane) * 2;
        *reinterpret_cast<uint2*>(dst) = make_uint2(p01, p23);
      }
    }
    __syncthreads();
  }

  // ---- query A fragments: row r = lane/4 (< G carries head g*G + r), k pairs 2t, 2t+8 ----
  const int r = lane >> 2, t = lane & 3;
  uint32_t qa0[8], qa2[8];
  if constexpr (FUSED) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qa0[kk] = r < G ? *reinterpret_cast<const uint32_t*>(&s_q[r < G ? r : 0][16 * kk + 2 * t]) : 0u;
      qa2[kk] = r < G ? *reinterpret_cast<const uint32_t*>(&s_q[r < G ? r : 0][16 * kk + 8 + 2 * t]) : 0u;
    }
  } else {
    const bool on = r < G;
    const int64_t qb = ((int64_t)b * a.Hq + g * G + (on ? r : 0)) * D;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t lo = 0, hi = 0;
      if (on) {
        const int d0 = 16 * kk + 2 * t;
        if (q_dtype == KVA_BF16) {
          lo = *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint16_t*>(a.q) + qb + d0);
          hi = *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint16_t*>(a.q) + qb + d0 + 8);
        } else {
          const float* qf = reinterpret_cast<const float*>(a.q) + qb;
          lo = pack_bf16x2(qf[d0], qf[d0 + 1]);
          hi = pack_bf16x2(qf[d0 + 8], qf[d0 + 9]);
        }
      }
      qa0[kk] = lo; qa2[kk] = hi;
    }
  }

  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  // statistics of row r (this lane's query head): m is a reference max, moved only when a score
  // exceeds it by more than 2^8 (so every P <= 256; the quad's shuffles and the O rescale run
  // only then); l is this lane's partial sum, reduced over the quad at the end
  float m = -INFINITY, l = 0.f;
  bool ok = true;

  for (int u = 0; u < n_mine; ++u) {
    if (!__all_sync(FULL_MASK, mbar_wait_bounded(&bar[u % NS], (uint32_t)((u / NS) & 1)))) { ok = false; break; }
    unsigned char* stg = ring + (u % NS) * STAGE;
    const int ks = k0 + (warp + u * WARPS) * KT;
    const int nk = min(KT, k1 - ks);
    if (nk < KT) {                              // keys past the chunk: zero V so 0 * V stays 0
      for (int i = lane; i < (KT - nk) * 16; i += 32) {
        const int key = nk + i / 16, half = (i / 8) & 1, ch = i & 7;
        *reinterpret_cast<uint4*>(stg + (2 + half) * BOX + swz(key, ch)) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    if constexpr (FUSED) {
      // the tile holding slot L-1 gets the freshly computed row (the TMA may have read the
      // cache before this CTA's own global write landed)
      const int row = (L - 1) - ks;
      if (last_chunk && row >= 0 && row < nk) {
        if (lane < 16) {
          const int half = lane >> 3, ch = lane & 7;
          *reinterpret_cast<uint4*>(stg + half * BOX + swz(row, ch)) =
              *reinterpret_cast<const uint4*>(&s_kv[0][half * 64 + ch * 8]);
        } else {
          const int half = (lane - 16) >> 3, ch = lane & 7;
          *reinterpret_cast<uint4*>(stg + (2 + half) * BOX + swz(row, ch)) =
              *reinterpret_cast<const uint4*>(&s_kv[1][half * 64 + ch * 8]);
        }
        __syncwarp();
      }
    }
    const uint32_t sK = smem_u32(stg), sV = sK + 2 * BOX;

    // ---- S = q K^T: n-tile 0 = keys 0..7, n-tile 1 = keys 8..15 ----
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int key = rr + 8 * (mi >> 1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int half = kk >> 2, ch = ((kk & 3) << 1) + (mi & 1);
        uint32_t bf[4];
        ldsm_x4(sK + half * BOX + swz(key, ch), bf);
        mma16816(s0, qa0[kk], qa2[kk], bf[0], bf[1]);
        mma16816(s1, qa0[kk], qa2[kk], bf[2], bf[3]);
      }
    }
    // ---- online softmax of row r over this tile's keys 2t, 2t+1, 8+2t, 9+2t ----
    float x[4] = {s0[0] * a.scale_log2, s0[1] * a.scale_log2, s1[0] * a.scale_log2, s1[1] * a.scale_log2};
    {
      const int kx[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
#pragma unroll
      for (int i = 0; i < 4; ++i) if (kx[i] >= nk) x[i] = -INFINITY;
    }
    float mt = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    if (__any_sync(FULL_MASK, mt > m + RESCALE_LOG2)) {
      mt = fmaxf(mt, __shfl_xor_sync(FULL_MASK, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(FULL_MASK, mt, 2));
      // quad-uniform (every tile has a valid key, so m is finite after the first tile, where
      // m = -inf gives alpha = 0 over an empty O)
      const bool grow = mt > m + RESCALE_LOG2;
      const float alpha = grow ? ex2(m - mt) : 1.f;
      if (grow) m = mt;
      l *= alpha;
#pragma unroll
      for (int n = 0; n < 16; ++n) { o[n][0] *= alpha; o[n][1] *= alpha; }
    }
    float p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = ex2(x[i] - m);    // hidden keys hold -inf: 0
    const uint32_t pa0 = pack_bf16x2(p[0], p[1]);     // keys 2t, 2t+1
    const uint32_t pa2 = pack_bf16x2(p[2], p[3]);     // keys 8+2t, 9+2t
    l += (bf16_lo(pa0) + bf16_hi(pa0)) + (bf16_lo(pa2) + bf16_hi(pa2));   // the weights P V uses

    // ---- O += P V: 16 n-tiles of 8 dims; ldmatrix.trans gives V as the B fragment ----
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int key = rr + 8 * (mi & 1);
#pragma unroll
      for (int nd = 0; nd < 8; ++nd) {
        const int half = nd >> 2, ch = ((nd & 3) << 1) + (mi >> 1);
        uint32_t bf[4];
        ldsm_x4_t(sV + half * BOX + swz(key, ch), bf);
        mma16816(o[2 * nd], pa0, pa2, bf[0], bf[1]);
        mma16816(o[2 * nd + 1], pa0, pa2, bf[2], bf[3]);
      }
    }
    __syncwarp();                               // all lanes are done with this stage
    if (lane == 0 && u + NS < n_mine) {
      fence_proxy_async_smem();                 // order this stage's generic accesses before the refill
      issue(u + NS);
    }
  }
  l += __shfl_xor_sync(FULL_MASK, l, 1);
  l += __shfl_xor_sync(FULL_MASK, l, 2);

  // ---- merge the warps (rows r < G live in lanes 4r..4r+3) ----
  __syncthreads();                              // rings drained: reuse them for the merge
  float* sm_m = reinterpret_cast<float*>(smem);           // [WARPS][G]
  float* sm_l = sm_m + WARPS * G;                         // [WARPS][G]
  float* sm_o = sm_l + WARPS * G;                         // [WARPS][G][D]
  if (r < G) {
    if (t == 0) { sm_m[warp * G + r] = ok ? m : NAN; sm_l[warp * G + r] = ok ? l : NAN; }
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      sm_o[(warp * G + r) * D + 8 * n + 2 * t] = o[n][0];
      sm_o[(warp * G + r) * D + 8 * n + 2 * t + 1] = o[n][1];
    }
  }
  __syncthreads();
  __shared__ float s_M[G], s_L[G];
  if (tid < G) {
    float M = -INFINITY;
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, sm_m[w * G + tid]);
    float Ls = 0.f;
    for (int w = 0; w < WARPS; ++w) {
      const float mw = sm_m[w * G + tid];
      Ls += (mw == -INFINITY) ? 0.f : exp2f(mw - M) * sm_l[w * G + tid];
    }
    s_M[tid] = M; s_L[tid] = Ls;
  }
  __syncthreads();
  const bool single = (n_chunks == 1);
  for (int idx = tid; idx < G * D; idx += THREADS) {
    const int hh = idx / D, d = idx % D;
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const float mw = sm_m[w * G + hh];
      if (mw != -INFINITY) tot += exp2f(mw - s_M[hh]) * sm_o[(w * G + hh) * D + d];
    }
    const int h = g * G + hh;
    if (single) {
      a.out[((int64_t)b * a.Hq + h) * D + d] = tot / s_L[hh];
    } else {
      const int64_t pidx = ((int64_t)b * a.Hq + h) * a.max_chunks + c;
      a.part_acc[pidx * D + d] = tot;
      if (d == 0) { a.part_ml[2 * pidx] = s_M[hh]; a.part_ml[2 * pidx + 1] = s_L[hh]; }
    }
  }
  if (single) return;

  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) s_last = (atomicAdd(&a.counters[b * a.Hkv + g], 1u) == (unsigned)(n_chunks - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int idx = tid; idx < G * D; idx += THREADS) {
    const int hh = idx / D, d = idx % D;
    const int64_t p0 = ((int64_t)b * a.Hq + g * G + hh) * a.max_chunks;
    float M = -INFINITY;
    for (int cc = 0; cc < n_chunks; ++cc) M = fmaxf(M, __ldcg(&a.part_ml[2 * (p0 + cc)]));
    float num = 0.f, den = 0.f;
    for (int cc = 0; cc < n_chunks; ++cc) {
      const float w = exp2f(__ldcg(&a.part_ml[2 * (p0 + cc)]) - M);
      num = fmaf(w, __ldcg(&a.part_acc[(p0 + cc) * D + d]), num);
      den = fmaf(w, __ldcg(&a.part_ml[2 * (p0 + cc) + 1]), den);
    }
    a.out[((int64_t)b * a.Hq + g * G + hh) * D + d] = num / den;
  }
  if (tid == 0) a.counters[b * a.Hkv + g] = 0u;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn_dec() {
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

// Whole cache as (head_dim, slot, kv head, instance); boxes of [16 slots x 64 dims].  A decode
// loop passes the same caches every step, so the last few maps built on this host thread are
// reused when every input of the encoding matches (encoding costs about a microsecond).
struct MapKey {
  const void* base;
  int capacity, Hkv, B;
  int64_t inst_stride;
  bool operator==(const MapKey& o) const {
    return base == o.base && capacity == o.capacity && Hkv == o.Hkv && B == o.B && inst_stride == o.inst_stride;
  }
};
cudaError_t encode_map(CUtensorMap* map, const void* base, const DecodeArgs& a);
cudaError_t make_map(CUtensorMap* map, const void* base, const DecodeArgs& a) {
  constexpr int SLOTS = 4;
  thread_local MapKey keys[SLOTS] = {};
  thread_local CUtensorMap maps[SLOTS];
  thread_local int next = 0;
  const MapKey key{base, a.capacity, a.Hkv, a.B, a.inst_stride};
  for (int i = 0; i < SLOTS; ++i)
    if (keys[i].base != nullptr && keys[i] == key) {
      *map = maps[i];
      return cudaSuccess;
    }
  const cudaError_t e = encode_map(map, base, a);
  if (e == cudaSuccess) {
    keys[next] = key;
    maps[next] = *map;
    next = (next + 1) % SLOTS;
  }
  return e;
}
cudaError_t encode_map(CUtensorMap* map, const void* base, const DecodeArgs& a) {
  EncodeTiledFn fn = encode_fn_dec();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)a.capacity, (cuuint64_t)a.Hkv, (cuuint64_t)a.B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)a.capacity * D * 2, (cuuint64_t)a.inst_stride * 2};
  const cuuint32_t box[4] = {64, KT, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int G, bool FUSED>
cudaError_t launch_g(const DecodeArgs& a, const StepArgs& st, kva_dtype q_dtype, cudaStream_t s) {
  const size_t smem = (size_t)WARPS * RING + WARPS * NS * 8 + 1024;
  static DeviceOnce configured;
  if (!configured.done()) {
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<G, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured.mark();
  }
  CUtensorMap mk, mv;
  cudaError_t e = make_map(&mk, a.kc, a);
  if (e != cudaSuccess) return e;
  if ((e = make_map(&mv, a.vc, a)) != cudaSuccess) return e;
  dim3 grid(a.max_chunks, a.Hkv, a.B);
  return launch_pdl(decode_mma_kernel<G, FUSED>, grid, dim3(THREADS), smem, s, a, mk, mv, q_dtype, st);
}

}  // namespace

bool decode_mma_supported() { return encode_fn_dec() != nullptr; }

cudaError_t decode_cache_map(CUtensorMap* map, const void* base, int capacity, int Hkv, int B, int64_t inst_stride) {
  DecodeArgs a{};
  a.capacity = capacity; a.Hkv = Hkv; a.B = B; a.inst_stride = inst_stride;
  return make_map(map, base, a);
}

cudaError_t launch_decode_mma(const DecodeArgs& a, kva_dtype q_dtype, cudaStream_t s) {
  const StepArgs none{};
  switch (a.Hq / a.Hkv) {
    case 1: return launch_g<1, false>(a, none, q_dtype, s);
    case 2: return launch_g<2, false>(a, none, q_dtype, s);
    case 4: return launch_g<4, false>(a, none, q_dtype, s);
    default: return cudaErrorInvalidValue;
  }
}

bool decode_step_supported(int G) { return G == 1 || G == 2 || G == 4; }

cudaError_t launch_decode_step(const DecodeArgs& a, const StepArgs& st, cudaStream_t s) {
  switch (a.Hq / a.Hkv) {
    case 1: return launch_g<1, true>(a, st, KVA_BF16, s);
    case 2: return launch_g<2, true>(a, st, KVA_BF16, s);
    case 4: return launch_g<4, true>(a, st, KVA_BF16, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kva
