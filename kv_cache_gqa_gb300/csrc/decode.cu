// Kernel (c), CUDA-core form (fp32 caches; bf16 caches use decode_mma.cu when TMA is
// available): split-KV single-token decode attention over the fixed-window cache.
//
// Work unit = (chunk c, KV head g, instance b).  A CTA streams its chunk of the K and V
// rows of head g through a 3-stage shared-memory ring filled by 1-D bulk async copies
// (one elected thread issues them; completion is an mbarrier transaction count), and
// serves all G = Hq/Hkv query heads of the group from each staged tile, so each cache
// byte is read from HBM once per step.  Scores stay in fp32 (log2 domain) with an
// online softmax across stages; the partial (max, sum, acc) of every chunk goes to the
// workspace and the last CTA to finish a (b, g) merges them - no CTA ever waits on
// another.  The K rows may be wider than the V rows: an asymmetric cache with Dk = 192,
// Dv = 128 (an MLA layer expanded to per-head K and V, Youtu-VL-4B ncnn port, section 6)
// takes the same kernel with wider K tiles.
//
// Method: one query against the valid prefix of the cache window (Youtu-VL-4B ncnn port,
// step 8: each new token attends to the whole cache behind the mask), GQA by
// repeat-interleave grouping (Penguin-VL ncnn port, section 3), softmax as
// max/subtract/exp/sum/divide (Youtu-VL-4B ncnn port, implementation difficulty 3),
// bf16 cache with fp32 accumulation (HunyuanOCR v1.5 ncnn port, section 3.7).
#include <cfloat>

#include "common.cuh"
#include "launch.h"

namespace kva {

namespace {

constexpr int D = DECODE_HEAD_DIM;    // V row width (and the output's)
constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int NSTAGE = 3;

template <typename CacheT> struct DecodeTile;
template <> struct DecodeTile<bf16_t> { static constexpr int KT = 64; };
template <> struct DecodeTile<float> { static constexpr int KT = 32; };

__device__ __forceinline__ float load_q(const void* q, kva_dtype dt, int64_t i) {
  if (dt == KVA_BF16)
    return __uint_as_float(((uint32_t) reinterpret_cast<const uint16_t*>(q)[i]) << 16);
  return reinterpret_cast<const float*>(q)[i];
}

// Convert one 16-byte chunk of cache row elements to floats.
template <typename CacheT, int N> __device__ __forceinline__ void chunk_to_f32(uint4 w, float (&x)[N]);
template <> __device__ __forceinline__ void chunk_to_f32<bf16_t, 8>(uint4 w, float (&x)[8]) {
  x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
  x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
}
template <> __device__ __forceinline__ void chunk_to_f32<float, 4>(uint4 w, float (&x)[4]) {
  x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
  x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
}

// One row of the new token (q of one head, k or v) held 8 elements per lane at dims
// [8 lane, 8 lane + 8): QK-Norm and RoPE in the configured order for q/k rows, none for v.  The
// rotation covers dims [ro, ro + rw) in rotate-half, 2D-halves or de-interleaved form; `mirror`
// (the row's shared buffer) lets every element read its partner wherever it sits.
__device__ __forceinline__ void step_row_general(float (&x)[8], int e0, bool on, int width, const float* w,
                                                 bool qk, const StepArgs& st, const float* cs, const float* sn,
                                                 float* mirror) {
  if (!qk) return;
  auto apply_norm = [&]() {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss += x[i] * x[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL_MASK, ss, o);
    if (w != nullptr && on) {
      float wv[8];
      load8(w + e0, wv);
      const float rinv = 1.0f / sqrtf(ss / (float)width + st.eps);
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = x[i] * rinv * wv[i];
    }
  };
  if (!st.after_rope) apply_norm();
  const int kind_r = st.rope.kind;
  if (kind_r != KVA_ROPE_NONE) {
    const int ro = st.rot_offset, rw = st.rot_dim, half = rw / 2, quarter = rw / 4;
    if (on) {
#pragma unroll
      for (int i = 0; i < 8; ++i) mirror[e0 + i] = x[i];
    }
    __syncwarp();
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int dd = e0 + i - ro;
      y[i] = x[i];
      if (on && dd >= 0 && dd < rw) {
        const float* xr = mirror + ro;
        if (kind_r == KVA_ROPE_INTERLEAVED) {
          const int j = dd < half ? dd : dd - half;
          const float ev = xr[2 * j], od = xr[2 * j + 1];
          y[i] = dd < half ? ev * cs[j] - od * sn[j] : od * cs[j] + ev * sn[j];
        } else if (kind_r == KVA_ROPE_2D) {
          const int bb = dd / half, e2 = dd - bb * half;
          const bool lo = e2 < quarter;
          const int j = bb * quarter + (lo ? e2 : e2 - quarter);
          const float pv = xr[lo ? dd + quarter : dd - quarter];
          y[i] = x[i] * cs[j] + (lo ? -pv : pv) * sn[j];
        } else {
          const bool lo = dd < half;
          const int j = lo ? dd : dd - half;
          const float pv = xr[lo ? dd + half : dd - half];
          y[i] = x[i] * cs[j] + (lo ? -pv : pv) * sn[j];
        }
      }
    }
    __syncwarp();                               // mirror reads done before it is rewritten
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = y[i];
  }
  if (st.after_rope) apply_norm();
}

__device__ __forceinline__ void load8_dt(const void* p, int dt, int64_t i, float (&x)[8]) {
  if (dt == KVA_BF16) load8(reinterpret_cast<const bf16_t*>(p) + i, x);
  else load8(reinterpret_cast<const float*>(p) + i, x);
}

__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ void store1(bf16_t* p, float v) { p->bits = (uint16_t)f32_to_bf16_rne(v); }

template <typename CacheT, int G, int DK, bool FUSED>
__global__ void __launch_bounds__(THREADS, DK > D ? 1 : 2)   // wide K tiles: one CTA per SM by smem
decode_kernel(const __grid_constant__ DecodeArgs a, kva_dtype q_dtype, const __grid_constant__ StepArgs st) {
  constexpr int ES = ElemSize<CacheT>::value;
  constexpr int KT = DecodeTile<CacheT>::KT;   // keys per stage
  constexpr int ROWK = DK * ES;                // bytes per K row
  constexpr int ROWB = D * ES;                 // bytes per V row
  constexpr int TILEK = KT * ROWK;             // bytes per K stage
  constexpr int TILEB = KT * ROWB;             // bytes per V stage
  constexpr int CH = 16 / ES;                  // elements per 16-byte chunk
  constexpr int QPL = DK / 8;                  // query dims per lane in the QK phase
  constexpr int NCH = QPL / CH;                // 16-byte chunks per lane in the QK phase
  static_assert(DK % (8 * CH) == 0, "K rows split into whole 16-byte chunks over 8 lanes");
  constexpr int KPW = KT / WARPS;              // keys per warp per stage
  constexpr int QK_PASSES = KPW / 4;           // 4 keys per warp pass (8 lanes per key)
  constexpr int SPL = KT / 32;                 // scores per lane in the softmax phase

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sK = smem;
  unsigned char* sV = smem + NSTAGE * TILEK;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSTAGE * (TILEK + TILEB));  // [NSTAGE]
  float* sS = reinterpret_cast<float*>(full + NSTAGE);               // [G][KT]
  float* sP = sS + G * KT;                                           // [KT][G]
  float* sAlpha = sP + KT * G;                                       // [G]
  float* sML = sAlpha + G;                                           // [G][2]
  __shared__ int s_flag;

  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned char* Kg = reinterpret_cast<const unsigned char*>(a.kc) +
      ((int64_t)b * a.inst_stride + (int64_t)g * a.capacity * DK) * ES;
  const unsigned char* Vg = reinterpret_cast<const unsigned char*>(a.vc) +
      ((int64_t)b * a.inst_stride_v + (int64_t)g * a.capacity * D) * ES;
  const int k0 = c * a.chunk;
  // Warm L2 with the length and the chunk's first stages while the kernel before this one
  // drains (prefetches return no data, so they may run before the wait: a write by that kernel
  // still lands in L2, where the copies after the wait read it)
  if (tid == 0) {
    prefetch_l2(a.lengths + b);
    if (k0 + NSTAGE * KT <= a.capacity) {
      bulk_prefetch_l2(Kg + (int64_t)k0 * ROWK, (uint32_t)(NSTAGE * TILEK));
      bulk_prefetch_l2(Vg + (int64_t)k0 * ROWB, (uint32_t)(NSTAGE * TILEB));
    }
  }
  griddep_wait();                               // inputs of this launch are complete from here on
  griddep_launch_dependents();
  const int L = a.lengths[b];
  const int n_chunks = (L + a.chunk - 1) / a.chunk;
  if (c >= n_chunks) return;
  const int k1 = min(L, k0 + a.chunk);
  const int n_sub = (k1 - k0 + KT - 1) / KT;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    s_flag = 0;
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < NSTAGE && s < n_sub; ++s) {
      const int ks = k0 + s * KT;
      const int nr = min(KT, k1 - ks);
      mbar_arrive_expect_tx(&full[s], (uint32_t)(nr * (ROWK + ROWB)));
      bulk_g2s(sK + s * TILEK, Kg + (int64_t)ks * ROWK, (uint32_t)(nr * ROWK), &full[s]);
      bulk_g2s(sV + s * TILEB, Vg + (int64_t)ks * ROWB, (uint32_t)(nr * ROWB), &full[s]);
    }
  }

  // ---- fused step: the new token's rows, transformed while the first copies are in flight.
  // Warps 0..G-1 take the group's query rows; in the last chunk warps G and G+1 take k and v,
  // write them into slot L-1 of the cache and keep them for the stage that holds that slot
  // (patched in shared memory: the copy may have read the slot before the write landed).
  constexpr int NROW = FUSED ? G + 2 : 1;
  constexpr int RW = FUSED ? 256 : 8;
  __shared__ float f_cos[FUSED ? MAX_ROPE_FREQ : 1], f_sin[FUSED ? MAX_ROPE_FREQ : 1];
  __shared__ __align__(16) float f_rows[NROW][RW];
  const bool last_chunk = (c == n_chunks - 1);
  if constexpr (FUSED) {
    if (st.rope.kind != KVA_ROPE_NONE)
      for (int j = tid; j < st.rot_dim / 2; j += THREADS) {
        const int32_t p = st.pos[(int64_t)b * st.pos_stride + st.rope.axis[j]];
        rope_cos_sin(p, st.rope.inv_hi[j], st.rope.inv_lo[j], st.rope.inv[j], &f_cos[j], &f_sin[j]);
      }
    __syncthreads();
    if (warp < G || (last_chunk && warp < G + 2)) {
      const int kind = warp < G ? 0 : (warp == G ? 1 : 2);   // q, k, v
      const int width = kind == 2 ? D : DK;
      const int e0 = lane * 8;
      const bool on = e0 < width;
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      const int64_t row = kind == 0 ? ((int64_t)b * a.Hq + g * G + warp) * DK
                                    : ((int64_t)b * a.Hkv + g) * (kind == 1 ? DK : D);
      if (on) load8_dt(kind == 0 ? st.q : (kind == 1 ? st.k : st.v), st.in_dtype, row + e0, x);
      const float* w = kind == 0 ? (st.q_w ? st.q_w + (int64_t)b * st.w_stride : nullptr)
                                 : (st.k_w ? st.k_w + (int64_t)b * st.w_stride : nullptr);
      step_row_general(x, e0, on, width, w, kind <= 1, st, f_cos, f_sin, f_rows[warp]);
      if (on) {
#pragma unroll
        for (int i = 0; i < 8; ++i) f_rows[warp][e0 + i] = x[i];
        if (kind == 0 && st.q_out && c == 0) {
          if (st.q_out_dtype == KVA_BF16) store8(reinterpret_cast<bf16_t*>(st.q_out) + row + e0, x);
          else store8(reinterpret_cast<float*>(st.q_out) + row + e0, x);
        }
        if (kind >= 1 && L - 1 < a.capacity) {
          CacheT* dst = kind == 1 ? reinterpret_cast<CacheT*>(const_cast<void*>(a.kc)) +
                                        (int64_t)b * a.inst_stride + ((int64_t)g * a.capacity + (L - 1)) * DK
                                  : reinterpret_cast<CacheT*>(const_cast<void*>(a.vc)) +
                                        (int64_t)b * a.inst_stride_v + ((int64_t)g * a.capacity + (L - 1)) * D;
          store8(dst + e0, x);
        }
      }
    }
    __syncthreads();
  }

  // Query registers for the QK phase: lane owns DK/8 dims, NCH chunks of CH elements at
  // element offsets CH*(lane&7) + 8*CH*i.  Pre-scaled so dots are log2-domain logits.
  const int l8 = lane & 7;
  float qv[G][QPL];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    const int64_t qbase = ((int64_t)b * a.Hq + g * G + hh) * DK;
#pragma unroll
    for (int i = 0; i < NCH; ++i)
#pragma unroll
      for (int e = 0; e < CH; ++e)
        qv[hh][i * CH + e] = (FUSED ? f_rows[FUSED ? hh : 0][(CH * l8 + 8 * CH * i + e) % RW]
                                    : load_q(a.q, q_dtype, qbase + CH * l8 + 8 * CH * i + e)) * a.scale_log2;
  }

  float acc[G][4];
#pragma unroll
  for (int hh = 0; hh < G; ++hh)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[hh][e] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;   // meaningful in warp hh < G only
  bool timed_out = false;

  for (int it = 0; it < n_sub; ++it) {
    const int stage = it % NSTAGE;
    const uint32_t parity = (uint32_t)((it / NSTAGE) & 1);
    if (!mbar_wait_bounded(&full[stage], parity)) s_flag = 1;
    __syncthreads();
    if (s_flag) { timed_out = true; break; }
    const int nk = min(KT, k1 - (k0 + it * KT));
    if constexpr (FUSED) {
      const int prow = (L - 1) - (k0 + it * KT);   // the new token's slot in this stage
      if (last_chunk && prow >= 0 && prow < nk) {
        CacheT* pk = reinterpret_cast<CacheT*>(sK + stage * TILEK + prow * ROWK);
        CacheT* pv = reinterpret_cast<CacheT*>(sV + stage * TILEB + prow * ROWB);
        for (int e = tid; e < DK; e += THREADS) store1(pk + e, f_rows[FUSED ? G : 0][e % RW]);
        for (int e = tid; e < D; e += THREADS) store1(pv + e, f_rows[FUSED ? G + 1 : 0][e % RW]);
        __syncthreads();
      }
    }
    const unsigned char* tK = sK + stage * TILEK;
    const unsigned char* tV = sV + stage * TILEB;

    // ---- S = q K^T (8 lanes per key, 4 keys per warp pass) ----
#pragma unroll
    for (int pass = 0; pass < QK_PASSES; ++pass) {
      const int j = warp * KPW + pass * 4 + (lane >> 3);
      float part[G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) part[hh] = 0.f;
      if (j < nk) {
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
          const uint4 w = *reinterpret_cast<const uint4*>(tK + j * ROWK + 16 * l8 + 128 * i);
          float x[CH];
          chunk_to_f32<CacheT, CH>(w, x);
#pragma unroll
          for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int e = 0; e < CH; ++e) part[hh] = fmaf(qv[hh][i * CH + e], x[e], part[hh]);
        }
      }
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float v = part[hh];
        v += __shfl_xor_sync(FULL_MASK, v, 1);
        v += __shfl_xor_sync(FULL_MASK, v, 2);
        v += __shfl_xor_sync(FULL_MASK, v, 4);
        if (l8 == 0) sS[hh * KT + j] = (j < nk) ? v : -INFINITY;
      }
    }
    __syncthreads();

    // ---- online softmax statistics: warp hh owns query head hh ----
    if (warp < G) {
      float s[SPL];
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < SPL; ++i) { s[i] = sS[warp * KT + lane + 32 * i]; mx = fmaxf(mx, s[i]); }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, o));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = exp2f(m_run - m_new);   // 0 on the first stage (m_run = -inf)
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < SPL; ++i) {
        const float p = exp2f(s[i] - m_new);      // 0 for masked keys
        sP[(lane + 32 * i) * G + warp] = p;
        sum += p;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL_MASK, sum, o);
      l_run = l_run * alpha + sum;
      m_run = m_new;
      if (lane == 0) sAlpha[warp] = alpha;
    }
    __syncthreads();

    // ---- acc = acc * alpha + P V (lane owns 4 dims; warp owns KPW keys) ----
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float al = sAlpha[hh];
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[hh][e] *= al;
    }
    const int jend = min(nk, (warp + 1) * KPW);
    for (int j = warp * KPW; j < jend; ++j) {
      float x[4];
      if constexpr (ES == 2) {
        const uint2 w = *reinterpret_cast<const uint2*>(tV + j * ROWB + 8 * lane);
        x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
      } else {
        const float4 w = *reinterpret_cast<const float4*>(tV + j * ROWB + 16 * lane);
        x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
      }
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float p = sP[j * G + hh];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[hh][e] = fmaf(p, x[e], acc[hh][e]);
      }
    }
    __syncthreads();   // stage consumed by every warp

    if (tid == 0 && it + NSTAGE < n_sub) {
      const int ks = k0 + (it + NSTAGE) * KT;
      const int nr = min(KT, k1 - ks);
      mbar_arrive_expect_tx(&full[stage], (uint32_t)(nr * (ROWK + ROWB)));
      bulk_g2s(sK + stage * TILEK, Kg + (int64_t)ks * ROWK, (uint32_t)(nr * ROWK), &full[stage]);
      bulk_g2s(sV + stage * TILEB, Vg + (int64_t)ks * ROWB, (uint32_t)(nr * ROWB), &full[stage]);
    }
  }

  // ---- reduce the warps' partial accumulators (stage buffers are free now) ----
  if (warp < G && lane == 0) {
    sML[2 * warp] = timed_out ? NAN : m_run;
    sML[2 * warp + 1] = timed_out ? NAN : l_run;
  }
  float* red = reinterpret_cast<float*>(smem);   // [WARPS][G][D]
#pragma unroll
  for (int hh = 0; hh < G; ++hh)
#pragma unroll
    for (int e = 0; e < 4; ++e) red[(warp * G + hh) * D + 4 * lane + e] = acc[hh][e];
  __syncthreads();

  // Each (head hh, dim d) of the group is owned by one thread per iteration.
  if (n_chunks == 1) {
    for (int idx = tid; idx < G * D; idx += THREADS) {
      const int hh = idx / D, d = idx % D;
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) tot += red[(w * G + hh) * D + d];
      a.out[((int64_t)b * a.Hq + g * G + hh) * D + d] = tot / sML[2 * hh + 1];
    }
    return;
  }

  for (int idx = tid; idx < G * D; idx += THREADS) {
    const int hh = idx / D, d = idx % D;
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) tot += red[(w * G + hh) * D + d];
    const int64_t pidx = ((int64_t)b * a.Hq + g * G + hh) * a.max_chunks + c;
    a.part_acc[pidx * D + d] = tot;
    if (d == 0) { a.part_ml[2 * pidx] = sML[2 * hh]; a.part_ml[2 * pidx + 1] = sML[2 * hh + 1]; }
  }
  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) {
    const unsigned ticket = atomicAdd(&a.counters[b * a.Hkv + g], 1u);
    s_last = (ticket == (unsigned)(n_chunks - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last CTA of (b, g): merge the chunk partials ----
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
  if (tid == 0) a.counters[b * a.Hkv + g] = 0u;   // ready for the next call
}

template <typename CacheT, int G, int DK>
size_t decode_smem_bytes() {
  constexpr int ES = ElemSize<CacheT>::value;
  constexpr int KT = DecodeTile<CacheT>::KT;
  return (size_t)NSTAGE * KT * (DK + D) * ES + sizeof(uint64_t) * NSTAGE +
         sizeof(float) * (2 * G * KT + 3 * G) + 16;
}

template <typename CacheT, int G, int DK, bool FUSED>
cudaError_t launch_g(const DecodeArgs& a, kva_dtype q_dtype, const StepArgs& st, cudaStream_t s) {
  const size_t smem = decode_smem_bytes<CacheT, G, DK>();
  static DeviceOnce configured;
  if (!configured.done()) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<CacheT, G, DK, FUSED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured.mark();
  }
  dim3 grid(a.max_chunks, a.Hkv, a.B);
  return launch_pdl(decode_kernel<CacheT, G, DK, FUSED>, grid, dim3(THREADS), smem, s, a, q_dtype, st);
}

template <typename CacheT, int DK, bool FUSED = false>
cudaError_t launch_t(const DecodeArgs& a, kva_dtype q_dtype, cudaStream_t s, const StepArgs& st = StepArgs{}) {
  switch (a.Hq / a.Hkv) {
    case 1: return launch_g<CacheT, 1, DK, FUSED>(a, q_dtype, st, s);
    case 2: return launch_g<CacheT, 2, DK, FUSED>(a, q_dtype, st, s);
    case 4: return launch_g<CacheT, 4, DK, FUSED>(a, q_dtype, st, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int decode_subtile(kva_dtype cache_dtype) {
  return cache_dtype == KVA_BF16 ? DecodeTile<bf16_t>::KT : DecodeTile<float>::KT;
}

int decode_num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

cudaError_t launch_decode_mma(const DecodeArgs& a, kva_dtype q_dtype, cudaStream_t s);

// bf16 caches: tensor-core tiles (decode_mma.cu); fp32 caches: the CUDA-core kernel above.
cudaError_t launch_decode(const DecodeArgs& a, kva_dtype q_dtype, kva_dtype cache_dtype,
                          cudaStream_t s) {
  if (cache_dtype == KVA_BF16 && decode_mma_supported()) return launch_decode_mma(a, q_dtype, s);
  if (cache_dtype == KVA_BF16) return launch_t<bf16_t, D>(a, q_dtype, s);
  return launch_t<float, D>(a, q_dtype, s);
}

bool decode_asym_supported(int Dk, int Dv) { return Dk == 192 && Dv == D; }

cudaError_t launch_decode_asym(const DecodeArgs& a, int Dk, int Dv, kva_dtype q_dtype, kva_dtype cache_dtype,
                               cudaStream_t s) {
  if (!decode_asym_supported(Dk, Dv)) return cudaErrorInvalidValue;
  if (cache_dtype == KVA_BF16) return launch_t<bf16_t, 192>(a, q_dtype, s);
  return launch_t<float, 192>(a, q_dtype, s);
}

bool decode_step_simt_supported(int Dk, int Dv, int G) {
  return (G == 1 || G == 2 || G == 4) && ((Dk == D && Dv == D) || decode_asym_supported(Dk, Dv));
}

// The fused decode step on the CUDA-core kernel: fp32 caches, the asymmetric cache, and RoPE
// over a sub-range of the head.
cudaError_t launch_decode_step_simt(const DecodeArgs& a, const StepArgs& st, int Dk, kva_dtype cache_dtype,
                                    cudaStream_t s) {
  if (Dk == D) {
    if (cache_dtype == KVA_BF16) return launch_t<bf16_t, D, true>(a, KVA_BF16, s, st);
    return launch_t<float, D, true>(a, KVA_F32, s, st);
  }
  if (Dk == 192) {
    if (cache_dtype == KVA_BF16) return launch_t<bf16_t, 192, true>(a, KVA_BF16, s, st);
    return launch_t<float, 192, true>(a, KVA_F32, s, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kva
