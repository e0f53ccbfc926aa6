// Multi-query verify block (speculative decoding): k query rows per instance attend to the
// cache with a causal limit inside the block, bf16 cache, head_dim 128.
//
// The split-KV decode structure with full 16-row MMA tiles: a CTA serves one (chunk c,
// KV head g, row tile rt, instance b).  Its 16 rows are r = rt*16 + (0..15) of the group's
// G*k rows, row r = (block position i = r / G, query head g*G + r % G); row i sees slots
// [0, L - k + i].  The CTA's four warps are independent: warp w takes the 16-key tiles w,
// w+4, ... of the chunk through a private 2-stage TMA ring (K and V as [16 keys x 64 dims]
// boxes, 128-byte swizzle), and per tile computes
//   S = Q K^T      16 rows x 16 keys, 16 mma.sync m16n8k16 (both row halves live)
//   online softmax per row in registers (each lane holds rows lane/4 and lane/4 + 8)
//   O += P V       P reused from the S accumulators as the A fragment, 16 MMAs
// so every K/V byte of the chunk is read once for all 16 rows.  Keys past a row's causal
// limit only occur in the last k - 1 slots and are masked there.  Warps merge in shared
// memory; with several chunks the CTA writes partials and the last CTA of (b, g, rt) merges.
//
// Method: the target-verification forward of a draft block with a multi-token causal mask
// over the existing cache (HunyuanOCR v1.5 ncnn port, section 3.8), GQA by repeat-interleave
// grouping (Penguin-VL ncnn port, section 3), bf16 storage with fp32 accumulation
// (HunyuanOCR v1.5 ncnn port, section 3.7).
#include "launch.h"
#include "tc.cuh"

namespace kva {

namespace {

constexpr int D = DECODE_HEAD_DIM;
constexpr int WARPS = 4;
constexpr int THREADS = WARPS * 32;
constexpr int KT = 16;                          // keys per warp tile
constexpr int NS = 2;                           // ring stages per warp (three CTAs fit an SM)
constexpr int BOX = KT * 128;                   // one [16 keys x 64 dims] swizzled box, 2 KB
constexpr int STAGE = 4 * BOX;                  // K lo, K hi, V lo, V hi
constexpr int RING = NS * STAGE;                // per warp
constexpr int ROWS = 16;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
// D = A B + D with all four A registers live (rows g and g + 8)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t swz(int key, int ch) { return key * 128 + ((ch ^ (key & 7)) << 4); }

__device__ __forceinline__ uint32_t q_pair(const void* q, kva_dtype dt, int64_t off) {
  if (dt == KVA_BF16) return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint16_t*>(q) + off);
  const float* f = reinterpret_cast<const float*>(q) + off;
  return pack_bf16x2(f[0], f[1]);
}

__global__ void __launch_bounds__(THREADS, 3)
verify_mma_kernel(const __grid_constant__ VerifyArgs a, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, kva_dtype q_dtype) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int c = blockIdx.x, g = blockIdx.y / a.RT, rt = blockIdx.y % a.RT, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.Hq / a.Hkv, R = G * a.k;

  unsigned char* ring = smem + warp * RING;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + WARPS * RING) + warp * NS;
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
    if (warp == 0) { tc::tma_prefetch_desc(&tmK); tc::tma_prefetch_desc(&tmV); }
  }
  griddep_wait();                               // inputs of this launch are complete from here on
  griddep_launch_dependents();
  const int L = a.lengths[b];
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

  // ---- this lane's rows: ra = lane/4 and rb = ra + 8 of the tile; pair t = lane % 4 ----
  const int t = lane & 3;
  const int ra = lane >> 2, rb = ra + 8;
  const int ga = rt * ROWS + ra, gb = rt * ROWS + rb;           // rows of the group
  const bool va = ga < R, vb = gb < R;
  // causal limit (exclusive) of each row; rows past the group see every valid key
  const int lim_a = va ? L - a.k + ga / G + 1 : L;
  const int lim_b = vb ? L - a.k + gb / G + 1 : L;
  auto q_off = [&](int gr) {                   // element offset of row gr's query
    return (((int64_t)b * a.k + gr / G) * a.Hq + g * G + gr % G) * D;
  };
  uint32_t qa[8][4];
  {
    const int64_t oa = va ? q_off(ga) : 0, ob = vb ? q_off(gb) : 0;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int d0 = 16 * kk + 2 * t;
      qa[kk][0] = va ? q_pair(a.q, q_dtype, oa + d0) : 0u;
      qa[kk][1] = vb ? q_pair(a.q, q_dtype, ob + d0) : 0u;
      qa[kk][2] = va ? q_pair(a.q, q_dtype, oa + d0 + 8) : 0u;
      qa[kk][3] = vb ? q_pair(a.q, q_dtype, ob + d0 + 8) : 0u;
    }
  }

  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
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
    const uint32_t sK = smem_u32(stg), sV = sK + 2 * BOX;

    // ---- S = Q K^T: n-tile 0 = keys 0..7, n-tile 1 = keys 8..15 ----
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int key = rr + 8 * (mi >> 1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int half = kk >> 2, ch = ((kk & 3) << 1) + (mi & 1);
        uint32_t bf[4];
        ldsm_x4(sK + half * BOX + swz(key, ch), bf);
        mma16816(s0, qa[kk], bf[0], bf[1]);
        mma16816(s1, qa[kk], bf[2], bf[3]);
      }
    }
    // ---- online softmax of rows a (s*[0..1]) and b (s*[2..3]) over keys 2t, 2t+1, 8+2t, 9+2t ----
    const int kx[4] = {ks + 2 * t, ks + 2 * t + 1, ks + 8 + 2 * t, ks + 9 + 2 * t};
    float xa[4] = {s0[0], s0[1], s1[0], s1[1]}, xb[4] = {s0[2], s0[3], s1[2], s1[3]};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      xa[i] = (kx[i] < ks + nk && kx[i] < lim_a) ? xa[i] * a.scale_log2 : -INFINITY;
      xb[i] = (kx[i] < ks + nk && kx[i] < lim_b) ? xb[i] * a.scale_log2 : -INFINITY;
    }
    float ta = fmaxf(fmaxf(xa[0], xa[1]), fmaxf(xa[2], xa[3]));
    float tb = fmaxf(fmaxf(xb[0], xb[1]), fmaxf(xb[2], xb[3]));
    ta = fmaxf(ta, __shfl_xor_sync(FULL_MASK, ta, 1)); ta = fmaxf(ta, __shfl_xor_sync(FULL_MASK, ta, 2));
    tb = fmaxf(tb, __shfl_xor_sync(FULL_MASK, tb, 1)); tb = fmaxf(tb, __shfl_xor_sync(FULL_MASK, tb, 2));
    // a tile can be entirely past a row's limit (the row keeps its state: alpha = 1, P = 0)
    const float mna = fmaxf(m_a, ta), mnb = fmaxf(m_b, tb);
    const float alpha_a = mna == -INFINITY ? 1.f : exp2f(m_a - mna);
    const float alpha_b = mnb == -INFINITY ? 1.f : exp2f(m_b - mnb);
    const float ra_ = mna == -INFINITY ? 0.f : mna, rb_ = mnb == -INFINITY ? 0.f : mnb;
    float pa[4], pb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) { pa[i] = exp2f(xa[i] - ra_); pb[i] = exp2f(xb[i] - rb_); }
    uint32_t pfrag[4];
    pfrag[0] = pack_bf16x2(pa[0], pa[1]);      // row a, keys 2t, 2t+1
    pfrag[1] = pack_bf16x2(pb[0], pb[1]);      // row b, keys 2t, 2t+1
    pfrag[2] = pack_bf16x2(pa[2], pa[3]);      // row a, keys 8+2t, 9+2t
    pfrag[3] = pack_bf16x2(pb[2], pb[3]);      // row b
    float sa = bf16_lo(pfrag[0]) + bf16_hi(pfrag[0]) + bf16_lo(pfrag[2]) + bf16_hi(pfrag[2]);
    float sb = bf16_lo(pfrag[1]) + bf16_hi(pfrag[1]) + bf16_lo(pfrag[3]) + bf16_hi(pfrag[3]);
    sa += __shfl_xor_sync(FULL_MASK, sa, 1); sa += __shfl_xor_sync(FULL_MASK, sa, 2);
    sb += __shfl_xor_sync(FULL_MASK, sb, 1); sb += __shfl_xor_sync(FULL_MASK, sb, 2);
    l_a = l_a * alpha_a + sa; m_a = mna;
    l_b = l_b * alpha_b + sb; m_b = mnb;
#pragma unroll
    for (int n = 0; n < 16; ++n) { o[n][0] *= alpha_a; o[n][1] *= alpha_a; o[n][2] *= alpha_b; o[n][3] *= alpha_b; }

    // ---- O += P V ----
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int key = rr + 8 * (mi & 1);
#pragma unroll
      for (int nd = 0; nd < 8; ++nd) {
        const int half = nd >> 2, ch = ((nd & 3) << 1) + (mi >> 1);
        uint32_t bf[4];
        ldsm_x4_t(sV + half * BOX + swz(key, ch), bf);
        mma16816(o[2 * nd], pfrag, bf[0], bf[1]);
        mma16816(o[2 * nd + 1], pfrag, bf[2], bf[3]);
      }
    }
    __syncwarp();                               // all lanes are done with this stage
    if (lane == 0 && u + NS < n_mine) {
      fence_proxy_async_smem();                 // order this stage's generic accesses before the refill
      issue(u + NS);
    }
  }

  // ---- merge the warps: 16 rows, row ra in lanes 4ra..4ra+3 (o[][0..1]), row rb (o[][2..3]) ----
  __syncthreads();                              // rings drained: reuse them for the merge
  float* sm_m = reinterpret_cast<float*>(smem);             // [WARPS][16]
  float* sm_l = sm_m + WARPS * ROWS;                        // [WARPS][16]
  float* sm_o = sm_l + WARPS * ROWS;                        // [WARPS][16][D]
  if (t == 0) {
    sm_m[warp * ROWS + ra] = ok ? m_a : NAN; sm_l[warp * ROWS + ra] = ok ? l_a : NAN;
    sm_m[warp * ROWS + rb] = ok ? m_b : NAN; sm_l[warp * ROWS + rb] = ok ? l_b : NAN;
  }
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    sm_o[(warp * ROWS + ra) * D + 8 * n + 2 * t] = o[n][0];
    sm_o[(warp * ROWS + ra) * D + 8 * n + 2 * t + 1] = o[n][1];
    sm_o[(warp * ROWS + rb) * D + 8 * n + 2 * t] = o[n][2];
    sm_o[(warp * ROWS + rb) * D + 8 * n + 2 * t + 1] = o[n][3];
  }
  __syncthreads();
  __shared__ float s_M[ROWS], s_L[ROWS];
  if (tid < ROWS) {
    float M = -INFINITY;
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, sm_m[w * ROWS + tid]);
    float Ls = 0.f;
    for (int w = 0; w < WARPS; ++w) {
      const float mw = sm_m[w * ROWS + tid];
      Ls += (mw == -INFINITY) ? 0.f : exp2f(mw - M) * sm_l[w * ROWS + tid];
    }
    s_M[tid] = M; s_L[tid] = Ls;
  }
  __syncthreads();
  const bool single = (n_chunks == 1);
  const int64_t pbase = ((int64_t)(b * a.Hkv + g) * a.RT + rt) * ROWS;      // partial row index base
  for (int idx = tid; idx < ROWS * D; idx += THREADS) {
    const int r = idx / D, d = idx % D;
    const int gr = rt * ROWS + r;
    if (gr >= R) continue;
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const float mw = sm_m[w * ROWS + r];
      if (mw != -INFINITY) tot += exp2f(mw - s_M[r]) * sm_o[(w * ROWS + r) * D + d];
    }
    if (single) {
      a.out[q_off(gr) + d] = tot / s_L[r];
    } else {
      const int64_t pidx = (pbase + r) * a.max_chunks + c;
      a.part_acc[pidx * D + d] = tot;
      if (d == 0) { a.part_ml[2 * pidx] = s_M[r]; a.part_ml[2 * pidx + 1] = s_L[r]; }
    }
  }
  if (single) return;

  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  const int64_t cidx = (int64_t)(b * a.Hkv + g) * a.RT + rt;
  if (tid == 0) s_last = (atomicAdd(&a.counters[cidx], 1u) == (unsigned)(n_chunks - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int idx = tid; idx < ROWS * D; idx += THREADS) {
    const int r = idx / D, d = idx % D;
    const int gr = rt * ROWS + r;
    if (gr >= R) continue;
    const int64_t p0 = (pbase + r) * a.max_chunks;
    float M = -INFINITY;
    for (int cc = 0; cc < n_chunks; ++cc) M = fmaxf(M, __ldcg(&a.part_ml[2 * (p0 + cc)]));
    float num = 0.f, den = 0.f;
    for (int cc = 0; cc < n_chunks; ++cc) {
      const float mc = __ldcg(&a.part_ml[2 * (p0 + cc)]);
      if (mc == -INFINITY) continue;           // a chunk wholly past this row's limit
      const float w = exp2f(mc - M);
      num = fmaf(w, __ldcg(&a.part_acc[(p0 + cc) * D + d]), num);
      den = fmaf(w, __ldcg(&a.part_ml[2 * (p0 + cc) + 1]), den);
    }
    a.out[q_off(gr) + d] = num / den;
  }
  if (tid == 0) a.counters[cidx] = 0u;
}

// One thread per instance: accepted prefix, next token and the committed length.
__global__ void verify_commit_kernel(const int32_t* posterior, const int32_t* block, int B, int k, int32_t* lengths,
                                     int32_t* accepted, int32_t* next_token) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int32_t* y = posterior + (int64_t)b * k;
  const int32_t* x = block + (int64_t)b * k;
  int acc = 0;
  while (acc < k - 1 && y[acc] == x[acc + 1]) ++acc;
  accepted[b] = acc;
  next_token[b] = y[acc];
  lengths[b] = lengths[b] - k + acc + 1;
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& a, kva_dtype q_dtype, cudaStream_t s) {
  const size_t smem = (size_t)WARPS * RING + WARPS * NS * 8 + 1024;
  static DeviceOnce configured;
  if (!configured.done()) {
    cudaError_t e = cudaFuncSetAttribute(verify_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured.mark();
  }
  CUtensorMap mk, mv;
  cudaError_t e = decode_cache_map(&mk, a.kc, a.capacity, a.Hkv, a.B, a.inst_stride);
  if (e != cudaSuccess) return e;
  if ((e = decode_cache_map(&mv, a.vc, a.capacity, a.Hkv, a.B, a.inst_stride)) != cudaSuccess) return e;
  dim3 grid(a.max_chunks, a.Hkv * a.RT, a.B);
  return launch_pdl(verify_mma_kernel, grid, dim3(THREADS), smem, s, a, mk, mv, q_dtype);
}

cudaError_t launch_verify_commit(const int32_t* posterior, const int32_t* block_tokens, int B, int k,
                                 int32_t* lengths, int32_t* accepted, int32_t* next_token, cudaStream_t s) {
  const int threads = 128;
  return launch_pdl(verify_commit_kernel, dim3((B + threads - 1) / threads), dim3(threads), 0, s, posterior,
                    block_tokens, B, k, lengths, accepted, next_token);
}

}  // namespace kva
