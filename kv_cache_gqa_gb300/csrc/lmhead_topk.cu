// Top-k of each row of a logits matrix [B, V]: the k best (logit, id) pairs ordered by logit
// descending, equal logits toward the lower id (the argmax tie rule extended to a ranking).
//
// A candidate is the 64-bit key (order-preserving logit bits above ~id), so "better" is
// "larger key".  Each row is cut into segments of SEG logits, one CTA of 256 threads each:
// every thread loads its 8 logits at once, keeps a sorted list of its TK best keys in registers
// (branch-free insertion), each warp merges its 32 lists by TK rounds of "warp max of the list
// heads, pop the winner", and warp 0 merges the 8 warp lists the same way.  The segment's list
// goes to the workspace; the last CTA of the row to finish (an atomic ticket, no waiting)
// merges the row's segment lists into the result and clears its ticket.  The row's logits
// come from the lm_head kernels (whose final-norm prologue and GEMV are shared with the
// greedy argmax).
//
// Method: the top_k generation option of the published runtime interface (HunyuanOCR v1.5
// ncnn port, section 3.6) over the lm_head logits (Youtu-VL-4B ncnn port, "decoding and
// sampling").
#include "common.cuh"
#include "launch.h"

namespace kva {

namespace {

constexpr int TK_THREADS = 256;
constexpr int TK_WARPS = TK_THREADS / 32;

template <int TK>
__device__ __forceinline__ void list_insert(unsigned long long (&L)[TK], unsigned long long key) {
  if (key <= L[TK - 1]) return;                      // not among this list's best
#pragma unroll
  for (int i = TK - 1; i > 0; --i) L[i] = key > L[i - 1] ? L[i - 1] : (key > L[i] ? key : L[i]);
  L[0] = key > L[0] ? key : L[0];
}

// k rounds over the warp's 32 sorted lists; round r leaves the r-th best key in `out` (lane 0).
template <int TK>
__device__ __forceinline__ void warp_merge(unsigned long long (&L)[TK], int k, unsigned long long* out) {
  const int lane = threadIdx.x & 31;
  for (int r = 0; r < k; ++r) {
    unsigned long long best = L[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(FULL_MASK, best, o);
      best = other > best ? other : best;
    }
    if (lane == 0) out[r] = best;
    if (best != 0ull && L[0] == best) {              // keys are unique: exactly one lane pops
#pragma unroll
      for (int i = 0; i < TK - 1; ++i) L[i] = L[i + 1];
      L[TK - 1] = 0ull;
    }
  }
}

constexpr int PER_THREAD = 8;
constexpr int SEG = TK_THREADS * PER_THREAD;          // logits per CTA

// Merge the CTA's per-thread lists into one sorted list of k keys in `out` (shared memory).
template <int TK>
__device__ __forceinline__ void cta_merge(unsigned long long (&L)[TK], int k, unsigned long long (*s_w)[TK],
                                          unsigned long long* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  warp_merge<TK>(L, k, &s_w[warp][0]);
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < TK; ++i) L[i] = (lane < TK_WARPS && i < k) ? s_w[lane][i] : 0ull;
    warp_merge<TK>(L, k, out);
  }
  __syncthreads();
}

template <int TK>
__global__ void __launch_bounds__(TK_THREADS)
topk_rows_kernel(const float* __restrict__ logits, int V, int k, int n_seg, unsigned long long* __restrict__ part,
                 unsigned int* __restrict__ tickets, int32_t* __restrict__ out_ids, float* __restrict__ out_vals) {
  __shared__ unsigned long long s_w[TK_WARPS][TK];
  __shared__ unsigned long long s_out[TK];
  __shared__ int s_last;
  griddep_wait();
  griddep_launch_dependents();
  const int seg = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const float* z = logits + (int64_t)b * V;
  unsigned long long L[TK];
#pragma unroll
  for (int i = 0; i < TK; ++i) L[i] = 0ull;
  {
    float x[PER_THREAD];
    const int v0 = seg * SEG + tid;
#pragma unroll
    for (int j = 0; j < PER_THREAD; ++j) {       // all of this thread's loads in flight together
      const int v = v0 + j * TK_THREADS;
      x[j] = v < V ? __ldg(z + v) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < PER_THREAD; ++j) {
      const int v = v0 + j * TK_THREADS;
      if (v < V) list_insert<TK>(L, argmax_key(x[j], (uint32_t)v));
    }
  }
  cta_merge<TK>(L, k, s_w, s_out);
  unsigned long long* my = part + ((int64_t)b * n_seg + seg) * TK;
  for (int r = tid; r < TK; r += TK_THREADS) my[r] = r < k ? s_out[r] : 0ull;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&tickets[b], 1u) == (unsigned)(n_seg - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last segment of the row: merge the n_seg lists (thread t folds lists t, t + 256, ...)
#pragma unroll
  for (int i = 0; i < TK; ++i) L[i] = 0ull;
  for (int sg = tid; sg < n_seg; sg += TK_THREADS) {
    const unsigned long long* q = part + ((int64_t)b * n_seg + sg) * TK;
    for (int i = 0; i < k; ++i) list_insert<TK>(L, __ldcg(q + i));
  }
  cta_merge<TK>(L, k, s_w, s_out);
  for (int r = tid; r < k; r += TK_THREADS) {
    const unsigned long long key = s_out[r];
    out_ids[(int64_t)b * k + r] = key ? (int32_t)(0xffffffffu - (uint32_t)(key & 0xffffffffull)) : -1;
    if (out_vals) out_vals[(int64_t)b * k + r] = float_from_order_bits((uint32_t)(key >> 32));
  }
  if (tid == 0) tickets[b] = 0u;
}

template <int TK>
cudaError_t launch_tk(const float* logits, int B, int V, int k, void* ws, int32_t* ids, float* vals, cudaStream_t s) {
  const int n_seg = (V + SEG - 1) / SEG;
  unsigned int* tickets = static_cast<unsigned int*>(ws);
  unsigned long long* part = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(ws) +
                                                                   ((sizeof(unsigned) * (size_t)B + 255) / 256) * 256);
  return launch_pdl(topk_rows_kernel<TK>, dim3(n_seg, B), dim3(TK_THREADS), 0, s, logits, V, k, n_seg, part, tickets,
                    ids, vals);
}

}  // namespace

size_t topk_rows_workspace_bytes(int B, int V) {
  const size_t n_seg = (size_t)(V + SEG - 1) / SEG;
  return ((sizeof(unsigned) * (size_t)B + 255) / 256) * 256 + sizeof(unsigned long long) * (size_t)B * n_seg * LMHEAD_TOPK_MAX;
}

cudaError_t launch_topk_rows(const float* logits, int B, int V, int k, void* workspace, int32_t* out_ids,
                             float* out_vals, cudaStream_t s) {
  if (k <= 4) return launch_tk<4>(logits, B, V, k, workspace, out_ids, out_vals, s);
  if (k <= 8) return launch_tk<8>(logits, B, V, k, workspace, out_ids, out_vals, s);
  if (k <= 16) return launch_tk<16>(logits, B, V, k, workspace, out_ids, out_vals, s);
  if (k <= LMHEAD_TOPK_MAX) return launch_tk<LMHEAD_TOPK_MAX>(logits, B, V, k, workspace, out_ids, out_vals, s);
  return cudaErrorInvalidValue;
}

}  // namespace kva
