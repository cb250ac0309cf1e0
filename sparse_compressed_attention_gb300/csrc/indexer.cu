// Lightning-indexer scoring on CUDA cores and the per-query top-k selection.
//
// Score: Primus PR #930 item 6a (per-head weights scaled by Hi^-1/2 Di^-1/2)
// and item 4 (fp32 scoring); "Enabling DeepSeek-V4-Flash Training ...",
// section "Kernel fusions", row "Indexer scoring tail" (ReLU, per-head
// multiply, head sum, causal mask built inline).  Selection: section "Three
// attention types, interleaved" (keep the best 512 entries).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace v4 {

namespace {

constexpr int kScoreThreads = 256;
constexpr int kHeadChunk = 16;

// One block per (query t, batch b).  Prepared queries and scaled weights of
// the row sit in shared memory; thread j scores entries s = j, j+256, ...
// for s < n_vis(t).  Per head: d = sum_c q[h][c] k[s][c] accumulated in
// order c = 0..Di-1 in fp32, then I += w'[h] * max(d, 0) in head order.
template <typename T>
__global__ void __launch_bounds__(kScoreThreads)
indexer_scores_kernel(const T* __restrict__ iqp, const T* __restrict__ ikey,
                      const float* __restrict__ w, float* __restrict__ scores,
                      int S, int N, int Hi, int Di, int ratio, float wscale) {
  extern __shared__ float sm[];
  float* s_q = sm;                 // [Hi][Di]
  float* s_w = sm + Hi * Di;       // [Hi]
  const int t = blockIdx.x;
  const int b = blockIdx.y;
  const int nv = min(n_visible(t, ratio), N);
  if (nv == 0) return;
  const T* qrow = iqp + ((size_t)b * S + t) * Hi * Di;
  for (int i = threadIdx.x; i < Hi * Di; i += kScoreThreads) s_q[i] = to_f(qrow[i]);
  for (int i = threadIdx.x; i < Hi; i += kScoreThreads)
    s_w[i] = w[((size_t)b * S + t) * Hi + i] * wscale;
  __syncthreads();
  float* out = scores + ((size_t)b * S + t) * N;
  const T* keys = ikey + (size_t)b * N * Di;
  for (int s = threadIdx.x; s < nv; s += kScoreThreads) {
    const T* k = keys + (size_t)s * Di;
    float total = 0.f;
    for (int h0 = 0; h0 < Hi; h0 += kHeadChunk) {
      float d[kHeadChunk];
#pragma unroll
      for (int j = 0; j < kHeadChunk; ++j) d[j] = 0.f;
      for (int c8 = 0; c8 < Di; c8 += 8) {
        float kv[8];
        load8(k + c8, kv);
#pragma unroll
        for (int j = 0; j < kHeadChunk; ++j) {
          if (h0 + j < Hi) {
            const float* qh = s_q + (h0 + j) * Di + c8;
#pragma unroll
            for (int e = 0; e < 8; ++e) d[j] = fmaf(qh[e], kv[e], d[j]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kHeadChunk; ++j)
        if (h0 + j < Hi) total = fmaf(s_w[h0 + j], fmaxf(d[j], 0.f), total);
    }
    out[s] = total;
  }
}

// Order-preserving map of a float to an unsigned key (larger float, larger key).
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTopkThreads = 256;

// Block-wide exclusive scan of one int per thread; returns the prefix and
// writes the block total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int wv = lane < kTopkThreads / 32 ? s_warp[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, wv, o);
      if (lane >= o) wv += y;
    }
    if (lane < kTopkThreads / 32) s_warp[lane] = wv;
  }
  __syncthreads();
  const int before = (wid > 0 ? s_warp[wid - 1] : 0) + x - v;
  *total = s_warp[kTopkThreads / 32 - 1];
  __syncthreads();
  return before;
}

// One block per (t, b): exact top-K of the row's n_vis scores by a 4-pass
// MSB-first radix select on the ordered 32-bit keys (8 bits per pass), then
// an index-ordered compaction: every key above the K-th key, plus the
// lowest-index keys equal to it until K are taken.  Output in ascending
// index order, -1 padded.
__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const float* __restrict__ scores, int32_t* __restrict__ idx, float* __restrict__ iscore,
            int S, int N, int K, int ratio) {
  __shared__ int s_hist[256];
  __shared__ int s_warp[kTopkThreads / 32];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_krem;
  const int t = blockIdx.x, b = blockIdx.y;
  const int nv = min(n_visible(t, ratio), N);
  const float* row = scores + ((size_t)b * S + t) * N;
  int32_t* orow = idx + ((size_t)b * S + t) * K;
  float* srow = iscore ? iscore + ((size_t)b * S + t) * K : nullptr;
  if (nv <= K) {
    for (int j = threadIdx.x; j < K; j += kTopkThreads) {
      orow[j] = j < nv ? j : -1;
      if (srow) srow[j] = j < nv ? row[j] : -INFINITY;
    }
    return;
  }
  if (threadIdx.x == 0) { s_prefix = 0u; s_mask = 0u; s_krem = K; }
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kTopkThreads) s_hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix, mask = s_mask;
    for (int s = threadIdx.x; s < nv; s += kTopkThreads) {
      const uint32_t u = ordered_key(row[s]);
      if ((u & mask) == prefix) atomicAdd(&s_hist[(u >> shift) & 0xFFu], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int krem = s_krem, acc = 0, dsel = 0;
      for (int d = 255; d >= 0; --d) {
        if (acc + s_hist[d] >= krem) { dsel = d; break; }
        acc += s_hist[d];
      }
      s_krem = krem - acc;
      s_prefix = prefix | ((uint32_t)dsel << shift);
      s_mask = mask | (0xFFu << shift);
    }
    __syncthreads();
  }
  const uint32_t kth = s_prefix;
  const int ties_needed = s_krem;      // keys equal to kth that are taken
  int out_base = 0, tie_base = 0;
  for (int c0 = 0; c0 < nv; c0 += kTopkThreads) {
    const int s = c0 + threadIdx.x;
    uint32_t u = 0;
    if (s < nv) u = ordered_key(row[s]);
    const int is_tie = (s < nv && u == kth) ? 1 : 0;
    int tie_tot;
    const int tie_rank = tie_base + block_exclusive_scan(is_tie, s_warp, &tie_tot);
    const int take = (s < nv) && (u > kth || (is_tie && tie_rank < ties_needed)) ? 1 : 0;
    int take_tot;
    const int pos = out_base + block_exclusive_scan(take, s_warp, &take_tot);
    if (take) {
      orow[pos] = s;
      if (srow) srow[pos] = row[s];
    }
    out_base += take_tot;
    tie_base += tie_tot;
  }
  for (int j = out_base + threadIdx.x; j < K; j += kTopkThreads) {
    orow[j] = -1;
    if (srow) srow[j] = -INFINITY;
  }
}

template <typename T>
cudaError_t scores_t(const v4_config& c, const void* iqp, const void* ikey, const float* w,
                     float* scores, cudaStream_t st) {
  const int N = c.seqlen / c.ratio;
  const size_t smem = (size_t)(c.idx_heads * c.idx_dim + c.idx_heads) * sizeof(float);
  auto kern = indexer_scores_kernel<T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const float wscale = 1.0f / sqrtf((float)c.idx_heads) / sqrtf((float)c.idx_dim);
  dim3 grid(c.seqlen, c.batch);
  kern<<<grid, kScoreThreads, smem, st>>>((const T*)iqp, (const T*)ikey, w, scores, c.seqlen, N,
                                          c.idx_heads, c.idx_dim, c.ratio, wscale);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_scores_simt(const v4_config& c, const void* iqp, const void* ikey,
                                       const float* w, float* scores, cudaStream_t st) {
  if (c.dtype == V4_BF16) return scores_t<bf16>(c, iqp, ikey, w, scores, st);
  return scores_t<float>(c, iqp, ikey, w, scores, st);
}

cudaError_t launch_topk(const v4_config& c, const float* scores, int32_t* idx, float* iscore,
                        cudaStream_t st) {
  const int N = c.seqlen / c.ratio;
  dim3 grid(c.seqlen, c.batch);
  topk_kernel<<<grid, kTopkThreads, 0, st>>>(scores, idx, iscore, c.seqlen, N, c.topk, c.ratio);
  note_launch();
  return cudaGetLastError();
}

}  // namespace v4
