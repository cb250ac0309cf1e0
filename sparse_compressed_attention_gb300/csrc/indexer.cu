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

// One block per (t, b): exact top-K of the row's n_vis scores.  The row is
// loaded once into shared memory as order-preserving 32-bit keys; a 4-pass
// MSB-first radix select (8 bits per pass) finds the K-th key: each pass
// builds per-warp 256-bin histograms (lanes that hit the same bin combine
// their increments first), sums them, and one warp locates the digit with a
// suffix scan.  The compaction keeps every key above the K-th key plus the
// lowest-index keys equal to it.  Output in ascending index
// order, -1 padded.  Rows longer than the shared-memory capacity fall back to
// reading the keys from global memory on every pass.
constexpr int kTopkWarps = kTopkThreads / 32;

__device__ __forceinline__ uint32_t row_key(const float* row, const uint32_t* skeys, bool in_smem, int s) {
  return in_smem ? skeys[s] : ordered_key(row[s]);
}

__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const float* __restrict__ scores, int32_t* __restrict__ idx, float* __restrict__ iscore,
            int S, int N, int K, int ratio, int smem_cap) {
  extern __shared__ uint32_t skeys[];
  __shared__ int s_hist[kTopkWarps][256];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_krem, s_done;
  const int t = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nv = min(n_visible(t, ratio), N);
  const float* row = scores + ((size_t)b * S + t) * N;
  int32_t* orow = idx + ((size_t)b * S + t) * K;
  float* srow = iscore ? iscore + ((size_t)b * S + t) * K : nullptr;
  if (nv <= K) {
    for (int j = tid; j < K; j += kTopkThreads) {
      orow[j] = j < nv ? j : -1;
      if (srow) srow[j] = j < nv ? row[j] : -INFINITY;
    }
    return;
  }
  const bool in_smem = nv <= smem_cap;
  if (in_smem)
    for (int s = tid; s < nv; s += kTopkThreads) skeys[s] = ordered_key(row[s]);
  for (int i = tid; i < kTopkWarps * 256; i += kTopkThreads) (&s_hist[0][0])[i] = 0;
  if (tid == 0) { s_prefix = 0u; s_mask = 0u; s_krem = K; s_done = 0; }
  __syncthreads();
  for (int shift = 24; shift >= 0 && !s_done; shift -= 8) {
    // histograms are zero here: cleared before the first pass, and by the
    // select phase of the previous one
    const uint32_t prefix = s_prefix, mask = s_mask;
    for (int s0 = 0; s0 < nv; s0 += kTopkThreads) {
      const int s = s0 + tid;
      int bin = -1;
      if (s < nv) {
        const uint32_t u = row_key(row, skeys, in_smem, s);
        if ((u & mask) == prefix) bin = (int)((u >> shift) & 0xFFu);
      }
      // lanes of the warp with the same bin add once (after the first pass
      // most keys no longer match the prefix: skip warps with none)
      if (shift == 24 || __any_sync(0xffffffffu, bin >= 0)) {
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (bin >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_hist[wid][bin], __popc(peers));
      }
    }
    __syncthreads();
    // totals per digit
    {
      const int d = tid;                       // kTopkThreads == 256 digits
      int sum = 0;
#pragma unroll
      for (int w = 0; w < kTopkWarps; ++w) sum += s_hist[w][d];
      s_hist[0][d] = sum;
    }
    __syncthreads();
    if (wid == 0) {
      // lane l owns digits 255-8l .. 248-8l (high digits first)
      const int krem = s_krem;                  // read before any lane of the warp writes it
      int cnt[8];
      int local = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = s_hist[0][255 - 8 * lane - i];
        local += cnt[i];
      }
      int incl = local;                         // inclusive scan over lanes (high digits first)
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int before = incl - local;
      const bool mine = before < krem && incl >= krem;
      if (mine) {
        int acc = before, dsel = 0, csel = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (acc + cnt[i] >= krem) { dsel = 255 - 8 * lane - i; csel = cnt[i]; break; }
          acc += cnt[i];
        }
        s_krem = krem - acc;
        s_prefix = prefix | ((uint32_t)dsel << shift);
        s_mask = mask | (0xFFu << shift);
        // every key of the digit is taken: the prefix already separates the
        // selection, the remaining digits need no pass
        if (csel == krem - acc) s_done = 1;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) s_hist[0][255 - 8 * lane - i] = 0;     // this lane's digits, read above
    } else {
      for (int i = lane; i < 256; i += 32) s_hist[wid][i] = 0;            // per-warp counts, summed above
    }
    __syncthreads();
  }
  // the k-th key's resolved digits; keys compare on those digits only (all
  // 32 bits unless the selection was separated earlier, in which case every
  // key equal to kth on them is taken)
  const uint32_t kth = s_prefix, kmask = s_mask;
  const int ties_needed = s_krem;      // keys equal to kth that are taken
  // Compaction: warp w owns the contiguous index range [lo, hi).  Counts of
  // keys above kth and equal to kth per warp give every warp its first
  // output slot and its first tie rank; each warp then writes its range in
  // index order.
  const int span = ((nv + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
  const int lo = min(wid * span, nv), hi = min(lo + span, nv);
  int gt = 0, eq = 0;
  for (int s0 = lo; s0 < hi; s0 += 32) {
    const int s = s0 + lane;
    const uint32_t u = s < hi ? row_key(row, skeys, in_smem, s) & kmask : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, s < hi && u > kth));
    eq += __popc(__ballot_sync(0xffffffffu, s < hi && u == kth));
  }
  if (lane == 0) { s_hist[1][wid] = gt; s_hist[2][wid] = eq; }
  __syncthreads();
  int out_pos = 0, tie_rank = 0;
  for (int w = 0; w < wid; ++w) {
    const int e = s_hist[2][w];
    out_pos += s_hist[1][w] + max(0, min(e, ties_needed - tie_rank));
    tie_rank += e;
  }
  const unsigned below = (1u << lane) - 1u;
  for (int s0 = lo; s0 < hi; s0 += 32) {
    const int s = s0 + lane;
    const uint32_t u = s < hi ? row_key(row, skeys, in_smem, s) & kmask : 0u;
    const unsigned tie_bits = __ballot_sync(0xffffffffu, s < hi && u == kth);
    const int my_tie = tie_rank + __popc(tie_bits & below);
    const bool take = s < hi && (u > kth || (u == kth && my_tie < ties_needed));
    const unsigned take_bits = __ballot_sync(0xffffffffu, take);
    if (take) {
      const int pos = out_pos + __popc(take_bits & below);
      orow[pos] = s;
      if (srow) srow[pos] = row[s];
    }
    out_pos += __popc(take_bits);
    tie_rank += __popc(tie_bits);
  }
  // slots past the selection (only when fewer than K keys exist; nv > K here)
  if (wid == kTopkWarps - 1)
    for (int j = out_pos + lane; j < K; j += 32) {
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
  // rows of up to 4096 keys stay in shared memory; longer rows re-read their
  // scores from L2 on every pass, which keeps more rows resident per SM
  // (measured faster at 16384 keys than staging 64 KB per row)
  const int cap = N < 4096 ? N : 4096;
  const size_t smem = (size_t)cap * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(c.seqlen, c.batch);
  topk_kernel<<<grid, kTopkThreads, smem, st>>>(scores, idx, iscore, c.seqlen, N, c.topk, c.ratio, cap);
  note_launch();
  return cudaGetLastError();
}

}  // namespace v4
