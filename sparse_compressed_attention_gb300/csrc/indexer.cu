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

// One block per (query row i, batch b), position t = t0 + i of Sq query rows
// per sequence.  Prepared queries and scaled weights of the row sit in shared memory; thread j scores entries s = j, j+256, ...
// for s < n_vis(t).  Per head: d = sum_c q[h][c] k[s][c] accumulated in
// order c = 0..Di-1 in fp32, then I += w'[h] * max(d, 0) in head order.
template <typename T>
__global__ void __launch_bounds__(kScoreThreads)
indexer_scores_kernel(const T* __restrict__ iqp, const T* __restrict__ ikey,
                      const float* __restrict__ w, float* __restrict__ scores,
                      int Sq, int t0, int N, int Hi, int Di, int ratio, float wscale) {
  extern __shared__ float sm[];
  float* s_q = sm;                 // [Hi][Di]
  float* s_w = sm + Hi * Di;       // [Hi]
  const int t = t0 + blockIdx.x;
  const int b = blockIdx.y;
  const size_t qr = (size_t)b * Sq + blockIdx.x;     // query row
  const int nv = min(n_visible(t, ratio), N);
  if (nv == 0) return;
  const T* qrow = iqp + qr * Hi * Di;
  for (int i = threadIdx.x; i < Hi * Di; i += kScoreThreads) s_q[i] = to_f(qrow[i]);
  for (int i = threadIdx.x; i < Hi; i += kScoreThreads)
    s_w[i] = w[qr * Hi + i] * wscale;
  __syncthreads();
  float* out = scores + qr * N;
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

// Four warps per row: the per-row fixed work (block barriers, the digit
// scan, clears, compaction offsets) is shared by fewer warps and more rows
// are resident per SM (measured 0.162 -> 0.156 ms at S=16384, 0.031 ->
// 0.024 ms at B=2, S=3000, K=64 against eight warps per row).
constexpr int kTopkThreads = 128;

// One block per (query row i, batch b), position t = t0 + i: exact top-K of
// the row's n_vis(t) scores.  The row is
// held in shared memory as order-preserving 32-bit keys; a 4-pass MSB-first
// radix select (8 bits per pass) finds the K-th key, and a compaction keeps
// every key above it plus the lowest-index keys equal to it.  Output in
// ascending index order, -1 padded.
//
// The kernel is bound by instruction issue, so each thread takes four
// consecutive keys per shared-memory load.  Each pass builds per-warp
// 256-bin histograms: in the first pass (sign and exponent bits) the scores
// crowd a few bins, so lanes that hit the same bin combine their increments
// before one shared-memory add, and that pass runs while the keys are
// loaded; later digits spread over the bins and each matching key adds
// directly.  One warp locates the digit with a scan.  The select stops once
// every key of the located digit is taken.  In the compaction each warp owns
// a contiguous range; per-warp counts give its first output slot and one
// packed lane scan per 128 keys orders its writes.  Rows longer than the
// shared-memory capacity read their keys from global memory on every pass.
constexpr int kTopkWarps = kTopkThreads / 32;

__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// keys 4c .. 4c+3 of the row (entries at or past nv are unspecified)
__device__ __forceinline__ uint4 row_key4(const float* row, const uint4* skeys4, bool in_smem, bool vec, int c,
                                          int nv) {
  if (in_smem) return skeys4[c];
  const int s = 4 * c;
  if (vec && s + 3 < nv) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(row) + c);
    return make_uint4(ordered_key(f.x), ordered_key(f.y), ordered_key(f.z), ordered_key(f.w));
  }
  return make_uint4(s < nv ? ordered_key(row[s]) : 0u, s + 1 < nv ? ordered_key(row[s + 1]) : 0u,
                    s + 2 < nv ? ordered_key(row[s + 2]) : 0u, s + 3 < nv ? ordered_key(row[s + 3]) : 0u);
}

// the four keys' contributions to this warp's histogram of digit `shift`
template <bool kFirst>
__device__ __forceinline__ void hist_add4(int* whist, uint4 k4, int s, int nv, uint32_t prefix, uint32_t mask,
                                          int shift, int lane) {
  const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int bin = -1;
    if (s + j < nv && (kk[j] & mask) == prefix) bin = (int)((kk[j] >> shift) & 0xFFu);
    if (kFirst) {
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (bin >= 0 && lane == __ffs(peers) - 1) atomicAdd(&whist[bin], __popc(peers));
    } else if (bin >= 0) {
      atomicAdd(&whist[bin], 1);
    }
  }
}

__global__ void __launch_bounds__(kTopkThreads, 12)
topk_kernel(const float* __restrict__ scores, int32_t* __restrict__ idx, float* __restrict__ iscore,
            int Sq, int t0, int N, int K, int ratio, int smem_cap) {
  extern __shared__ uint4 skeys4[];
  __shared__ int s_hist[kTopkWarps][256];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_krem, s_done;
  const int t = t0 + blockIdx.x, b = blockIdx.y;
  const size_t qr = (size_t)b * Sq + blockIdx.x;     // query row
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nv = min(n_visible(t, ratio), N);
  const float* row = scores + qr * N;
  int32_t* orow = idx + qr * K;
  float* srow = iscore ? iscore + qr * K : nullptr;
  if (nv <= K) {
    for (int j = tid; j < K; j += kTopkThreads) {
      orow[j] = j < nv ? j : -1;
      if (srow) srow[j] = j < nv ? row[j] : -INFINITY;
    }
    return;
  }
  const bool in_smem = nv <= smem_cap;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const int nc = (nv + 3) >> 2;                        // 4-key chunks
  int* whist = s_hist[wid];
#pragma unroll
  for (int i = 0; i < 8; ++i) whist[lane + 32 * i] = 0;  // each warp adds to its own row only
  __syncwarp();
  if (in_smem)
    for (int c0 = 0; c0 < nc; c0 += kTopkThreads) {   // load, with the first pass's histogram
      const int c = c0 + tid;
      uint4 k4 = make_uint4(0u, 0u, 0u, 0u);
      if (c < nc) {
        k4 = row_key4(row, skeys4, false, vec, c, nv);
        skeys4[c] = k4;
      }
      hist_add4<true>(whist, k4, 4 * c, nv, 0u, 0u, 24, lane);
    }
  if (tid == 0) { s_prefix = 0u; s_mask = 0u; s_krem = K; s_done = 0; }
  __syncthreads();
  for (int shift = 24; shift >= 0 && !s_done; shift -= 8) {
    // histograms are zero here: cleared before the first pass, and by the
    // select phase of the previous one
    const uint32_t prefix = s_prefix, mask = s_mask;
    if (shift != 24 || !in_smem) {
      for (int c0 = 0; c0 < nc; c0 += kTopkThreads) {
        const int c = c0 + tid;
        const uint4 k4 = c < nc ? row_key4(row, skeys4, in_smem, vec, c, nv) : make_uint4(0u, 0u, 0u, 0u);
        if (shift == 24) hist_add4<true>(whist, k4, 4 * c, nv, prefix, mask, shift, lane);
        else hist_add4<false>(whist, k4, 4 * c, nv, prefix, mask, shift, lane);
      }
      __syncthreads();
    }
    // totals per digit
    for (int d = tid; d < 256; d += kTopkThreads) {
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
  // warp w owns the chunks [lo, hi), in index order
  const int span = ((nc + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
  const int lo = min(wid * span, nc), hi = min(lo + span, nc);
  int gt = 0, eq = 0;
  for (int c0 = lo; c0 < hi; c0 += 32) {
    const int c = c0 + lane;
    if (c < hi) {
      const uint4 k4 = row_key4(row, skeys4, in_smem, vec, c, nv);
      const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t u = kk[j] & kmask;
        const bool v = 4 * c + j < nv;
        gt += (v && u > kth) ? 1 : 0;
        eq += (v && u == kth) ? 1 : 0;
      }
    }
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  if (lane == 0) { s_hist[1][wid] = gt; s_hist[2][wid] = eq; }
  __syncthreads();
  // first output slot and first tie rank of this warp's range
  int out_pos = 0, tie_rank = 0;
  for (int w = 0; w < wid; ++w) {
    const int e = s_hist[2][w];
    out_pos += s_hist[1][w] + max(0, min(e, ties_needed - tie_rank));
    tie_rank += e;
  }
  for (int c0 = lo; c0 < hi; c0 += 32) {
    const int c = c0 + lane;
    uint32_t kk[4] = {0u, 0u, 0u, 0u};
    int n_gt = 0, n_eq = 0;
    if (c < hi) {
      const uint4 k4 = row_key4(row, skeys4, in_smem, vec, c, nv);
      kk[0] = k4.x; kk[1] = k4.y; kk[2] = k4.z; kk[3] = k4.w;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t u = kk[j] & kmask;
        const bool v = 4 * c + j < nv;
        n_gt += (v && u > kth) ? 1 : 0;
        n_eq += (v && u == kth) ? 1 : 0;
      }
    }
    // exclusive lane scan of (keys above kth, keys equal to it), 16 bits each
    // (at most 128 per step)
    const int packed = n_gt | (n_eq << 16);
    int incl = packed;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int excl = incl - packed;
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    const int gt_lo = excl & 0xFFFF, eq_lo = excl >> 16;
    int tie_r = tie_rank + eq_lo;                          // rank of this lane's first tie
    int pos = out_pos + gt_lo + max(0, min(eq_lo, ties_needed - tie_rank));
    if (c < hi) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t u = kk[j] & kmask;
        if (4 * c + j < nv) {
          const bool tie = u == kth;
          const bool take = u > kth || (tie && tie_r < ties_needed);
          tie_r += tie ? 1 : 0;
          if (take && pos < K) {
            orow[pos] = 4 * c + j;
            if (srow) srow[pos] = key_to_float(kk[j]);
            ++pos;
          }
        }
      }
    }
    const int tot_eq = total >> 16;
    out_pos += (total & 0xFFFF) + max(0, min(tot_eq, ties_needed - tie_rank));
    tie_rank += tot_eq;
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
  dim3 grid(q_rows(c), c.batch);
  kern<<<grid, kScoreThreads, smem, st>>>((const T*)iqp, (const T*)ikey, w, scores, q_rows(c), c.q_begin, N,
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
  const size_t smem = (size_t)((cap + 3) & ~3) * sizeof(uint32_t);      // whole 4-key chunks
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(q_rows(c), c.batch);
  topk_kernel<<<grid, kTopkThreads, smem, st>>>(scores, idx, iscore, q_rows(c), c.q_begin, N, c.topk, c.ratio,
                                                cap);
  note_launch();
  return cudaGetLastError();
}

}  // namespace v4
