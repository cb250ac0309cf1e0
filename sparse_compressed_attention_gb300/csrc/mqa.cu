// Sparse / dense multi-query attention on CUDA cores (any shape, fp32 or
// bf16 storage).  This is the kernel of the fp32 mode and of shapes the
// tensor-core kernel does not cover.
//
// "Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X GPUs with
// Primus", sections "The DeepSeek-V4-Flash architecture" (all query heads
// read one latent that is both key and value), "Three attention types,
// interleaved" (selected or all entries plus a 128-token window) and "Kernel
// fusions", row "SWA / CSA / HCA attention" (window and sink folded into one
// softmax); Primus PR #930 item 1 (scale D^-1/2) and item 3 (output rotated
// at -t before the output projection).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace v4 {

namespace {

constexpr int kHG = 8;        // heads per block (one warp per head)
constexpr int kKT = 32;       // keys per tile (one lane per key)
constexpr int kMqaThreads = kHG * 32;

struct KeySet {
  int ne;        // entry slots (K with a selection, n_vis without)
  int lo, nw;    // window tokens [lo, lo + nw)
};

// Block per (query t, head group, batch).  Warp h owns head h0 + h: it
// scores a tile of 32 keys (lane j <- key j), updates the running max and
// denominator, and accumulates p * key into its D-wide output, each lane
// owning channels lane, lane+32, ...
template <typename T>
__global__ void __launch_bounds__(kMqaThreads)
mqa_simt_kernel(const T* __restrict__ q, const T* __restrict__ kv_rot, const T* __restrict__ ent,
                const int32_t* __restrict__ idx, const float* __restrict__ sink,
                const float* __restrict__ inv_freq, T* __restrict__ o, float* __restrict__ lse,
                int* __restrict__ status, const int* __restrict__ list, int S, int Sq, int t0, int H, int D,
                int R, int N, int ratio, int window, int K, float scale) {
  extern __shared__ float sm[];
  const int ldk = D + 1;                      // padded key rows: conflict-free columns
  float* s_q = sm;                            // [kHG][D] rotated query rows
  float* s_k = s_q + kHG * D;                 // [kKT][D+1]
  float* s_p = s_k + kKT * ldk;               // [kHG][kKT]
  __shared__ const T* s_ptr[kKT];
  __shared__ float s_cs[2][512];

  const int h0 = blockIdx.y * kHG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = h0 + warp;
  const bool head_live = h < H;
  // without a list: query row blockIdx.x of batch blockIdx.z; with a list:
  // the listed query rows, strided over blockIdx.x.  Query row r of batch b
  // is position t = t0 + r; q, o, lse and idx are indexed by query row.
  for (int item = blockIdx.x;; item += gridDim.x) {
  int t, b, r;
  if (list != nullptr) {
    if (item >= list[0]) break;
    const int br = list[1 + item];
    b = br / Sq;
    r = br % Sq;
  } else {
    if (item >= Sq) break;
    r = item;
    b = blockIdx.z;
  }
  t = t0 + r;
  const size_t qrow = (size_t)b * Sq + r;
  __syncthreads();

  // RoPE angles of position t (shared by all heads)
  for (int j = threadIdx.x; j < R / 2; j += kMqaThreads) {
    float cs, sn;
    rope_cos_sin(t, inv_freq[j], &cs, &sn);
    s_cs[0][j] = cs;
    s_cs[1][j] = sn;
  }
  __syncthreads();
  // rotated queries of the group
  for (int i = threadIdx.x; i < kHG * D; i += kMqaThreads) {
    const int hh = h0 + i / D, c = i % D;
    float v = 0.f;
    if (hh < H) {
      const T* qr = q + (qrow * H + hh) * D;
      v = to_f(qr[c]);
      if (c >= D - R) {
        const int j = (c - (D - R)) >> 1;
        const float other = to_f(qr[c ^ 1]);
        v = (c & 1) ? (other * s_cs[1][j] + v * s_cs[0][j]) : (v * s_cs[0][j] - other * s_cs[1][j]);
      }
    }
    s_q[i] = v;
  }

  KeySet ks;
  const int nv = ratio > 0 ? min(n_visible(t, ratio), N) : 0;
  ks.ne = ratio > 0 ? (K > 0 ? K : nv) : 0;
  if (window == 0) { ks.lo = t + 1; ks.nw = 0; }
  else if (window < 0) { ks.lo = 0; ks.nw = t + 1; }
  else { ks.lo = max(0, t - window + 1); ks.nw = t + 1 - ks.lo; }
  const int nk = ks.ne + ks.nw;

  float m = -INFINITY, l = 0.f;
  const bool has_sink = sink != nullptr && head_live && sink[h] > -INFINITY;
  if (has_sink) { m = sink[h]; l = 1.f; }
  float acc[32];                              // D / 32 <= 32 channels per lane
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  const int per_lane = D / 32;

  for (int k0 = 0; k0 < nk; k0 += kKT) {
    __syncthreads();
    if (threadIdx.x < kKT) {
      const int j = k0 + threadIdx.x;
      const T* p = nullptr;
      if (j < ks.ne) {
        int s = j;
        if (K > 0) {
          s = idx[qrow * K + j];
          if (s < -1 || s >= nv) { set_status(status, kStatusBadIndex); s = -1; }
        }
        if (s >= 0) p = ent + ((size_t)b * N + s) * D;
      } else if (j < nk) {
        p = kv_rot + ((size_t)b * S + ks.lo + (j - ks.ne)) * D;
      }
      s_ptr[threadIdx.x] = p;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kKT * (D / 8); i += kMqaThreads) {
      const int j = i / (D / 8), c8 = (i % (D / 8)) * 8;
      float v[8];
      const T* p = s_ptr[j];
      if (p) load8(p + c8, v);
      else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) s_k[j * ldk + c8 + e] = v[e];
    }
    __syncthreads();
    // logits: lane = key
    float lg = -INFINITY;
    if (head_live && s_ptr[lane] != nullptr) {
      const float* qh = s_q + warp * D;
      const float* kr = s_k + lane * ldk;
      float d = 0.f;
      for (int c = 0; c < D; ++c) d = fmaf(qh[c], kr[c], d);
      lg = d * scale;
    }
    float tmax = lg;
    for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float mnew = fmaxf(m, tmax);
    float p = 0.f, alpha = 1.f;
    if (mnew > -INFINITY) {
      p = (lg > -INFINITY) ? expf(lg - mnew) : 0.f;
      alpha = (m > -INFINITY) ? expf(m - mnew) : 0.f;
    }
    float psum = p;
    for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    l = l * alpha + psum;
    m = mnew;
    s_p[warp * kKT + lane] = p;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i < per_lane) {
        const int c = lane + 32 * i;
        float a = acc[i] * alpha;
        for (int j = 0; j < kKT; ++j) a = fmaf(s_p[warp * kKT + j], s_k[j * ldk + c], a);
        acc[i] = a;
      }
    }
  }

  if (head_live) {
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
  T* orow = o + (qrow * H + h) * D;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (i < per_lane) {
      const int c = lane + 32 * i;
      float v = acc[i] * inv_l;
      // de-rotation at -t: the pair partner of channel c sits on lane ^ 1
      const float other = __shfl_xor_sync(0xffffffffu, v, 1);
      if (c >= D - R) {
        const int j = (c - (D - R)) >> 1;
        const float cs = s_cs[0][j], sn = -s_cs[1][j];
        v = (c & 1) ? (other * sn + v * cs) : (v * cs - other * sn);
      }
      from_f(orow + c, v);
    }
  }
  if (lse && lane == 0) lse[qrow * H + h] = l > 0.f ? m + logf(l) : -INFINITY;
  }
  }
}

template <typename T>
cudaError_t mqa_t(const v4_config& c, const void* q, const void* kv_rot, const void* ent,
                  const int32_t* idx, const float* sink, const float* inv_freq, void* o,
                  float* lse, int* status, const int* list, cudaStream_t st) {
  const int D = c.head_dim;
  const size_t smem = (size_t)(kHG * D + kKT * (D + 1) + kHG * kKT) * sizeof(float);
  auto kern = mqa_simt_kernel<T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int N = c.ratio > 0 ? c.seqlen / c.ratio : 0;
  const float scale = c.softmax_scale > 0.f ? c.softmax_scale : 1.0f / sqrtf((float)D);
  dim3 grid(q_rows(c), (c.n_heads + kHG - 1) / kHG, c.batch);
  if (list != nullptr) grid = dim3(256, (c.n_heads + kHG - 1) / kHG, 1);
  kern<<<grid, kMqaThreads, smem, st>>>((const T*)q, (const T*)kv_rot, (const T*)ent, idx, sink,
                                        inv_freq, (T*)o, lse, status, list, c.seqlen, q_rows(c), c.q_begin,
                                        c.n_heads, D, c.rope_dim, N, c.ratio, c.window, c.topk, scale);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mqa_simt(const v4_config& c, const void* q, const void* kv_rot,
                            const void* ent, const int32_t* idx, const float* sink,
                            const float* inv_freq, void* o, float* lse, int* status,
                            const int* list, cudaStream_t st) {
  if (c.dtype == V4_BF16)
    return mqa_t<bf16>(c, q, kv_rot, ent, idx, sink, inv_freq, o, lse, status, list, st);
  return mqa_t<float>(c, q, kv_rot, ent, idx, sink, inv_freq, o, lse, status, list, st);
}

}  // namespace v4
