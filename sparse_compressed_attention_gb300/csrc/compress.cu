// Compressor (learned softmax pooling of the shared latent into entries),
// window-key rotation and indexer query preparation.
//
// Compressor: "Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X
// GPUs with Primus", section "Three attention types, interleaved" (softmax
// over the group with a learnable per-position bias; CSA groups overlap) and
// section "Kernel fusions", row "Compressor pooling" (bias add, softmax over
// the window of 8 or 128, weighted reduce, all in fp32, one kernel).  Entry
// RMSNorm and the rotation at r*s follow Primus PR #930 items 1 and 2; the
// indexer-key Hadamard follows item 6e.
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace v4 {

namespace {

// One block per (entry s, batch b); 256 threads, or 512 for groups of 32
// members and more.  Thread tid works on channel vector cv = tid % ncv (8
// channels) and member slice ms = tid / ncv; it runs an online softmax over
// the members m with m % nms == ms (with PAIR, two members' loads at a time:
// for the long groups, whose slices hold many members each).  The nms
// partial states of a channel are merged in shared memory, then the block
// finishes the entry: RMSNorm, weight, RoPE at r*s (from the per-call cos/sin
// table when one is given), optional Hadamard, store.
template <typename T, bool PAIR>
__global__ void __launch_bounds__(PAIR ? 512 : 256)
compress_kernel(const T* __restrict__ ckv, const T* __restrict__ cscore,
                const float* __restrict__ ape, const float* __restrict__ norm_w,
                const float* __restrict__ inv_freq, const float2* __restrict__ cs_table, T* __restrict__ out,
                int S, int N, int dim, int R, int ratio, int overlap, float eps,
                int hadamard) {
  extern __shared__ float sm[];
  const int nthr = blockDim.x;
  const int ncv = dim / 8;
  const int nms = nthr / ncv;                // >= 1 because dim <= 2048
  float* s_m = sm;                           // [nms][dim]
  float* s_l = s_m + nms * dim;              // [nms][dim]
  float* s_a = s_l + nms * dim;              // [nms][dim]
  float* s_e = s_a + nms * dim;              // [dim] finished entry
  __shared__ float s_red[32];

  const int s = blockIdx.x;
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  const int cv = tid % ncv;
  const int ms = tid / ncv;
  const int P = 1 + overlap;
  const int G = (overlap && s >= 1) ? 2 * ratio : ratio;  // members present
  const int first_row = (overlap && s >= 1) ? 0 : overlap * ratio;

  if (ms < nms) {
    float m[8], l[8], acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) { m[k] = -INFINITY; l[k] = 0.f; acc[k] = 0.f; }
    // member mi in chronological order: ape row first_row + mi
    auto member_off = [&](int mi, size_t* off, int* row) {
      *row = first_row + mi;
      int tok, half;
      if (overlap && *row < ratio) { tok = ratio * (s - 1) + *row; half = 1; }
      else { tok = ratio * s + (*row - overlap * ratio); half = 0; }
      *off = (((size_t)b * S + tok) * P + half) * dim + cv * 8;
    };
    auto update = [&](const float* sc, const float* x, const float* a) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float lam = sc[k] + a[k];
        if (lam > m[k]) {
          float f = expf(m[k] - lam);
          l[k] = l[k] * f + 1.f;
          acc[k] = acc[k] * f + x[k];
          m[k] = lam;
        } else {
          float e = expf(lam - m[k]);
          l[k] += e;
          acc[k] += e * x[k];
        }
      }
    };
    int mi = ms;
    for (; PAIR && mi + nms < G; mi += 2 * nms) {   // two members' loads in flight
      size_t off0, off1;
      int row0, row1;
      member_off(mi, &off0, &row0);
      member_off(mi + nms, &off1, &row1);
      float sc0[8], x0[8], a0[8], sc1[8], x1[8], a1[8];
      load8(cscore + off0, sc0);
      load8(ckv + off0, x0);
      load8(ape + (size_t)row0 * dim + cv * 8, a0);
      load8(cscore + off1, sc1);
      load8(ckv + off1, x1);
      load8(ape + (size_t)row1 * dim + cv * 8, a1);
      update(sc0, x0, a0);
      update(sc1, x1, a1);
    }
    for (; mi < G; mi += nms) {
      size_t off0;
      int row0;
      member_off(mi, &off0, &row0);
      float sc0[8], x0[8], a0[8];
      load8(cscore + off0, sc0);
      load8(ckv + off0, x0);
      load8(ape + (size_t)row0 * dim + cv * 8, a0);
      update(sc0, x0, a0);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      s_m[ms * dim + cv * 8 + k] = m[k];
      s_l[ms * dim + cv * 8 + k] = l[k];
      s_a[ms * dim + cv * 8 + k] = acc[k];
    }
  }
  __syncthreads();

  // merge the member slices, accumulate the sum of squares
  float ss = 0.f;
  for (int c = tid; c < dim; c += nthr) {
    float mm = -INFINITY;
    for (int j = 0; j < nms; ++j) mm = fmaxf(mm, s_m[j * dim + c]);
    float ll = 0.f, aa = 0.f;
    for (int j = 0; j < nms; ++j) {
      float mj = s_m[j * dim + c];
      if (mj == -INFINITY) continue;
      float f = expf(mj - mm);
      ll += s_l[j * dim + c] * f;
      aa += s_a[j * dim + c] * f;
    }
    float v = aa / ll;
    s_e[c] = v;
    ss += v * v;
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) s_red[tid >> 5] = ss;
  __syncthreads();
  if (tid < 32) {
    float v = tid < nthr / 32 ? s_red[tid] : 0.f;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (tid == 0) s_red[0] = v;
  }
  __syncthreads();
  const float rinv = 1.0f / sqrtf(s_red[0] / (float)dim + eps);
  for (int c = tid; c < dim; c += nthr)
    s_e[c] = s_e[c] * rinv * (norm_w ? norm_w[c] : 1.f);
  __syncthreads();
  // RoPE on interleaved pairs of the last R channels, position r*s
  const long long pos = (long long)ratio * s;
  for (int j = tid; j < R / 2; j += nthr) {
    float cs, sn;
    if (cs_table) {
      const float2 v = cs_table[pos * (R / 2) + j];
      cs = v.x;
      sn = v.y;
    } else {
      rope_cos_sin(pos, inv_freq[j], &cs, &sn);
    }
    const int c0 = dim - R + 2 * j;
    float a = s_e[c0], bb = s_e[c0 + 1];
    rot_pair(a, bb, cs, sn);
    s_e[c0] = a;
    s_e[c0 + 1] = bb;
  }
  __syncthreads();
  if (hadamard) {
    for (int h = 1; h < dim; h <<= 1) {
      for (int i = tid; i < dim / 2; i += nthr) {
        const int lo = (i / h) * 2 * h + (i % h);
        float a = s_e[lo], bb = s_e[lo + h];
        s_e[lo] = a + bb;
        s_e[lo + h] = a - bb;
      }
      __syncthreads();
    }
    const float hs = 1.0f / sqrtf((float)dim);
    for (int c = tid; c < dim; c += nthr) s_e[c] *= hs;
    __syncthreads();
  }
  T* dst = out + ((size_t)b * N + s) * dim;
  for (int c8 = tid; c8 < ncv; c8 += nthr) store8(dst + c8 * 8, s_e + c8 * 8);
}

// Rotate every row of kv [rows, D] at its own position u = row % S (last R
// dims), writing the storage dtype.  One thread per 8-element vector.
template <typename T>
__global__ void rotate_rows_kernel(const T* __restrict__ x, const float* __restrict__ inv_freq,
                                   T* __restrict__ y, long long rows, int S, int D, int R) {
  const int nv = D / 8;
  const long long total = rows * nv;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / nv;
    const int v = (int)(i % nv);
    float e[8];
    load8(x + row * D + v * 8, e);
    const int c0 = v * 8;
    if (c0 >= D - R) {
      const long long u = row % S;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float cs, sn;
        rope_cos_sin(u, inv_freq[(c0 - (D - R)) / 2 + k], &cs, &sn);
        rot_pair(e[2 * k], e[2 * k + 1], cs, sn);
      }
    }
    store8(y + row * D + v * 8, e);
  }
}

// cos/sin of pos * inv_freq[j] for every position pos < S and pair j, one
// thread per entry: the table all position-dependent rotations read.
__global__ void rope_table_kernel(const float* __restrict__ inv_freq, float2* __restrict__ table,
                                  long long S, int half_r) {
  const long long total = S * half_r;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    float cs, sn;
    rope_cos_sin(i / half_r, inv_freq[i % half_r], &cs, &sn);
    table[i] = make_float2(cs, sn);
  }
}

// Key prep: one warp per window row u of kv (rows [0, B*S)): rotated at
// its position on the last R dims and stored in the storage dtype.
template <typename T>
__global__ void key_prep_kernel(const T* __restrict__ kv, const float2* __restrict__ cs_table,
                                T* __restrict__ kv_rot, long long kv_rows, int S, int D, int R) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long row = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5); row < kv_rows;
       row += warps) {
    const T* src = kv + row * D;
    for (int v = lane; v < D / 8; v += 32) {
      float e[8];
      load8(src + v * 8, e);
      const int c0 = v * 8;
      if (c0 >= D - R) {
        const float2* cs = cs_table + (row % S) * (R / 2) + (c0 - (D - R)) / 2;
#pragma unroll
        for (int k = 0; k < 4; ++k) rot_pair(e[2 * k], e[2 * k + 1], cs[k].x, cs[k].y);
      }
      store8(kv_rot + row * D + c0, e);
    }
  }
}

// Indexer query prep: rows of Di elements (row = (b, query row i, h) with
// Sq query rows per sequence, position t = t0 + i), RoPE at t on the last R dims, then the normalised Hadamard via butterflies: stages 1,2,4
// inside a thread's 8 elements, larger stages across the Di/8 lanes of the
// row with warp shuffles.  Requires Di/8 <= 32.
template <typename T>
__global__ void indexer_prep_kernel(const T* __restrict__ iq, const float2* __restrict__ cs_table,
                                    const float* __restrict__ inv_freq, T* __restrict__ out,
                                    long long rows, int Sq, int t0, int Hi, int Di, int R) {
  const int lanes = Di / 8;                                  // lanes per row (power of 2)
  const long long gt = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long row = gt / lanes;
  const int lane = (int)(gt % lanes);
  const bool live = row < rows;
  float e[8];
  if (live) load8(iq + row * Di + lane * 8, e);
  else {
#pragma unroll
    for (int k = 0; k < 8; ++k) e[k] = 0.f;
  }
  const int c0 = lane * 8;
  if (live && c0 >= Di - R) {
    const long long t = t0 + (row / Hi) % Sq;
    const int j0 = (c0 - (Di - R)) / 2;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float cs, sn;
      if (cs_table) {
        const float2 v = cs_table[t * (R / 2) + j0 + k];
        cs = v.x;
        sn = v.y;
      } else {
        rope_cos_sin(t, inv_freq[j0 + k], &cs, &sn);
      }
      rot_pair(e[2 * k], e[2 * k + 1], cs, sn);
    }
  }
  // in-thread butterflies (h = 1, 2, 4)
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if ((k & h) == 0) {
        float a = e[k], b = e[k + h];
        e[k] = a + b;
        e[k + h] = a - b;
      }
    }
  }
  // cross-lane butterflies (h = 8 .. Di/2)
  for (int hl = 1; hl < lanes; hl <<= 1) {
    const bool upper = (lane & hl) != 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float other = __shfl_xor_sync(0xffffffffu, e[k], hl);
      e[k] = upper ? (other - e[k]) : (e[k] + other);
    }
  }
  const float hs = 1.0f / sqrtf((float)Di);
#pragma unroll
  for (int k = 0; k < 8; ++k) e[k] *= hs;
  if (live) store8(out + row * Di + lane * 8, e);
}

// The same transform for Di = 128 with four lanes per row: a lane holds 32
// elements (chunk `lane` of 8 in each 32-element block), so five butterfly
// stages run inside the thread and only two cross lanes (a quarter of the
// shuffles of the kernel above), each load of the row's four lanes covers 64
// contiguous bytes (bf16), and each thread has 64 bytes in flight.
// With kCodes (bf16 only) the prepared row is not stored: its bf16 values are
// quantised to E4M3 by the row's absolute maximum (the rule of the
// standalone quantiser: scale = amax / 448, codes of x * (448 / amax) in fp32,
// round to nearest, saturating), and only the codes and the scale are written.
template <typename T, bool kCodes = false>
__global__ void __launch_bounds__(256)
indexer_prep_d128_kernel(const T* __restrict__ iq, const float2* __restrict__ cs_table,
                         const float* __restrict__ inv_freq, T* __restrict__ out,
                         long long rows, int Sq, int t0, int Hi, int R, uint8_t* __restrict__ codes = nullptr,
                         float* __restrict__ scales = nullptr) {
  constexpr int Di = 128, kLanes = 4, kPer = 32;
  const long long gt = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long row = gt / kLanes;
  const int lane = (int)(gt % kLanes);
  const bool live = row < rows;
  // e[8q + i] holds dim 32q + 8 lane + i: the row's four lanes read 64
  // contiguous bytes per load (bf16), and the butterflies over dim bits 1, 2,
  // 4, 32 and 64 stay in the thread
  float e[kPer];
#pragma unroll
  for (int q = 0; q < kPer / 8; ++q) {
    if (live) load8(iq + row * Di + 32 * q + 8 * lane, e + 8 * q);
    else {
#pragma unroll
      for (int k = 0; k < 8; ++k) e[8 * q + k] = 0.f;
    }
  }
  if (live) {
    const long long t = t0 + (row / Hi) % Sq;
#pragma unroll
    for (int k = 0; k < kPer / 2; ++k) {
      const int c = 32 * (k / 4) + 8 * lane + 2 * (k % 4);       // dim of e[2k]
      if (c >= Di - R) {
        const int j = (c - (Di - R)) / 2;
        float cs, sn;
        if (cs_table) {
          const float2 v = cs_table[t * (R / 2) + j];
          cs = v.x;
          sn = v.y;
        } else {
          rope_cos_sin(t, inv_freq[j], &cs, &sn);
        }
        rot_pair(e[2 * k], e[2 * k + 1], cs, sn);
      }
    }
  }
  // in-thread butterflies (element strides 1 .. 16: dim bits 1, 2, 4, 32,
  // 64): stride 1 in scalars, the others on element pairs with paired fp32
  // adds (x - y as fma(y, -1, x), exact)
#pragma unroll
  for (int k = 0; k < kPer; k += 2) {
    const float a = e[k], b = e[k + 1];
    e[k] = a + b;
    e[k + 1] = a - b;
  }
  const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
  for (int h = 2; h < kPer; h <<= 1) {
#pragma unroll
    for (int k = 0; k < kPer; k += 2) {
      if ((k & h) == 0) {
        const float2 x = make_float2(e[k], e[k + 1]), y = make_float2(e[k + h], e[k + h + 1]);
        const float2 sum = __fadd2_rn(x, y), dif = __ffma2_rn(y, neg1, x);
        e[k] = sum.x;
        e[k + 1] = sum.y;
        e[k + h] = dif.x;
        e[k + h + 1] = dif.y;
      }
    }
  }
  // cross-lane butterflies (dim bits 8, 16): the lower lane keeps a + b, the
  // upper a - b, both as fma(own, +-1, partner)
#pragma unroll
  for (int hl = 1; hl < kLanes; hl <<= 1) {
    const float sg = (lane & hl) ? -1.f : 1.f;
    const float2 sg2 = make_float2(sg, sg);
#pragma unroll
    for (int k = 0; k < kPer; k += 2) {
      const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, e[k], hl),
                                       __shfl_xor_sync(0xffffffffu, e[k + 1], hl));
      const float2 r = __ffma2_rn(make_float2(e[k], e[k + 1]), sg2, other);
      e[k] = r.x;
      e[k + 1] = r.y;
    }
  }
  const float hs = 1.0f / sqrtf((float)Di);
  const float2 hs2 = make_float2(hs, hs);
#pragma unroll
  for (int k = 0; k < kPer; k += 2) {
    const float2 r = __fmul2_rn(make_float2(e[k], e[k + 1]), hs2);
    e[k] = r.x;
    e[k + 1] = r.y;
  }
  if constexpr (kCodes) {
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      e[k] = __bfloat162float(__float2bfloat16_rn(e[k]));
      amax = fmaxf(amax, fabsf(e[k]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));     // the row's four lanes
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float inv = amax > 0.f ? 448.0f / amax : 0.f;
    if (live) {
      if (lane == 0) scales[row] = amax > 0.f ? amax / 448.0f : 0.f;
      uint32_t wv[kPer / 4];
#pragma unroll
      for (int q = 0; q < kPer / 4; ++q) {
        const __nv_fp8x2_storage_t lo =
            __nv_cvt_float2_to_fp8x2(make_float2(e[4 * q] * inv, e[4 * q + 1] * inv), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(e[4 * q + 2] * inv, e[4 * q + 3] * inv), __NV_SATFINITE, __NV_E4M3);
        wv[q] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
#pragma unroll
      for (int q = 0; q < kPer / 8; ++q)
        *reinterpret_cast<uint2*>(codes + row * Di + 32 * q + 8 * lane) = make_uint2(wv[2 * q], wv[2 * q + 1]);
    }
  } else {
    if (live) {
#pragma unroll
      for (int q = 0; q < kPer / 8; ++q) store8(out + row * Di + 32 * q + 8 * lane, e + 8 * q);
    }
  }
}

// Short groups (G <= 16 members, e.g. CSA's 8) with dim/8 a power of two in
// [16, 256]: one thread per 8 channels runs the whole online softmax over
// the members (no merge step), the entry's threads reduce the RMS by warp
// shuffles (and shared memory when the entry spans warps), rotate their own
// pairs and, for dim/8 <= 32, run the Hadamard as the query prep does (three
// stages in the thread, the rest across lanes).  Several entries per block.
template <typename T>
__global__ void __launch_bounds__(256)
compress_short_kernel(const T* __restrict__ ckv, const T* __restrict__ cscore,
                      const float* __restrict__ ape, const float* __restrict__ norm_w,
                      const float* __restrict__ inv_freq, const float2* __restrict__ cs_table,
                      T* __restrict__ out, int S, int N, int dim, int R, int ratio, int overlap, float eps,
                      int hadamard) {
  __shared__ float s_part[8];                        // per-warp partial sums of squares
  const int ncv = dim / 8;
  const int per_block = 256 / ncv;
  const int e_in = threadIdx.x / ncv, cv = threadIdx.x % ncv;
  const int s = blockIdx.x * per_block + e_in;
  const int b = blockIdx.y;
  const bool live = s < N;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int P = 1 + overlap;
  const int ss_ = live ? s : 0;
  const int G = (overlap && ss_ >= 1) ? 2 * ratio : ratio;
  const int first_row = (overlap && ss_ >= 1) ? 0 : overlap * ratio;
  float m[8], l[8], acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) { m[k] = -INFINITY; l[k] = 0.f; acc[k] = 0.f; }
  if (live) {
    for (int mi = 0; mi < G; ++mi) {
      const int row = first_row + mi;
      int tok, half;
      if (overlap && row < ratio) { tok = ratio * (ss_ - 1) + row; half = 1; }
      else { tok = ratio * ss_ + (row - overlap * ratio); half = 0; }
      const size_t off = (((size_t)b * S + tok) * P + half) * dim + cv * 8;
      float sc[8], x[8], a[8];
      load8(cscore + off, sc);
      load8(ckv + off, x);
      load8(ape + (size_t)row * dim + cv * 8, a);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float lam = sc[k] + a[k];
        if (lam > m[k]) {
          float f = expf(m[k] - lam);
          l[k] = l[k] * f + 1.f;
          acc[k] = acc[k] * f + x[k];
          m[k] = lam;
        } else {
          float e = expf(lam - m[k]);
          l[k] += e;
          acc[k] += e * x[k];
        }
      }
    }
  }
  float v[8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    v[k] = live ? acc[k] / l[k] : 0.f;
    ss += v[k] * v[k];
  }
  // sum of squares over the entry's ncv threads
  if (ncv <= 32) {
    for (int o = ncv / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  } else {
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) s_part[wid] = ss;
    __syncthreads();
    const int w0 = (e_in * ncv) >> 5, nw = ncv >> 5;
    ss = 0.f;
    for (int w = 0; w < nw; ++w) ss += s_part[w0 + w];
  }
  const float rinv = 1.0f / sqrtf(ss / (float)dim + eps);
  const int c0 = cv * 8;
#pragma unroll
  for (int k = 0; k < 8; ++k) v[k] = v[k] * rinv * (norm_w ? norm_w[c0 + k] : 1.f);
  if (c0 >= dim - R) {
    const long long pos = (long long)ratio * ss_;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = (c0 - (dim - R)) / 2 + k;
      float cs, sn;
      if (cs_table) {
        const float2 cvv = cs_table[pos * (R / 2) + j];
        cs = cvv.x;
        sn = cvv.y;
      } else {
        rope_cos_sin(pos, inv_freq[j], &cs, &sn);
      }
      rot_pair(v[2 * k], v[2 * k + 1], cs, sn);
    }
  }
  if (hadamard) {                                     // dim/8 <= 32 (checked by the launcher)
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if ((k & h) == 0) {
          const float a = v[k], d = v[k + h];
          v[k] = a + d;
          v[k + h] = a - d;
        }
      }
    }
    for (int hl = 1; hl < ncv; hl <<= 1) {
      const bool upper = (cv & hl) != 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float other = __shfl_xor_sync(0xffffffffu, v[k], hl);
        v[k] = upper ? (other - v[k]) : (v[k] + other);
      }
    }
    const float hs = 1.0f / sqrtf((float)dim);
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] *= hs;
  }
  if (live) store8(out + ((size_t)b * N + s) * dim + c0, v);
}

template <typename T>
cudaError_t compress_t(const v4_config& c, const void* ckv, const void* cscore, const float* ape,
                       const float* norm_w, const float* inv_freq, const float2* cs_table, int dim,
                       int hadamard, void* out, cudaStream_t st) {
  const int N = c.seqlen / c.ratio;
  if (N == 0) return cudaSuccess;
  const int ncv = dim / 8;
  const int G = (1 + c.overlap) * c.ratio;
  const bool pow2 = (ncv & (ncv - 1)) == 0;
  if (G <= 16 && pow2 && ncv >= 16 && ncv <= 256 && (!hadamard || ncv <= 32)) {
    const int per_block = 256 / ncv;
    dim3 grid((N + per_block - 1) / per_block, c.batch);
    compress_short_kernel<T><<<grid, 256, 0, st>>>((const T*)ckv, (const T*)cscore, ape, norm_w, inv_freq,
                                                    cs_table, (T*)out, c.seqlen, N, dim, c.rope_dim, c.ratio,
                                                    c.overlap, c.rms_eps, hadamard);
    note_launch();
    return cudaGetLastError();
  }
  int threads = G >= 32 ? 512 : 256;
  while (threads > 32 && threads / ncv < 1) threads *= 2;   // dim <= 2048: 256 threads cover it
  const int nms = threads / ncv;
  const size_t smem = (size_t)(3 * nms * dim + dim) * sizeof(float);
  auto kern = G >= 32 ? compress_kernel<T, true> : compress_kernel<T, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(N, c.batch);
  kern<<<grid, threads, smem, st>>>((const T*)ckv, (const T*)cscore, ape, norm_w, inv_freq, cs_table,
                                    (T*)out, c.seqlen, N, dim, c.rope_dim, c.ratio,
                                    c.overlap, c.rms_eps, hadamard);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compress(const v4_config& c, const void* ckv, const void* cscore,
                            const float* ape, const float* norm_w, const float* inv_freq,
                            const float2* cs_table, int dim, int hadamard, void* out, cudaStream_t st) {
  if (c.dtype == V4_BF16)
    return compress_t<bf16>(c, ckv, cscore, ape, norm_w, inv_freq, cs_table, dim, hadamard, out, st);
  return compress_t<float>(c, ckv, cscore, ape, norm_w, inv_freq, cs_table, dim, hadamard, out, st);
}

cudaError_t launch_rotate_rows(const v4_config& c, const void* kv, const float* inv_freq,
                               void* kv_rot, cudaStream_t st) {
  const long long rows = (long long)c.batch * c.seqlen;
  const long long total = rows * (c.head_dim / 8);
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  if (c.dtype == V4_BF16)
    rotate_rows_kernel<bf16><<<(int)blocks, threads, 0, st>>>(
        (const bf16*)kv, inv_freq, (bf16*)kv_rot, rows, c.seqlen, c.head_dim, c.rope_dim);
  else
    rotate_rows_kernel<float><<<(int)blocks, threads, 0, st>>>(
        (const float*)kv, inv_freq, (float*)kv_rot, rows, c.seqlen, c.head_dim, c.rope_dim);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_rope_table(const v4_config& c, const float* inv_freq, float2* table, cudaStream_t st) {
  const long long total = (long long)c.seqlen * (c.rope_dim / 2);
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  if (blocks > 152LL * 8) blocks = 152LL * 8;
  rope_table_kernel<<<(int)blocks, 256, 0, st>>>(inv_freq, table, c.seqlen, c.rope_dim / 2);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_key_prep(const v4_config& c, const void* kv, const float2* cs_table, void* kv_rot,
                            cudaStream_t st) {
  const long long kv_rows = (long long)c.batch * c.seqlen;
  const int threads = 256;
  long long blocks = (kv_rows + 7) / 8;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  if (blocks < 1) blocks = 1;
  if (c.dtype == V4_BF16)
    key_prep_kernel<bf16><<<(int)blocks, threads, 0, st>>>((const bf16*)kv, cs_table, (bf16*)kv_rot, kv_rows,
                                                            c.seqlen, c.head_dim, c.rope_dim);
  else
    key_prep_kernel<float><<<(int)blocks, threads, 0, st>>>((const float*)kv, cs_table, (float*)kv_rot, kv_rows,
                                                             c.seqlen, c.head_dim, c.rope_dim);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_indexer_prep_e4m3(const v4_config& c, const void* iq, const float2* cs_table,
                                     const float* inv_freq, uint8_t* codes, float* scales, cudaStream_t st) {
  if (c.idx_dim != 128 || c.dtype != V4_BF16) return cudaErrorInvalidValue;
  const long long rows = (long long)c.batch * q_rows(c) * c.idx_heads;
  if (rows == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (rows * 4 + threads - 1) / threads;
  indexer_prep_d128_kernel<bf16, true><<<(unsigned)blocks, threads, 0, st>>>(
      (const bf16*)iq, cs_table, inv_freq, nullptr, rows, q_rows(c), c.q_begin, c.idx_heads, c.rope_dim, codes,
      scales);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_indexer_prep(const v4_config& c, const void* iq, const float2* cs_table,
                                const float* inv_freq, void* iqp, cudaStream_t st) {
  const long long rows = (long long)c.batch * q_rows(c) * c.idx_heads;
  if (rows == 0) return cudaSuccess;
  const int threads = 256;
  const int Sq = q_rows(c), t0 = c.q_begin;
  if (c.idx_dim == 128) {
    const long long blocks = (rows * 4 + threads - 1) / threads;
    if (c.dtype == V4_BF16)
      indexer_prep_d128_kernel<bf16><<<(unsigned)blocks, threads, 0, st>>>(
          (const bf16*)iq, cs_table, inv_freq, (bf16*)iqp, rows, Sq, t0, c.idx_heads, c.rope_dim);
    else
      indexer_prep_d128_kernel<float><<<(unsigned)blocks, threads, 0, st>>>(
          (const float*)iq, cs_table, inv_freq, (float*)iqp, rows, Sq, t0, c.idx_heads, c.rope_dim);
    note_launch();
    return cudaGetLastError();
  }
  const int lanes = c.idx_dim / 8;
  const long long blocks = (rows * lanes + threads - 1) / threads;
  if (c.dtype == V4_BF16)
    indexer_prep_kernel<bf16><<<(unsigned)blocks, threads, 0, st>>>(
        (const bf16*)iq, cs_table, inv_freq, (bf16*)iqp, rows, Sq, t0, c.idx_heads, c.idx_dim, c.rope_dim);
  else
    indexer_prep_kernel<float><<<(unsigned)blocks, threads, 0, st>>>(
        (const float*)iq, cs_table, inv_freq, (float*)iqp, rows, Sq, t0, c.idx_heads, c.idx_dim,
        c.rope_dim);
  note_launch();
  return cudaGetLastError();
}

}  // namespace v4
