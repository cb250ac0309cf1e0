// Lightning-indexer scores on the 5th-generation tensor cores.
//
// Primus PR #930 item 6a (per-head weights scaled by Hi^-1/2 Di^-1/2) and
// item 4 (bf16 QK with fp32 accumulation and scoring); "Enabling
// DeepSeek-V4-Flash Training ...", section "Kernel fusions", row "Indexer
// scoring tail" (ReLU, per-head weight, head sum and causal mask in one
// kernel).
//
//   D^T[s, (t,h)] = ikey[s] . iq~[t,h]     M = 128 entries (TMEM lanes),
//                                          N = 4 queries x 64 heads, K = 128
//   I[t, s] = sum_h w'[t,h] * max(D^T[s,(t,h)], 0)   for s < n_vis(t)
//
// One CTA owns a group of 4 consecutive queries at a time (its prepared
// query rows, 64 KB, stay in shared memory; two buffers, so the next group's
// rows load while this group's tiles run) and streams the causally visible
// entry tiles through a 3-stage TMA ring.  The accumulator is
// double-buffered in TMEM (2 x 256 columns) so the epilogue of one tile (one
// thread per entry: 4 x 64 TMEM columns, ReLU, weighted head sum, masked
// store of the four scores) overlaps the MMAs of the next; the scaled head
// weights of the next group are fetched during the current one.
// Warp roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-9 epilogue (two per TMEM lane quarter, each summing two of
// the four queries: one warp per quarter could not keep up with the MMAs).  Groups are handed out round-robin, heaviest
// (largest t) first.  Flash shapes only: Hi = 64, Di = 128, bf16.
//
// The opt-in E4M3 variant (same kernel, kE4M3 = true) takes per-row scaled
// E4M3 codes of the prepared queries and of the keys: one 128-byte K-block
// per row instead of two, kind::f8f6f4 MMAs (K = 32), twice the stages.
// With x ~= code * scale per row and positive scales,
//   I[t, s] = kscale[s] * sum_h (w'[t,h] * qscale[t,h]) * max(acc[s,(t,h)], 0),
// so the query scales fold into the head weights and the key scale is one
// product after the head sum.  A quantisation kernel (one warp per row,
// absolute maximum by shuffles, scale = amax / 448, codes = satfinite e4m3
// of x * (448 / amax) rounded to nearest) makes the codes from bf16 rows.
#include <cuda.h>
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace v4 {

using namespace sm100;

namespace {

constexpr int kHi = 64, kDi = 128;
constexpr int kQG = 4;                                // queries per group
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr uint32_t kABlock = 128 * 128;               // 128 entries x 128 bytes (64 bf16 / 128 e4m3 dims)
constexpr uint32_t kBBlock = 256 * 128;               // 256 query rows x 128 bytes

// Shared-memory plan of one variant: two query-row buffers, the entry-tile
// ring, the scaled head weights and the barriers.
template <bool kE4M3>
struct Shape {
  static constexpr int kKB = kE4M3 ? 1 : 2;           // 128-byte K-blocks per row (Di = 128)
  static constexpr int kStages = kE4M3 ? 8 : 3;
  static constexpr uint32_t kAStage = kKB * kABlock;
  static constexpr uint32_t OFF_B = 0;
  static constexpr uint32_t OFF_A = 2 * kKB * kBBlock;
  static constexpr uint32_t OFF_W = OFF_A + kStages * kAStage;   // w' [2][4][64] fp32
  static constexpr uint32_t OFF_CTL = OFF_W + 2 * kQG * kHi * 4;
};

template <int kStages>
struct Ctl {
  uint64_t a_full[kStages], a_empty[kStages];
  uint64_t b_full[2], b_empty[2];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t fin;
  uint32_t tmem_base;
  int abort;
};
template <bool kE4M3>
constexpr uint32_t smem_bytes() {
  return Shape<kE4M3>::OFF_CTL + sizeof(Ctl<Shape<kE4M3>::kStages>);
}
static_assert(smem_bytes<false>() <= 232448 && smem_bytes<true>() <= 232448, "shared memory budget");

struct Params {
  const float* w;          // [B,Sq,64] unscaled weights
  const float* qscale;     // [B,Sq,64] query-row scales (E4M3 only)
  const float* kscale;     // [B,N] key-row scales (E4M3 only)
  float* scores;           // [B,Sq,N]
  int* status;
  int B, Sq, t0, N, ratio; // Sq query rows per sequence at positions t0 .. t0+Sq-1
  float wscale;
};

// (a0, a1) += (w0 * max(x0, 0), w1 * max(x1, 0)): one paired fp32 FMA
// (fma.rn.f32x2, two round-to-nearest FMAs) after the two ReLUs.
__device__ __forceinline__ void fma2_relu(float& a0, float& a1, float w0, float w1, float x0, float x1) {
  const float r0 = fmaxf(x0, 0.f), r1 = fmaxf(x1, 0.f);
  asm("{\n\t.reg .b64 wv, rv, av;\n\t"
      "mov.b64 wv, {%2, %3};\n\tmov.b64 rv, {%4, %5};\n\tmov.b64 av, {%0, %1};\n\t"
      "fma.rn.f32x2 av, wv, rv, av;\n\tmov.b64 {%0, %1}, av;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(w0), "f"(w1), "f"(r0), "f"(r1));
}

// Group gi: batch b, first query row r0 of its kQG rows (positions p.t0 + r0 ..),
// entry tiles of its last query.
__device__ __forceinline__ void group_of(int gi, const Params& p, int groups_per_b, int& b, int& r0,
                                         int& tiles) {
  b = gi % p.B;
  const int grp = groups_per_b - 1 - gi / p.B;
  r0 = grp * kQG;
  const int tmax = p.t0 + min(r0 + kQG - 1, p.Sq - 1);
  const int nv = min((tmax + 1) / p.ratio, p.N);
  tiles = (nv + 127) / 128;
}

template <bool kE4M3>
__global__ void __launch_bounds__(kThreads, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const Params p) {
  using Sh = Shape<kE4M3>;
  constexpr int kStages = Sh::kStages, kKB = Sh::kKB;
  constexpr uint32_t kAStage = Sh::kAStage, OFF_A = Sh::OFF_A, OFF_B = Sh::OFF_B;
  constexpr int kXStep = kE4M3 ? 128 : 64;              // elements per 128-byte K-block
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctl<kStages>* c = reinterpret_cast<Ctl<kStages>*>(smem + Sh::OFF_CTL);
  float* s_w = reinterpret_cast<float*>(smem + Sh::OFF_W);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) set_status(p.status, V4_ERR_UNSUPPORTED);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&c->a_full[i], 1); mbar_init(&c->a_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&c->b_full[i], 1); mbar_init(&c->b_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&c->acc_full[i], 1); mbar_init(&c->acc_empty[i], kEpiThreads); }
    mbar_init(&c->fin, 1);
    c->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_q);
    prefetch_tmap(&map_k);
  }
  if (warp == 1) {
    tmem_alloc(&c->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;
  const int groups_per_b = (p.Sq + kQG - 1) / kQG;
  const int total = p.B * groups_per_b;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int gq = 0, st = 0, use = 0;
      bool ok = true;
      for (int gi = blockIdx.x; gi < total && ok; gi += gridDim.x) {
        int b, r0, tiles;
        group_of(gi, p, groups_per_b, b, r0, tiles);
        if (tiles == 0) continue;
        const int bb = gq & 1;
        if (gq >= 2) ok = mbar_wait(&c->b_empty[bb], ((gq >> 1) - 1) & 1, &c->abort, p.status);
        if (!ok) break;
        mbar_expect_tx(&c->b_full[bb], kKB * kBBlock);
        for (int kb = 0; kb < kKB; ++kb)
          tma_load_2d(smem + OFF_B + (kKB * bb + kb) * kBBlock, &map_q, kXStep * kb, (b * p.Sq + r0) * kHi,
                      &c->b_full[bb]);
        for (int j = 0; j < tiles && ok; ++j) {
          if (use >= kStages) ok = mbar_wait(&c->a_empty[st], ((use / kStages) - 1) & 1, &c->abort, p.status);
          if (!ok) break;
          mbar_expect_tx(&c->a_full[st], kAStage);
          for (int kb = 0; kb < kKB; ++kb)
            tma_load_2d(smem + OFF_A + st * kAStage + kb * kABlock, &map_k, kXStep * kb, b * p.N + 128 * j,
                        &c->a_full[st]);
          ++use;
          st = (st + 1) % kStages;
        }
        ++gq;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = kE4M3 ? idesc_e4m3_f32(128, 256) : idesc_bf16_f32(128, 256, 0, 0);
      const uint64_t dA0 = smem_desc(smem_u32(smem + OFF_A), 16, 1024, kLayoutSW128);
      const uint64_t dB0 = smem_desc(smem_u32(smem + OFF_B), 16, 1024, kLayoutSW128);
      int gq = 0, st = 0, use = 0, tile_ct = 0;
      bool ok = true;
      for (int gi = blockIdx.x; gi < total && ok; gi += gridDim.x) {
        int b, r0, tiles;
        group_of(gi, p, groups_per_b, b, r0, tiles);
        if (tiles == 0) continue;
        const int bb = gq & 1;
        ok = mbar_wait(&c->b_full[bb], (gq >> 1) & 1, &c->abort, p.status);
        const uint64_t dB = dB0 + (uint64_t)((kKB * bb * kBBlock) >> 4);
        for (int j = 0; j < tiles && ok; ++j) {
          const int ab = tile_ct & 1;
          ok = mbar_wait(&c->a_full[st], (use / kStages) & 1, &c->abort, p.status);
          if (ok && tile_ct >= 2) ok = mbar_wait(&c->acc_empty[ab], ((tile_ct >> 1) - 1) & 1, &c->abort, p.status);
          tc_fence_after();
          if (!ok) break;
          const uint32_t d = tmem + 256 * ab;
          const uint64_t dA = dA0 + (uint64_t)((st * kAStage) >> 4);
#pragma unroll
          for (int kb = 0; kb < kKB; ++kb) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {           // 32 bytes of K per instruction
              const uint64_t da = dA + (uint64_t)((kb * kABlock + 32 * ks) >> 4);
              const uint64_t db = dB + (uint64_t)((kb * kBBlock + 32 * ks) >> 4);
              if constexpr (kE4M3)
                umma_e4m3_ss(d, da, db, idesc, (kb | ks) != 0);
              else
                umma_f16_ss(d, da, db, idesc, (kb | ks) != 0);
            }
          }
          umma_commit(&c->a_empty[st]);
          umma_commit(&c->acc_full[ab]);
          ++use;
          st = (st + 1) % kStages;
          ++tile_ct;
        }
        umma_commit(&c->b_empty[bb]);
        ++gq;
      }
      umma_commit(&c->fin);
      mbar_wait(&c->fin, 0, &c->abort, p.status, 200000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ts = threadIdx.x - 64;          // 0..255
    const int quarter = warp & 3;
    const int q0 = 2 * ((warp - 2) >> 2);     // this warp's queries q0, q0+1
    const int krow = 32 * quarter + lane;
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    // scaled weight ts of a group (query ts/64, head ts%64), one group ahead
    float pf_w = 0.f;
    int pf_gi = -1;
    auto fetch_w = [&](int g) -> float {
      int bg = 0, tg = 0, tl = 0;
      if (g >= total) return 0.f;
      group_of(g, p, groups_per_b, bg, tg, tl);
      const int r = tg + ts / kHi;             // query row
      if (r >= p.Sq) return 0.f;
      const size_t wi = ((size_t)bg * p.Sq + r) * kHi + (ts % kHi);
      if constexpr (kE4M3)
        return p.w[wi] * p.wscale * p.qscale[wi];
      else
        return p.w[wi] * p.wscale;
    };
    pf_w = fetch_w(blockIdx.x);
    pf_gi = blockIdx.x;
    int gq = 0, tile_ct = 0;
    for (int gi = blockIdx.x; gi < total; gi += gridDim.x) {
      int b, r0, tiles;
      group_of(gi, p, groups_per_b, b, r0, tiles);
      if (tiles == 0) continue;
      const float wv = pf_gi == gi ? pf_w : fetch_w(gi);
      // buffer gq & 1 was last read for group gq-2, which every thread has
      // finished before the barrier of group gq-1
      float* sw = s_w + (gq & 1) * kQG * kHi;
      sw[ts] = wv;
      named_bar_sync(1, kEpiThreads);
      pf_w = fetch_w(gi + gridDim.x);
      pf_gi = gi + gridDim.x;
      for (int j = 0; j < tiles; ++j) {
        const int ab = tile_ct & 1;
        const int s = 128 * j + krow;
        float ksc = 1.f;                         // key-row scale, loaded before the wait
        if constexpr (kE4M3) ksc = s < p.N ? p.kscale[(size_t)b * p.N + s] : 0.f;
        mbar_wait(&c->acc_full[ab], (tile_ct >> 1) & 1, &c->abort, p.status);
        tc_fence_after();
        float sc[2];
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const int q = q0 + qq;
          const float* wq = sw + q * kHi;
          // both halves of the query's 64 heads in one wait; four partial
          // sums (heads h mod 4), two of them per paired fp32 FMA
          float v[64];
          if (!V4_BOUND(256 * ab + 64 * q + 64 <= 512, p.status)) break;   // accumulator columns
          tmem_ld32(tmem + lane_base + 256 * ab + 64 * q, v);
          tmem_ld32(tmem + lane_base + 256 * ab + 64 * q + 32, v + 32);
          tmem_wait_ld();
          float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int h = 0; h < kHi; h += 2)
            fma2_relu(a[h & 3], a[(h & 3) + 1], wq[h], wq[h + 1], v[h], v[h + 1]);
          sc[qq] = (a[0] + a[1]) + (a[2] + a[3]);
        }
        tc_fence_before();
        mbar_arrive(&c->acc_empty[ab]);
        if constexpr (kE4M3) {
          sc[0] *= ksc;
          sc[1] *= ksc;
        }
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const int r = r0 + q0 + qq;            // query row, position p.t0 + r
          if (r < p.Sq && s < min((p.t0 + r + 1) / p.ratio, p.N) && V4_BOUND(b < p.B && s >= 0, p.status))
            p.scores[((size_t)b * p.Sq + r) * p.N + s] = sc[qq];
        }
        ++tile_ct;
      }
      ++gq;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool indexer_tc_supported(const v4_config& c) {
  return c.dtype == V4_BF16 && c.idx_heads == kHi && c.idx_dim == kDi && c.ratio >= 1;
}

bool indexer_e4m3_supported(const v4_config& c) { return indexer_tc_supported(c); }

template <bool kE4M3>
static cudaError_t launch_scores(const v4_config& cfg, const CUtensorMap& mq, const CUtensorMap& mk,
                                 const Params& prm, cudaStream_t st) {
  const uint32_t bytes = smem_bytes<kE4M3>();
  cudaError_t err = cudaFuncSetAttribute(indexer_tc_kernel<kE4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
  if (err != cudaSuccess) return err;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int total = cfg.batch * ((q_rows(cfg) + kQG - 1) / kQG);
  const int grid = total < sms ? total : sms;
  indexer_tc_kernel<kE4M3><<<grid, kThreads, bytes, st>>>(mq, mk, prm);
  note_launch();
  return cudaGetLastError();
}

static Params make_params(const v4_config& cfg, const float* w, float* scores, int* status) {
  Params prm;
  prm.w = w;
  prm.qscale = nullptr;
  prm.kscale = nullptr;
  prm.scores = scores;
  prm.status = status;
  prm.B = cfg.batch;
  prm.Sq = q_rows(cfg);
  prm.t0 = cfg.q_begin;
  prm.N = cfg.seqlen / cfg.ratio;
  prm.ratio = cfg.ratio;
  prm.wscale = 1.0f / sqrtf((float)kHi) / sqrtf((float)kDi);
  return prm;
}

cudaError_t launch_indexer_scores_tc(const v4_config& cfg, const void* iqp, const void* ikey, const float* w,
                                     float* scores, int* status, cudaStream_t st) {
  const int B = cfg.batch, S = cfg.seqlen;
  const int N = S / cfg.ratio;
  if (N == 0) return cudaSuccess;
  CUtensorMap mq, mk;
  int e = 0;
  e |= make_tmap_bf16_2d(&mq, iqp, kDi, (uint64_t)B * q_rows(cfg) * kHi, 64, 256, true);
  e |= make_tmap_bf16_2d(&mk, ikey, kDi, (uint64_t)B * N, 64, 128, true);
  if (e) return cudaErrorInvalidValue;
  return launch_scores<false>(cfg, mq, mk, make_params(cfg, w, scores, status), st);
}

cudaError_t launch_indexer_scores_e4m3(const v4_config& cfg, const uint8_t* qc, const float* qs, const uint8_t* kc,
                                       const float* ks, const float* w, float* scores, int* status,
                                       cudaStream_t st) {
  const int B = cfg.batch, S = cfg.seqlen;
  const int N = S / cfg.ratio;
  if (N == 0) return cudaSuccess;
  CUtensorMap mq, mk;
  int e = 0;
  e |= make_tmap_u8_2d(&mq, qc, kDi, (uint64_t)B * q_rows(cfg) * kHi, 128, 256, true);
  e |= make_tmap_u8_2d(&mk, kc, kDi, (uint64_t)B * N, 128, 128, true);
  if (e) return cudaErrorInvalidValue;
  Params prm = make_params(cfg, w, scores, status);
  prm.qscale = qs;
  prm.kscale = ks;
  return launch_scores<true>(cfg, mq, mk, prm, st);
}

// ---------------------------------------------------------------------------
// E4M3 quantisation of bf16 rows: one warp per row, lane l holds the 4-value
// chunks l, l + 32, ... (dim / 128 of them); absolute maximum by shuffles.
// ---------------------------------------------------------------------------
template <int kChunks>
__global__ void __launch_bounds__(256)
quant_e4m3_kernel(const bf16* __restrict__ x, long long rows, uint8_t* __restrict__ codes,
                  float* __restrict__ scales) {
  constexpr int dim = 128 * kChunks;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    const bf16* xr = x + r * dim;
    float v[4 * kChunks];
    float amax = 0.f;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const uint2 u = *reinterpret_cast<const uint2*>(xr + 4 * (32 * c + lane));
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
      const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
      v[4 * c] = a.x;
      v[4 * c + 1] = a.y;
      v[4 * c + 2] = b.x;
      v[4 * c + 3] = b.y;
#pragma unroll
      for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(v[4 * c + i]));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float inv = amax > 0.f ? 448.0f / amax : 0.f;
    if (lane == 0) scales[r] = amax > 0.f ? amax / 448.0f : 0.f;
    uint8_t* cr = codes + r * dim;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const __nv_fp8x2_storage_t lo =
          __nv_cvt_float2_to_fp8x2(make_float2(v[4 * c] * inv, v[4 * c + 1] * inv), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi =
          __nv_cvt_float2_to_fp8x2(make_float2(v[4 * c + 2] * inv, v[4 * c + 3] * inv), __NV_SATFINITE, __NV_E4M3);
      *reinterpret_cast<uint32_t*>(cr + 4 * (32 * c + lane)) = (uint32_t)lo | ((uint32_t)hi << 16);
    }
  }
}

cudaError_t launch_quant_e4m3(const void* x, long long rows, int dim, uint8_t* codes, float* scales,
                              cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (rows + 7) / 8;
  const int grid = (int)(want < 8LL * sms ? want : 8LL * sms);
  const bf16* xb = (const bf16*)x;
  switch (dim / 128) {
    case 1: quant_e4m3_kernel<1><<<grid, 256, 0, st>>>(xb, rows, codes, scales); break;
    case 2: quant_e4m3_kernel<2><<<grid, 256, 0, st>>>(xb, rows, codes, scales); break;
    case 4: quant_e4m3_kernel<4><<<grid, 256, 0, st>>>(xb, rows, codes, scales); break;
    case 8: quant_e4m3_kernel<8><<<grid, 256, 0, st>>>(xb, rows, codes, scales); break;
    default: return cudaErrorInvalidValue;
  }
  note_launch();
  return cudaGetLastError();
}

}  // namespace v4
