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
#include <cuda.h>
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
constexpr int kStages = 3;
constexpr uint32_t kABlock = 128 * 128;               // 128 entries x 64 dims x 2 B
constexpr uint32_t kAStage = 2 * kABlock;             // both K-blocks of a tile
constexpr uint32_t kBBlock = 256 * 128;               // 256 rows x 64 dims x 2 B
constexpr uint32_t OFF_B = 0;                         // 2 buffers x 2 K-blocks: 131072
constexpr uint32_t OFF_A = 4 * kBBlock;               // stages: 3 x 32768
constexpr uint32_t OFF_W = OFF_A + kStages * kAStage; // 229376: w' [2][4][64] fp32
constexpr uint32_t OFF_CTL = OFF_W + 2 * kQG * kHi * 4;   // 231424

struct Ctl {
  uint64_t a_full[kStages], a_empty[kStages];
  uint64_t b_full[2], b_empty[2];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t fin;
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t kSmemBytes = OFF_CTL + sizeof(Ctl);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  const float* w;          // [B,S,64] unscaled weights
  float* scores;           // [B,S,N]
  int* status;
  int B, S, N, ratio;
  float wscale;
};

__device__ __forceinline__ void group_of(int gi, const Params& p, int groups_per_b, int& b, int& t0,
                                         int& tiles) {
  b = gi % p.B;
  const int grp = groups_per_b - 1 - gi / p.B;
  t0 = grp * kQG;
  const int tmax = min(t0 + kQG - 1, p.S - 1);
  const int nv = min((tmax + 1) / p.ratio, p.N);
  tiles = (nv + 127) / 128;
}

__global__ void __launch_bounds__(kThreads, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctl* c = reinterpret_cast<Ctl*>(smem + OFF_CTL);
  float* s_w = reinterpret_cast<float*>(smem + OFF_W);
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
  const int groups_per_b = (p.S + kQG - 1) / kQG;
  const int total = p.B * groups_per_b;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int gq = 0, st = 0, use = 0;
      bool ok = true;
      for (int gi = blockIdx.x; gi < total && ok; gi += gridDim.x) {
        int b, t0, tiles;
        group_of(gi, p, groups_per_b, b, t0, tiles);
        if (tiles == 0) continue;
        const int bb = gq & 1;
        if (gq >= 2) ok = mbar_wait(&c->b_empty[bb], ((gq >> 1) - 1) & 1, &c->abort, p.status);
        if (!ok) break;
        mbar_expect_tx(&c->b_full[bb], 2 * kBBlock);
        for (int kb = 0; kb < 2; ++kb)
          tma_load_2d(smem + OFF_B + (2 * bb + kb) * kBBlock, &map_q, 64 * kb, (b * p.S + t0) * kHi,
                      &c->b_full[bb]);
        for (int j = 0; j < tiles && ok; ++j) {
          if (use >= kStages) ok = mbar_wait(&c->a_empty[st], ((use / kStages) - 1) & 1, &c->abort, p.status);
          if (!ok) break;
          mbar_expect_tx(&c->a_full[st], kAStage);
          for (int kb = 0; kb < 2; ++kb)
            tma_load_2d(smem + OFF_A + st * kAStage + kb * kABlock, &map_k, 64 * kb, b * p.N + 128 * j,
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
      const uint32_t idesc = idesc_bf16_f32(128, 256, 0, 0);
      const uint64_t dA0 = smem_desc(smem_u32(smem + OFF_A), 16, 1024, kLayoutSW128);
      const uint64_t dB0 = smem_desc(smem_u32(smem + OFF_B), 16, 1024, kLayoutSW128);
      int gq = 0, st = 0, use = 0, tile_ct = 0;
      bool ok = true;
      for (int gi = blockIdx.x; gi < total && ok; gi += gridDim.x) {
        int b, t0, tiles;
        group_of(gi, p, groups_per_b, b, t0, tiles);
        if (tiles == 0) continue;
        const int bb = gq & 1;
        ok = mbar_wait(&c->b_full[bb], (gq >> 1) & 1, &c->abort, p.status);
        const uint64_t dB = dB0 + (uint64_t)((2 * bb * kBBlock) >> 4);
        for (int j = 0; j < tiles && ok; ++j) {
          const int ab = tile_ct & 1;
          ok = mbar_wait(&c->a_full[st], (use / kStages) & 1, &c->abort, p.status);
          if (ok && tile_ct >= 2) ok = mbar_wait(&c->acc_empty[ab], ((tile_ct >> 1) - 1) & 1, &c->abort, p.status);
          tc_fence_after();
          if (!ok) break;
          const uint32_t d = tmem + 256 * ab;
          const uint64_t dA = dA0 + (uint64_t)((st * kAStage) >> 4);
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_f16_ss(d, dA + (uint64_t)((kb * kABlock + 32 * ks) >> 4),
                          dB + (uint64_t)((kb * kBBlock + 32 * ks) >> 4), idesc, (kb | ks) != 0);
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
      const int t = tg + ts / kHi;
      return t < p.S ? p.w[((size_t)bg * p.S + t) * kHi + (ts % kHi)] * p.wscale : 0.f;
    };
    pf_w = fetch_w(blockIdx.x);
    pf_gi = blockIdx.x;
    int gq = 0, tile_ct = 0;
    for (int gi = blockIdx.x; gi < total; gi += gridDim.x) {
      int b, t0, tiles;
      group_of(gi, p, groups_per_b, b, t0, tiles);
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
        mbar_wait(&c->acc_full[ab], (tile_ct >> 1) & 1, &c->abort, p.status);
        tc_fence_after();
        const int s = 128 * j + krow;
        float sc[2];
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const int q = q0 + qq;
          const float* wq = sw + q * kHi;
          float acc = 0.f;
#pragma unroll
          for (int half = 0; half < 2; ++half) {       // heads in order 0..63
            float v[32];
            tmem_ld32(tmem + lane_base + 256 * ab + 64 * q + 32 * half, v);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 32; ++h) acc = fmaf(wq[32 * half + h], fmaxf(v[h], 0.f), acc);
          }
          sc[qq] = acc;
        }
        tc_fence_before();
        mbar_arrive(&c->acc_empty[ab]);
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const int t = t0 + q0 + qq;
          if (t < p.S && s < min((t + 1) / p.ratio, p.N)) p.scores[((size_t)b * p.S + t) * p.N + s] = sc[qq];
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

cudaError_t launch_indexer_scores_tc(const v4_config& cfg, const void* iqp, const void* ikey, const float* w,
                                     float* scores, int* status, cudaStream_t st) {
  const int B = cfg.batch, S = cfg.seqlen;
  const int N = S / cfg.ratio;
  if (N == 0) return cudaSuccess;
  CUtensorMap mq, mk;
  int e = 0;
  e |= make_tmap_bf16_2d(&mq, iqp, kDi, (uint64_t)B * S * kHi, 64, 256, true);
  e |= make_tmap_bf16_2d(&mk, ikey, kDi, (uint64_t)B * N, 64, 128, true);
  if (e) return cudaErrorInvalidValue;
  Params prm;
  prm.w = w;
  prm.scores = scores;
  prm.status = status;
  prm.B = B;
  prm.S = S;
  prm.N = N;
  prm.ratio = cfg.ratio;
  prm.wscale = 1.0f / sqrtf((float)kHi) / sqrtf((float)kDi);
  cudaError_t err = cudaFuncSetAttribute(indexer_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int total = B * ((S + kQG - 1) / kQG);
  const int grid = total < sms ? total : sms;
  indexer_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mq, mk, prm);
  note_launch();
  return cudaGetLastError();
}

}  // namespace v4
