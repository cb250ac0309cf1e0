// Grouped low-rank output projection on the 5th-generation tensor cores.
//
// "Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X GPUs with
// Primus", section "The DeepSeek-V4-Flash architecture": the 64 x 512 head
// output projects back down in 8 groups, each through a 1024-d bottleneck.
// Group g holds heads g*H/G .. (g+1)*H/G - 1 concatenated along D, so for a
// token its group input is Kg = (H/G)*D contiguous elements of o.
//
//   y[t, g*N + n] = sum_k o[t, g*Kg + k] * wo_a[g, k, n]
//
// Tile: 128 tokens x 256 outputs of one group, K streamed in 64-wide blocks
// through a 4-stage TMA ring: A = 128 token rows x 64 (K-major, 128-byte
// swizzle), B = 64 K-rows x 256 outputs read straight from wo_a's [K][N]
// layout (MN-major, four 64-column blocks).  tcgen05 MMAs (M=128, N=256,
// K=16) accumulate in TMEM, double-buffered (2 x 256 columns) so the
// epilogue of one tile (one thread per token row: fp32 -> bf16, 16-byte
// stores) overlaps the next tile's MMAs.  Persistent CTAs walk the tiles.
//
// The same kernel runs the query projections of the rank-1024 path (one
// group: y = qlat . W).  With per-head normalisation a CTA takes the two
// 256-column tiles of a 512-wide head back to back, into the two TMEM
// buffers; the epilogue sums the squares of both halves, then scales and
// stores them (y / sqrt(mean(y^2) + eps) * g), releasing each buffer as it
// is written so the next head's first half can start.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace v4 {

using namespace sm100;

namespace {

constexpr int kThreads = 192;       // warp 0 producer, warp 1 MMA, warps 2-5 epilogue
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr uint32_t kABytes = kBM * kBK * 2;                 // 16 KB
constexpr uint32_t kBBlock = kBK * 64 * 2;                  // 64 K-rows x 64 columns: 8 KB
constexpr uint32_t kBBytes = 4 * kBBlock;                   // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;         // 48 KB
constexpr uint32_t OFF_CTL = kStages * kStageBytes;         // 196608

struct Ctl {
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t fin;
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t kSmemBytes = OFF_CTL + sizeof(Ctl);

struct Params {
  bf16* y;             // [T, G*N]
  const float* norm_w; // [512] RMSNorm weight of a head (pair_norm), null = ones
  int* status;
  int T, G, N, Kg;     // tokens, groups, outputs per group, inputs per group
  int pair_norm;       // 1: RMS-normalise each pair of consecutive 256-column tiles (a 512-wide head)
  int m_fast;          // 1: token tiles vary fastest (each weight block is read once from DRAM)
  float eps;
};

// The k-th tile of this CTA (tiles in tile_of order).  With pair_norm the
// CTA owns pairs: tiles 2i and 2i+1 hold the two halves of one head.
__device__ __forceinline__ int my_tile(int k, const Params& p) {
  if (p.pair_norm) return 2 * (blockIdx.x + (k >> 1) * gridDim.x) + (k & 1);
  return blockIdx.x + k * gridDim.x;
}

__device__ __forceinline__ void tile_of(int tile, const Params& p, int& g, int& m0, int& n0) {
  const int nt = p.N / kBN;
  const int mt = (p.T + kBM - 1) / kBM;
  g = tile / (mt * nt);
  const int r = tile % (mt * nt);
  if (!p.m_fast) {               // grouped projection: a token tile's outputs side by side
    m0 = (r / nt) * kBM;
    n0 = (r % nt) * kBN;
  } else if (p.pair_norm) {      // (head, token tile) pairs, token tiles fastest
    const int pr = r >> 1;
    m0 = (pr % mt) * kBM;
    n0 = (pr / mt) * 2 * kBN + (r & 1) * kBN;
  } else {
    m0 = (r % mt) * kBM;
    n0 = (r / mt) * kBN;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
oproj_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctl* c = reinterpret_cast<Ctl*>(smem + OFF_CTL);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) set_status(p.status, V4_ERR_UNSUPPORTED);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&c->full[i], 1); mbar_init(&c->empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&c->acc_full[i], 1); mbar_init(&c->acc_empty[i], 128); }
    mbar_init(&c->fin, 1);
    c->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_x);
    prefetch_tmap(&map_w);
  }
  if (warp == 1) {
    tmem_alloc(&c->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;
  const int tiles = p.G * ((p.T + kBM - 1) / kBM) * (p.N / kBN);
  const int kblocks = p.Kg / kBK;

  if (warp == 0) {
    if (lane == 0) {
      int use = 0;
      bool ok = true;
      for (int k = 0, tile = my_tile(0, p); tile < tiles && ok; tile = my_tile(++k, p)) {
        int g, m0, n0;
        tile_of(tile, p, g, m0, n0);
        for (int kb = 0; kb < kblocks; ++kb) {
          const int st = use % kStages;
          if (use >= kStages) ok = mbar_wait(&c->empty[st], ((use / kStages) - 1) & 1, &c->abort, p.status);
          if (!ok) break;
          uint8_t* sa = smem + st * kStageBytes;
          mbar_expect_tx(&c->full[st], kStageBytes);
          tma_load_2d(sa, &map_x, g * p.Kg + kb * kBK, m0, &c->full[st]);
#pragma unroll
          for (int nb = 0; nb < 4; ++nb)
            tma_load_2d(sa + kABytes + nb * kBBlock, &map_w, n0 + 64 * nb, g * p.Kg + kb * kBK, &c->full[st]);
          ++use;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 256, 0, 1);
      const uint64_t dA0 = smem_desc(smem_u32(smem), 16, 1024, kLayoutSW128);
      const uint64_t dB0 = smem_desc(smem_u32(smem + kABytes), kBBlock, 1024, kLayoutSW128);
      int use = 0, tc = 0;
      bool ok = true;
      for (int k = 0, tile = my_tile(0, p); tile < tiles && ok; tile = my_tile(++k, p)) {
        const int ab = tc & 1;
        if (tc >= 2) ok = mbar_wait(&c->acc_empty[ab], ((tc >> 1) - 1) & 1, &c->abort, p.status);
        tc_fence_after();
        const uint32_t d = tmem + 256 * ab;
        for (int kb = 0; kb < kblocks && ok; ++kb) {
          const int st = use % kStages;
          ok = mbar_wait(&c->full[st], (use / kStages) & 1, &c->abort, p.status);
          tc_fence_after();
          const uint64_t da = dA0 + (uint64_t)((st * kStageBytes) >> 4);
          const uint64_t db = dB0 + (uint64_t)((st * kStageBytes) >> 4);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_f16_ss(d, da + (uint64_t)((32 * ks) >> 4), db + (uint64_t)((2048 * ks) >> 4), idesc,
                        (kb | ks) != 0);
          umma_commit(&c->empty[st]);
          ++use;
        }
        umma_commit(&c->acc_full[ab]);
        ++tc;
      }
      umma_commit(&c->fin);
      mbar_wait(&c->fin, 0, &c->abort, p.status, 200000000ull);
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    int tc = 0;
    if (!p.pair_norm) {
      for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        int g, m0, n0;
        tile_of(tile, p, g, m0, n0);
        const int ab = tc & 1;
        mbar_wait(&c->acc_full[ab], (tc >> 1) & 1, &c->abort, p.status);
        tc_fence_after();
        const int t = m0 + row;
        bf16* yrow = p.y + (size_t)t * p.G * p.N + (size_t)g * p.N + n0;
#pragma unroll 1
        for (int cb = 0; cb < kBN / 32; ++cb) {
          float v[32];
          tmem_ld32(tmem + lane_base + 256 * ab + 32 * cb, v);
          tmem_wait_ld();
          if (t < p.T) {
#pragma unroll
            for (int q = 0; q < 4; ++q) store8(yrow + 32 * cb + 8 * q, v + 8 * q);
          }
        }
        tc_fence_before();
        mbar_arrive(&c->acc_empty[ab]);
        ++tc;
      }
    } else {
      // one 512-wide head per pair: halves in buffers 0 and 1
      for (int k = 0, tile = my_tile(0, p); tile < tiles; k += 2, tile = my_tile(k, p)) {
        int g, m0, n0;
        tile_of(tile, p, g, m0, n0);
        const uint32_t ph = (tc >> 1) & 1;
        float ss[4] = {0.f, 0.f, 0.f, 0.f};
        // squares of the first half while the second half's products run
#pragma unroll 1
        for (int ab = 0; ab < 2; ++ab) {
          mbar_wait(&c->acc_full[ab], ph, &c->abort, p.status);
          tc_fence_after();
#pragma unroll 1
          for (int cb = 0; cb < kBN / 32; ++cb) {
            float v[32];
            tmem_ld32(tmem + lane_base + 256 * ab + 32 * cb, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ss[i & 3] = fmaf(v[i], v[i], ss[i & 3]);
          }
        }
        const float rs = 1.0f / sqrtf(((ss[0] + ss[1]) + (ss[2] + ss[3])) / (float)(2 * kBN) + p.eps);
        const int t = m0 + row;
        bf16* yrow = p.y + (size_t)t * p.G * p.N + (size_t)g * p.N + n0;
#pragma unroll 1
        for (int ab = 0; ab < 2; ++ab) {
#pragma unroll 1
          for (int cb = 0; cb < kBN / 32; ++cb) {
            float v[32];
            tmem_ld32(tmem + lane_base + 256 * ab + 32 * cb, v);
            tmem_wait_ld();
            const int c0 = kBN * ab + 32 * cb;            // column within the head
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= p.norm_w ? rs * p.norm_w[c0 + i] : rs;
            if (t < p.T) {
#pragma unroll
              for (int q = 0; q < 4; ++q) store8(yrow + c0 + 8 * q, v + 8 * q);
            }
          }
          tc_fence_before();
          mbar_arrive(&c->acc_empty[ab]);
        }
        tc += 2;
      }
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

bool oproj_tc_supported(const v4_config& c) {
  if (c.dtype != V4_BF16 || c.o_groups < 1 || c.n_heads % c.o_groups) return false;
  const long long kg = (long long)(c.n_heads / c.o_groups) * c.head_dim;
  return kg % kBK == 0 && c.o_rank % kBN == 0 && c.o_rank > 0;
}

cudaError_t launch_oproj_tc(const v4_config& cfg, const void* o, const void* wo_a, void* y, int* status,
                            cudaStream_t st) {
  const long long T = (long long)cfg.batch * q_rows(cfg);      // the call's query rows
  const int G = cfg.o_groups, N = cfg.o_rank;
  const int Kg = (cfg.n_heads / G) * cfg.head_dim;
  CUtensorMap mx, mw;
  int e = 0;
  e |= make_tmap_bf16_2d(&mx, o, (uint64_t)G * Kg, (uint64_t)T, kBK, kBM, true);
  e |= make_tmap_bf16_2d(&mw, wo_a, (uint64_t)N, (uint64_t)G * Kg, 64, kBK, true);
  if (e) return cudaErrorInvalidValue;
  Params prm;
  prm.y = (bf16*)y;
  prm.norm_w = nullptr;
  prm.status = status;
  prm.T = (int)T;
  prm.G = G;
  prm.N = N;
  prm.Kg = Kg;
  prm.pair_norm = 0;
  prm.m_fast = 0;
  prm.eps = 0.f;
  cudaError_t err = cudaFuncSetAttribute(oproj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long tiles = (long long)G * ((T + kBM - 1) / kBM) * (N / kBN);
  const int grid = (int)(tiles < sms ? tiles : sms);
  if (grid == 0) return cudaSuccess;
  oproj_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mx, mw, prm);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_qproj_tc(long long T, int rank, const void* x, const void* w, int N, void* y, int norm,
                            float eps, const float* norm_w, int* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  CUtensorMap mx, mw;
  int e = 0;
  e |= make_tmap_bf16_2d(&mx, x, (uint64_t)rank, (uint64_t)T, kBK, kBM, true);
  e |= make_tmap_bf16_2d(&mw, w, (uint64_t)N, (uint64_t)rank, 64, kBK, true);
  if (e) return cudaErrorInvalidValue;
  Params prm;
  prm.y = (bf16*)y;
  prm.norm_w = norm_w;
  prm.status = status;
  prm.T = (int)T;
  prm.G = 1;
  prm.N = N;
  prm.Kg = rank;
  prm.pair_norm = norm ? 1 : 0;
  prm.m_fast = 1;
  prm.eps = eps;
  cudaError_t err = cudaFuncSetAttribute(oproj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long tiles = ((T + kBM - 1) / kBM) * (N / kBN);
  const long long units = norm ? tiles / 2 : tiles;
  const int grid = (int)(units < sms ? units : sms);
  oproj_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mx, mw, prm);
  note_launch();
  return cudaGetLastError();
}

}  // namespace v4
