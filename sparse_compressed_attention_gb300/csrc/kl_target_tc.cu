// Sparse indexer distillation target on the 5th-generation tensor cores.
//
// Primus PR #930 item 5 (KL(attention || indexer) over the selected entries,
// the sparse top-k variant that stays in [B, S, K]) and item 11 (the target
// branch is detached: gather and GEMM at the model dtype, heads summed inside
// the loop so [B, H, S, K] never exists).
//
// For query t and its selected entries e_k, with the forward's lse:
//   raw[t, k] = sum_h exp(scale * rot(q_h, t) . ent[e_k] - lse[t, h])
// i.e. the main attention's probabilities (window and sink stay in lse) on
// the selected entries, summed over the heads; a row kernel then normalises
// raw over the slots, forms the indexer's softmax over the same slots, the
// KL loss and its gradient with respect to the indexer scores.
//
// Per (query, 64-head slice) work item (one CTA, persistent): the selected
// entries in tiles of 128 gathered into eight 128-byte-swizzled K-block
// slots, S^T[key, head] = K_tile . Qr^T (M = 128 keys, N = 64, K = 512) into
// a double-buffered TMEM accumulator; the slots are released K-block by
// K-block as the products read them, so the next tile's gathers overlap.
// Eight softmax warps (two per TMEM lane quarter, 32 heads each) exponentiate
// against lse, sum their heads and add into raw (fp32 atomics: the two head
// halves and any further 64-head slices of the query).
// Warp roles (384 threads): warp 0 producer (selection list with slots,
// query rows by TMA, a third of the gathers), warp 1 MMA issuer and TMEM
// owner, warps 2-3 the other gathers, warps 4-11 softmax.
#include <cuda.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace v4 {

using namespace sm100;

namespace {

constexpr int kH = 64, kD = 512, kR = 64;
constexpr int kThreads = 384;
constexpr int kSoftThreads = 256;                 // warps 4-11
constexpr int kGatherLanes = 96;                  // warps 0, 2, 3
constexpr int kTileKeys = 128;
constexpr int kSlots = 8;
constexpr uint32_t kSlotBytes = 128 * 128;        // 128 keys x 64 dims x 2 B
constexpr uint32_t kQBlockBytes = 64 * 128;       // 64 heads x 64 dims x 2 B
constexpr int kMaxSel = 1024;
constexpr int kMaxGroups = 11;

constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_SLOT = OFF_Q + 8 * kQBlockBytes;                 // 65536
constexpr uint32_t OFF_LIST = OFF_SLOT + kSlots * kSlotBytes;           // 196608: [2][entry u16 | slot u16]
constexpr uint32_t OFF_CTL = OFF_LIST + 2 * kMaxSel * 4;                // 204800

struct QInfo {
  int b, t, hs, n_ent, tiles, done;
};

struct Ctl {
  uint64_t full[kSlots], empty[kSlots];
  uint64_t list_free[2];
  uint64_t q_full, q_ready, q_empty;
  uint64_t s_full[2], s_empty[2];
  uint64_t info_full[2], info_empty[2];
  uint64_t fin;
  QInfo info[2];
  float lse2[2][kH];
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t kSmemBytes = OFF_CTL + sizeof(Ctl);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  const bf16* q;               // [B,S,H,512] (L2 prefetch of the next query's rows)
  const bf16* ent;             // [B*N, 512] rotated entries
  const int32_t* idx;          // [B,S,K]
  const float* lse;            // [B,S,H]
  const float2* rope_cs;       // [S][32]
  float* raw;                  // [B,S,K] pre-zeroed
  int* status;
  int B, S, N, ratio, K, H, HS;
  float scale;
};

__device__ __forceinline__ bool wait_ok(uint64_t* bar, uint32_t parity, Ctl* c, int* status) {
  return mbar_wait(bar, parity, &c->abort, status);
}

// One K-block (64 dims) of the selected entries of a tile: lane covers row
// 4*grp + lane/8, 16-byte chunk lane%8 (128-byte-swizzled K-major layout);
// one arrival when the copies land.
__device__ __forceinline__ void gather_kblock(uint8_t* slot, const bf16* ent, const int* sidx, int gw, int nw,
                                              int lane, int kb, uint64_t* full, int n_rows, int* status) {
  const int chunk = lane & 7;
  const bf16* src = ent + kb * 64 + chunk * 8;
  const uint32_t d0 = smem_u32(slot);
#pragma unroll
  for (int i = 0; i < kMaxGroups; ++i) {
    const int grp = gw + nw * i;
    if (grp < 32) {
      const int row = 4 * grp + (lane >> 3);
      if (V4_BOUND(sidx[i] >= 0 && sidx[i] < n_rows, status))
        cp_async_16(d0 + row * 128 + ((chunk ^ (row & 7)) << 4), src + (size_t)sidx[i] * kD);
    }
  }
  cp_async_mbar_arrive(full);
}

// Global entry rows of tile j for gather warp gw of nw (row 0 pads short tiles).
__device__ __forceinline__ void load_rows(const uint32_t* list, int n_ent, int j, int gw, int nw, int lane,
                                          int* sidx, int b, int N) {
#pragma unroll
  for (int i = 0; i < kMaxGroups; ++i) {
    const int grp = gw + nw * i;
    const int k = j * kTileKeys + 4 * grp + (lane >> 3);
    sidx[i] = b * N + ((grp < 32 && k < n_ent) ? (int)(list[k] & 0xFFFFu) : 0);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
kl_target_tc_kernel(const __grid_constant__ CUtensorMap map_q, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctl* c = reinterpret_cast<Ctl*>(smem + OFF_CTL);
  uint32_t* lists = reinterpret_cast<uint32_t*>(smem + OFF_LIST);   // [2][kMaxSel]: entry | slot << 16
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) set_status(p.status, V4_ERR_UNSUPPORTED);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&c->full[i], kGatherLanes);
      mbar_init(&c->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->list_free[i], 64 + kSoftThreads);
      mbar_init(&c->s_full[i], 1);
      mbar_init(&c->s_empty[i], kSoftThreads);
      mbar_init(&c->info_full[i], 1);
      mbar_init(&c->info_empty[i], 1 + 64 + kSoftThreads);
    }
    mbar_init(&c->q_full, 1);
    mbar_init(&c->q_ready, kSoftThreads);
    mbar_init(&c->q_empty, 1);
    mbar_init(&c->fin, 1);
    c->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&map_q);
  if (warp == 1) {
    tmem_alloc(&c->tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;
  const int total = p.B * p.S * p.HS;

  // every consumer copies the query's description and releases the slot
  auto receive = [&](int qc, QInfo& inf) -> bool {
    const int is = qc & 1;
    const bool ok = wait_ok(&c->info_full[is], (qc >> 1) & 1, c, p.status);
    inf = c->info[is];
    mbar_arrive(&c->info_empty[is]);
    return ok && !inf.done;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int qc = 0, g = 0;
    bool ok = true;
    int item = blockIdx.x;
    while (ok) {
      // the next work item whose query selected at least one entry
      QInfo inf;
      inf.done = 1;
      inf.b = inf.t = inf.hs = inf.n_ent = inf.tiles = 0;
      const int is = qc & 1;
      if (lane == 0 && qc >= 2) ok = wait_ok(&c->list_free[is], ((qc >> 1) - 1) & 1, c, p.status);
      ok = __shfl_sync(0xffffffffu, (int)ok, 0);
      if (!ok) break;
      uint32_t* lst = lists + is * kMaxSel;
      for (; item < total; item += gridDim.x) {
        const int qi = item / p.HS;
        const int b = qi % p.B, t = p.S - 1 - qi / p.B;
        const int nv = min((t + 1) / p.ratio, p.N);
        const int32_t* row = p.idx + ((size_t)b * p.S + t) * p.K;
        const unsigned below = (1u << lane) - 1u;
        // every load first, then the ballots: one memory latency per row
        int sv[kMaxSel / 32];
#pragma unroll
        for (int i = 0; i < kMaxSel / 32; ++i) sv[i] = 32 * i + lane < p.K ? row[32 * i + lane] : -1;
        int n = 0;
#pragma unroll
        for (int i = 0; i < kMaxSel / 32; ++i) {
          const int k = 32 * i + lane;
          int v = sv[i];
          if (v < -1 || v >= nv) {
            set_status(p.status, kStatusBadIndex);
            v = -1;
          }
          const unsigned msk = __ballot_sync(0xffffffffu, v >= 0);
          if (v >= 0) lst[n + __popc(msk & below)] = (uint32_t)v | ((uint32_t)k << 16);
          n += __popc(msk);
        }
        if (n > 0) {
          // warm L2 with the query rows of this CTA's next item
          const int nx = item + gridDim.x;
          if (lane == 0 && nx < total) {
            const int qn = nx / p.HS;
            const bf16* nrows = p.q + (((size_t)(qn % p.B) * p.S + (p.S - 1 - qn / p.B)) * p.H + kH * (nx % p.HS)) * kD;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(nrows), "r"(kH * kD * 2) : "memory");
          }
          inf.done = 0;
          inf.b = b;
          inf.t = t;
          inf.hs = item % p.HS;
          inf.n_ent = n;
          inf.tiles = (n + kTileKeys - 1) / kTileKeys;
          break;
        }
      }
      __syncwarp();
      if (lane == 0) {
        if (qc >= 2) (void)wait_ok(&c->info_empty[is], ((qc >> 1) - 1) & 1, c, p.status);
        c->info[is] = inf;
        mbar_arrive(&c->info_full[is]);
      }
      __syncwarp();
      if (inf.done) break;
      // query rows of this head slice: one 8 KB box per lane 0..7
      if (lane == 0 && qc >= 1) ok = wait_ok(&c->q_empty, (qc - 1) & 1, c, p.status);
      ok = __shfl_sync(0xffffffffu, (int)ok, 0);
      if (!ok) break;
      if (lane == 0) mbar_expect_tx(&c->q_full, 8 * kQBlockBytes);
      __syncwarp();
      if (lane < 8)
        tma_load_2d(smem + OFF_Q + lane * kQBlockBytes, &map_q, 64 * lane, (inf.b * p.S + inf.t) * p.H + kH * inf.hs,
                    &c->q_full);
      for (int j = 0; j < inf.tiles && ok; ++j) {
        int sidx[kMaxGroups];
        load_rows(lst, inf.n_ent, j, 0, 3, lane, sidx, inf.b, p.N);
        for (int kb = 0; kb < kSlots; ++kb) {
          if (lane == 0 && g >= 1) ok = wait_ok(&c->empty[kb], (g - 1) & 1, c, p.status);
          ok = __shfl_sync(0xffffffffu, (int)ok, 0);
          if (!ok) break;
          gather_kblock(smem + OFF_SLOT + kb * kSlotBytes, p.ent, sidx, 0, 3, lane, kb, &c->full[kb], p.B * p.N,
                        p.status);
        }
        ++g;
      }
      ++qc;
      item += gridDim.x;
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ gather helpers
    const int gw = warp - 1;
    int qc = 0, g = 0;
    QInfo inf;
    bool ok = true;
    while (ok && receive(qc, inf)) {
      const int is = qc & 1;
      const uint32_t* lst = lists + is * kMaxSel;
      for (int j = 0; j < inf.tiles && ok; ++j) {
        int sidx[kMaxGroups];
        load_rows(lst, inf.n_ent, j, gw, 3, lane, sidx, inf.b, p.N);
        for (int kb = 0; kb < kSlots; ++kb) {
          if (lane == 0 && g >= 1) ok = wait_ok(&c->empty[kb], (g - 1) & 1, c, p.status);
          ok = __shfl_sync(0xffffffffu, (int)ok, 0);
          if (!ok) break;
          gather_kblock(smem + OFF_SLOT + kb * kSlotBytes, p.ent, sidx, gw, 3, lane, kb, &c->full[kb], p.B * p.N,
                        p.status);
        }
        ++g;
      }
      mbar_arrive(&c->list_free[is]);
      ++qc;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id1 = idesc_bf16_f32(128, 64, 0, 0);
      const uint64_t dA = smem_desc(smem_u32(smem + OFF_SLOT), 16, 1024, kLayoutSW128);
      const uint64_t dQ = smem_desc(smem_u32(smem + OFF_Q), 16, 1024, kLayoutSW128);
      int qc = 0, g = 0;
      bool ok = true;
      QInfo inf;
      while (ok && receive(qc, inf)) {
        ok = wait_ok(&c->q_ready, qc & 1, c, p.status);
        tc_fence_after();
        for (int j = 0; j < inf.tiles && ok; ++j) {
          const int sb = g & 1;
          if (g >= 2) ok = wait_ok(&c->s_empty[sb], ((g >> 1) - 1) & 1, c, p.status);
          tc_fence_after();
#pragma unroll
          for (int kb = 0; kb < kSlots; ++kb) {
            ok = ok && wait_ok(&c->full[kb], g & 1, c, p.status);
            fence_proxy_async_smem();                 // cp.async writes -> tensor-core reads
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_f16_ss(tmem + 64 * sb, dA + (uint64_t)((kb * kSlotBytes + 32 * ks) >> 4),
                          dQ + (uint64_t)((kb * kQBlockBytes + 32 * ks) >> 4), id1, (kb | ks) != 0);
            umma_commit(&c->empty[kb]);
          }
          umma_commit(&c->s_full[sb]);
          if (j == inf.tiles - 1) umma_commit(&c->q_empty);
          ++g;
        }
        ++qc;
      }
      // every issued MMA completes before TMEM is released
      umma_commit(&c->fin);
      mbar_wait(&c->fin, 0, &c->abort, p.status, 200000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int ts = threadIdx.x - 128;         // 0..255
    const int quarter = warp & 3;
    const int hh = (warp - 4) >> 2;
    const int krow = 32 * quarter + lane;
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    const float log2e = 1.4426950408889634f;
    const float c1 = p.scale * log2e;
    int qc = 0, g = 0;
    QInfo inf;
    while (receive(qc, inf)) {
      const int is = qc & 1;
      // rotate the last 64 dims of every head at t (K-block 7 of the query
      // rows, in place: 256 threads, 4 per head, 16 pairs each) and stage lse
      {
        const int h = ts >> 2, part = ts & 3;
        float4 csv[4];
        const float4* csp = reinterpret_cast<const float4*>(p.rope_cs + (size_t)inf.t * (kR / 2) + 8 * part);
#pragma unroll
        for (int i = 0; i < 4; ++i) csv[i] = csp[i];
        if (ts < kH) c->lse2[is][ts] = p.lse[((size_t)inf.b * p.S + inf.t) * p.H + kH * inf.hs + ts] * log2e;
        wait_ok(&c->q_full, qc & 1, c, p.status);
        uint8_t* qrow = smem + OFF_Q + 7 * kQBlockBytes + h * 128;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int ch = 2 * part + cc;
          uint4* ptr = reinterpret_cast<uint4*>(qrow + ((ch ^ (h & 7)) * 16));
          uint4 u = *ptr;
          __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&u);
          const float4 cs01 = csv[2 * cc], cs23 = csv[2 * cc + 1];
          const float cs[8] = {cs01.x, cs01.y, cs01.z, cs01.w, cs23.x, cs23.y, cs23.z, cs23.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(hv[i]);
            rot_pair(f.x, f.y, cs[2 * i], cs[2 * i + 1]);
            hv[i] = __floats2bfloat162_rn(f.x, f.y);
          }
          *ptr = u;
        }
        fence_proxy_async_smem();
        named_bar_sync(1, kSoftThreads);
        mbar_arrive(&c->q_ready);
      }
      const float* lse2 = c->lse2[is] + 32 * hh;
      const uint32_t* lst = lists + is * kMaxSel;
      float* rawrow = p.raw + ((size_t)inf.b * p.S + inf.t) * p.K;
      for (int j = 0; j < inf.tiles; ++j) {
        const int sb = g & 1;
        const int k = j * kTileKeys + krow;
        const bool valid = k < inf.n_ent;
        const int slot = valid ? (int)(lst[k] >> 16) : 0;
        wait_ok(&c->s_full[sb], (g >> 1) & 1, c, p.status);
        tc_fence_after();
        float v[32];
        tmem_ld32(tmem + lane_base + 64 * sb + 32 * hh, v);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&c->s_empty[sb]);
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i & 3] += exp2f(fmaf(v[i], c1, -lse2[i]));
        if (valid) atomicAdd(rawrow + slot, (a[0] + a[1]) + (a[2] + a[3]));
        ++g;
      }
      mbar_arrive(&c->list_free[is]);
      ++qc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ---------------------------------------------------------------------------
// Row pass: target = raw / sum(raw) over the valid slots; with iscore the
// indexer's softmax over the same slots, loss = KL(target || softmax) and
// dscore = softmax - target.  One warp per (b, t) row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
kl_finish_kernel(const int32_t* __restrict__ idx, const float* __restrict__ iscore, float* __restrict__ target,
                 float* __restrict__ loss, float* __restrict__ dscore, long long rows, int K) {
  const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int32_t* ir = idx + r * K;
  float* tr = target + r * K;
  float tot = 0.f, mx = -INFINITY;
  for (int k = lane; k < K; k += 32) {
    if (ir[k] >= 0) {
      tot += tr[k];
      if (iscore) mx = fmaxf(mx, iscore[r * K + k]);
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const float inv = tot > 0.f ? 1.0f / tot : 0.f;
  float es = 0.f;
  if (iscore) {
    for (int k = lane; k < K; k += 32)
      if (ir[k] >= 0) es += expf(iscore[r * K + k] - mx);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) es += __shfl_xor_sync(0xffffffffu, es, o);
  }
  const float lz = mx + logf(es);            // log of the softmax denominator
  float kl = 0.f;
  for (int k = lane; k < K; k += 32) {
    const bool valid = ir[k] >= 0;
    const float pk = valid ? tr[k] * inv : 0.f;
    tr[k] = pk;
    if (iscore) {
      const float lq = valid ? iscore[r * K + k] - lz : 0.f;
      if (pk > 0.f) kl += pk * (logf(pk) - lq);
      if (dscore) dscore[r * K + k] = valid ? expf(lq) - pk : 0.f;
    }
  }
  if (iscore && loss) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) kl += __shfl_xor_sync(0xffffffffu, kl, o);
    if (lane == 0) loss[r] = kl;
  }
}

}  // namespace

bool kl_target_tc_supported(const v4_config& c) {
  return c.dtype == V4_BF16 && c.n_heads >= kH && c.n_heads % kH == 0 && c.n_heads <= 8 * kH &&
         c.head_dim == kD && c.rope_dim == kR && c.ratio >= 1 && c.topk >= 1 && c.topk <= kMaxSel &&
         c.seqlen / c.ratio <= 65536;
}

cudaError_t launch_kl_target(const v4_config& cfg, const void* q, const void* ent, const int32_t* idx,
                             const float* lse, const float* iscore, const float2* cs_table, float* target,
                             float* loss, float* dscore, int* status, cudaStream_t st) {
  const int B = cfg.batch, S = cfg.seqlen, K = cfg.topk;
  const int N = S / cfg.ratio;
  const long long rows = (long long)B * S;
  cudaError_t err = cudaMemsetAsync(target, 0, (size_t)rows * K * sizeof(float), st);
  if (err != cudaSuccess) return err;
  if (N > 0) {
    CUtensorMap mq;
    if (make_tmap_bf16_2d(&mq, q, kD, (uint64_t)rows * cfg.n_heads, 64, 64, true)) return cudaErrorInvalidValue;
    Params prm;
    prm.q = (const bf16*)q;
    prm.ent = (const bf16*)ent;
    prm.idx = idx;
    prm.lse = lse;
    prm.rope_cs = cs_table;
    prm.raw = target;
    prm.status = status;
    prm.B = B;
    prm.S = S;
    prm.N = N;
    prm.ratio = cfg.ratio;
    prm.K = K;
    prm.H = cfg.n_heads;
    prm.HS = cfg.n_heads / kH;
    prm.scale = cfg.softmax_scale > 0.f ? cfg.softmax_scale : 1.0f / sqrtf((float)kD);
    err = cudaFuncSetAttribute(kl_target_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long items = rows * prm.HS;
    const int grid = (int)(items < sms ? items : sms);
    kl_target_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mq, prm);
    note_launch();
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  kl_finish_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(idx, iscore, target, loss, dscore, rows, K);
  note_launch();
  return cudaGetLastError();
}

}  // namespace v4
