// Sparse / dense multi-query attention on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators, TMA) for the DeepSeek-V4-Flash shapes:
// 64 query heads sharing one 512-d latent that is both key and value, the
// last 64 dims rotated, bf16 storage, window <= 128.
//
// Method: "Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X GPUs
// with Primus", sections "The DeepSeek-V4-Flash architecture", "Three
// attention types, interleaved" and "Kernel fusions" (row "SWA / CSA / HCA
// attention": in-kernel gather of the selected entries, window branch and
// sink in one softmax); Primus PR #930 item 1 (scale D^-1/2) and item 3
// (output de-rotated at -t).  The softmax follows the page's "fixed max via
// shift invariance" (section "Attention kernels for the three layer types"):
// each head's largest logit over the query's first key tile is the shift
// for all its tiles, so there is no running max and no rescaling and
// partial sums simply add.  A later key above that shift only makes its P
// exceed 1; a query whose denominator leaves [nk * 1e-26, 2^100) (an
// overflow, or mass lost to underflow) is recomputed by the CUDA-core
// kernel with a running max.
//
// Layout per query t (one CTA, persistent over queries):
//   S^T[key, head] = K_tile[128 keys x 512] . Q^T          (M=128 keys, N=64)
//   P^T = exp(S^T * scale - m) in bf16 (one thread per key row)
//   O^T[dim, head] += K_tile^T[512 x 128 keys] . P^T     (4 x M=128 dims, N=64)
// The key tile in shared memory (8 K-blocks of [128 keys x 64 dims], 128-byte
// swizzle) is the K-major A operand of the first product and, read as
// MN-major, the A operand of the second.  TMEM: S^T double buffer (2 x 64
// columns) and O^T (256 columns).  The softmax denominators sum exactly the
// bf16 P the output uses: after publishing its P row, each softmax warp folds
// its 32 key rows per head with a lane butterfly while the MMAs run, and the
// four warp partials meet in shared memory at the end of the query.
// Contiguous key tiles (window rows, HCA entries) and the query rows arrive
// by TMA boxes; selected entries are gathered row by row with 16-byte
// cp.async (many small TMA gathers would serialise in the TMA unit).  Each
// output row leaves with direct stores (the 32 lanes of a warp cover 64
// contiguous bytes per head; a lane transpose to 16-byte stores measured
// slower, its shuffles being latency-bound with one softmax warp per SM
// sub-partition).  Rotations read a per-position cos/sin table built once per
// call.
//
// Warp roles (384 threads): warp 0 producer (per-query selection list, query
// rows and contiguous tiles by TMA, one third of the gathers), warp 1 MMA
// issuer and TMEM owner, warps 2-3 gather the other two thirds, warps 4-11
// softmax + epilogue (two per TMEM lane quarter, 32 heads each).
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
constexpr int kSlots = 8;                         // one tile: 8 K-blocks of 64 dims
constexpr uint32_t kSlotBytes = 128 * 128;        // 128 keys x 64 dims x 2 B
constexpr uint32_t kQBlockBytes = 64 * 128;       // 64 heads x 64 dims x 2 B
constexpr uint32_t kPBytes = 128 * 64 * 2;        // 128 keys x 64 heads x 2 B
constexpr int kMaxSel = 1024;

constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_SLOT = OFF_Q + 8 * kQBlockBytes;           // 65536
constexpr uint32_t OFF_P = OFF_SLOT + kSlots * kSlotBytes;        // 196608
constexpr uint32_t OFF_LIST = OFF_P + kPBytes;                    // 212992 (one P^T buffer)
constexpr uint32_t OFF_CTL = OFF_LIST + 2 * kMaxSel * 2;          // 217088 (two 16-bit lists)

struct QInfo {
  int b, t, hs, n_ent, ent_tiles, tiles, w_lo, done;     // hs: head slice (64 heads each)
};

struct Ctl {
  uint64_t full_g[kSlots];                 // gathered K-block landed: 96 gather-lane arrivals
  uint64_t full_t[kSlots];                 // contiguous K-block landed: one arrival + TMA bytes
  uint64_t empty[kSlots];
  uint64_t list_free[2];                   // warps 2-3 have read selection list 0 / 1
  uint64_t q_full, q_ready, q_empty;
  uint64_t s_full[2], p_ready[2];
  uint64_t o_full, o_empty;
  uint64_t info_full[2], info_empty[2];
  uint64_t fin;
  QInfo info[2];
  float mlog2[2][kH];          // per-query shift (log2 units), double-buffered by query parity
  float hmax[4][kH];           // first tile: each TMEM lane quarter's largest logit per head
  uint32_t tmem_base;
  int abort;
  int decision;
  int redo;
};

constexpr uint32_t kSmemBytes = OFF_CTL + sizeof(Ctl);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  const bf16* q;               // [B,Sq,H,512] (L2 prefetch of upcoming queries)
  const bf16* ent;             // [B,N,512] gathered entries
  bf16* o;                     // [B,Sq,H,512]
  const int32_t* idx;          // [B,Sq,K] or null
  const float* sink;           // [H] or null
  const float2* rope_cs;       // [S][32] cos/sin
  // Two unused slots: with them the parameter block keeps the layout the
  // kernel was tuned at, which measured 1.7% faster on the CSA + HCA layer
  // pair at S=16384 than the same code without them (outputs identical;
  // a code-generation effect of the layout, not of the values).
  const void* reserved0;
  const void* reserved1;
  float* lse;                  // [B,Sq,H] or null
  int* status;
  int* counters;               // [0] work item, [1] redo count, [2..] redo list (query rows)
  int B, S, N, ratio, window, K;
  int Sq, t0;                  // query rows per sequence, at positions t0 .. t0+Sq-1
  int H, HS;                   // heads, head slices of 64
  float scale;
};

__device__ __forceinline__ bool wait_ok(uint64_t* bar, uint32_t parity, Ctl* c, int* status) {
  return mbar_wait(bar, parity, &c->abort, status);
}

// Row groups (4 rows each) of a 128-key tile: with nw gathering warps, warp
// gw takes groups gw, gw+nw, ... (three warps: at most 11 groups each).
// More gathering warps do not speed the kernel: with one tile of slots per
// SM a K-block's gather can start only when the O products free its slot,
// and seven gathering warps (512 threads) measured slower than three (the
// O products lose shared-memory bandwidth to the extra copies).
constexpr int kMaxGroups = 11;

// Gather one K-block (64 dims) of the selected entries of a tile: lane
// covers row 4*grp + lane/8, 16-byte chunk lane%8, written into the
// 128-byte-swizzled K-major slot layout; one arrival when the copies land.
__device__ __forceinline__ void gather_kblock(uint8_t* slot, const bf16* ent_b, const int* sidx, int gw, int nw,
                                              int lane, int kb, uint64_t* full, int n_rows, int* status) {
  const int chunk = lane & 7;
  const bf16* src = ent_b + kb * 64 + chunk * 8;
  const uint32_t d0 = smem_u32(slot);
#pragma unroll
  for (int i = 0; i < kMaxGroups; ++i) {
    const int grp = gw + nw * i;
    if (grp < 32) {
      const int row = 4 * grp + (lane >> 3);
      if (V4_BOUND(sidx[i] >= 0 && sidx[i] < n_rows && kb >= 0 && kb < kSlots, status))
        cp_async_16(d0 + row * 128 + ((chunk ^ (row & 7)) << 4), src + (size_t)sidx[i] * kD);
    }
  }
  cp_async_mbar_arrive(full);
}

// Selection-list rows of tile j for gather warp gw of nw (row 0 pads short tiles).
__device__ __forceinline__ void load_rows(const uint16_t* list, int n_ent, int j, int gw, int nw, int lane,
                                          int* sidx) {
#pragma unroll
  for (int i = 0; i < kMaxGroups; ++i) {
    const int grp = gw + nw * i;
    const int k = j * 128 + 4 * grp + (lane >> 3);
    sidx[i] = (grp < 32 && k < n_ent) ? list[k] : 0;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
mqa_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv,
              const __grid_constant__ CUtensorMap map_ent, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctl* c = reinterpret_cast<Ctl*>(smem + OFF_CTL);
  uint16_t* lists = reinterpret_cast<uint16_t*>(smem + OFF_LIST);   // [2][kMaxSel], by query parity
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0) {          // swizzled operands need 1 KB alignment
    if (threadIdx.x == 0) set_status(p.status, V4_ERR_UNSUPPORTED);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&c->full_g[i], kGatherLanes);
      mbar_init(&c->full_t[i], 1);
      mbar_init(&c->empty[i], 1);
    }
    mbar_init(&c->list_free[0], 64);
    mbar_init(&c->list_free[1], 64);
    mbar_init(&c->q_full, 1);
    mbar_init(&c->q_ready, kSoftThreads);
    mbar_init(&c->q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->s_full[i], 1);
      mbar_init(&c->p_ready[i], kSoftThreads);
      mbar_init(&c->info_full[i], 1);
      mbar_init(&c->info_empty[i], 1 + kSoftThreads + 64);
    }
    mbar_init(&c->o_full, 1);
    mbar_init(&c->o_empty, kSoftThreads);
    mbar_init(&c->fin, 1);
    c->abort = 0;
    c->redo = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_q);
    prefetch_tmap(&map_kv);
    prefetch_tmap(&map_ent);
  }
  if (warp == 1) {
    tmem_alloc(&c->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;
  const int total = p.B * p.Sq * p.HS;       // work items: (query, head slice)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Query qc+1 is described (selection list, tile counts) and published
    // while query qc's first tile loads, so every role can move on to it
    // without waiting; its selection row is read one more query ahead.
    // Lists alternate between two 16-bit buffers.
    const bool gathered = p.ratio > 0 && p.idx != nullptr;
    int sv[kMaxSel / 32];
    auto fetch_ahead = [&](int it) {
      if (it >= total) return;
      const int qi = it / p.HS;
      const int nb = qi % p.B, nr = p.Sq - 1 - qi / p.B;
      if (gathered) {
        const int32_t* row = p.idx + ((size_t)nb * p.Sq + nr) * p.K;
#pragma unroll
        for (int i = 0; i < kMaxSel / 32; ++i) {
          const int j = lane + 32 * i;
          sv[i] = j < p.K ? row[j] : -1;
        }
      }
    };
    auto prepare = [&](int qn, int it) -> QInfo {
      QInfo inf;
      inf.done = it >= total ? 1 : 0;
      inf.b = inf.done ? 0 : (it / p.HS) % p.B;
      inf.t = inf.done ? 0 : p.t0 + p.Sq - 1 - (it / p.HS) / p.B;
      inf.hs = inf.done ? 0 : it % p.HS;
      inf.n_ent = 0;
      inf.w_lo = 0;
      if (!inf.done) {
        if (lane == 0) {                      // warm L2 with its query rows, loaded one query later
          const bf16* qn_rows = p.q + (((size_t)inf.b * p.Sq + inf.t - p.t0) * p.H + kH * inf.hs) * kD;
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(qn_rows), "r"(kH * kD * 2) : "memory");
        }
        const int nv = p.ratio > 0 ? min((inf.t + 1) / p.ratio, p.N) : 0;
        if (gathered) {
          // the helpers must have read the list this buffer held two queries ago
          if (lane == 0 && qn >= 2) (void)wait_ok(&c->list_free[qn & 1], ((qn >> 1) - 1) & 1, c, p.status);
          __syncwarp();
          uint16_t* lst = lists + (qn & 1) * kMaxSel;
          // every ballot first, then the stores: no chain through the count
          unsigned msk[kMaxSel / 32];
#pragma unroll
          for (int i = 0; i < kMaxSel / 32; ++i) {
            if (sv[i] < -1 || sv[i] >= nv) {
              set_status(p.status, kStatusBadIndex);
              sv[i] = -1;
            }
            msk[i] = __ballot_sync(0xffffffffu, sv[i] >= 0);
          }
          const unsigned below = (1u << lane) - 1u;
          int base = 0;
#pragma unroll
          for (int i = 0; i < kMaxSel / 32; ++i) {
            const int pos = base + __popc(msk[i] & below);
            if (sv[i] >= 0 && V4_BOUND(pos < kMaxSel, p.status)) lst[pos] = (uint16_t)sv[i];
            base += __popc(msk[i]);
          }
          inf.n_ent = base;
        } else if (p.ratio > 0) {
          inf.n_ent = nv;
        }
        inf.w_lo = max(0, inf.t - p.window + 1);
        __syncwarp();
        fetch_ahead(it + gridDim.x);
      }
      inf.ent_tiles = (inf.n_ent + kTileKeys - 1) / kTileKeys;
      inf.tiles = inf.ent_tiles + 1;            // + the window tile
      if (lane == 0) {
        const int is = qn & 1;
        if (qn >= 2) (void)wait_ok(&c->info_empty[is], ((qn >> 1) - 1) & 1, c, p.status);
        c->info[is] = inf;
        mbar_arrive(&c->info_full[is]);
      }
      __syncwarp();
      return inf;
    };

    int qc = 0, g = 0;
    fetch_ahead(blockIdx.x);
    QInfo cur = prepare(0, blockIdx.x);
    bool ok = true;
    for (int item = blockIdx.x; !cur.done; item += gridDim.x) {
      // query rows: one 8 KB box per lane 0..7
      if (lane == 0 && qc >= 1) ok = wait_ok(&c->q_empty, (qc - 1) & 1, c, p.status);
      ok = __shfl_sync(0xffffffffu, (int)ok, 0);
      if (!ok) break;
      if (lane == 0) mbar_expect_tx(&c->q_full, 8 * kQBlockBytes);
      __syncwarp();
      if (lane < 8)
        tma_load_2d(smem + OFF_Q + lane * kQBlockBytes, &map_q, 64 * lane,
                    (cur.b * p.Sq + cur.t - p.t0) * p.H + kH * cur.hs, &c->q_full);
      const uint16_t* lst = lists + (qc & 1) * kMaxSel;
      QInfo nxt;
      nxt.done = 1;
      for (int j = 0; j < cur.tiles && ok; ++j) {
        const bool window_tile = j == cur.ent_tiles;
        if (window_tile || !gathered) {
          // contiguous rows: lane kb loads K-block kb as soon as its slot is free
          bool lok = true;
          if (lane < kSlots) {
            const int kb = lane;
            if (g >= 1) lok = wait_ok(&c->empty[kb], (g - 1) & 1, c, p.status);
            if (lok) {
              uint8_t* dst = smem + OFF_SLOT + kb * kSlotBytes;
              mbar_expect_tx(&c->full_t[kb], kSlotBytes);
              if (window_tile)
                tma_load_2d(dst, &map_kv, 64 * kb, cur.b * p.S + cur.t - (kTileKeys - 1), &c->full_t[kb]);
              else
                tma_load_2d(dst, &map_ent, 64 * kb, cur.b * p.N + j * kTileKeys, &c->full_t[kb]);
            }
          }
          ok = __all_sync(0xffffffffu, lok);
        } else {
          int sidx[kMaxGroups];
          const int nw = 3;
          load_rows(lst, cur.n_ent, j, 0, nw, lane, sidx);
          for (int kb = 0; kb < kSlots; ++kb) {
            if (lane == 0 && g >= 1) ok = wait_ok(&c->empty[kb], (g - 1) & 1, c, p.status);
            ok = __shfl_sync(0xffffffffu, (int)ok, 0);
            if (!ok) break;
            gather_kblock(smem + OFF_SLOT + kb * kSlotBytes, p.ent + (size_t)cur.b * p.N * kD, sidx, 0, nw, lane,
                          kb, &c->full_g[kb], p.N, p.status);
          }
        }
        if (j == 0) nxt = prepare(qc + 1, item + gridDim.x);
        ++g;
      }
      if (!ok) break;
      ++qc;
      cur = nxt;
      __syncwarp();
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ gather helpers
    const int gw = warp - 1;                  // row groups gw, gw+3, ...
    const bool gathered = p.ratio > 0 && p.idx != nullptr;
    int qc = 0, g = 0;
    bool ok = true;
    while (ok) {
      const int is = qc & 1;
      QInfo inf;
      ok = wait_ok(&c->info_full[is], (qc >> 1) & 1, c, p.status);    // every lane acquires
      ok = __shfl_sync(0xffffffffu, (int)ok, 0);
      inf = c->info[is];
      __syncwarp();
      mbar_arrive(&c->info_empty[is]);
      if (inf.done || !ok) break;
      if (!gathered || inf.ent_tiles == 0) mbar_arrive(&c->list_free[is]);
      const uint16_t* lst = lists + is * kMaxSel;
      const bf16* ent_b = p.ent + (size_t)inf.b * p.N * kD;
      for (int j = 0; j < inf.tiles && ok; ++j) {
        // Contiguous tiles come by TMA alone, but their slot releases are still
        // awaited: a parity wait is only unambiguous one phase ahead.
        const bool contiguous = j == inf.ent_tiles || !gathered;
        int sidx[kMaxGroups];
        const int nw = 3;
        if (!contiguous) {
          load_rows(lst, inf.n_ent, j, gw, nw, lane, sidx);
          if (j == inf.ent_tiles - 1) mbar_arrive(&c->list_free[is]);
        }
        for (int kb = 0; kb < kSlots; ++kb) {
          if (lane == 0 && g >= 1) ok = wait_ok(&c->empty[kb], (g - 1) & 1, c, p.status);
          ok = __shfl_sync(0xffffffffu, (int)ok, 0);
          if (!ok) break;
          if (!contiguous)
            gather_kblock(smem + OFF_SLOT + kb * kSlotBytes, ent_b, sidx, gw, nw, lane, kb, &c->full_g[kb], p.N,
                          p.status);
        }
        ++g;
      }
      ++qc;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id1 = idesc_bf16_f32(128, 64, 0, 0);
      const uint32_t id2 = idesc_bf16_f32(128, 64, 1, 1);
      // descriptors are affine in the start address (14-bit field, no carry
      // below 256 KB): build the bases once, add byte offsets >> 4 per MMA
      const uint64_t dA1 = smem_desc(smem_u32(smem + OFF_SLOT), 16, 1024, kLayoutSW128);
      const uint64_t dQ = smem_desc(smem_u32(smem + OFF_Q), 16, 1024, kLayoutSW128);
      const uint64_t dA2 = smem_desc(smem_u32(smem + OFF_SLOT), kSlotBytes, 1024, kLayoutSW128);
      const uint64_t dP0 = smem_desc(smem_u32(smem + OFF_P), 128, 2048, kLayoutNone);
      const bool gathered = p.ratio > 0 && p.idx != nullptr;
      int qc = 0, g = 0, gg = 0, gt = 0;      // all tiles, gathered tiles, contiguous tiles
      bool ok = true;
      while (ok) {
        const int is = qc & 1;
        ok = wait_ok(&c->info_full[is], (qc >> 1) & 1, c, p.status);
        if (!ok) break;
        const QInfo inf = c->info[is];
        mbar_arrive(&c->info_empty[is]);
        if (inf.done) break;
        ok = wait_ok(&c->q_ready, qc & 1, c, p.status);
        tc_fence_after();
        for (int j = 0; j < inf.tiles && ok; ++j) {
          const int sb = g & 1;
          const uint32_t s_tmem = tmem + 64 * sb;
          const bool contiguous = j == inf.ent_tiles || !gathered;
          uint64_t* fullb = contiguous ? c->full_t : c->full_g;
          const uint32_t fpar = (contiguous ? gt : gg) & 1;
          // The S buffer's TMEM hand-off was fenced after the p_ready wait that
          // freed it; the key tile needs only its full barriers.
          if (contiguous) {
            // TMA writes (async proxy): no proxy fence; the products go out in
            // two runs of 16 once each half of the tile has landed (fewer
            // barrier polls between products: measured 1.002 -> 0.959 ms for
            // the HCA layer at S=16384)
#pragma unroll
            for (int k0 = 0; k0 < kSlots; k0 += kSlots / 2) {
#pragma unroll
              for (int kb = k0; kb < k0 + kSlots / 2; ++kb) ok = ok && wait_ok(&fullb[kb], fpar, c, p.status);
#pragma unroll
              for (int kb = k0; kb < k0 + kSlots / 2; ++kb)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                  umma_f16_ss(s_tmem, dA1 + (uint64_t)((kb * kSlotBytes + 32 * ks) >> 4),
                              dQ + (uint64_t)((kb * kQBlockBytes + 32 * ks) >> 4), id1, (kb | ks) != 0);
            }
          } else {
            // gathered K-blocks, consumed as they land
#pragma unroll
            for (int kb = 0; kb < kSlots; ++kb) {
              ok = ok && wait_ok(&fullb[kb], fpar, c, p.status);
              fence_proxy_async_smem();               // cp.async writes -> tensor-core reads
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                umma_f16_ss(s_tmem, dA1 + (uint64_t)((kb * kSlotBytes + 32 * ks) >> 4),
                            dQ + (uint64_t)((kb * kQBlockBytes + 32 * ks) >> 4), id1, (kb | ks) != 0);
            }
          }
          umma_commit(&c->s_full[sb]);
          if (j == inf.tiles - 1) umma_commit(&c->q_empty);
          if (!ok) break;
          ok = wait_ok(&c->p_ready[sb], (g >> 1) & 1, c, p.status);
          if (ok && j == 0 && qc >= 1) ok = wait_ok(&c->o_empty, (qc - 1) & 1, c, p.status);
          tc_fence_after();
          const uint64_t dP = dP0;                   // one P^T buffer: S(j+1) commits after O(j)
#pragma unroll
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              umma_f16_ss(tmem + 128 + 64 * m, dA2 + (uint64_t)((2 * m * kSlotBytes + 2048 * ks) >> 4),
                          dP + (uint64_t)((256 * ks) >> 4), id2, (j > 0 || ks > 0) ? 1u : 0u);
            umma_commit(&c->empty[2 * m]);
            umma_commit(&c->empty[2 * m + 1]);
          }
          if (contiguous) ++gt; else ++gg;
          ++g;
        }
        umma_commit(&c->o_full);
        ++qc;
      }
      // every issued MMA completes before TMEM is released
      umma_commit(&c->fin);
      mbar_wait(&c->fin, 0, &c->abort, p.status, 200000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Eight warps: two per TMEM lane quarter, head halves hh = 0 / 1 (heads
    // 32*hh .. 32*hh+31 of every row the quarter holds).
    const int ts = threadIdx.x - 128;         // 0..255
    const int quarter = warp & 3;             // TMEM lane quarter of this warp
    const int hh = (warp - 4) >> 2;           // head half
    const int h0 = 32 * hh;
    const int krow = 32 * quarter + lane;     // key row / dim row owned in TMEM
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    const float log2e = 1.4426950408889634f;
    const float c1 = p.scale * log2e;

    // Receive query qc's description; returns false when the work is over.
    auto next_query = [&](int qc, QInfo& inf) -> bool {
      const int is = qc & 1;
      wait_ok(&c->info_full[is], (qc >> 1) & 1, c, p.status);
      inf = c->info[is];
      mbar_arrive(&c->info_empty[is]);
      if (ts == 0) c->decision = (c->abort || inf.done) ? 1 : 0;
      named_bar_sync(1, kSoftThreads);
      const bool more = c->decision == 0;
      named_bar_sync(1, kSoftThreads);
      return more;
    };
    // Rotate the last 64 dims of each head of query qc at position t (four
    // threads per head, two 16-byte chunks each) and publish the rows.
    auto setup_query = [&](int qc, const QInfo& inf) {
      const int h = ts >> 2, part = ts & 3;
      // cos/sin of this thread's 8 rotation pairs, fetched before the wait
      float4 csv[4];
      {
        const float4* csp = reinterpret_cast<const float4*>(p.rope_cs + (size_t)inf.t * (kR / 2) + 8 * part);
#pragma unroll
        for (int i = 0; i < 4; ++i) csv[i] = csp[i];
      }
      wait_ok(&c->q_full, qc & 1, c, p.status);
      uint8_t* qrow = smem + OFF_Q + 7 * kQBlockBytes + h * 128;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int ch = 2 * part + cc;                        // 16-byte chunk of dims 448..511
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
      mbar_arrive(&c->q_ready);                // the products wait for all 256 arrivals
    };

    int qc = 0, g = 0;
    QInfo inf;
    bool more = next_query(0, inf);
    if (more) setup_query(0, inf);
    while (more) {
      const float* mlog2 = c->mlog2[qc & 1] + h0;
      const int t = inf.t, b = inf.b, hsl = inf.hs;
      const int nk_total = inf.n_ent + (t - inf.w_lo + 1);
      float lsum = 0.f;                         // this warp's denominator of head h0 + lane
      for (int j = 0; j < inf.tiles; ++j) {
        int sb = g & 1;
        bool valid;
        if (j < inf.ent_tiles) {
          valid = j * kTileKeys + krow < inf.n_ent;
        } else {
          const int u = t - (kTileKeys - 1) + krow;
          valid = u >= inf.w_lo && u <= t;
        }
        wait_ok(&c->s_full[sb], (g >> 1) & 1, c, p.status);
        tc_fence_after();
        float v[32];
        if (!V4_BOUND(64 * sb + h0 + 32 <= 128, p.status)) sb = 0;     // S columns [0, 128)
        tmem_ld32(tmem + lane_base + 64 * sb + h0, v);
        tmem_wait_ld();
        if (j == 0) {
          // the query's shift: each head's largest logit over this tile's
          // valid keys (the tile always holds one: entry 0 or the query's
          // own token).  Five butterfly rounds leave lane L with head h0 + L
          // of this warp's 32 rows, the four lane quarters meet in shared
          // memory.
          float r[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = valid ? v[i] : -INFINITY;
#pragma unroll
          for (int o = 16, w = 16; o >= 1; o >>= 1, w >>= 1) {
            const bool hi = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < w; ++i) {
              const float send = hi ? r[i] : r[w + i];
              const float keep = hi ? r[w + i] : r[i];
              r[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
            }
          }
          c->hmax[quarter][h0 + lane] = r[0];
          named_bar_sync(1, kSoftThreads);
          // lane L publishes head h0 + L's shift for its warp (the four
          // warps of a head half write the same values)
          const int hd = h0 + lane;
          float m = fmaxf(fmaxf(c->hmax[0][hd], c->hmax[1][hd]), fmaxf(c->hmax[2][hd], c->hmax[3][hd])) * c1;
          if (p.sink != nullptr) m = fmaxf(m, p.sink[kH * hsl + hd] * log2e);
          c->mlog2[qc & 1][hd] = m;
          __syncwarp();
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0 = valid ? ex2_approx(fmaf(v[2 * i], c1, -mlog2[2 * i])) : 0.f;
          float x1 = valid ? ex2_approx(fmaf(v[2 * i + 1], c1, -mlog2[2 * i + 1])) : 0.f;
          pk[i] = pack_bf16x2(x0, x1);
        }
        // P^T [8-head column block][key]: this half's four blocks
        // (one buffer: this tile's S completing implies the previous tile's
        // O products, issued before it, have completed too)
        uint8_t* prow = smem + OFF_P + krow * 16 + (4 * hh) * 2048;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          if (V4_BOUND(krow * 16 + (4 * hh + cc) * 2048 + 16 <= (int)kPBytes, p.status))
            *reinterpret_cast<uint4*>(prow + cc * 2048) =
                make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&c->p_ready[sb]);
        // Sum the warp's 32 rows per head while the products run: five
        // butterfly rounds, each lane keeping half of its heads, leave lane L
        // with head h0 + L (pk[i] packs heads h0 + 2i, h0 + 2i + 1).
        {
          float r[16];
          const bool up = (lane & 16) != 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t keep = up ? pk[8 + i] : pk[i];
            const uint32_t got = __shfl_xor_sync(0xffffffffu, up ? pk[i] : pk[8 + i], 16);
            r[2 * i] = __uint_as_float(keep << 16) + __uint_as_float(got << 16);
            r[2 * i + 1] = __uint_as_float(keep & 0xFFFF0000u) + __uint_as_float(got & 0xFFFF0000u);
          }
#pragma unroll
          for (int o = 8, w = 8; o >= 1; o >>= 1, w >>= 1) {
            const bool hi = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < w; ++i) {
              const float send = hi ? r[i] : r[w + i];
              const float keep = hi ? r[w + i] : r[i];
              r[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
          }
          lsum += r[0];
        }
        ++g;
      }

      // the next query's queries go first, so its first products overlap
      // this query's epilogue
      QInfo nxt;
      more = next_query(qc + 1, nxt);
      if (more) setup_query(qc + 1, nxt);

      // ---- epilogue: denominators, lse, O^T / l, de-rotation, store
      // de-rotation of this thread's dim pair (M-block 3 holds dims 384..511)
      float dc = 1.f, ds = 0.f;
      const int dim3 = 384 + krow;
      if (dim3 >= kD - kR) {
        const float2 cs = p.rope_cs[(size_t)t * (kR / 2) + ((dim3 - (kD - kR)) >> 1)];
        dc = cs.x;
        ds = cs.y;
      }
      wait_ok(&c->o_full, qc & 1, c, p.status);
      tc_fence_after();
      // per-head scalars, one head per thread; the P buffers are idle here:
      // [0,256) the four quarter partials of l, [256,320) 1/l
      float* hs = reinterpret_cast<float*>(smem + OFF_P);
      const float* mlog2_all = c->mlog2[qc & 1];
      hs[64 * quarter + h0 + lane] = lsum;
      named_bar_sync(1, kSoftThreads);
      if (ts < kH) {
        float l = (hs[ts] + hs[64 + ts]) + (hs[128 + ts] + hs[192 + ts]);
        const float m = mlog2_all[ts] * 0.6931471805599453f;
        if (p.sink != nullptr) l += expf(p.sink[kH * hsl + ts] - m);
        // too little mass under the shift (exp underflow may have lost keys)
        // or so much above it that the fp32 output sums could overflow
        const bool bad = !(l >= (float)nk_total * 1.0e-26f) || !(l < 0x1p100f);
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&c->redo, 1);
        if (p.lse) p.lse[((size_t)b * p.Sq + t - p.t0) * p.H + kH * hsl + ts] = m + logf(l);
        hs[256 + ts] = 1.0f / l;
      }
      named_bar_sync(1, kSoftThreads);
      if (ts == 0 && c->redo) {                 // queue the query once for the running-max kernel
        const int slot = atomicAdd(&p.counters[1], 1);
        if (V4_BOUND(slot < p.B * p.Sq * p.HS, p.status)) p.counters[2 + slot] = b * p.Sq + t - p.t0;
        c->redo = 0;
      }
      float inv_l[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 v4 = *reinterpret_cast<const float4*>(hs + 256 + h0 + i);
        inv_l[i] = v4.x;
        inv_l[i + 1] = v4.y;
        inv_l[i + 2] = v4.z;
        inv_l[i + 3] = v4.w;
      }
      // o[t, h, 128m + krow]: for each head the 32 lanes of a warp write 64
      // contiguous bytes
      bf16* obase = p.o + (((size_t)b * p.Sq + t - p.t0) * p.H + kH * hsl + h0) * kD + krow;
      for (int m = 0; m < 4; ++m) {
        float v[32];
        if (!V4_BOUND(128 + 64 * m + h0 + 32 <= 384, p.status)) break;   // O columns [128, 384)
        tmem_ld32(tmem + lane_base + 128 + 64 * m + h0, v);
        tmem_wait_ld();
        if (m == 3) {
          tc_fence_before();
          mbar_arrive(&c->o_empty);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= inv_l[i];
        if (m == 3 && quarter >= 2) {
          // rotated dims 448..511: the partner of each pair is the
          // neighbouring lane; the values cross through the idle P buffer
          // (after the per-head scalars), sixteen heads per round
          float4* xb = reinterpret_cast<float4*>(smem + OFF_P + 2048 + (2 * (quarter - 2) + hh) * 2048);
          const bool odd = lane & 1;
#pragma unroll
          for (int rnd = 0; rnd < 2; ++rnd) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const int i = 16 * rnd + 4 * c4;
              xb[c4 * 32 + lane] = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
            }
            __syncwarp();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const float4 o4 = xb[c4 * 32 + (lane ^ 1)];
              const float oth[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = 16 * rnd + 4 * c4 + e;
                v[i] = odd ? (v[i] * dc - oth[e] * ds) : (v[i] * dc + oth[e] * ds);
              }
            }
            __syncwarp();
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) obase[(size_t)i * kD + 128 * m] = __float2bfloat16_rn(v[i]);
      }
      named_bar_sync(1, kSoftThreads);          // the scalars in the P buffers are read; P may be rewritten
      inf = nxt;
      ++qc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// host side: tensor maps and launch
// ---------------------------------------------------------------------------
}  // namespace

cudaError_t launch_mqa_tc(const v4_config& cfg, const void* q, const void* kv_rot, const void* ent,
                          const int32_t* idx, const float* sink, const float2* cs_table, void* o, float* lse,
                          int* counters, int* status, cudaStream_t st) {
  const int B = cfg.batch, S = cfg.seqlen;
  const int N = cfg.ratio > 0 ? S / cfg.ratio : 0;
  CUtensorMap mq, mkv, ment;
  const uint64_t qrows = (uint64_t)B * q_rows(cfg) * cfg.n_heads;
  int e = 0;
  e |= make_tmap_bf16_2d(&mq, q, kD, qrows, 64, 64, true);
  e |= make_tmap_bf16_2d(&mkv, kv_rot, kD, (uint64_t)B * S, 64, kTileKeys, true);
  const void* ent_base = (ent != nullptr && N > 0) ? ent : kv_rot;      // unused when there are no entries
  const uint64_t ent_rows = (ent != nullptr && N > 0) ? (uint64_t)B * N : (uint64_t)B * S;
  e |= make_tmap_bf16_2d(&ment, ent_base, kD, ent_rows, 64, kTileKeys, true);
  if (e) return cudaErrorInvalidValue;
  Params prm;
  prm.q = (const bf16*)q;
  prm.ent = (const bf16*)ent_base;
  prm.o = (bf16*)o;
  prm.idx = idx;
  prm.sink = sink;
  prm.rope_cs = cs_table;
  prm.reserved0 = nullptr;
  prm.reserved1 = nullptr;
  prm.lse = lse;
  prm.status = status;
  prm.counters = counters;
  prm.B = B;
  prm.S = S;
  prm.N = N;
  prm.ratio = cfg.ratio;
  prm.window = cfg.window;
  prm.K = cfg.topk;
  prm.H = cfg.n_heads;
  prm.HS = cfg.n_heads / kH;
  prm.Sq = q_rows(cfg);
  prm.t0 = cfg.q_begin;
  prm.scale = cfg.softmax_scale > 0.f ? cfg.softmax_scale : 1.0f / sqrtf((float)kD);
  cudaError_t err = cudaFuncSetAttribute(mqa_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long total = (long long)B * q_rows(cfg) * (cfg.n_heads / kH);
  const int grid = (int)(total < sms ? total : sms);
  err = cudaMemsetAsync(counters + 1, 0, sizeof(int), st);
  if (err != cudaSuccess) return err;
  mqa_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mq, mkv, ment, prm);
  note_launch();
  return cudaGetLastError();
}

bool mqa_tc_supported(const v4_config& c) {
  return c.dtype == V4_BF16 && c.n_heads >= kH && c.n_heads % kH == 0 && c.n_heads <= 8 * kH &&
         c.head_dim == kD && c.rope_dim == kR &&
         c.window >= 1 && c.window <= kTileKeys && c.topk <= kMaxSel && (c.ratio == 0 || c.ratio >= 1) &&
         (c.topk == 0 || c.ratio == 0 || c.seqlen / c.ratio <= 65536);    // 16-bit selection lists
}

}  // namespace v4
