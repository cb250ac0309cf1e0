// Backward of the sparse / dense multi-query attention on the 5th-generation
// tensor cores (tcgen05, TMEM accumulators, TMA) for the DeepSeek-V4 shapes:
// query heads in slices of 64 sharing one 512-d latent that is both key and
// value, the last 64 dims rotated, bf16 storage, window <= 128.
//
// Method: "Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X GPUs
// with Primus", section "Attention kernels for the three layer types"
// (backward): a dQ pass that regathers the selected entries and recomputes
// the softmax, the delta rowsum(O * dO) folded in ahead of it, and a
// head-dimension contraction ("interm") whose result is scattered into the
// key/value gradient.  Here the contraction and the scatter are fused into
// the dQ kernel: each (query, key) pair's 512-d gradient is reduced into an
// fp32 accumulator in L2 (red.global.add), so the intermediate tensor never
// reaches HBM.
//
// Per query t and 64-head slice (one CTA, persistent over queries), keys in
// tiles of 32 (the query's selected or visible entries, then its window):
//   [S; dP] = [Qr; dO'] . K^T               (M = 128 = 64 heads + 64 heads, N = 32 keys)
//   P  = exp(scale S - lse),  dS = scale P (dP - delta)          (fp32, in registers)
//   dQ^T  += K^T . dS^T                     (4 x M=128 dims, N = 64 heads, K = 32 keys)
//   dKV^T  = [Qr; dO']^T . [dS; P]          (4 x M=128 dims, N = 32 keys, K = 128)
// Qr = rot(q, t) and dO' = rot(dO, t) are written by a prep kernel that also
// forms delta = dO . o and the sink gradient.  The [Qr; dO'] block (128 KB,
// 128-byte swizzle) is the K-major A operand of the first product and, read
// as MN-major, the A operand of the last; the key tile is K-major B of the
// first and MN-major A of the second.  [dS; P] is written once in a
// no-swizzle core-matrix layout that is the K-major B of dQ^T (rows 0..63)
// and the MN-major B of dKV^T.  TMEM: [S; dP] double buffer (2 x 32
// columns), dQ^T (256), dKV^T (128).
//
// Warp roles (384 threads): warp 0 producer (per-query selection list, [Qr; dO']
// by TMA, a third of the key gathers), warp 1 MMA issuer and TMEM owner,
// warps 2-3 the other gathers, warps 4-7 softmax (TMEM lane quarters 0-1
// hold the S rows, 2-3 the dP rows; P crosses through shared memory; they
// also reduce keys 16..31 of each dKV^T tile), warps 8-11 reduce keys 0..15
// and write dQ.  Element-wise fp32 reductions from the SM reach the L2's
// rate only with many warps issuing them: four warps alone measured about
// 14 GB/s per SM and bounded the whole kernel.
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
constexpr int kT = 32;                            // keys per tile
constexpr int kGatherLanes = 96;                  // warps 0, 2, 3
constexpr int kSoftThreads = 128;                 // warps 4-7
constexpr int kEpiThreads = 128;                  // warps 8-11
constexpr uint32_t kABlock = 128 * 128;           // [Qr; dO'] K-block: 128 rows x 64 dims x 2 B
constexpr uint32_t kKBlock = kT * 128;            // key K-block: 32 keys x 64 dims x 2 B
constexpr uint32_t kKBuf = 8 * kKBlock;           // one key tile
constexpr uint32_t kDSBytes = 128 * kT * 2;       // [dS; P]: 128 rows x 32 keys x 2 B
constexpr uint32_t kPSBytes = kH * kT * 4;        // P in fp32: 64 heads x 32 keys
constexpr int kMaxSel = 1024;

constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_K = OFF_A + 8 * kABlock;             // 131072
constexpr uint32_t OFF_DS = OFF_K + 2 * kKBuf;              // 196608
constexpr uint32_t OFF_PS = OFF_DS + kDSBytes;              // 204800 (two buffers)
constexpr uint32_t OFF_LIST = OFF_PS + 2 * kPSBytes;        // 221184
constexpr uint32_t OFF_CTL = OFF_LIST + 2 * kMaxSel * 4;    // 229376

// TMEM columns
constexpr uint32_t TM_SD = 0;        // [S; dP] buffers at 0 and 32
constexpr uint32_t TM_DQ = 64;       // dQ^T: 64 + 64 m
constexpr uint32_t TM_DKV = 320;     // dKV^T: 320 + 32 m

struct QInfo {
  int b, t, hs, n_ent, w_lo, n_keys, tiles, done;
  int listed;                   // entries come from the selection list (else 0 .. n_ent-1)
};

// Accumulator row of key k of a query: its entries first (selection list or
// all visible), then its window tokens.  Rows [0, B*N) are entries, rows
// B*N + b*S + u window tokens.
__device__ __forceinline__ int key_row(const QInfo& q, const int32_t* lst, int k, int N, int S, int BN) {
  if (k < q.n_ent) return q.listed ? lst[k] : q.b * N + k;
  return BN + q.b * S + q.w_lo + (k - q.n_ent);
}

struct Ctl {
  uint64_t a_full, a_empty;
  uint64_t kfull[2], kempty[2];
  uint64_t s_full[2], sd_empty[2];
  uint64_t ds_ready, ds_free;
  uint64_t dkv_full, dkv_empty[4];
  uint64_t dq_full, dq_empty;
  uint64_t info_full[2], info_empty[2];
  uint64_t list_free[2];
  uint64_t fin;
  QInfo info[2];
  uint32_t tmem_base;
  int abort;
};

constexpr uint32_t kSmemBytes = OFF_CTL + sizeof(Ctl);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  const bf16* ent;             // [B*N, 512] rotated entries
  const bf16* kr;              // [B*S, 512] rotated window keys
  const int32_t* idx;          // [B,S,K] or null (every visible entry)
  const float* lse;            // [B,S,H]
  const float* delta;          // [B,S,H]
  const float2* rope_cs;       // [S][32] cos/sin
  bf16* dq;                    // [B,S,H,512]
  float* dent;                 // [B*N, 512] accumulators
  float* dkr;                  // [B*S, 512] accumulators (gradient of the rotated window keys)
  int* status;
  int B, S, N, ratio, window, K;
  int H, HS;
  float scale;
};

__device__ __forceinline__ bool wait_ok(uint64_t* bar, uint32_t parity, Ctl* c, int* status) {
  return mbar_wait(bar, parity, &c->abort, status);
}

// Gather key tile j of a query into a key buffer: 32 rows x 8 16-byte chunks
// per 64-dim K-block; gather lane gl (of 96) takes (row, chunk) pairs gl,
// gl + 96, gl + 192 across all eight K-blocks.  Rows past the query's last
// key repeat the tile's first key (finite values; their P and dS are zero).
// One arrival on `full` when this lane's copies have landed.
__device__ __forceinline__ void gather_tile(uint8_t* kbuf, const QInfo& q, const int32_t* lst, int j, int gl,
                                            const bf16* ent, const bf16* kr, int N, int S, int BN,
                                            uint64_t* full, int kv_rows, int* status) {
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int pr = gl + kGatherLanes * i;
    if (pr < kT * 8) {
      const int row = pr >> 3, ch = pr & 7;
      int k = j * kT + row;
      if (k >= q.n_keys) k = j * kT;
      const int r = key_row(q, lst, k, N, S, BN);
      const bf16* src = (r < BN ? ent + (size_t)r * kD : kr + (size_t)(r - BN) * kD) + ch * 8;
      const uint32_t d0 = smem_u32(kbuf) + row * 128 + ((ch ^ (row & 7)) << 4);
      if (V4_BOUND(r >= 0 && r < BN + kv_rows, status)) {
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) cp_async_16(d0 + kb * kKBlock, src + kb * 64);
      }
    }
  }
  cp_async_mbar_arrive(full);
}

// Reduce keys [k0, k0 + 16) of tile j's dKV^T (all four M-blocks) into the
// fp32 accumulators and release each M-block's TMEM columns.  The warp's 32
// TMEM lanes are 32 consecutive dims of an M-block: one warp-wide 128-byte
// reduction per key.  Keys past the query's last carry exact zeros; they add
// into the tile's first key row, so the loop has no branch.
__device__ __forceinline__ void drain_dkv(uint32_t t_dkv, int k0, const QInfo& q, const int32_t* lst, int j,
                                          int lane, int quarter, const Params& p, int BN, Ctl* c) {
  const int kk = kT * j + k0 + (lane & 15);
  const int rid = key_row(q, lst, kk < q.n_keys ? kk : kT * j, p.N, p.S, BN);
  float* rowp = rid < BN ? p.dent + (size_t)rid * kD : p.dkr + (size_t)(rid - BN) * kD;
  const unsigned long long rowv = reinterpret_cast<unsigned long long>(rowp);
#pragma unroll 1
  for (int m = 0; m < 4; ++m) {
    float v[16];
    tmem_ld16(t_dkv + kT * m + k0, v);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(&c->dkv_empty[m]);
    const int d = 128 * m + 32 * quarter + lane;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      float* dst = reinterpret_cast<float*>(__shfl_sync(0xffffffffu, rowv, k)) + d;
      atomicAdd(dst, v[k]);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
mqa_bwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                  const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctl* c = reinterpret_cast<Ctl*>(smem + OFF_CTL);
  int32_t* lists = reinterpret_cast<int32_t*>(smem + OFF_LIST);   // [2][kMaxSel] selections, by query parity
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0) {          // swizzled operands need 1 KB alignment
    if (threadIdx.x == 0) set_status(p.status, V4_ERR_UNSUPPORTED);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&c->a_full, 1);
    mbar_init(&c->a_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->kfull[i], kGatherLanes);
      mbar_init(&c->kempty[i], 1);
      mbar_init(&c->s_full[i], 1);
      mbar_init(&c->sd_empty[i], kSoftThreads);
      mbar_init(&c->info_full[i], 1);
      mbar_init(&c->info_empty[i], 64 + 1 + kSoftThreads + kEpiThreads);
      mbar_init(&c->list_free[i], 64 + kSoftThreads + kEpiThreads);
    }
    mbar_init(&c->ds_ready, kSoftThreads);
    mbar_init(&c->ds_free, 1);
    mbar_init(&c->dkv_full, 1);
    for (int m = 0; m < 4; ++m) mbar_init(&c->dkv_empty[m], kSoftThreads + kEpiThreads);
    mbar_init(&c->dq_full, 1);
    mbar_init(&c->dq_empty, kEpiThreads);
    mbar_init(&c->fin, 1);
    c->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_q);
    prefetch_tmap(&map_do);
  }
  if (warp == 1) {
    tmem_alloc(&c->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c->tmem_base;
  const int total = p.B * p.S * p.HS;        // work items: (query, head slice)
  const int BN = p.B * p.N;

  // Every consumer copies the query's description and releases the slot.
  auto receive = [&](int qc, QInfo& inf) -> bool {
    const int is = qc & 1;
    const bool ok = wait_ok(&c->info_full[is], (qc >> 1) & 1, c, p.status);
    inf = c->info[is];
    mbar_arrive(&c->info_empty[is]);
    return ok && !inf.done;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Query qc+1's selection list is compacted and published while query
    // qc's first tile loads; lists alternate between two buffers.
    auto prepare = [&](int qn, int it) -> QInfo {
      QInfo inf;
      inf.done = it >= total ? 1 : 0;
      inf.b = inf.done ? 0 : (it / p.HS) % p.B;
      inf.t = inf.done ? 0 : p.S - 1 - (it / p.HS) / p.B;
      inf.hs = inf.done ? 0 : it % p.HS;
      int n = 0;
      inf.listed = p.ratio > 0 && p.idx != nullptr;
      inf.w_lo = 0;
      if (!inf.done) {
        if (lane == 0 && qn >= 2) (void)wait_ok(&c->list_free[qn & 1], ((qn >> 1) - 1) & 1, c, p.status);
        __syncwarp();
        int32_t* lst = lists + (qn & 1) * kMaxSel;
        const int t = inf.t, b = inf.b;
        const int nv = p.ratio > 0 ? min((t + 1) / p.ratio, p.N) : 0;
        const unsigned below = (1u << lane) - 1u;
        if (inf.listed) {
          // every load first, then the ballots: one memory latency per row
          const int32_t* row = p.idx + ((size_t)b * p.S + t) * p.K;
          int sv[kMaxSel / 32];
#pragma unroll
          for (int i = 0; i < kMaxSel / 32; ++i) sv[i] = 32 * i + lane < p.K ? row[32 * i + lane] : -1;
#pragma unroll
          for (int i = 0; i < kMaxSel / 32; ++i) {
            int v = sv[i];
            if (v < -1 || v >= nv) {
              set_status(p.status, kStatusBadIndex);
              v = -1;
            }
            const unsigned msk = __ballot_sync(0xffffffffu, v >= 0);
            if (v >= 0) lst[n + __popc(msk & below)] = b * p.N + v;
            n += __popc(msk);
          }
        } else {
          n = nv;
        }
        inf.w_lo = max(0, t - p.window + 1);
        __syncwarp();
      }
      inf.n_ent = n;
      inf.n_keys = inf.done ? 0 : n + (inf.t - inf.w_lo + 1);
      inf.tiles = (inf.n_keys + kT - 1) / kT;
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
    QInfo cur = prepare(0, blockIdx.x);
    bool ok = true;
    for (int item = blockIdx.x; !cur.done; item += gridDim.x) {
      // [Qr; dO'] rows of this query and head slice: sixteen 8 KB boxes
      if (lane == 0 && qc >= 1) ok = wait_ok(&c->a_empty, (qc - 1) & 1, c, p.status);
      ok = __shfl_sync(0xffffffffu, (int)ok, 0);
      if (!ok) break;
      if (lane == 0) mbar_expect_tx(&c->a_full, 8 * kABlock);
      __syncwarp();
      if (lane < 16) {
        const int kb = lane & 7;
        const int y = (cur.b * p.S + cur.t) * p.H + kH * cur.hs;
        if (lane < 8)
          tma_load_2d(smem + OFF_A + kb * kABlock, &map_q, 64 * kb, y, &c->a_full);
        else
          tma_load_2d(smem + OFF_A + kb * kABlock + 64 * 128, &map_do, 64 * kb, y, &c->a_full);
      }
      const int32_t* lst = lists + (qc & 1) * kMaxSel;
      QInfo nxt;
      nxt.done = 1;
      for (int j = 0; j < cur.tiles; ++j) {
        if (lane == 0 && g >= 2) ok = wait_ok(&c->kempty[g & 1], ((g >> 1) - 1) & 1, c, p.status);
        ok = __shfl_sync(0xffffffffu, (int)ok, 0);
        if (!ok) break;
        gather_tile(smem + OFF_K + (g & 1) * kKBuf, cur, lst, j, lane, p.ent, p.kr, p.N, p.S, BN, &c->kfull[g & 1],
                    p.B * p.S, p.status);
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
    const int gl = 32 * (warp - 1) + lane;
    int qc = 0, g = 0;
    QInfo inf;
    while (receive(qc, inf)) {
      const int is = qc & 1;
      const int32_t* lst = lists + is * kMaxSel;
      bool ok = true;
      for (int j = 0; j < inf.tiles; ++j) {
        if (lane == 0 && g >= 2) ok = wait_ok(&c->kempty[g & 1], ((g >> 1) - 1) & 1, c, p.status);
        ok = __shfl_sync(0xffffffffu, (int)ok, 0);
        if (!ok) break;
        gather_tile(smem + OFF_K + (g & 1) * kKBuf, inf, lst, j, gl, p.ent, p.kr, p.N, p.S, BN, &c->kfull[g & 1],
                    p.B * p.S, p.status);
        ++g;
      }
      mbar_arrive(&c->list_free[is]);
      if (!ok) break;
      ++qc;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id1 = idesc_bf16_f32(128, kT, 0, 0);    // [S; dP]
      const uint32_t id2 = idesc_bf16_f32(128, kH, 1, 0);    // dQ^T
      const uint32_t id3 = idesc_bf16_f32(128, kT, 1, 1);    // dKV^T
      // descriptors are affine in the start address (14-bit field, no carry
      // below 256 KB): build the bases once, add byte offsets >> 4 per MMA
      const uint64_t dA1 = smem_desc(smem_u32(smem + OFF_A), 16, 1024, kLayoutSW128);
      const uint64_t dB1 = smem_desc(smem_u32(smem + OFF_K), 16, 1024, kLayoutSW128);
      const uint64_t dA2 = smem_desc(smem_u32(smem + OFF_K), kKBlock, 1024, kLayoutSW128);
      const uint64_t dB2 = smem_desc(smem_u32(smem + OFF_DS), 2048, 128, kLayoutNone);
      const uint64_t dA3 = smem_desc(smem_u32(smem + OFF_A), kABlock, 1024, kLayoutSW128);
      const uint64_t dB3 = smem_desc(smem_u32(smem + OFF_DS), 128, 2048, kLayoutNone);
      bool ok = true;
      auto issue_s = [&](int gg) {
        const int kbuf = gg & 1;
        ok = ok && wait_ok(&c->kfull[kbuf], (gg >> 1) & 1, c, p.status);
        if (gg >= 2) ok = ok && wait_ok(&c->sd_empty[kbuf], ((gg >> 1) - 1) & 1, c, p.status);
        fence_proxy_async_smem();                 // cp.async writes -> tensor-core reads
        tc_fence_after();
#pragma unroll
        for (int kb = 0; kb < 8; ++kb)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_f16_ss(tmem + TM_SD + kT * kbuf, dA1 + (uint64_t)((kb * kABlock + 32 * ks) >> 4),
                        dB1 + (uint64_t)((kbuf * kKBuf + kb * kKBlock + 32 * ks) >> 4), id1, (kb | ks) != 0);
        umma_commit(&c->s_full[kbuf]);
      };
      int qc = 0, g = 0;
      QInfo inf;
      while (ok && receive(qc, inf)) {
        ok = wait_ok(&c->a_full, qc & 1, c, p.status);
        tc_fence_after();
        issue_s(g);
        for (int j = 0; j < inf.tiles && ok; ++j) {
          const int gj = g + j, kbuf = gj & 1;
          if (j + 1 < inf.tiles) issue_s(gj + 1);
          ok = ok && wait_ok(&c->ds_ready, gj & 1, c, p.status);
          if (j == 0 && qc >= 1) ok = ok && wait_ok(&c->dq_empty, (qc - 1) & 1, c, p.status);
          tc_fence_after();
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks)
              umma_f16_ss(tmem + TM_DQ + 64 * m,
                          dA2 + (uint64_t)((kbuf * kKBuf + 2 * m * kKBlock + 2048 * ks) >> 4),
                          dB2 + (uint64_t)((4096 * ks) >> 4), id2, (j > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            if (gj >= 1) ok = ok && wait_ok(&c->dkv_empty[m], (gj - 1) & 1, c, p.status);
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              umma_f16_ss(tmem + TM_DKV + kT * m, dA3 + (uint64_t)((2 * m * kABlock + 2048 * ks) >> 4),
                          dB3 + (uint64_t)((256 * ks) >> 4), id3, ks > 0 ? 1u : 0u);
          }
          umma_commit(&c->dkv_full);
          umma_commit(&c->kempty[kbuf]);
          umma_commit(&c->ds_free);
          if (j == inf.tiles - 1) {
            umma_commit(&c->dq_full);
            umma_commit(&c->a_empty);
          }
        }
        g += inf.tiles;
        ++qc;
      }
      // every issued MMA completes before TMEM is released
      umma_commit(&c->fin);
      mbar_wait(&c->fin, 0, &c->abort, p.status, 200000000ull);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax
    // Quarter 0-1 threads own S rows (head h), quarter 2-3 threads the dP
    // rows of the same heads; P crosses in fp32 through shared memory.
    const int quarter = warp & 3;
    const bool is_s = quarter < 2;
    const int h = 32 * (quarter & 1) + lane;
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    const float log2e = 1.4426950408889634f;
    const float c1 = p.scale * log2e;
    int qc = 0, g = 0;
    QInfo inf;
    while (receive(qc, inf)) {
      const int32_t* lst = lists + (qc & 1) * kMaxSel;
      const size_t hrow = ((size_t)inf.b * p.S + inf.t) * p.H + kH * inf.hs + h;
      const float lse2 = is_s ? p.lse[hrow] * log2e : 0.f;
      const float dlt = is_s ? 0.f : p.delta[hrow];
      for (int j = 0; j < inf.tiles; ++j) {
        const int gj = g + j, sb = gj & 1;
        const int nvalid = min(kT, inf.n_keys - kT * j);
        wait_ok(&c->s_full[sb], (gj >> 1) & 1, c, p.status);
        tc_fence_after();
        float v[32];
        tmem_ld32(tmem + lane_base + TM_SD + kT * sb, v);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&c->sd_empty[sb]);
        float* ps = reinterpret_cast<float*>(smem + OFF_PS + sb * kPSBytes) + h * kT;
        float x[32];
        if (is_s) {
#pragma unroll
          for (int k = 0; k < 32; ++k) x[k] = k < nvalid ? ex2_approx(fmaf(v[k], c1, -lse2)) : 0.f;
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            *reinterpret_cast<float4*>(ps + 4 * (c4 ^ (h & 7))) =
                make_float4(x[4 * c4], x[4 * c4 + 1], x[4 * c4 + 2], x[4 * c4 + 3]);
        }
        named_bar_sync(2, kSoftThreads);
        if (!is_s) {
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 f = *reinterpret_cast<const float4*>(ps + 4 * (c4 ^ (h & 7)));
            x[4 * c4] = p.scale * f.x * (v[4 * c4] - dlt);
            x[4 * c4 + 1] = p.scale * f.y * (v[4 * c4 + 1] - dlt);
            x[4 * c4 + 2] = p.scale * f.z * (v[4 * c4 + 2] - dlt);
            x[4 * c4 + 3] = p.scale * f.w * (v[4 * c4 + 3] - dlt);
          }
        }
        // [dS; P] row (dS rows 0..63, P rows 64..127): 8-key core-matrix
        // columns 2048 B apart, 8-row groups 128 B apart
        if (gj >= 1) wait_ok(&c->ds_free, (gj - 1) & 1, c, p.status);
        const int row = is_s ? 64 + h : h;
        uint8_t* base = smem + OFF_DS + (row >> 3) * 128 + (row & 7) * 16;
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8)
          *reinterpret_cast<uint4*>(base + c8 * 2048) =
              make_uint4(pack_bf16x2(x[8 * c8], x[8 * c8 + 1]), pack_bf16x2(x[8 * c8 + 2], x[8 * c8 + 3]),
                         pack_bf16x2(x[8 * c8 + 4], x[8 * c8 + 5]), pack_bf16x2(x[8 * c8 + 6], x[8 * c8 + 7]));
        fence_proxy_async_smem();
        mbar_arrive(&c->ds_ready);
        // keys 16..31 of the previous tile's dKV^T (its products completed
        // with the ds_free phase waited above); the query's last tile is
        // drained once its products finish
        if (j >= 1) {
          wait_ok(&c->dkv_full, (gj - 1) & 1, c, p.status);
          tc_fence_after();
          drain_dkv(tmem + lane_base + TM_DKV, 16, inf, lst, j - 1, lane, quarter, p, BN, c);
        }
        if (j == inf.tiles - 1) {
          wait_ok(&c->dkv_full, gj & 1, c, p.status);
          tc_fence_after();
          drain_dkv(tmem + lane_base + TM_DKV, 16, inf, lst, j, lane, quarter, p, BN, c);
          mbar_arrive(&c->list_free[qc & 1]);
        }
      }
      g += inf.tiles;
      ++qc;
    }
  } else {
    // ------------------------------------------------------------ dKV reduction + dQ epilogue
    const int quarter = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    int qc = 0, g = 0;
    QInfo inf;
    while (receive(qc, inf)) {
      const int is = qc & 1;
      const int32_t* lst = lists + is * kMaxSel;
      for (int j = 0; j < inf.tiles; ++j) {
        const int gj = g + j;
        wait_ok(&c->dkv_full, gj & 1, c, p.status);
        tc_fence_after();
        drain_dkv(tmem + lane_base + TM_DKV, 0, inf, lst, j, lane, quarter, p, BN, c);      // keys 0..15
        if (j == inf.tiles - 1) mbar_arrive(&c->list_free[is]);
      }
      g += inf.tiles;
      // dQ^T [dim, head]: de-rotate the last 64 dims at -t, store bf16
      wait_ok(&c->dq_full, qc & 1, c, p.status);
      tc_fence_after();
      bf16* dqb = p.dq + (((size_t)inf.b * p.S + inf.t) * p.H + kH * inf.hs) * kD;
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        const int d = 128 * m + 32 * quarter + lane;
        float dc = 1.f, dsn = 0.f;
        const bool rot = d >= kD - kR;                 // warp-uniform (m = 3, quarters 2-3)
        if (rot) {
          const float2 cs = p.rope_cs[(size_t)inf.t * (kR / 2) + ((d - (kD - kR)) >> 1)];
          dc = cs.x;
          dsn = cs.y;
        }
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          float v[32];
          tmem_ld32(tmem + lane_base + TM_DQ + 64 * m + 32 * hf, v);
          tmem_wait_ld();
          if (rot) {
            const bool odd = lane & 1;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float o = __shfl_xor_sync(0xffffffffu, v[i], 1);
              v[i] = odd ? (v[i] * dc - o * dsn) : (v[i] * dc + o * dsn);
            }
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) dqb[(size_t)(32 * hf + i) * kD + d] = __float2bfloat16_rn(v[i]);
        }
      }
      tc_fence_before();
      mbar_arrive(&c->dq_empty);
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
// Prep: Qr = rot(q, t), dO' = rot(dO, t), delta = dO . o per (query, head),
// and the sink gradient -sum_t exp(sink - lse) delta.  One warp per row,
// 16 dims per lane (two 8-dim chunks); the grid's warp count is a multiple
// of H so that each warp keeps one head and adds its sink share once.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
mqa_bwd_prep_kernel(const bf16* __restrict__ q, const bf16* __restrict__ o, const bf16* __restrict__ dout,
                    const float* __restrict__ lse, const float* __restrict__ sink, const float2* __restrict__ cs,
                    bf16* __restrict__ qr, bf16* __restrict__ dor, float* __restrict__ delta,
                    float* __restrict__ dsink, long long rows, int S, int H) {
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  const long long w0 = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  float sacc = 0.f;
  for (long long r = w0; r < rows; r += nwarps) {
    const int t = (int)((r / H) % S);
    const size_t base = (size_t)r * kD;
    float dsum = 0.f;
#pragma unroll
    for (int cidx = 0; cidx < 2; ++cidx) {
      const int d0 = 8 * lane + 256 * cidx;
      float a[8], b[8], c8[8];
      load8(q + base + d0, a);
      load8(dout + base + d0, b);
      load8(o + base + d0, c8);
#pragma unroll
      for (int i = 0; i < 8; ++i) dsum = fmaf(b[i], c8[i], dsum);
      if (d0 >= kD - kR) {
        const float2* csr = cs + (size_t)t * (kR / 2) + ((d0 - (kD - kR)) >> 1);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = csr[i];
          rot_pair(a[2 * i], a[2 * i + 1], f.x, f.y);
          rot_pair(b[2 * i], b[2 * i + 1], f.x, f.y);
        }
      }
      store8(qr + base + d0, a);
      store8(dor + base + d0, b);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
    if (lane == 0) {
      delta[r] = dsum;
      if (sink) sacc -= expf(sink[r % H] - lse[r]) * dsum;
    }
  }
  if (sink && lane == 0 && w0 < rows) atomicAdd(dsink + (w0 % H), sacc);
}

// The window gradient w.r.t. the un-rotated latent: rot(dk_u, -u) on the last
// 64 dims, in place.  One thread per rotated pair.
__global__ void mqa_bwd_derotate_kernel(float* __restrict__ dkv, const float2* __restrict__ cs, long long n,
                                        int S) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const long long row = i / (kR / 2);
  const int j = (int)(i % (kR / 2));
  const int u = (int)(row % S);
  const float2 f = cs[(size_t)u * (kR / 2) + j];
  float* x = dkv + (size_t)row * kD + (kD - kR) + 2 * j;
  const float a = x[0], b = x[1];
  x[0] = a * f.x + b * f.y;
  x[1] = b * f.x - a * f.y;
}

}  // namespace

bool mqa_bwd_tc_supported(const v4_config& c) {
  const long long BS = (long long)c.batch * c.seqlen;
  const long long BN = c.ratio > 0 ? (long long)c.batch * (c.seqlen / c.ratio) : 0;
  return mqa_tc_supported(c) && BS + BN < (1LL << 31) && BS * c.n_heads < (1LL << 31);
}

cudaError_t launch_mqa_bwd_prep(const v4_config& c, const void* q, const void* o, const void* dout,
                                const float* lse, const float* sink, const float2* cs_table, void* qr, void* dor,
                                float* delta, float* dsink, cudaStream_t st) {
  const long long rows = (long long)c.batch * c.seqlen * c.n_heads;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // warps (8 per block) a multiple of H: blocks a multiple of H / 8
  const long long step = c.n_heads / 8;
  long long blocks = (rows + 7) / 8;
  const long long cap = 8LL * sms;
  if (blocks > cap) blocks = cap;
  blocks = (blocks + step - 1) / step * step;
  mqa_bwd_prep_kernel<<<(unsigned)blocks, 256, 0, st>>>((const bf16*)q, (const bf16*)o, (const bf16*)dout, lse,
                                                      sink, cs_table, (bf16*)qr, (bf16*)dor, delta, dsink, rows,
                                                      c.seqlen, c.n_heads);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_mqa_bwd_tc(const v4_config& cfg, const void* qr, const void* dor, const void* kv_rot,
                              const void* ent, const int32_t* idx, const float* lse, const float* delta,
                              const float2* cs_table, void* dq, float* dkv, float* dent, int* status,
                              cudaStream_t st) {
  const int B = cfg.batch, S = cfg.seqlen;
  const int N = cfg.ratio > 0 ? S / cfg.ratio : 0;
  CUtensorMap mq, mdo;
  const uint64_t rows = (uint64_t)B * S * cfg.n_heads;
  int e = 0;
  e |= make_tmap_bf16_2d(&mq, qr, kD, rows, 64, 64, true);
  e |= make_tmap_bf16_2d(&mdo, dor, kD, rows, 64, 64, true);
  if (e) return cudaErrorInvalidValue;
  Params prm;
  prm.ent = (const bf16*)ent;
  prm.kr = (const bf16*)kv_rot;
  prm.idx = cfg.topk > 0 ? idx : nullptr;
  prm.lse = lse;
  prm.delta = delta;
  prm.rope_cs = cs_table;
  prm.dq = (bf16*)dq;
  prm.dent = dent;
  prm.dkr = dkv;
  prm.status = status;
  prm.B = B;
  prm.S = S;
  prm.N = (ent != nullptr) ? N : 0;
  prm.ratio = (ent != nullptr) ? cfg.ratio : 0;
  prm.window = cfg.window;
  prm.K = cfg.topk;
  prm.H = cfg.n_heads;
  prm.HS = cfg.n_heads / kH;
  prm.scale = cfg.softmax_scale > 0.f ? cfg.softmax_scale : 1.0f / sqrtf((float)kD);
  cudaError_t err = cudaFuncSetAttribute(mqa_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long total = (long long)B * S * (cfg.n_heads / kH);
  const int grid = (int)(total < sms ? total : sms);
  mqa_bwd_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mq, mdo, prm);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_mqa_bwd_derotate(const v4_config& c, float* dkv, const float2* cs_table, cudaStream_t st) {
  const long long n = (long long)c.batch * c.seqlen * (kR / 2);
  if (n == 0) return cudaSuccess;
  mqa_bwd_derotate_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(dkv, cs_table, n, c.seqlen);
  note_launch();
  return cudaGetLastError();
}

}  // namespace v4
