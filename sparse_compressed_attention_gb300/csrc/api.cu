// C ABI of the compressed-attention library: argument checks, workspace
// carve-up, kernel dispatch, error text and the device status word.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace v4 {

static std::atomic<uint64_t> g_launches{0};
void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

// Sticky device status word (one per device that loads the library).
__device__ int g_device_status = 0;

static thread_local std::string g_err;

static v4_status fail(v4_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

static v4_status cuda_fail(cudaError_t e, const char* what) {
  return fail(V4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device address of the status word on the current device.
static int* status_ptr() {
  static std::mutex mu;
  static int* cache[128] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    cache[dev] = (int*)p;
  }
  return cache[dev];
}

// ---------------------------------------------------------------------------
// Optional per-launch timing: when enabled, every stage launch is bracketed
// by a pair of CUDA events recorded on its stream.
// ---------------------------------------------------------------------------
struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};
static std::mutex g_prof_mu;
static bool g_prof_on = false;
static std::vector<ProfRec> g_prof;

enum { K_COMPRESS = 0, K_ROTATE = 1, K_IDX_PREP = 2, K_IDX_SCORE = 3, K_TOPK = 4, K_ATTN = 5,
       K_OPROJ = 6, K_BWD_PREP = 7, K_BWD_ATTN = 8, K_BWD_FIN = 9, K_IDX_QUANT = 10,
       K_QPROJ = 11, K_KL_TARGET = 12 };

struct ProfScope {
  bool on = false;
  ProfRec r{};
  cudaStream_t st;
  ProfScope(int kind, cudaStream_t s) : st(s) {
    {
      std::lock_guard<std::mutex> lk(g_prof_mu);
      on = g_prof_on;
    }
    if (!on) return;
    r.kind = kind;
    if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) {
      on = false;
      return;
    }
    cudaEventRecord(r.a, st);
  }
  ~ProfScope() {
    if (!on) return;
    cudaEventRecord(r.b, st);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof.push_back(r);
  }
};

StageTiming::StageTiming(int kind, cudaStream_t st) : rec_(nullptr), st_(st) {
  ProfScope* ps = new ProfScope(kind, st);
  if (ps->on) rec_ = ps;
  else delete ps;
}

StageTiming::~StageTiming() { delete static_cast<ProfScope*>(rec_); }

static void prof_clear() {
  for (auto& r : g_prof) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  g_prof.clear();
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Workspace plan_workspace(const v4_config& c) {
  Workspace w;
  const size_t es = c.dtype == V4_BF16 ? 2 : 4;
  const size_t B = c.batch, S = c.seqlen, D = c.head_dim;
  const size_t Sq = (size_t)q_rows(c);            // query rows of the call
  const size_t N = c.ratio > 0 ? S / c.ratio : 0;
  const bool sel = c.topk > 0 && c.ratio > 0;
  size_t off = 0;
  auto take = [&](size_t& at, size_t& bytes, size_t n) {
    at = off;
    bytes = n;
    off = align256(off + n);
  };
  take(w.kv_rot, w.kv_rot_bytes, B * S * D * es);
  take(w.ent, w.ent_bytes, B * N * D * es);
  take(w.ikey, w.ikey_bytes, sel ? B * N * c.idx_dim * es : 0);
  // bf16 prepared queries (the E4M3 path writes codes instead)
  take(w.iqp, w.iqp_bytes, sel && !c.indexer_fp8 ? B * Sq * c.idx_heads * c.idx_dim * es : 0);
  take(w.scores, w.scores_bytes, sel ? B * Sq * N * 4 : 0);
  take(w.idx, w.idx_bytes, sel ? B * Sq * c.topk * 4 : 0);
  // redo list: one entry per (query, 64-head slice) at most
  take(w.counters, w.counters_bytes, (2 + B * Sq * (size_t)(c.n_heads > 64 ? (c.n_heads + 63) / 64 : 1)) * 4);
  take(w.rope, w.rope_bytes, S * (size_t)(c.rope_dim / 2) * 8);
  const bool e4m3 = sel && c.indexer_fp8 == 1;
  take(w.qc8, w.qc8_bytes, e4m3 ? B * Sq * c.idx_heads * c.idx_dim : 0);
  take(w.qs8, w.qs8_bytes, e4m3 ? B * Sq * c.idx_heads * 4 : 0);
  take(w.kc8, w.kc8_bytes, e4m3 ? B * N * c.idx_dim : 0);
  take(w.ks8, w.ks8_bytes, e4m3 ? B * N * 4 : 0);
  w.total = off;
  return w;
}

// Backward workspace: cos/sin table, rotated window keys, rotated queries
// and output gradients, delta.
struct BwdWorkspace {
  size_t rope = 0, kv_rot = 0, qr = 0, dor = 0, delta = 0, total = 0;
};

static BwdWorkspace plan_bwd_workspace(const v4_config& c) {
  BwdWorkspace w;
  const size_t es = c.dtype == V4_BF16 ? 2 : 4;
  const size_t B = c.batch, S = c.seqlen, D = c.head_dim, H = c.n_heads;
  size_t off = 0;
  auto take = [&](size_t& at, size_t n) {
    at = off;
    off = align256(off + n);
  };
  take(w.rope, S * (size_t)(c.rope_dim / 2) * 8);
  take(w.kv_rot, B * S * D * es);
  take(w.qr, B * S * H * D * es);
  take(w.dor, B * S * H * D * es);
  take(w.delta, B * S * H * 4);
  w.total = off;
  return w;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
static bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

static v4_status check_cfg(const v4_config* c) {
  if (!c) return fail(V4_ERR_INVALID_ARG, "cfg is NULL");
  if (c->batch < 1 || c->seqlen < 1 || c->n_heads < 1)
    return fail(V4_ERR_INVALID_ARG, "batch, seqlen and n_heads must be >= 1");
  if (c->seqlen > (1 << 28)) return fail(V4_ERR_INVALID_ARG, "seqlen above 2^28");
  if (c->head_dim < 32 || c->head_dim > 1024 || c->head_dim % 32)
    return fail(V4_ERR_INVALID_ARG, "head_dim must be a multiple of 32 in [32, 1024]");
  if (c->rope_dim < 0 || c->rope_dim > c->head_dim || c->rope_dim % 8)
    return fail(V4_ERR_INVALID_ARG, "rope_dim must be a multiple of 8 in [0, head_dim]");
  if (c->ratio < 0) return fail(V4_ERR_INVALID_ARG, "ratio must be >= 0");
  if (c->overlap != 0 && c->overlap != 1) return fail(V4_ERR_INVALID_ARG, "overlap must be 0 or 1");
  if (c->overlap && c->ratio < 1) return fail(V4_ERR_INVALID_ARG, "overlap needs ratio >= 1");
  if (c->window < -1) return fail(V4_ERR_INVALID_ARG, "window must be >= -1");
  if (c->topk < 0) return fail(V4_ERR_INVALID_ARG, "topk must be >= 0");
  if (c->topk > 0 && c->ratio < 1) return fail(V4_ERR_INVALID_ARG, "topk needs ratio >= 1");
  if (c->topk > 0) {
    if (c->idx_heads < 1) return fail(V4_ERR_INVALID_ARG, "idx_heads must be >= 1");
    if (!pow2(c->idx_dim) || c->idx_dim < 8 || c->idx_dim > 256)
      return fail(V4_ERR_INVALID_ARG, "idx_dim must be a power of two in [8, 256]");
    if (c->rope_dim > c->idx_dim) return fail(V4_ERR_INVALID_ARG, "rope_dim exceeds idx_dim");
  }
  if (c->dtype != V4_F32 && c->dtype != V4_BF16) return fail(V4_ERR_INVALID_ARG, "unknown dtype");
  if (c->path < V4_PATH_AUTO || c->path > V4_PATH_TC) return fail(V4_ERR_INVALID_ARG, "unknown path");
  if (!(c->rms_eps >= 0.f)) return fail(V4_ERR_INVALID_ARG, "rms_eps must be >= 0");
  if (c->indexer_fp8 != 0 && c->indexer_fp8 != 1) return fail(V4_ERR_INVALID_ARG, "indexer_fp8 must be 0 or 1");
  if (c->q_begin < 0 || c->q_begin >= c->seqlen)
    return fail(V4_ERR_INVALID_ARG, "q_begin must be in [0, seqlen)");
  return V4_OK;
}

#define REQ(p, name)                                                              \
  do {                                                                            \
    if (!(p)) return fail(V4_ERR_INVALID_ARG, "%s is NULL", name);                \
    if (!aligned16(p)) return fail(V4_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
  } while (0)
#define OPT(p, name)                                                              \
  do {                                                                            \
    if ((p) && !aligned16(p)) return fail(V4_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
  } while (0)
#define CU(call, what)                                  \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, what);  \
  } while (0)

static v4_status check_ws(const v4_config& c, void* ws, size_t bytes) {
  const Workspace w = plan_workspace(c);
  if (bytes < w.total)
    return fail(V4_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", bytes, w.total);
  if (w.total > 0 && !ws) return fail(V4_ERR_WORKSPACE, "workspace is NULL");
  if (ws && ((uintptr_t)ws & 255u)) return fail(V4_ERR_WORKSPACE, "workspace not 256-byte aligned");
  return V4_OK;
}

// ---------------------------------------------------------------------------
// Stage bodies (no argument checks); shared by the single-stage entry points
// and the layer call.
// ---------------------------------------------------------------------------
static v4_status do_compress(const v4_config& c, const void* ckv, const void* cs, const float* ape,
                             const float* nw, const float* f, const float2* table, int dim, int had,
                             void* out, cudaStream_t st) {
  ProfScope ps(K_COMPRESS, st);
  CU(launch_compress(c, ckv, cs, ape, nw, f, table, dim, had, out, st), "compress kernel");
  return V4_OK;
}

// cos/sin table of every position (kept in the workspace for the call)
static v4_status do_rope_table(const v4_config& c, const float* f, char* ws, cudaStream_t st) {
  const Workspace plan = plan_workspace(c);
  CU(launch_rope_table(c, f, (float2*)(ws + plan.rope), st), "rope table kernel");
  return V4_OK;
}

static v4_status do_indexer(const v4_config& c, const void* iq, int prepared, const void* ikey,
                            const float* w, const float* f, int32_t* idx, float* iscore,
                            char* ws, cudaStream_t st, bool table_ready) {
  const Workspace plan = plan_workspace(c);
  if (!prepared && !table_ready) {
    v4_status s = do_rope_table(c, f, ws, st);
    if (s != V4_OK) return s;
  }
  const float2* table = (const float2*)(ws + plan.rope);
  float* scores = (float*)(ws + plan.scores);
  if (c.indexer_fp8) {
    // opt-in E4M3: queries prepared and quantised in one kernel (or, when the
    // caller prepared them, quantised alone), keys quantised per row
    uint8_t* qc = (uint8_t*)(ws + plan.qc8);
    float* qs = (float*)(ws + plan.qs8);
    uint8_t* kc = (uint8_t*)(ws + plan.kc8);
    float* ks = (float*)(ws + plan.ks8);
    const long long N = c.seqlen / c.ratio;
    const long long qrows = (long long)c.batch * q_rows(c) * c.idx_heads;
    if (!prepared) {
      ProfScope ps(K_IDX_PREP, st);
      CU(launch_indexer_prep_e4m3(c, iq, table, f, qc, qs, st), "indexer prep kernel (E4M3)");
    }
    {
      ProfScope ps(K_IDX_QUANT, st);
      if (prepared) CU(launch_quant_e4m3(iq, qrows, c.idx_dim, qc, qs, st), "E4M3 query quantisation kernel");
      CU(launch_quant_e4m3(ikey, (long long)c.batch * N, c.idx_dim, kc, ks, st), "E4M3 key quantisation kernel");
    }
    int* status = status_ptr();
    if (!status) return fail(V4_ERR_CUDA, "device status word unavailable");
    {
      ProfScope ps(K_IDX_SCORE, st);
      CU(launch_indexer_scores_e4m3(c, qc, qs, kc, ks, w, scores, status, st), "E4M3 indexer kernel");
    }
  } else {
    const void* iqp = iq;
    if (!prepared) {
      ProfScope ps(K_IDX_PREP, st);
      CU(launch_indexer_prep(c, iq, table, f, ws + plan.iqp, st), "indexer prep kernel");
      iqp = ws + plan.iqp;
    }
    ProfScope ps(K_IDX_SCORE, st);
    if (c.path != V4_PATH_SIMT && indexer_tc_supported(c)) {
      int* status = status_ptr();
      if (!status) return fail(V4_ERR_CUDA, "device status word unavailable");
      CU(launch_indexer_scores_tc(c, iqp, ikey, w, scores, status, st), "tensor-core indexer kernel");
    } else {
      CU(launch_indexer_scores_simt(c, iqp, ikey, w, scores, st), "indexer score kernel");
    }
  }
  {
    ProfScope ps(K_TOPK, st);
    CU(launch_topk(c, scores, idx, iscore, st), "top-k kernel");
  }
  return V4_OK;
}

static bool use_tc_attention(const v4_config& c) {
  return c.path != V4_PATH_SIMT && mqa_tc_supported(c);
}

static v4_status do_mqa(const v4_config& c, const void* q, const void* kv, const void* ent,
                        const int32_t* idx, const float* sink, const float* f, void* o,
                        float* lse, char* ws, cudaStream_t st, bool table_ready) {
  const Workspace plan = plan_workspace(c);
  const float2* table = (const float2*)(ws + plan.rope);
  int* status = status_ptr();
  if (!status) return fail(V4_ERR_CUDA, "device status word unavailable");
  void* kv_rot = ws + plan.kv_rot;
  const bool tc = use_tc_attention(c);
  {
    ProfScope ps(K_ROTATE, st);
    if (tc) {
      if (!table_ready) {
        v4_status s = do_rope_table(c, f, ws, st);
        if (s != V4_OK) return s;
      }
      CU(launch_key_prep(c, kv, table, kv_rot, st), "key prep kernel");
    } else {
      CU(launch_rotate_rows(c, kv, f, kv_rot, st), "window-key rotation kernel");
    }
  }
  if (tc) {
    int* counters = (int*)(ws + plan.counters);
    {
      ProfScope ps(K_ATTN, st);
      CU(launch_mqa_tc(c, q, kv_rot, ent, idx, sink, table, o, lse, counters, status, st),
         "tensor-core attention kernel");
    }
    // queries whose fixed-shift softmax overflowed or kept too little mass
    // are recomputed with the running-max kernel (normally none)
    CU(launch_mqa_simt(c, q, kv_rot, ent, idx, sink, f, o, lse, status, counters + 1, st),
       "attention fix-up kernel");
    return V4_OK;
  }
  {
    ProfScope ps(K_ATTN, st);
    CU(launch_mqa_simt(c, q, kv_rot, ent, idx, sink, f, o, lse, status, nullptr, st), "attention kernel");
  }
  return V4_OK;
}

// Accessors for other translation units of the library.
v4_status validate_config(const v4_config* c) { return check_cfg(c); }
v4_status set_error(v4_status st, const char* msg) { return fail(st, "%s", msg); }
int* device_status_ptr() { return status_ptr(); }

}  // namespace v4

using namespace v4;

extern "C" {

v4_status v4_rope_inv_freq(float theta, int32_t rope_dim, float yarn_factor, int32_t original_len,
                           float beta_fast, float beta_slow, float* inv_freq) {
  if (!inv_freq) return fail(V4_ERR_INVALID_ARG, "inv_freq is NULL");
  if (rope_dim < 2 || rope_dim % 2) return fail(V4_ERR_INVALID_ARG, "rope_dim must be even and >= 2");
  if (!(theta > 1.f)) return fail(V4_ERR_INVALID_ARG, "theta must be > 1");
  const bool yarn = yarn_factor > 1.f && original_len > 0;
  if (yarn && !(beta_fast > beta_slow)) return fail(V4_ERR_INVALID_ARG, "beta_fast must exceed beta_slow");
  const double pi = 3.14159265358979323846;
  for (int j = 0; j < rope_dim / 2; ++j) {
    double f = pow((double)theta, -2.0 * j / (double)rope_dim);
    if (yarn) {
      // YaRN NTK-by-parts: ratio of the original length to the wavelength
      const double r = (double)original_len * f / (2.0 * pi);
      double g = (r - beta_slow) / ((double)beta_fast - beta_slow);
      g = g < 0.0 ? 0.0 : (g > 1.0 ? 1.0 : g);
      f = (1.0 - g) * f / (double)yarn_factor + g * f;
    }
    inv_freq[j] = (float)f;
  }
  return V4_OK;
}

v4_status v4_workspace_size(const v4_config* cfg, size_t* bytes) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  if (!bytes) return fail(V4_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = plan_workspace(*cfg).total;
  return V4_OK;
}

v4_status v4_compress(const v4_config* cfg, const void* ckv, const void* cscore, const float* ape,
                      const float* norm_w, const float* inv_freq, int32_t dim, int32_t hadamard,
                      void* out, void* stream) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  if (cfg->ratio < 1) return fail(V4_ERR_INVALID_ARG, "compressor needs ratio >= 1");
  if (dim < 8 || dim > 1024 || dim % 8 || cfg->rope_dim > dim)
    return fail(V4_ERR_INVALID_ARG, "dim must be a multiple of 8 in [max(8, rope_dim), 1024]");
  if (hadamard && !pow2(dim)) return fail(V4_ERR_INVALID_ARG, "Hadamard needs a power-of-two dim");
  REQ(ckv, "ckv");
  REQ(cscore, "cscore");
  REQ(ape, "ape");
  OPT(norm_w, "norm_w");
  if (cfg->rope_dim > 0) REQ(inv_freq, "inv_freq");
  if (cfg->seqlen / cfg->ratio > 0) REQ(out, "out");
  return do_compress(*cfg, ckv, cscore, ape, norm_w, inv_freq, nullptr, dim, hadamard ? 1 : 0, out,
                     (cudaStream_t)stream);
}

v4_status v4_indexer_prep(const v4_config* cfg, const void* iq, const float* inv_freq, void* iq_prep,
                          void* stream) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  if (cfg->topk < 1) return fail(V4_ERR_INVALID_ARG, "indexer needs topk >= 1");
  REQ(iq, "iq");
  REQ(iq_prep, "iq_prep");
  if (cfg->rope_dim > 0) REQ(inv_freq, "inv_freq");
  CU(launch_indexer_prep(*cfg, iq, nullptr, inv_freq, iq_prep, (cudaStream_t)stream), "indexer prep kernel");
  return V4_OK;
}

v4_status v4_indexer_topk(const v4_config* cfg, const void* iq, int32_t iq_prepared, const void* ikey,
                          const float* w, const float* inv_freq, int32_t* idx, float* iscore,
                          void* workspace, size_t ws_bytes, void* stream) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  if (cfg->topk < 1) return fail(V4_ERR_INVALID_ARG, "indexer needs topk >= 1");
  REQ(iq, "iq");
  REQ(w, "w");
  REQ(idx, "idx");
  OPT(iscore, "iscore");
  if (cfg->seqlen / cfg->ratio > 0) REQ(ikey, "ikey");
  if (!iq_prepared && cfg->rope_dim > 0) REQ(inv_freq, "inv_freq");
  if (cfg->path == V4_PATH_TC && !indexer_tc_supported(*cfg))
    return fail(V4_ERR_UNSUPPORTED, "tensor-core indexer needs bf16, idx_heads 64, idx_dim 128");
  if (cfg->indexer_fp8 && (cfg->path == V4_PATH_SIMT || !indexer_e4m3_supported(*cfg)))
    return fail(V4_ERR_UNSUPPORTED, "E4M3 indexer needs the tensor-core shapes: bf16, idx_heads 64, idx_dim 128");
  s = check_ws(*cfg, workspace, ws_bytes);
  if (s != V4_OK) return s;
  return do_indexer(*cfg, iq, iq_prepared ? 1 : 0, ikey, w, inv_freq, idx, iscore, (char*)workspace,
                    (cudaStream_t)stream, false);
}

v4_status v4_quantize_e4m3(const void* x, int64_t rows, int32_t dim, uint8_t* codes, float* scales,
                           void* stream) {
  if (rows < 0) return fail(V4_ERR_INVALID_ARG, "rows must be >= 0");
  if (dim != 128 && dim != 256 && dim != 512 && dim != 1024)
    return fail(V4_ERR_INVALID_ARG, "dim must be 128, 256, 512 or 1024");
  if (rows == 0) return V4_OK;
  REQ(x, "x");
  REQ(codes, "codes");
  REQ(scales, "scales");
  CU(launch_quant_e4m3(x, (long long)rows, dim, codes, scales, (cudaStream_t)stream), "E4M3 quantisation kernel");
  return V4_OK;
}

v4_status v4_indexer_topk_e4m3(const v4_config* cfg, const uint8_t* q_codes, const float* q_scales,
                               const uint8_t* k_codes, const float* k_scales, const float* w, int32_t* idx,
                               float* iscore, void* workspace, size_t ws_bytes, void* stream) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  if (cfg->topk < 1) return fail(V4_ERR_INVALID_ARG, "indexer needs topk >= 1");
  if (!indexer_e4m3_supported(*cfg) || cfg->path == V4_PATH_SIMT)
    return fail(V4_ERR_UNSUPPORTED, "E4M3 indexer needs the tensor-core shapes: bf16, idx_heads 64, idx_dim 128");
  REQ(q_codes, "q_codes");
  REQ(q_scales, "q_scales");
  REQ(w, "w");
  REQ(idx, "idx");
  OPT(iscore, "iscore");
  if (cfg->seqlen / cfg->ratio > 0) {
    REQ(k_codes, "k_codes");
    REQ(k_scales, "k_scales");
  }
  s = check_ws(*cfg, workspace, ws_bytes);
  if (s != V4_OK) return s;
  const Workspace plan = plan_workspace(*cfg);
  cudaStream_t st = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  float* scores = (float*)(ws + plan.scores);
  int* status = status_ptr();
  if (!status) return fail(V4_ERR_CUDA, "device status word unavailable");
  {
    ProfScope ps(K_IDX_SCORE, st);
    CU(launch_indexer_scores_e4m3(*cfg, q_codes, q_scales, k_codes, k_scales, w, scores, status, st),
       "E4M3 indexer kernel");
  }
  {
    ProfScope ps(K_TOPK, st);
    CU(launch_topk(*cfg, scores, idx, iscore, st), "top-k kernel");
  }
  return V4_OK;
}

v4_status v4_sparse_mqa_fwd(const v4_config* cfg, const void* q, const void* kv, const void* ent,
                            const int32_t* idx, const float* sink, const float* inv_freq, void* o,
                            float* lse, void* workspace, size_t ws_bytes, void* stream) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  REQ(q, "q");
  REQ(kv, "kv");
  REQ(o, "o");
  if (cfg->ratio > 0 && cfg->seqlen / cfg->ratio > 0) REQ(ent, "ent");
  if (cfg->topk > 0) REQ(idx, "idx");
  OPT(sink, "sink");
  OPT(lse, "lse");
  if (cfg->rope_dim > 0) REQ(inv_freq, "inv_freq");
  if (cfg->path == V4_PATH_TC && !mqa_tc_supported(*cfg))
    return fail(V4_ERR_UNSUPPORTED, "tensor-core attention needs bf16, H a multiple of 64 up to 512, D=512, R=64, 1 <= W <= 128, K <= 1024");
  s = check_ws(*cfg, workspace, ws_bytes);
  if (s != V4_OK) return s;
  return do_mqa(*cfg, q, kv, ent, cfg->topk > 0 ? idx : nullptr, sink, inv_freq, o, lse,
                (char*)workspace, (cudaStream_t)stream, false);
}

v4_status v4_bwd_workspace_size(const v4_config* cfg, size_t* bytes) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  if (!bytes) return fail(V4_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = plan_bwd_workspace(*cfg).total;
  return V4_OK;
}

v4_status v4_sparse_mqa_bwd(const v4_config* cfg, const void* q, const void* kv, const void* ent,
                            const int32_t* idx, const float* sink, const float* inv_freq, const void* o,
                            const float* lse, const void* dout, void* dq, float* dkv, float* dent,
                            float* dsink, void* workspace, size_t ws_bytes, void* stream) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  const v4_config& c = *cfg;
  if (c.q_begin != 0) return fail(V4_ERR_UNSUPPORTED, "attention backward needs q_begin = 0");
  if (!mqa_bwd_tc_supported(c))
    return fail(V4_ERR_UNSUPPORTED,
                "attention backward needs bf16, H a multiple of 64 up to 512, D=512, R=64, 1 <= W <= 128, K <= 1024");
  const bool comp = c.ratio > 0 && c.seqlen / c.ratio > 0;
  REQ(q, "q");
  REQ(kv, "kv");
  REQ(o, "o");
  REQ(lse, "lse");
  REQ(dout, "dout");
  REQ(dq, "dq");
  REQ(dkv, "dkv");
  REQ(inv_freq, "inv_freq");
  if (comp) {
    REQ(ent, "ent");
    REQ(dent, "dent");
  }
  if (c.topk > 0) REQ(idx, "idx");
  OPT(sink, "sink");
  if (sink) REQ(dsink, "dsink");
  const BwdWorkspace plan = plan_bwd_workspace(c);
  if (ws_bytes < plan.total) return fail(V4_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, plan.total);
  if (!workspace) return fail(V4_ERR_WORKSPACE, "workspace is NULL");
  if ((uintptr_t)workspace & 255u) return fail(V4_ERR_WORKSPACE, "workspace not 256-byte aligned");
  int* status = status_ptr();
  if (!status) return fail(V4_ERR_CUDA, "device status word unavailable");
  char* ws = (char*)workspace;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t B = c.batch, S = c.seqlen, D = c.head_dim;
  const size_t N = comp ? S / c.ratio : 0;
  const float2* table = (const float2*)(ws + plan.rope);
  float* delta = (float*)(ws + plan.delta);
  void* kv_rot = ws + plan.kv_rot;
  {
    ProfScope ps(K_BWD_PREP, st);
    CU(cudaMemsetAsync(dkv, 0, B * S * D * 4, st), "dkv clear");
    if (comp) CU(cudaMemsetAsync(dent, 0, B * N * D * 4, st), "dent clear");
    if (sink) CU(cudaMemsetAsync(dsink, 0, (size_t)c.n_heads * 4, st), "dsink clear");
    CU(launch_rope_table(c, inv_freq, (float2*)(ws + plan.rope), st), "rope table kernel");
    CU(launch_key_prep(c, kv, table, kv_rot, st), "key prep kernel");
    CU(launch_mqa_bwd_prep(c, q, o, dout, lse, sink, table, ws + plan.qr, ws + plan.dor, delta, sink ? dsink : nullptr,
                           st),
       "backward prep kernel");
  }
  {
    ProfScope ps(K_BWD_ATTN, st);
    CU(launch_mqa_bwd_tc(c, ws + plan.qr, ws + plan.dor, kv_rot, comp ? ent : nullptr, c.topk > 0 ? idx : nullptr,
                         lse, delta, table, dq, dkv, comp ? dent : nullptr, status, st),
       "tensor-core attention backward kernel");
  }
  {
    ProfScope ps(K_BWD_FIN, st);
    CU(launch_mqa_bwd_derotate(c, dkv, table, st), "window-gradient de-rotation kernel");
  }
  return V4_OK;
}

static v4_status check_oproj(const v4_config& c) {
  if (c.o_groups < 1 || c.n_heads % c.o_groups) return fail(V4_ERR_INVALID_ARG, "o_groups must divide n_heads");
  if (c.o_rank < 1) return fail(V4_ERR_INVALID_ARG, "o_rank must be >= 1");
  if (!oproj_tc_supported(c))
    return fail(V4_ERR_UNSUPPORTED,
                "grouped projection needs bf16, (n_heads/o_groups)*head_dim a multiple of 64, o_rank a multiple of 256");
  return V4_OK;
}

static v4_status do_oproj(const v4_config& c, const void* o, const void* wo_a, void* y, cudaStream_t st) {
  int* status = status_ptr();
  if (!status) return fail(V4_ERR_CUDA, "device status word unavailable");
  ProfScope ps(K_OPROJ, st);
  CU(launch_oproj_tc(c, o, wo_a, y, status, st), "grouped projection kernel");
  return V4_OK;
}

v4_status v4_grouped_o_proj(const v4_config* cfg, const void* o, const void* wo_a, void* y,
                            void* stream) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  s = check_oproj(*cfg);
  if (s != V4_OK) return s;
  REQ(o, "o");
  REQ(wo_a, "wo_a");
  REQ(y, "y");
  return do_oproj(*cfg, o, wo_a, y, (cudaStream_t)stream);
}

v4_status v4_indexer_kl_target(const v4_config* cfg, const void* q, const void* ent, const int32_t* idx,
                               const float* lse, const float* iscore, const float* inv_freq, float* target,
                               float* loss, float* dscore, void* workspace, size_t ws_bytes, void* stream) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  const v4_config& c = *cfg;
  if (c.topk < 1 || c.ratio < 1) return fail(V4_ERR_INVALID_ARG, "the target needs a selection (topk >= 1, ratio >= 1)");
  if (c.q_begin != 0) return fail(V4_ERR_UNSUPPORTED, "the distillation target needs q_begin = 0");
  if (!kl_target_tc_supported(c))
    return fail(V4_ERR_UNSUPPORTED, "the distillation target needs bf16, H a multiple of 64 up to 512, D=512, R=64, "
                                    "K <= 1024");
  REQ(q, "q");
  REQ(idx, "idx");
  REQ(lse, "lse");
  REQ(target, "target");
  if (c.seqlen / c.ratio > 0) REQ(ent, "ent");
  if (c.rope_dim > 0) REQ(inv_freq, "inv_freq");
  OPT(iscore, "iscore");
  OPT(loss, "loss");
  OPT(dscore, "dscore");
  if ((loss || dscore) && !iscore) return fail(V4_ERR_INVALID_ARG, "loss and dscore need iscore");
  s = check_ws(c, workspace, ws_bytes);
  if (s != V4_OK) return s;
  int* status = status_ptr();
  if (!status) return fail(V4_ERR_CUDA, "device status word unavailable");
  cudaStream_t st = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  s = do_rope_table(c, inv_freq, ws, st);
  if (s != V4_OK) return s;
  const Workspace plan = plan_workspace(c);
  ProfScope ps(K_KL_TARGET, st);
  CU(launch_kl_target(c, q, ent, idx, lse, iscore, (const float2*)(ws + plan.rope), target, loss, dscore, status, st),
     "distillation target kernel");
  return V4_OK;
}

v4_status v4_q_proj(const v4_config* cfg, const void* qlat, int32_t rank, const void* wq, int32_t q_norm,
                    const float* q_norm_w, const void* wiq, void* q, void* iq, void* stream) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  const v4_config& c = *cfg;
  if (q_norm != 0 && q_norm != 1) return fail(V4_ERR_INVALID_ARG, "q_norm must be 0 or 1");
  if (rank < 1) return fail(V4_ERR_INVALID_ARG, "rank must be >= 1");
  const long long nq = (long long)c.n_heads * c.head_dim;
  const long long ni = (long long)c.idx_heads * c.idx_dim;
  if (c.dtype != V4_BF16 || rank % 64 || rank > 65536 || nq % 256 || (q_norm && c.head_dim != 512) ||
      (wiq && (c.idx_heads < 1 || ni % 256)))
    return fail(V4_ERR_UNSUPPORTED, "query projections need bf16, rank a multiple of 64, H*D and Hi*Di multiples "
                                    "of 256, D = 512 with q_norm");
  REQ(qlat, "qlat");
  REQ(wq, "wq");
  REQ(q, "q");
  OPT(q_norm_w, "q_norm_w");
  OPT(wiq, "wiq");
  if (wiq) REQ(iq, "iq");
  int* status = status_ptr();
  if (!status) return fail(V4_ERR_CUDA, "device status word unavailable");
  cudaStream_t st = (cudaStream_t)stream;
  const long long T = (long long)c.batch * q_rows(c);          // the call's query rows
  ProfScope ps(K_QPROJ, st);
  CU(launch_qproj_tc(T, rank, qlat, wq, (int)nq, q, q_norm, c.rms_eps, q_norm ? q_norm_w : nullptr, status, st),
     "query projection kernel");
  if (wiq) CU(launch_qproj_tc(T, rank, qlat, wiq, (int)ni, iq, 0, 0.f, nullptr, status, st),
              "indexer query projection kernel");
  return V4_OK;
}

v4_status v4_attn_layer_fwd(const v4_config* cfg, const v4_layer_inputs* in, v4_layer_outputs* out,
                            void* workspace, size_t ws_bytes, void* stream) {
  v4_status s = check_cfg(cfg);
  if (s != V4_OK) return s;
  if (!in || !out) return fail(V4_ERR_INVALID_ARG, "inputs or outputs struct is NULL");
  const v4_config& c = *cfg;
  const bool comp = c.ratio > 0 && c.seqlen / c.ratio > 0;
  const bool sel = c.topk > 0;
  REQ(in->q, "q");
  REQ(in->kv, "kv");
  REQ(out->o, "o");
  OPT(out->lse, "lse");
  OPT(in->sink, "sink");
  if (c.rope_dim > 0) REQ(in->inv_freq, "inv_freq");
  if (comp) {
    REQ(in->ckv, "ckv");
    REQ(in->cscore, "cscore");
    REQ(in->ape, "ape");
    OPT(in->norm_w, "norm_w");
    OPT(out->ent, "ent");
  }
  if (sel) {
    REQ(in->iq, "iq");
    REQ(in->w, "w");
    OPT(out->idx, "idx");
    OPT(out->iscore, "iscore");
    if (comp) {
      REQ(in->ickv, "ickv");
      REQ(in->icscore, "icscore");
      REQ(in->iape, "iape");
      OPT(in->inorm_w, "inorm_w");
      OPT(out->ikey, "ikey");
    }
  }
  if (in->wo_a) {
    REQ(in->wo_a, "wo_a");
    REQ(out->y, "y");
    s = check_oproj(c);
    if (s != V4_OK) return s;
  }
  if (c.path == V4_PATH_TC && !mqa_tc_supported(c))
    return fail(V4_ERR_UNSUPPORTED, "tensor-core attention needs bf16, H a multiple of 64 up to 512, D=512, R=64, 1 <= W <= 128, K <= 1024");
  if (sel && c.indexer_fp8 && (c.path == V4_PATH_SIMT || !indexer_e4m3_supported(c)))
    return fail(V4_ERR_UNSUPPORTED, "E4M3 indexer needs the tensor-core shapes: bf16, idx_heads 64, idx_dim 128");
  s = check_ws(c, workspace, ws_bytes);
  if (s != V4_OK) return s;
  char* ws = (char*)workspace;
  const Workspace plan = plan_workspace(c);
  cudaStream_t st = (cudaStream_t)stream;
  void* ent = out->ent ? out->ent : (void*)(ws + plan.ent);
  void* ikey = out->ikey ? out->ikey : (void*)(ws + plan.ikey);
  int32_t* idx = out->idx ? out->idx : (int32_t*)(ws + plan.idx);
  s = do_rope_table(c, in->inv_freq, ws, st);
  if (s != V4_OK) return s;
  if (comp) {
    s = do_compress(c, in->ckv, in->cscore, in->ape, in->norm_w, in->inv_freq, (const float2*)(ws + plan.rope),
                    c.head_dim, 0, ent, st);
    if (s != V4_OK) return s;
  }
  if (sel) {
    if (comp) {
      s = do_compress(c, in->ickv, in->icscore, in->iape, in->inorm_w, in->inv_freq,
                      (const float2*)(ws + plan.rope), c.idx_dim, 1, ikey, st);
      if (s != V4_OK) return s;
    }
    s = do_indexer(c, in->iq, 0, ikey, in->w, in->inv_freq, idx, out->iscore, ws, st, true);
    if (s != V4_OK) return s;
  }
  s = do_mqa(c, in->q, in->kv, comp ? ent : nullptr, sel ? idx : nullptr, in->sink, in->inv_freq, out->o,
             out->lse, ws, st, true);
  if (s != V4_OK || !in->wo_a) return s;
  return do_oproj(c, out->o, in->wo_a, out->y, st);
}

const char* v4_last_error(void) { return g_err.c_str(); }

const char* v4_build_info(void) {
#ifdef V4_DEBUG
  return "sm_103a V4_DEBUG (bound checks)";
#else
  return "sm_103a";
#endif
}

v4_status v4_get_device_status(void* stream, int32_t* status) {
  if (!status) return fail(V4_ERR_INVALID_ARG, "status is NULL");
  int* p = status_ptr();
  if (!p) return fail(V4_ERR_CUDA, "device status word unavailable");
  int v = 0;
  CU(cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream), "status copy");
  CU(cudaStreamSynchronize((cudaStream_t)stream), "status sync");
  *status = v;
  return V4_OK;
}

v4_status v4_reset_device_status(void* stream) {
  int* p = status_ptr();
  if (!p) return fail(V4_ERR_CUDA, "device status word unavailable");
  CU(cudaMemsetAsync(p, 0, sizeof(int), (cudaStream_t)stream), "status reset");
  return V4_OK;
}

uint64_t v4_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

v4_status v4_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (on) prof_clear();
  g_prof_on = on != 0;
  return V4_OK;
}

int32_t v4_profile_count(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  return (int32_t)g_prof.size();
}

v4_status v4_profile_get(int32_t i, int32_t* kind, float* ms) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (i < 0 || i >= (int32_t)g_prof.size()) return fail(V4_ERR_INVALID_ARG, "profile record out of range");
  if (!kind || !ms) return fail(V4_ERR_INVALID_ARG, "kind or ms is NULL");
  CU(cudaEventSynchronize(g_prof[i].b), "profile event sync");
  CU(cudaEventElapsedTime(ms, g_prof[i].a, g_prof[i].b), "profile elapsed time");
  *kind = g_prof[i].kind;
  return V4_OK;
}

}  // extern "C"
