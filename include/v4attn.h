/*
 * v4attn.h - C ABI of the DeepSeek-V4-Flash compressed attention forward
 * (compressor, CSA lightning indexer with top-k, sparse/dense multi-query
 * attention with sliding window and de-rotated output) on one GB300 GPU.
 *
 * Sources of the operations:
 *   [PR]   Primus PR #930 "fix(deepseek-v4): correct V4-Flash attention math,
 *          wire the MoE balance loss", Part 1 (items 1-6, 8).
 *   [BLOG] "Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X GPUs
 *          with Primus", sections "The DeepSeek-V4-Flash architecture",
 *          "Three attention types, interleaved", "Kernel fusions".
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, row-major, in device memory owned by the caller.
 *     The library never allocates device memory; scratch space is the
 *     caller's workspace (see v4_workspace_size).  One exception:
 *     v4_sparse_mqa_fwd_noalloc keeps its scratch in a library-owned static
 *     device array (see its section).  Every device pointer must be 16-byte
 *     aligned.
 *   - "Storage dtype" (cfg->dtype) is the element type of q, kv, the pooling
 *     projections, entries, indexer keys/queries and the output: V4_F32 or
 *     V4_BF16.  ape, norm weights, indexer weights w, sink, inv_freq, lse
 *     and iscore are always float32.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously.  A non-V4_OK return means nothing was
 *     enqueued; v4_last_error() gives the reason.  Arguments are validated on
 *     the host before any launch.
 *   - Problems found on the device (an out-of-range selected index, a timed
 *     out wait) never trap: they set a sticky status word that
 *     v4_get_device_status() reads.  Offending keys are skipped.
 *   - Entry points may be called from several host threads; the error text
 *     is per thread.
 *
 * Notation: B batch, S sequence length, H query heads, D latent (head) dim,
 * R rotated dims (the last R of D), r compression ratio, ov overlap (0/1),
 * N = S / r entries (floor), Hi / Di indexer heads / dim, K top-k, W window.
 */
#ifndef V4ATTN_H
#define V4ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  V4_OK = 0,
  V4_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or combination */
  V4_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. forced path) */
  V4_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
  V4_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  V4_ERR_TIMEOUT = 5,       /* device status: a bounded wait gave up */
  V4_ERR_BAD_INDEX = 6,     /* device status: a selected index was not visible */
  V4_ERR_BOUND = 7          /* device status, V4_DEBUG builds only: an index failed its
                               bound check (gather row, ring slot, TMEM column) and the
                               access was skipped */
} v4_status;

typedef enum { V4_F32 = 0, V4_BF16 = 1 } v4_dtype;

/* Kernel family selection (cfg->path). AUTO picks the tensor-core kernels
 * when the shapes and dtype allow it, otherwise the CUDA-core kernels.
 * Tensor-core attention: bf16, n_heads a multiple of 64 up to 512 (each
 * 64-head slice of a query is one work item), head_dim 512, rope_dim 64,
 * 1 <= window <= 128, topk <= 1024.  Tensor-core indexer: bf16,
 * idx_heads 64, idx_dim 128.  V4_PATH_TC returns V4_ERR_UNSUPPORTED for
 * other shapes. */
typedef enum { V4_PATH_AUTO = 0, V4_PATH_SIMT = 1, V4_PATH_TC = 2 } v4_path;

typedef struct v4_config {
  int32_t batch;          /* B >= 1 */
  int32_t seqlen;         /* S >= 1 */
  int32_t n_heads;        /* H >= 1 (Flash: 64) */
  int32_t head_dim;       /* D, multiple of 32, 32..1024 (Flash: 512) */
  int32_t rope_dim;       /* R, multiple of 8, <= D (Flash: 64) */
  int32_t ratio;          /* r: 0 = window-only layer, 4 = CSA, 128 = HCA; any r >= 1 */
  int32_t overlap;        /* ov: 1 = each entry also pools the previous r tokens (CSA) */
  int32_t window;         /* W: tokens [t-W+1, t]; 0 = no window; -1 = all tokens <= t */
  int32_t topk;           /* K: 0 = attend to every visible entry (HCA); > 0 = CSA selection */
  int32_t idx_heads;      /* Hi (Flash: 64) */
  int32_t idx_dim;        /* Di, power of two, 8..256, >= R (Flash: 128) */
  int32_t o_groups;       /* grouped output projection: groups (Flash: 8) */
  int32_t o_rank;         /* grouped output projection: rank per group (Flash: 1024) */
  float softmax_scale;    /* <= 0 selects D^-0.5, the only value [PR] item 1 allows */
  float rms_eps;          /* entry RMSNorm epsilon (1e-6) */
  int32_t dtype;          /* v4_dtype: storage dtype */
  int32_t path;           /* v4_path */
  int32_t indexer_fp8;    /* 1 = opt-in E4M3 indexer QK (see v4_indexer_topk_e4m3);
                             0 = bf16 operands, fp32 scoring (the default [PR] item 4 asks for) */
  int32_t q_begin;        /* first query position of the call, 0 <= q_begin < seqlen (0 = all).
                             The call computes queries q_begin .. seqlen-1 of every sequence
                             against the whole causal prefix: [BLOG] "Three attention types,
                             interleaved" gives each query its own keys (selected entries and
                             window), so query rows are independent given the prefix.  Row
                             tensors (q, iq, w, o, lse, idx, iscore, y; Sq = seqlen - q_begin
                             rows per sequence, row i = position q_begin + i) hold only these
                             rows; sequence tensors (kv, ckv, cscore, ickv, icscore, entries,
                             indexer keys) hold all seqlen positions.  A chunk [a, b) of a
                             sequence is the call with seqlen = b and q_begin = a: causality
                             means it needs no token past b-1.  The backward and the indexer
                             distillation target take q_begin = 0 only (V4_ERR_UNSUPPORTED). */
} v4_config;

/* ----------------------------------------------------------------------
 * RoPE inverse-frequency table (host function, no GPU).
 * [PR] items 2 and 8: compressed layers rotate with base 40000 paired with a
 * YaRN factor (16) acting on the inverse frequencies.  Base table
 * theta^(-2j/R); YaRN "NTK-by-parts" (Peng et al. 2023, section 3.2) with
 * ramp bounds beta_slow..beta_fast applies when yarn_factor > 1 and
 * original_len > 0.  inv_freq: host array of R/2 floats, written.
 * --------------------------------------------------------------------*/
v4_status v4_rope_inv_freq(float theta, int32_t rope_dim, float yarn_factor,
                           int32_t original_len, float beta_fast, float beta_slow,
                           float* inv_freq);

/* Bytes of workspace that every entry point below needs for `cfg` (the
 * largest of their needs, so one buffer serves them all). */
v4_status v4_workspace_size(const v4_config* cfg, size_t* bytes);

/* ----------------------------------------------------------------------
 * Compressor (one learned pooling operator for CSA and HCA).
 * [BLOG] "Three attention types, interleaved" (softmax over the group biased
 * by a learnable per-position term; CSA groups overlap: own r tokens plus
 * the previous r) and "Kernel fusions", row "Compressor pooling";
 * [PR] item 1 (entries are RMSNormed), item 2 (entry s rotated at r*s),
 * item 6e (indexer keys: RoPE then normalised Hadamard).
 *
 *   ckv, cscore : [B, S, 1+ov, dim] storage dtype. Half 0 is the token's
 *                 projection for its own group, half 1 for the next group
 *                 (used as "previous" members).
 *   ape         : [(1+ov)*r, dim] fp32. Rows are chronological: with
 *                 overlap rows 0..r-1 bias the previous group's tokens,
 *                 rows r..2r-1 the own tokens.
 *   norm_w      : [dim] fp32 RMSNorm weight, NULL = ones.
 *   inv_freq    : [R/2] fp32 device array.
 *   dim         : channel count (D for the attention entries, Di for the
 *                 indexer keys); R <= dim.
 *   hadamard    : 1 = apply the normalised Sylvester Hadamard (dim must be a
 *                 power of two) after the rotation.
 *   out         : [B, N, dim] storage dtype, N = S / r.
 * Per entry s and channel c: pooled = sum_m softmax_m(cscore + ape) * ckv over
 * the members m (entry 0 has no previous group; absent members are left out),
 * then e = pooled / sqrt(mean_c pooled^2 + eps) * g, rotated at position r*s.
 * --------------------------------------------------------------------*/
v4_status v4_compress(const v4_config* cfg, const void* ckv, const void* cscore,
                      const float* ape, const float* norm_w, const float* inv_freq,
                      int32_t dim, int32_t hadamard, void* out, void* stream);

/* ----------------------------------------------------------------------
 * Indexer query preparation.  [PR] item 6e: queries rotated at their own
 * position t (partial RoPE at the compressed base), then the normalised
 * Hadamard.  iq: [B, S, Hi, Di] -> iq_prep: [B, S, Hi, Di], storage dtype.
 * --------------------------------------------------------------------*/
v4_status v4_indexer_prep(const v4_config* cfg, const void* iq, const float* inv_freq,
                          void* iq_prep, void* stream);

/* ----------------------------------------------------------------------
 * Lightning indexer scores and top-k selection (CSA).
 * [PR] item 6a (per-head weights scaled by Hi^-1/2 * Di^-1/2), item 4 (the
 * QK stays in high precision: bf16 operands, fp32 accumulation, fp32
 * scoring and selection); [BLOG] "Kernel fusions", row "Indexer scoring tail"
 * (ReLU, per-head weight, head sum, inline causal mask) and "Three attention
 * types" (keep the best 512).
 *
 *   I[t,s] = sum_h w[t,h] * (Hi*Di)^-1/2 * max(0, iq~[t,h] . ikey[s]),
 *   defined for s < n_vis(t) = (t+1)/r; the best min(K, n_vis(t)) are kept,
 *   equal scores going to the lower index.
 *
 *   iq          : [B, S, Hi, Di]; un-rotated (iq_prepared = 0) or already
 *                 prepared by v4_indexer_prep (iq_prepared = 1).
 *   ikey        : [B, N, Di] from v4_compress(dim = Di, hadamard = 1).
 *   w           : [B, S, Hi] fp32 per-head weights (unscaled).
 *   idx         : [B, S, K] int32 out. The selected entries of row t in
 *                 ascending index order, then -1 padding.
 *   iscore      : [B, S, K] fp32 out, nullable: I[t, idx] (-inf on padding).
 *   workspace   : at least v4_workspace_size bytes.
 * --------------------------------------------------------------------*/
v4_status v4_indexer_topk(const v4_config* cfg, const void* iq, int32_t iq_prepared,
                          const void* ikey, const float* w, const float* inv_freq,
                          int32_t* idx, float* iscore, void* workspace,
                          size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------
 * Opt-in E4M3 indexer.  [PR] item 4 keeps the indexer QK in high precision
 * by default, because quantisation error there changes which entries are
 * selected, and puts FP8 behind its own switch; [BLOG] closing section: an
 * E4M3 path for the indexer QK ships.  The pages name the format, not the
 * scaling: here every row (one prepared query head, one indexer key) is
 * scaled by its absolute maximum.
 *
 * v4_quantize_e4m3: x [rows, dim] bf16 -> codes [rows, dim] (E4M3 bytes,
 *   OCP "FN" encoding) and scales [rows] fp32 with x ~= code * scale:
 *   scale = amax / 448, code = E4M3(x * (448 / amax)), every step in fp32
 *   rounded to nearest (the conversion saturates at +-448); an all-zero row
 *   gets scale 0 and zero codes.  dim is 128, 256, 512 or 1024; rows >= 0.
 *
 * v4_indexer_topk_e4m3: the selection of v4_indexer_topk from quantised
 *   operands (cfg as for the tensor-core indexer: bf16, Hi = 64, Di = 128):
 *     q_codes [B, S, Hi, Di] with q_scales [B, S, Hi]  (prepared queries),
 *     k_codes [B, N, Di]     with k_scales [B, N]      (indexer keys),
 *     I[t,s] = sum_h w[t,h] (Hi*Di)^-1/2 max(0, (q_code q_scale) . (k_code k_scale)),
 *   E4M3 tensor-core products with fp32 accumulation and fp32 scoring; idx,
 *   iscore, tie rule and workspace as v4_indexer_topk.  Other shapes return
 *   V4_ERR_UNSUPPORTED.
 *
 * With cfg->indexer_fp8 = 1, v4_indexer_topk and v4_attn_layer_fwd prepare
 * the queries in bf16 as before, quantise queries and keys into the
 * workspace with v4_quantize_e4m3's rule and select from the E4M3 scores.
 * --------------------------------------------------------------------*/
v4_status v4_quantize_e4m3(const void* x, int64_t rows, int32_t dim, uint8_t* codes, float* scales,
                           void* stream);
v4_status v4_indexer_topk_e4m3(const v4_config* cfg, const uint8_t* q_codes, const float* q_scales,
                               const uint8_t* k_codes, const float* k_scales, const float* w,
                               int32_t* idx, float* iscore, void* workspace, size_t ws_bytes,
                               void* stream);

/* ----------------------------------------------------------------------
 * Sparse / dense multi-query attention with sliding window, sink and
 * de-rotated output.
 * [BLOG] "The DeepSeek-V4-Flash architecture" (64 heads read one 512-d latent
 * that is both key and value), "Three attention types" (selected entries or
 * all HCA entries, plus the 128-token window), "Kernel fusions", row
 * "SWA / CSA / HCA attention" (window and softmax sink in one kernel);
 * [PR] item 1 (scale exactly D^-0.5), item 3 (output de-rotated at -t).
 *
 * For query t and head h: keys J(t) = idx[t] (K > 0), or every visible entry
 * s < n_vis(t) (K = 0, r > 0), or none (r = 0); plus window tokens u in
 * [max(0,t-W+1), t] rotated at u.  logits = scale * rot(q[t,h], t) . key;
 * softmax over J(t) with the optional sink logit sink[h] in the
 * denominator; o = sum p * key (V = K); o's last R dims rotated at -t.
 *
 *   q    : [B, S, H, D] un-rotated.           kv   : [B, S, D] un-rotated.
 *   ent  : [B, N, D] rotated entries (v4_compress); NULL iff r == 0.
 *   idx  : [B, S, K] int32; -1 = unused slot; NULL = all visible entries.
 *          Values >= n_vis(t) or < -1 are skipped and flagged
 *          (V4_ERR_BAD_INDEX in the device status).
 *   sink : [H] fp32, nullable.
 *   o    : [B, S, H, D] out.   lse : [B, S, H] fp32 out (natural log), nullable.
 * An empty key set without a sink yields o = 0 and lse = -inf.
 * --------------------------------------------------------------------*/
v4_status v4_sparse_mqa_fwd(const v4_config* cfg, const void* q, const void* kv,
                            const void* ent, const int32_t* idx, const float* sink,
                            const float* inv_freq, void* o, float* lse,
                            void* workspace, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------
 * v4_sparse_mqa_fwd without a workspace: the method has no counterpart for
 * this entry point; it exists for callers that cannot allocate device memory
 * where they run the attention (a serving stack whose planner owns all
 * device memory up front, a plugin that may not call cudaMalloc inside a
 * host framework, a latency-critical path that cannot absorb an
 * allocation).  Arguments and results are those of v4_sparse_mqa_fwd.
 *
 * Scratch comes from one library-owned device array of about 10 MiB, held by
 * every GPU that loads the library until the process exits.  Limits:
 * batch*seqlen <= 8192, batch*seqlen*head_dim*element size <= 8 MiB and
 * seqlen*rope_dim <= 524288; larger problems return V4_ERR_INVALID_ARG with
 * a message.  The call allocates nothing.  The first call on a device looks
 * up the array's device address (cudaGetSymbolAddress, with that device
 * current), so make that first call before any stream capture.  All calls
 * share the array and it keeps the last call's contents: calls that overlap
 * on the GPU (unordered streams, several host threads) race on it.
 * --------------------------------------------------------------------*/
v4_status v4_sparse_mqa_fwd_noalloc(const v4_config* cfg, const void* q, const void* kv,
                                    const void* ent, const int32_t* idx, const float* sink,
                                    const float* inv_freq, void* o, float* lse, void* stream);

/* ----------------------------------------------------------------------
 * Backward of v4_sparse_mqa_fwd: the gradients of L = sum(dout * o).
 * [BLOG] "Attention kernels for the three layer types", backward: a dQ pass
 * that regathers the keys and recomputes the softmax, the delta
 * rowsum(O * dO), and a head-dimension contraction scattered into the
 * key/value gradient (fused here with dQ; fp32 reductions in L2).
 *
 * With p = softmax probabilities of v4_sparse_mqa_fwd (from lse), g =
 * rot(dout, t), delta = dout . o and ds = p (g . key - delta):
 *   dq   = rot(scale * sum_j ds_j key_j, -t)
 *   dkey = scale * sum_h ds_h rot(q_h, t) + sum_h p_h g_h     (key = value)
 *   dent[b, e] = sum of dkey over every (query, slot) that read entry e
 *   dkv[b, u]  = rot(sum of dkey over queries whose window holds u, -u)
 *   dsink[h]   = -sum_t exp(sink[h] - lse[t, h]) delta[t, h]
 *
 * Inputs are those of the forward call plus its outputs:
 *   o    : [B, S, H, D] the forward output.   lse : [B, S, H] fp32 (required).
 *   dout : [B, S, H, D] gradient of o.
 * Outputs (overwritten):
 *   dq    : [B, S, H, D] (storage dtype).
 *   dkv   : [B, S, D] fp32, gradient of the un-rotated window latent kv.
 *   dent  : [B, N, D] fp32, gradient of the rotated entries; required iff
 *           r > 0 and N > 0, else NULL.
 *   dsink : [H] fp32; required iff sink != NULL.
 * Shapes: those of the tensor-core forward (bf16, H a multiple of 64 up to
 * 512, D = 512, R = 64, 1 <= W <= 128, K <= 1024); others return
 * V4_ERR_UNSUPPORTED.  Reduction order of dkv / dent / dsink follows the
 * GPU's scheduling, so they are not bitwise reproducible.
 * workspace : at least v4_bwd_workspace_size bytes, 256-byte aligned.
 * --------------------------------------------------------------------*/
v4_status v4_bwd_workspace_size(const v4_config* cfg, size_t* bytes);
v4_status v4_sparse_mqa_bwd(const v4_config* cfg, const void* q, const void* kv,
                            const void* ent, const int32_t* idx, const float* sink,
                            const float* inv_freq, const void* o, const float* lse,
                            const void* dout, void* dq, float* dkv, float* dent,
                            float* dsink, void* workspace, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------
 * Query projections of the rank-r latent.  [BLOG] "The DeepSeek-V4-Flash
 * architecture": queries arrive through a low-rank path of rank 1024 that
 * the sparse-selection indexer shares.
 *   qlat : [B, S, rank] bf16, the shared latent.
 *   wq   : [rank, H*D] bf16 (row k holds the weights of latent dim k).
 *   q    : [B, S, H, D] out: qlat . wq, and with q_norm = 1 every head
 *          RMS-normalised over its D dims, q / sqrt(mean(q^2) + cfg->rms_eps)
 *          * g with g = q_norm_w [D] fp32 (NULL = ones).
 *   wiq  : [rank, Hi*Di] bf16, nullable; iq : [B, S, Hi, Di] out (required
 *          iff wiq): qlat . wiq.
 * bf16 storage only, fp32 accumulation, one rounding to bf16; rank a
 * multiple of 64 (at most 65536), H*D and Hi*Di multiples of 256, and D =
 * 512 when q_norm = 1; other shapes return V4_ERR_UNSUPPORTED.
 * --------------------------------------------------------------------*/
v4_status v4_q_proj(const v4_config* cfg, const void* qlat, int32_t rank, const void* wq,
                    int32_t q_norm, const float* q_norm_w, const void* wiq, void* q, void* iq,
                    void* stream);

/* ----------------------------------------------------------------------
 * Sparse indexer distillation target.  [PR] item 5: KL(attention ||
 * indexer) over the selected entries, the sparse top-k variant that stays
 * in [B, S, K]; item 11: the target branch is detached and its heads are
 * summed inside the loop, so [B, H, S, K] never exists.
 *
 * With A_h the attention probabilities of v4_sparse_mqa_fwd for head h
 * (window and sink included in the normalisation, given by lse):
 *   target[t,k] = sum_h A_h[idx[t,k]] / sum_k' sum_h A_h[idx[t,k']]
 * over the valid slots (0 on padding and on rows without selections).  With
 * iscore (the indexer scores of the slots, as v4_indexer_topk returns
 * them) and qd = softmax of iscore over the valid slots:
 *   loss[t]     = sum_k target (log target - log qd)     (nullable)
 *   dscore[t,k] = qd - target, the gradient of sum_t loss[t] with respect
 *                 to iscore (0 on padding)                 (nullable)
 *   q    : [B, S, H, D] un-rotated queries.   ent : [B, N, D] rotated entries.
 *   idx  : [B, S, K] selections.              lse : [B, S, H] of the forward.
 * Tensor-core shapes only (bf16, H a multiple of 64 up to 512, D = 512,
 * R = 64, K <= 1024, N <= 65536); others return V4_ERR_UNSUPPORTED.
 * Heads and slices are summed with fp32 atomics (not bitwise reproducible).
 * workspace : at least v4_workspace_size bytes.
 * --------------------------------------------------------------------*/
v4_status v4_indexer_kl_target(const v4_config* cfg, const void* q, const void* ent,
                               const int32_t* idx, const float* lse, const float* iscore,
                               const float* inv_freq, float* target, float* loss, float* dscore,
                               void* workspace, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------
 * Grouped low-rank output projection.  [BLOG] "The DeepSeek-V4-Flash
 * architecture": the 64 x 512 output splits into o_groups groups, each
 * through an o_rank bottleneck.  Group g holds heads g*H/G .. (g+1)*H/G-1
 * concatenated along D.
 *   o    : [B, S, H, D];  wo_a : [G, (H/G)*D, o_rank];  y : [B, S, G*o_rank].
 * bf16 storage; (H/G)*D a multiple of 64 and o_rank a multiple of 256 (other
 * shapes return V4_ERR_UNSUPPORTED).  fp32 accumulation, bf16 result.
 * --------------------------------------------------------------------*/
v4_status v4_grouped_o_proj(const v4_config* cfg, const void* o, const void* wo_a,
                            void* y, void* stream);

/* Pointers of one layer call. Nullable fields are marked. */
typedef struct v4_layer_inputs {
  const void* q;         /* [B,S,H,D] */
  const void* kv;        /* [B,S,D] window latent */
  const void* ckv;       /* [B,S,1+ov,D]     (r > 0) */
  const void* cscore;    /* [B,S,1+ov,D]     (r > 0) */
  const float* ape;      /* [(1+ov)r, D]     (r > 0) */
  const float* norm_w;   /* [D], nullable */
  const void* ickv;      /* [B,S,1+ov,Di]    (K > 0) */
  const void* icscore;   /* [B,S,1+ov,Di]    (K > 0) */
  const float* iape;     /* [(1+ov)r, Di]    (K > 0) */
  const float* inorm_w;  /* [Di], nullable */
  const void* iq;        /* [B,S,Hi,Di] un-rotated (K > 0) */
  const float* w;        /* [B,S,Hi]         (K > 0) */
  const float* sink;     /* [H], nullable */
  const float* inv_freq; /* [R/2] */
  const void* wo_a;      /* [G,(H/G)D,o_rank], nullable = no projection */
} v4_layer_inputs;

typedef struct v4_layer_outputs {
  void* o;               /* [B,S,H,D] */
  float* lse;            /* [B,S,H], nullable */
  void* ent;             /* [B,N,D], nullable (kept in the workspace) */
  void* ikey;            /* [B,N,Di], nullable (kept in the workspace) */
  int32_t* idx;          /* [B,S,K], nullable (kept in the workspace) */
  float* iscore;         /* [B,S,K], nullable */
  void* y;               /* [B,S,G*o_rank], required iff wo_a != NULL */
} v4_layer_outputs;

/* ----------------------------------------------------------------------
 * One attention layer: compressor (r > 0), indexer keys + query prep +
 * scores + top-k (K > 0), attention with window and de-rotation, optional
 * grouped output projection; all on `stream`, no host synchronisation.
 * [PR] Part 1 as a whole; [BLOG] "Three attention types, interleaved".
 * --------------------------------------------------------------------*/
v4_status v4_attn_layer_fwd(const v4_config* cfg, const v4_layer_inputs* in,
                            v4_layer_outputs* out, void* workspace, size_t ws_bytes,
                            void* stream);

/* Text of the last non-OK status returned on this host thread ("" if none). */
const char* v4_last_error(void);

/* Static text naming the build: the target architecture and, for the
 * bound-checking build (compiled with V4_DEBUG), "V4_DEBUG". */
const char* v4_build_info(void);

/* Copy the sticky device status word (a v4_status value, 0 = clean) after
 * synchronising `stream`.  v4_reset_device_status clears it (async). */
v4_status v4_get_device_status(void* stream, int32_t* status);
v4_status v4_reset_device_status(void* stream);

/* Number of kernels this library has launched since it was loaded. */
uint64_t v4_launch_count(void);

/* ----------------------------------------------------------------------
 * Self-test of the device-side failure path (no counterpart in the method).
 * Launches one warp whose lane 0 waits, with the same bounded wait the
 * tensor-core kernels use, on a shared-memory barrier that nothing ever
 * completes; after limit_us microseconds (1 .. 1000000) the wait gives up,
 * records V4_ERR_TIMEOUT in the sticky device status word and the kernel
 * returns.  Nothing traps and no tensor-core or TMA work is in flight, so the
 * context stays usable: the host reads the status with
 * v4_get_device_status and clears it with v4_reset_device_status.
 * --------------------------------------------------------------------*/
v4_status v4_selftest_wait_timeout(int32_t limit_us, void* stream);

/* ----------------------------------------------------------------------
 * Per-stage timing.  While enabled, every stage launch is bracketed by two
 * CUDA events recorded on the stage's stream, so the timing sees exactly the
 * stage's kernels in stream order.  v4_profile_enable(1) discards earlier
 * records and starts recording; v4_profile_enable(0) stops.  Record i
 * (launch order, 0-based) is read with v4_profile_get, which waits for its
 * stop event.  kind: 0 compressor, 1 window-key rotation, 2 indexer query
 * prep, 3 indexer scores, 4 top-k, 5 attention, 6 output projection,
 * 7 backward prep (clears, tables, key rotation, query/gradient rotation and
 * delta), 8 attention backward, 9 window-gradient de-rotation, 10 E4M3
 * quantisation of the indexer operands, 11 query projections, 12 indexer
 * distillation target.
 * --------------------------------------------------------------------*/
v4_status v4_profile_enable(int32_t on);
int32_t v4_profile_count(void);
v4_status v4_profile_get(int32_t i, int32_t* kind, float* ms);

#ifdef __cplusplus
}
#endif
#endif /* V4ATTN_H */
