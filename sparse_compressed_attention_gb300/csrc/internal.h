// Internal launch interface between the C ABI (api.cu) and the kernels.
// Every launcher enqueues on `stream` and returns the launch error (if any).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "v4attn.h"

namespace v4 {

// Counts kernel launches made by the library (reported by v4_launch_count).
void note_launch(int n = 1);

// Query rows per sequence of a call: positions q_begin .. seqlen-1.  Row
// tensors (q, iq, w, o, lse, idx, scores) are indexed by b * q_rows + (t - q_begin);
// sequence tensors (kv, entries) by b * seqlen + t.
inline int q_rows(const v4_config& c) { return c.seqlen - c.q_begin; }

// Argument checks, error text and the device status word (api.cu).
v4_status validate_config(const v4_config* c);
v4_status set_error(v4_status st, const char* msg);
int* device_status_ptr();

// Per-stage timing (v4_profile_*): while timing is on, the launches between
// construction and destruction are bracketed by two CUDA events on `st`
// (api.cu).  `kind` is a stage number of v4_profile_enable's list.
class StageTiming {
 public:
  StageTiming(int kind, cudaStream_t st);
  ~StageTiming();
  StageTiming(const StageTiming&) = delete;
  StageTiming& operator=(const StageTiming&) = delete;

 private:
  void* rec_;
  cudaStream_t st_;
};

// Workspace carve-up for one configuration (Sq = q_rows).  Offsets are
// 256-byte aligned.
struct Workspace {
  size_t kv_rot = 0, kv_rot_bytes = 0;     // rotated window keys [B,S,D]
  size_t ent = 0, ent_bytes = 0;           // entries [B,N,D] (layer call)
  size_t ikey = 0, ikey_bytes = 0;         // indexer keys [B,N,Di] (layer call)
  size_t iqp = 0, iqp_bytes = 0;           // prepared indexer queries [B,Sq,Hi,Di]
  size_t scores = 0, scores_bytes = 0;     // indexer scores [B,Sq,N] fp32
  size_t idx = 0, idx_bytes = 0;           // selected entries [B,Sq,K] (layer call)
  size_t counters = 0, counters_bytes = 0; // work counter, redo count, redo list [2 + B*Sq*slices]
  size_t rope = 0, rope_bytes = 0;         // cos/sin table [S][R/2] float2
  size_t qc8 = 0, qc8_bytes = 0;           // E4M3 indexer: query codes [B,Sq,Hi,Di] u8
  size_t qs8 = 0, qs8_bytes = 0;           //   query scales [B,Sq,Hi] fp32
  size_t kc8 = 0, kc8_bytes = 0;           //   key codes [B,N,Di] u8
  size_t ks8 = 0, ks8_bytes = 0;           //   key scales [B,N] fp32
  size_t total = 0;
};
Workspace plan_workspace(const v4_config& c);

// ---- compressor and preparation kernels (compress.cu)
// cs_table: the per-call cos/sin table of positions < S, or null (angles
// computed in place).
cudaError_t launch_compress(const v4_config& c, const void* ckv, const void* cscore,
                            const float* ape, const float* norm_w, const float* inv_freq,
                            const float2* cs_table, int dim, int hadamard, void* out, cudaStream_t st);
cudaError_t launch_rotate_rows(const v4_config& c, const void* kv, const float* inv_freq,
                               void* kv_rot, cudaStream_t st);
// Rotated window keys: token u of kv rotated at u on the last R dims,
// stored in the storage dtype, from the per-call cos/sin table.
cudaError_t launch_key_prep(const v4_config& c, const void* kv, const float2* cs_table, void* kv_rot,
                            cudaStream_t st);
// cos/sin of every (position < S, rotated pair): table[pos * R/2 + j].
cudaError_t launch_rope_table(const v4_config& c, const float* inv_freq, float2* table, cudaStream_t st);

// ---- TMA descriptors (tma_host.cu); returns 0 on success
int make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                      uint32_t box_rows, bool swizzle128);
int make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                    uint32_t box_rows, bool swizzle128);
// cs_table may be null (angles are then computed in the kernel from inv_freq)
cudaError_t launch_indexer_prep(const v4_config& c, const void* iq, const float2* cs_table,
                                const float* inv_freq, void* iqp, cudaStream_t st);
// The same preparation quantised to E4M3 rows in the kernel (bf16, Di = 128):
// codes [B,Sq,Hi,128] and scales [B,Sq,Hi] instead of the bf16 rows.
cudaError_t launch_indexer_prep_e4m3(const v4_config& c, const void* iq, const float2* cs_table,
                                     const float* inv_freq, uint8_t* codes, float* scales, cudaStream_t st);

// ---- indexer (indexer.cu)
cudaError_t launch_indexer_scores_simt(const v4_config& c, const void* iqp, const void* ikey,
                                       const float* w, float* scores, cudaStream_t st);
bool indexer_tc_supported(const v4_config& c);
cudaError_t launch_indexer_scores_tc(const v4_config& c, const void* iqp, const void* ikey, const float* w,
                                     float* scores, int* status, cudaStream_t st);
// Opt-in E4M3 indexer (indexer_tc.cu): per-row absmax quantisation of bf16
// rows (dim a multiple of 128, <= 1024) and the scores of quantised
// operands (Hi = 64, Di = 128): q codes [B,Sq,64,128] with scales [B,Sq,64],
// key codes [B,N,128] with scales [B,N].
cudaError_t launch_quant_e4m3(const void* x, long long rows, int dim, uint8_t* codes, float* scales,
                              cudaStream_t st);
bool indexer_e4m3_supported(const v4_config& c);
cudaError_t launch_indexer_scores_e4m3(const v4_config& c, const uint8_t* qc, const float* qs, const uint8_t* kc,
                                       const float* ks, const float* w, float* scores, int* status,
                                       cudaStream_t st);
cudaError_t launch_topk(const v4_config& c, const float* scores, int32_t* idx, float* iscore,
                        cudaStream_t st);

// ---- attention (mqa.cu)
// `list` (nullable): list[0] = number of queries, list[1..] = b*Sq + (t - q_begin)
// of each (its query row); when given, only those queries are computed.
cudaError_t launch_mqa_simt(const v4_config& c, const void* q, const void* kv_rot,
                            const void* ent, const int32_t* idx, const float* sink,
                            const float* inv_freq, void* o, float* lse, int* status,
                            const int* list, cudaStream_t st);
bool mqa_tc_supported(const v4_config& c);

// ---- grouped output projection (oproj_tc.cu)
bool oproj_tc_supported(const v4_config& c);
cudaError_t launch_oproj_tc(const v4_config& c, const void* o, const void* wo_a, void* y, int* status,
                            cudaStream_t st);
// Query projection y[T, N] = x[T, rank] . w[rank, N] (bf16, fp32 accumulate);
// norm = 1 RMS-normalises every 512-wide column block (N % 512 == 0),
// weight norm_w [512] or ones.  rank % 64 == 0, N % 256 == 0.
cudaError_t launch_qproj_tc(long long T, int rank, const void* x, const void* w, int N, void* y, int norm,
                            float eps, const float* norm_w, int* status, cudaStream_t st);
cudaError_t launch_mqa_tc(const v4_config& c, const void* q, const void* kv_rot, const void* ent,
                          const int32_t* idx, const float* sink, const float2* cs_table, void* o, float* lse,
                          int* counters, int* status, cudaStream_t st);

// ---- sparse indexer distillation target (kl_target_tc.cu)
bool kl_target_tc_supported(const v4_config& c);
// target [B,S,K] (written), loss [B,S] and dscore [B,S,K] nullable (need iscore)
cudaError_t launch_kl_target(const v4_config& c, const void* q, const void* ent, const int32_t* idx,
                             const float* lse, const float* iscore, const float2* cs_table, float* target,
                             float* loss, float* dscore, int* status, cudaStream_t st);

// ---- attention backward (mqa_bwd_tc.cu)
bool mqa_bwd_tc_supported(const v4_config& c);
// qr = rot(q, t), dor = rot(dout, t) (storage dtype), delta = dout . o per
// (query, head); dsink (nullable, pre-zeroed) += -exp(sink - lse) delta.
cudaError_t launch_mqa_bwd_prep(const v4_config& c, const void* q, const void* o, const void* dout,
                                const float* lse, const float* sink, const float2* cs_table, void* qr, void* dor,
                                float* delta, float* dsink, cudaStream_t st);
// dq, and the fp32 reductions into dkv (gradient of the rotated window keys,
// pre-zeroed) and dent (pre-zeroed; nullable when there are no entries).
cudaError_t launch_mqa_bwd_tc(const v4_config& c, const void* qr, const void* dor, const void* kv_rot,
                              const void* ent, const int32_t* idx, const float* lse, const float* delta,
                              const float2* cs_table, void* dq, float* dkv, float* dent, int* status,
                              cudaStream_t st);
// dkv[b, u] = rot(dkv[b, u], -u) in place
cudaError_t launch_mqa_bwd_derotate(const v4_config& c, float* dkv, const float2* cs_table, cudaStream_t st);

}  // namespace v4
