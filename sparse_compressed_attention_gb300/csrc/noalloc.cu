// Sparse / dense multi-query attention forward whose scratch memory is owned
// by the library: a file-scope device array instead of a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// attention: an inference server whose memory planner hands out every byte of
// device memory up front, a plugin loaded into another framework that must not
// call cudaMalloc or reach into that framework's allocator, or a
// latency-critical path where an allocation and its implicit synchronisation
// are not acceptable.  They still own their inputs and outputs; this entry
// point needs nothing else from them.
//
// The scratch array below lives in every GPU that loads the library, until
// the process exits.  All calls share it: two calls that overlap on the GPU
// (different streams, no ordering between them) race on it.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace v4 {

namespace {

// Limits of the shared scratch: at most 8192 tokens (B*S), at most 8 MiB of
// rotated window keys (B*S*D*element size) and S*R <= 524288 (the cos/sin
// table).  The Flash shapes (D=512, R=64, bf16) reach all three at B*S=8192.
constexpr long long kMaxTokens = 8192;
constexpr size_t kKvBytes = 8u << 20;
constexpr size_t kCounterBytes = (2 + 8 * kMaxTokens) * sizeof(int);      // up to 8 head slices
constexpr size_t kRopeBytes = 524288 / 2 * sizeof(float2);
constexpr size_t kOffCounters = kKvBytes;
constexpr size_t kOffRope = (kOffCounters + kCounterBytes + 255) & ~(size_t)255;
constexpr size_t kScratchBytes = kOffRope + kRopeBytes;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch for the current device.  Host code cannot use
// the symbol itself (it names a host-side stand-in), so the address is looked
// up once per device with that device current, and cached.
unsigned char* scratch_ptr(v4_status* st) {
  static std::mutex mu;
  static unsigned char* cache[128] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    *st = set_error(V4_ERR_CUDA, "no current CUDA device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) {
      *st = set_error(V4_ERR_CUDA, cudaGetErrorString(e));
      return nullptr;
    }
    cache[dev] = (unsigned char*)p;
  }
  return cache[dev];
}

}  // namespace

}  // namespace v4

using namespace v4;

extern "C" v4_status v4_sparse_mqa_fwd_noalloc(const v4_config* cfg, const void* q, const void* kv,
                                               const void* ent, const int32_t* idx, const float* sink,
                                               const float* inv_freq, void* o, float* lse, void* stream) {
  v4_status s = validate_config(cfg);
  if (s != V4_OK) return s;
  const v4_config& c = *cfg;
  const long long tokens = (long long)c.batch * c.seqlen;
  const size_t es = c.dtype == V4_BF16 ? 2 : 4;
  if (tokens > kMaxTokens) return set_error(V4_ERR_INVALID_ARG, "no-alloc attention: batch*seqlen above 8192");
  if ((size_t)tokens * c.head_dim * es > kKvBytes)
    return set_error(V4_ERR_INVALID_ARG, "no-alloc attention: window keys above 8 MiB (batch*seqlen*head_dim*size)");
  if ((long long)c.seqlen * c.rope_dim > 524288)
    return set_error(V4_ERR_INVALID_ARG, "no-alloc attention: seqlen*rope_dim above 524288");
  const int N = c.ratio > 0 ? c.seqlen / c.ratio : 0;
  auto aligned = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
  if (!q || !kv || !o || !aligned(q) || !aligned(kv) || !aligned(o))
    return set_error(V4_ERR_INVALID_ARG, "q, kv and o must be non-null and 16-byte aligned");
  if (c.ratio > 0 && N > 0 && (!ent || !aligned(ent)))
    return set_error(V4_ERR_INVALID_ARG, "ent must be non-null and 16-byte aligned");
  if (c.topk > 0 && (!idx || !aligned(idx))) return set_error(V4_ERR_INVALID_ARG, "idx must be non-null and 16-byte aligned");
  if ((sink && !aligned(sink)) || (lse && !aligned(lse)))
    return set_error(V4_ERR_INVALID_ARG, "sink and lse must be 16-byte aligned");
  if (c.rope_dim > 0 && (!inv_freq || !aligned(inv_freq)))
    return set_error(V4_ERR_INVALID_ARG, "inv_freq must be non-null and 16-byte aligned");
  if (c.path == V4_PATH_TC && !mqa_tc_supported(c))
    return set_error(V4_ERR_UNSUPPORTED, "tensor-core attention needs bf16, H a multiple of 64 up to 512, D=512, R=64, 1 <= W <= 128, K <= 1024");
  unsigned char* base = scratch_ptr(&s);
  if (!base) return s;
  int* status = device_status_ptr();
  if (!status) return set_error(V4_ERR_CUDA, "device status word unavailable");
  cudaStream_t st = (cudaStream_t)stream;
  void* kv_rot = base;
  int* counters = (int*)(base + kOffCounters);
  float2* table = (float2*)(base + kOffRope);
  const int32_t* sel = c.topk > 0 ? idx : nullptr;
  cudaError_t e;
  // stage timing as in v4_sparse_mqa_fwd: kind 1 (window keys), kind 5 (attention)
  constexpr int kKindRotate = 1, kKindAttention = 5;
  if (c.path != V4_PATH_SIMT && mqa_tc_supported(c)) {
    {
      StageTiming tm(kKindRotate, st);
      if ((e = launch_rope_table(c, inv_freq, table, st)) != cudaSuccess)
        return set_error(V4_ERR_CUDA, cudaGetErrorString(e));
      if ((e = launch_key_prep(c, kv, table, kv_rot, st)) != cudaSuccess)
        return set_error(V4_ERR_CUDA, cudaGetErrorString(e));
    }
    {
      StageTiming tm(kKindAttention, st);
      // launch_mqa_tc clears the redo count it needs before its kernel runs
      if ((e = launch_mqa_tc(c, q, kv_rot, ent, sel, sink, table, o, lse, counters, status, st)) != cudaSuccess)
        return set_error(V4_ERR_CUDA, cudaGetErrorString(e));
    }
    if ((e = launch_mqa_simt(c, q, kv_rot, ent, sel, sink, inv_freq, o, lse, status, counters + 1, st)) != cudaSuccess)
      return set_error(V4_ERR_CUDA, cudaGetErrorString(e));
    return V4_OK;
  }
  {
    StageTiming tm(kKindRotate, st);
    if ((e = launch_rotate_rows(c, kv, inv_freq, kv_rot, st)) != cudaSuccess)
      return set_error(V4_ERR_CUDA, cudaGetErrorString(e));
  }
  StageTiming tm(kKindAttention, st);
  if ((e = launch_mqa_simt(c, q, kv_rot, ent, sel, sink, inv_freq, o, lse, status, nullptr, st)) != cudaSuccess)
    return set_error(V4_ERR_CUDA, cudaGetErrorString(e));
  return V4_OK;
}
