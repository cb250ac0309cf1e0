// Device helpers shared by the kernels of the compressed-attention library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace v4 {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// 8-element vector loads / stores (16 B for bf16, 32 B for f32); values are
// widened to / rounded from float (round to nearest even for bf16).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void load8(const float* p, float* v) {
  float4 a = reinterpret_cast<const float4*>(p)[0];
  float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const bf16* p, float* v) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ void store8(float* p, const float* v) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ void store8(bf16* p, const float* v) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void from_f(bf16* p, float x) { *p = __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------
// RoPE angle.  phi = pos * inv_freq is formed exactly in double (a 64-bit
// integer times a float fits the double mantissa for |pos| < 2^29), reduced
// by the nearest multiple of 2*pi in double, and only then narrowed to float
// for CUDA's sincosf.  This keeps the angle error near one float ulp of the
// reduced angle even at positions of 10^6.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void rope_cos_sin(long long pos, float inv_freq, float* c, float* s) {
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  double a = (double)pos * (double)inv_freq;
  double k = rint(a * inv_two_pi);
  double red = fma(-k, two_pi, a);
  sincosf((float)red, s, c);
}

// Rotate one interleaved pair (a, b) by (c, s).
__device__ __forceinline__ void rot_pair(float& a, float& b, float c, float s) {
  float x = a * c - b * s;
  float y = a * s + b * c;
  a = x;
  b = y;
}

// ---------------------------------------------------------------------------
// Sticky device status: the first non-zero code wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

constexpr int kStatusTimeout = 5;
constexpr int kStatusBadIndex = 6;
constexpr int kStatusBound = 7;

// Bound checks of the V4_DEBUG build (compiled out otherwise): an index that
// fails its bound records kStatusBound and the guarded access is skipped, so
// a bad gather row, ring slot or TMEM column shows up in the status word
// instead of touching memory outside its buffer.
#ifdef V4_DEBUG
#define V4_BOUND(cond, status) ((cond) ? true : (::v4::set_status((status), ::v4::kStatusBound), false))
#else
#define V4_BOUND(cond, status) true
#endif

__device__ __forceinline__ int n_visible(long long t, int ratio) {
  return ratio > 0 ? (int)((t + 1) / ratio) : 0;
}

}  // namespace v4
