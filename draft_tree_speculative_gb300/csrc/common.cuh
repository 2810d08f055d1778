// Shared device helpers of the CUDA path: error reporting, bf16 packing and
// RoPE angles. Nothing here is shared with the CPU oracle.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "dts.h"

namespace dts {

constexpr int kMaxNodes = 64;

// First error wins: a zero word becomes `code`; later errors leave it alone.
__device__ __forceinline__ void report(int32_t *err, int code) {
  if (err != nullptr) atomicCAS(reinterpret_cast<int *>(err), 0, code);
}

// Programmatic dependent launch. A kernel of the verify step may be launched
// before the kernel ahead of it in the stream has finished (launch_chained
// below), so its launch and block scheduling overlap that kernel's tail.
// grid_dep_wait() blocks until the kernel ahead has completed and its memory
// operations are visible; every such kernel calls it before it touches
// global memory. grid_dep_launch_next() lets the next kernel in the stream
// be launched once every block of this grid has issued it (or exited); its
// blocks then wait in their own grid_dep_wait(). Both are no-ops for a
// kernel launched the ordinary way.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_next() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float f16_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// Pack two floats as bf16 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
// Pack two floats as f16 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
// Two E4M3 bytes (the low byte is the first element) widened to f16, exactly:
// every E4M3 value, subnormals included, is a normal f16 value (or zero), and
// the E4M3 NaN becomes an f16 NaN.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_bytes), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}
// Two floats to E4M3 bytes (`lo` in the low byte): round to nearest even,
// saturating at +-448; NaN stays NaN.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3)) & 0xFFFFu;
}

// ---------------------------------------------------------------------------
// RoPE angles.
//
// Position p (an integer < 2^24) and frequency w_k = theta^(-2k/d) give the
// angle p * w_k, which reaches ~1.3e5 rad at the long-context positions. A
// plain fp32 product would carry ~1e-2 rad of error there. The host passes
// w_k as an unevaluated sum hi + lo of two floats (from a double); the device
// forms p * w exactly as a float-float pair (Dekker's product by FMA: the
// rounding error of p*hi is fma(p, hi, -p*hi)), then reduces modulo 2*pi
// with a three-part constant (Cody and Waite's additive range reduction).
// The first FMA of the reduction is exact because both terms are multiples of
// ulp(2*pi) and the result is below 2^24 of those units. The reduced angle is
// in [-pi, pi] up to ~3e-7 rad, where the hardware sine/cosine are accurate
// to ~5e-7; both are far below bf16 resolution.
// ---------------------------------------------------------------------------
struct RopeFreqs {
  float2 w[64];  // (hi, lo) for k < d/2, d <= 128
};

__device__ __forceinline__ float rope_reduced_angle(int pos, float2 w) {
  const float p = static_cast<float>(pos);
  const float a_hi = __fmul_rn(p, w.x);  // rounded product, never contracted
  const float a_err = fmaf(p, w.x, -a_hi);
  const float a_lo = fmaf(p, w.y, a_err);
  const float kTwoPi1 = 6.28318548202514648438f;        // float(2*pi)
  const float kTwoPi2 = -1.74845553146951715462e-07f;   // float(2*pi - kTwoPi1)
  const float kTwoPi3 = -6.86049804002352749122e-15f;   // float(2*pi - kTwoPi1 - kTwoPi2)
  const float kInvTwoPi = 0.15915493667125701904f;
  const float n = rintf(a_hi * kInvTwoPi);
  float r = fmaf(-n, kTwoPi1, a_hi);
  r = fmaf(-n, kTwoPi2, r);
  r = fmaf(-n, kTwoPi3, r);
  return r + a_lo;
}

__device__ __forceinline__ void rope_sincos(int pos, float2 w, float *s, float *c) {
  __sincosf(rope_reduced_angle(pos, w), s, c);
}

}  // namespace dts

// Host helpers (defined in api.cu).
namespace dts_host {
// Launches `kernel` on stream `s` with programmatic stream serialization: it
// may start while the kernel ahead of it in the stream is still running and
// must call dts::grid_dep_wait() before its first global-memory access.
template <typename... Params, typename... Args>
cudaError_t launch_chained(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                           Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
void make_rope_freqs(float theta, int d, dts::RopeFreqs *out);
int launch_status();  // DTS_OK or DTS_ERR_CUDA from cudaGetLastError()
int sm_count();
}  // namespace dts_host
