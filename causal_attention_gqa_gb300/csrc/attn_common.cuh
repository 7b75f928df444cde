// Shared device helpers of the attention library: problem geometry, the
// library status word, NEOX RoPE angles and bf16 conversions.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace attn {

// Status codes (mirror attn_status_t of the public header).
constexpr int kOk = 0;
constexpr int kErrDeviceTimeout = -7;
constexpr int kErrBadArgument = -8;

// Geometry of one call.  Packed qkv rows hold Q | K | V column blocks:
// query head h at h*hd, kv head kh at C + kh*hd (K) and C + NKV*hd + kh*hd
// (V) -- the layout of "nanoeuler -- CUDA kernels", causal GQA attention.
struct Geometry {
  int B, T, C, NH, NKV;
  int hd;        // head size C / NH
  int grp;       // query heads per kv head NH / NKV
  int W;         // packed row width (NH + 2*NKV) * hd
  float scale;   // 1 / sqrt(hd)
  float rope_theta;  // <= 0: no RoPE
  // 0: NEOX pairs (i, i + hd/2); 1: interleaved (GPT-J) pairs (2i, 2i+1).  The
  // kernels work on NEOX-ordered rotated rows either way: an interleaved head
  // row is read with its even elements first (pair i moves to slots i and
  // i + hd/2), and gradients are written back through the same permutation.
  // Scores q . k are unchanged by a permutation shared by Q and K.
  int rope_interleaved;
  // RoPE inverse frequencies theta^(-2i/hd), i < hd/2, as float head + tail
  // (computed once on the host in double precision).
  float rope_f_hi[64];
  float rope_f_lo[64];
};

// Record the first device-side error in the library status word.
__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, kOk, code);
}

// ---------------------------------------------------------------------------
// NEOX RoPE ("nx_f32_qwen2_train_gate.nx source", build_rope / rope_node):
// pair (i, i + hd/2) at position t turns by angle t * theta^(-2i/hd):
//   y_i        = x_i cos(a) - x_{i+hd/2} sin(a)
//   y_{i+hd/2} = x_{i+hd/2} cos(a) + x_i sin(a)
// ---------------------------------------------------------------------------

// The angle t * f reduced to about [-pi, pi], good to ~1e-6 rad for any
// t < 2^24.  The product is formed error-free with an FMA (Dekker's
// two-product), and 2*pi is subtracted in three parts (Cody & Waite, 1980):
// C1 has 8 significant bits so k*C1 is exact for |k| < 2^16, and C2, C3 are
// the float head and tail of 2*pi - C1.
__device__ __forceinline__ float rope_angle(int t, float f_hi, float f_lo) {
  const float kInv2Pi = 0.159154943091895336f;
  const float kC1 = 6.28125f;
  const float kC2 = 1.9353071693331003e-3f;    // float(2*pi - C1)
  const float kC3 = 1.0253376273028358e-11f;   // float(2*pi - C1 - C2)
  float tf = (float)t;
  float p = tf * f_hi;
  float e = fmaf(tf, f_hi, -p);      // exact rounding error of the product
  float lo = fmaf(tf, f_lo, e);
  float k = rintf(p * kInv2Pi);
  float r = p - k * kC1;              // exact (Sterbenz)
  r = fmaf(-k, kC2, r);
  r = fmaf(-k, kC3, r);
  return r + lo;
}

// The rounding steps are spelled out (one product, then one fused
// multiply-add) so that every kernel that rotates a row gets the same bits,
// whatever the compiler would contract.
__device__ __forceinline__ void rope_pair(float x0, float x1, float c, float s, float& y0, float& y1) {
  y0 = __fmaf_rn(x0, c, __fmul_rn(-x1, s));
  y1 = __fmaf_rn(x1, c, __fmul_rn(x0, s));
}

// Adjoint (inverse) rotation: R^T applied to a gradient pair.
__device__ __forceinline__ void rope_pair_transpose(float g0, float g1, float c, float s, float& y0, float& y1) {
  y0 = __fmaf_rn(g0, c, __fmul_rn(g1, s));
  y1 = __fmaf_rn(g1, c, __fmul_rn(-g0, s));
}

// ---------------------------------------------------------------------------
// bf16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The eight pairs 8 gi .. 8 gi + 7 of one bf16 head row as two 16-byte words:
// x0 holds the first elements of the pairs, x1 the second ones.  NEOX pairs
// (i, i + hd/2) are two contiguous runs; interleaved pairs (2i, 2i+1) are the
// sixteen elements 16 gi .. 16 gi + 15, split into even and odd ones.
__device__ __forceinline__ void load_rope_pairs(const __nv_bfloat16* head_row, int gi, int half, bool interleaved,
                                                uint4& x0, uint4& x1) {
  if (!interleaved) {
    x0 = *reinterpret_cast<const uint4*>(head_row + gi * 8);
    x1 = *reinterpret_cast<const uint4*>(head_row + half + gi * 8);
    return;
  }
  const uint4 u = *reinterpret_cast<const uint4*>(head_row + gi * 16);
  const uint4 v = *reinterpret_cast<const uint4*>(head_row + gi * 16 + 8);
  auto even = [](uint32_t a, uint32_t b) { return (a & 0xFFFFu) | (b << 16); };
  auto odd = [](uint32_t a, uint32_t b) { return (a >> 16) | (b & 0xFFFF0000u); };
  x0 = make_uint4(even(u.x, u.y), even(u.z, u.w), even(v.x, v.y), even(v.z, v.w));
  x1 = make_uint4(odd(u.x, u.y), odd(u.z, u.w), odd(v.x, v.y), odd(v.z, v.w));
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace attn
