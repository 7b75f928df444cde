// Exact float32 causal MHA/GQA attention on CUDA cores (dtype F32).
//
// The float32 path keeps every product and sum in IEEE float32 FMAs (no
// tensor-core rounding), so it meets a 1e-4 relative bar against a float64
// restatement of the method.  It serves the tiny heads (hd 4 and 16) where
// tensor-core tiles would be mostly padding, and any other head size up to
// 128.
//
// Forward: one CTA per (32-query tile, head, batch row); 8 warps, 4 queries
// per warp.  Key/value tiles of 32 rows are staged in shared memory (RoPE
// applied as they land), each lane scores one key, and the row softmax is
// kept online (running max m, running sum l, rescaled accumulator), which
// reorders -- but does not change -- the sums of "nanoeuler -- CUDA kernels",
// attention_forward_kernel.
//
// Backward: the gradient of "nanoeuler"'s attention_backward_kernel, with the
// softmax Jacobian folded into dS = P * (dP - D) where D = rowsum(dO * O)
// ("CUDA C microgpt", attention_backward_kernel's weighted_sum).  Two
// kernels, both free of atomics: one owns a key tile and sums dK, dV over
// every query tile and every query head of its group; the other owns a query
// tile and sums dQ over its key tiles.
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_profile.h"

#include <math.h>

namespace attn {
namespace {

constexpr int kTile = 32;        // queries per CTA tile and keys per key tile
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerWarp = kTile / kWarps;

// Load `rows` rows of one head (columns col0 .. col0+hd) starting at position
// t0 into shared memory with row pitch hd+1, optionally NEOX-rotated.
__device__ void load_head_tile(float* dst, const float* src, const Geometry& g, int b, int t0,
                               int col0, bool rope, const float* f_hi, const float* f_lo) {
  const int hd = g.hd, pitch = hd + 1;
  if (!rope) {
    for (int idx = threadIdx.x; idx < kTile * hd; idx += blockDim.x) {
      int r = idx / hd, d = idx % hd, t = t0 + r;
      dst[r * pitch + d] = (t < g.T) ? src[((size_t)b * g.T + t) * g.W + col0 + d] : 0.f;
    }
    return;
  }
  const int half = hd / 2;
  for (int idx = threadIdx.x; idx < kTile * half; idx += blockDim.x) {
    int r = idx / half, i = idx % half, t = t0 + r;
    float y0 = 0.f, y1 = 0.f;
    if (t < g.T) {
      const float* row = src + ((size_t)b * g.T + t) * g.W + col0;
      float s, c;
      sincosf(rope_angle(t, f_hi[i], f_lo[i]), &s, &c);
      // Interleaved pair i is (2i, 2i+1); it lands in NEOX slots i, i + hd/2.
      const int i0 = g.rope_interleaved ? 2 * i : i, i1 = g.rope_interleaved ? 2 * i + 1 : i + half;
      rope_pair(row[i0], row[i1], c, s, y0, y1);
    }
    dst[r * pitch + i] = y0;
    dst[r * pitch + i + half] = y1;
  }
}

__device__ void init_rope_freqs(const Geometry& g, float* f_hi, float* f_lo) {
  for (int i = threadIdx.x; i < 64; i += blockDim.x) {
    f_hi[i] = g.rope_f_hi[i];
    f_lo[i] = g.rope_f_lo[i];
  }
}

// Write `rows` rows of a float32 gradient tile (pitch hd+1 in shared memory)
// to dqkv columns col0.., undoing the RoPE rotation at each row's position.
__device__ void store_grad_tile(float* dqkv, const float* tile, const Geometry& g, int b, int t0,
                                int col0, bool rope, const float* f_hi, const float* f_lo) {
  const int hd = g.hd, pitch = hd + 1;
  if (!rope) {
    for (int idx = threadIdx.x; idx < kTile * hd; idx += blockDim.x) {
      int r = idx / hd, d = idx % hd, t = t0 + r;
      if (t < g.T) dqkv[((size_t)b * g.T + t) * g.W + col0 + d] = tile[r * pitch + d];
    }
    return;
  }
  const int half = hd / 2;
  for (int idx = threadIdx.x; idx < kTile * half; idx += blockDim.x) {
    int r = idx / half, i = idx % half, t = t0 + r;
    if (t >= g.T) continue;
    float s, c, y0, y1;
    sincosf(rope_angle(t, f_hi[i], f_lo[i]), &s, &c);
    rope_pair_transpose(tile[r * pitch + i], tile[r * pitch + i + half], c, s, y0, y1);
    float* row = dqkv + ((size_t)b * g.T + t) * g.W + col0;
    row[g.rope_interleaved ? 2 * i : i] = y0;
    row[g.rope_interleaved ? 2 * i + 1 : i + half] = y1;
  }
}

// ---------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------
template <int DPL>  // head dims per lane: ceil(hd / 32)
__global__ void __launch_bounds__(kThreads)
simt_fwd_kernel(float* __restrict__ out, float* __restrict__ lse, const float* __restrict__ qkv, Geometry g) {
  extern __shared__ float smem[];
  const int pitch = g.hd + 1;
  float* Qs = smem;
  float* Ks = Qs + kTile * pitch;
  float* Vs = Ks + kTile * pitch;
  float* f_hi = Vs + kTile * pitch;
  float* f_lo = f_hi + 64;

  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int kh = h / g.grp;
  const int q0 = qt * kTile;
  const bool rope = g.rope_theta > 0.f;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  init_rope_freqs(g, f_hi, f_lo);
  __syncthreads();
  load_head_tile(Qs, qkv, g, b, q0, h * g.hd, rope, f_hi, f_lo);

  float m[kRowsPerWarp], l[kRowsPerWarp], o[kRowsPerWarp][DPL];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) o[r][j] = 0.f;
  }

  const int q_last = min(q0 + kTile, g.T) - 1;
  for (int k0 = 0; k0 <= q_last; k0 += kTile) {
    __syncthreads();
    load_head_tile(Ks, qkv, g, b, k0, g.C + kh * g.hd, rope, f_hi, f_lo);
    load_head_tile(Vs, qkv, g, b, k0, g.C + g.NKV * g.hd + kh * g.hd, false, f_hi, f_lo);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int qr = warp * kRowsPerWarp + r, tq = q0 + qr;
      if (tq >= g.T || k0 > tq) continue;  // warp-uniform
      const int key = k0 + lane;
      float s = -INFINITY;
      if (key <= tq) {
        float acc = 0.f;
        for (int d = 0; d < g.hd; ++d) acc = fmaf(Qs[qr * pitch + d], Ks[lane * pitch + d], acc);
        s = acc * g.scale;
      }
      const float m_new = fmaxf(m[r], warp_max(s));  // finite: key k0 <= tq is allowed
      const float p = (key <= tq) ? expf(s - m_new) : 0.f;
      const float corr = expf(m[r] - m_new);         // 0 on the first tile (m = -inf)
      l[r] = l[r] * corr + warp_sum(p);
      m[r] = m_new;
#pragma unroll
      for (int j = 0; j < DPL; ++j) o[r][j] *= corr;
      for (int k = 0; k < kTile; ++k) {
        const float pk = __shfl_sync(0xffffffffu, p, k);
#pragma unroll
        for (int j = 0; j < DPL; ++j) {
          const int d = lane + 32 * j;
          if (d < g.hd) o[r][j] = fmaf(pk, Vs[k * pitch + d], o[r][j]);
        }
      }
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int tq = q0 + warp * kRowsPerWarp + r;
    if (tq >= g.T) continue;
    const float inv_l = 1.f / l[r];
    float* orow = out + ((size_t)b * g.T + tq) * g.C + h * g.hd;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const int d = lane + 32 * j;
      if (d < g.hd) orow[d] = o[r][j] * inv_l;
    }
    if (lane == 0) lse[((size_t)b * g.NH + h) * g.T + tq] = m[r] + logf(l[r]);
  }
}

// ---------------------------------------------------------------------------
// Backward, key-stationary part: dK and dV of one key tile of one kv head.
// ---------------------------------------------------------------------------
template <int DPL>
__global__ void __launch_bounds__(kThreads)
simt_bwd_dkdv_kernel(float* __restrict__ dqkv, const float* __restrict__ qkv, const float* __restrict__ dout,
                     const float* __restrict__ lse, const float* __restrict__ Drow, Geometry g) {
  extern __shared__ float smem[];
  const int pitch = g.hd + 1;
  float* Ks = smem;
  float* Vs = Ks + kTile * pitch;
  float* Qs = Vs + kTile * pitch;
  float* dOs = Qs + kTile * pitch;
  float* lse_s = dOs + kTile * pitch;
  float* D_s = lse_s + kTile;
  float* f_hi = D_s + kTile;
  float* f_lo = f_hi + 64;

  const int kt = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int k0 = kt * kTile;
  const bool rope = g.rope_theta > 0.f;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  init_rope_freqs(g, f_hi, f_lo);
  __syncthreads();
  load_head_tile(Ks, qkv, g, b, k0, g.C + kh * g.hd, rope, f_hi, f_lo);
  load_head_tile(Vs, qkv, g, b, k0, g.C + g.NKV * g.hd + kh * g.hd, false, f_hi, f_lo);

  float dk[kRowsPerWarp][DPL], dv[kRowsPerWarp][DPL];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int j = 0; j < DPL; ++j) dk[r][j] = dv[r][j] = 0.f;

  for (int h = kh * g.grp; h < (kh + 1) * g.grp; ++h) {
    for (int q0 = k0; q0 < g.T; q0 += kTile) {  // query tiles that can see this key tile
      __syncthreads();
      load_head_tile(Qs, qkv, g, b, q0, h * g.hd, rope, f_hi, f_lo);
      for (int idx = threadIdx.x; idx < kTile * g.hd; idx += blockDim.x) {
        int r = idx / g.hd, d = idx % g.hd, t = q0 + r;
        dOs[r * pitch + d] = (t < g.T) ? dout[((size_t)b * g.T + t) * g.C + h * g.hd + d] : 0.f;
      }
      for (int r = threadIdx.x; r < kTile; r += blockDim.x) {
        int t = q0 + r;
        lse_s[r] = (t < g.T) ? lse[((size_t)b * g.NH + h) * g.T + t] : 0.f;
        D_s[r] = (t < g.T) ? Drow[((size_t)b * g.NH + h) * g.T + t] : 0.f;
      }
      __syncthreads();
      const int tq = q0 + lane;  // this lane's query
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        const int kr = warp * kRowsPerWarp + r, ks = k0 + kr;
        if (ks >= g.T) continue;  // warp-uniform
        float P = 0.f, dS = 0.f;
        if (tq >= ks && tq < g.T) {
          float sacc = 0.f, pacc = 0.f;
          for (int d = 0; d < g.hd; ++d) {
            sacc = fmaf(Qs[lane * pitch + d], Ks[kr * pitch + d], sacc);
            pacc = fmaf(dOs[lane * pitch + d], Vs[kr * pitch + d], pacc);
          }
          P = expf(sacc * g.scale - lse_s[lane]);
          dS = P * (pacc - D_s[lane]);
        }
        for (int q = 0; q < kTile; ++q) {
          const float Pq = __shfl_sync(0xffffffffu, P, q);
          const float dSq = __shfl_sync(0xffffffffu, dS, q);
#pragma unroll
          for (int j = 0; j < DPL; ++j) {
            const int d = lane + 32 * j;
            if (d < g.hd) {
              dv[r][j] = fmaf(Pq, dOs[q * pitch + d], dv[r][j]);
              dk[r][j] = fmaf(dSq, Qs[q * pitch + d], dk[r][j]);
            }
          }
        }
      }
    }
  }

  // dK goes back through the rotation; reuse the Q tile buffer for staging.
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int kr = warp * kRowsPerWarp + r;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const int d = lane + 32 * j;
      if (d < g.hd) {
        Qs[kr * pitch + d] = dk[r][j] * g.scale;
        dOs[kr * pitch + d] = dv[r][j];
      }
    }
  }
  __syncthreads();
  store_grad_tile(dqkv, Qs, g, b, k0, g.C + kh * g.hd, rope, f_hi, f_lo);
  store_grad_tile(dqkv, dOs, g, b, k0, g.C + g.NKV * g.hd + kh * g.hd, false, f_hi, f_lo);
}

// ---------------------------------------------------------------------------
// Backward, query-stationary part: dQ of one query tile of one head.
// ---------------------------------------------------------------------------
template <int DPL>
__global__ void __launch_bounds__(kThreads)
simt_bwd_dq_kernel(float* __restrict__ dqkv, const float* __restrict__ qkv, const float* __restrict__ dout,
                   const float* __restrict__ lse, const float* __restrict__ Drow, Geometry g) {
  extern __shared__ float smem[];
  const int pitch = g.hd + 1;
  float* Qs = smem;
  float* dOs = Qs + kTile * pitch;
  float* Ks = dOs + kTile * pitch;
  float* Vs = Ks + kTile * pitch;
  float* f_hi = Vs + kTile * pitch;
  float* f_lo = f_hi + 64;

  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int kh = h / g.grp;
  const int q0 = qt * kTile;
  const bool rope = g.rope_theta > 0.f;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  init_rope_freqs(g, f_hi, f_lo);
  __syncthreads();
  load_head_tile(Qs, qkv, g, b, q0, h * g.hd, rope, f_hi, f_lo);
  for (int idx = threadIdx.x; idx < kTile * g.hd; idx += blockDim.x) {
    int r = idx / g.hd, d = idx % g.hd, t = q0 + r;
    dOs[r * pitch + d] = (t < g.T) ? dout[((size_t)b * g.T + t) * g.C + h * g.hd + d] : 0.f;
  }

  float dq[kRowsPerWarp][DPL], lse_r[kRowsPerWarp], D_r[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int tq = q0 + warp * kRowsPerWarp + r;
    lse_r[r] = (tq < g.T) ? lse[((size_t)b * g.NH + h) * g.T + tq] : 0.f;
    D_r[r] = (tq < g.T) ? Drow[((size_t)b * g.NH + h) * g.T + tq] : 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) dq[r][j] = 0.f;
  }

  const int q_last = min(q0 + kTile, g.T) - 1;
  for (int k0 = 0; k0 <= q_last; k0 += kTile) {
    __syncthreads();
    load_head_tile(Ks, qkv, g, b, k0, g.C + kh * g.hd, rope, f_hi, f_lo);
    load_head_tile(Vs, qkv, g, b, k0, g.C + g.NKV * g.hd + kh * g.hd, false, f_hi, f_lo);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int qr = warp * kRowsPerWarp + r, tq = q0 + qr;
      if (tq >= g.T || k0 > tq) continue;  // warp-uniform
      const int key = k0 + lane;
      float dS = 0.f;
      if (key <= tq) {
        float sacc = 0.f, pacc = 0.f;
        for (int d = 0; d < g.hd; ++d) {
          sacc = fmaf(Qs[qr * pitch + d], Ks[lane * pitch + d], sacc);
          pacc = fmaf(dOs[qr * pitch + d], Vs[lane * pitch + d], pacc);
        }
        const float P = expf(sacc * g.scale - lse_r[r]);
        dS = P * (pacc - D_r[r]);
      }
      for (int k = 0; k < kTile; ++k) {
        const float dSk = __shfl_sync(0xffffffffu, dS, k);
#pragma unroll
        for (int j = 0; j < DPL; ++j) {
          const int d = lane + 32 * j;
          if (d < g.hd) dq[r][j] = fmaf(dSk, Ks[k * pitch + d], dq[r][j]);
        }
      }
    }
  }

  __syncthreads();
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int qr = warp * kRowsPerWarp + r;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const int d = lane + 32 * j;
      if (d < g.hd) Ks[qr * pitch + d] = dq[r][j] * g.scale;
    }
  }
  __syncthreads();
  store_grad_tile(dqkv, Ks, g, b, q0, h * g.hd, rope, f_hi, f_lo);
}

template <int DPL>
cudaError_t launch_simt(const SimtArgs& a, cudaStream_t stream) {
  const Geometry& g = a.g;
  const int pitch = g.hd + 1;
  const int n_tiles = (g.T + kTile - 1) / kTile;
  const size_t freq_bytes = 128 * sizeof(float);
  if (a.forward) {
    size_t smem = 3 * kTile * pitch * sizeof(float) + freq_bytes;
    cudaError_t e = cudaFuncSetAttribute(simt_fwd_kernel<DPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prof_begin(kKernelFwdSimt, stream);
    simt_fwd_kernel<DPL><<<dim3(n_tiles, g.NH, g.B), kThreads, smem, stream>>>(
        (float*)a.out, a.lse, (const float*)a.qkv, g);
    prof_end(kKernelFwdSimt, stream);
    return cudaGetLastError();
  }
  size_t smem_kv = 4 * kTile * pitch * sizeof(float) + 2 * kTile * sizeof(float) + freq_bytes;
  size_t smem_q = 4 * kTile * pitch * sizeof(float) + freq_bytes;
  cudaError_t e = cudaFuncSetAttribute(simt_bwd_dkdv_kernel<DPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_kv);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(simt_bwd_dq_kernel<DPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q);
  if (e != cudaSuccess) return e;
  prof_begin(kKernelBwdDkdvSimt, stream);
  simt_bwd_dkdv_kernel<DPL><<<dim3(n_tiles, g.NKV, g.B), kThreads, smem_kv, stream>>>(
      (float*)a.dqkv, (const float*)a.qkv, (const float*)a.dout, a.lse, a.Drow, g);
  prof_end(kKernelBwdDkdvSimt, stream);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_begin(kKernelBwdDqSimt, stream);
  simt_bwd_dq_kernel<DPL><<<dim3(n_tiles, g.NH, g.B), kThreads, smem_q, stream>>>(
      (float*)a.dqkv, (const float*)a.qkv, (const float*)a.dout, a.lse, a.Drow, g);
  prof_end(kKernelBwdDqSimt, stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t simt_launch(const SimtArgs& a, cudaStream_t stream) {
  if (simt_tiled_supported(a)) return simt_tiled_launch(a, stream);
  if (a.g.hd <= 32) return launch_simt<1>(a, stream);
  if (a.g.hd <= 64) return launch_simt<2>(a, stream);
  return launch_simt<4>(a, stream);
}

size_t simt_max_smem_bytes(int hd) {
  return 4 * kTile * (hd + 1) * sizeof(float) + 2 * kTile * sizeof(float) + 128 * sizeof(float);
}

}  // namespace attn
