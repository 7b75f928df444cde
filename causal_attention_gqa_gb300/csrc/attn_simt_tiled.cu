// Exact float32 causal MHA/GQA attention on CUDA cores, register-tiled, for
// head size 64 (dtype F32 / TF32).
//
// Same arithmetic contract as the row-per-warp kernels of the float32 path:
// every product and sum is an IEEE float32 FMA (no tensor-core rounding), the
// softmax is kept online, and the backward folds the softmax Jacobian into
// dS = P * (dP - D) with D = rowsum(dO * O) (the gradient of "nanoeuler --
// CUDA kernels", attention_backward_kernel; "CUDA C microgpt",
// attention_backward_kernel's weighted_sum).  What changes is the blocking:
// a CTA of 256 threads works on a 64 x 64 tile of scores, each thread on a
// 4 x 4 block of it, so that every pair of 16-byte shared-memory loads feeds
// 16 FMAs (the row-per-warp kernels issue about one load per FMA and are
// bound by shared-memory bandwidth).
//
// Thread (ty, tx), ty, tx in 0..15, owns score rows ty + 16 i and columns
// tx + 16 j (i, j < 4).  Tiles are row-major in shared memory with a pitch of
// 68 floats: rows tx, tx+1, ... of one 16-byte column then fall into distinct
// banks, so the loads of a quarter-warp are conflict-free without
// transposing anything.  The 16 threads of one ty are one half-warp, so row
// maxima and sums are shuffles over 16 lanes.
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_profile.h"

#include <math.h>

namespace attn {
namespace {

constexpr int kB = 64;             // queries per tile and keys per tile
constexpr int kP = 68;             // shared-memory row pitch (floats)
constexpr int kThreadsT = 256;
constexpr int kHD = 64;            // head size of these kernels
constexpr int kTileFloats = kB * kP;

// 16-lane (half-warp) reductions.
__device__ __forceinline__ float half_max(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Stage rows t0 .. t0+63 of one head (qkv or dout columns col0 .. col0+63,
// row width `width`) into dst (pitch kP), zero past T, NEOX-rotated if rope.
// Consecutive threads take consecutive 16-byte pieces of a row.
__device__ void stage_rows(float* dst, const float* src, int width, const Geometry& g, int b, int t0, int col0,
                           bool rope, const float* f_hi, const float* f_lo) {
  if (!rope) {
    for (int u = threadIdx.x; u < kB * (kHD / 4); u += kThreadsT) {
      const int r = u / (kHD / 4), c = u % (kHD / 4), t = t0 + r;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < g.T) v = *reinterpret_cast<const float4*>(src + ((size_t)b * g.T + t) * width + col0 + 4 * c);
      *reinterpret_cast<float4*>(dst + r * kP + 4 * c) = v;
    }
    return;
  }
  constexpr int half = kHD / 2;
  for (int u = threadIdx.x; u < kB * (half / 4); u += kThreadsT) {
    const int r = u / (half / 4), c = u % (half / 4), t = t0 + r;
    float y0[4] = {0.f, 0.f, 0.f, 0.f}, y1[4] = {0.f, 0.f, 0.f, 0.f};
    if (t < g.T) {
      const float* row = src + ((size_t)b * g.T + t) * width + col0;
      float4 a, e;
      if (!g.rope_interleaved) {
        a = *reinterpret_cast<const float4*>(row + 4 * c);
        e = *reinterpret_cast<const float4*>(row + half + 4 * c);
      } else {            // pairs (2i, 2i+1), i = 4c .. 4c+3: elements 8c .. 8c+7
        const float4 u = *reinterpret_cast<const float4*>(row + 8 * c);
        const float4 w = *reinterpret_cast<const float4*>(row + 8 * c + 4);
        a = make_float4(u.x, u.z, w.x, w.z);
        e = make_float4(u.y, u.w, w.y, w.w);
      }
      const float x0[4] = {a.x, a.y, a.z, a.w}, x1[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float s, co;
        sincosf(rope_angle(t, f_hi[4 * c + k], f_lo[4 * c + k]), &s, &co);
        rope_pair(x0[k], x1[k], co, s, y0[k], y1[k]);
      }
    }
    *reinterpret_cast<float4*>(dst + r * kP + 4 * c) = make_float4(y0[0], y0[1], y0[2], y0[3]);
    *reinterpret_cast<float4*>(dst + r * kP + half + 4 * c) = make_float4(y1[0], y1[1], y1[2], y1[3]);
  }
}

// acc[i][j] (+)= sum_d A[ty + 16 i][d] * B[tx + 16 j][d] over d < kHD (both
// tiles row-major with pitch kP).
__device__ __forceinline__ void tile_abt(float (&acc)[4][4], const float* A, const float* B, int ty, int tx) {
#pragma unroll 4
  for (int d = 0; d < kHD; d += 4) {
    float4 a[4], bb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(A + (ty + 16 * i) * kP + d);
#pragma unroll
    for (int j = 0; j < 4; ++j) bb[j] = *reinterpret_cast<const float4*>(B + (tx + 16 * j) * kP + d);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[i][j] = fmaf(a[i].x, bb[j].x, acc[i][j]);
        acc[i][j] = fmaf(a[i].y, bb[j].y, acc[i][j]);
        acc[i][j] = fmaf(a[i].z, bb[j].z, acc[i][j]);
        acc[i][j] = fmaf(a[i].w, bb[j].w, acc[i][j]);
      }
  }
}

// out[i][c] += sum_k W[k][4 ty' + i] * X[k][4 tx + c] over the 64 rows k of a
// tile: W is a 64 x 64 block stored as W[k * kP + 4 * ty + i] (the four rows
// a thread owns contiguous), X row-major with pitch kP.
__device__ __forceinline__ void tile_wtx(float (&out)[4][4], const float* W, const float* X, int ty, int tx) {
#pragma unroll 4
  for (int k = 0; k < kB; ++k) {
    const float4 w = *reinterpret_cast<const float4*>(W + k * kP + 4 * ty);
    const float4 x = *reinterpret_cast<const float4*>(X + k * kP + 4 * tx);
    const float wv[4] = {w.x, w.y, w.z, w.w}, xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) out[i][c] = fmaf(wv[i], xv[c], out[i][c]);
  }
}

// ---------------------------------------------------------------------------
// Forward: one CTA per (64-query tile, query head, batch row), heaviest tiles
// first; key tiles 0 .. qt.  O[q][d] for d = 4 tx .. 4 tx + 3 and q = ty + 16 i.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreadsT, 2)
simt64_fwd_kernel(float* __restrict__ out, float* __restrict__ lse, const float* __restrict__ qkv, Geometry g) {
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  float* Qs = smem;
  float* Ks = Qs + kTileFloats;
  float* Vs = Ks + kTileFloats;
  float* Ps = Vs + kTileFloats;          // Ps[k * kP + 4 ty + i] = P[ty + 16 i][k]
  float* f_hi = Ps + kTileFloats;
  float* f_lo = f_hi + 64;
  const int n_qt = (g.T + kB - 1) / kB;
  const int qt = n_qt - 1 - (int)blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int kh = h / g.grp, q0 = qt * kB;
  const bool rope = g.rope_theta > 0.f;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  for (int i = threadIdx.x; i < 64; i += kThreadsT) {
    f_hi[i] = g.rope_f_hi[i];
    f_lo[i] = g.rope_f_lo[i];
  }
  __syncthreads();
  stage_rows(Qs, qkv, g.W, g, b, q0, h * kHD, rope, f_hi, f_lo);

  float m[4], l[4], o[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) o[i][c] = 0.f;
  }
  for (int kt = 0; kt <= qt; ++kt) {
    const int k0 = kt * kB;
    __syncthreads();   // the previous tile's K, V and P are consumed
    stage_rows(Ks, qkv, g.W, g, b, k0, g.C + kh * kHD, rope, f_hi, f_lo);
    stage_rows(Vs, qkv, g.W, g, b, k0, g.C + g.NKV * kHD + kh * kHD, false, f_hi, f_lo);
    __syncthreads();
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
    tile_abt(s, Qs, Ks, ty, tx);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tq = q0 + ty + 16 * i;
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = k0 + tx + 16 * j;
        s[i][j] = (key <= tq) ? s[i][j] * g.scale : -INFINITY;
        mx = fmaxf(mx, s[i][j]);
      }
      // Key k0 <= tq for every row this tile reaches except rows past T
      // (tq >= k0 always holds here), so m_new is finite.
      const float m_new = fmaxf(m[i], half_max(mx));
      const float corr = expf(m[i] - m_new);       // 0 on the first tile (m = -inf)
      float ps = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float p = (s[i][j] == -INFINITY) ? 0.f : expf(s[i][j] - m_new);
        s[i][j] = p;
        ps += p;
      }
      l[i] = l[i] * corr + ps;                      // this thread's partial row sum
      m[i] = m_new;
#pragma unroll
      for (int c = 0; c < 4; ++c) o[i][c] *= corr;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<float4*>(Ps + (tx + 16 * j) * kP + 4 * ty) = make_float4(s[0][j], s[1][j], s[2][j], s[3][j]);
    __syncthreads();
    tile_wtx(o, Ps, Vs, ty, tx);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lt = half_sum(l[i]);
    const int tq = q0 + ty + 16 * i;
    if (tq < g.T) {
      const float inv = 1.f / lt;
      *reinterpret_cast<float4*>(out + ((size_t)b * g.T + tq) * g.C + h * kHD + 4 * tx) =
          make_float4(o[i][0] * inv, o[i][1] * inv, o[i][2] * inv, o[i][3] * inv);
      if (tx == 0) lse[((size_t)b * g.NH + h) * g.T + tq] = m[i] + logf(lt);
    }
  }
}

// Write rows t0 .. t0+63 (< T) of a float32 gradient tile (pitch kP) to
// dqkv columns col0 .. col0+63, undoing the NEOX rotation at each row's
// position when rope is set (the gradient with respect to the unrotated
// input is R^T times the gradient with respect to the rotated one).
__device__ void store_rows(float* dqkv, const float* tile, const Geometry& g, int b, int t0, int col0, bool rope,
                           const float* f_hi, const float* f_lo) {
  if (!rope) {
    for (int u = threadIdx.x; u < kB * (kHD / 4); u += kThreadsT) {
      const int r = u / (kHD / 4), c = u % (kHD / 4), t = t0 + r;
      if (t < g.T)
        *reinterpret_cast<float4*>(dqkv + ((size_t)b * g.T + t) * g.W + col0 + 4 * c) =
            *reinterpret_cast<const float4*>(tile + r * kP + 4 * c);
    }
    return;
  }
  constexpr int half = kHD / 2;
  for (int u = threadIdx.x; u < kB * (half / 4); u += kThreadsT) {
    const int r = u / (half / 4), c = u % (half / 4), t = t0 + r;
    if (t >= g.T) continue;
    const float4 a = *reinterpret_cast<const float4*>(tile + r * kP + 4 * c);
    const float4 e = *reinterpret_cast<const float4*>(tile + r * kP + half + 4 * c);
    const float g0[4] = {a.x, a.y, a.z, a.w}, g1[4] = {e.x, e.y, e.z, e.w};
    float y0[4], y1[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float sn, co;
      sincosf(rope_angle(t, f_hi[4 * c + k], f_lo[4 * c + k]), &sn, &co);
      rope_pair_transpose(g0[k], g1[k], co, sn, y0[k], y1[k]);
    }
    float* row = dqkv + ((size_t)b * g.T + t) * g.W + col0;
    if (!g.rope_interleaved) {
      *reinterpret_cast<float4*>(row + 4 * c) = make_float4(y0[0], y0[1], y0[2], y0[3]);
      *reinterpret_cast<float4*>(row + half + 4 * c) = make_float4(y1[0], y1[1], y1[2], y1[3]);
    } else {
      *reinterpret_cast<float4*>(row + 8 * c) = make_float4(y0[0], y1[0], y0[1], y1[1]);
      *reinterpret_cast<float4*>(row + 8 * c + 4) = make_float4(y0[2], y1[2], y0[3], y1[3]);
    }
  }
}

// Put a thread's 4 x 4 accumulator block (rows ty + 16 i, columns
// 4 tx .. 4 tx + 3), times `scale`, into a row-major tile.
__device__ __forceinline__ void put_block(float* tile, const float (&acc)[4][4], float scale, int ty, int tx) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(tile + (ty + 16 * i) * kP + 4 * tx) =
        make_float4(acc[i][0] * scale, acc[i][1] * scale, acc[i][2] * scale, acc[i][3] * scale);
}

// ---------------------------------------------------------------------------
// Backward, key-stationary: one CTA per (64-key tile, kv head, batch row),
// heaviest first.  Walks the group's query heads and the query tiles at or
// after the key tile; per query tile, with k = key row ty + 16 i and q =
// query column tx + 16 j:
//   S^T = scale K Q^T,  P^T = exp(S^T - lse_q) (0 where q < k or q >= T),
//   dP^T = V dO^T,      dS^T = P^T (dP^T - D_q),
//   dV += P^T dO,       dK += dS^T Q      (dK scaled once at the end).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreadsT, 2)
simt64_bwd_dkdv_kernel(float* __restrict__ dqkv, const float* __restrict__ qkv, const float* __restrict__ dout,
                       const float* __restrict__ lse, const float* __restrict__ Drow, Geometry g) {
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  float* Ks = smem;
  float* Vs = Ks + kTileFloats;
  float* Qs = Vs + kTileFloats;
  float* dOs = Qs + kTileFloats;
  float* Ps = dOs + kTileFloats;      // Ps[q * kP + 4 ty + i] = P^T[ty + 16 i][q]
  float* dSs = Ps + kTileFloats;      // same layout for dS^T
  float* Ls = dSs + kTileFloats;      // lse of the query tile
  float* Ds = Ls + kB;                // D of the query tile
  float* f_hi = Ds + kB;
  float* f_lo = f_hi + 64;
  const int n_qt = (g.T + kB - 1) / kB;
  const int kt = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int k0 = kt * kB;
  const bool rope = g.rope_theta > 0.f;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  for (int i = threadIdx.x; i < 64; i += kThreadsT) {
    f_hi[i] = g.rope_f_hi[i];
    f_lo[i] = g.rope_f_lo[i];
  }
  __syncthreads();
  stage_rows(Ks, qkv, g.W, g, b, k0, g.C + kh * kHD, rope, f_hi, f_lo);
  stage_rows(Vs, qkv, g.W, g, b, k0, g.C + g.NKV * kHD + kh * kHD, false, f_hi, f_lo);

  float dk[4][4], dv[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) dk[i][c] = dv[i][c] = 0.f;

  for (int hh = 0; hh < g.grp; ++hh) {
    const int h = kh * g.grp + hh;
    const size_t row_base = ((size_t)b * g.NH + h) * g.T;
    for (int qt = kt; qt < n_qt; ++qt) {
      const int q0 = qt * kB;
      __syncthreads();   // the previous step's Q, dO, P^T, dS^T are consumed
      stage_rows(Qs, qkv, g.W, g, b, q0, h * kHD, rope, f_hi, f_lo);
      stage_rows(dOs, dout, g.C, g, b, q0, h * kHD, false, f_hi, f_lo);
      for (int r = threadIdx.x; r < kB; r += kThreadsT) {
        const int t = q0 + r;
        Ls[r] = (t < g.T) ? lse[row_base + t] : 0.f;
        Ds[r] = (t < g.T) ? Drow[row_base + t] : 0.f;
      }
      __syncthreads();
      float st[4][4], dpt[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) st[i][j] = dpt[i][j] = 0.f;
      tile_abt(st, Ks, Qs, ty, tx);
      tile_abt(dpt, Vs, dOs, ty, tx);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int q = tx + 16 * j, tq = q0 + q;
        const float lq = Ls[q], dq = Ds[q];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tk = k0 + ty + 16 * i;
          const float p = (tq >= tk && tq < g.T) ? expf(st[i][j] * g.scale - lq) : 0.f;
          st[i][j] = p;
          dpt[i][j] = p * (dpt[i][j] - dq);
        }
        *reinterpret_cast<float4*>(Ps + q * kP + 4 * ty) = make_float4(st[0][j], st[1][j], st[2][j], st[3][j]);
        *reinterpret_cast<float4*>(dSs + q * kP + 4 * ty) =
            make_float4(dpt[0][j], dpt[1][j], dpt[2][j], dpt[3][j]);
      }
      __syncthreads();
      tile_wtx(dv, Ps, dOs, ty, tx);
      tile_wtx(dk, dSs, Qs, ty, tx);
    }
  }
  __syncthreads();
  put_block(Qs, dk, g.scale, ty, tx);
  put_block(dOs, dv, 1.f, ty, tx);
  __syncthreads();
  store_rows(dqkv, Qs, g, b, k0, g.C + kh * kHD, rope, f_hi, f_lo);
  store_rows(dqkv, dOs, g, b, k0, g.C + g.NKV * kHD + kh * kHD, false, f_hi, f_lo);
}

// ---------------------------------------------------------------------------
// Backward, query-stationary: one CTA per (64-query tile, query head, batch
// row), heaviest first; key tiles 0 .. qt.  With q = query row ty + 16 i and
// k = key column tx + 16 j:
//   P = exp(scale Q K^T - lse_q) (0 where k > q),  dP = dO V^T,
//   dS = P (dP - D_q),  dQ += dS K                  (scaled once at the end).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreadsT, 2)
simt64_bwd_dq_kernel(float* __restrict__ dqkv, const float* __restrict__ qkv, const float* __restrict__ dout,
                     const float* __restrict__ lse, const float* __restrict__ Drow, Geometry g) {
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  float* Qs = smem;
  float* dOs = Qs + kTileFloats;
  float* Ks = dOs + kTileFloats;
  float* Vs = Ks + kTileFloats;
  float* dSs = Vs + kTileFloats;      // dSs[k * kP + 4 ty + i] = dS[ty + 16 i][k]
  float* f_hi = dSs + kTileFloats;
  float* f_lo = f_hi + 64;
  const int n_qt = (g.T + kB - 1) / kB;
  const int qt = n_qt - 1 - (int)blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int kh = h / g.grp, q0 = qt * kB;
  const bool rope = g.rope_theta > 0.f;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  for (int i = threadIdx.x; i < 64; i += kThreadsT) {
    f_hi[i] = g.rope_f_hi[i];
    f_lo[i] = g.rope_f_lo[i];
  }
  __syncthreads();
  stage_rows(Qs, qkv, g.W, g, b, q0, h * kHD, rope, f_hi, f_lo);
  stage_rows(dOs, dout, g.C, g, b, q0, h * kHD, false, f_hi, f_lo);
  const size_t row_base = ((size_t)b * g.NH + h) * g.T;
  float lq[4], dq_row[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int tq = q0 + ty + 16 * i;
    lq[i] = (tq < g.T) ? lse[row_base + tq] : 0.f;
    dq_row[i] = (tq < g.T) ? Drow[row_base + tq] : 0.f;
  }
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
  for (int kt = 0; kt <= qt; ++kt) {
    const int k0 = kt * kB;
    __syncthreads();   // the previous tile's K, V, dS are consumed
    stage_rows(Ks, qkv, g.W, g, b, k0, g.C + kh * kHD, rope, f_hi, f_lo);
    stage_rows(Vs, qkv, g.W, g, b, k0, g.C + g.NKV * kHD + kh * kHD, false, f_hi, f_lo);
    __syncthreads();
    float sc[4][4], dp[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[i][j] = dp[i][j] = 0.f;
    tile_abt(sc, Qs, Ks, ty, tx);
    tile_abt(dp, dOs, Vs, ty, tx);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int tk = k0 + tx + 16 * j;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int tq = q0 + ty + 16 * i;
        const float p = (tk <= tq && tq < g.T) ? expf(sc[i][j] * g.scale - lq[i]) : 0.f;
        dp[i][j] = p * (dp[i][j] - dq_row[i]);
      }
      *reinterpret_cast<float4*>(dSs + (tx + 16 * j) * kP + 4 * ty) =
          make_float4(dp[0][j], dp[1][j], dp[2][j], dp[3][j]);
    }
    __syncthreads();
    tile_wtx(acc, dSs, Ks, ty, tx);
  }
  __syncthreads();
  put_block(Ks, acc, g.scale, ty, tx);
  __syncthreads();
  store_rows(dqkv, Ks, g, b, q0, h * kHD, rope, f_hi, f_lo);
}

}  // namespace

// Head size 64, and every tensor 16-byte aligned (the tiles move as float4;
// the float32 entry points otherwise only require 4-byte alignment).
bool simt_tiled_supported(const SimtArgs& a) {
  const uintptr_t bits = reinterpret_cast<uintptr_t>(a.qkv) | reinterpret_cast<uintptr_t>(a.out) |
                         reinterpret_cast<uintptr_t>(a.dqkv) | reinterpret_cast<uintptr_t>(a.dout);
  return a.g.hd == kHD && (bits & 15u) == 0;
}

size_t simt_tiled_smem_bytes() { return (size_t)(4 * kTileFloats + 128) * sizeof(float); }
size_t simt_tiled_dkdv_smem_bytes() { return (size_t)(6 * kTileFloats + 2 * kB + 128) * sizeof(float); }
size_t simt_tiled_dq_smem_bytes() { return (size_t)(5 * kTileFloats + 128) * sizeof(float); }

cudaError_t simt_tiled_launch(const SimtArgs& a, cudaStream_t stream) {
  const Geometry& g = a.g;
  const int n_qt = (g.T + kB - 1) / kB;
  if (a.forward) {
    const size_t smem = simt_tiled_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(simt64_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prof_begin(kKernelFwdSimt, stream);
    simt64_fwd_kernel<<<dim3(n_qt, g.NH, g.B), kThreadsT, smem, stream>>>((float*)a.out, a.lse,
                                                                          (const float*)a.qkv, g);
    prof_end(kKernelFwdSimt, stream);
    return cudaGetLastError();
  }
  const int n_kt = n_qt;
  const size_t smem_kv = simt_tiled_dkdv_smem_bytes(), smem_q = simt_tiled_dq_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(simt64_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_kv);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(simt64_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q);
  if (e != cudaSuccess) return e;
  prof_begin(kKernelBwdDkdvSimt, stream);
  simt64_bwd_dkdv_kernel<<<dim3(n_kt, g.NKV, g.B), kThreadsT, smem_kv, stream>>>(
      (float*)a.dqkv, (const float*)a.qkv, (const float*)a.dout, a.lse, a.Drow, g);
  prof_end(kKernelBwdDkdvSimt, stream);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_begin(kKernelBwdDqSimt, stream);
  simt64_bwd_dq_kernel<<<dim3(n_qt, g.NH, g.B), kThreadsT, smem_q, stream>>>(
      (float*)a.dqkv, (const float*)a.qkv, (const float*)a.dout, a.lse, a.Drow, g);
  prof_end(kKernelBwdDqSimt, stream);
  return cudaGetLastError();
}

}  // namespace attn
