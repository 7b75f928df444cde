// Backward prologue kernels (HBM-bound, CUDA cores).
//
// Row dots: D[b,h,t] = dO[b,t,h] . O[b,t,h].  This is the identity
// sum_s P_ts dP_ts = dO_t . O_t that "CUDA C microgpt"'s
// attention_backward_kernel accumulates as `weighted_sum`; computing it once
// per row up front lets the main backward form dS = P * (dP - D) tile by tile.
//
// Rotated Q/K copy (bf16 path with RoPE): the backward reads every Q and K
// tile many times, so it rotates them once into the caller's workspace
// instead of once per use.
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_profile.h"
#include "attn_ptx.cuh"

namespace attn {
namespace {

// One warp per (b, t) row of out/dout; lanes stride across the C columns in
// 16-byte vectors and reduce per head.
template <typename T>
__global__ void __launch_bounds__(256) row_dot_kernel(float* __restrict__ D, const T* __restrict__ out,
                                                      const T* __restrict__ dout, Geometry g) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
  const long long rows = (long long)g.B * g.T;
  if (warp >= rows) return;
  const int b = warp / g.T, t = warp % g.T;
  const T* o = out + (size_t)warp * g.C;
  const T* d = dout + (size_t)warp * g.C;
  for (int h = 0; h < g.NH; ++h) {
    float acc = 0.f;
    for (int c = lane; c < g.hd; c += 32) acc = fmaf(to_f32(o[h * g.hd + c]), to_f32(d[h * g.hd + c]), acc);
    acc = warp_sum(acc);
    if (lane == 0) D[((size_t)b * g.NH + h) * g.T + t] = acc;
  }
}

// bf16, hd a multiple of 8: lane handles 8 columns (one 16-byte vector) of a
// head; a warp covers 256 columns = 2 heads of 128 or 4 of 64 per step.
__global__ void __launch_bounds__(256) row_dot_bf16_vec_kernel(float* __restrict__ D, const uint4* __restrict__ out,
                                                                const uint4* __restrict__ dout, Geometry g) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
  const long long rows = (long long)g.B * g.T;
  if (warp >= rows) return;
  const int b = warp / g.T, t = warp % g.T;
  const int vec_per_row = g.C / 8, vec_per_head = g.hd / 8;
  const uint4* o = out + (size_t)warp * vec_per_row;
  const uint4* d = dout + (size_t)warp * vec_per_row;
  for (int v0 = 0; v0 < vec_per_row; v0 += 32) {
    const int v = v0 + lane;
    float acc = 0.f;
    if (v < vec_per_row) {
      uint4 a = o[v], c = d[v];
      acc = bf16_lo(a.x) * bf16_lo(c.x) + bf16_hi(a.x) * bf16_hi(c.x) + bf16_lo(a.y) * bf16_lo(c.y) +
            bf16_hi(a.y) * bf16_hi(c.y) + bf16_lo(a.z) * bf16_lo(c.z) + bf16_hi(a.z) * bf16_hi(c.z) +
            bf16_lo(a.w) * bf16_lo(c.w) + bf16_hi(a.w) * bf16_hi(c.w);
    }
    // reduce within groups of vec_per_head lanes (a power of two <= 32)
    for (int off = vec_per_head / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (v < vec_per_row && (v % vec_per_head) == 0) {
      const int h = v / vec_per_head;
      D[((size_t)b * g.NH + h) * g.T + t] = acc;
    }
  }
}

// Rotated Q/K copy.  One thread per unit (token row, chunk of up to 4 heads,
// group of 8 consecutive NEOX pairs): it forms the 8 angles of its pairs at
// its row once and applies them to each head of its chunk (heads 0..NH-1 are
// query heads, NH..NH+NKV-1 kv heads; K heads follow Q heads at column C in
// qkv, so head `head` sits at column head*hd in both arrays).  All loads of
// a unit are issued before the first is used (the kernel is HBM-bound); the
// units of one token row are adjacent threads.
// dst[b,t,head*hd + ...] = rotated qkv[b,t,head*hd + ...].
constexpr int kRopeHeadsPerThread = 4;
__global__ void __launch_bounds__(256, 3) rope_qk_bf16_kernel(__nv_bfloat16* __restrict__ dst,
                                                               const __nv_bfloat16* __restrict__ qkv, Geometry g,
                                                               int gph_log2, int n_units) {
  // The forward kernel that follows may get resident as blocks of this grid
  // retire (it waits for this grid before touching memory).
  ptx::grid_dep_launch();
  constexpr int HC = kRopeHeadsPerThread;
  const int half = g.hd >> 1;
  const int heads = g.NH + g.NKV;
  const int n_chunks = (heads + HC - 1) / HC;
  const int dst_w = heads * g.hd;
  for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += gridDim.x * blockDim.x) {
    const int gi = u & ((1 << gph_log2) - 1);
    const int rc = u >> gph_log2;
    const int row = rc / n_chunks, h0 = (rc - row * n_chunks) * HC;
    const int nh = min(HC, heads - h0);
    const int t = row % g.T;
    const __nv_bfloat16* src = qkv + (size_t)row * g.W + h0 * g.hd;
    uint4 x0[HC], x1[HC];
#pragma unroll
    for (int k = 0; k < HC; ++k)
      if (k < nh) load_rope_pairs(src + k * g.hd, gi, half, g.rope_interleaved != 0, x0[k], x1[k]);
    float cs[8], sn[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) __sincosf(rope_angle(t, g.rope_f_hi[gi * 8 + e], g.rope_f_lo[gi * 8 + e]), &sn[e], &cs[e]);
    __nv_bfloat16* out = dst + (size_t)row * dst_w + h0 * g.hd + gi * 8;
#pragma unroll
    for (int k = 0; k < HC; ++k) {
      if (k >= nh) break;
      const uint32_t a[4] = {x0[k].x, x0[k].y, x0[k].z, x0[k].w}, c[4] = {x1[k].x, x1[k].y, x1[k].z, x1[k].w};
      uint32_t ya[4], yc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float y00, y01, y10, y11;
        rope_pair(bf16_lo(a[q]), bf16_lo(c[q]), cs[2 * q], sn[2 * q], y00, y10);
        rope_pair(bf16_hi(a[q]), bf16_hi(c[q]), cs[2 * q + 1], sn[2 * q + 1], y01, y11);
        ya[q] = pack_bf16x2(y00, y01);
        yc[q] = pack_bf16x2(y10, y11);
      }
      *reinterpret_cast<uint4*>(out + k * g.hd) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
      *reinterpret_cast<uint4*>(out + k * g.hd + half) = make_uint4(yc[0], yc[1], yc[2], yc[3]);
    }
  }
}

// bf16 backward prologue, one launch.
//  * -D[b,h,t] with D = dO . O, into the second row table of (b, h): each
//    thread multiplies 16-byte chunks of out and dout, the hd/8 lanes of a
//    head (aligned: C/8 is a multiple of hd/8) sum their partials with
//    shuffles and one of them writes the table entry.  Rows of at least 256
//    chunks: block-stride over groups of four token rows, threads over the
//    chunks of the group's rows.  Narrower rows: the chunks of all B*T rows
//    flattened, four per thread and pass (a block per group of rows would
//    leave most of a block idle).  All loads of a pass are issued before the
//    first of them is used.
//  * (RoPE only) block-stride over groups of four token rows: threads
//    0..(NH+NKV)*hd/16-1 each rotate 8 NEOX pairs of one Q or K head of the
//    four rows into the workspace copy.
// The kernel is bound by HBM latency and bandwidth, not arithmetic.
// Afterwards the first row table, -lse[b,h,t] * log2(e), is written from lse
// along t, and the rows T..Tp-1 of both tables are cleared, so that whole
// 64-row tiles of the tables can be copied.  The two tables hold the per-row
// values the backward's elementwise steps use, already in the form they
// enter the exponent and the dS difference.  All index arithmetic is 32-bit
// with shifts: hd/8 and hd/16 are powers of two.
template <bool ROPE>
__global__ void __launch_bounds__(256, ROPE ? 3 : 4) bwd_prologue_bf16_kernel(float* __restrict__ LD, const uint4* __restrict__ out,
                                                                 const uint4* __restrict__ dout,
                                                                 const float* __restrict__ lse,
                                                                 __nv_bfloat16* __restrict__ rot,
                                                                 int* __restrict__ item_counter,
                                                                 float* __restrict__ rope_cs,
                                                                 const __nv_bfloat16* __restrict__ qkv, Geometry g,
                                                                 int vph_log2) {
  // out is written by the forward that may still be finishing (programmatic
  // launch): wait for it, then let the dK/dV kernel get resident.
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  if (blockIdx.x == 0 && threadIdx.x == 0) *item_counter = 0;
  constexpr int R = 4;                            // token rows per iteration
  const int vph = 1 << vph_log2;                  // 16-byte chunks per head (hd / 8)
  const int dot_units = g.C >> 3;                 // chunks per token row
  const int dot_threads = (dot_units + 31) & ~31;  // rounded to whole warps
  const int gph_log2 = vph_log2 - 1;              // 8-pair groups per head (hd / 16), log2
  const int heads = g.NH + g.NKV, half = g.hd >> 1;
  const int rope_units = ROPE ? heads << gph_log2 : 0;
  const int rows = g.B * g.T, Tp = row_table_rows(g.T);
  const int rot_w = heads * g.hd;
  const int n_groups = (rows + R - 1) / R;
  if (dot_units < (int)blockDim.x) {
    // Rows narrower than a block (C/8 < 256 chunks): flattened chunks.
    constexpr int U = 4;
    const long long n_units = (long long)rows * dot_units;
    const int lane = threadIdx.x & 31;
    for (long long base = ((long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31)) * U; base < n_units;
         base += (long long)gridDim.x * blockDim.x * U) {
      uint4 a[U], d[U];
#pragma unroll
      for (int i = 0; i < U; ++i) {
        const long long u = base + 32 * i + lane;
        a[i] = make_uint4(0u, 0u, 0u, 0u);
        d[i] = a[i];
        if (u < n_units) {
          a[i] = out[u];
          d[i] = dout[u];
        }
      }
      // Row (b, t) and chunk c of the thread's first unit of the pass from
      // one division; its other units, 32, 64 and 96 chunks on, by carrying.
      const long long u0 = base + lane;
      const int row0 = n_units < 0x7fff0000LL ? (int)u0 / dot_units : (int)(u0 / dot_units);
      int c = (int)(u0 - (long long)row0 * dot_units);
      int b = row0 / g.T, t = row0 - b * g.T;
#pragma unroll
      for (int i = 0; i < U; ++i) {
        float acc = bf16_lo(a[i].x) * bf16_lo(d[i].x) + bf16_hi(a[i].x) * bf16_hi(d[i].x) +
                    bf16_lo(a[i].y) * bf16_lo(d[i].y) + bf16_hi(a[i].y) * bf16_hi(d[i].y) +
                    bf16_lo(a[i].z) * bf16_lo(d[i].z) + bf16_hi(a[i].z) * bf16_hi(d[i].z) +
                    bf16_lo(a[i].w) * bf16_lo(d[i].w) + bf16_hi(a[i].w) * bf16_hi(d[i].w);
        for (int off = vph >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const long long u = base + 32 * i + lane;
        if (u < n_units && (lane & (vph - 1)) == 0)
          LD[(size_t)(2 * (b * g.NH + (c >> vph_log2)) + 1) * Tp + t] = -acc;
        for (c += 32; c >= dot_units; c -= dot_units) {
          if (++t == g.T) {
            t = 0;
            ++b;
          }
        }
      }
    }
  }
  const bool dot_by_group = dot_units >= (int)blockDim.x;
  for (int grp = blockIdx.x; grp < n_groups; grp += gridDim.x) {
    const int row0 = grp * R;
    const int nr = min(R, rows - row0);
    const int b0 = row0 / g.T, t0 = row0 - b0 * g.T;  // the group's first row; the others follow in t
    // Rows at least a block wide: the block's threads take the chunks of the
    // group's four rows (eight loads in flight per chunk column); whole
    // warps take part in the shuffles.
    for (int c = threadIdx.x; dot_by_group && c < dot_threads; c += blockDim.x) {
      uint4 a[R], d[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        a[r] = make_uint4(0u, 0u, 0u, 0u);
        d[r] = a[r];
        if (c < dot_units && r < nr) {
          a[r] = out[(size_t)(row0 + r) * dot_units + c];
          d[r] = dout[(size_t)(row0 + r) * dot_units + c];
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float acc = bf16_lo(a[r].x) * bf16_lo(d[r].x) + bf16_hi(a[r].x) * bf16_hi(d[r].x) +
                    bf16_lo(a[r].y) * bf16_lo(d[r].y) + bf16_hi(a[r].y) * bf16_hi(d[r].y) +
                    bf16_lo(a[r].z) * bf16_lo(d[r].z) + bf16_hi(a[r].z) * bf16_hi(d[r].z) +
                    bf16_lo(a[r].w) * bf16_lo(d[r].w) + bf16_hi(a[r].w) * bf16_hi(d[r].w);
        for (int off = vph >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (c < dot_units && r < nr && (c & (vph - 1)) == 0) {
          int t = t0 + r, b = b0;
          while (t >= g.T) {                          // the group runs into the next batch row
            t -= g.T;
            ++b;
          }
          LD[(size_t)(2 * (b * g.NH + (c >> vph_log2)) + 1) * Tp + t] = -acc;
        }
      }
    }
    for (int u = threadIdx.x; u < rope_units; u += blockDim.x) {
      const int head = u >> gph_log2, gi = u & ((1 << gph_log2) - 1);
      uint4 x0[R], x1[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (r < nr) {
          const __nv_bfloat16* src = qkv + (size_t)(row0 + r) * g.W + head * g.hd;  // K heads follow Q heads
          load_rope_pairs(src, gi, half, g.rope_interleaved != 0, x0[r], x1[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (r >= nr) break;
        const int row = row0 + r;
        const int t = row % g.T;
        const uint32_t a[4] = {x0[r].x, x0[r].y, x0[r].z, x0[r].w}, c[4] = {x1[r].x, x1[r].y, x1[r].z, x1[r].w};
        uint32_t ya[4], yc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float s0, c0, s1, c1, y00, y01, y10, y11;
          const int i0 = gi * 8 + 2 * q;
          __sincosf(rope_angle(t, g.rope_f_hi[i0], g.rope_f_lo[i0]), &s0, &c0);
          __sincosf(rope_angle(t, g.rope_f_hi[i0 + 1], g.rope_f_lo[i0 + 1]), &s1, &c1);
          rope_pair(bf16_lo(a[q]), bf16_lo(c[q]), c0, s0, y00, y10);
          rope_pair(bf16_hi(a[q]), bf16_hi(c[q]), c1, s1, y01, y11);
          ya[q] = pack_bf16x2(y00, y01);
          yc[q] = pack_bf16x2(y10, y11);
        }
        __nv_bfloat16* dst = rot + (size_t)row * rot_w + head * g.hd;
        *reinterpret_cast<uint4*>(dst + gi * 8) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
        *reinterpret_cast<uint4*>(dst + half + gi * 8) = make_uint4(yc[0], yc[1], yc[2], yc[3]);
      }
    }
  }
  // The -lse * log2(e) table of every (b, h), read and written along t
  // (coalesced on both sides), and the padding rows T..Tp-1 of both tables.
  const int n_tab = g.B * g.NH * Tp;
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < n_tab; k += gridDim.x * blockDim.x) {
    const int bh = k / Tp, t = k - bh * Tp;
    if (t < g.T) {
      LD[(size_t)(2 * bh) * Tp + t] = -lse[(size_t)bh * g.T + t] * 1.4426950408889634f;
    } else {
      LD[(size_t)(2 * bh) * Tp + t] = 0.f;
      LD[(size_t)(2 * bh + 1) * Tp + t] = 0.f;
    }
  }
  // The (cos, sin) of every RoPE angle, for the gradient epilogues: pair i,
  // position t at rope_cs[2 (i T + t)], so that the 32 consecutive rows of a
  // warp read one contiguous run per pair.
  if (rope_cs != nullptr) {
    const int half = g.hd >> 1, n_cs = g.T * half;
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < n_cs; k += gridDim.x * blockDim.x) {
      const int i = k / g.T, t = k - i * g.T;
      float sn, cs;
      __sincosf(rope_angle(t, g.rope_f_hi[i], g.rope_f_lo[i]), &sn, &cs);
      *reinterpret_cast<float2*>(rope_cs + 2 * (size_t)k) = make_float2(cs, sn);
    }
  }
}

}  // namespace

cudaError_t launch_bwd_prologue_bf16(float* LD, void* rot, int* item_counter, float* rope_cs, const void* out,
                                     const void* dout, const float* lse, const void* qkv, const Geometry& g,
                                     cudaStream_t stream) {
  const int vph = g.hd / 8;  // 8 or 16
  int vph_log2 = 0;
  while ((1 << vph_log2) < vph) ++vph_log2;
  const int groups = (g.B * g.T + 3) / 4;           // groups of four token rows
  const int per_sm = rot != nullptr ? 3 : 4;         // resident 256-thread blocks per SM
  const int blocks = groups < 152 * per_sm ? groups : 152 * per_sm;
  prof_begin(kKernelBwdPrologue, stream);
  cudaError_t e = rot != nullptr
                      ? launch_pdl(bwd_prologue_bf16_kernel<true>, dim3((unsigned)blocks), dim3(256), 0, stream, LD,
                                   (const uint4*)out, (const uint4*)dout, lse, (__nv_bfloat16*)rot, item_counter, rope_cs,
                                   (const __nv_bfloat16*)qkv, g, vph_log2)
                      : launch_pdl(bwd_prologue_bf16_kernel<false>, dim3((unsigned)blocks), dim3(256), 0, stream, LD,
                                   (const uint4*)out, (const uint4*)dout, lse, (__nv_bfloat16*)rot, item_counter, rope_cs,
                                   (const __nv_bfloat16*)qkv, g, vph_log2);
  prof_end(kKernelBwdPrologue, stream);
  return e;
}

cudaError_t launch_row_dot(float* D, const void* out, const void* dout, const Geometry& g, bool bf16,
                           cudaStream_t stream) {
  const long long rows = (long long)g.B * g.T;
  const int blocks = (int)((rows + 7) / 8);
  prof_begin(kKernelBwdRowDot, stream);
  if (bf16 && g.hd % 8 == 0 && (g.hd / 8) <= 32 && ((g.hd / 8) & (g.hd / 8 - 1)) == 0) {
    row_dot_bf16_vec_kernel<<<blocks, 256, 0, stream>>>(D, (const uint4*)out, (const uint4*)dout, g);
  } else if (bf16) {
    row_dot_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(D, (const __nv_bfloat16*)out,
                                                               (const __nv_bfloat16*)dout, g);
  } else {
    row_dot_kernel<float><<<blocks, 256, 0, stream>>>(D, (const float*)out, (const float*)dout, g);
  }
  prof_end(kKernelBwdRowDot, stream);
  return cudaGetLastError();
}

cudaError_t launch_rope_qk_bf16(void* dst, const void* qkv, const Geometry& g, cudaStream_t stream) {
  int gph_log2 = 0;                                   // log2(hd / 16)
  while ((16 << gph_log2) < g.hd) ++gph_log2;
  const int heads = g.NH + g.NKV;
  const long long units = (long long)g.B * g.T * ((heads + kRopeHeadsPerThread - 1) / kRopeHeadsPerThread)
                          << gph_log2;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  const long long need = (units + 255) / 256;
  // One unit per thread: blocks retire and refill the SMs while others wait
  // on their loads (measured faster than 3 resident blocks per SM walking the
  // units).
  const int blocks = (int)need;
  prof_begin(kKernelRopeQK, stream);
  rope_qk_bf16_kernel<<<blocks, 256, 0, stream>>>((__nv_bfloat16*)dst, (const __nv_bfloat16*)qkv, g, gph_log2,
                                                  (int)units);
  prof_end(kKernelRopeQK, stream);
  return cudaGetLastError();
}

}  // namespace attn
