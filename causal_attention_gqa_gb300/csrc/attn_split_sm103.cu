// Causal MHA/GQA attention on sm_103a tensor cores for float32 tensors
// (dtype TF32), head size 64: every product of two float32 operands is taken
// as three bf16 products.
//
// Each float32 operand x is split into bf16 parts hi = bf16(x) and
// lo = bf16(x - hi) (x = hi + lo to about 2^-17 relative), and a product is
// formed as hi*hi + hi*lo + lo*hi in float32 tensor-core accumulation (the
// lo*lo term, ~2^-16 relative, is dropped): the split of Ootomo & Yokota
// (2022), "Recovering single precision accuracy from Tensor Cores while
// surpassing the FP32 theoretical peak performance", with bf16 parts instead
// of tf32 ones, so that the bf16 tcgen05 MMAs run at their full rate.  The
// softmax weights P and the gradient weights dS are split the same way before
// their second-stage products; exponentials, the online softmax and the row
// statistics stay in float32.  On float32 inputs of the GPT-2-shaped workload
// this reaches ~1e-5 of the float64 result, inside the 1e-4 bar of the float32
// dtypes.
//
// The method is that of "nanoeuler -- CUDA kernels" (attention_forward_kernel
// and attention_backward_kernel: scale 1/sqrt(hd), kv head h/(NH/NKV), causal
// softmax, P V; dP = dO V^T, dS = P * (dP - D), dQ = scale dS K,
// dK = scale dS^T Q, dV = P^T dO, dK/dV summed over the group, RoPE undone on
// dQ/dK).  Kernels:
//   split_rope_kernel / split_plain_kernel: hi/lo parts of (rotated) Q, K, V
//     and of dO into the workspace, in the column layout of qkv / dout;
//   split_tables_kernel: the backward's row tables -lse log2(e) and -D with
//     D = dO . O, over T rounded up to 128 rows;
//   split_fwd_kernel: one CTA per (128-query tile, head, batch row);
//   split_bwd_dkdv_kernel: one CTA per (128-key tile, kv head, batch row),
//     walking the group's query heads and query tiles;
//   split_bwd_dq_kernel: one CTA per (128-query tile, head, batch row).
// Each step runs its MMAs and its elementwise work one after the other (no
// cross-step overlap): the float32 path is held to its accuracy bar first.
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, the
// others elementwise with one TMEM lane (row) per thread.  Every wait is
// bounded.
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_profile.h"
#include "attn_ptx.cuh"

namespace attn {
namespace {

constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kHD = 64;
constexpr int kTile = 128 * kHD * 2;       // one bf16 [128 x 64] tile: one 128-byte swizzle atom column
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// hi = bf16(x), lo = bf16(x - hi), two values at a time (packed bf16 pairs).
__device__ __forceinline__ void split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_bf16x2(x - hf.x, y - hf.y);
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// TMEM column, inside a 128-column block, of the bf16 pairs of elements
// 16 kk .. 16 kk + 15 of a split row whose owner group w = kk / 4 writes its
// 64 elements as 32 hi columns at 64 w and 32 lo columns at 64 w + 32.
__device__ __forceinline__ uint32_t hi_col(int kk) { return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8); }

// 64 float32 columns of this thread's TMEM lane.  Warp-collective.
__device__ __forceinline__ void load64(uint32_t t, float (&v)[64]) {
  uint32_t a[32], b[32];
  ptx::tmem_ld32(t, a);
  ptx::tmem_ld32(t + 32, b);
  ptx::tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    v[c] = __uint_as_float(a[c]);
    v[32 + c] = __uint_as_float(b[c]);
  }
}

// Split 64 float32 values of this thread's row into hi/lo pairs and store
// them at `t` (32 hi columns) and `t + 32` (32 lo columns).  Warp-collective.
__device__ __forceinline__ void store_split64(uint32_t t, const float (&v)[64]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) split2(v[32 * h + 2 * c], v[32 * h + 2 * c + 1], hi[c], lo[c]);
    ptx::tmem_st16(t + 16 * h, hi);
    ptx::tmem_st16(t + 32 + 16 * h, lo);
  }
}

// ===========================================================================
// Split passes
// ===========================================================================
// Columns [col0, col0 + ncols) of a float32 [rows, src_w] array into bf16
// hi/lo arrays [rows, dst_w] at the same columns; 8 columns per thread.
__global__ void split_plain_kernel(const float* __restrict__ src, int src_w, int col0, int ncols,
                                   __nv_bfloat16* __restrict__ hi, __nv_bfloat16* __restrict__ lo, int dst_w,
                                   long long rows) {
  const int per_row = ncols / 8;
  const long long n = rows * per_row;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < n;
       u += (long long)gridDim.x * blockDim.x) {
    const long long r = u / per_row;
    const int c = col0 + (int)(u % per_row) * 8;
    const float4 a = *reinterpret_cast<const float4*>(src + r * src_w + c);
    const float4 b = *reinterpret_cast<const float4*>(src + r * src_w + c + 4);
    uint4 h, l;
    split2(a.x, a.y, h.x, l.x);
    split2(a.z, a.w, h.y, l.y);
    split2(b.x, b.y, h.z, l.z);
    split2(b.z, b.w, h.w, l.w);
    *reinterpret_cast<uint4*>(hi + r * dst_w + c) = h;
    *reinterpret_cast<uint4*>(lo + r * dst_w + c) = l;
  }
}

// The Q and K heads of a float32 qkv rotated at their positions and split:
// pair i of a head turns by t * theta^(-2i/hd) (NEOX pairs (i, i + hd/2); an
// interleaved (2i, 2i+1) row is read even-first so that pair i lands in slots
// i and i + hd/2, as in the bf16 kernels).  One thread per (row, head, group
// of eight pairs).
__global__ void split_rope_kernel(const float* __restrict__ qkv, __nv_bfloat16* __restrict__ hi,
                                  __nv_bfloat16* __restrict__ lo, Geometry g) {
  const int half = g.hd / 2, groups = half / 8, heads = g.NH + g.NKV;
  const long long n = (long long)g.B * g.T * heads * groups;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < n;
       u += (long long)gridDim.x * blockDim.x) {
    const int gi = (int)(u % groups);
    const long long rh = u / groups;
    const int head = (int)(rh % heads);
    const long long row = rh / heads;
    const int t = (int)(row % g.T);
    const float* x = qkv + row * g.W + head * g.hd;
    float x0[8], x1[8];
    if (!g.rope_interleaved) {
      const float4 a = *reinterpret_cast<const float4*>(x + 8 * gi);
      const float4 b = *reinterpret_cast<const float4*>(x + 8 * gi + 4);
      const float4 c = *reinterpret_cast<const float4*>(x + half + 8 * gi);
      const float4 d = *reinterpret_cast<const float4*>(x + half + 8 * gi + 4);
      const float xa[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w}, xc[8] = {c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        x0[k] = xa[k];
        x1[k] = xc[k];
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 a = *reinterpret_cast<const float4*>(x + 16 * gi + 4 * q);
        x0[2 * q] = a.x;
        x1[2 * q] = a.y;
        x0[2 * q + 1] = a.z;
        x1[2 * q + 1] = a.w;
      }
    }
    float y0[8], y1[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = 8 * gi + k;
      float sn, cs;
      __sincosf(rope_angle(t, g.rope_f_hi[i], g.rope_f_lo[i]), &sn, &cs);
      rope_pair(x0[k], x1[k], cs, sn, y0[k], y1[k]);
    }
    uint4 h0, l0, h1, l1;
    split2(y0[0], y0[1], h0.x, l0.x);
    split2(y0[2], y0[3], h0.y, l0.y);
    split2(y0[4], y0[5], h0.z, l0.z);
    split2(y0[6], y0[7], h0.w, l0.w);
    split2(y1[0], y1[1], h1.x, l1.x);
    split2(y1[2], y1[3], h1.y, l1.y);
    split2(y1[4], y1[5], h1.z, l1.z);
    split2(y1[6], y1[7], h1.w, l1.w);
    const size_t o = (size_t)row * g.W + head * g.hd;
    *reinterpret_cast<uint4*>(hi + o + 8 * gi) = h0;
    *reinterpret_cast<uint4*>(lo + o + 8 * gi) = l0;
    *reinterpret_cast<uint4*>(hi + o + half + 8 * gi) = h1;
    *reinterpret_cast<uint4*>(lo + o + half + 8 * gi) = l1;
  }
}

// Row tables of the backward, Tp = T rounded up to 128 per (b, h):
// LD[2 bh Tp + t] = -lse log2(e), LD[(2 bh + 1) Tp + t] = -D with
// D = sum_d dO[b,t,h,d] O[b,t,h,d] (float32); zeros for t >= T.
__global__ void split_tables_kernel(float* __restrict__ LD, const float* __restrict__ out,
                                    const float* __restrict__ dout, const float* __restrict__ lse, Geometry g,
                                    int Tp) {
  const long long n = (long long)g.B * g.NH * Tp;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < n;
       u += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(u % Tp);
    const long long bh = u / Tp;
    const int h = (int)(bh % g.NH), b = (int)(bh / g.NH);
    float nl = 0.f, nd = 0.f;
    if (t < g.T) {
      const float* o = out + ((size_t)b * g.T + t) * g.C + h * g.hd;
      const float* d = dout + ((size_t)b * g.T + t) * g.C + h * g.hd;
      float acc = 0.f;
      for (int k = 0; k < g.hd; k += 4) {
        const float4 a = *reinterpret_cast<const float4*>(o + k);
        const float4 c = *reinterpret_cast<const float4*>(d + k);
        acc = fmaf(a.x, c.x, acc);
        acc = fmaf(a.y, c.y, acc);
        acc = fmaf(a.z, c.z, acc);
        acc = fmaf(a.w, c.w, acc);
      }
      nl = -lse[bh * g.T + t] * kLog2e;
      nd = -acc;
    }
    LD[(2 * bh) * Tp + t] = nl;
    LD[(2 * bh + 1) * Tp + t] = nd;
  }
}

// ===========================================================================
// Forward
// ===========================================================================
// Per key tile j: S = Qh Kh^T + Qh Kl^T + Ql Kh^T; online softmax over S's row
// (exact rescale of O whenever the row maximum grows); P split into hi/lo in
// TMEM; O += Ph Vh + Ph Vl + Pl Vh, as one N = 128 product Ph [Vh | Vl] (Vh and
// Vl sit side by side in shared memory: the accumulator's first 64 columns
// get Ph Vh, the next 64 Ph Vl) and one N = 64 product Pl Vh into the first
// half; the epilogue adds the halves.  Sixteen MMAs a tile instead of 24 of
// N = 64 (the issue of the PV products sits on the tile's critical path).  S
// is double-buffered and the issuer runs two score tiles ahead of the PV
// products (S(j+2) right after PV(j)), so the softmax of tile j+1 overlaps
// PV(j).  TMEM: S0 [0, 128), S1 [128, 256), Ph [256, 320), Pl [320, 384),
// O [384, 512).  Shared memory: Qh, Ql, then a
// K ring and a V ring of two stages of (hi, lo) each: K(j) is released as soon
// as S(j) has read it, V(j) once PV(j) has.
constexpr int kFwdThreads = 192;   // producer, issuer, four softmax warps
constexpr int kFwdSmem = 2 * kTile + 2 * 2 * kTile + 2 * 2 * kTile + 256 + 1024;
constexpr uint32_t kFPh = 256, kFPl = 320, kFO = 384;

struct SplitFwdBars {
  uint64_t q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full, pv_done, drain;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(kFwdThreads, 1)
split_fwd_kernel(const __grid_constant__ CUtensorMap tm_hi, const __grid_constant__ CUtensorMap tm_lo,
                 float* __restrict__ out, float* __restrict__ lse, int* __restrict__ status, Geometry g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;                          // Qh, Ql
  uint8_t* sK = smem + 2 * kTile;              // stage s: Kh, Kl at sK + 2 s kTile
  uint8_t* sV = smem + 6 * kTile;              // stage s: Vh, Vl at sV + 2 s kTile
  SplitFwdBars* bars = reinterpret_cast<SplitFwdBars*>(smem + 10 * kTile);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nq = (g.T + 127) / 128, bh_count = g.B * g.NH;
  const int qt = nq - 1 - (int)(blockIdx.x / bh_count);    // longest causal ranges first
  const int b = (int)(blockIdx.x % bh_count) / g.NH, h = (int)(blockIdx.x % bh_count) % g.NH;
  const int kh = h / g.grp;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->q_full), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->k_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->k_empty[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->v_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->v_empty[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->s_full[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->p_full), 4);
    ptx::mbar_init(ptx::smem_u32(&bars->pv_done), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->drain), 1);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  auto fail = [&]() {
    *abort_flag = 1;
    record_status(status, kErrDeviceTimeout);
  };
  int k_issued = 0, v_issued = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t qf = ptx::smem_u32(&bars->q_full);
      ptx::mbar_arrive_expect_tx(qf, 2 * kTile);
      ptx::tma_load_3d(ptx::smem_u32(sQ), &tm_hi, h * kHD, qt * 128, b, qf);
      ptx::tma_load_3d(ptx::smem_u32(sQ + kTile), &tm_lo, h * kHD, qt * 128, b, qf);
      for (int j = 0; j <= qt; ++j) {
        const int st = j & 1;
        if (j >= 2 &&
            !ptx::mbar_wait(ptx::smem_u32(&bars->k_empty[st]), ((j >> 1) - 1) & 1, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
        const uint32_t kf = ptx::smem_u32(&bars->k_full[st]);
        ptx::mbar_arrive_expect_tx(kf, 2 * kTile);
        ptx::tma_load_3d(ptx::smem_u32(sK + 2 * st * kTile), &tm_hi, g.C + kh * kHD, j * 128, b, kf);
        ptx::tma_load_3d(ptx::smem_u32(sK + (2 * st + 1) * kTile), &tm_lo, g.C + kh * kHD, j * 128, b, kf);
        k_issued = j + 1;
        if (j >= 2 &&
            !ptx::mbar_wait(ptx::smem_u32(&bars->v_empty[st]), ((j >> 1) - 1) & 1, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
        const uint32_t vf = ptx::smem_u32(&bars->v_full[st]);
        ptx::mbar_arrive_expect_tx(vf, 2 * kTile);
        ptx::tma_load_3d(ptx::smem_u32(sV + 2 * st * kTile), &tm_hi, g.C + g.NKV * kHD + kh * kHD, j * 128, b, vf);
        ptx::tma_load_3d(ptx::smem_u32(sV + (2 * st + 1) * kTile), &tm_lo, g.C + g.NKV * kHD + kh * kHD, j * 128,
                         b, vf);
        v_issued = j + 1;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp runs the issue loop; one elected lane issues each MMA
    // and commit, and every wait is warp-collective)
    {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(128, kHD, false, true);
      constexpr uint32_t idesc_o2 = ptx::idesc_bf16_f32(128, 2 * kHD, false, true);
      const uint64_t dQh = ptx::sw128_desc(ptx::smem_u32(sQ), 16, 1024);
      const uint64_t dQl = ptx::sw128_desc(ptx::smem_u32(sQ + kTile), 16, 1024);
      // S(j) into buffer j & 1 (free: the softmax read S(j-2) before it
      // signalled p_full(j-2), which this thread waited for before PV(j-2)).
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (!ptx::mbar_wait_all(ptx::smem_u32(&bars->k_full[st]), (j >> 1) & 1, abort_flag, kWaitLimitNs)) return false;
        ptx::tc_fence_after();
        const uint64_t dKh = ptx::sw128_desc(ptx::smem_u32(sK + 2 * st * kTile), 16, 1024);
        const uint64_t dKl = ptx::sw128_desc(ptx::smem_u32(sK + (2 * st + 1) * kTile), 16, 1024);
        const uint32_t d_s = tmem + 128u * (uint32_t)st;
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t off = kk * 32;
          ptx::mma_bf16_ss_w(d_s, ptx::desc_advance(dQh, off), ptx::desc_advance(dKh, off), idesc_s, kk > 0 ? 1u : 0u);
          ptx::mma_bf16_ss_w(d_s, ptx::desc_advance(dQh, off), ptx::desc_advance(dKl, off), idesc_s, 1u);
          ptx::mma_bf16_ss_w(d_s, ptx::desc_advance(dQl, off), ptx::desc_advance(dKh, off), idesc_s, 1u);
        }
        ptx::mma_commit_w(ptx::smem_u32(&bars->s_full[st]));
        ptx::mma_commit_w(ptx::smem_u32(&bars->k_empty[st]));
        return true;
      };
      bool ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->q_full), 0, abort_flag, kWaitLimitNs);
      if (ok) ok = issue_s(0);
      if (ok && qt >= 1) ok = issue_s(1);
      for (int j = 0; j <= qt && ok; ++j) {
        const int st = j & 1;
        ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->p_full), j & 1, abort_flag, kWaitLimitNs);
        if (ok) ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->v_full[st]), (j >> 1) & 1, abort_flag, kWaitLimitNs);
        if (!ok) break;
        ptx::tc_fence_after();
        // B: [Vh | Vl] MN-major, the two 64-column atoms kTile apart.
        const uint64_t dV2 = ptx::sw128_desc(ptx::smem_u32(sV + 2 * st * kTile), kTile, 1024);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk) {
          ptx::mma_bf16_ts_w(tmem + kFO, tmem + kFPh + kk * 8, ptx::desc_advance(dV2, kk * 2048), idesc_o2,
                           (j > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_bf16_ts_w(tmem + kFO, tmem + kFPl + kk * 8, ptx::desc_advance(dV2, kk * 2048), idesc_o, 1u);
        }
        ptx::mma_commit_w(ptx::smem_u32(&bars->pv_done));
        ptx::mma_commit_w(ptx::smem_u32(&bars->v_empty[st]));
        if (j + 2 <= qt) ok = issue_s(j + 2);
      }
      if (!ok) fail();
      ptx::mma_commit_w(ptx::smem_u32(&bars->drain));
      ptx::mbar_wait_all(ptx::smem_u32(&bars->drain), 0, nullptr, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;               // query row within the tile
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = g.scale * kLog2e;
    float m = -INFINITY, l = 0.f;                      // log2 units
    bool ok = true;
    for (int j = 0; j <= qt; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu,
                      ptx::mbar_wait(ptx::smem_u32(&bars->s_full[sb]), (j >> 1) & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      ptx::tc_fence_after();
      float s[128];
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t r[32];
        ptx::tmem_ld32(t_lane + 128u * (uint32_t)sb + c0, r);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) s[c0 + c] = __uint_as_float(r[c]);
      }
      if (j == qt) {   // diagonal tile: key c is visible to row `row` iff c <= row
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > row) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m, mx * sl2);
      const float corr = (m == -INFINITY) ? 0.f : ptx::ex2_approx(m - m_new);
      float lsum = 0.f;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        s[c] = ptx::ex2_approx(fmaf(s[c], sl2, -m_new));
        lsum += s[c];
      }
      l = l * corr + lsum;
      // P(j) goes over P(j-1) and O may be rescaled: PV(j-1) must be done.
      if (j > 0) {
        ok = __all_sync(0xffffffffu,
                        ptx::mbar_wait(ptx::smem_u32(&bars->pv_done), (j - 1) & 1, abort_flag, kWaitLimitNs));
        if (!ok) break;
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, m_new > m)) {
#pragma unroll 1
          for (int c0 = 0; c0 < 2 * kHD; c0 += 32) {
            uint32_t o[32];
            ptx::tmem_ld32(t_lane + kFO + c0, o);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * corr);
            ptx::tmem_st32(t_lane + kFO + c0, o);
          }
        }
      }
      m = m_new;
      // P as hi/lo bf16 pairs: key c at column c/2 of Ph and of Pl.
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) split2(s[c0 + 2 * c], s[c0 + 2 * c + 1], ph[c], pl[c]);
        ptx::tmem_st16(t_lane + kFPh + c0 / 2, ph);
        ptx::tmem_st16(t_lane + kFPl + c0 / 2, pl);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->p_full));
    }
    if (ok)
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->pv_done), qt & 1, abort_flag, kWaitLimitNs));
    if (ok) {
      ptx::tc_fence_after();
      float o[64];
      {
        uint32_t a[32], b2[32];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          ptx::tmem_ld32(t_lane + kFO + 32 * h2, a);
          ptx::tmem_ld32(t_lane + kFO + kHD + 32 * h2, b2);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[32 * h2 + c] = __uint_as_float(a[c]) + __uint_as_float(b2[c]);
        }
      }
      const int t = qt * 128 + row;
      if (t < g.T) {
        const float inv_l = 1.f / l;
        float* dst = out + ((size_t)b * g.T + t) * g.C + h * kHD;
#pragma unroll
        for (int q = 0; q < 16; ++q)
          *reinterpret_cast<float4*>(dst + 4 * q) =
              make_float4(o[4 * q] * inv_l, o[4 * q + 1] * inv_l, o[4 * q + 2] * inv_l, o[4 * q + 3] * inv_l);
        lse[((size_t)b * g.NH + h) * g.T + t] = (m + log2f(l)) * kLn2;
      }
    } else {
      fail();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // Every copy issued has landed before shared memory is released.
    for (int st = 0; st < 2 && st < k_issued; ++st)
      ptx::mbar_wait(ptx::smem_u32(&bars->k_full[st]), ((k_issued - 1 - st) / 2) & 1, nullptr, kWaitLimitNs);
    for (int st = 0; st < 2 && st < v_issued; ++st)
      ptx::mbar_wait(ptx::smem_u32(&bars->v_full[st]), ((v_issued - 1 - st) / 2) & 1, nullptr, kWaitLimitNs);
    ptx::mbar_wait(ptx::smem_u32(&bars->q_full), 0, nullptr, kWaitLimitNs);
  }
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Float32 epilogue of one gradient row held in TMEM (kHD columns at `acc`,
// plus the kHD columns after them when `two`: an accumulator kept as two
// halves that add up to the row): scaled by `s`, the RoPE rotation at
// position `t` undone if `rope`, written to `dst` (interleaved pairs back to
// columns 2i, 2i+1).  The row is shared by `nparts` callers: this one takes
// 16 of the 32 pairs (RoPE) or 32 of the 64 columns (no RoPE) when
// nparts = 2.  Warp-collective.
__device__ __forceinline__ void split_grad_row(uint32_t acc, bool two, float s, bool rope, int t,
                                               const Geometry& g, float* dst, bool valid, int part, int nparts) {
  constexpr int HALF = kHD / 2;
  if (!rope) {
    const int n = kHD / nparts, c0 = part * n;
#pragma unroll 1
    for (int c = c0; c < c0 + n; c += 16) {
      uint32_t v[16], w[16];
      ptx::tmem_ld16(acc + c, v);
      if (two) ptx::tmem_ld16(acc + kHD + c, w);
      ptx::tmem_wait_ld();
      float x[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) x[e] = two ? __uint_as_float(v[e]) + __uint_as_float(w[e]) : __uint_as_float(v[e]);
      if (valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<float4*>(dst + c + 4 * q) =
              make_float4(x[4 * q] * s, x[4 * q + 1] * s, x[4 * q + 2] * s, x[4 * q + 3] * s);
      }
    }
    return;
  }
  const int n = HALF / nparts, i0 = part * n;
  uint32_t a[16], c[16], a2[16], c2[16];
  ptx::tmem_ld16(acc + i0, a);
  ptx::tmem_ld16(acc + HALF + i0, c);
  if (two) {
    ptx::tmem_ld16(acc + kHD + i0, a2);
    ptx::tmem_ld16(acc + kHD + HALF + i0, c2);
  }
  ptx::tmem_wait_ld();
  if (!valid) return;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const int i = i0 + e;
    const float xa = two ? __uint_as_float(a[e]) + __uint_as_float(a2[e]) : __uint_as_float(a[e]);
    const float xc = two ? __uint_as_float(c[e]) + __uint_as_float(c2[e]) : __uint_as_float(c[e]);
    float sn, cs, y0, y1;
    __sincosf(rope_angle(t, g.rope_f_hi[i], g.rope_f_lo[i]), &sn, &cs);
    rope_pair_transpose(xa * s, xc * s, cs, sn, y0, y1);
    if (!g.rope_interleaved) {
      dst[i] = y0;
      dst[HALF + i] = y1;
    } else {
      *reinterpret_cast<float2*>(dst + 2 * i) = make_float2(y0, y1);
    }
  }
}

// ===========================================================================
// Backward: dK / dV (key-stationary)
// ===========================================================================
// Per step (query head h of the group, query tile i >= j): S^T = K Q^T and
// dP^T = V dO^T (three products each); P^T = exp2(S^T scale log2e - lse
// log2e) split into TMEM over S^T; dV += P^T dO; dS^T = P^T (dP^T - D) split
// into TMEM over dP^T; dK += dS^T Q.  The gradient products take the hi and
// lo parts of dO (of Q) as one N = 128 B operand [dOh | dOl] (they sit side
// by side in shared memory): P^Th [dOh | dOl] at N = 128 and P^Tl dOh at
// N = 64 into the first half of a two-half accumulator that the epilogue
// adds up, 16 MMAs a product instead of 24 of N = 64.  S^T(n+1) is issued
// one step ahead (dP^T(n), dV(n), S^T(n+1), dK(n)), so that the elementwise
// warps form P^T(n+1) while the tensor core runs dK(n); it goes over P^T(n)
// in the one S^T buffer after dV(n) has read it (MMAs from one thread run in
// order).  Elementwise group w owns queries 64 w .. 64 w + 63: its hi parts at
// columns 64 w .. + 31, lo parts at 64 w + 32 .. + 63 of each 128-column
// block.  TMEM: S^T [0, 128), dP^T [128, 256), dK [256, 384), dV [384, 512).  Shared memory:
// Kh, Kl, Vh, Vl, then two ring stages of (Qh, Ql, dOh, dOl, row tables).
constexpr int kBwdThreads = 320;
constexpr int kDkvStage = 4 * kTile + 1024;
constexpr int kDkvSmem = 4 * kTile + 2 * kDkvStage + 256 + 1024;
constexpr uint32_t kBS = 0, kBDP = 128, kBDK = 256, kBDV = 384;

struct SplitDkvBars {
  uint64_t kv_full, qdo_full[2], qdo_empty[2], s_full[2], dp_full, p_full, ds_full, acc_done, drain;
  uint32_t tmem_base;
  int abort;
};

template <bool ROPE>
__global__ void __launch_bounds__(kBwdThreads, 1)
split_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_hi, const __grid_constant__ CUtensorMap tm_lo,
                      const __grid_constant__ CUtensorMap tm_dohi, const __grid_constant__ CUtensorMap tm_dolo,
                      const float* __restrict__ LD, float* __restrict__ dqkv, int* __restrict__ status, Geometry g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sKV = smem;                                    // Kh, Kl, Vh, Vl
  uint8_t* sRing = smem + 4 * kTile;                      // stage s at sRing + s kDkvStage: Qh, Ql, dOh, dOl, table
  SplitDkvBars* bars = reinterpret_cast<SplitDkvBars*>(sRing + 2 * kDkvStage);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bk = g.B * g.NKV;
  const int j = (int)(blockIdx.x / bk);
  const int b = (int)(blockIdx.x % bk) / g.NKV, kh = (int)(blockIdx.x % bk) % g.NKV;
  const int nq = (g.T + 127) / 128, nqj = nq - j;
  const int n_steps = g.grp * nqj;
  const int Tp = nq * 128;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->kv_full), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->qdo_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->qdo_empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->s_full[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->s_full[1]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->dp_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->p_full), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->ds_full), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->acc_done), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->drain), 1);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // The split passes and tables are written by the grids before this one.
  ptx::grid_dep_wait();
  auto fail = [&]() {
    *abort_flag = 1;
    record_status(status, kErrDeviceTimeout);
  };
  int q_issued = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t kvf = ptx::smem_u32(&bars->kv_full);
      ptx::mbar_arrive_expect_tx(kvf, 4 * kTile);
      ptx::tma_load_3d(ptx::smem_u32(sKV), &tm_hi, g.C + kh * kHD, j * 128, b, kvf);
      ptx::tma_load_3d(ptx::smem_u32(sKV + kTile), &tm_lo, g.C + kh * kHD, j * 128, b, kvf);
      ptx::tma_load_3d(ptx::smem_u32(sKV + 2 * kTile), &tm_hi, g.C + g.NKV * kHD + kh * kHD, j * 128, b, kvf);
      ptx::tma_load_3d(ptx::smem_u32(sKV + 3 * kTile), &tm_lo, g.C + g.NKV * kHD + kh * kHD, j * 128, b, kvf);
      for (int n = 0; n < n_steps; ++n) {
        const int st = n & 1;
        if (n >= 2 &&
            !ptx::mbar_wait(ptx::smem_u32(&bars->qdo_empty[st]), ((n >> 1) - 1) & 1, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
        const int h = kh * g.grp + n / nqj, qi = j + n % nqj;
        uint8_t* s5 = sRing + st * kDkvStage;
        const uint32_t full = ptx::smem_u32(&bars->qdo_full[st]);
        ptx::mbar_arrive_expect_tx(full, 4 * kTile + 1024);
        ptx::tma_load_3d(ptx::smem_u32(s5), &tm_hi, h * kHD, qi * 128, b, full);
        ptx::tma_load_3d(ptx::smem_u32(s5 + kTile), &tm_lo, h * kHD, qi * 128, b, full);
        ptx::tma_load_3d(ptx::smem_u32(s5 + 2 * kTile), &tm_dohi, h * kHD, qi * 128, b, full);
        ptx::tma_load_3d(ptx::smem_u32(s5 + 3 * kTile), &tm_dolo, h * kHD, qi * 128, b, full);
        const float* tab = LD + (size_t)(2 * (b * g.NH + h)) * Tp + qi * 128;
        ptx::bulk_load(ptx::smem_u32(s5 + 4 * kTile), tab, 512, full);
        ptx::bulk_load(ptx::smem_u32(s5 + 4 * kTile + 512), tab + Tp, 512, full);
        q_issued = n + 1;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp runs the issue loop; one elected lane issues each MMA
    // and commit, and every wait is warp-collective)
    {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_g = ptx::idesc_bf16_f32(128, kHD, false, true);
      constexpr uint32_t idesc_g2 = ptx::idesc_bf16_f32(128, 2 * kHD, false, true);
      const uint64_t dKh = ptx::sw128_desc(ptx::smem_u32(sKV), 16, 1024);
      const uint64_t dKl = ptx::sw128_desc(ptx::smem_u32(sKV + kTile), 16, 1024);
      const uint64_t dVh = ptx::sw128_desc(ptx::smem_u32(sKV + 2 * kTile), 16, 1024);
      const uint64_t dVl = ptx::sw128_desc(ptx::smem_u32(sKV + 3 * kTile), 16, 1024);
      // S^T(n) = K Q(n)^T over P^T(n-1), read by dV(n-1) issued before.
      auto issue_s = [&](int n) -> bool {
        const int st = n & 1;
        if (!ptx::mbar_wait_all(ptx::smem_u32(&bars->qdo_full[st]), (n >> 1) & 1, abort_flag, kWaitLimitNs))
          return false;
        ptx::tc_fence_after();
        const uint32_t aQh = ptx::smem_u32(sRing + st * kDkvStage);
        const uint64_t kQh = ptx::sw128_desc(aQh, 16, 1024), kQl = ptx::sw128_desc(aQh + kTile, 16, 1024);
        const uint32_t d_s = tmem + kBS;
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t off = kk * 32;
          ptx::mma_bf16_ss_w(d_s, ptx::desc_advance(dKh, off), ptx::desc_advance(kQh, off), idesc_s, kk > 0 ? 1u : 0u);
          ptx::mma_bf16_ss_w(d_s, ptx::desc_advance(dKh, off), ptx::desc_advance(kQl, off), idesc_s, 1u);
          ptx::mma_bf16_ss_w(d_s, ptx::desc_advance(dKl, off), ptx::desc_advance(kQh, off), idesc_s, 1u);
        }
        ptx::mma_commit_w(ptx::smem_u32(&bars->s_full[st]));
        return true;
      };
      bool ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->kv_full), 0, abort_flag, kWaitLimitNs);
      if (ok && n_steps > 0) ok = issue_s(0);
      for (int n = 0; n < n_steps && ok; ++n) {
        const int st = n & 1;
        const uint32_t aQh = ptx::smem_u32(sRing + st * kDkvStage);
        const uint32_t aDh = aQh + 2 * kTile, aDl = aQh + 3 * kTile;
        const uint64_t kDh = ptx::sw128_desc(aDh, 16, 1024), kDl = ptx::sw128_desc(aDl, 16, 1024);
        // dP^T = V dO^T (over dS^T(n-1), read by dK(n-1) issued before).
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t off = kk * 32;
          ptx::mma_bf16_ss_w(tmem + kBDP, ptx::desc_advance(dVh, off), ptx::desc_advance(kDh, off), idesc_s,
                           kk > 0 ? 1u : 0u);
          ptx::mma_bf16_ss_w(tmem + kBDP, ptx::desc_advance(dVh, off), ptx::desc_advance(kDl, off), idesc_s, 1u);
          ptx::mma_bf16_ss_w(tmem + kBDP, ptx::desc_advance(dVl, off), ptx::desc_advance(kDh, off), idesc_s, 1u);
        }
        ptx::mma_commit_w(ptx::smem_u32(&bars->dp_full));
        // dV += P^T dO (B: [dOh | dOl] MN-major, 16 queries per K step).
        ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->p_full), n & 1, abort_flag, kWaitLimitNs);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint64_t mD2 = ptx::sw128_desc(aDh, kTile, 1024);
        const uint32_t t_p = tmem + kBS;
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk) {
          const uint32_t ph = t_p + hi_col(kk), pl = ph + 32;
          ptx::mma_bf16_ts_w(tmem + kBDV, ph, ptx::desc_advance(mD2, kk * 2048), idesc_g2, (n > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_bf16_ts_w(tmem + kBDV, pl, ptx::desc_advance(mD2, kk * 2048), idesc_g, 1u);
        }
        // The next step's scores, over P^T(n) (dV(n) above read it).
        if (n + 1 < n_steps && !(ok = issue_s(n + 1))) break;
        // dK += dS^T Q (B: [Qh | Ql] MN-major).
        ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->ds_full), n & 1, abort_flag, kWaitLimitNs);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint64_t mQ2 = ptx::sw128_desc(aQh, kTile, 1024);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk) {
          const uint32_t dh = tmem + kBDP + hi_col(kk), dl = dh + 32;
          ptx::mma_bf16_ts_w(tmem + kBDK, dh, ptx::desc_advance(mQ2, kk * 2048), idesc_g2, (n > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_bf16_ts_w(tmem + kBDK, dl, ptx::desc_advance(mQ2, kk * 2048), idesc_g, 1u);
        }
        ptx::mma_commit_w(ptx::smem_u32(&bars->qdo_empty[st]));
      }
      if (ok) ptx::mma_commit_w(ptx::smem_u32(&bars->acc_done));
      else fail();
      ptx::mma_commit_w(ptx::smem_u32(&bars->drain));
      ptx::mbar_wait_all(ptx::smem_u32(&bars->drain), 0, nullptr, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ elementwise + epilogue
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;                // key row within the tile
    const int ks = j * 128 + row;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = g.scale * kLog2e;
    const int q0 = 64 * wg;
    bool ok = true;
    for (int n = 0; n < n_steps; ++n) {
      const int qi = j + n % nqj;
      const bool diag = qi == j;
      const float* tab = reinterpret_cast<const float*>(sRing + (n & 1) * kDkvStage + 4 * kTile);
      const uint32_t t_s = t_lane + kBS;
      ok = __all_sync(0xffffffffu,
                      ptx::mbar_wait(ptx::smem_u32(&bars->s_full[n & 1]), (n >> 1) & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      ptx::tc_fence_after();
      float p[64];
      load64(t_s + q0, p);
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float e = ptx::ex2_approx(fmaf(p[c], sl2, tab[q0 + c]));
        p[c] = (diag && q0 + c < row) ? 0.f : e;        // query q0 + c comes before key `row`
      }
      store_split64(t_s + q0, p);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->p_full));
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->dp_full), n & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      ptx::tc_fence_after();
      float d[64];
      load64(t_lane + kBDP + q0, d);
#pragma unroll
      for (int c = 0; c < 64; ++c) d[c] = p[c] * (d[c] + tab[128 + q0 + c]);
      store_split64(t_lane + kBDP + q0, d);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->ds_full));
    }
    if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->acc_done), 0, abort_flag, kWaitLimitNs));
    if (ok) {
      ptx::tc_fence_after();
      const bool valid = ks < g.T;
      float* drow = dqkv + ((size_t)b * g.T + (valid ? ks : 0)) * g.W;
      split_grad_row(t_lane + kBDV, true, 1.f, false, ks, g, drow + g.C + g.NKV * kHD + kh * kHD, valid, wg, 2);
      split_grad_row(t_lane + kBDK, true, g.scale, ROPE, ks, g, drow + g.C + kh * kHD, valid, wg, 2);
    } else {
      fail();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0) {
    ptx::mbar_wait(ptx::smem_u32(&bars->kv_full), 0, nullptr, kWaitLimitNs);
    for (int st = 0; st < 2 && st < q_issued; ++st)
      ptx::mbar_wait(ptx::smem_u32(&bars->qdo_full[st]), ((q_issued - 1 - st) / 2) & 1, nullptr, kWaitLimitNs);
  }
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// Backward: dQ (query-stationary)
// ===========================================================================
// Per key tile j <= i: S = Q K^T and dP = dO V^T (three products each),
// P = exp2(S scale log2e - lse log2e), dS = P (dP - D) split into TMEM over
// dP, dQ += dSh Kh + dSh Kl + dSl Kh as one N = 128 product dSh [Kh | Kl]
// and one N = 64 product dSl Kh into the accumulator's first half (the
// epilogue adds the halves).  S is double-buffered and issued one tile ahead (dP(j),
// S(j+1), dQ(j)), so that P(j+1) is formed while the tensor core runs dQ(j).
// Elementwise group w owns keys 64 w .. 64 w + 63.  TMEM: S buffers [0, 128)
// and [128, 256), dP [256, 384), dQ [384, 512) as two halves.  Shared memory: Qh, Ql, dOh,
// dOl, a K ring of three stages (K(j) is read by S(j) and by dQ(j), which
// trails S(j+1)) and a V ring of two stages (V(j) is read by dP(j) only).
constexpr int kDqSmem = 4 * kTile + 3 * 2 * kTile + 2 * 2 * kTile + 256 + 1024;
constexpr uint32_t kQDP = 256, kQDQ = 384;

struct SplitDqBars {
  uint64_t qdo_full, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2], dp_full, ds_full, acc_done, drain;
  uint32_t tmem_base;
  int abort;
};

template <bool ROPE>
__global__ void __launch_bounds__(kBwdThreads, 1)
split_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_hi, const __grid_constant__ CUtensorMap tm_lo,
                    const __grid_constant__ CUtensorMap tm_dohi, const __grid_constant__ CUtensorMap tm_dolo,
                    const float* __restrict__ LD, float* __restrict__ dqkv, int* __restrict__ status, Geometry g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQD = smem;                                    // Qh, Ql, dOh, dOl
  uint8_t* sK = smem + 4 * kTile;                         // stage s at sK + 2 s kTile: Kh, Kl
  uint8_t* sV = smem + 10 * kTile;                        // stage s at sV + 2 s kTile: Vh, Vl
  SplitDqBars* bars = reinterpret_cast<SplitDqBars*>(smem + 14 * kTile);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nq = (g.T + 127) / 128, bh_count = g.B * g.NH;
  const int qt = nq - 1 - (int)(blockIdx.x / bh_count);
  const int b = (int)(blockIdx.x % bh_count) / g.NH, h = (int)(blockIdx.x % bh_count) % g.NH;
  const int kh = h / g.grp;
  const int Tp = nq * 128;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->qdo_full), 1);
    for (int s = 0; s < 3; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->k_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->k_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->v_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->v_empty[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->s_full[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->dp_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->ds_full), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->acc_done), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->drain), 1);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  ptx::grid_dep_wait();
  auto fail = [&]() {
    *abort_flag = 1;
    record_status(status, kErrDeviceTimeout);
  };
  int k_issued = 0, v_issued = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t qf = ptx::smem_u32(&bars->qdo_full);
      ptx::mbar_arrive_expect_tx(qf, 4 * kTile);
      ptx::tma_load_3d(ptx::smem_u32(sQD), &tm_hi, h * kHD, qt * 128, b, qf);
      ptx::tma_load_3d(ptx::smem_u32(sQD + kTile), &tm_lo, h * kHD, qt * 128, b, qf);
      ptx::tma_load_3d(ptx::smem_u32(sQD + 2 * kTile), &tm_dohi, h * kHD, qt * 128, b, qf);
      ptx::tma_load_3d(ptx::smem_u32(sQD + 3 * kTile), &tm_dolo, h * kHD, qt * 128, b, qf);
      for (int jj = 0; jj <= qt; ++jj) {
        const int ks = jj % 3, vs = jj & 1;
        if (jj >= 3 &&
            !ptx::mbar_wait(ptx::smem_u32(&bars->k_empty[ks]), (jj / 3 - 1) & 1, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
        const uint32_t kf = ptx::smem_u32(&bars->k_full[ks]);
        ptx::mbar_arrive_expect_tx(kf, 2 * kTile);
        ptx::tma_load_3d(ptx::smem_u32(sK + 2 * ks * kTile), &tm_hi, g.C + kh * kHD, jj * 128, b, kf);
        ptx::tma_load_3d(ptx::smem_u32(sK + (2 * ks + 1) * kTile), &tm_lo, g.C + kh * kHD, jj * 128, b, kf);
        k_issued = jj + 1;
        if (jj >= 2 &&
            !ptx::mbar_wait(ptx::smem_u32(&bars->v_empty[vs]), ((jj >> 1) - 1) & 1, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
        const uint32_t vf = ptx::smem_u32(&bars->v_full[vs]);
        ptx::mbar_arrive_expect_tx(vf, 2 * kTile);
        ptx::tma_load_3d(ptx::smem_u32(sV + 2 * vs * kTile), &tm_hi, g.C + g.NKV * kHD + kh * kHD, jj * 128, b, vf);
        ptx::tma_load_3d(ptx::smem_u32(sV + (2 * vs + 1) * kTile), &tm_lo, g.C + g.NKV * kHD + kh * kHD, jj * 128,
                         b, vf);
        v_issued = jj + 1;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp runs the issue loop; one elected lane issues each MMA
    // and commit, and every wait is warp-collective)
    {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_g = ptx::idesc_bf16_f32(128, kHD, false, true);
      constexpr uint32_t idesc_g2 = ptx::idesc_bf16_f32(128, 2 * kHD, false, true);
      const uint64_t dQh = ptx::sw128_desc(ptx::smem_u32(sQD), 16, 1024);
      const uint64_t dQl = ptx::sw128_desc(ptx::smem_u32(sQD + kTile), 16, 1024);
      const uint64_t dDh = ptx::sw128_desc(ptx::smem_u32(sQD + 2 * kTile), 16, 1024);
      const uint64_t dDl = ptx::sw128_desc(ptx::smem_u32(sQD + 3 * kTile), 16, 1024);
      // S(j) = Q K(j)^T into buffer j & 1 (free: the elementwise warps read
      // S(j-2) before they signalled ds_full(j-2), waited for before dQ(j-2)).
      auto issue_s = [&](int jj) -> bool {
        const int ks = jj % 3;
        if (!ptx::mbar_wait_all(ptx::smem_u32(&bars->k_full[ks]), (jj / 3) & 1, abort_flag, kWaitLimitNs)) return false;
        ptx::tc_fence_after();
        const uint32_t aKh = ptx::smem_u32(sK + 2 * ks * kTile);
        const uint64_t kKh = ptx::sw128_desc(aKh, 16, 1024), kKl = ptx::sw128_desc(aKh + kTile, 16, 1024);
        const uint32_t d_s = tmem + 128u * (uint32_t)(jj & 1);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t off = kk * 32;
          ptx::mma_bf16_ss_w(d_s, ptx::desc_advance(dQh, off), ptx::desc_advance(kKh, off), idesc_s, kk > 0 ? 1u : 0u);
          ptx::mma_bf16_ss_w(d_s, ptx::desc_advance(dQh, off), ptx::desc_advance(kKl, off), idesc_s, 1u);
          ptx::mma_bf16_ss_w(d_s, ptx::desc_advance(dQl, off), ptx::desc_advance(kKh, off), idesc_s, 1u);
        }
        ptx::mma_commit_w(ptx::smem_u32(&bars->s_full[jj & 1]));
        return true;
      };
      bool ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->qdo_full), 0, abort_flag, kWaitLimitNs);
      if (ok) ok = issue_s(0);
      for (int jj = 0; jj <= qt && ok; ++jj) {
        const int ks = jj % 3, vs = jj & 1;
        // dP = dO V^T (over dS(j-1), read by dQ(j-1) issued before).
        if (!(ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->v_full[vs]), (jj >> 1) & 1, abort_flag, kWaitLimitNs)))
          break;
        ptx::tc_fence_after();
        const uint32_t aVh = ptx::smem_u32(sV + 2 * vs * kTile);
        const uint64_t kVh = ptx::sw128_desc(aVh, 16, 1024), kVl = ptx::sw128_desc(aVh + kTile, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint32_t off = kk * 32;
          ptx::mma_bf16_ss_w(tmem + kQDP, ptx::desc_advance(dDh, off), ptx::desc_advance(kVh, off), idesc_s,
                           kk > 0 ? 1u : 0u);
          ptx::mma_bf16_ss_w(tmem + kQDP, ptx::desc_advance(dDh, off), ptx::desc_advance(kVl, off), idesc_s, 1u);
          ptx::mma_bf16_ss_w(tmem + kQDP, ptx::desc_advance(dDl, off), ptx::desc_advance(kVh, off), idesc_s, 1u);
        }
        ptx::mma_commit_w(ptx::smem_u32(&bars->dp_full));
        ptx::mma_commit_w(ptx::smem_u32(&bars->v_empty[vs]));
        // The next tile's scores, into the other S buffer.
        if (jj + 1 <= qt && !(ok = issue_s(jj + 1))) break;
        // dQ += dS K (B: [Kh | Kl] MN-major, the two 64-column atoms kTile
        // apart; 16 keys per K step).
        ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->ds_full), jj & 1, abort_flag, kWaitLimitNs);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t aKh = ptx::smem_u32(sK + 2 * ks * kTile);
        const uint64_t mK2 = ptx::sw128_desc(aKh, kTile, 1024);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk) {
          const uint32_t dh = tmem + kQDP + hi_col(kk), dl = dh + 32;
          ptx::mma_bf16_ts_w(tmem + kQDQ, dh, ptx::desc_advance(mK2, kk * 2048), idesc_g2,
                           (jj > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_bf16_ts_w(tmem + kQDQ, dl, ptx::desc_advance(mK2, kk * 2048), idesc_g, 1u);
        }
        ptx::mma_commit_w(ptx::smem_u32(&bars->k_empty[ks]));
      }
      if (ok) ptx::mma_commit_w(ptx::smem_u32(&bars->acc_done));
      else fail();
      ptx::mma_commit_w(ptx::smem_u32(&bars->drain));
      ptx::mbar_wait_all(ptx::smem_u32(&bars->drain), 0, nullptr, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ elementwise + epilogue
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;                // query row within the tile
    const int tq = qt * 128 + row;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = g.scale * kLog2e;
    const int k0 = 64 * wg;
    const size_t tab = (size_t)(2 * (b * g.NH + h)) * Tp + tq;   // tq < Tp: padded rows read zeros
    const float nl = LD[tab], nd = LD[tab + Tp];
    bool ok = true;
    for (int jj = 0; jj <= qt; ++jj) {
      const bool diag = jj == qt;
      ok = __all_sync(0xffffffffu,
                      ptx::mbar_wait(ptx::smem_u32(&bars->s_full[jj & 1]), (jj >> 1) & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      ptx::tc_fence_after();
      float p[64];
      load64(t_lane + 128u * (uint32_t)(jj & 1) + k0, p);
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float e = ptx::ex2_approx(fmaf(p[c], sl2, nl));
        p[c] = (diag && k0 + c > row) ? 0.f : e;        // key k0 + c comes after query `row`
      }
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->dp_full), jj & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      ptx::tc_fence_after();
      float d[64];
      load64(t_lane + kQDP + k0, d);
#pragma unroll
      for (int c = 0; c < 64; ++c) d[c] = p[c] * (d[c] + nd);
      store_split64(t_lane + kQDP + k0, d);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->ds_full));
    }
    if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->acc_done), 0, abort_flag, kWaitLimitNs));
    if (ok) {
      ptx::tc_fence_after();
      const bool valid = tq < g.T;
      float* drow = dqkv + ((size_t)b * g.T + (valid ? tq : 0)) * g.W + h * kHD;
      split_grad_row(t_lane + kQDQ, true, g.scale, ROPE, tq, g, drow, valid, wg, 2);
    } else {
      fail();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0) {
    ptx::mbar_wait(ptx::smem_u32(&bars->qdo_full), 0, nullptr, kWaitLimitNs);
    for (int st = 0; st < 3 && st < k_issued; ++st)
      ptx::mbar_wait(ptx::smem_u32(&bars->k_full[st]), ((k_issued - 1 - st) / 3) & 1, nullptr, kWaitLimitNs);
    for (int st = 0; st < 2 && st < v_issued; ++st)
      ptx::mbar_wait(ptx::smem_u32(&bars->v_full[st]), ((v_issued - 1 - st) / 2) & 1, nullptr, kWaitLimitNs);
  }
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

unsigned grid_for(long long units, int per_block) {
  const long long blocks = (units + per_block - 1) / per_block;
  return (unsigned)(blocks < 152 * 8 ? (blocks > 0 ? blocks : 1) : 152 * 8);
}

cudaError_t launch_split(const SplitArgs& a, cudaStream_t stream, bool with_dout) {
  const Geometry& g = a.g;
  const long long rows = (long long)g.B * g.T;
  const bool rope = g.rope_theta > 0.f;
  const int qk_cols = (g.NH + g.NKV) * g.hd;
  if (a.qkv_given) {   // the forward's parts of this qkv: only dO is split
    split_plain_kernel<<<grid_for(rows * (g.C / 8), 256), 256, 0, stream>>>(
        static_cast<const float*>(a.dout), g.C, 0, g.C, a.dout_hi, a.dout_lo, g.C, rows);
    return cudaGetLastError();
  }
  // Q and K (rotated when RoPE is on), then V, then dO.
  if (rope) {
    split_rope_kernel<<<grid_for(rows * (g.NH + g.NKV) * (g.hd / 16), 256), 256, 0, stream>>>(
        static_cast<const float*>(a.qkv), a.qkv_hi, a.qkv_lo, g);
  } else {
    split_plain_kernel<<<grid_for(rows * (qk_cols / 8), 256), 256, 0, stream>>>(
        static_cast<const float*>(a.qkv), g.W, 0, qk_cols, a.qkv_hi, a.qkv_lo, g.W, rows);
  }
  split_plain_kernel<<<grid_for(rows * (g.NKV * g.hd / 8), 256), 256, 0, stream>>>(
      static_cast<const float*>(a.qkv), g.W, qk_cols, g.NKV * g.hd, a.qkv_hi, a.qkv_lo, g.W, rows);
  if (with_dout)
    split_plain_kernel<<<grid_for(rows * (g.C / 8), 256), 256, 0, stream>>>(
        static_cast<const float*>(a.dout), g.C, 0, g.C, a.dout_hi, a.dout_lo, g.C, rows);
  return cudaGetLastError();
}

}  // namespace

bool split_supported(const Geometry& g) { return g.hd == kHD; }

cudaError_t split_fwd_launch(const SplitArgs& a, cudaStream_t stream) {
  const Geometry& g = a.g;
  cudaError_t e = cudaFuncSetAttribute(split_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdSmem);
  if (e != cudaSuccess) return e;
  prof_begin(kKernelSplitPrep, stream);
  e = launch_split(a, stream, false);
  prof_end(kKernelSplitPrep, stream);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(((g.T + 127) / 128) * g.B * g.NH);
  prof_begin(kKernelFwdSplit, stream);
  split_fwd_kernel<<<grid, kFwdThreads, kFwdSmem, stream>>>(a.tm_hi, a.tm_lo, static_cast<float*>(a.out), a.lse,
                                                            a.status, g);
  prof_end(kKernelFwdSplit, stream);
  return cudaGetLastError();
}

cudaError_t split_bwd_launch(const SplitArgs& a, cudaStream_t stream) {
  const Geometry& g = a.g;
  const bool rope = g.rope_theta > 0.f;
  auto k1 = rope ? split_bwd_dkdv_kernel<true> : split_bwd_dkdv_kernel<false>;
  auto k2 = rope ? split_bwd_dq_kernel<true> : split_bwd_dq_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, kDkvSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmem);
  if (e != cudaSuccess) return e;
  const int nq = (g.T + 127) / 128, Tp = nq * 128;
  prof_begin(kKernelSplitPrep, stream);
  e = launch_split(a, stream, true);
  if (e == cudaSuccess) {
    split_tables_kernel<<<grid_for((long long)g.B * g.NH * Tp, 256), 256, 0, stream>>>(
        a.LD, static_cast<const float*>(a.out), static_cast<const float*>(a.dout), a.lse, g, Tp);
    e = cudaGetLastError();
  }
  prof_end(kKernelSplitPrep, stream);
  if (e != cudaSuccess) return e;
  prof_begin(kKernelBwdDkdvSplit, stream);
  e = launch_pdl(k1, dim3((unsigned)(nq * g.B * g.NKV)), dim3(kBwdThreads), kDkvSmem, stream, a.tm_hi, a.tm_lo,
                 a.tm_dohi, a.tm_dolo, (const float*)a.LD, static_cast<float*>(a.dqkv), a.status, g);
  prof_end(kKernelBwdDkdvSplit, stream);
  if (e != cudaSuccess) return e;
  prof_begin(kKernelBwdDqSplit, stream);
  e = launch_pdl(k2, dim3((unsigned)(nq * g.B * g.NH)), dim3(kBwdThreads), kDqSmem, stream, a.tm_hi, a.tm_lo,
                 a.tm_dohi, a.tm_dolo, (const float*)a.LD, static_cast<float*>(a.dqkv), a.status, g);
  prof_end(kKernelBwdDqSplit, stream);
  return e;
}

}  // namespace attn
