// Causal MHA/GQA attention backward on sm_103a tensor cores (bf16 in, f32
// accumulation), head size 64 or 128.  Deterministic and free of atomics.
//
// The gradient is that of "nanoeuler -- CUDA kernels", attention_backward_kernel:
// with P recomputed from the saved log-sum-exp, P_ts = exp(s_ts - lse_t),
//   dP = dO V^T,  dS = P * (dP - D)  with D_t = dO_t . O_t  (the row dot of
//   "CUDA C microgpt"'s attention_backward_kernel, computed by a prologue),
//   dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K,
// dK and dV summed over the query heads that share a kv head (the page's
// atomicAdd into the shared dk/dv), and dQ/dK carried back through the RoPE
// rotation (the page's rope_kernel with inverse=1 on dqkv).
//
// Two kernels split the work so that every output element has exactly one
// writer:
//  * dkdv: one CTA per (128-key tile j, kv head, batch row).  K_j and V_j stay
//    in shared memory; the CTA walks every query head of the group and every
//    128-query tile that can see tile j.  Per step: S^T = K Q^T and
//    dP^T = V dO^T into TMEM, P^T and dS^T (bf16) back into TMEM over the
//    score columns already read, then dV += P^T dO and dK += dS^T Q (A
//    operand from TMEM) accumulate in TMEM.
//  * dq:   one CTA per (128-query tile i, query head, batch row).  Q_i and dO_i
//    stay in shared memory; the CTA walks the 128-key tiles 0..i.  Per step:
//    S = Q K^T and dP = dO V^T into TMEM, dS (bf16) back into TMEM over the
//    dP columns already read, then dQ += dS K (A operand from TMEM)
//    accumulates in TMEM.
// Warp roles in both: warp 0 TMA producer; warp 1 TMEM owner and the single
// MMA issuer; two elementwise warpgroups with one TMEM lane (one key or query
// row) per thread, each owning half of every step's 128 columns, which also
// split the epilogue.  Every MMA has N = 128.  All waits are bounded.
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_profile.h"
#include "attn_ptx.cuh"

namespace attn {
namespace {

constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kThreadsDkdv = 320;   // producer, MMA issuer, two elementwise warpgroups
constexpr int kThreadsDq = 352;     // producer, MMA issuer, two elementwise warpgroups, Q producer
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint4 pack8(const uint32_t* f, float s) {
  return make_uint4(pack_bf16x2(__uint_as_float(f[0]) * s, __uint_as_float(f[1]) * s),
                    pack_bf16x2(__uint_as_float(f[2]) * s, __uint_as_float(f[3]) * s),
                    pack_bf16x2(__uint_as_float(f[4]) * s, __uint_as_float(f[5]) * s),
                    pack_bf16x2(__uint_as_float(f[6]) * s, __uint_as_float(f[7]) * s));
}

// Byte offset of the 16-byte chunk holding columns col..col+7 (col a multiple
// of 8) of row `row` in a 128-row bf16 tile stored as 128-byte-swizzled atom
// columns of 64 elements: the layout of the tensor maps' 64 x 128 boxes.
__device__ __forceinline__ uint32_t sw128_chunk(int row, int col) {
  return (uint32_t)((col >> 6) * (128 * 128) + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4));
}

// Epilogue of one gradient row held in TMEM (HD float32 columns at `acc`):
// multiply by `s`, undo the RoPE rotation at position `t` if `rope` (cos and
// sin of each pair's angle from the prologue's table `cs` when given: in the
// dQ kernel, where the epilogue overlaps the next item's MMAs, forming them
// per pair took as long as a step), round to
// bf16 and write row `row` of the swizzled staging tile `stile` (HD columns),
// from which one thread then writes the whole tile with TMA stores (coalesced;
// one 16-byte store per thread and row would not be).  Every lane of the warp
// must call this (tcgen05.ld is warp-collective).  Chunks of 32 columns (32
// pairs with RoPE) are dealt round-robin to `nparts` callers; this caller
// handles part `part`.
template <int HD>
__device__ __forceinline__ void stage_grad_row(uint32_t acc, float s, bool rope, int t, const Geometry& g,
                                               const float* __restrict__ cs, uint8_t* stile, int row, int part,
                                               int nparts) {
  if (!rope) {
#pragma unroll 1
    for (int c0 = 32 * part; c0 < HD; c0 += 32 * nparts) {
      uint32_t v[32];
      ptx::tmem_ld32(acc + c0, v);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(stile + sw128_chunk(row, c0 + 8 * q)) = pack8(&v[8 * q], s);
    }
    return;
  }
  constexpr int HALF = HD / 2;
#pragma unroll 1
  for (int c0 = 32 * part; c0 < HALF; c0 += 32 * nparts) {
    uint32_t lo[32], hi[32];
    // Pair i of position t at cs[2 (i T + t)]: the warp's 32 consecutive rows
    // read one contiguous run per pair.  Rows past T (clipped by the TMA
    // store) read the last row's angles.  Without a table (cs == NULL) the
    // angles are formed here.
    float2 a[32];
    if (cs != nullptr) {
      const float2* cs2 = reinterpret_cast<const float2*>(cs) + (size_t)c0 * g.T + (t < g.T ? t : g.T - 1);
#pragma unroll
      for (int e = 0; e < 32; ++e) a[e] = __ldg(cs2 + (size_t)e * g.T);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) __sincosf(rope_angle(t, g.rope_f_hi[c0 + e], g.rope_f_lo[c0 + e]), &a[e].y, &a[e].x);
    }
    ptx::tmem_ld32(acc + c0, lo);
    ptx::tmem_ld32(acc + HALF + c0, hi);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      float y0, y1;
      rope_pair_transpose(__uint_as_float(lo[e]) * s, __uint_as_float(hi[e]) * s, a[e].x, a[e].y, y0, y1);
      lo[e] = __float_as_uint(y0);
      hi[e] = __float_as_uint(y1);
    }
    if (!g.rope_interleaved) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        *reinterpret_cast<uint4*>(stile + sw128_chunk(row, c0 + 8 * q)) = pack8(&lo[8 * q], 1.f);
        *reinterpret_cast<uint4*>(stile + sw128_chunk(row, HALF + c0 + 8 * q)) = pack8(&hi[8 * q], 1.f);
      }
    } else {
      // Interleaved pairing: pair i goes back to columns 2i and 2i + 1.
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t w[8] = {lo[4 * q], hi[4 * q], lo[4 * q + 1], hi[4 * q + 1],
                               lo[4 * q + 2], hi[4 * q + 2], lo[4 * q + 3], hi[4 * q + 3]};
        *reinterpret_cast<uint4*>(stile + sw128_chunk(row, 2 * c0 + 8 * q)) = pack8(w, 1.f);
      }
    }
  }
}

// ===========================================================================
// dK / dV kernel
// ===========================================================================
// One step = 128 queries of one query head of the group, so that every MMA
// has N = 128 (full tensor-core rate; N = 64 runs at about two thirds).  TMEM:
// S^T [0, 128), dP^T [128, 256), dK and dV accumulators from column 256.  The
// elementwise groups write P^T / dS^T (bf16 pairs) back into TMEM over score
// columns they have already read, and the gradient MMAs take their A operand
// from there; the MMA issue order (see the issuer) keeps the tensor core busy
// with the previous step's dK while P^T is formed.
template <int HD>
struct DkdvCfg {
  static constexpr int kKeys = 128, kQ = 128;
  static constexpr int kKTile = kKeys * HD * 2;        // K_j or V_j
  static constexpr int kQTile = kQ * HD * 2;           // Q_i or dO_i
  static constexpr int kAtom = 128 * 128;              // one 64-column atom column of a 128-row tile
  // Q/dO ring depth: a slot is recycled after the step's gradient MMAs.
  static constexpr int kQStages = (HD == 128) ? 2 : 4;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKTile;
  static constexpr int kQOff = kVOff + kKTile;
  static constexpr int kDOOff = kQOff + kQStages * kQTile;
  static constexpr int kLDOff = kDOOff + kQStages * kQTile;  // per stage: lse2[128], then D[128] (float)
  static constexpr int kBarOff = kLDOff + kQStages * kQ * 8;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDK = 256, kTmemDV = 256 + HD, kTmemCols = 512;
  // Head size 64 leaves TMEM columns 384-511 free: S^T is double-buffered
  // there and issued a step ahead (see the issuer).
  static constexpr bool kDblS = (HD == 64);
  static constexpr uint32_t kTmemS2 = 384;
  static_assert(!kDblS || kTmemDV + HD <= kTmemS2, "second score buffer overlaps the gradient accumulators");
  static_assert(kSmemBytes <= 232448, "dK/dV kernel exceeds the 227 KB shared-memory limit");
};

struct DkdvBarriers {
  uint64_t kv_full, acc_done, drain, staged;
  uint64_t qdo_full[4], qdo_empty[4];
  // p_full[2 * b + h]: half h of P^T of the steps using score buffer b
  // (head size 128: b = 0 only).  With the scores a step ahead, the
  // elementwise groups can finish P^T(n+1) before the issuer has waited for
  // P^T(n); one barrier per buffer keeps each wait within one phase.
  uint64_t s_full[2], dp_full, p_full[4], ds_full;
  uint32_t tmem_base;
  int abort;
};

// TMEM column (relative to a score block) of the bf16 pairs of queries
// 16*kk .. 16*kk+15: elementwise group w writes the 32 columns of its queries
// 64w .. 64w+63 at 64w.
__device__ __forceinline__ uint32_t pair_col(int kk) { return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8); }

template <int HD, bool ROPE>
__global__ void __launch_bounds__(kThreadsDkdv, 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dqkv, const float* __restrict__ LD,
                int* __restrict__ status, Geometry g) {
  using Cfg = DkdvCfg<HD>;
  constexpr int NQS = Cfg::kQStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + Cfg::kKOff;
  uint8_t* sV = smem + Cfg::kVOff;
  uint8_t* sQ = smem + Cfg::kQOff;
  uint8_t* sDO = smem + Cfg::kDOOff;
  float* sLD = reinterpret_cast<float*>(smem + Cfg::kLDOff);
  DkdvBarriers* bars = reinterpret_cast<DkdvBarriers*>(smem + Cfg::kBarOff);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // Heaviest key tiles (small j) first.
  const int bk = g.B * g.NKV;
  const int j = (int)(blockIdx.x / bk);
  const int b = (blockIdx.x % bk) / g.NKV, kh = (blockIdx.x % bk) % g.NKV;
  const int nq128 = (g.T + 127) / 128;
  const int nq = nq128 - j;                     // 128-query tiles that can see key tile j
  const int n_steps = g.grp * nq;
  const int Tp = row_table_rows(g.T);

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->kv_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->acc_done), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->drain), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->staged), 8);
    for (int i = 0; i < NQS; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->qdo_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->qdo_empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->s_full[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->s_full[1]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->dp_full), 1);
    for (int i = 0; i < 4; ++i) ptx::mbar_init(ptx::smem_u32(&bars->p_full[i]), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->ds_full), 8);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), Cfg::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // Everything above overlapped the prologue's tail; its outputs (row table,
  // rotated Q/K) are read below.  Once every CTA of this grid is past this
  // point the dQ kernel may start: it depends on the prologue only, which has
  // then completed.
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  auto fail = [&]() {
    *abort_flag = 1;
    record_status(status, kErrDeviceTimeout);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Per step: Q_i and dO_i (TMA, 128 rows) and the step's 128 row-table
    // entries of each kind (two bulk copies; the table is padded to whole
    // 128-row tiles with zeros, and padding query rows have zero Q and dO, so
    // they add nothing).
    int issued = 0;
    if (lane == 0) {
      const uint32_t kvf = ptx::smem_u32(&bars->kv_full);
      ptx::mbar_arrive_expect_tx(kvf, 2 * Cfg::kKTile);
#pragma unroll
      for (int a = 0; a < HD / 64; ++a) {
        ptx::tma_load_3d(ptx::smem_u32(sK + a * Cfg::kAtom), &tm_k, g.C + kh * HD + 64 * a, j * 128, b, kvf);
        ptx::tma_load_3d(ptx::smem_u32(sV + a * Cfg::kAtom), &tm_v, g.C + g.NKV * HD + kh * HD + 64 * a, j * 128, b,
                         kvf);
      }
      int h = kh * g.grp, qi = j;                  // step n's query head and 128-query tile
      for (int n = 0; n < n_steps; ++n) {
        const int st = n % NQS, u = n / NQS;
        if (u > 0 && !ptx::mbar_wait(ptx::smem_u32(&bars->qdo_empty[st]), (u - 1) & 1, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
        const uint32_t full = ptx::smem_u32(&bars->qdo_full[st]);
        ptx::mbar_arrive_expect_tx(full, 2 * Cfg::kQTile + Cfg::kQ * 8);
#pragma unroll
        for (int a = 0; a < HD / 64; ++a) {
          ptx::tma_load_3d(ptx::smem_u32(sQ + st * Cfg::kQTile + a * Cfg::kAtom), &tm_q, h * HD + 64 * a, qi * 128, b,
                           full);
          ptx::tma_load_3d(ptx::smem_u32(sDO + st * Cfg::kQTile + a * Cfg::kAtom), &tm_do, h * HD + 64 * a, qi * 128,
                           b, full);
        }
        const float* tab = LD + (size_t)(2 * (b * g.NH + h)) * Tp + qi * 128;
        ptx::bulk_load(ptx::smem_u32(sLD + st * 256), tab, Cfg::kQ * 4, full);
        ptx::bulk_load(ptx::smem_u32(sLD + st * 256 + 128), tab + Tp, Cfg::kQ * 4, full);
        issued = n + 1;
        if (++qi == nq128) {
          qi = j;
          ++h;
        }
      }
    }
    if (lane == 0 && *abort_flag) {
      ptx::mbar_wait(ptx::smem_u32(&bars->kv_full), 0, nullptr, kWaitLimitNs);
      for (int st = 0; st < NQS && st < issued; ++st)
        ptx::mbar_wait(ptx::smem_u32(&bars->qdo_full[st]), ((issued - 1 - st) / NQS) & 1, nullptr, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the whole warp
    // runs the loop; one elected lane issues each MMA and commit)
    {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_g = ptx::idesc_bf16_f32(128, HD, false, true);
      const uint64_t dK = ptx::sw128_desc(ptx::smem_u32(sK), 16, 1024);
      const uint64_t dV = ptx::sw128_desc(ptx::smem_u32(sV), 16, 1024);
      const uint64_t dQk = ptx::sw128_desc(ptx::smem_u32(sQ), 16, 1024);
      const uint64_t dDOk = ptx::sw128_desc(ptx::smem_u32(sDO), 16, 1024);
      const uint64_t dQm = ptx::sw128_desc(ptx::smem_u32(sQ), Cfg::kAtom, 1024);
      const uint64_t dDOm = ptx::sw128_desc(ptx::smem_u32(sDO), Cfg::kAtom, 1024);
      bool ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->kv_full), 0, abort_flag, kWaitLimitNs);
      // dK += dS^T Q of step m once both groups wrote dS^T(m); frees the
      // step's ring slot.
      auto issue_dk = [&](int m) -> bool {
        if (!ptx::mbar_wait_all(ptx::smem_u32(&bars->ds_full), m & 1, abort_flag, kWaitLimitNs)) return false;
        ptx::tc_fence_after();
        const int ms = m % NQS;
        const uint64_t gq = ptx::desc_advance(dQm, ms * Cfg::kQTile);
#pragma unroll
        for (int kk = 0; kk < Cfg::kQ / 16; ++kk)
          ptx::mma_bf16_ts_w(tmem + Cfg::kTmemDK, tmem + Cfg::kTmemDP + pair_col(kk), ptx::desc_advance(gq, kk * 2048),
                           idesc_g, (m > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit_w(ptx::smem_u32(&bars->qdo_empty[ms]));
        return true;
      };
      // S^T(n) into its score buffer, once Q_n landed.
      auto sbuf = [&](int n) -> uint32_t { return (Cfg::kDblS && (n & 1)) ? Cfg::kTmemS2 : Cfg::kTmemS; };
      auto issue_s = [&](int n) -> bool {
        const int qs = n % NQS;
        if (!ptx::mbar_wait_all(ptx::smem_u32(&bars->qdo_full[qs]), (n / NQS) & 1, abort_flag, kWaitLimitNs))
          return false;
        ptx::tc_fence_after();
        const uint64_t bq = ptx::desc_advance(dQk, qs * Cfg::kQTile);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Cfg::kAtom + (kk & 3) * 32;
          ptx::mma_bf16_ss_w(tmem + sbuf(n), ptx::desc_advance(dK, off), ptx::desc_advance(bq, off), idesc_s,
                             kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit_w(ptx::smem_u32(&bars->s_full[Cfg::kDblS ? (n & 1) : 0]));
        return true;
      };
      // Issue order S^T(n), dK(n-1), dP^T(n), dV(n) (head size 128), or with
      // the scores a step ahead in two buffers S^T(n+1), dK(n-1), dP^T(n),
      // dV(n) (head size 64, whose shorter MMAs would leave the tensor core
      // idle while P^T(n) is formed): the tensor core works on dK(n-1) and
      // dP^T(n) while the elementwise groups turn S^T(n) into P^T(n), and on
      // dV(n) and the next scores while they form dS^T(n).  dP^T(n)
      // overwrites dS^T(n-1) after dK(n-1) has been issued, and a score MMA
      // overwrites P^T of the step that last used its buffer after that
      // step's dV: MMAs from one thread run in order.
      if (Cfg::kDblS) ok = ok && issue_s(0);
      for (int n = 0; n < n_steps && ok; ++n) {
        const int qs = n % NQS;
        if (!(ok = Cfg::kDblS ? (n + 1 >= n_steps || issue_s(n + 1)) : issue_s(n))) break;
        const uint64_t bdo = ptx::desc_advance(dDOk, qs * Cfg::kQTile);
        if (n > 0 && !(ok = issue_dk(n - 1))) break;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Cfg::kAtom + (kk & 3) * 32;
          ptx::mma_bf16_ss_w(tmem + Cfg::kTmemDP, ptx::desc_advance(dV, off), ptx::desc_advance(bdo, off), idesc_s,
                           kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit_w(ptx::smem_u32(&bars->dp_full));
        // dV += P^T dO once both groups wrote P^T.
        // P^T arrives in halves: queries 0-31 and 64-95 (K steps 0, 1, 4,
        // 5), then 32-63 and 96-127, so dV starts before it is complete.
        const uint64_t gdo = ptx::desc_advance(dDOm, qs * Cfg::kQTile);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int pb = Cfg::kDblS ? (n & 1) : 0;
          if (!(ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->p_full[2 * pb + hh]), Cfg::kDblS ? (n >> 1) & 1 : n & 1,
                                        abort_flag, kWaitLimitNs)))
            break;
          ptx::tc_fence_after();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int kk = (i >> 1) * 4 + hh * 2 + (i & 1);
            ptx::mma_bf16_ts_w(tmem + Cfg::kTmemDV, tmem + sbuf(n) + pair_col(kk),
                               ptx::desc_advance(gdo, kk * 2048), idesc_g, (n > 0 || kk > 0) ? 1u : 0u);
          }
        }
        if (!ok) break;
      }
      if (ok && n_steps > 0) ok = issue_dk(n_steps - 1);
      if (ok) ptx::mma_commit_w(ptx::smem_u32(&bars->acc_done));
      if (!ok) fail();
      ptx::mma_commit_w(ptx::smem_u32(&bars->drain));
      ptx::mbar_wait_all(ptx::smem_u32(&bars->drain), 0, nullptr, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ elementwise + epilogue
    // Group wg owns queries 64*wg .. 64*wg+63 of every step (TMEM columns
    // 64*wg .. of each score block); thread = key row = TMEM lane.
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;           // key row within the tile
    const int ks = j * 128 + row;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t t_dp = t_lane + Cfg::kTmemDP + 64 * wg;
    const float sl2 = g.scale * kLog2e;
    const float2 sl2x2 = make_float2(sl2, sl2);
    bool ok = true;
    for (int n = 0; n < n_steps; ++n) {
      const int qi = j + n % nq;
      const bool diag = qi == j;                   // query tile == key tile: query q is before key row iff q < row
      const int q0 = 64 * wg;                      // first query (within the tile) of this group
      // This group's row-table entries: -lse * log2(e) and -D of its 64 queries.
      const float4* lse4 = reinterpret_cast<const float4*>(sLD + (n % NQS) * 256 + q0);
      const float4* d4 = reinterpret_cast<const float4*>(sLD + (n % NQS) * 256 + 128 + q0);
      // ---- P^T = exp2(S^T * scale * log2(e) - lse * log2(e)), while dP^T is computed.
      float p[64];
      float4 Lw[2];
      // s_full(n) also means the step's loads (table included) have landed:
      // the issuer waited for them before the score MMAs.
      const int sb = Cfg::kDblS ? (n & 1) : 0;
      const uint32_t t_s = t_lane + (sb ? Cfg::kTmemS2 : Cfg::kTmemS) + 64 * wg;
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->s_full[sb]), Cfg::kDblS ? (n >> 1) & 1 : n & 1,
                                                  abort_flag, kWaitLimitNs));
      if (!ok) break;
      ptx::tc_fence_after();
      Lw[0] = lse4[0];
      Lw[1] = lse4[1];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sr[32], pw[16];
        ptx::tmem_ld32(t_s + 32 * half, sr);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const int k = (32 * half + c) >> 2;       // float4 index 0..15
          const float4 L = Lw[k & 1];
          if (k + 2 < 16) Lw[k & 1] = lse4[k + 2];
          const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2,
                                       make_float2(L.x, L.y));
          const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), sl2x2,
                                       make_float2(L.z, L.w));
          float e[4] = {ptx::ex2_approx(x0.x), ptx::ex2_approx(x0.y), ptx::ex2_approx(x1.x), ptx::ex2_approx(x1.y)};
          if (diag) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
              if (q0 + 32 * half + c + t < row) e[t] = 0.f;
          }
#pragma unroll
          for (int t = 0; t < 4; ++t) p[32 * half + c + t] = e[t];
          pw[c >> 1] = pack_bf16x2(e[0], e[1]);
          pw[(c >> 1) + 1] = pack_bf16x2(e[2], e[3]);
        }
        ptx::tmem_st16(t_s + 16 * half, pw);
        // Each half of this group's queries is signalled once it is in TMEM.
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->p_full[2 * sb + half]));
      }
      // ---- dS^T = P^T * (dP^T - D), while dV is accumulated.
      Lw[0] = d4[0];
      Lw[1] = d4[1];
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->dp_full), n & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      ptx::tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t dr[32], dw[16];
        ptx::tmem_ld32(t_dp + 32 * half, dr);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const int k = (32 * half + c) >> 2;
          const float4 L = Lw[k & 1];
          if (k + 2 < 16) Lw[k & 1] = d4[k + 2];
          const float2 a0 = __fmul2_rn(make_float2(p[32 * half + c], p[32 * half + c + 1]),
                                       __fadd2_rn(make_float2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])),
                                                  make_float2(L.x, L.y)));
          const float2 a1 = __fmul2_rn(make_float2(p[32 * half + c + 2], p[32 * half + c + 3]),
                                       __fadd2_rn(make_float2(__uint_as_float(dr[c + 2]), __uint_as_float(dr[c + 3])),
                                                  make_float2(L.z, L.w)));
          dw[c >> 1] = pack_bf16x2(a0.x, a0.y);
          dw[(c >> 1) + 1] = pack_bf16x2(a1.x, a1.y);
        }
        ptx::tmem_st16(t_dp + 16 * half, dw);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->ds_full));
    }
    if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->acc_done), 0, abort_flag, kWaitLimitNs));
    // Every MMA has completed: the first Q and dO ring stages are free and
    // stage the dV and dK tiles; rows past T are clipped by the TMA store.
    uint8_t* stV = sQ;
    uint8_t* stK = sDO;
    if (ok) {
      ptx::tc_fence_after();
      stage_grad_row<HD>(t_lane + Cfg::kTmemDV, 1.f, false, ks, g, nullptr, stV, row, wg, 2);
      // The angles are formed here: at the CTA's end nothing overlaps the
      // epilogue, and the table reads measured slower than forming them.
      stage_grad_row<HD>(t_lane + Cfg::kTmemDK, g.scale, ROPE, ks, g, nullptr, stK, row, wg, 2);
    } else {
      fail();
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->staged));
    if (warp == 2 && lane == 0) {
      if (ptx::mbar_wait(ptx::smem_u32(&bars->staged), 0, abort_flag, kWaitLimitNs) && !*abort_flag) {
#pragma unroll
        for (int a = 0; a < HD / 64; ++a) {
          ptx::tma_store_3d(&tm_dqkv, ptx::smem_u32(stV + a * Cfg::kAtom), g.C + g.NKV * HD + kh * HD + 64 * a,
                            j * 128, b);
          ptx::tma_store_3d(&tm_dqkv, ptx::smem_u32(stK + a * Cfg::kAtom), g.C + kh * HD + 64 * a, j * 128, b);
        }
        ptx::bulk_commit();
        ptx::bulk_wait();
      } else {
        fail();
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// ===========================================================================
// dQ kernel
// ===========================================================================
// Persistent: one CTA per SM claims work items (128-query tile, query head,
// batch row), heaviest (longest causal key range) first, from a counter in
// the workspace that the prologue clears: CTAs that become resident early
// (the kernel starts while the dK/dV kernel drains) take more items.  Per
// item, Q_i and dO_i stay in shared memory and the CTA walks the 128-key
// tiles 0..i (every MMA N = 128).  A Q producer warp loads the next item's Q
// into the other of two Q buffers while the current item runs (an item's dQ
// tile is staged in its own Q buffer for the TMA store); its dO follows as
// soon as the current item's last dP MMA has read the one dO buffer, and its
// first MMAs overlap the current item's epilogue.
// TMEM: S [0, 128), dP [128, 256), two dQ accumulators from 256 (items
// alternate).  The elementwise groups turn S into P (kept in registers) while
// dP is computed, then dP into dS, written (bf16 pairs) into TMEM over the dP
// columns they have read; the dQ MMA takes its A operand from there.  Issue
// order S(n), dQ(n-1), dP(n): the tensor core works on dQ(n-1) and dP(n)
// while P(n) is formed.
template <int HD>
struct DqCfg {
  static constexpr int kQ = 128, kKeys = 128;
  static constexpr int kQTile = kQ * HD * 2;           // Q_i, dO_i or a staged dQ tile
  static constexpr int kKTile = kKeys * HD * 2;        // K_j or V_j
  static constexpr int kAtom = 128 * 128;              // one 64-column atom column of a 128-row tile
  // K(t) is read by S(t) and by dQ(t), which is issued a step later, so its
  // ring needs a stage more than V's (read by dP(t) only) to keep each load
  // a step ahead of its use.
  static constexpr int kKStages = (HD == 128) ? 3 : 4; // K ring depth
  static constexpr int kVStages = (HD == 128) ? 1 : 4; // V ring depth
  // Two Q buffers (items alternate; an item's dQ tile is staged for its TMA
  // store in the item's own Q buffer once its last score MMA has read it).
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = kQOff + 2 * kQTile;
  static constexpr int kKOff = kDOOff + kQTile;
  static constexpr int kVOff = kKOff + kKStages * kKTile;
  static constexpr int kBarOff = kVOff + kVStages * kKTile;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDQ = 256, kTmemCols = 512;
  static constexpr int kItemSlots = 4;                 // claimed-item queue depth
  static_assert(kSmemBytes <= 232448, "dQ kernel exceeds the 227 KB shared-memory limit");
};

struct DqBarriers {
  uint64_t q_full[2], do_full, do_empty, drain;
  // v_empty: V stage free (a ring of more than one stage; with one stage the
  // producer waits for dp_full instead, dP being V's only reader).
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full, s_free, dp_full, ds_full;
  uint64_t acc_done[2], dq_free[2], staged, stage_free[2];
  uint64_t item_full[4], item_empty[4];
  int item[4];
  uint32_t tmem_base;
  int abort;
};

// Work item w -> (batch row, query head, 128-query tile); heaviest first.
struct DqItem {
  int b, h, qt;
};
__device__ __forceinline__ DqItem dq_item(int w, const Geometry& g) {
  const int n_qt = (g.T + 127) / 128, bh_count = g.B * g.NH;
  DqItem it;
  it.qt = n_qt - 1 - w / bh_count;
  const int bh = w % bh_count;
  it.b = bh / g.NH;
  it.h = bh % g.NH;
  return it;
}

template <int HD, bool ROPE>
__global__ void __launch_bounds__(kThreadsDq, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_dqkv, const float* __restrict__ LD,
              const float* __restrict__ rope_cs, int* __restrict__ item_counter, int n_items,
              int* __restrict__ status, Geometry g) {
  using Cfg = DqCfg<HD>;
  constexpr int NKS = Cfg::kKStages, NVS = Cfg::kVStages, NIS = Cfg::kItemSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Cfg::kQOff;
  uint8_t* sDO = smem + Cfg::kDOOff;
  uint8_t* sK = smem + Cfg::kKOff;
  uint8_t* sV = smem + Cfg::kVOff;
  DqBarriers* bars = reinterpret_cast<DqBarriers*>(smem + Cfg::kBarOff);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->q_full[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->q_full[1]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->do_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->do_empty), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->drain), 1);
    for (int i = 0; i < NKS; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->k_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->k_empty[i]), 1);
    }
    for (int i = 0; i < NVS; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->v_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->v_empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->s_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->s_free), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->dp_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->ds_full), 8);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->acc_done[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->dq_free[i]), 8);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->staged), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->stage_free[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->stage_free[1]), 1);
    for (int i = 0; i < NIS; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->item_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->item_empty[i]), 10);  // MMA issuer, 8 elementwise warps, Q producer
    }
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), Cfg::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // Launched as a programmatic dependent of the dK/dV kernel, whose CTAs all
  // waited for the prologue before allowing this grid to start; this kernel
  // reads only the prologue's outputs (row tables, rotated Q/K, the cleared
  // item counter) and the inputs, and writes dqkv columns the dK/dV kernel
  // does not touch, so it needs no wait of its own.
  auto fail = [&]() {
    *abort_flag = 1;
    record_status(status, kErrDeviceTimeout);
  };
  // Claimed item `it` of this CTA (-1: no more work), published by the producer.
  auto next_item = [&](int it, bool* okp) -> int {
    const int slot = it % NIS;
    if (!ptx::mbar_wait(ptx::smem_u32(&bars->item_full[slot]), (it / NIS) & 1, abort_flag, kWaitLimitNs)) {
      *okp = false;
      return -1;
    }
    return *reinterpret_cast<volatile int*>(&bars->item[slot]);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int k_issued = 0, v_issued = 0, do_issued = 0;  // global sequence counters
      int gs = 0;                                    // global index of the item's first key step
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int slot = it % NIS;
        if (it >= NIS &&
            !(ok = ptx::mbar_wait(ptx::smem_u32(&bars->item_empty[slot]), (it / NIS - 1) & 1, abort_flag,
                                  kWaitLimitNs)))
          break;
        int w = atomicAdd(item_counter, 1);
        if (w >= n_items) w = -1;
        bars->item[slot] = w;
        ptx::mbar_arrive(ptx::smem_u32(&bars->item_full[slot]));
        if (w < 0) break;
        const DqItem item = dq_item(w, g);
        const int kh = item.h / g.grp, n_steps = item.qt + 1;
        // K, V and dO of this item (Q comes from the Q producer warp); dO once
        // the previous item's last dP MMA has read it.
        bool do_loaded = false;
        for (int n = 0; n < n_steps && ok; ++n) {
          const int gi = gs + n, st = gi % NKS, u = gi / NKS;
          if (u > 0 && !(ok = ptx::mbar_wait(ptx::smem_u32(&bars->k_empty[st]), (u - 1) & 1, abort_flag,
                                             kWaitLimitNs)))
            break;
          const uint32_t kf = ptx::smem_u32(&bars->k_full[st]);
          ptx::mbar_arrive_expect_tx(kf, Cfg::kKTile);
#pragma unroll
          for (int a = 0; a < HD / 64; ++a)
            ptx::tma_load_3d(ptx::smem_u32(sK + st * Cfg::kKTile + a * Cfg::kAtom), &tm_k, g.C + kh * HD + 64 * a,
                             n * 128, item.b, kf);
          k_issued = gi + 1;
          if (!do_loaded) {
            if (it > 0 &&
                !(ok = ptx::mbar_wait(ptx::smem_u32(&bars->do_empty), (it - 1) & 1, abort_flag, kWaitLimitNs)))
              break;
            const uint32_t df = ptx::smem_u32(&bars->do_full);
            ptx::mbar_arrive_expect_tx(df, Cfg::kQTile);
#pragma unroll
            for (int a = 0; a < HD / 64; ++a)
              ptx::tma_load_3d(ptx::smem_u32(sDO + a * Cfg::kAtom), &tm_do, item.h * HD + 64 * a, item.qt * 128,
                               item.b, df);
            do_loaded = true;
            do_issued = it + 1;
          }
          const int vs = gi % NVS, vu = gi / NVS;
          // One V stage: dP(gi-1), its only reader, has completed once
          // dp_full has (dP(gi) cannot complete before V(gi) is loaded).
          if (vu > 0 && !(ok = (NVS == 1 ? ptx::mbar_wait(ptx::smem_u32(&bars->dp_full), (gi - 1) & 1, abort_flag,
                                                          kWaitLimitNs)
                                         : ptx::mbar_wait(ptx::smem_u32(&bars->v_empty[vs]), (vu - 1) & 1, abort_flag,
                                                          kWaitLimitNs))))
            break;
          const uint32_t vf = ptx::smem_u32(&bars->v_full[vs]);
          ptx::mbar_arrive_expect_tx(vf, Cfg::kKTile);
#pragma unroll
          for (int a = 0; a < HD / 64; ++a)
            ptx::tma_load_3d(ptx::smem_u32(sV + vs * Cfg::kKTile + a * Cfg::kAtom), &tm_v,
                             g.C + g.NKV * HD + kh * HD + 64 * a, n * 128, item.b, vf);
          v_issued = gi + 1;
        }
        gs += n_steps;
      }
      if (!ok) fail();
      if (*abort_flag) {
        // Let every copy already in flight land before shared memory is released.
        if (do_issued > 0)
          ptx::mbar_wait(ptx::smem_u32(&bars->do_full), (do_issued - 1) & 1, nullptr, kWaitLimitNs);
        for (int st = 0; st < NKS && st < k_issued; ++st)
          ptx::mbar_wait(ptx::smem_u32(&bars->k_full[st]), ((k_issued - 1 - st) / NKS) & 1, nullptr, kWaitLimitNs);
        for (int st = 0; st < NVS && st < v_issued; ++st)
          ptx::mbar_wait(ptx::smem_u32(&bars->v_full[st]), ((v_issued - 1 - st) / NVS) & 1, nullptr, kWaitLimitNs);
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ Q producer
    // Q of item it into buffer it & 1 as soon as the TMA store of item it-2's
    // dQ tile, staged there, has read it (which also means item it-2's score
    // MMAs have completed): the next item's Q lands while this one runs.
    if (lane == 0) {
      int q_issued = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int w = next_item(it, &ok);
        ptx::mbar_arrive(ptx::smem_u32(&bars->item_empty[it % NIS]));
        if (!ok || w < 0) break;
        const DqItem item = dq_item(w, g);
        const int qb = it & 1;
        if (it >= 2 && !(ok = ptx::mbar_wait(ptx::smem_u32(&bars->stage_free[qb]), ((it >> 1) - 1) & 1, abort_flag,
                                             kWaitLimitNs)))
          break;
        const uint32_t qf = ptx::smem_u32(&bars->q_full[qb]);
        ptx::mbar_arrive_expect_tx(qf, Cfg::kQTile);
#pragma unroll
        for (int a = 0; a < HD / 64; ++a)
          ptx::tma_load_3d(ptx::smem_u32(sQ + qb * Cfg::kQTile + a * Cfg::kAtom), &tm_q, item.h * HD + 64 * a,
                           item.qt * 128, item.b, qf);
        q_issued = it + 1;
      }
      if (!ok) fail();
      // Let the Q loads already in flight land before shared memory is released.
      for (int i = q_issued - 2 > 0 ? q_issued - 2 : 0; i < q_issued; ++i)
        ptx::mbar_wait(ptx::smem_u32(&bars->q_full[i & 1]), (i >> 1) & 1, nullptr, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the whole warp
    // runs the loop; one elected lane issues each MMA and commit)
    {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_g = ptx::idesc_bf16_f32(128, HD, false, true);
      const uint64_t dQ = ptx::sw128_desc(ptx::smem_u32(sQ), 16, 1024);
      const uint64_t dDO = ptx::sw128_desc(ptx::smem_u32(sDO), 16, 1024);
      const uint64_t dK = ptx::sw128_desc(ptx::smem_u32(sK), 16, 1024);
      const uint64_t dV = ptx::sw128_desc(ptx::smem_u32(sV), 16, 1024);
      const uint64_t dKm = ptx::sw128_desc(ptx::smem_u32(sK), Cfg::kAtom, 1024);
      bool ok = true;
      // The pending dQ MMA group: global step index, its item, and whether it
      // is that item's first / last step.
      int p_g = -1, p_it = 0;
      bool p_first = false, p_last = false;
      auto issue_dq = [&]() -> bool {
        if (!ptx::mbar_wait_all(ptx::smem_u32(&bars->ds_full), p_g & 1, abort_flag, kWaitLimitNs)) return false;
        const int db = p_it & 1;
        // The item's first dQ MMA overwrites accumulator db: the epilogue of
        // the item two before must have read it.
        if (p_first && p_it >= 2 &&
            !ptx::mbar_wait_all(ptx::smem_u32(&bars->dq_free[db]), ((p_it >> 1) - 1) & 1, abort_flag, kWaitLimitNs))
          return false;
        ptx::tc_fence_after();
        const int ms = p_g % NKS;
        const uint64_t bk = ptx::desc_advance(dKm, ms * Cfg::kKTile);
#pragma unroll
        for (int kk = 0; kk < Cfg::kKeys / 16; ++kk)
          ptx::mma_bf16_ts_w(tmem + Cfg::kTmemDQ + 128 * db, tmem + Cfg::kTmemDP + pair_col(kk),
                           ptx::desc_advance(bk, kk * 2048), idesc_g, (!p_first || kk > 0) ? 1u : 0u);
        ptx::mma_commit_w(ptx::smem_u32(&bars->k_empty[ms]));
        if (p_last) ptx::mma_commit_w(ptx::smem_u32(&bars->acc_done[db]));
        return true;
      };
      int gs = 0;
      for (int it = 0; ok; ++it) {
        const int w = next_item(it, &ok);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->item_empty[it % NIS]));
        if (!ok || w < 0) break;
        const DqItem item = dq_item(w, g);
        const int n_steps = item.qt + 1;
        ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->q_full[it & 1]), (it >> 1) & 1, abort_flag, kWaitLimitNs);
        const uint64_t dQb = ptx::desc_advance(dQ, (it & 1) * Cfg::kQTile);
        for (int n = 0; n < n_steps && ok; ++n) {
          const int gi = gs + n, ks = gi % NKS, u = gi / NKS, vs = gi % NVS, vu = gi / NVS;
          // K landed; the groups have read the previous S out of TMEM.
          ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->k_full[ks]), u & 1, abort_flag, kWaitLimitNs);
          if (ok && gi > 0) ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->s_free), (gi - 1) & 1, abort_flag, kWaitLimitNs);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint64_t bk = ptx::desc_advance(dK, ks * Cfg::kKTile), bv = ptx::desc_advance(dV, vs * Cfg::kKTile);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * Cfg::kAtom + (kk & 3) * 32;
            ptx::mma_bf16_ss_w(tmem + Cfg::kTmemS, ptx::desc_advance(dQb, off), ptx::desc_advance(bk, off), idesc_s,
                             kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit_w(ptx::smem_u32(&bars->s_full));
          // The previous step's dQ reads its dS in the dP columns: issued
          // before dP overwrites them (MMAs from one thread run in order).
          if (p_g >= 0 && !(ok = issue_dq())) break;
          if (n == 0 && !(ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->do_full), it & 1, abort_flag, kWaitLimitNs)))
            break;
          if (!(ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->v_full[vs]), vu & 1, abort_flag, kWaitLimitNs))) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * Cfg::kAtom + (kk & 3) * 32;
            ptx::mma_bf16_ss_w(tmem + Cfg::kTmemDP, ptx::desc_advance(dDO, off), ptx::desc_advance(bv, off), idesc_s,
                             kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit_w(ptx::smem_u32(&bars->dp_full));
          if (NVS > 1) ptx::mma_commit_w(ptx::smem_u32(&bars->v_empty[vs]));
          if (n == n_steps - 1) ptx::mma_commit_w(ptx::smem_u32(&bars->do_empty));
          p_g = gi;
          p_it = it;
          p_first = n == 0;
          p_last = n == n_steps - 1;
        }
        gs += n_steps;
      }
      if (ok && p_g >= 0) ok = issue_dq();
      if (!ok) fail();
      ptx::mma_commit_w(ptx::smem_u32(&bars->drain));
      ptx::mbar_wait_all(ptx::smem_u32(&bars->drain), 0, nullptr, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ elementwise + epilogue
    // Group wg owns keys 64*wg .. 64*wg+63 of every step (TMEM columns 64*wg
    // .. of each score block); thread = query row = TMEM lane.
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;           // query row within the tile
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t t_s = t_lane + Cfg::kTmemS + 64 * wg, t_dp = t_lane + Cfg::kTmemDP + 64 * wg;
    const float sl2 = g.scale * kLog2e;
    const float2 sl2x2 = make_float2(sl2, sl2);
    const int Tp = row_table_rows(g.T);
    const int k0 = 64 * wg;                        // first key (within a tile) of this group
    // Warp 2's store in flight (the Q buffer it reads, -1: none): released
    // once the store has read it, at warp 2's next dS arrival or at the start
    // of the next item, whichever comes first (never later: the Q producer
    // waits for the release before loading the item after next).
    int store_db = -1;
    auto release_store = [&]() {
      if (warp == 2 && lane == 0 && store_db >= 0) {
        ptx::bulk_wait_read();
        ptx::mbar_arrive(ptx::smem_u32(&bars->stage_free[store_db]));   // the Q producer may reload it
        store_db = -1;
      }
    };
    // dQ of a finished item: staged in the item's Q buffer (its last score
    // MMA, which precedes its last dQ MMA, has read it) and written with TMA
    // stores (rows past T are clipped).  It runs after the next item's first
    // dS is out (the RoPE undo in it takes about as long as a step), so that
    // the tensor core works on that item's first MMAs meanwhile.
    auto epilogue = [&](int pit, const DqItem& pitem) -> bool {
      const int db = pit & 1;
      const int ptq = pitem.qt * 128 + row;
      uint8_t* sSt = sQ + db * Cfg::kQTile;
      if (!__all_sync(0xffffffffu,
                      ptx::mbar_wait(ptx::smem_u32(&bars->acc_done[db]), (pit >> 1) & 1, abort_flag, kWaitLimitNs)))
        return false;
      ptx::tc_fence_after();
      stage_grad_row<HD>(t_lane + Cfg::kTmemDQ + 128 * db, g.scale, ROPE, ptq, g, rope_cs, sSt, row, wg, 2);
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(ptx::smem_u32(&bars->dq_free[db]));
        ptx::mbar_arrive(ptx::smem_u32(&bars->staged));
      }
      bool sok = true;
      if (warp == 2 && lane == 0) {
        sok = ptx::mbar_wait(ptx::smem_u32(&bars->staged), pit & 1, abort_flag, kWaitLimitNs);
        if (sok) {
#pragma unroll
          for (int a = 0; a < HD / 64; ++a)
            ptx::tma_store_3d(&tm_dqkv, ptx::smem_u32(sSt + a * Cfg::kAtom), pitem.h * HD + 64 * a, pitem.qt * 128,
                              pitem.b);
          ptx::bulk_commit();
          store_db = db;                           // released by release_store()
        }
      }
      return __shfl_sync(0xffffffffu, sok ? 1 : 0, 0) != 0;
    };
    int pend_it = -1;                              // finished item whose epilogue is due
    DqItem pend_item{};
    bool ok = true;
    int gs = 0;
    for (int it = 0; ok; ++it) {
      const int w = __shfl_sync(0xffffffffu, lane == 0 ? next_item(it, &ok) : 0, 0);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->item_empty[it % NIS]));
      if (!ok || w < 0) break;
      release_store();
      const DqItem item = dq_item(w, g);
      const int n_steps = item.qt + 1;
      const int tq = item.qt * 128 + row;
      // This row's table entries -lse * log2(e) and -D; padding rows have
      // zero Q and dO, hence dP = 0 and dS = 0.
      const size_t tab = (size_t)(2 * (item.b * g.NH + item.h)) * Tp + tq;
      const float2 ldr = (tq < g.T) ? make_float2(LD[tab], LD[tab + Tp]) : make_float2(0.f, 0.f);
      const float2 nl2 = make_float2(ldr.x, ldr.x), nd2 = make_float2(ldr.y, ldr.y);
      for (int n = 0; n < n_steps; ++n) {
        const int gi = gs + n;
        const bool diag = n == item.qt;            // key tile == query tile: key k is after row iff k > row
        // ---- P = exp2(S * scale * log2(e) - lse * log2(e)), while dP is computed.
        float p[64];
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->s_full), gi & 1, abort_flag, kWaitLimitNs));
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sr[32];
          ptx::tmem_ld32(t_s + 32 * half, sr);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2, nl2);
            float e0 = ptx::ex2_approx(x.x), e1 = ptx::ex2_approx(x.y);
            if (diag) {
              if (k0 + 32 * half + c > row) e0 = 0.f;
              if (k0 + 32 * half + c + 1 > row) e1 = 0.f;
            }
            p[32 * half + c] = e0;
            p[32 * half + c + 1] = e1;
          }
        }
        // S is in registers: the next score MMA may overwrite it.
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->s_free));
        // ---- dS = P * (dP - D), while the previous dQ is accumulated.
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->dp_full), gi & 1, abort_flag, kWaitLimitNs));
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t dr[32], dw[16];
          ptx::tmem_ld32(t_dp + 32 * half, dr);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 ds = __fmul2_rn(make_float2(p[32 * half + c], p[32 * half + c + 1]),
                                         __fadd2_rn(make_float2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])),
                                                    nd2));
            dw[c >> 1] = pack_bf16x2(ds.x, ds.y);
          }
          ptx::tmem_st16(t_dp + 16 * half, dw);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->ds_full));
        release_store();
        if (n == 0 && pend_it >= 0) {
          if (!(ok = epilogue(pend_it, pend_item))) break;
          pend_it = -1;
        }
      }
      if (!ok) break;
      gs += n_steps;
      pend_it = it;
      pend_item = item;
    }
    if (ok && pend_it >= 0) ok = epilogue(pend_it, pend_item);
    if (!ok) fail();
    // Every tile store has landed in global memory before the CTA exits.
    if (warp == 2 && lane == 0) ptx::bulk_wait();
  }

  // Finish only after the dK/dV kernel this grid overlapped has completed, so
  // that work later in the stream (which waits for this grid only) never
  // overwrites the workspace while the dK/dV kernel still reads it.
  ptx::grid_dep_wait();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

template <int HD, bool ROPE>
cudaError_t launch_bwd(const Tc05BwdArgs& a, cudaStream_t stream) {
  const Geometry& g = a.g;
  auto k1 = bwd_dkdv_kernel<HD, ROPE>;
  auto k2 = bwd_dq_kernel<HD, ROPE>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, DkdvCfg<HD>::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<HD>::kSmemBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid1 = (unsigned)(((g.T + 127) / 128) * g.B * g.NKV);
  prof_begin(kKernelBwdDkdvTc05, stream);
  e = launch_pdl(k1, dim3(grid1), dim3(kThreadsDkdv), DkdvCfg<HD>::kSmemBytes, stream, a.tm_qk[1], a.tm_v[1],
                 a.tm_qk[1], a.tm_do[1], a.tm_dqkv, a.LD, a.status, g);
  prof_end(kKernelBwdDkdvTc05, stream);
  if (e != cudaSuccess) return e;
  const int n_items = ((g.T + 127) / 128) * g.B * g.NH;
  const unsigned grid2 = (unsigned)(n_items < a.num_sms ? n_items : a.num_sms);
  prof_begin(kKernelBwdDqTc05, stream);
  e = launch_pdl(k2, dim3(grid2), dim3(kThreadsDq), DqCfg<HD>::kSmemBytes, stream, a.tm_qk[1], a.tm_do[1],
                 a.tm_qk[1], a.tm_v[1], a.tm_dqkv, a.LD, a.rope_cs, a.item_counter, n_items, a.status, g);
  prof_end(kKernelBwdDqTc05, stream);
  return e;
}

}  // namespace

cudaError_t tc05_bwd_launch(const Tc05BwdArgs& a, cudaStream_t stream) {
  const bool rope = a.g.rope_theta > 0.f;
  if (a.g.hd == 128) return rope ? launch_bwd<128, true>(a, stream) : launch_bwd<128, false>(a, stream);
  if (a.g.hd == 64) return rope ? launch_bwd<64, true>(a, stream) : launch_bwd<64, false>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
