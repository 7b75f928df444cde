// Causal MHA/GQA attention forward on sm_103a tensor cores (bf16 in, f32
// accumulation), head size 64 or 128.
//
// Persistent kernel: one CTA per SM walks its share of a list of work items
// (dealt back and forth across the CTAs, see snake_item), one item = a
// 128-query tile of one (batch row, query head), heaviest (longest causal row
// range) first; query heads that share a kv head are adjacent in
// the list, so concurrently running CTAs reuse K/V tiles through L2.  Every
// role runs one continuous stream of key tiles across its items, so the next
// item's loads and first MMAs overlap the current item's last softmax and
// epilogue; barriers and TMEM are set up once per CTA.  Within an item the
// key tiles 0..qt are visited (causal tile skipping).  Warp roles:
//   warp 0      TMA producer: Q (double-buffered across items), then K_j and
//               V_j into separate rings; K runs two tiles ahead of V so that
//               the score MMA never waits on a load.
//   warp 1      TMEM owner and score-MMA issuer (one thread): S_j = Q K_j^T
//               into one of two TMEM score buffers.
//   warp 2      PV-MMA issuer (one thread): O += P_j V_j with P_j read from
//               tensor memory (A operand) and V_j from shared memory.
//               Two issuers keep the tensor core fed: each one's barrier
//               checks and commits overlap the other's queued MMAs.
//   warps 4-7   softmax: thread = query row = TMEM lane.  Reads S_j, keeps the
//               running max m and sum l, writes P_j (bf16) into one of two
//               TMEM P buffers, rescales O in TMEM when m grows past a
//               threshold (exact: l and O share the stale max), and at the end
//               of an item writes out = O / l and lse = m + ln l.
//   warps 8-11  (RoPE only) rotate each item's Q and every landed K tile in
//               shared memory before the score MMA may read them.
// TMEM columns: S0, S1 (128 each), P0, P1 (64 each, bf16 pairs), then O (one
// buffer at head size 128, two at 64).
// The math is that of "nanoeuler -- CUDA kernels", attention_forward_kernel
// (scale 1/sqrt(hd), kv head h/(NH/NKV), causal mask, row softmax, PV), with
// the softmax evaluated online over key tiles; lse follows the forward kernel
// declaration of the same page (one float per (b, h, t)).
//
// Every wait is bounded (see ptx::mbar_wait); on expiry the CTA records
// ATTN_ERR_DEVICE_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM
// and exits.
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_profile.h"
#include "attn_ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;                      // queries per tile
constexpr int kBN = 128;                      // keys per tile
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr float kRescaleThreshold = 8.0f;     // log2 units: P may reach 2^8 before O is rescaled
constexpr int kPvWarp = 2;
constexpr int kSoftmaxWarp0 = 4;              // warpgroup 1
constexpr int kRopeWarp0 = 8;                 // warpgroup 2 (RoPE only)

template <int HD, bool ROPE>
struct FwdCfg {
  static constexpr int kAtomBytes = kBM * 128;              // 128 rows x 128 B swizzle-atom column
  static constexpr int kTileBytes = kBM * HD * 2;           // Q / K / V tile
  static constexpr int kKStages = (HD == 128) ? 3 : 4;      // K ring depth
  static constexpr int kVStages = (HD == 128) ? 2 : 4;      // V ring depth
  static constexpr int kQOff = 0;                           // two Q buffers (items in flight)
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;   // barriers + alignment slack
  static_assert(kSmemBytes <= 232448, "forward kernel exceeds the 227 KB shared-memory limit");
  static constexpr int kThreads = ROPE ? 384 : 256;
  static constexpr int kOBuffers = (HD == 128) ? 1 : 2;
  static constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemP0 = 256, kTmemP1 = 320, kTmemO0 = 384,
                            kTmemO1 = 384 + HD, kTmemCols = 512;
};

struct FwdBarriers {
  uint64_t q_full[2], q_ready[2], q_empty[2], o_free[2];
  uint64_t pv_done[2], p_full[2], drain, drain2, o_staged;
  uint64_t s_full[2], s_free[2];
  uint64_t k_full[4], k_ready[4], k_empty[4], v_full[4], v_empty[4];
  uint32_t tmem_base;
  int abort;
};

// Work item w -> (batch row, query head, query tile).  Items are ordered by
// decreasing query tile (longest causal range first); within a tile, the
// heads of one batch row are consecutive.
struct FwdItem {
  int b, h, kh, qt;
};

__device__ __forceinline__ FwdItem fwd_item(int w, const Geometry& g) {
  const int n_qt = (g.T + kBM - 1) / kBM;
  const int bh_count = g.B * g.NH;
  FwdItem it;
  it.qt = n_qt - 1 - w / bh_count;
  const int bh = w % bh_count;
  it.b = bh / g.NH;
  it.h = bh % g.NH;
  it.kh = it.h / g.grp;
  return it;
}

// The it-th item of the CTA with index w0 in a grid of dw CTAs.  Items are
// dealt in rounds of dw, forward in even rounds and backward in odd ones
// (boustrophedon), so that the CTA that took the heaviest item of one round
// takes the lightest of the next: with items sorted by decreasing weight this
// keeps the per-CTA totals within a few percent of each other, where a plain
// stride leaves the first CTAs with up to ~25 % more work.
__device__ __forceinline__ int snake_item(int it, int w0, int dw) {
  return it * dw + ((it & 1) ? dw - 1 - w0 : w0);
}

// Byte offset of element (row, col) inside a 128-row bf16 tile stored as
// 128-byte-swizzled atom columns of 64 elements.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col) {
  const int atom = col >> 6, chunk = (col & 63) >> 3;
  return atom * (kBM * 128) + row * 128 + ((chunk ^ (row & 7)) << 4) + ((col & 7) << 1);
}

// Rotate a 128-row tile in shared memory (NEOX pairs (i, i+HD/2)).  128
// threads: thread tid owns pairs 8p..8p+7 (p = tid % NCH) for rows
// r0, r0 + RS, ..., r0 = tid / NCH.  Angles advance by RS rows with the
// angle-addition recurrence, from an accurately reduced start per tile.  The
// two pairs held in one 32-bit bf16x2 word are processed together with
// packed FP32 (f32x2) arithmetic.
template <int HD>
struct TileRotator {
  static constexpr int NCH = HD / 16;        // 8-pair groups per row
  static constexpr int RS = 128 / NCH;       // row stride between a thread's rows
  static constexpr int ROWS = 128 / RS;      // rows per thread
  float f_hi[8], f_lo[8];
  float2 step_c[4], step_s[4];               // cos/sin of RS * f for pairs (2q, 2q+1)
  int p, r0;

  __device__ void init(int tid, const Geometry& g) {
    p = tid % NCH;
    r0 = tid / NCH;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      f_hi[e] = g.rope_f_hi[8 * p + e];
      f_lo[e] = g.rope_f_lo[8 * p + e];
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float s0, c0, s1, c1;
      __sincosf(rope_angle(RS, f_hi[2 * q], f_lo[2 * q]), &s0, &c0);
      __sincosf(rope_angle(RS, f_hi[2 * q + 1], f_lo[2 * q + 1]), &s1, &c1);
      step_c[q] = make_float2(c0, c1);
      step_s[q] = make_float2(s0, s1);
    }
  }

  __device__ void rotate(uint8_t* tile, int pos0) {
    float2 c[4], sn[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float s0, c0, s1, c1;
      __sincosf(rope_angle(pos0 + r0, f_hi[2 * q], f_lo[2 * q]), &s0, &c0);
      __sincosf(rope_angle(pos0 + r0, f_hi[2 * q + 1], f_lo[2 * q + 1]), &s1, &c1);
      c[q] = make_float2(c0, c1);
      sn[q] = make_float2(s0, s1);
    }
#pragma unroll 1
    for (int k = 0; k < ROWS; ++k) {
      const int r = r0 + k * RS;
      uint4* a_ptr = reinterpret_cast<uint4*>(tile + sw128_offset(r, 8 * p));
      uint4* b_ptr = reinterpret_cast<uint4*>(tile + sw128_offset(r, 8 * p + HD / 2));
      const uint4 a = *a_ptr, b = *b_ptr;
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
      uint32_t ya[4], yb[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // x0 = first elements of pairs (2q, 2q+1), x1 = their partners.
        const float2 x0 = make_float2(bf16_lo(av[q]), bf16_hi(av[q]));
        const float2 x1 = make_float2(bf16_lo(bv[q]), bf16_hi(bv[q]));
        const float2 ns = make_float2(-sn[q].x, -sn[q].y);
        const float2 y0 = __ffma2_rn(x0, c[q], __fmul2_rn(x1, ns));     // x0 cos - x1 sin
        const float2 y1 = __ffma2_rn(x1, c[q], __fmul2_rn(x0, sn[q]));  // x1 cos + x0 sin
        ya[q] = pack_bf16x2(y0.x, y0.y);
        yb[q] = pack_bf16x2(y1.x, y1.y);
      }
      *a_ptr = make_uint4(ya[0], ya[1], ya[2], ya[3]);
      *b_ptr = make_uint4(yb[0], yb[1], yb[2], yb[3]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // advance the angles by RS positions
        const float2 nss = make_float2(-step_s[q].x, -step_s[q].y);
        const float2 cn = __ffma2_rn(c[q], step_c[q], __fmul2_rn(sn[q], nss));
        sn[q] = __ffma2_rn(sn[q], step_c[q], __fmul2_rn(c[q], step_s[q]));
        c[q] = cn;
      }
    }
  }

  // Interleaved (GPT-J) pairs (2i, 2i+1) of "nanoeuler -- CUDA kernels",
  // rope_kernel: each bf16x2 word of the tile is one pair, rotated in place
  // (scores q . k do not depend on the element order Q and K share).  Thread
  // p owns the sixteen columns 16p .. 16p + 15, i.e. pairs 8p .. 8p + 7, the
  // same pairs (and angles) as in the NEOX layout.
  __device__ void rotate_interleaved(uint8_t* tile, int pos0) {
    float2 c[4], sn[4];   // pair 8p + e: component e & 1 of entry e >> 1
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float s0, c0, s1, c1;
      __sincosf(rope_angle(pos0 + r0, f_hi[2 * q], f_lo[2 * q]), &s0, &c0);
      __sincosf(rope_angle(pos0 + r0, f_hi[2 * q + 1], f_lo[2 * q + 1]), &s1, &c1);
      c[q] = make_float2(c0, c1);
      sn[q] = make_float2(s0, s1);
    }
#pragma unroll 1
    for (int k = 0; k < ROWS; ++k) {
      const int r = r0 + k * RS;
      uint4* a_ptr = reinterpret_cast<uint4*>(tile + sw128_offset(r, 16 * p));
      uint4* b_ptr = reinterpret_cast<uint4*>(tile + sw128_offset(r, 16 * p + 8));
      const uint4 a = *a_ptr, b = *b_ptr;
      uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float cs = (e & 1) ? c[e >> 1].y : c[e >> 1].x;
        const float ss = (e & 1) ? sn[e >> 1].y : sn[e >> 1].x;
        float y0, y1;
        rope_pair(bf16_lo(w[e]), bf16_hi(w[e]), cs, ss, y0, y1);
        w[e] = pack_bf16x2(y0, y1);
      }
      *a_ptr = make_uint4(w[0], w[1], w[2], w[3]);
      *b_ptr = make_uint4(w[4], w[5], w[6], w[7]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // advance the angles by RS positions
        const float2 nss = make_float2(-step_s[q].x, -step_s[q].y);
        const float2 cn = __ffma2_rn(c[q], step_c[q], __fmul2_rn(sn[q], nss));
        sn[q] = __ffma2_rn(sn[q], step_c[q], __fmul2_rn(c[q], step_s[q]));
        c[q] = cn;
      }
    }
  }

  __device__ void rotate_tile(uint8_t* tile, int pos0, bool interleaved) {
    if (interleaved)
      rotate_interleaved(tile, pos0);
    else
      rotate(tile, pos0);
  }
};

template <int HD, bool ROPE>
__global__ void __launch_bounds__(FwdCfg<HD, ROPE>::kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_qk, const __grid_constant__ CUtensorMap tm_v,
           const __grid_constant__ CUtensorMap tm_out, float* __restrict__ lse,
           int* __restrict__ status, Geometry g, int n_items) {
  using Cfg = FwdCfg<HD, ROPE>;
  constexpr int NK = Cfg::kKStages, NV = Cfg::kVStages, NO = Cfg::kOBuffers;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Cfg::kQOff;
  uint8_t* sK = smem + Cfg::kKOff;
  uint8_t* sV = smem + Cfg::kVOff;
  FwdBarriers* bars = reinterpret_cast<FwdBarriers*>(smem + Cfg::kBarOff);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int w0 = blockIdx.x, dw = gridDim.x;   // this CTA's items: snake_item(0..., w0, dw)

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->q_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->q_ready[i]), 4);
      ptx::mbar_init(ptx::smem_u32(&bars->q_empty[i]), 2);  // last score MMA + epilogue store
      ptx::mbar_init(ptx::smem_u32(&bars->o_free[i]), 4);
      ptx::mbar_init(ptx::smem_u32(&bars->s_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->s_free[i]), 4);
      ptx::mbar_init(ptx::smem_u32(&bars->p_full[i]), 4);
      ptx::mbar_init(ptx::smem_u32(&bars->pv_done[i]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->drain), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->drain2), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->o_staged), 4);
    for (int i = 0; i < NK; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->k_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->k_ready[i]), 4);
      ptx::mbar_init(ptx::smem_u32(&bars->k_empty[i]), 1);
    }
    for (int i = 0; i < NV; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->v_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->v_empty[i]), 1);
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
  // A following backward prologue may get resident now; it waits for this
  // grid to complete before reading out.
  ptx::grid_dep_launch();

  auto fail = [&]() {
    *abort_flag = 1;
    record_status(status, kErrDeviceTimeout);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_qk);
      ptx::tma_prefetch_desc(&tm_v);
      int k_issued = 0, v_issued = 0, q_issued = 0;  // global sequence counters
      bool ok = true;
      for (int it = 0, w = w0; w < n_items && ok; ++it, w = snake_item(it, w0, dw)) {
        const FwdItem item = fwd_item(w, g);
        const int n_kv = item.qt + 1;
        const int k_col = g.C + item.kh * HD, v_col = g.C + g.NKV * HD + item.kh * HD;
        // Q of this item into buffer it & 1 once item it-2 issued its last S.
        const int qb = it & 1;
        if (it >= 2 && !ptx::mbar_wait(ptx::smem_u32(&bars->q_empty[qb]), ((it >> 1) - 1) & 1, abort_flag,
                                       kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint32_t qf = ptx::smem_u32(&bars->q_full[qb]);
        ptx::mbar_arrive_expect_tx(qf, Cfg::kTileBytes);
#pragma unroll
        for (int a = 0; a < HD / 64; ++a)
          ptx::tma_load_3d(ptx::smem_u32(sQ + qb * Cfg::kTileBytes + a * Cfg::kAtomBytes), &tm_qk,
                           item.h * HD + 64 * a, item.qt * kBM, item.b, qf);
        q_issued = it + 1;
        const int kbase = k_issued;  // global index of this item's key tile 0
        auto load_k = [&](int j) -> bool {
          const int gi = kbase + j, st = gi % NK, u = gi / NK;
          if (u > 0 && !ptx::mbar_wait(ptx::smem_u32(&bars->k_empty[st]), (u - 1) & 1, abort_flag, kWaitLimitNs))
            return false;
          const uint32_t kf = ptx::smem_u32(&bars->k_full[st]);
          ptx::mbar_arrive_expect_tx(kf, Cfg::kTileBytes);
#pragma unroll
          for (int a = 0; a < HD / 64; ++a)
            ptx::tma_load_3d(ptx::smem_u32(sK + st * Cfg::kTileBytes + a * Cfg::kAtomBytes), &tm_qk,
                             k_col + 64 * a, j * kBN, item.b, kf);
          k_issued = gi + 1;
          return true;
        };
        auto load_v = [&](int j) -> bool {
          const int gi = kbase + j, st = gi % NV, u = gi / NV;
          if (u > 0 && !ptx::mbar_wait(ptx::smem_u32(&bars->v_empty[st]), (u - 1) & 1, abort_flag, kWaitLimitNs))
            return false;
          const uint32_t vf = ptx::smem_u32(&bars->v_full[st]);
          ptx::mbar_arrive_expect_tx(vf, Cfg::kTileBytes);
#pragma unroll
          for (int a = 0; a < HD / 64; ++a)
            ptx::tma_load_3d(ptx::smem_u32(sV + st * Cfg::kTileBytes + a * Cfg::kAtomBytes), &tm_v,
                             v_col + 64 * a, j * kBN, item.b, vf);
          v_issued = gi + 1;
          return true;
        };
        // Issue order within an item: K_0, K_1, then V_j, K_{j+2}.
        for (int j = 0; j < 2 && j < n_kv && ok; ++j) ok = load_k(j);
        for (int j = 0; j < n_kv && ok; ++j) {
          ok = load_v(j);
          if (ok && j + 2 < n_kv) ok = load_k(j + 2);
        }
      }
      if (!ok) fail();
      if (*abort_flag) {
        // Let every copy already in flight land before shared memory is released.
        for (int qb = 0; qb < 2 && qb < q_issued; ++qb)
          ptx::mbar_wait(ptx::smem_u32(&bars->q_full[qb]), ((q_issued - 1 - qb) >> 1) & 1, nullptr, kWaitLimitNs);
        for (int st = 0; st < NK && st < k_issued; ++st)
          ptx::mbar_wait(ptx::smem_u32(&bars->k_full[st]), ((k_issued - 1 - st) / NK) & 1, nullptr, kWaitLimitNs);
        for (int st = 0; st < NV && st < v_issued; ++st)
          ptx::mbar_wait(ptx::smem_u32(&bars->v_full[st]), ((v_issued - 1 - st) / NV) & 1, nullptr, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ score-MMA issuer
    // (the whole warp runs the issue loop; one elected lane issues each MMA
    // and commit, and every wait is warp-collective)
    {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(kBM, kBN, false, false);
      const uint64_t dQ = ptx::sw128_desc(ptx::smem_u32(sQ), 16, 1024);
      const uint64_t dK = ptx::sw128_desc(ptx::smem_u32(sK), 16, 1024);
      bool ok = true;
      int gi = 0;  // global key-tile index of this CTA's stream
      for (int it = 0, w = w0; w < n_items && ok; ++it, w = snake_item(it, w0, dw)) {
        const FwdItem item = fwd_item(w, g);
        const int n_kv = item.qt + 1, qb = it & 1;
        ok = ptx::mbar_wait_all(ptx::smem_u32(ROPE ? &bars->q_ready[qb] : &bars->q_full[qb]), (it >> 1) & 1, abort_flag,
                            kWaitLimitNs);
        for (int j = 0; j < n_kv && ok; ++j, ++gi) {
          const int s = gi % NK, sb = gi & 1;
          const uint32_t kb = ptx::smem_u32(ROPE ? &bars->k_ready[s] : &bars->k_full[s]);
          const uint32_t fb = ptx::smem_u32(&bars->s_free[sb]);
          // K_j landed (and rotated); score buffer sb read out by the softmax of tile gi-2.
          if (!(ptx::mbar_ready(kb, (gi / NK) & 1) & (gi < 2 ? 1u : ptx::mbar_ready(fb, ((gi >> 1) - 1) & 1)))) {
            ok = ptx::mbar_wait_all(kb, (gi / NK) & 1, abort_flag, kWaitLimitNs);
            if (ok && gi >= 2) ok = ptx::mbar_wait_all(fb, ((gi >> 1) - 1) & 1, abort_flag, kWaitLimitNs);
            if (!ok) break;
          }
          ptx::tc_fence_after();
          const uint64_t bk = ptx::desc_advance(dK, s * Cfg::kTileBytes);
          const uint64_t aq = ptx::desc_advance(dQ, qb * Cfg::kTileBytes);
          const uint32_t d_s = tmem + (sb ? Cfg::kTmemS1 : Cfg::kTmemS0);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * Cfg::kAtomBytes + (kk & 3) * 32;
            ptx::mma_bf16_ss_w(d_s, ptx::desc_advance(aq, off), ptx::desc_advance(bk, off), idesc_s, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit_w(ptx::smem_u32(&bars->s_full[sb]));
          ptx::mma_commit_w(ptx::smem_u32(&bars->k_empty[s]));
          if (j == n_kv - 1) ptx::mma_commit_w(ptx::smem_u32(&bars->q_empty[qb]));
        }
      }
      if (!ok) fail();
      // Drain: every MMA this thread issued has finished before TMEM is freed.
      ptx::mma_commit_w(ptx::smem_u32(&bars->drain));
      ptx::mbar_wait_all(ptx::smem_u32(&bars->drain), 0, nullptr, kWaitLimitNs);
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ PV-MMA issuer
    // (the whole warp runs the issue loop; one elected lane issues each MMA
    // and commit, and every wait is warp-collective)
    {
      constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(kBM, HD, false, true);
      const uint64_t dV = ptx::sw128_desc(ptx::smem_u32(sV), Cfg::kAtomBytes, 1024);
      bool ok = true;
      int gi = 0;
      for (int it = 0, w = w0; w < n_items && ok; ++it, w = snake_item(it, w0, dw)) {
        const FwdItem item = fwd_item(w, g);
        const int n_kv = item.qt + 1, ob = (NO == 2) ? (it & 1) : 0;
        // The first PV of an item overwrites its O buffer: the epilogue of the
        // item that last used it must have read it out.
        if (it >= NO)
          ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->o_free[ob]), (((it - NO) / NO)) & 1, abort_flag, kWaitLimitNs);
        for (int j = 0; j < n_kv && ok; ++j, ++gi) {
          const int pb = gi & 1, sp = gi % NV;
          const uint32_t pf = ptx::smem_u32(&bars->p_full[pb]), vf = ptx::smem_u32(&bars->v_full[sp]);
          if (!(ptx::mbar_ready(pf, (gi >> 1) & 1) & ptx::mbar_ready(vf, (gi / NV) & 1))) {
            ok = ptx::mbar_wait_all(pf, (gi >> 1) & 1, abort_flag, kWaitLimitNs);
            if (ok) ok = ptx::mbar_wait_all(vf, (gi / NV) & 1, abort_flag, kWaitLimitNs);
            if (!ok) break;
          }
          ptx::tc_fence_after();
          const uint64_t bv = ptx::desc_advance(dV, sp * Cfg::kTileBytes);
          const uint32_t d_o = tmem + (ob ? Cfg::kTmemO1 : Cfg::kTmemO0);
          const uint32_t a_p = tmem + (pb ? Cfg::kTmemP1 : Cfg::kTmemP0);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            ptx::mma_bf16_ts_w(d_o, a_p + kk * 8, ptx::desc_advance(bv, kk * 2048), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit_w(ptx::smem_u32(&bars->pv_done[pb]));
          ptx::mma_commit_w(ptx::smem_u32(&bars->v_empty[sp]));
        }
      }
      if (!ok) fail();
      ptx::mma_commit_w(ptx::smem_u32(&bars->drain2));
      ptx::mbar_wait_all(ptx::smem_u32(&bars->drain2), 0, nullptr, kWaitLimitNs);
    }
  } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = g.scale * 1.4426950408889634f;  // scale * log2(e)
    bool ok = true;
    int gi = 0;
    for (int it = 0, w = w0; w < n_items && ok; ++it, w = snake_item(it, w0, dw)) {
      const FwdItem item = fwd_item(w, g);
      const int n_kv = item.qt + 1;
      const int tq = item.qt * kBM + row;
      const int ob = (NO == 2) ? (it & 1) : 0;
      const uint32_t o_addr = t_lane + (ob ? Cfg::kTmemO1 : Cfg::kTmemO0);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n_kv; ++j, ++gi) {
        const int sb = gi & 1;
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->s_full[sb]), (gi >> 1) & 1, abort_flag,
                                                      kWaitLimitNs));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sr[kBN];
        const uint32_t s_addr = t_lane + (sb ? Cfg::kTmemS1 : Cfg::kTmemS0);
        ptx::tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        ptx::tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        ptx::tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
        ptx::tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->s_free[sb]));
        // Non-blocking checks issued now and consumed after the math: P
        // buffer gi&1 was read by PV(gi-2); O may be rescaled only once
        // PV(gi-1) (same item) has finished.
        const int pb = gi & 1;
        const uint32_t pfree_now = gi < 2 ? 1u : ptx::mbar_test(ptx::smem_u32(&bars->pv_done[pb]), ((gi - 2) >> 1) & 1);
        const uint32_t prev_now =
            j < 1 ? 1u : ptx::mbar_test(ptx::smem_u32(&bars->pv_done[pb ^ 1]), ((gi - 1) >> 1) & 1);

        if (j == n_kv - 1) {  // diagonal tile: key c is visible to row `row` iff c <= row
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c > row) sr[c] = __float_as_uint(-INFINITY);
        }
        // Row max with 4 independent partial maxima (no 128-long dependency chain).
        float mx[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) mx[k] = __uint_as_float(sr[k]);
#pragma unroll
        for (int c = 4; c < kBN; c += 4)
#pragma unroll
          for (int k = 0; k < 4; ++k) mx[k] = fmaxf(mx[k], __uint_as_float(sr[c + k]));
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        const float m_cand = mt * sl2;
        const bool grow = m_cand > m + kRescaleThreshold;   // always true on an item's first tile
        const float m_new = grow ? m_cand : m;
        const float corr = grow ? ptx::ex2_approx(m - m_new) : 1.f;
        // p = 2^(s * scale * log2(e) - m): exponent arguments two at a time
        // (packed FMA), row sum in 4 independent partial sums (packed adds).
        const float2 sl2x2 = make_float2(sl2, sl2), negm2 = make_float2(-m_new, -m_new);
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < kBN; c += 2) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2, negm2);
          const float2 p = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
          sr[c] = __float_as_uint(p.x);
          sr[c + 1] = __float_as_uint(p.y);
          acc[(c >> 1) & 1] = __fadd2_rn(acc[(c >> 1) & 1], p);
        }
        const float2 acc2 = __fadd2_rn(acc[0], acc[1]);
        const float rs = acc2.x + acc2.y;
        l = l * corr + rs;
        m = m_new;

        const bool rescale = (j >= 1) && __any_sync(0xffffffffu, grow);
        if (!__all_sync(0xffffffffu, pfree_now)) {
          ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->pv_done[pb]), ((gi - 2) >> 1) & 1,
                                                        abort_flag, kWaitLimitNs));
          if (!ok) break;
        }
        ptx::tc_fence_after();
        // P (bf16, two keys per 32-bit column) into TMEM P buffer pb.  Packed
        // first, so that the 128 score registers are dead before the O rescale
        // below needs its own 32.
        {
          const uint32_t p_addr = t_lane + (pb ? Cfg::kTmemP1 : Cfg::kTmemP0);
          uint32_t pw[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) pw[c] = pack_bf16x2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1]));
          ptx::tmem_st32(p_addr, pw);
#pragma unroll
          for (int c = 0; c < 32; ++c)
            pw[c] = pack_bf16x2(__uint_as_float(sr[64 + 2 * c]), __uint_as_float(sr[64 + 2 * c + 1]));
          ptx::tmem_st32(p_addr + 32, pw);
        }
        if (rescale) {
          if (!__all_sync(0xffffffffu, prev_now)) {
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->pv_done[pb ^ 1]), ((gi - 1) >> 1) & 1,
                                                          abort_flag, kWaitLimitNs));
            if (!ok) break;
          }
          ptx::tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < HD; c0 += 32) {
            uint32_t o[32];
            ptx::tmem_ld32(o_addr + c0, o);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * corr);
            ptx::tmem_st32(o_addr + c0, o);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->p_full[pb]));
      }
      if (!ok) break;
      // Epilogue of this item: O is complete once its last PV has finished.
      // out = O / l is staged in this item's Q buffer (every score MMA of the
      // item has completed) in the tensor-map layout and written with TMA
      // stores (rows past T are clipped), instead of one scattered 16-byte
      // store per thread and chunk.
      const int last = gi - 1;
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->pv_done[last & 1]), (last >> 1) & 1,
                                                    abort_flag, kWaitLimitNs));
      if (!ok) break;
      ptx::tc_fence_after();
      const float inv_l = 1.f / l;
      uint8_t* stile = sQ + (it & 1) * Cfg::kTileBytes;
#pragma unroll 1
      for (int c0 = 0; c0 < HD; c0 += 32) {
        uint32_t o[32];
        ptx::tmem_ld32(o_addr + c0, o);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 w4 = make_uint4(
              pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l),
              pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l),
              pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l),
              pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l));
          *reinterpret_cast<uint4*>(stile + sw128_offset(row, c0 + 8 * v)) = w4;
        }
      }
      ptx::tc_fence_before();
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(ptx::smem_u32(&bars->o_free[ob]));
        ptx::mbar_arrive(ptx::smem_u32(&bars->o_staged));
      }
      if (tq < g.T) lse[((size_t)item.b * g.NH + item.h) * g.T + tq] = (m + log2f(l)) * 0.6931471805599453f;
      if (warp == kSoftmaxWarp0 && lane == 0) {
        // All four warps staged their rows: store the tile, and release the
        // Q buffer once the TMA engine has read it.
        if (ptx::mbar_wait(ptx::smem_u32(&bars->o_staged), it & 1, abort_flag, kWaitLimitNs)) {
#pragma unroll
          for (int a = 0; a < HD / 64; ++a)
            ptx::tma_store_3d(&tm_out, ptx::smem_u32(stile + a * Cfg::kAtomBytes), item.h * HD + 64 * a,
                              item.qt * kBM, item.b);
          ptx::bulk_commit();
          ptx::bulk_wait_read();
        } else {
          fail();
        }
        ptx::mbar_arrive(ptx::smem_u32(&bars->q_empty[it & 1]));
      }
    }
    // Every tile store has landed in global memory before the CTA exits.
    if (warp == kSoftmaxWarp0 && lane == 0) ptx::bulk_wait();
    if (!ok) fail();
  } else if (ROPE && warp >= kRopeWarp0) {
    // ------------------------------------------------------------ RoPE transform
    const int tid = threadIdx.x - kRopeWarp0 * 32;
    TileRotator<HD> rot;
    rot.init(tid, g);
    bool ok = true;
    int gi = 0;
    for (int it = 0, w = w0; w < n_items && ok; ++it, w = snake_item(it, w0, dw)) {
      const FwdItem item = fwd_item(w, g);
      const int qb = it & 1;
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->q_full[qb]), (it >> 1) & 1, abort_flag,
                                                    kWaitLimitNs));
      if (!ok) break;
      rot.rotate_tile(sQ + qb * Cfg::kTileBytes, item.qt * kBM, g.rope_interleaved != 0);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->q_ready[qb]));
      for (int j = 0; j <= item.qt && ok; ++j, ++gi) {
        const int s = gi % NK;
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->k_full[s]), (gi / NK) & 1, abort_flag,
                                                      kWaitLimitNs));
        if (!ok) break;
        rot.rotate_tile(sK + s * Cfg::kTileBytes, j * kBN, g.rope_interleaved != 0);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->k_ready[s]));
      }
    }
    if (!ok) fail();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

template <int HD, bool ROPE>
cudaError_t launch_fwd(const Tc05FwdArgs& a, cudaStream_t stream) {
  using Cfg = FwdCfg<HD, ROPE>;
  auto kern = fwd_kernel<HD, ROPE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_qt = (a.g.T + kBM - 1) / kBM;
  const int n_items = n_qt * a.g.B * a.g.NH;
  const unsigned grid = (unsigned)(n_items < a.num_sms ? n_items : a.num_sms);
  prof_begin(kKernelFwdTc05, stream);
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(a.tm_qk, a.tm_v, a.tm_out, a.lse, a.status, a.g, n_items);
  prof_end(kKernelFwdTc05, stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc05_fwd_launch(const Tc05FwdArgs& a, cudaStream_t stream) {
  const bool rope = a.g.rope_theta > 0.f && !a.pre_rotated;
  if (!rope && tc05_fwd2_supported(a.g)) return tc05_fwd2_launch(a, stream);
  if (a.g.hd == 128) return rope ? launch_fwd<128, true>(a, stream) : launch_fwd<128, false>(a, stream);
  if (a.g.hd == 64) return rope ? launch_fwd<64, true>(a, stream) : launch_fwd<64, false>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
