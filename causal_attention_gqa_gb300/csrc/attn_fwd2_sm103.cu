// Causal GQA attention forward on sm_103a tensor cores for two query heads
// per work item (bf16 in, f32 accumulation): head size 128 with two query
// heads of one kv head (they read the same K/V tiles), or head size 64 with
// any two query heads (sharing K/V tiles when they share a kv head, else
// each brings its own K/V tiles into the same ring stage).
//
// Persistent kernel: one CTA per SM walks its share of a list of work items
// (dealt back and forth across the CTAs), one item = a 128-query tile of two
// query heads 2p, 2p+1 of one batch row (with a shared kv head every K/V
// tile loaded feeds two score and two PV MMAs), heaviest (longest causal key
// range) first.  Two softmax warpgroups, one per query head, work
// in ping-pong: while group A turns S_A(j) into P_A(j), the tensor core runs
// PV_B(j-1) and S_B(j), and the other way round, so neither the tensor core
// nor the softmax waits for the other as long as one tile's softmax takes
// less than two tiles' MMAs.  Warp roles:
//   warp 0      TMA producer: both Q tiles of an item, then K_j and V_j (of
//               one kv head, or of both heads' kv heads) together into a
//               two-stage ring (one barrier per key tile).
//   warp 1      TMEM owner and the single MMA issuer, in the order
//               S_A(0), S_B(0), then per key tile PV_A(j), S_A(j+1), PV_B(j),
//               S_B(j+1).
//   warps 2-5   softmax of head 2p (group A), warps 6-9 of head 2p+1 (group
//               B): thread = query row = TMEM lane.  Reads S(j), keeps the
//               running max m and sum l, writes P(j) (bf16 pairs) into TMEM
//               over the score columns it has read, rescales O in TMEM when m
//               grows past a threshold (exact: l and O share the stale max),
//               and at the end of an item writes out = O / l (staged in shared
//               memory, TMA store) and lse = m + ln l.
// TMEM columns: S_A, S_B (128 each), O_A, O_B (128 each, of which the head
// size is used).  P(j) overwrites
// S(j) and the next score MMA into the same columns is issued after the PV
// MMA that reads P(j): MMAs issued by one thread execute in order.
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

constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr float kRescaleThreshold = 8.0f;     // log2 units: P may reach 2^8 before O is rescaled
constexpr int kThreads = 320;

// SHARED: the two heads of an item read one kv head's K/V tiles; else each
// ring stage holds K_A, K_B (and V_A, V_B).
template <int HD, bool SHARED>
struct Fwd2Cfg {
  static constexpr int kAtom = 128 * 128;               // 128 rows x one 128-byte swizzle-atom column
  static constexpr int kTileBytes = 128 * HD * 2;       // Q / K / V / output tile
  static constexpr int kKT = SHARED ? 1 : 2;            // K (and V) tiles per ring stage
  static constexpr int kStageBytes = kKT * kTileBytes;
  static constexpr int kKStages = 2, kVStages = 2;
  static constexpr int kQOff = 0;                       // Q_A, Q_B
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kStageBytes;
  static constexpr int kStOff = kVOff + kVStages * kStageBytes;   // output staging tile
  static constexpr int kBarOff = kStOff + kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;
  static_assert(kSmemBytes <= 232448, "paired forward kernel exceeds the 227 KB shared-memory limit");
};

__device__ __forceinline__ uint32_t tmem_s(int x) { return 128u * (uint32_t)x; }
__device__ __forceinline__ uint32_t tmem_o(int x) { return 256u + 128u * (uint32_t)x; }

struct Fwd2Barriers {
  uint64_t q_full, q_empty;
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t staged[2], stage_free, drain;
  uint32_t tmem_base;
  int abort;
};

// Work item w -> (batch row, head pair, query tile); heaviest first.
struct Fwd2Item {
  int b, h0, kh, qt;
};
__device__ __forceinline__ Fwd2Item fwd2_item(int w, const Geometry& g) {
  const int n_qt = (g.T + 127) / 128, pairs = g.NH / 2, bp_count = g.B * pairs;
  Fwd2Item it;
  it.qt = n_qt - 1 - w / bp_count;
  const int bp = w % bp_count;
  it.b = bp / pairs;
  it.h0 = 2 * (bp % pairs);
  it.kh = it.h0 / g.grp;
  return it;
}

// The it-th item of CTA w0 in a grid of dw CTAs, dealt forward in even rounds
// and backward in odd ones, which balances the per-CTA totals of a list
// sorted by decreasing weight.
__device__ __forceinline__ int snake(int it, int w0, int dw) { return it * dw + ((it & 1) ? dw - 1 - w0 : w0); }

// Byte offset of the 16-byte chunk holding columns col..col+7 of row `row` in
// a 128-row bf16 tile of 128-byte-swizzled 64-column atoms.
__device__ __forceinline__ uint32_t sw128_chunk(int row, int col) {
  return (uint32_t)((col >> 6) * (128 * 128) + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4));
}

template <int HD, bool SHARED>
__global__ void __launch_bounds__(kThreads, 1)
fwd2_kernel(const __grid_constant__ CUtensorMap tm_qk, const __grid_constant__ CUtensorMap tm_v,
            const __grid_constant__ CUtensorMap tm_out, float* __restrict__ lse, int* __restrict__ status, Geometry g,
            int n_items) {
  using Cfg = Fwd2Cfg<HD, SHARED>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Cfg::kQOff;
  uint8_t* sK = smem + Cfg::kKOff;
  uint8_t* sV = smem + Cfg::kVOff;
  uint8_t* sSt = smem + Cfg::kStOff;
  Fwd2Barriers* bars = reinterpret_cast<Fwd2Barriers*>(smem + Cfg::kBarOff);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int w0 = blockIdx.x, dw = gridDim.x;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->q_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->q_empty), 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->kv_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->kv_empty[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->s_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->p_full[i]), 4);
      ptx::mbar_init(ptx::smem_u32(&bars->o_done[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->o_free[i]), 4);
      ptx::mbar_init(ptx::smem_u32(&bars->staged[i]), 4);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->stage_free), 1);
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
  // Launched as a programmatic dependent of the preceding kernel (the Q/K
  // rotation pass of attn_fwd_ws): the set-up above overlapped its tail;
  // wait for it to complete before reading or writing global memory.  A
  // following backward prologue may get resident now; it waits for this grid
  // to complete before reading out.
  ptx::grid_dep_wait();
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
      int kv_issued = 0, q_issued = 0;   // global sequence counters
      bool ok = true;
      for (int it = 0, w = w0; w < n_items && ok; ++it, w = snake(it, w0, dw)) {
        const Fwd2Item item = fwd2_item(w, g);
        const int n_kv = item.qt + 1;
        // kv heads of the item's two query heads (the same one when SHARED)
        const int kh2[2] = {item.h0 / g.grp, (item.h0 + 1) / g.grp};
        if (it >= 1 && !(ok = ptx::mbar_wait(ptx::smem_u32(&bars->q_empty), (it - 1) & 1, abort_flag, kWaitLimitNs)))
          break;
        const uint32_t qf = ptx::smem_u32(&bars->q_full);
        ptx::mbar_arrive_expect_tx(qf, 2 * Cfg::kTileBytes);
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int a = 0; a < HD / 64; ++a)
            ptx::tma_load_3d(ptx::smem_u32(sQ + x * Cfg::kTileBytes + a * Cfg::kAtom), &tm_qk,
                             (item.h0 + x) * HD + 64 * a, item.qt * 128, item.b, qf);
        q_issued = it + 1;
        // K_j and V_j into one ring stage with one barrier (each barrier the
        // MMA issuer checks stalls the tensor pipe).
        for (int j = 0; j < n_kv && ok; ++j) {
          const int gk = kv_issued, st = gk % 2;
          if (gk >= 2 && !(ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_empty[st]), ((gk >> 1) - 1) & 1, abort_flag,
                                               kWaitLimitNs)))
            break;
          const uint32_t kvf = ptx::smem_u32(&bars->kv_full[st]);
          ptx::mbar_arrive_expect_tx(kvf, 2 * Cfg::kStageBytes);
#pragma unroll
          for (int y = 0; y < Cfg::kKT; ++y) {
            const int k_col = g.C + kh2[y] * HD, v_col = g.C + g.NKV * HD + kh2[y] * HD;
            const int off = st * Cfg::kStageBytes + y * Cfg::kTileBytes;
#pragma unroll
            for (int a = 0; a < HD / 64; ++a) {
              ptx::tma_load_3d(ptx::smem_u32(sK + off + a * Cfg::kAtom), &tm_qk, k_col + 64 * a, j * 128, item.b,
                               kvf);
              ptx::tma_load_3d(ptx::smem_u32(sV + off + a * Cfg::kAtom), &tm_v, v_col + 64 * a, j * 128, item.b,
                               kvf);
            }
          }
          kv_issued = gk + 1;
        }
      }
      if (!ok) fail();
      if (*abort_flag) {
        // Let every copy already in flight land before shared memory is released.
        if (q_issued > 0) ptx::mbar_wait(ptx::smem_u32(&bars->q_full), (q_issued - 1) & 1, nullptr, kWaitLimitNs);
        for (int st = 0; st < 2 && st < kv_issued; ++st)
          ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[st]), ((kv_issued - 1 - st) >> 1) & 1, nullptr, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp runs the issue loop; one elected lane issues each MMA
    // and commit, and every wait is warp-collective)
    {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(128, HD, false, true);
      const uint64_t dQ = ptx::sw128_desc(ptx::smem_u32(sQ), 16, 1024);
      const uint64_t dK = ptx::sw128_desc(ptx::smem_u32(sK), 16, 1024);
      const uint64_t dV = ptx::sw128_desc(ptx::smem_u32(sV), Cfg::kAtom, 1024);
      bool ok = true;
      // S_x(g) = Q_x K_g^T into the score columns of group x.
      auto issue_s = [&](int x, int gk) {
        const uint64_t bk = ptx::desc_advance(dK, (gk % 2) * Cfg::kStageBytes + (SHARED ? 0 : x) * Cfg::kTileBytes);
        const uint64_t aq = ptx::desc_advance(dQ, x * Cfg::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Cfg::kAtom + (kk & 3) * 32;
          ptx::mma_bf16_ss_w(tmem + tmem_s(x), ptx::desc_advance(aq, off), ptx::desc_advance(bk, off), idesc_s,
                           kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit_w(ptx::smem_u32(&bars->s_full[x]));
      };
      // O_x += P_x(g) V_g with P from TMEM.
      auto issue_pv = [&](int x, int gk, bool first) {
        const uint64_t bv = ptx::desc_advance(dV, (gk % 2) * Cfg::kStageBytes + (SHARED ? 0 : x) * Cfg::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk)
          ptx::mma_bf16_ts_w(tmem + tmem_o(x), tmem + tmem_s(x) + kk * 8, ptx::desc_advance(bv, kk * 2048), idesc_o,
                           (!first || kk > 0) ? 1u : 0u);
      };
      int g0 = 0;   // global index of the item's first key tile
      for (int it = 0, w = w0; w < n_items && ok; ++it, w = snake(it, w0, dw)) {
        const Fwd2Item item = fwd2_item(w, g);
        const int n_kv = item.qt + 1;
        ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->q_full), it & 1, abort_flag, kWaitLimitNs) &&
             ptx::mbar_wait_all(ptx::smem_u32(&bars->kv_full[g0 % 2]), (g0 >> 1) & 1, abort_flag, kWaitLimitNs);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_s(0, g0);
        issue_s(1, g0);
        if (n_kv == 1) ptx::mma_commit_w(ptx::smem_u32(&bars->q_empty));
        for (int j = 0; j < n_kv && ok; ++j) {
          const int gk = g0 + j;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            // PV_x(j) once group x wrote P_x(j) and V_j landed; the item's
            // first PV overwrites O_x, which the previous item's epilogue
            // must have read.
            // (V_j landed with K_j, checked before the score MMAs.)
            ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->p_full[x]), gk & 1, abort_flag, kWaitLimitNs);
            if (ok && j == 0 && it >= 1)
              ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->o_free[x]), (it - 1) & 1, abort_flag, kWaitLimitNs);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_pv(x, gk, j == 0);
            if (x == 1) ptx::mma_commit_w(ptx::smem_u32(&bars->kv_empty[gk % 2]));   // last reader of K_j, V_j
            if (j == n_kv - 1) ptx::mma_commit_w(ptx::smem_u32(&bars->o_done[x]));
            // S_x(j+1) after PV_x(j): it overwrites P_x(j).
            if (j + 1 < n_kv) {
              if (x == 0 &&
                  !(ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->kv_full[(gk + 1) % 2]), ((gk + 1) >> 1) & 1,
                                        abort_flag, kWaitLimitNs)))
                break;
              ptx::tc_fence_after();
              issue_s(x, gk + 1);
              if (x == 1 && j + 1 == n_kv - 1) ptx::mma_commit_w(ptx::smem_u32(&bars->q_empty));
            }
          }
        }
        g0 += n_kv;
      }
      if (!ok) fail();
      // Drain: every MMA this thread issued has finished before TMEM is freed.
      ptx::mma_commit_w(ptx::smem_u32(&bars->drain));
      ptx::mbar_wait_all(ptx::smem_u32(&bars->drain), 0, nullptr, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int x = (warp - 2) >> 2;               // 0: head 2p, 1: head 2p+1
    const int quarter = warp & 3;                // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_addr = t_lane + tmem_s(x), o_addr = t_lane + tmem_o(x);
    const float sl2 = g.scale * 1.4426950408889634f;  // scale * log2(e)
    const bool storer = (warp & 3) == 2 && lane == 0;  // first warp of the group
    bool ok = true;
    int gk = 0;
    for (int it = 0, w = w0; w < n_items && ok; ++it, w = snake(it, w0, dw)) {
      const Fwd2Item item = fwd2_item(w, g);
      const int n_kv = item.qt + 1;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n_kv; ++j, ++gk) {
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->s_full[x]), gk & 1, abort_flag,
                                                      kWaitLimitNs));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sr[128];
        ptx::tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        ptx::tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        ptx::tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
        ptx::tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
        ptx::tmem_wait_ld();
        if (j == n_kv - 1) {  // diagonal tile: key c is visible to row `row` iff c <= row
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > row) sr[c] = __float_as_uint(-INFINITY);
        }
        // Row max with 4 independent partial maxima.
        float mx[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) mx[k] = __uint_as_float(sr[k]);
#pragma unroll
        for (int c = 4; c < 128; c += 4)
#pragma unroll
          for (int k = 0; k < 4; ++k) mx[k] = fmaxf(mx[k], __uint_as_float(sr[c + k]));
        const float m_cand = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
        const bool grow = m_cand > m + kRescaleThreshold;   // always true on an item's first tile
        const float m_new = grow ? m_cand : m;
        const float corr = grow ? ptx::ex2_approx(m - m_new) : 1.f;
        // p = 2^(s * scale * log2(e) - m), packed to bf16 pairs and written
        // over the score columns 16 at a time (columns 16h.. hold keys 32h..,
        // already read); row sum in 4 partial sums.
        const float2 sl2x2 = make_float2(sl2, sl2), negm2 = make_float2(-m_new, -m_new);
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t pw[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const int cc = 32 * h + c;
            const float2 xv = __ffma2_rn(make_float2(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])), sl2x2,
                                         negm2);
            const float2 p = make_float2(ptx::ex2_approx(xv.x), ptx::ex2_approx(xv.y));
            acc[(c >> 1) & 1] = __fadd2_rn(acc[(c >> 1) & 1], p);
            pw[c >> 1] = pack_bf16x2(p.x, p.y);
          }
          ptx::tmem_st16(s_addr + 16 * h, pw);
        }
        const float2 acc2 = __fadd2_rn(acc[0], acc[1]);
        l = l * corr + (acc2.x + acc2.y);
        m = m_new;
        // O_x is idle here: PV_x(j-1) was issued before S_x(j), whose
        // completion this group waited for.
        if ((j >= 1) && __any_sync(0xffffffffu, grow)) {
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
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->p_full[x]));
      }
      if (!ok) break;
      // ---- Epilogue of this item: out = O / l staged in shared memory (one
      // tile shared by the two groups, A then B) and written with TMA stores
      // (rows past T are clipped); lse = m + ln l.
      const int use = 2 * it + x;                // global use index of the staging tile
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->o_done[x]), it & 1, abort_flag, kWaitLimitNs));
      if (ok && use > 0)
        ok = __all_sync(0xffffffffu,
                        ptx::mbar_wait(ptx::smem_u32(&bars->stage_free), (use - 1) & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      ptx::tc_fence_after();
      const float inv_l = 1.f / l;
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
          *reinterpret_cast<uint4*>(sSt + sw128_chunk(row, c0 + 8 * v)) = w4;
        }
      }
      ptx::tc_fence_before();
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(ptx::smem_u32(&bars->o_free[x]));
        ptx::mbar_arrive(ptx::smem_u32(&bars->staged[x]));
      }
      const int tq = item.qt * 128 + row;
      if (tq < g.T) lse[((size_t)item.b * g.NH + item.h0 + x) * g.T + tq] = (m + log2f(l)) * 0.6931471805599453f;
      if (storer) {
        // All four warps staged their rows: store the tile, and release the
        // staging tile once the TMA engine has read it.
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->staged[x]), it & 1, abort_flag, kWaitLimitNs);
        if (ok) {
#pragma unroll
          for (int a = 0; a < HD / 64; ++a)
            ptx::tma_store_3d(&tm_out, ptx::smem_u32(sSt + a * Cfg::kAtom), (item.h0 + x) * HD + 64 * a,
                              item.qt * 128, item.b);
          ptx::bulk_commit();
          ptx::bulk_wait_read();
          ptx::mbar_arrive(ptx::smem_u32(&bars->stage_free));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (!ok) fail();
    // Every tile store has landed in global memory before the CTA exits.
    if (storer) ptx::bulk_wait();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool tc05_fwd2_supported(const Geometry& g) {
  return (g.hd == 128 && g.grp % 2 == 0) || (g.hd == 64 && g.NH % 2 == 0);
}

namespace {
template <int HD, bool SHARED>
cudaError_t launch_fwd2(const Tc05FwdArgs& a, cudaStream_t stream) {
  using Cfg = Fwd2Cfg<HD, SHARED>;
  auto kern = fwd2_kernel<HD, SHARED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_qt = (a.g.T + 127) / 128;
  const int n_items = n_qt * a.g.B * (a.g.NH / 2);
  const unsigned grid = (unsigned)(n_items < a.num_sms ? n_items : a.num_sms);
  prof_begin(kKernelFwdTc05, stream);
  e = launch_pdl(kern, dim3(grid), dim3(kThreads), Cfg::kSmemBytes, stream, a.tm_qk, a.tm_v, a.tm_out, a.lse,
                 a.status, a.g, n_items);
  prof_end(kKernelFwdTc05, stream);
  return e;
}
}  // namespace

cudaError_t tc05_fwd2_launch(const Tc05FwdArgs& a, cudaStream_t stream) {
  if (a.g.hd == 128 && a.g.grp % 2 == 0) return launch_fwd2<128, true>(a, stream);
  if (a.g.hd == 64) return a.g.grp % 2 == 0 ? launch_fwd2<64, true>(a, stream) : launch_fwd2<64, false>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
