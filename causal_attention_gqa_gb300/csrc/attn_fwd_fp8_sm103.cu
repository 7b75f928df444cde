// Causal GQA attention forward with e4m3 (FP8) operands on sm_103a tensor
// cores: two query heads that share a kv head, head size 128, bf16 in and out.
//
// The structure is that of the paired-head bf16 forward (persistent CTAs, two
// softmax warpgroups in ping-pong, K and V tiles through a two-stage ring, one
// MMA issuer, P written into TMEM over the scores it replaces), with the
// operands quantized first (fp8_quant_kernel below):
//   * Q and K, rotated, in e4m3 with one scale per (batch row, head, 128-row
//     tile): x8 = rn(x * 448 / amax(tile)), dequantized by amax/448;
//   * V in e4m3 with one scale per (batch row, kv head), stored transposed
//     (V^T, keys contiguous) so that both operands of the PV MMA are K-major;
//   * P = 2^(s - m) with m the running row maximum, renewed only when a
//     tile's maximum exceeds it by more than 2 (so P <= 4), stored as
//     rn(112 * P) <= 448 in e4m3 in TMEM; the factor 112 is added to the
//     exponent (2^(s - m + log2 112)), not multiplied in.
// The scores S = Q8 K8^T come out of kind::f8f6f4 MMAs (32 elements per K
// step, twice the bf16 rate) and are dequantized in the exponent: s =
// S * scale * log2(e) * deq_q * deq_k.  O accumulates (112 P) V8 and l the
// float32 112 P, so the epilogue scales O by deq_v / l; lse = m + log2(l) -
// log2(112), in natural-log units.
// The arithmetic is that of "nanoeuler -- CUDA kernels",
// attention_forward_kernel, with the inputs rounded to e4m3 (3 mantissa bits)
// and P rounded to e4m3 before the PV product.
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_profile.h"
#include "attn_ptx.cuh"

namespace attn {
namespace {

constexpr int kHD = 128;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// Lazy rescale: the running max m is renewed (and O, l rescaled) only when a
// tile's maximum exceeds it by more than kRescaleThreshold, so P = 2^(s - m)
// stays <= 4 and 112 P <= 448, the largest finite e4m3 value.
constexpr float kRescaleThreshold = 2.0f;
constexpr float kLog2PScale = 6.807354922057604f;   // log2(112)
constexpr int kThreads = 320;

struct Fp8Cfg {
  static constexpr int kTileBytes = 128 * kHD;          // e4m3 Q / K / V^T tile: one atom
  static constexpr int kOutBytes = 128 * kHD * 2;       // bf16 output tile
  static constexpr int kKStages = 2, kVStages = 2;
  static constexpr int kQOff = 0;                       // Q_A, Q_B
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kStOff = kVOff + kVStages * kTileBytes;   // output staging tile
  static constexpr int kBarOff = kStOff + kOutBytes;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;
  static_assert(kSmemBytes <= 232448, "FP8 forward kernel exceeds the 227 KB shared-memory limit");
};

__device__ __forceinline__ uint32_t tmem_s(int x) { return 128u * (uint32_t)x; }
__device__ __forceinline__ uint32_t tmem_o(int x) { return 256u + 128u * (uint32_t)x; }

struct Fp8Barriers {
  uint64_t q_full, q_empty;
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t staged[2], stage_free, drain;
  uint32_t tmem_base;
  int abort;
};

// Work item w -> (batch row, head pair, query tile); heaviest first.
struct Fp8Item {
  int b, h0, kh, qt;
};
__device__ __forceinline__ Fp8Item fp8_item(int w, const Geometry& g) {
  const int n_qt = (g.T + 127) / 128, pairs = g.NH / 2, bp_count = g.B * pairs;
  Fp8Item it;
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

__global__ void __launch_bounds__(kThreads, 1)
fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_qk, const __grid_constant__ CUtensorMap tm_v,
               const __grid_constant__ CUtensorMap tm_out, float* __restrict__ lse, int* __restrict__ status,
               Geometry g, int n_items, const float* __restrict__ deq_qk, const float* __restrict__ deq_v) {
  using Cfg = Fp8Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Cfg::kQOff;
  uint8_t* sK = smem + Cfg::kKOff;
  uint8_t* sV = smem + Cfg::kVOff;
  uint8_t* sSt = smem + Cfg::kStOff;
  Fp8Barriers* bars = reinterpret_cast<Fp8Barriers*>(smem + Cfg::kBarOff);
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
  // Launched as a programmatic dependent of the quantization pass: wait for
  // it before reading its outputs.
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
        const Fp8Item item = fp8_item(w, g);
        const int n_kv = item.qt + 1;
        const int k_col = g.C + item.kh * kHD, vt_z = item.b * g.NKV + item.kh;
        if (it >= 1 && !(ok = ptx::mbar_wait(ptx::smem_u32(&bars->q_empty), (it - 1) & 1, abort_flag, kWaitLimitNs)))
          break;
        const uint32_t qf = ptx::smem_u32(&bars->q_full);
        ptx::mbar_arrive_expect_tx(qf, 2 * Cfg::kTileBytes);
#pragma unroll
        for (int x = 0; x < 2; ++x)
          ptx::tma_load_3d(ptx::smem_u32(sQ + x * Cfg::kTileBytes), &tm_qk, (item.h0 + x) * kHD, item.qt * 128,
                           item.b, qf);
        q_issued = it + 1;
        // K_j and V_j into one ring stage with one barrier (each barrier the
        // MMA issuer checks stalls the tensor pipe).
        for (int j = 0; j < n_kv && ok; ++j) {
          const int gk = kv_issued, st = gk % 2;
          if (gk >= 2 && !(ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_empty[st]), ((gk >> 1) - 1) & 1, abort_flag,
                                               kWaitLimitNs)))
            break;
          const uint32_t kvf = ptx::smem_u32(&bars->kv_full[st]);
          ptx::mbar_arrive_expect_tx(kvf, 2 * Cfg::kTileBytes);
          ptx::tma_load_3d(ptx::smem_u32(sK + st * Cfg::kTileBytes), &tm_qk, k_col, j * 128, item.b, kvf);
          ptx::tma_load_3d(ptx::smem_u32(sV + st * Cfg::kTileBytes), &tm_v, j * 128, 0, vt_z, kvf);
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
      constexpr uint32_t idesc_s = ptx::idesc_e4m3_f32(128, 128);
      constexpr uint32_t idesc_o = ptx::idesc_e4m3_f32(128, kHD);
      const uint64_t dQ = ptx::sw128_desc(ptx::smem_u32(sQ), 16, 1024);
      const uint64_t dK = ptx::sw128_desc(ptx::smem_u32(sK), 16, 1024);
      const uint64_t dV = ptx::sw128_desc(ptx::smem_u32(sV), 16, 1024);   // V^T: K-major too
      bool ok = true;
      // S_x(g) = Q_x K_g^T into the score columns of group x.
      auto issue_s = [&](int x, int gk) {
        const uint64_t bk = ptx::desc_advance(dK, (gk % 2) * Cfg::kTileBytes);
        const uint64_t aq = ptx::desc_advance(dQ, x * Cfg::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kHD / 32; ++kk)
          ptx::mma_e4m3_ss_w(tmem + tmem_s(x), ptx::desc_advance(aq, kk * 32), ptx::desc_advance(bk, kk * 32), idesc_s,
                           kk > 0 ? 1u : 0u);
        ptx::mma_commit_w(ptx::smem_u32(&bars->s_full[x]));
      };
      // O_x += P8_x(g) V8_g with P from TMEM (four e4m3 per column).
      auto issue_pv = [&](int x, int gk, bool first) {
        const uint64_t bv = ptx::desc_advance(dV, (gk % 2) * Cfg::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 128 / 32; ++kk)
          ptx::mma_e4m3_ts_w(tmem + tmem_o(x), tmem + tmem_s(x) + kk * 8, ptx::desc_advance(bv, kk * 32), idesc_o,
                           (!first || kk > 0) ? 1u : 0u);
      };
      int g0 = 0;   // global index of the item's first key tile
      for (int it = 0, w = w0; w < n_items && ok; ++it, w = snake(it, w0, dw)) {
        const Fp8Item item = fp8_item(w, g);
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
      const Fp8Item item = fp8_item(w, g);
      const int n_kv = item.qt + 1;
      const int n_qt = (g.T + 127) / 128, heads = g.NH + g.NKV;
      const float dq = deq_qk[((size_t)item.b * heads + item.h0 + x) * n_qt + item.qt];
      const float* dk_row = deq_qk + ((size_t)item.b * heads + g.NH + item.kh) * n_qt;
      float m = -INFINITY, l = 0.f;
      float dk_next = dk_row[0];
      for (int j = 0; j < n_kv; ++j, ++gk) {
        // K-tile scale of this step, and the next one's load issued early.
        const float dk_j = dk_next;
        if (j + 1 < n_kv) dk_next = dk_row[j + 1];
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
        // Row max with 4 independent partial maxima, two new scores per
        // three-input max.
        float mx[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) mx[k] = __uint_as_float(sr[k]);
#pragma unroll
        for (int c = 4; c < 128; c += 8)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mx[k] = ptx::fmax3(mx[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 4 + k]));
        const float sl2j = sl2 * dq * dk_j;             // scale * log2(e) * dequantization
        const float m_cand = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2j;
        const bool grow = m_cand > m + kRescaleThreshold;   // always true on an item's first tile
        const float m_new = grow ? m_cand : m;
        const float corr = grow ? ptx::ex2_approx(m - m_new) : 1.f;
        // 112 p = 2^(s - m + log2 112) with s the dequantized scaled score, in
        // e4m3, four per column, written over the score columns 8 at a time
        // (columns 8h.. hold keys 32h.., already read); row sum of the
        // float32 112 p in 4 partial sums.
        const float2 sl2x2 = make_float2(sl2j, sl2j);
        const float2 negm2 = make_float2(kLog2PScale - m_new, kLog2PScale - m_new);
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t pw[8];
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const int cc = 32 * h + c;
            const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])), sl2x2,
                                         negm2);
            const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sr[cc + 2]), __uint_as_float(sr[cc + 3])),
                                         sl2x2, negm2);
            const float2 p0 = make_float2(ptx::ex2_approx(x0.x), ptx::ex2_approx(x0.y));
            const float2 p1 = make_float2(ptx::ex2_approx(x1.x), ptx::ex2_approx(x1.y));
            acc[0] = __fadd2_rn(acc[0], p0);
            acc[1] = __fadd2_rn(acc[1], p1);
            pw[c >> 2] = ptx::cvt_e4m3x2(p0.x, p0.y) | (ptx::cvt_e4m3x2(p1.x, p1.y) << 16);
          }
          ptx::tmem_st8(s_addr + 8 * h, pw);
        }
        const float2 acc2 = __fadd2_rn(acc[0], acc[1]);
        l = l * corr + (acc2.x + acc2.y);
        m = m_new;
        // O_x is idle here: PV_x(j-1) was issued before S_x(j), whose
        // completion this group waited for.
        if ((j >= 1) && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int c0 = 0; c0 < kHD; c0 += 32) {
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
      const float inv_l = deq_v[(size_t)item.b * g.NKV + item.kh] / l;
#pragma unroll 1
      for (int c0 = 0; c0 < kHD; c0 += 32) {
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
      if (tq < g.T)
        lse[((size_t)item.b * g.NH + item.h0 + x) * g.T + tq] = (m + (log2f(l) - kLog2PScale)) * 0.6931471805599453f;
      if (storer) {
        // All four warps staged their rows: store the tile, and release the
        // staging tile once the TMA engine has read it.
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->staged[x]), it & 1, abort_flag, kWaitLimitNs);
        if (ok) {
#pragma unroll
          for (int a = 0; a < kHD / 64; ++a)
            ptx::tma_store_3d(&tm_out, ptx::smem_u32(sSt + a * (128 * 128)), (item.h0 + x) * kHD + 64 * a,
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


// ---------------------------------------------------------------------------
// Quantization pass.
// ---------------------------------------------------------------------------
// amax of V over one 128-row tile of one (batch row, kv head), into
// vtile_amax[b][kv][tile]; the quantization pass takes the maximum over the
// tiles of a head (deq_v = amax / 448), so every tile of a head shares one
// scale and the result does not depend on the order of anything.
__global__ void __launch_bounds__(256) fp8_vamax_kernel(float* __restrict__ vtile_amax,
                                                        const __nv_bfloat16* __restrict__ qkv, Geometry g) {
  __shared__ float red[256];
  const int tile = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  // The quantization grid is launched as a programmatic dependent: its Q/K
  // blocks need nothing from here and may start at once.
  ptx::grid_dep_launch();
  float mx = 0.f;
  for (int u = threadIdx.x; u < 128 * (kHD / 8); u += 256) {
    const int t = tile * 128 + u / (kHD / 8), c = u % (kHD / 8);
    if (t >= g.T) break;
    const uint4 v = *reinterpret_cast<const uint4*>(qkv + ((size_t)b * g.T + t) * g.W + g.C + g.NKV * kHD + kh * kHD +
                                                    8 * c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
  }
  red[threadIdx.x] = mx;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + s]);
    __syncthreads();
  }
  if (threadIdx.x == 0) vtile_amax[((size_t)b * g.NKV + kh) * gridDim.x + tile] = red[0];
}

// One CTA per (128-row tile, head, batch row); heads 0..NH+NKV-1 are the Q
// and K heads (rotated, one scale per tile, into the e4m3 copy with the
// layout of the bf16 rotated copy), heads NH+NKV.. the V heads (scale per
// head from the tile maxima of fp8_vamax_kernel, written transposed into
// V^T [b][kv][d][Tp]).  In a Q/K block, thread = (row r = tid / 4, quarter of
// the head's pairs), so a thread holds 32 rotated values.
constexpr int kQuantThreads = 512;

__global__ void __launch_bounds__(kQuantThreads) fp8_quant_kernel(uint8_t* __restrict__ qk8, uint8_t* __restrict__ vt8,
                                                                  float* __restrict__ deq_qk,
                                                                  float* __restrict__ deq_v,
                                                                  const float* __restrict__ vtile_amax,
                                                                  const __nv_bfloat16* __restrict__ qkv, Geometry g,
                                                                  int Tp) {
  __shared__ float red[kQuantThreads / 32];
  __shared__ __align__(16) uint8_t tile8[kHD][128 + 16];
  const int tile = blockIdx.x, head = blockIdx.y, b = blockIdx.z;
  const int heads = g.NH + g.NKV, n_qt = (g.T + 127) / 128;
  if (head < heads) {
    const int r = threadIdx.x >> 2, part = threadIdx.x & 3;
    const int t = tile * 128 + r;
    const bool valid = t < g.T;
    const __nv_bfloat16* src = qkv + ((size_t)b * g.T + (valid ? t : 0)) * g.W + head * kHD;
    float y0[16], y1[16];
    float mx = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int gi = part * 2 + q;                          // 8 pairs 8 gi .. 8 gi + 7
      uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0;
      if (valid) load_rope_pairs(src, gi, kHD / 2, g.rope_interleaved != 0, x0, x1);
      const uint32_t a[4] = {x0.x, x0.y, x0.z, x0.w}, c[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float u0 = (k & 1) ? bf16_hi(a[k >> 1]) : bf16_lo(a[k >> 1]);
        const float u1 = (k & 1) ? bf16_hi(c[k >> 1]) : bf16_lo(c[k >> 1]);
        float v0 = u0, v1 = u1;
        if (g.rope_theta > 0.f) {
          float sn, cs;
          const int i = 8 * gi + k;
          __sincosf(rope_angle(valid ? t : 0, g.rope_f_hi[i], g.rope_f_lo[i]), &sn, &cs);
          rope_pair(u0, u1, cs, sn, v0, v1);
        }
        y0[8 * q + k] = v0;
        y1[8 * q + k] = v1;
        mx = fmaxf(mx, fmaxf(fabsf(v0), fabsf(v1)));
      }
    }
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    const float scale = amax > 0.f ? 448.f / amax : 1.f;
    if (threadIdx.x == 0) deq_qk[((size_t)b * heads + head) * n_qt + tile] = amax > 0.f ? amax / 448.f : 1.f;
    if (valid) {
      // Pairs 16 part .. 16 part + 15 -> slots i and i + hd/2 of the head.
      uint8_t* dst = qk8 + ((size_t)b * g.T + t) * (size_t)(heads * kHD) + head * kHD;
      uint32_t w0[4], w1[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w0[k] = ptx::cvt_e4m3x2(y0[4 * k] * scale, y0[4 * k + 1] * scale) |
                (ptx::cvt_e4m3x2(y0[4 * k + 2] * scale, y0[4 * k + 3] * scale) << 16);
        w1[k] = ptx::cvt_e4m3x2(y1[4 * k] * scale, y1[4 * k + 1] * scale) |
                (ptx::cvt_e4m3x2(y1[4 * k + 2] * scale, y1[4 * k + 3] * scale) << 16);
      }
      *reinterpret_cast<uint4*>(dst + 16 * part) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
      *reinterpret_cast<uint4*>(dst + kHD / 2 + 16 * part) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
    }
    return;
  }
  // V head kv, transposed, with the head's scale (maximum of its tile
  // maxima, written by fp8_vamax_kernel, which this grid may overlap: wait
  // for it here).  Warp cw takes columns 8 cw .. 8 cw + 7, lane rg rows
  // 4 rg .. 4 rg + 3, and writes each column's four bytes as one word, so
  // the 32 lanes of a warp store 32 consecutive words.
  ptx::grid_dep_wait();
  const int kv = head - heads;
  float mx = 0.f;
  for (int k = 0; k < n_qt; ++k) mx = fmaxf(mx, vtile_amax[((size_t)b * g.NKV + kv) * n_qt + k]);
  const float scale = mx > 0.f ? 448.f / mx : 1.f;
  if (tile == 0 && threadIdx.x == 0) deq_v[(size_t)b * g.NKV + kv] = mx > 0.f ? mx / 448.f : 1.f;
  const int cw = threadIdx.x >> 5, rg = threadIdx.x & 31;
  uint4 raw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int tv = tile * 128 + 4 * rg + i;
    raw[i] = make_uint4(0, 0, 0, 0);
    if (tv < g.T)
      raw[i] = *reinterpret_cast<const uint4*>(qkv + ((size_t)b * g.T + tv) * g.W + g.C + g.NKV * kHD + kv * kHD +
                                               8 * cw);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {          // bf16 pair k = columns 2k, 2k+1
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = (&raw[i].x)[k];
    const uint32_t lo01 = ptx::cvt_e4m3x2(bf16_lo(w[0]) * scale, bf16_lo(w[1]) * scale);
    const uint32_t lo23 = ptx::cvt_e4m3x2(bf16_lo(w[2]) * scale, bf16_lo(w[3]) * scale);
    const uint32_t hi01 = ptx::cvt_e4m3x2(bf16_hi(w[0]) * scale, bf16_hi(w[1]) * scale);
    const uint32_t hi23 = ptx::cvt_e4m3x2(bf16_hi(w[2]) * scale, bf16_hi(w[3]) * scale);
    *reinterpret_cast<uint32_t*>(&tile8[8 * cw + 2 * k][4 * rg]) = lo01 | (lo23 << 16);
    *reinterpret_cast<uint32_t*>(&tile8[8 * cw + 2 * k + 1][4 * rg]) = hi01 | (hi23 << 16);
  }
  __syncthreads();
  // Row d of V^T (keys tile*128 .. +127) in eight 16-byte chunks.
#pragma unroll
  for (int k = 0; k < (kHD * 8) / kQuantThreads; ++k) {
    const int id = threadIdx.x + k * kQuantThreads, d = id >> 3, q = id & 7;
    uint8_t* dst = vt8 + (((size_t)b * g.NKV + kv) * kHD + d) * (size_t)Tp + tile * 128 + 16 * q;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&tile8[d][16 * q]);
  }
}

}  // namespace

bool fp8_fwd_supported(const Geometry& g) { return g.hd == kHD && g.grp % 2 == 0; }

cudaError_t fp8_fwd_launch(const Fp8FwdArgs& a, cudaStream_t stream) {
  const Geometry& g = a.g;
  const int n_qt = (g.T + 127) / 128, heads = g.NH + g.NKV;
  prof_begin(kKernelFp8Prep, stream);
  fp8_vamax_kernel<<<dim3(n_qt, g.NKV, g.B), 256, 0, stream>>>(a.vtile_amax, (const __nv_bfloat16*)a.qkv, g);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    e = launch_pdl(fp8_quant_kernel, dim3(n_qt, heads + g.NKV, g.B), dim3(kQuantThreads), 0, stream, a.qk8, a.vt8,
                   a.deq_qk, a.deq_v, (const float*)a.vtile_amax, (const __nv_bfloat16*)a.qkv, g, a.Tp);
  }
  prof_end(kKernelFp8Prep, stream);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Fp8Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_items = n_qt * g.B * (g.NH / 2);
  const unsigned grid = (unsigned)(n_items < a.num_sms ? n_items : a.num_sms);
  prof_begin(kKernelFwdFp8, stream);
  e = launch_pdl(fwd_fp8_kernel, dim3(grid), dim3(kThreads), Fp8Cfg::kSmemBytes, stream, a.tm_qk8, a.tm_vt, a.tm_out,
                 a.lse, a.status, g, n_items, (const float*)a.deq_qk, (const float*)a.deq_v);
  prof_end(kKernelFwdFp8, stream);
  return e;
}

}  // namespace attn
