// Causal MHA/GQA attention forward on sm_103a tensor cores (bf16 in, f32
// accumulation), head size 64 or 128.
//
// One CTA owns a 128-query tile of one (batch row, query head) and walks the
// key tiles 0..qt (causal tile skipping: tiles entirely above the diagonal are
// never loaded).  Warp roles:
//   warp 0      TMA producer: Q once, then K_j and V_j into separate rings;
//               K runs two tiles ahead of V so that S_j never waits on a load.
//   warp 1      TMEM owner and MMA issuer (one thread): S_j = Q K_j^T into one
//               of two TMEM score buffers, O += P_j V_j into the TMEM output.
//   warps 2-5   softmax: thread = query row = TMEM lane.  Reads S_j, keeps the
//               running max m and sum l, writes P_j (bf16) to shared memory in
//               the MMA's swizzled layout, rescales O in TMEM when m grows
//               past a threshold (exact: l and O share the stale max), and in
//               the epilogue writes out = O / l and lse = m + ln l.
//   warps 6-9   (RoPE only) rotate Q and every landed K tile in shared memory
//               before the MMA warp may read them.
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
constexpr int kSoftmaxWarp0 = 2;
constexpr int kRopeWarp0 = 6;

template <int HD, bool ROPE>
struct FwdCfg {
  static constexpr int kAtomBytes = kBM * 128;              // 128 rows x 128 B swizzle-atom column
  static constexpr int kTileBytes = kBM * HD * 2;           // Q / K / V tile
  static constexpr int kKStages = (HD == 128) ? 3 : 4;      // K ring depth
  static constexpr int kVStages = (HD == 128) ? 2 : 4;      // V ring depth
  static constexpr int kQOff = 0;
  static constexpr int kPOff = kQOff + kTileBytes;
  static constexpr int kPBytes = kBM * kBN * 2;
  static constexpr int kKOff = kPOff + kPBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;   // barriers + alignment slack
  static_assert(kSmemBytes <= 232448, "forward kernel exceeds the 227 KB shared-memory limit");
  static constexpr int kThreads = ROPE ? 320 : 192;
  static constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256, kTmemCols = 512;
};

struct FwdBarriers {
  uint64_t q_full, q_ready, pv_done, p_full, drain;
  uint64_t s_full[2], s_free[2];
  uint64_t k_full[4], k_ready[4], k_empty[4], v_full[4], v_empty[4];
  uint32_t tmem_base;
  int abort;
};

// Byte offset of element (row, col) inside a 128-row bf16 tile stored as
// 128-byte-swizzled atom columns of 64 elements.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col) {
  const int atom = col >> 6, chunk = (col & 63) >> 3;
  return atom * (kBM * 128) + row * 128 + ((chunk ^ (row & 7)) << 4) + ((col & 7) << 1);
}

// Rotate a 128-row tile in shared memory (NEOX pairs (i, i+HD/2)).  128
// threads: thread tid owns pairs 8p..8p+7 (p = tid % NCH) for rows
// r0, r0 + RS, ..., r0 = tid / NCH.  Angles advance by RS rows with the
// angle-addition recurrence, from an accurately reduced start per tile.
template <int HD>
struct TileRotator {
  static constexpr int NCH = HD / 16;        // 8-pair groups per row
  static constexpr int RS = 128 / NCH;       // row stride between a thread's rows
  static constexpr int ROWS = 128 / RS;      // rows per thread
  float f_hi[8], f_lo[8], step_c[8], step_s[8];
  int p, r0;

  __device__ void init(int tid, const Geometry& g) {
    p = tid % NCH;
    r0 = tid / NCH;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      f_hi[e] = g.rope_f_hi[8 * p + e];
      f_lo[e] = g.rope_f_lo[8 * p + e];
      __sincosf(rope_angle(RS, f_hi[e], f_lo[e]), &step_s[e], &step_c[e]);
    }
  }

  __device__ void rotate(uint8_t* tile, int pos0) {
    float c[8], s[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) __sincosf(rope_angle(pos0 + r0, f_hi[e], f_lo[e]), &s[e], &c[e]);
#pragma unroll 1
    for (int k = 0; k < ROWS; ++k) {
      const int r = r0 + k * RS;
      uint4* a_ptr = reinterpret_cast<uint4*>(tile + sw128_offset(r, 8 * p));
      uint4* b_ptr = reinterpret_cast<uint4*>(tile + sw128_offset(r, 8 * p + HD / 2));
      uint4 a = *a_ptr, b = *b_ptr;
      uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float y0l, y1l, y0h, y1h;
        rope_pair(bf16_lo(av[q]), bf16_lo(bv[q]), c[2 * q], s[2 * q], y0l, y1l);
        rope_pair(bf16_hi(av[q]), bf16_hi(bv[q]), c[2 * q + 1], s[2 * q + 1], y0h, y1h);
        av[q] = pack_bf16x2(y0l, y0h);
        bv[q] = pack_bf16x2(y1l, y1h);
      }
      *a_ptr = make_uint4(av[0], av[1], av[2], av[3]);
      *b_ptr = make_uint4(bv[0], bv[1], bv[2], bv[3]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {  // advance the angle by RS positions
        const float cn = c[e] * step_c[e] - s[e] * step_s[e];
        s[e] = s[e] * step_c[e] + c[e] * step_s[e];
        c[e] = cn;
      }
    }
  }
};

template <int HD, bool ROPE>
__global__ void __launch_bounds__(FwdCfg<HD, ROPE>::kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_qkv, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
           int* __restrict__ status, Geometry g) {
  using Cfg = FwdCfg<HD, ROPE>;
  constexpr int NK = Cfg::kKStages, NV = Cfg::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Cfg::kQOff;
  uint8_t* sP = smem + Cfg::kPOff;
  uint8_t* sK = smem + Cfg::kKOff;
  uint8_t* sV = smem + Cfg::kVOff;
  FwdBarriers* bars = reinterpret_cast<FwdBarriers*>(smem + Cfg::kBarOff);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // Tile order: heaviest query tiles first; heads sharing a kv head adjacent.
  const int n_qt = (g.T + kBM - 1) / kBM;
  const int bh_count = g.B * g.NH;
  const int qt = n_qt - 1 - (int)(blockIdx.x / bh_count);
  const int bh = blockIdx.x % bh_count;
  const int b = bh / g.NH, h = bh % g.NH;
  const int kh = h / g.grp;
  const int q0 = qt * kBM;
  const int n_kv = qt + 1;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->q_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->q_ready), 4);
    ptx::mbar_init(ptx::smem_u32(&bars->pv_done), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->p_full), 4);
    ptx::mbar_init(ptx::smem_u32(&bars->drain), 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->s_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->s_free[i]), 4);
    }
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

  auto fail = [&]() {
    *abort_flag = 1;
    record_status(status, kErrDeviceTimeout);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_qkv);
      const int q_col = h * HD, k_col = g.C + kh * HD, v_col = g.C + g.NKV * HD + kh * HD;
      const uint32_t q_full = ptx::smem_u32(&bars->q_full);
      ptx::mbar_arrive_expect_tx(q_full, Cfg::kTileBytes);
#pragma unroll
      for (int a = 0; a < HD / 64; ++a)
        ptx::tma_load_3d(ptx::smem_u32(sQ + a * Cfg::kAtomBytes), &tm_qkv, q_col + 64 * a, q0, b, q_full);
      // Issue order: K_0, K_1, then V_j, K_{j+2} for j = 0, 1, ...
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      auto load_k = [&](int j) -> bool {
        const int st = j % NK, u = j / NK;
        if (u > 0 && !ptx::mbar_wait(ptx::smem_u32(&bars->k_empty[st]), (u - 1) & 1, abort_flag, kWaitLimitNs))
          return false;
        const uint32_t kf = ptx::smem_u32(&bars->k_full[st]);
        ptx::mbar_arrive_expect_tx(kf, Cfg::kTileBytes);
#pragma unroll
        for (int a = 0; a < HD / 64; ++a)
          ptx::tma_load_3d(ptx::smem_u32(sK + st * Cfg::kTileBytes + a * Cfg::kAtomBytes), &tm_qkv, k_col + 64 * a,
                           j * kBN, b, kf);
        k_issued = j + 1;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int st = j % NV, u = j / NV;
        if (u > 0 && !ptx::mbar_wait(ptx::smem_u32(&bars->v_empty[st]), (u - 1) & 1, abort_flag, kWaitLimitNs))
          return false;
        const uint32_t vf = ptx::smem_u32(&bars->v_full[st]);
        ptx::mbar_arrive_expect_tx(vf, Cfg::kTileBytes);
#pragma unroll
        for (int a = 0; a < HD / 64; ++a)
          ptx::tma_load_3d(ptx::smem_u32(sV + st * Cfg::kTileBytes + a * Cfg::kAtomBytes), &tm_qkv, v_col + 64 * a,
                           j * kBN, b, vf);
        v_issued = j + 1;
        return true;
      };
      for (int j = 0; j < 2 && j < n_kv && ok; ++j) ok = load_k(j);
      for (int j = 0; j < n_kv && ok; ++j) {
        ok = load_v(j);
        if (ok && j + 2 < n_kv) ok = load_k(j + 2);
      }
      if (!ok) fail();
      if (*abort_flag) {
        // Let every copy already in flight land before shared memory is released.
        ptx::mbar_wait(q_full, 0, nullptr, kWaitLimitNs);
        for (int st = 0; st < NK && st < k_issued; ++st)
          ptx::mbar_wait(ptx::smem_u32(&bars->k_full[st]), ((k_issued - 1 - st) / NK) & 1, nullptr, kWaitLimitNs);
        for (int st = 0; st < NV && st < v_issued; ++st)
          ptx::mbar_wait(ptx::smem_u32(&bars->v_full[st]), ((v_issued - 1 - st) / NV) & 1, nullptr, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(kBM, HD, false, true);
      const uint32_t sQa = ptx::smem_u32(sQ), sPa = ptx::smem_u32(sP);
      const uint32_t sKa = ptx::smem_u32(sK), sVa = ptx::smem_u32(sV);
      bool ok = ptx::mbar_wait(ptx::smem_u32(ROPE ? &bars->q_ready : &bars->q_full), 0, abort_flag, kWaitLimitNs);

      auto issue_pv = [&](int i) -> bool {
        const int sp = i % NV;
        if (!ptx::mbar_wait(ptx::smem_u32(&bars->p_full), i & 1, abort_flag, kWaitLimitNs)) return false;
        if (!ptx::mbar_wait(ptx::smem_u32(&bars->v_full[sp]), (i / NV) & 1, abort_flag, kWaitLimitNs)) return false;
        ptx::tc_fence_after();
        const uint32_t v_base = sVa + sp * Cfg::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t a = ptx::sw128_desc(sPa + (kk >> 2) * Cfg::kAtomBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t bdesc = ptx::sw128_desc(v_base + kk * 2048, Cfg::kAtomBytes, 1024);
          ptx::mma_bf16_ss(tmem + Cfg::kTmemO, a, bdesc, idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(ptx::smem_u32(&bars->pv_done));
        ptx::mma_commit(ptx::smem_u32(&bars->v_empty[sp]));
        return true;
      };

      for (int j = 0; j < n_kv && ok; ++j) {
        const int s = j % NK, sb = j & 1;
        ok = ptx::mbar_wait(ptx::smem_u32(ROPE ? &bars->k_ready[s] : &bars->k_full[s]), (j / NK) & 1, abort_flag,
                            kWaitLimitNs);
        if (ok && j >= 2) ok = ptx::mbar_wait(ptx::smem_u32(&bars->s_free[sb]), ((j >> 1) - 1) & 1, abort_flag,
                                              kWaitLimitNs);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t k_base = sKa + s * Cfg::kTileBytes;
        const uint32_t d_s = tmem + (sb ? Cfg::kTmemS1 : Cfg::kTmemS0);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Cfg::kAtomBytes + (kk & 3) * 32;
          ptx::mma_bf16_ss(d_s, ptx::sw128_desc(sQa + off, 16, 1024), ptx::sw128_desc(k_base + off, 16, 1024),
                           idesc_s, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(ptx::smem_u32(&bars->s_full[sb]));
        ptx::mma_commit(ptx::smem_u32(&bars->k_empty[s]));
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) ok = issue_pv(n_kv - 1);
      if (!ok) fail();
      // Drain: every MMA this thread issued has finished before TMEM is freed.
      ptx::mma_commit(ptx::smem_u32(&bars->drain));
      ptx::mbar_wait(ptx::smem_u32(&bars->drain), 0, nullptr, kWaitLimitNs);
    }
  } else if (warp < kSoftmaxWarp0 + 4) {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const int tq = q0 + row;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = g.scale * 1.4426950408889634f;  // scale * log2(e)
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->s_full[sb]), (j >> 1) & 1, abort_flag,
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

      if (j == n_kv - 1) {  // diagonal tile: key c is visible to row `row` iff c <= row
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c > row) sr[c] = __float_as_uint(-INFINITY);
      }
      float mt = __uint_as_float(sr[0]);
#pragma unroll
      for (int c = 1; c < kBN; ++c) mt = fmaxf(mt, __uint_as_float(sr[c]));
      const float m_cand = mt * sl2;
      const bool grow = m_cand > m + kRescaleThreshold;   // always true on the first tile
      const float m_new = grow ? m_cand : m;
      const float corr = grow ? ptx::ex2_approx(m - m_new) : 1.f;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kBN; ++c) {
        const float p = ptx::ex2_approx(fmaf(__uint_as_float(sr[c]), sl2, -m_new));
        sr[c] = __float_as_uint(p);
        rs += p;
      }
      l = l * corr + rs;
      m = m_new;

      // P_j may overwrite P_{j-1} and O may be rescaled only after PV_{j-1}.
      if (j >= 1) {
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->pv_done), (j - 1) & 1, abort_flag,
                                                      kWaitLimitNs));
        if (!ok) break;
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int c0 = 0; c0 < HD; c0 += 32) {
            uint32_t o[32];
            ptx::tmem_ld32(t_lane + Cfg::kTmemO + c0, o);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * corr);
            ptx::tmem_st32(t_lane + Cfg::kTmemO + c0, o);
          }
          ptx::tmem_wait_st();
        }
      }
#pragma unroll
      for (int ch = 0; ch < kBN / 8; ++ch) {
        const uint32_t* q = &sr[8 * ch];
        const uint4 v = make_uint4(pack_bf16x2(__uint_as_float(q[0]), __uint_as_float(q[1])),
                                   pack_bf16x2(__uint_as_float(q[2]), __uint_as_float(q[3])),
                                   pack_bf16x2(__uint_as_float(q[4]), __uint_as_float(q[5])),
                                   pack_bf16x2(__uint_as_float(q[6]), __uint_as_float(q[7])));
        *reinterpret_cast<uint4*>(sP + sw128_offset(row, 8 * ch)) = v;
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->p_full));
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->pv_done), (n_kv - 1) & 1, abort_flag,
                                                    kWaitLimitNs));
    }
    if (ok) {
      ptx::tc_fence_after();
      const float inv_l = 1.f / l;
      __nv_bfloat16* orow = out + ((size_t)b * g.T + tq) * g.C + h * HD;
#pragma unroll 1
      for (int c0 = 0; c0 < HD; c0 += 32) {
        uint32_t o[32];
        ptx::tmem_ld32(t_lane + Cfg::kTmemO + c0, o);
        ptx::tmem_wait_ld();
        if (tq < g.T) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 w = make_uint4(
                pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l),
                pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l),
                pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l),
                pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l));
            *reinterpret_cast<uint4*>(orow + c0 + 8 * v) = w;
          }
        }
      }
      if (tq < g.T) lse[((size_t)b * g.NH + h) * g.T + tq] = (m + log2f(l)) * 0.6931471805599453f;
    } else {
      fail();
    }
  } else if (ROPE) {
    // ------------------------------------------------------------ RoPE transform
    const int tid = threadIdx.x - kRopeWarp0 * 32;
    TileRotator<HD> rot;
    rot.init(tid, g);
    bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->q_full), 0, abort_flag, kWaitLimitNs));
    if (ok) {
      rot.rotate(sQ, q0);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->q_ready));
    }
    for (int j = 0; j < n_kv && ok; ++j) {
      const int s = j % NK;
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->k_full[s]), (j / NK) & 1, abort_flag,
                                                    kWaitLimitNs));
      if (!ok) break;
      rot.rotate(sK + s * Cfg::kTileBytes, j * kBN);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->k_ready[s]));
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
  const unsigned grid = (unsigned)(n_qt * a.g.B * a.g.NH);
  prof_begin(kKernelFwdTc05, stream);
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(a.tm_qkv, (__nv_bfloat16*)a.out, a.lse, a.status, a.g);
  prof_end(kKernelFwdTc05, stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tc05_fwd_launch(const Tc05FwdArgs& a, cudaStream_t stream) {
  const bool rope = a.g.rope_theta > 0.f;
  if (a.g.hd == 128) return rope ? launch_fwd<128, true>(a, stream) : launch_fwd<128, false>(a, stream);
  if (a.g.hd == 64) return rope ? launch_fwd<64, true>(a, stream) : launch_fwd<64, false>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
