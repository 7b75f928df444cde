// QKV projection with the RoPE rotation fused into its epilogue (bf16,
// tcgen05 on CTA pairs, persistent).
//
// The trainers on the pages project the layer input into the packed Q | K | V
// activation with a GEMM and then run separate RoPE passes over its Q and K
// column blocks ("nanoeuler -- CUDA kernels": the matmul into qkv, then
// rope_kernel over the query heads and the kv heads).  Here the projection
// writes the packed qkv (unrotated, what attn_bwd differentiates against)
// and, from the same float32 accumulators, the rotated copy of its Q and K
// heads that the attention kernels read (the copy attn_fwd_ws's rotation pass
// would otherwise make), so no separate rotation pass is left.
//
//   qkv[m, n] = sum_k x[m, k] w[n, k],  m < M = B*T, n < N = (NH + 2*NKV)*hd
//
// Tiles of 256 x 256 outputs, each computed by a pair of CTAs (a cluster of
// two on neighbouring SMs) with tcgen05.mma.cta_group::2, M = 256: the first
// CTA's shared memory holds rows 0-127 of the x tile and w rows 0-127 of the
// tile, the second CTA's x rows 128-255 and w rows 128-255, so per 64-column
// k-block each CTA stages 32 KB (a 128 x 256 tile on one SM stages 48 KB for
// the same MMA work per SM), and one thread of the first CTA issues the MMAs
// of both.  Each CTA's tensor memory receives its 128 output rows x 256
// columns, in one of two accumulators (256 columns each), so the epilogue of
// a tile overlaps the next tile's MMAs.  6-stage TMA ring per CTA.
//
//   warp 0      TMA producer (each CTA: its x rows and its half of the w rows)
//   warp 1      TMEM (both CTAs); first CTA: MMA issuer
//   warps 2-5   epilogue (both CTAs): TMEM -> bf16 qkv rows, rotated Q/K rows
//
// Barriers live at the same shared-memory offsets in both CTAs.  Both CTAs'
// stage copies signal the first CTA's stage barrier (which expects the bytes
// of both); MMA completion (stage free, accumulator full, drain) is
// committed to both CTAs' barriers at once (multicast); both CTAs' epilogue
// warps release an accumulator on the first CTA's barrier.
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_profile.h"
#include "attn_ptx.cuh"

namespace attn {
namespace {

constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kBM = 256, kBN = 256, kBK = 64, kStages = 6;
constexpr int kRowsCta = kBM / 2;                   // x rows (and w rows) staged per CTA
constexpr int kATile = kRowsCta * kBK * 2;          // 16 KB: one 128-row swizzle atom
constexpr int kBTile = (kBN / 2) * kBK * 2;         // 16 KB
constexpr int kStageBytes = kATile + kBTile;
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kSmemBytes = kBarOff + 256 + 1024;    // + barriers + alignment slack
constexpr int kThreadsP = 192;
static_assert(kSmemBytes <= 232448, "projection kernel exceeds the 227 KB shared-memory limit");

struct ProjBarriers {
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort;
};

// Column n of the rotated copy for pair i of the head at column base h: the
// copy is in NEOX slot order (pair i at slots i and i + hd/2) for either
// pairing, as the attention kernels read it.
__global__ void __launch_bounds__(kThreadsP, 1)
proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
            __nv_bfloat16* __restrict__ qkv, __nv_bfloat16* __restrict__ rot, ProjGeometry pg,
            int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  ProjBarriers* bars = reinterpret_cast<ProjBarriers*>(smem + kBarOff);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = ptx::cluster_rank();          // 0: issuing CTA of the pair
  const int pair = blockIdx.x / 2, n_pairs = gridDim.x / 2;
  const int n_mt = (pg.M + kBM - 1) / kBM, n_nt = (pg.N + kBN - 1) / kBN, n_tiles = n_mt * n_nt;
  const int n_kb = (pg.Cm + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->full[i]), 1);     // used in the first CTA
      ptx::mbar_init(ptx::smem_u32(&bars->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->acc_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->acc_empty[i]), 8);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->drain), 1);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc2(ptx::smem_u32(&bars->tmem_base), 512);
    ptx::tmem_relinquish2();
  }
  ptx::tc_fence_before();
  __syncthreads();
  // Both CTAs' barriers are initialised before either CTA signals the other.
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  auto fail = [&]() {
    *abort_flag = 1;
    ptx::st_cluster_u32(ptx::cluster_addr(ptx::smem_u32(&bars->abort), rank ^ 1u), 1u);
    record_status(status, kErrDeviceTimeout);
  };
  // The pair's MMAs write both CTAs' tensor memory at the first CTA's
  // address: the collective allocation returns the same one to both.
  if (threadIdx.x == 0 && rank == 1 && ptx::ld_cluster_u32(ptx::cluster_addr(ptx::smem_u32(&bars->tmem_base), 0)) != tmem)
    fail();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_x);
      ptx::tma_prefetch_desc(&tm_w);
      bool ok = true;
      int it = 0;
      for (int tile = pair; tile < n_tiles && ok; tile += n_pairs) {
        const int m0 = (tile / n_nt) * kBM + kRowsCta * (int)rank, n0 = (tile % n_nt) * kBN + (kBN / 2) * (int)rank;
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % kStages, u = it / kStages;
          if (u > 0 && !(ok = ptx::mbar_wait_cl(ptx::smem_u32(&bars->empty[st]), (u - 1) & 1, abort_flag,
                                                kWaitLimitNs)))
            break;
          const uint32_t fb = ptx::smem_u32(&bars->full[st]);
          uint8_t* sa = smem + st * kStageBytes;
          if (rank == 0) {
            // The stage barrier takes both CTAs' bytes; the second CTA's
            // copies may land before this arrival (the transaction count
            // goes negative until it).
            ptx::mbar_arrive_expect_tx(fb, 2 * kStageBytes);
            ptx::tma_load_3d(ptx::smem_u32(sa), &tm_x, kb * kBK, m0, 0, fb);
            ptx::tma_load_3d(ptx::smem_u32(sa + kATile), &tm_w, kb * kBK, n0, 0, fb);
          } else {
            const uint32_t lead_fb = ptx::cluster_addr(fb, 0);
            ptx::tma_load_3d_pair(ptx::smem_u32(sa), &tm_x, kb * kBK, m0, 0, lead_fb);
            ptx::tma_load_3d_pair(ptx::smem_u32(sa + kATile), &tm_w, kb * kBK, n0, 0, lead_fb);
          }
        }
      }
      if (!ok) fail();
      if (*abort_flag && rank == 0) {
        // Let the copies in flight (both CTAs') land before shared memory is
        // released; the second CTA exits only after the final cluster barrier.
        for (int st = 0; st < kStages && st < it; ++st)
          ptx::mbar_wait(ptx::smem_u32(&bars->full[st]), ((it - 1 - st) / kStages) & 1, nullptr, kWaitLimitNs);
      }
    }
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp runs the issue loop; one elected lane issues each MMA
    // and commit, and every wait is warp-collective)
    {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint16_t kBoth = 3;
      const uint64_t d0 = ptx::sw128_desc(ptx::smem_u32(smem), 16, 1024);
      bool ok = true;
      int it = 0, lt = 0;
      for (int tile = pair; tile < n_tiles && ok; tile += n_pairs, ++lt) {
        const int buf = lt & 1;
        // The accumulator's previous tile (two back) has been read out by
        // both CTAs.
        if (lt >= 2 &&
            !(ok = ptx::mbar_wait_cl_all(ptx::smem_u32(&bars->acc_empty[buf]), ((lt >> 1) - 1) & 1, abort_flag,
                                         kWaitLimitNs)))
          break;
        ptx::tc_fence_after();
        // Each stage's barrier is checked (non-blocking) one k-block ahead.
        uint32_t ready = __all_sync(
            0xffffffffu, ptx::mbar_test_cl(ptx::smem_u32(&bars->full[it % kStages]), (it / kStages) & 1) != 0);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % kStages, u = it / kStages;
          if (!ready &&
              !(ok = ptx::mbar_wait_cl_all(ptx::smem_u32(&bars->full[st]), u & 1, abort_flag, kWaitLimitNs)))
            break;
          ptx::tc_fence_after();
          ready = (kb + 1 < n_kb)
                      ? __all_sync(0xffffffffu, ptx::mbar_test_cl(ptx::smem_u32(&bars->full[(it + 1) % kStages]),
                                                                  ((it + 1) / kStages) & 1) != 0)
                      : 1u;
          const uint64_t da = ptx::desc_advance(d0, st * kStageBytes);
          const uint64_t db = ptx::desc_advance(d0, st * kStageBytes + kATile);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            ptx::mma2_bf16_ss_w(tmem + buf * kBN, ptx::desc_advance(da, kk * 32), ptx::desc_advance(db, kk * 32),
                                idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          ptx::mma2_commit_mc_w(ptx::smem_u32(&bars->empty[st]), kBoth);
        }
        if (!ok) break;
        ptx::mma2_commit_mc_w(ptx::smem_u32(&bars->acc_full[buf]), kBoth);
      }
      if (!ok) fail();
      ptx::mma2_commit_mc_w(ptx::smem_u32(&bars->drain), kBoth);
      ptx::mbar_wait_cl_all(ptx::smem_u32(&bars->drain), 0, nullptr, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ second CTA's TMEM warp
    // Wait until the pair's MMAs have drained: they read this CTA's shared
    // memory and write its tensor memory.
    if (lane == 0) ptx::mbar_wait_cl(ptx::smem_u32(&bars->drain), 0, nullptr, kWaitLimitNs);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;                       // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;                // output row within the tile
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const int half = pg.hd / 2;
    bool ok = true;
    int lt = 0;
    const uint32_t acc_empty0 = ptx::cluster_addr(ptx::smem_u32(&bars->acc_empty[0]), 0);
    const uint32_t acc_empty1 = ptx::cluster_addr(ptx::smem_u32(&bars->acc_empty[1]), 0);
    for (int tile = pair; tile < n_tiles && ok; tile += n_pairs, ++lt) {
      const int buf = lt & 1;
      // This CTA's 128 rows of the pair's 256 x 256 tile, all 256 columns.
      const int m0 = (tile / n_nt) * kBM + kRowsCta * (int)rank, n0 = (tile % n_nt) * kBN;
      ok = ptx::mbar_wait_cl_all(ptx::smem_u32(&bars->acc_full[buf]), (lt >> 1) & 1, abort_flag, kWaitLimitNs);
      if (!ok) break;
      ptx::tc_fence_after();
      const int m = m0 + row;
      const bool live = m < pg.M;
      const int t = live ? m % pg.T : 0;
      __nv_bfloat16* qrow = qkv + (size_t)(live ? m : 0) * pg.N;
      __nv_bfloat16* rrow = rot ? rot + (size_t)(live ? m : 0) * pg.NQK : nullptr;
      // One head at a time: its columns [hb, hb + hd) of the tile.
      for (int hb = 0; hb < kBN && n0 + hb < pg.N; hb += pg.hd) {
        const int nh = n0 + hb;                          // the head's first output column
        const bool rotate = pg.rope && rrow != nullptr && nh < pg.NQK;
        // 32-column chunks c and c + hd/2 hold pair partners (NEOX); the
        // interleaved pairing keeps partners inside one chunk.
        for (int c = 0; c < half; c += 32) {
          uint32_t lo[32], hi[32];
          ptx::tmem_ld32(t_lane + buf * kBN + hb + c, lo);
          ptx::tmem_ld32(t_lane + buf * kBN + hb + half + c, hi);
          ptx::tmem_wait_ld();
          if (live) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              *reinterpret_cast<uint4*>(qrow + nh + c + 8 * q) =
                  make_uint4(pack_bf16x2(__uint_as_float(lo[8 * q]), __uint_as_float(lo[8 * q + 1])),
                             pack_bf16x2(__uint_as_float(lo[8 * q + 2]), __uint_as_float(lo[8 * q + 3])),
                             pack_bf16x2(__uint_as_float(lo[8 * q + 4]), __uint_as_float(lo[8 * q + 5])),
                             pack_bf16x2(__uint_as_float(lo[8 * q + 6]), __uint_as_float(lo[8 * q + 7])));
              *reinterpret_cast<uint4*>(qrow + nh + half + c + 8 * q) =
                  make_uint4(pack_bf16x2(__uint_as_float(hi[8 * q]), __uint_as_float(hi[8 * q + 1])),
                             pack_bf16x2(__uint_as_float(hi[8 * q + 2]), __uint_as_float(hi[8 * q + 3])),
                             pack_bf16x2(__uint_as_float(hi[8 * q + 4]), __uint_as_float(hi[8 * q + 5])),
                             pack_bf16x2(__uint_as_float(hi[8 * q + 6]), __uint_as_float(hi[8 * q + 7])));
            }
          }
          if (rotate && live) {
            if (!pg.interleaved) {
              // Pairs (c + e, c + e + hd/2), e < 32.
              uint32_t y0[16], y1[16];
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float a0, a1, b0, b1, s0, c0, s1, c1;
                __sincosf(rope_angle(t, pg.rope_f_hi[c + e], pg.rope_f_lo[c + e]), &s0, &c0);
                __sincosf(rope_angle(t, pg.rope_f_hi[c + e + 1], pg.rope_f_lo[c + e + 1]), &s1, &c1);
                rope_pair(__uint_as_float(lo[e]), __uint_as_float(hi[e]), c0, s0, a0, b0);
                rope_pair(__uint_as_float(lo[e + 1]), __uint_as_float(hi[e + 1]), c1, s1, a1, b1);
                y0[e / 2] = pack_bf16x2(a0, a1);
                y1[e / 2] = pack_bf16x2(b0, b1);
              }
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                *reinterpret_cast<uint4*>(rrow + nh + c + 8 * q) =
                    make_uint4(y0[4 * q], y0[4 * q + 1], y0[4 * q + 2], y0[4 * q + 3]);
                *reinterpret_cast<uint4*>(rrow + nh + half + c + 8 * q) =
                    make_uint4(y1[4 * q], y1[4 * q + 1], y1[4 * q + 2], y1[4 * q + 3]);
              }
            } else {
              // Pairs (2i, 2i+1) inside each chunk: chunk columns c .. c+31
              // (in lo) are pairs c/2 .. c/2+15, columns half + c .. (in hi)
              // pairs (half + c)/2 .. ; pair i goes to slots i, i + hd/2.
#pragma unroll
              for (int part = 0; part < 2; ++part) {
                const uint32_t* v = part ? hi : lo;
                const int p0 = (part ? half + c : c) / 2;  // first pair of this chunk
                uint32_t y0[8], y1[8];
#pragma unroll
                for (int k = 0; k < 16; k += 2) {
                  float a0, a1, b0, b1, s0, c0, s1, c1;
                  __sincosf(rope_angle(t, pg.rope_f_hi[p0 + k], pg.rope_f_lo[p0 + k]), &s0, &c0);
                  __sincosf(rope_angle(t, pg.rope_f_hi[p0 + k + 1], pg.rope_f_lo[p0 + k + 1]), &s1, &c1);
                  rope_pair(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]), c0, s0, a0, b0);
                  rope_pair(__uint_as_float(v[2 * k + 2]), __uint_as_float(v[2 * k + 3]), c1, s1, a1, b1);
                  y0[k / 2] = pack_bf16x2(a0, a1);
                  y1[k / 2] = pack_bf16x2(b0, b1);
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                  *reinterpret_cast<uint4*>(rrow + nh + p0 + 8 * q) =
                      make_uint4(y0[4 * q], y0[4 * q + 1], y0[4 * q + 2], y0[4 * q + 3]);
                  *reinterpret_cast<uint4*>(rrow + nh + half + p0 + 8 * q) =
                      make_uint4(y1[4 * q], y1[4 * q + 1], y1[4 * q + 2], y1[4 * q + 3]);
                }
              }
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      // Released on the first CTA's barrier (both CTAs' four warps).
      if (lane == 0) ptx::mbar_arrive_remote(buf ? acc_empty1 : acc_empty0);
    }
    if (!ok) fail();
  }
  ptx::tc_fence_before();
  __syncthreads();
  // Neither CTA releases its tensor or shared memory while the other may
  // still signal it.
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc2(tmem, 512);
  }
}

}  // namespace

// CTA pairs that can be resident at once (one CTA per SM), per device.
int proj_max_pairs() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreadsP);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, proj_kernel, &cfg) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

cudaError_t proj_launch(const ProjArgs& a, cudaStream_t stream) {
  const ProjGeometry& pg = a.pg;
  const int n_tiles = ((pg.M + kBM - 1) / kBM) * ((pg.N + kBN - 1) / kBN);
  cudaError_t e = cudaFuncSetAttribute(proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int max_pairs = proj_max_pairs();
  if (max_pairs <= 0) return cudaErrorLaunchOutOfResources;
  const int pairs = n_tiles < max_pairs ? n_tiles : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreadsP);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  prof_begin(kKernelProj, stream);
  e = cudaLaunchKernelEx(&cfg, proj_kernel, a.tm_x, a.tm_w, (__nv_bfloat16*)a.qkv, (__nv_bfloat16*)a.rot, pg,
                         a.status);
  prof_end(kKernelProj, stream);
  return e;
}

}  // namespace attn
