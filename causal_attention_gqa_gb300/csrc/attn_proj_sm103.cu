// QKV projection with the RoPE rotation fused into its epilogue (bf16,
// tcgen05, persistent).
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
// Tiles of 128 x 256 outputs; x and w tiles of 64 columns (one 128-byte
// swizzle atom) through a 4-stage TMA ring; one issuing thread runs
// M=128, N=256, K=16 MMAs into one of two TMEM accumulators (256 columns
// each), so the epilogue of a tile (four warps, one output row per thread)
// overlaps the next tile's MMAs.
//
//   warp 0      TMA producer
//   warp 1      TMEM owner and MMA issuer
//   warps 2-5   epilogue: TMEM -> bf16 qkv rows, rotated Q/K rows
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_profile.h"
#include "attn_ptx.cuh"

namespace attn {
namespace {

constexpr uint64_t kWaitLimitNs = 1000000000ull;
#ifndef PROJ_BK
#define PROJ_BK 64
#endif
#ifndef PROJ_STAGES
#define PROJ_STAGES 4
#endif
constexpr int kBM = 128, kBN = 256, kBK = PROJ_BK, kStages = PROJ_STAGES;
constexpr int kAtoms = kBK / 64;                    // 64-column swizzle atoms per k-block
constexpr int kAAtom = kBM * 128, kBAtom = kBN * 128;
constexpr int kATile = kBM * kBK * 2;
constexpr int kBTile = kBN * kBK * 2;
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
  const int n_mt = (pg.M + kBM - 1) / kBM, n_nt = (pg.N + kBN - 1) / kBN, n_tiles = n_mt * n_nt;
  const int n_kb = (pg.Cm + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars->acc_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->acc_empty[i]), 4);
    }
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_x);
      ptx::tma_prefetch_desc(&tm_w);
      bool ok = true;
      int it = 0;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int m0 = (tile / n_nt) * kBM, n0 = (tile % n_nt) * kBN;
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % kStages, u = it / kStages;
          if (u > 0 && !(ok = ptx::mbar_wait(ptx::smem_u32(&bars->empty[st]), (u - 1) & 1, abort_flag,
                                             kWaitLimitNs)))
            break;
          const uint32_t fb = ptx::smem_u32(&bars->full[st]);
          ptx::mbar_arrive_expect_tx(fb, kStageBytes);
          uint8_t* sa = smem + st * kStageBytes;
#pragma unroll
          for (int a = 0; a < kAtoms; ++a) {
            ptx::tma_load_3d(ptx::smem_u32(sa + a * kAAtom), &tm_x, kb * kBK + 64 * a, m0, 0, fb);
            ptx::tma_load_3d(ptx::smem_u32(sa + kATile + a * kBAtom), &tm_w, kb * kBK + 64 * a, n0, 0, fb);
          }
        }
      }
      if (!ok) fail();
      if (*abort_flag) {
        // Let the copies in flight land before shared memory is released.
        for (int st = 0; st < kStages && st < it; ++st)
          ptx::mbar_wait(ptx::smem_u32(&bars->full[st]), ((it - 1 - st) / kStages) & 1, nullptr, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp runs the issue loop; one elected lane issues each MMA
    // and commit, and every wait is warp-collective)
    {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBM, kBN, false, false);
      const uint64_t d0 = ptx::sw128_desc(ptx::smem_u32(smem), 16, 1024);
      bool ok = true;
      int it = 0, lt = 0;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++lt) {
        const int buf = lt & 1;
        // The accumulator's previous tile (two back) has been read out.
        if (lt >= 2 &&
            !(ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->acc_empty[buf]), ((lt >> 1) - 1) & 1, abort_flag,
                                  kWaitLimitNs)))
          break;
        ptx::tc_fence_after();
        // Each stage's barrier is checked (non-blocking) one k-block ahead.
        uint32_t ready =
            __all_sync(0xffffffffu, ptx::mbar_test(ptx::smem_u32(&bars->full[it % kStages]), (it / kStages) & 1) != 0);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % kStages, u = it / kStages;
          if (!ready && !(ok = ptx::mbar_wait_all(ptx::smem_u32(&bars->full[st]), u & 1, abort_flag, kWaitLimitNs)))
            break;
          ptx::tc_fence_after();
          ready = (kb + 1 < n_kb) ? __all_sync(0xffffffffu, ptx::mbar_test(ptx::smem_u32(&bars->full[(it + 1) % kStages]),
                                                                            ((it + 1) / kStages) & 1) != 0)
                                  : 1u;
          const uint64_t da = ptx::desc_advance(d0, st * kStageBytes);
          const uint64_t db = ptx::desc_advance(d0, st * kStageBytes + kATile);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            ptx::mma_bf16_ss_w(tmem + buf * kBN, ptx::desc_advance(da, (kk >> 2) * kAAtom + (kk & 3) * 32),
                             ptx::desc_advance(db, (kk >> 2) * kBAtom + (kk & 3) * 32), idesc,
                             (kb > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit_w(ptx::smem_u32(&bars->empty[st]));
        }
        if (!ok) break;
        ptx::mma_commit_w(ptx::smem_u32(&bars->acc_full[buf]));
      }
      if (!ok) fail();
      ptx::mma_commit_w(ptx::smem_u32(&bars->drain));
      ptx::mbar_wait_all(ptx::smem_u32(&bars->drain), 0, nullptr, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;                       // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;                // output row within the tile
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const int half = pg.hd / 2;
    bool ok = true;
    int lt = 0;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++lt) {
      const int buf = lt & 1;
      const int m0 = (tile / n_nt) * kBM, n0 = (tile % n_nt) * kBN;
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(&bars->acc_full[buf]), (lt >> 1) & 1, abort_flag,
                                                  kWaitLimitNs));
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
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->acc_empty[buf]));
    }
    if (!ok) fail();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t proj_launch(const ProjArgs& a, cudaStream_t stream) {
  const ProjGeometry& pg = a.pg;
  const int n_tiles = ((pg.M + kBM - 1) / kBM) * ((pg.N + kBN - 1) / kBN);
  const int grid = n_tiles < a.num_sms ? n_tiles : a.num_sms;
  cudaError_t e = cudaFuncSetAttribute(proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  prof_begin(kKernelProj, stream);
  proj_kernel<<<grid, kThreadsP, kSmemBytes, stream>>>(a.tm_x, a.tm_w, (__nv_bfloat16*)a.qkv,
                                                       (__nv_bfloat16*)a.rot, pg, a.status);
  prof_end(kKernelProj, stream);
  return cudaGetLastError();
}

}  // namespace attn
