// Single-query (decode) attention over a KV cache: one new token per batch
// row attends to the cached keys and values 0 .. len-1 of its sequence.
//
// The per-position form of the method ("CUDA C microgpt",
// attention_forward_kernel: one query at position pos_id against keys
// 0 .. pos_id) with the grouped heads of "nanoeuler -- CUDA kernels" (query
// head h reads kv head h / (NH/NKV)).  Nothing here is a contraction worth a
// tensor core: each cached row is read once and used for a handful of dot
// products, so the kernels are bound by HBM bandwidth (4 FLOP per byte of
// bf16 cache at four query heads per kv head).
//
// Split over the cache length (flash-decoding): a CTA takes a chunk of cache
// rows (a multiple of 32, sized by a small wave-count cost model) of one kv
// head and up to kHeads of its query heads, keeps
// an online softmax per head, and writes a partial (max m, sum l, unnormalised
// output o) to the workspace; a second kernel merges the chunks of each
// (batch row, head) in chunk order, so the result is deterministic.
//
// Inside a CTA each warp walks blocks of 8 rows: lanes hold HD/32 elements of
// every row (coalesced 8-row loads of K and V), form the 8 x kHeads partial
// dot products, and reduce all 32 of them across the warp in one butterfly
// (31 shuffles; lane 4r + h ends with the full score of row r, head h).
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_profile.h"

#include <math.h>

namespace attn {
namespace {

constexpr int kTargetCtas = 152 * 3;   // one wave: 152 SMs, three CTAs each
constexpr int kHeads = 4;        // query heads per CTA (sharing one kv head)
constexpr int kWarpsD = 4;
constexpr int kThreadsD = 32 * kWarpsD;

// EPL consecutive elements of a row: loaded as one raw vector, widened to
// float where they are used.
template <typename T, int EPL> struct Vec;
template <> struct Vec<__nv_bfloat16, 4> {
  using Raw = uint2;
  static __device__ __forceinline__ Raw load(const __nv_bfloat16* p) { return *reinterpret_cast<const uint2*>(p); }
  static __device__ __forceinline__ void widen(Raw u, float (&x)[4]) {
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
  }
};
template <> struct Vec<__nv_bfloat16, 2> {
  using Raw = uint32_t;
  static __device__ __forceinline__ Raw load(const __nv_bfloat16* p) { return *reinterpret_cast<const uint32_t*>(p); }
  static __device__ __forceinline__ void widen(Raw u, float (&x)[2]) { x[0] = bf16_lo(u); x[1] = bf16_hi(u); }
};
template <> struct Vec<float, 4> {
  using Raw = float4;
  static __device__ __forceinline__ Raw load(const float* p) { return *reinterpret_cast<const float4*>(p); }
  static __device__ __forceinline__ void widen(Raw u, float (&x)[4]) { x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w; }
};
template <> struct Vec<float, 2> {
  using Raw = float2;
  static __device__ __forceinline__ Raw load(const float* p) { return *reinterpret_cast<const float2*>(p); }
  static __device__ __forceinline__ void widen(Raw u, float (&x)[2]) { x[0] = u.x; x[1] = u.y; }
};
__device__ __forceinline__ void store_elem(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store_elem(float* p, float v) { *p = v; }

__device__ __forceinline__ int clamp_len(const int* lens, int b, int max_len, int* status) {
  int n = lens[b];
  if (n < 1 || n > max_len) {
    record_status(status, kErrBadArgument);
    n = n < 1 ? 1 : max_len;
  }
  return n;
}

// Partial of one (batch row, head, chunk): m, l, then o[HD].  KH query heads
// per CTA: 4, or 1 when a kv head serves a single query head (each lane then
// reduces 8 partial sums instead of 32).
template <typename T, int HD, int KH>
__global__ void __launch_bounds__(kThreadsD, sizeof(T) == 2 ? 3 : 2)
decode_split_kernel(float* __restrict__ part, const T* __restrict__ q, const T* __restrict__ kc,
                    const T* __restrict__ vc, const int* __restrict__ lens, int NH, int NKV, int max_len,
                    int chunk, int n_split, float scale, int* status) {
  // The merge kernel is launched as a programmatic dependent; it waits for
  // this grid before reading the partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int EPL = HD / 32;
  // Per warp: the probabilities of a block of rows, then the heads' corrections.
  __shared__ __align__(16) float p_sh[kWarpsD][2][32];
  __shared__ float m_sh[kWarpsD][KH], l_sh[kWarpsD][KH];
  __shared__ float o_sh[kWarpsD][KH][HD];
  const int grp = NH / NKV, hgroups = (grp + KH - 1) / KH;
  const int s = blockIdx.x, kh = blockIdx.y / hgroups, hg = blockIdx.y % hgroups, b = blockIdx.z;
  const int h0 = kh * grp + hg * KH, gcnt = min(KH, grp - hg * KH);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int len = clamp_len(lens, b, max_len, status);
  const int r0 = s * chunk, r1 = min(r0 + chunk, len);

  // This lane's elements of the queries (heads past gcnt: zero).
  float qv[KH][EPL];
#pragma unroll
  for (int h = 0; h < KH; ++h) {
    if (h < gcnt) {
      Vec<T, EPL>::widen(Vec<T, EPL>::load(q + ((size_t)b * NH + h0 + h) * HD + lane * EPL), qv[h]);
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) qv[h][e] = 0.f;
    }
  }
  // Running state: m, l of head (lane % 4) (replicated over its 8 lanes; KH = 1:
  // all lanes hold head 0), and
  // this lane's elements of every head's unnormalised output.
  float m = -INFINITY, l = 0.f, o[KH][EPL];
#pragma unroll
  for (int h = 0; h < KH; ++h)
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[h][e] = 0.f;

  const size_t row_stride = (size_t)NKV * HD;
  const T* kbase = kc + ((size_t)b * max_len * NKV + kh) * HD + lane * EPL;
  const T* vbase = vc + ((size_t)b * max_len * NKV + kh) * HD + lane * EPL;
  // Blocks of 8 rows, one warp each in turn; the next block's K and V rows are
  // fetched (raw) before the current block is worked on.
  using Raw = typename Vec<T, EPL>::Raw;
  Raw kr[8], vr[8];
  auto fetch = [&](int base, Raw (&kk)[8], Raw (&vv)[8]) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (base + r < r1) {
        kk[r] = Vec<T, EPL>::load(kbase + (size_t)(base + r) * row_stride);
        vv[r] = Vec<T, EPL>::load(vbase + (size_t)(base + r) * row_stride);
      } else {
        kk[r] = Raw{};
        vv[r] = Raw{};
      }
    }
  };
  if (r0 + 8 * warp < r1) fetch(r0 + 8 * warp, kr, vr);
  for (int rb = r0 + 8 * warp; rb < r1; rb += 8 * kWarpsD) {
    Raw kn[8], vn[8];
    if (rb + 8 * kWarpsD < r1) fetch(rb + 8 * kWarpsD, kn, vn);
    // Partial dot products, value index KH r + h (rows widened one at a time).
    constexpr int NV = 8 * KH;
    float v[NV];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float kv[EPL];
      Vec<T, EPL>::widen(kr[r], kv);
#pragma unroll
      for (int h = 0; h < KH; ++h) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc = fmaf(qv[h][e], kv[e], acc);
        v[KH * r + h] = acc;
      }
    }
    // Butterfly: while a lane holds several values, the stage with offset o
    // keeps the half selected by its lane bit o and adds the partner's copy of
    // that half; once one value is left the stages just add.  Lane l ends
    // with value index l >> (5 - log2(NV)), i.e. row l / 4 and head l % 4
    // (KH = 4) or row l / 4 (KH = 1).
#pragma unroll
    for (int stage = 0; stage < 5; ++stage) {
      const int o2 = 16 >> stage, n = NV >> stage;   // compile-time once unrolled
      if (n > 1) {
        const bool upper = (lane & o2) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
          const float send = upper ? v[i] : v[i + n / 2];
          const float keep = upper ? v[i + n / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o2);
        }
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], o2);
      }
    }
    // Lane 4 r + h: score of row rb + r for head h (KH = 1: head 0 on all four).
    const int row = rb + lane / 4;
    const float sc = (row < r1) ? v[0] * scale : -INFINITY;
    float bm = sc;
    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
    const float m_new = fmaxf(m, bm);                  // finite: row rb < r1 is in the block
    const float corr = expf(m - m_new);                // 0 while m = -inf
    const float p = (row < r1) ? expf(sc - m_new) : 0.f;
    float ps = p;
    ps += __shfl_xor_sync(0xffffffffu, ps, 4);
    ps += __shfl_xor_sync(0xffffffffu, ps, 8);
    ps += __shfl_xor_sync(0xffffffffu, ps, 16);
    l = l * corr + ps;
    m = m_new;
    p_sh[warp][0][lane] = p;
    p_sh[warp][1][lane] = corr;
    __syncwarp();
#pragma unroll
    for (int h = 0; h < KH; ++h) {
      const float c = p_sh[warp][1][h];
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[h][e] *= c;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float4 pr = *reinterpret_cast<const float4*>(&p_sh[warp][0][4 * r]);
      const float pv[4] = {pr.x, pr.y, pr.z, pr.w};   // heads 0..3 (KH = 1: head 0 in pv[0])
      float vrow[EPL];
      Vec<T, EPL>::widen(vr[r], vrow);
#pragma unroll
      for (int h = 0; h < KH; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[h][e] = fmaf(pv[h], vrow[e], o[h][e]);
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      kr[r] = kn[r];
      vr[r] = vn[r];
    }
  }
  // Merge the warps: lanes 0..3 hold m, l of heads 0..3.
  if (lane < KH) {
    m_sh[warp][lane] = m;
    l_sh[warp][lane] = l;
  }
#pragma unroll
  for (int h = 0; h < KH; ++h)
#pragma unroll
    for (int e = 0; e < EPL; ++e) o_sh[warp][h][lane * EPL + e] = o[h][e];
  __syncthreads();
  for (int idx = threadIdx.x; idx < gcnt * (HD + 2); idx += kThreadsD) {
    const int h = idx / (HD + 2), c = idx % (HD + 2);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarpsD; ++w) M = fmaxf(M, m_sh[w][h]);
    float acc = 0.f;
    if (c == 0) {
      acc = M;
    } else {
#pragma unroll
      for (int w = 0; w < kWarpsD; ++w) {
        const float f = (M == -INFINITY) ? 0.f : expf(m_sh[w][h] - M);
        acc += f * (c == 1 ? l_sh[w][h] : o_sh[w][h][c - 2]);
      }
    }
    part[(((size_t)b * NH + h0 + h) * n_split + s) * (HD + 2) + c] = acc;
  }
}

// out[b,h,:] and lse[b,h] from the chunks of (b, h), merged in a fixed order.
// 4 x HD threads: the chunk maxima and sums are read in parallel and reduced
// through shared memory; thread group g sums chunks g, g+4, ... of each
// output element, and the four group sums are added in group order.
constexpr int kMergeGroups = 4;
template <typename T, int HD>
__global__ void __launch_bounds__(kMergeGroups * HD)
decode_merge_kernel(T* __restrict__ out, float* __restrict__ lse, const float* __restrict__ part,
                    const int* __restrict__ lens, int NH, int max_len, int chunk, int n_split, int* status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int NT = kMergeGroups * HD;
  __shared__ float red[NT];
  __shared__ float o_part[kMergeGroups][HD];
  __shared__ float M_sh, L_sh;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int len = clamp_len(lens, b, max_len, status);
  const int n_used = (len + chunk - 1) / chunk;
  const float* pp = part + ((size_t)b * NH + h) * n_split * (HD + 2);
  // Maximum of the chunk maxima.
  float mx = -INFINITY;
  for (int s = tid; s < n_used; s += NT) mx = fmaxf(mx, pp[s * (HD + 2)]);
  red[tid] = mx;
  __syncthreads();
  for (int w = NT / 2; w > 0; w >>= 1) {
    if (tid < w) red[tid] = fmaxf(red[tid], red[tid + w]);
    __syncthreads();
  }
  if (tid == 0) M_sh = red[0];
  __syncthreads();
  const float M = M_sh;
  // Sum of the rescaled chunk sums (a fixed tree: deterministic).
  float ls = 0.f;
  for (int s = tid; s < n_used; s += NT) ls = fmaf(expf(pp[s * (HD + 2)] - M), pp[s * (HD + 2) + 1], ls);
  red[tid] = ls;
  __syncthreads();
  for (int w = NT / 2; w > 0; w >>= 1) {
    if (tid < w) red[tid] += red[tid + w];
    __syncthreads();
  }
  if (tid == 0) L_sh = red[0];
  // Output elements: group g takes chunks g, g + 4, ...
  const int grp_id = tid / HD, d = tid % HD;
  float o = 0.f;
#pragma unroll 4
  for (int s = grp_id; s < n_used; s += kMergeGroups)
    o = fmaf(expf(pp[s * (HD + 2)] - M), pp[s * (HD + 2) + 2 + d], o);
  o_part[grp_id][d] = o;
  __syncthreads();
  if (tid < HD) {
    float acc = 0.f;
#pragma unroll
    for (int g2 = 0; g2 < kMergeGroups; ++g2) acc += o_part[g2][tid];
    const float L = L_sh;
    store_elem(out + ((size_t)b * NH + h) * HD + tid, acc / L);
    if (tid == 0) lse[(size_t)b * NH + h] = M + logf(L);
  }
}

template <typename T, int HD>
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const int grp = a.NH / a.NKV, hgroups = (grp + kHeads - 1) / kHeads;   // grp 1: one group either way
  const int chunk = decode_chunk_rows(a.B, a.NH, a.NKV, a.max_len);
  const int n_split = (a.max_len + chunk - 1) / chunk;
  const float scale = (float)(1.0 / sqrt((double)HD));
  prof_begin(kKernelDecode, stream);
  const dim3 grid(n_split, a.NKV * hgroups, a.B);
  if (grp == 1)
    decode_split_kernel<T, HD, 1><<<grid, kThreadsD, 0, stream>>>(
        a.part, (const T*)a.q, (const T*)a.k_cache, (const T*)a.v_cache, a.lens, a.NH, a.NKV, a.max_len, chunk,
        n_split, scale, a.status);
  else
    decode_split_kernel<T, HD, kHeads><<<grid, kThreadsD, 0, stream>>>(
        a.part, (const T*)a.q, (const T*)a.k_cache, (const T*)a.v_cache, a.lens, a.NH, a.NKV, a.max_len, chunk,
        n_split, scale, a.status);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess)
    e = launch_pdl(decode_merge_kernel<T, HD>, dim3(a.NH, a.B), dim3(kMergeGroups * HD), 0, stream, (T*)a.out, a.lse,
                   (const float*)a.part, a.lens, a.NH, a.max_len, chunk, n_split, a.status);
  prof_end(kKernelDecode, stream);
  return e;
}

}  // namespace

// Cache rows per chunk: a multiple of 32 (four warps x 8-row blocks), from a
// small cost model: the split grid runs in waves of kTargetCtas CTAs, a CTA
// costs its rows plus a fixed ~96 rows' worth (queries, merge of its warps,
// partial store), and the merge kernel ~2 rows' worth per chunk.  Too few
// chunks leave SMs idle (a grid of slightly more than one wave waits on its
// tail); too many make CTAs mostly overhead.
int decode_chunk_rows(int B, int NH, int NKV, int max_len) {
  const long long hgroups = (NH / NKV + kHeads - 1) / kHeads;
  const long long units = (long long)B * NKV * hgroups;             // CTAs per chunk index
  long long best_chunk = ((long long)max_len + 31) / 32 * 32, best_cost = -1;
  // Candidate split counts 1, 2, 3, ... growing by about 1/8 each step.
  for (long long want = 1; want <= ((long long)max_len + 31) / 32; want += (want + 7) / 8) {
    const long long chunk = (((long long)max_len + want - 1) / want + 31) / 32 * 32;
    const long long n_split = ((long long)max_len + chunk - 1) / chunk;
    const long long waves = (units * n_split + kTargetCtas - 1) / kTargetCtas;
    const long long cost = waves * (chunk + 96) + 2 * n_split;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_chunk = chunk;
    }
  }
  return (int)best_chunk;
}

size_t decode_workspace_floats(int B, int NH, int NKV, int hd, int max_len) {
  const int chunk = decode_chunk_rows(B, NH, NKV, max_len);
  return (size_t)B * NH * ((max_len + chunk - 1) / chunk) * (hd + 2);
}

cudaError_t decode_launch(const DecodeArgs& a, cudaStream_t stream) {
  if (a.bf16) return a.hd == 128 ? launch_decode<__nv_bfloat16, 128>(a, stream)
                                 : launch_decode<__nv_bfloat16, 64>(a, stream);
  return a.hd == 128 ? launch_decode<float, 128>(a, stream) : launch_decode<float, 64>(a, stream);
}

}  // namespace attn
