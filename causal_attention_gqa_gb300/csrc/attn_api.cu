// C ABI of the attention library (declared in include/attn_gb300.h).
//
// Host-side argument validation, TMA tensor-map encoding, workspace carving
// and kernel dispatch.  Every entry point validates before it enqueues
// anything; nothing here allocates device memory or synchronises (except the
// explicitly synchronous status / self-test calls).
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn_gb300.h"
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_ptx.cuh"

namespace attn {
namespace {

__device__ int g_status;           // first device-side error since the last reset
__device__ int g_selftest_status;  // result of attn_selftest_wait_timeout

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};

int* status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

int g_num_sms[kMaxDevices] = {};

// Streaming multiprocessors of the current device (persistent grid size).
int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_num_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D bf16 tensor map over a row-major [B, T, width] array, box {64, rows, 1},
// 128-byte swizzle; rows past T read as zeros.
bool make_tmap(CUtensorMap* m, const void* base, int width, int T, int B, int rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * (cuuint64_t)T};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte (e4m3) tensor of d0 x d1 x d2 elements, rows of d0 bytes, 128 x 128 boxes.
bool make_tmap_u8(CUtensorMap* m, const void* base, int d0, int d1, int d2) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  cuuint64_t strides[2] = {(cuuint64_t)d0, (cuuint64_t)d0 * (cuuint64_t)d1};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// `dtype` may carry ATTN_FLAG_ROPE_INTERLEAVED; it is stripped here (the
// element type stays in `dtype`) and recorded in the geometry.
int check_shape(int B, int T, int C, int NH, int NKV, float rope_theta, int& dtype, Geometry* g) {
  const int flags = dtype & ~0xFF;
  if (flags & ~ATTN_FLAG_ROPE_INTERLEAVED) return ATTN_ERR_BAD_ARGUMENT;
  dtype &= 0xFF;
  if (B < 1 || T < 1 || C < 1 || NH < 1 || NKV < 1) return ATTN_ERR_BAD_SHAPE;
  if (C % NH != 0 || NH % NKV != 0) return ATTN_ERR_BAD_SHAPE;
  if (!std::isfinite(rope_theta)) return ATTN_ERR_BAD_ARGUMENT;
  const int hd = C / NH;
  const bool rope = rope_theta > 0.f;
  if (rope && hd % 2 != 0) return ATTN_ERR_BAD_SHAPE;
  const long long W = (long long)(NH + 2 * NKV) * hd;
  if ((long long)B * T > INT_MAX / 8 || (long long)B * T * NH > INT_MAX || W > INT_MAX / 4 ||
      (long long)T > (1LL << 24))
    return ATTN_ERR_BAD_SHAPE;
  switch (dtype) {
    case ATTN_DTYPE_F32:
    case ATTN_DTYPE_TF32:   // float32 storage and the 1e-4 bar: the exact float32 kernels
      if (hd > 128) return ATTN_ERR_UNSUPPORTED;
      break;
    case ATTN_DTYPE_BF16:
      if (hd != 64 && hd != 128) return ATTN_ERR_UNSUPPORTED;
      if ((long long)((T + 127) / 128) * B * NH > INT_MAX) return ATTN_ERR_BAD_SHAPE;
      break;
    default:
      return ATTN_ERR_BAD_ARGUMENT;
  }
  g->B = B;
  g->T = T;
  g->C = C;
  g->NH = NH;
  g->NKV = NKV;
  g->hd = hd;
  g->grp = NH / NKV;
  g->W = (int)W;
  g->scale = (float)(1.0 / std::sqrt((double)hd));
  g->rope_theta = rope ? rope_theta : 0.f;
  g->rope_interleaved = (rope && (flags & ATTN_FLAG_ROPE_INTERLEAVED)) ? 1 : 0;
  for (int i = 0; i < 64; ++i) {
    double f = 0.0;
    if (rope && i < hd / 2) f = std::exp(-2.0 * i * std::log((double)rope_theta) / hd);
    g->rope_f_hi[i] = (float)f;
    g->rope_f_lo[i] = (float)(f - (double)g->rope_f_hi[i]);
  }
  return ATTN_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Leading part of the workspace: float32 row dots [B,NH,T] (F32), or the
// bf16 path's two row tables per (b, h), Tp floats each.
size_t row_part_bytes(const Geometry& g, int dtype) {
  if (dtype == ATTN_DTYPE_BF16) return align256((size_t)g.B * g.NH * row_table_rows(g.T) * 2 * sizeof(float));
  return align256((size_t)g.B * g.NH * g.T * sizeof(float));
}

// bf16: row tables, then the rotated Q/K copy, then 256 bytes for the dQ
// kernel's work-item counter.
size_t rot_part_bytes(const Geometry& g) { return align256((size_t)g.B * g.T * (g.NH + g.NKV) * g.hd * 2); }

// bf16: after the counter, the RoPE angle table [hd/2][T] of (cos, sin) float
// pairs the prologue writes for the gradient epilogues (reserved whether or
// not RoPE is on: the size query takes no rope_theta).
size_t rope_table_bytes(const Geometry& g) { return align256((size_t)g.T * g.hd * sizeof(float)); }

// dtype TF32 on tensor cores (head size 64): bf16 hi/lo parts of qkv (and,
// for the backward, of dout), each array rounded up to 256 bytes.
bool split_path(const Geometry& g, int dtype) { return dtype == ATTN_DTYPE_TF32 && split_supported(g); }
size_t split_part_bytes(const Geometry& g, int width) { return align256((size_t)g.B * g.T * width * 2); }
size_t split_table_bytes(const Geometry& g) { return align256((size_t)g.B * g.NH * row_table_rows(g.T) * 2 * 4); }

size_t workspace_bytes(const Geometry& g, int dtype) {
  if (split_path(g, dtype))
    return split_table_bytes(g) + 2 * split_part_bytes(g, g.W) + 2 * split_part_bytes(g, g.C);
  size_t bytes = row_part_bytes(g, dtype);
  if (dtype == ATTN_DTYPE_BF16) bytes += rot_part_bytes(g) + 256 + rope_table_bytes(g);
  return bytes;
}

// Tensor maps of the split path: the qkv parts at `qkv_parts` (hi, then lo),
// and, when `dout_parts` is set, the dout parts there (hi, then lo).
bool split_maps(SplitArgs* a, uint8_t* qkv_parts, uint8_t* dout_parts) {
  const Geometry& g = a->g;
  a->qkv_hi = reinterpret_cast<__nv_bfloat16*>(qkv_parts);
  a->qkv_lo = reinterpret_cast<__nv_bfloat16*>(qkv_parts + split_part_bytes(g, g.W));
  if (!make_tmap(&a->tm_hi, a->qkv_hi, g.W, g.T, g.B) || !make_tmap(&a->tm_lo, a->qkv_lo, g.W, g.T, g.B))
    return false;
  if (!dout_parts) return true;
  a->dout_hi = reinterpret_cast<__nv_bfloat16*>(dout_parts);
  a->dout_lo = reinterpret_cast<__nv_bfloat16*>(dout_parts + split_part_bytes(g, g.C));
  return make_tmap(&a->tm_dohi, a->dout_hi, g.C, g.T, g.B) && make_tmap(&a->tm_dolo, a->dout_lo, g.C, g.T, g.B);
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// One block waits on an mbarrier nobody arrives on; the bounded wait must
// expire, record the timeout and let the kernel exit.
__global__ void wait_timeout_selftest_kernel(int* result, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const bool ok = ptx::mbar_wait(ptx::smem_u32(&bar), 0, &abort_flag, limit_ns);
  if (!ok && threadIdx.x == 0) record_status(result, kErrDeviceTimeout);
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_abi_version(void) { return 1; }

extern "C" const char* attn_strerror(int status) {
  switch (status) {
    case ATTN_OK: return "success";
    case ATTN_ERR_NULL_POINTER: return "a required pointer is NULL";
    case ATTN_ERR_BAD_SHAPE: return "invalid shape (B,T,C,NH,NKV; C%NH, NH%NKV, odd head size with RoPE, or size limits)";
    case ATTN_ERR_UNSUPPORTED: return "unsupported (dtype, head size) combination";
    case ATTN_ERR_MISALIGNED: return "a pointer is not 16-byte aligned";
    case ATTN_ERR_WORKSPACE: return "workspace missing or smaller than the *_workspace_bytes() size";
    case ATTN_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a device-side bounded wait expired";
    case ATTN_ERR_BAD_ARGUMENT: return "invalid argument";
    default: return "unknown status";
  }
}

namespace {

// Forward shared by attn_fwd (workspace == NULL: RoPE rotated inside the
// attention kernel) and attn_fwd_ws (bf16 with RoPE: one rotation pass writes
// the rotated Q/K copy into the workspace, and the attention kernel reads Q
// and K from there).
int fwd_impl(void* out, float* lse, const void* qkv, int B, int T, int C, int NH, int NKV, float rope_theta,
             int dtype, void* workspace, size_t ws_bytes, void* stream, bool rotated_given = false) {
  Geometry g;
  int st = check_shape(B, T, C, NH, NKV, rope_theta, dtype, &g);
  if (st != ATTN_OK) return st;
  if (!out || !lse || !qkv) return ATTN_ERR_NULL_POINTER;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (split_path(g, dtype) && workspace != nullptr) {
    // float32 tensors on the tensor cores: hi/lo parts in the workspace.
    if (!aligned16(out) || !aligned16(qkv) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return ATTN_ERR_MISALIGNED;
    SplitArgs a{};
    a.g = g;
    a.qkv = qkv;
    a.out = out;
    a.lse = lse;
    a.status = status_word();
    if (!a.status || !split_maps(&a, static_cast<uint8_t*>(workspace), nullptr)) return ATTN_ERR_CUDA;
    return from_cuda(split_fwd_launch(a, s));
  }
  if (dtype == ATTN_DTYPE_F32 || dtype == ATTN_DTYPE_TF32) {
    if ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(qkv)) & 3u)
      return ATTN_ERR_MISALIGNED;
    SimtArgs a{};
    a.g = g;
    a.forward = true;
    a.out = out;
    a.lse = lse;
    a.qkv = qkv;
    return from_cuda(simt_launch(a, s));
  }
  if (!aligned16(out) || !aligned16(qkv) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_MISALIGNED;
  const bool pre_rotate = workspace != nullptr && g.rope_theta > 0.f;
  if (pre_rotate && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTN_ERR_MISALIGNED;
  Tc05FwdArgs a{};
  a.g = g;
  a.out = out;
  a.lse = lse;
  a.status = status_word();
  a.num_sms = num_sms();
  a.pre_rotated = pre_rotate;
  if (!a.status || a.num_sms <= 0) return ATTN_ERR_CUDA;
  const void* qk_src = pre_rotate ? workspace : qkv;
  const int qk_width = pre_rotate ? (g.NH + g.NKV) * g.hd : g.W;
  if (!make_tmap(&a.tm_qk, qk_src, qk_width, g.T, g.B) || !make_tmap(&a.tm_v, qkv, g.W, g.T, g.B) ||
      !make_tmap(&a.tm_out, out, g.C, g.T, g.B))
    return ATTN_ERR_CUDA;
  if (pre_rotate && !rotated_given) {
    cudaError_t e = launch_rope_qk_bf16(workspace, qkv, g, s);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return from_cuda(tc05_fwd_launch(a, s));
}

}  // namespace

extern "C" int attn_fwd(void* out, float* lse, const void* qkv, int B, int T, int C, int NH, int NKV,
                        float rope_theta, int dtype, void* stream) {
  return fwd_impl(out, lse, qkv, B, T, C, NH, NKV, rope_theta, dtype, nullptr, 0, stream);
}

extern "C" size_t attn_fwd_workspace_bytes(int B, int T, int C, int NH, int NKV, int dtype) {
  Geometry g;
  if (check_shape(B, T, C, NH, NKV, 0.f, dtype, &g) != ATTN_OK) return 0;
  if (split_path(g, dtype)) return 2 * split_part_bytes(g, g.W);
  if (dtype != ATTN_DTYPE_BF16) return 0;
  return align256((size_t)g.B * g.T * (g.NH + g.NKV) * g.hd * 2);
}

extern "C" int attn_fwd_ws(void* out, float* lse, const void* qkv, int B, int T, int C, int NH, int NKV,
                           float rope_theta, int dtype, void* workspace, size_t ws_bytes, void* stream) {
  Geometry g;
  int type = dtype;   // dtype keeps its flags for fwd_impl
  int st = check_shape(B, T, C, NH, NKV, rope_theta, type, &g);
  if (st != ATTN_OK) return st;
  const size_t need = attn_fwd_workspace_bytes(B, T, C, NH, NKV, type);
  if (need > 0 && (!workspace || ws_bytes < need)) return ATTN_ERR_WORKSPACE;
  return fwd_impl(out, lse, qkv, B, T, C, NH, NKV, rope_theta, dtype, need > 0 ? workspace : nullptr, ws_bytes,
                  stream);
}

extern "C" size_t attn_bwd_workspace_bytes(int B, int T, int C, int NH, int NKV, int dtype) {
  Geometry g;
  if (check_shape(B, T, C, NH, NKV, 0.f, dtype, &g) != ATTN_OK) return 0;
  return workspace_bytes(g, dtype);
}

namespace {

// Backward shared by attn_bwd (qk_rot == NULL: with RoPE the prologue rotates
// Q/K into the workspace) and attn_bwd_rot (qk_rot: the rotated copy an
// attn_fwd_ws call left in its workspace).
int bwd_impl(void* dqkv, const void* qkv, const void* out, const void* dout, const float* lse, int B, int T, int C,
             int NH, int NKV, float rope_theta, int dtype, const void* qk_rot, void* workspace, size_t ws_bytes,
             void* stream) {
  Geometry g;
  int st = check_shape(B, T, C, NH, NKV, rope_theta, dtype, &g);
  if (st != ATTN_OK) return st;
  if (!dqkv || !qkv || !out || !dout || !lse) return ATTN_ERR_NULL_POINTER;
  if (!workspace || ws_bytes < workspace_bytes(g, dtype)) return ATTN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* Drow = static_cast<float*>(workspace);
  if (split_path(g, dtype)) {
    // float32 tensors on the tensor cores; with qk_rot (the workspace of the
    // attn_fwd_ws call, which holds the hi/lo parts of this qkv) the parts are
    // not formed again.
    if (!aligned16(dqkv) || !aligned16(qkv) || !aligned16(out) || !aligned16(dout) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(qk_rot) & 255u))
      return ATTN_ERR_MISALIGNED;
    SplitArgs a{};
    a.g = g;
    a.qkv = qkv;
    a.dout = dout;
    a.out = const_cast<void*>(out);
    a.lse = const_cast<float*>(lse);
    a.dqkv = dqkv;
    a.LD = static_cast<float*>(workspace);
    a.status = status_word();
    uint8_t* ws = static_cast<uint8_t*>(workspace) + split_table_bytes(g);
    uint8_t* dout_parts = ws + 2 * split_part_bytes(g, g.W);
    a.qkv_given = qk_rot != nullptr;
    uint8_t* qkv_parts = a.qkv_given ? static_cast<uint8_t*>(const_cast<void*>(qk_rot)) : ws;
    if (!a.status || !split_maps(&a, qkv_parts, dout_parts)) return ATTN_ERR_CUDA;
    return from_cuda(split_bwd_launch(a, s));
  }
  if (dtype == ATTN_DTYPE_F32 || dtype == ATTN_DTYPE_TF32) {
    if ((reinterpret_cast<uintptr_t>(dqkv) | reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(out) |
         reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(lse)) & 3u)
      return ATTN_ERR_MISALIGNED;
    cudaError_t e = launch_row_dot(Drow, out, dout, g, false, s);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    SimtArgs a{};
    a.g = g;
    a.forward = false;
    a.lse = const_cast<float*>(lse);
    a.qkv = qkv;
    a.dqkv = dqkv;
    a.dout = dout;
    a.Drow = Drow;
    return from_cuda(simt_launch(a, s));
  }
  if (!aligned16(dqkv) || !aligned16(qkv) || !aligned16(out) || !aligned16(dout) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return ATTN_ERR_MISALIGNED;
  const bool rope = g.rope_theta > 0.f;
  const bool reuse = rope && qk_rot != nullptr;
  if (reuse && (reinterpret_cast<uintptr_t>(qk_rot) & 255u)) return ATTN_ERR_MISALIGNED;
  Tc05BwdArgs a{};
  a.g = g;
  a.dqkv = dqkv;
  a.LD = static_cast<const float*>(workspace);
  a.status = status_word();
  a.num_sms = num_sms();
  if (!a.status || a.num_sms <= 0) return ATTN_ERR_CUDA;
  // With RoPE, Q and K are read from a rotated copy (the caller's, or one the
  // prologue writes into the workspace); its layout keeps query head h at
  // column h*hd and kv head kh at C + kh*hd.
  void* rot = static_cast<uint8_t*>(workspace) + row_part_bytes(g, dtype);
  a.item_counter = reinterpret_cast<int*>(static_cast<uint8_t*>(rot) + rot_part_bytes(g));
  float* rope_cs = reinterpret_cast<float*>(static_cast<uint8_t*>(rot) + rot_part_bytes(g) + 256);
  a.rope_cs = rope_cs;
  const void* qk_src = !rope ? qkv : (reuse ? qk_rot : rot);
  const int qk_width = rope ? (g.NH + g.NKV) * g.hd : g.W;
  for (int r = 0; r < 2; ++r) {
    const int rows = r ? 128 : 64;
    if (!make_tmap(&a.tm_qk[r], qk_src, qk_width, g.T, g.B, rows) ||
        !make_tmap(&a.tm_v[r], qkv, g.W, g.T, g.B, rows) || !make_tmap(&a.tm_do[r], dout, g.C, g.T, g.B, rows))
      return ATTN_ERR_CUDA;
  }
  if (!make_tmap(&a.tm_dqkv, dqkv, g.W, g.T, g.B, 128)) return ATTN_ERR_CUDA;
  cudaError_t e = launch_bwd_prologue_bf16(static_cast<float*>(workspace), rope && !reuse ? rot : nullptr,
                                           a.item_counter, rope ? rope_cs : nullptr, out, dout, lse, qkv, g, s);
  if (e == cudaSuccess) e = tc05_bwd_launch(a, s);
  return from_cuda(e);
}

}  // namespace

extern "C" int attn_bwd(void* dqkv, const void* qkv, const void* out, const void* dout, const float* lse, int B,
                        int T, int C, int NH, int NKV, float rope_theta, int dtype, void* workspace,
                        size_t ws_bytes, void* stream) {
  return bwd_impl(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, rope_theta, dtype, nullptr, workspace, ws_bytes,
                  stream);
}

extern "C" int attn_bwd_rot(void* dqkv, const void* qkv, const void* out, const void* dout, const float* lse, int B,
                            int T, int C, int NH, int NKV, float rope_theta, int dtype, const void* qk_rot,
                            void* workspace, size_t ws_bytes, void* stream) {
  return bwd_impl(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, rope_theta, dtype, qk_rot, workspace, ws_bytes,
                  stream);
}

// ---------------------------------------------------------------- FP8 forward
namespace {
struct Fp8Layout {
  size_t qk8, vt8, deq_qk, deq_v, vtile_amax, total;
  int Tp;
};
Fp8Layout fp8_layout(const Geometry& g) {
  Fp8Layout L;
  const int n_qt = (g.T + 127) / 128;
  L.Tp = n_qt * 128;
  const size_t heads = (size_t)(g.NH + g.NKV);
  L.qk8 = 0;
  L.vt8 = L.qk8 + align256((size_t)g.B * g.T * heads * g.hd);
  L.deq_qk = L.vt8 + align256((size_t)g.B * g.NKV * g.hd * L.Tp);
  L.deq_v = L.deq_qk + align256((size_t)g.B * heads * n_qt * sizeof(float));
  L.vtile_amax = L.deq_v + align256((size_t)g.B * g.NKV * sizeof(float));
  L.total = L.vtile_amax + align256((size_t)g.B * g.NKV * n_qt * sizeof(float));
  return L;
}
}  // namespace

extern "C" size_t attn_fwd_fp8_workspace_bytes(int B, int T, int C, int NH, int NKV, int dtype) {
  Geometry g;
  if (check_shape(B, T, C, NH, NKV, 0.f, dtype, &g) != ATTN_OK || dtype != ATTN_DTYPE_BF16) return 0;
  if (!fp8_fwd_supported(g)) return 0;
  return fp8_layout(g).total;
}

extern "C" int attn_fwd_fp8(void* out, float* lse, const void* qkv, int B, int T, int C, int NH, int NKV,
                            float rope_theta, int dtype, void* workspace, size_t ws_bytes, void* stream) {
  Geometry g;
  int type = dtype;
  int st = check_shape(B, T, C, NH, NKV, rope_theta, type, &g);
  if (st != ATTN_OK) return st;
  if (type != ATTN_DTYPE_BF16 || !fp8_fwd_supported(g)) return ATTN_ERR_UNSUPPORTED;
  if (!out || !lse || !qkv) return ATTN_ERR_NULL_POINTER;
  if (!aligned16(out) || !aligned16(qkv) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_MISALIGNED;
  const Fp8Layout L = fp8_layout(g);
  if (!workspace || ws_bytes < L.total) return ATTN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_MISALIGNED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Fp8FwdArgs a{};
  a.g = g;
  a.qkv = qkv;
  a.qk8 = ws + L.qk8;
  a.vt8 = ws + L.vt8;
  a.deq_qk = reinterpret_cast<float*>(ws + L.deq_qk);
  a.deq_v = reinterpret_cast<float*>(ws + L.deq_v);
  a.vtile_amax = reinterpret_cast<float*>(ws + L.vtile_amax);
  a.Tp = L.Tp;
  a.lse = lse;
  a.status = status_word();
  a.num_sms = num_sms();
  if (!a.status || a.num_sms <= 0) return ATTN_ERR_CUDA;
  if (!make_tmap_u8(&a.tm_qk8, a.qk8, (g.NH + g.NKV) * g.hd, g.T, g.B) ||
      !make_tmap_u8(&a.tm_vt, a.vt8, L.Tp, g.hd, g.B * g.NKV) || !make_tmap(&a.tm_out, out, g.C, g.T, g.B))
    return ATTN_ERR_CUDA;
  return from_cuda(fp8_fwd_launch(a, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- QKV projection
extern "C" int attn_qkv_proj(void* qkv, void* qk_rot, const void* x, const void* w, int B, int T, int Cm, int NH,
                             int NKV, int hd, float rope_theta, int flags, void* stream) {
  if (B < 1 || T < 1 || Cm < 1 || NH < 1 || NKV < 1 || hd < 1 || NH % NKV != 0) return ATTN_ERR_BAD_SHAPE;
  if (flags & ~ATTN_FLAG_ROPE_INTERLEAVED) return ATTN_ERR_BAD_ARGUMENT;
  if (!std::isfinite(rope_theta)) return ATTN_ERR_BAD_ARGUMENT;
  if (hd != 64 && hd != 128) return ATTN_ERR_UNSUPPORTED;
  if (Cm % 8 != 0) return ATTN_ERR_BAD_SHAPE;           // 16-byte rows for the tensor maps
  const long long M = (long long)B * T, N = (long long)(NH + 2 * NKV) * hd;
  if (M > INT_MAX / 2 || N > 65535 * 8 || (long long)T > (1LL << 24)) return ATTN_ERR_BAD_SHAPE;
  if (!qkv || !x || !w) return ATTN_ERR_NULL_POINTER;
  if (!aligned16(qkv) || !aligned16(x) || !aligned16(w) || (qk_rot && !aligned16(qk_rot))) return ATTN_ERR_MISALIGNED;
  ProjArgs a{};
  ProjGeometry& pg = a.pg;
  pg.M = (int)M;
  pg.N = (int)N;
  pg.Cm = Cm;
  pg.T = T;
  pg.NQK = (NH + NKV) * hd;
  pg.hd = hd;
  pg.rope = rope_theta > 0.f ? 1 : 0;
  pg.interleaved = (flags & ATTN_FLAG_ROPE_INTERLEAVED) ? 1 : 0;
  for (int i = 0; i < 64; ++i) {
    double f = 0.0;
    if (pg.rope && i < hd / 2) f = std::exp(-2.0 * i * std::log((double)rope_theta) / hd);
    pg.rope_f_hi[i] = (float)f;
    pg.rope_f_lo[i] = (float)(f - (double)pg.rope_f_hi[i]);
  }
  a.qkv = qkv;
  a.rot = (pg.rope && qk_rot) ? qk_rot : nullptr;
  a.status = status_word();
  a.num_sms = num_sms();
  if (!a.status || a.num_sms <= 0) return ATTN_ERR_CUDA;
  if (!make_tmap(&a.tm_x, x, Cm, (int)M, 1, 128) || !make_tmap(&a.tm_w, w, Cm, (int)N, 1, 128)) return ATTN_ERR_CUDA;
  return from_cuda(proj_launch(a, static_cast<cudaStream_t>(stream)));
}

extern "C" int attn_fwd_rot(void* out, float* lse, const void* qkv, const void* qk_rot, int B, int T, int C, int NH,
                            int NKV, float rope_theta, int dtype, void* stream) {
  Geometry g;
  int type = dtype;
  int st = check_shape(B, T, C, NH, NKV, rope_theta, type, &g);
  if (st != ATTN_OK) return st;
  if (type != ATTN_DTYPE_BF16 || g.rope_theta <= 0.f)   // the copy only matters on the bf16 RoPE path
    return fwd_impl(out, lse, qkv, B, T, C, NH, NKV, rope_theta, dtype, nullptr, 0, stream);
  if (!qk_rot) return ATTN_ERR_NULL_POINTER;
  return fwd_impl(out, lse, qkv, B, T, C, NH, NKV, rope_theta, dtype, const_cast<void*>(qk_rot), 0, stream, true);
}

// ---------------------------------------------------------------- decode
namespace {
int decode_check(int B, int NH, int NKV, int hd, int max_len, int dtype) {
  if (B < 1 || NH < 1 || NKV < 1 || max_len < 1 || hd < 1) return ATTN_ERR_BAD_SHAPE;
  if (NH % NKV != 0) return ATTN_ERR_BAD_SHAPE;
  if (dtype != ATTN_DTYPE_F32 && dtype != ATTN_DTYPE_TF32 && dtype != ATTN_DTYPE_BF16) return ATTN_ERR_BAD_ARGUMENT;
  if (hd != 64 && hd != 128) return ATTN_ERR_UNSUPPORTED;
  const long long hgroups = (NH / NKV + 3) / 4;
  if (B > 65535 || (long long)NKV * hgroups > 65535 || (long long)max_len * NKV * hd > (1LL << 40))
    return ATTN_ERR_BAD_SHAPE;
  return ATTN_OK;
}
}  // namespace

extern "C" size_t attn_decode_workspace_bytes(int B, int NH, int NKV, int hd, int max_len, int dtype) {
  if (decode_check(B, NH, NKV, hd, max_len, dtype) != ATTN_OK) return 0;
  return align256(decode_workspace_floats(B, NH, NKV, hd, max_len) * sizeof(float));
}

extern "C" int attn_decode(void* out, float* lse, const void* q, const void* k_cache, const void* v_cache,
                           const int* seq_lens, int B, int NH, int NKV, int hd, int max_len, int dtype,
                           void* workspace, size_t ws_bytes, void* stream) {
  int st = decode_check(B, NH, NKV, hd, max_len, dtype);
  if (st != ATTN_OK) return st;
  if (!out || !lse || !q || !k_cache || !v_cache || !seq_lens) return ATTN_ERR_NULL_POINTER;
  if (!workspace || ws_bytes < attn_decode_workspace_bytes(B, NH, NKV, hd, max_len, dtype)) return ATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(workspace)) & 15u)
    return ATTN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(seq_lens)) & 3u) return ATTN_ERR_MISALIGNED;
  DecodeArgs a{};
  a.B = B;
  a.NH = NH;
  a.NKV = NKV;
  a.hd = hd;
  a.max_len = max_len;
  a.bf16 = dtype == ATTN_DTYPE_BF16;
  a.out = out;
  a.lse = lse;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.lens = seq_lens;
  a.part = static_cast<float*>(workspace);
  a.status = status_word();
  if (!a.status) return ATTN_ERR_CUDA;
  return from_cuda(decode_launch(a, static_cast<cudaStream_t>(stream)));
}

extern "C" int attn_device_status(int* status, int reset) {
  if (!status) return ATTN_ERR_NULL_POINTER;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  *status = v;
  if (reset) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

extern "C" int attn_selftest_wait_timeout(long long limit_ns, int* status) {
  if (!status) return ATTN_ERR_NULL_POINTER;
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > 1000000000LL) limit_ns = 1000000000LL;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_selftest_status, &zero, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_selftest_status) != cudaSuccess) return ATTN_ERR_CUDA;
  wait_timeout_selftest_kernel<<<1, 32>>>(static_cast<int*>(p), (unsigned long long)limit_ns);
  if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_selftest_status, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  *status = v;
  return ATTN_OK;
}
