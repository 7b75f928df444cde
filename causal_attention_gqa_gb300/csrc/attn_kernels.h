// Internal launch interfaces between the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include <utility>

#include "attn_common.cuh"

namespace attn {

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream is still running; it must call
// griddepcontrol.wait before touching anything that kernel writes, unless
// an earlier grid already guarantees it (see the backward kernels).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ------------------------------------------------------------ float32 SIMT path
struct SimtArgs {
  Geometry g;
  bool forward;
  void* out;          // fwd: [B,T,C] float32
  float* lse;         // fwd: written; bwd: read
  const void* qkv;    // [B,T,W] float32
  void* dqkv;         // bwd: [B,T,W] float32
  const void* dout;   // bwd: [B,T,C] float32
  const float* Drow;  // bwd: [B,NH,T] row dots
};
cudaError_t simt_launch(const SimtArgs& a, cudaStream_t stream);
// Register-tiled float32 kernels (head size 64, 16-byte aligned tensors).
bool simt_tiled_supported(const SimtArgs& a);
cudaError_t simt_tiled_launch(const SimtArgs& a, cudaStream_t stream);
size_t simt_max_smem_bytes(int hd);

// ------------------------------------------------------------ float32 on tensor cores
// dtype TF32, head size 64: every product of float32 operands as three bf16
// products of hi/lo parts (attn_split_sm103.cu).  The parts of Q, K, V (Q and
// K rotated when RoPE is on) and of dO live in the workspace in the column
// layout of qkv / dout.
struct SplitArgs {
  Geometry g;
  CUtensorMap tm_hi, tm_lo;       // over qkv_hi / qkv_lo [B, T, W] bf16 (64-column, 128-row boxes)
  CUtensorMap tm_dohi, tm_dolo;   // over dout_hi / dout_lo [B, T, C] bf16 (backward)
  const void* qkv;                // float32 [B, T, W]
  const void* dout;               // float32 [B, T, C] (backward)
  void* out;                      // float32 [B, T, C]: forward writes it, backward reads it
  float* lse;                     // float32 [B, NH, T]: forward writes it, backward reads it
  void* dqkv;                     // float32 [B, T, W] (backward)
  __nv_bfloat16* qkv_hi;
  __nv_bfloat16* qkv_lo;
  __nv_bfloat16* dout_hi;
  __nv_bfloat16* dout_lo;
  float* LD;                      // backward row tables: -lse log2(e) and -D over T rounded up to 128
  bool qkv_given;                 // backward: qkv_hi / qkv_lo already hold the forward's parts
  int* status;
};
bool split_supported(const Geometry& g);
cudaError_t split_fwd_launch(const SplitArgs& a, cudaStream_t stream);
cudaError_t split_bwd_launch(const SplitArgs& a, cudaStream_t stream);

// ------------------------------------------------------------ FP8 forward
// e4m3 operands with per-tile (Q, K) and per-head (V) scales; head size 128,
// an even number of query heads per kv head.
struct Fp8FwdArgs {
  Geometry g;
  CUtensorMap tm_qk8, tm_vt, tm_out;
  const void* qkv;
  uint8_t* qk8;      // [B*T, (NH+NKV)*hd] e4m3, rotated Q | K
  uint8_t* vt8;      // [B, NKV, hd, Tp] e4m3, V transposed
  float* deq_qk;     // [B, NH+NKV, T/128] dequantization factors
  float* deq_v;      // [B, NKV]
  float* vtile_amax; // [B, NKV, T/128] amax of each V tile
  int Tp;            // T rounded up to 128
  float* lse;
  int* status;
  int num_sms;
};
bool fp8_fwd_supported(const Geometry& g);
cudaError_t fp8_fwd_launch(const Fp8FwdArgs& a, cudaStream_t stream);

// ------------------------------------------------------------ QKV projection
// qkv = x w^T with the rotated Q/K copy written from the same accumulators.
struct ProjGeometry {
  int M, N, Cm, T;   // rows B*T, packed width (NH+2NKV)*hd, input width, sequence length
  int NQK;           // (NH+NKV)*hd: the Q and K columns (rotated copy width)
  int hd;
  int rope;          // rotate (and write the copy) at all
  int interleaved;   // pairing of the rotation (see Geometry::rope_interleaved)
  float rope_f_hi[64];
  float rope_f_lo[64];
};
struct ProjArgs {
  CUtensorMap tm_x, tm_w;   // x [M, Cm] and w [N, Cm] bf16: 64-column, 128-row boxes, 128-byte swizzle
  void* qkv;
  void* rot;         // may be null
  ProjGeometry pg;
  int* status;
  int num_sms;
};
cudaError_t proj_launch(const ProjArgs& a, cudaStream_t stream);

// ------------------------------------------------------------ decode
// Single-query attention over a KV cache (attn_decode).
struct DecodeArgs {
  int B, NH, NKV, hd, max_len;
  bool bf16;
  void* out;             // [B,NH,hd]
  float* lse;            // [B,NH]
  const void* q;         // [B,NH,hd]
  const void* k_cache;   // [B,max_len,NKV,hd]
  const void* v_cache;   // [B,max_len,NKV,hd]
  const int* lens;       // [B], device
  float* part;           // workspace: per (b, h, chunk) m, l, o[hd]
  int* status;
};
int decode_chunk_rows(int B, int NH, int NKV, int max_len);
size_t decode_workspace_floats(int B, int NH, int NKV, int hd, int max_len);
cudaError_t decode_launch(const DecodeArgs& a, cudaStream_t stream);

// ------------------------------------------------------------ backward prologue
// D[b,h,t] = sum_d dout[b,t,h,d] * out[b,t,h,d] (float32 accumulation).
cudaError_t launch_row_dot(float* D, const void* out, const void* dout, const Geometry& g, bool bf16,
                           cudaStream_t stream);
// NEOX-rotated bf16 copy of every Q and K head: dst [B,T,(NH+NKV)*hd], query
// head h at column h*hd and kv head kh at C + kh*hd (the columns they have
// in qkv).  hd must be a multiple of 16.
cudaError_t launch_rope_qk_bf16(void* dst, const void* qkv, const Geometry& g, cudaStream_t stream);
// Rows of each per-(b, h) row table the bf16 backward reads: T rounded up to
// whole 128-row query tiles.
__host__ __device__ inline int row_table_rows(int T) { return (T + 127) / 128 * 128; }
// bf16 (hd a multiple of 16): the row tables, two float arrays of Tp rows per
// (b, h): LD[(2*(b*NH + h))*Tp + t] = -lse * log2(e) and
// LD[(2*(b*NH + h) + 1)*Tp + t] = -D with D = dO . O (zeros for t >= T); and,
// when `rot` is not NULL, the RoPE-rotated Q/K copy; when `rope_cs` is not
// NULL, the table rope_cs[2(i*T + t)], [2(i*T + t) + 1] = cos, sin of the RoPE
// angle of position t and pair i that the gradient epilogues read; it also
// clears *item_counter; in one launch.
cudaError_t launch_bwd_prologue_bf16(float* LD, void* rot, int* item_counter, float* rope_cs, const void* out,
                                     const void* dout, const float* lse, const void* qkv, const Geometry& g,
                                     cudaStream_t stream);

// ------------------------------------------------------------ tcgen05 bf16 path
struct Tc05FwdArgs {
  Geometry g;
  // Q and K come from tm_qk (qkv itself, or the RoPE-rotated copy written by
  // launch_rope_qk_bf16), V from tm_v (qkv); query head h starts at column
  // h*hd and kv head kh at column C + kh*hd in both layouts.  Box {64, 128, 1},
  // 128-byte swizzle.
  CUtensorMap tm_qk;
  CUtensorMap tm_v;
  bool pre_rotated;    // RoPE on, Q/K already rotated: no rotation in the kernel
  CUtensorMap tm_out;  // out [B,T,C] bf16, same box and swizzle (tile stores)
  void* out;          // [B,T,C] bf16
  float* lse;         // [B,NH,T]
  int* status;        // library status word
  int num_sms;        // persistent grid size
};
cudaError_t tc05_fwd_launch(const Tc05FwdArgs& a, cudaStream_t stream);
// Paired-head forward (two query heads per work item), Q/K not rotated in
// the kernel: head size 128 with an even number of query heads per kv head
// (the pair shares its K/V tiles), or head size 64 with an even number of
// query heads (sharing K/V tiles when the pair shares a kv head).
bool tc05_fwd2_supported(const Geometry& g);
cudaError_t tc05_fwd2_launch(const Tc05FwdArgs& a, cudaStream_t stream);

struct Tc05BwdArgs {
  Geometry g;
  // Tensor maps with 128-byte swizzle and 64-column boxes; index 0 has 64-row
  // boxes, index 1 128-row boxes.  Q and K come from the same source (qkv, or
  // the rotated copy when RoPE is on); query head h starts at column h*hd and
  // kv head kh at column C + kh*hd in both layouts.
  CUtensorMap tm_qk[2];
  CUtensorMap tm_v[2];   // over qkv
  CUtensorMap tm_do[2];  // over dout
  CUtensorMap tm_dqkv;   // over dqkv, 128-row boxes (tile stores of the gradients)
  void* dqkv;            // [B,T,W] bf16
  const float* LD;       // row tables: -lse * log2(e) and -D per (b, h), see launch_bwd_prologue_bf16
  int* item_counter;     // dQ work-item counter (workspace), cleared by the prologue
  const float* rope_cs;  // RoPE (cos, sin) table [hd/2][T] written by the prologue (RoPE only)
  int* status;
  int num_sms;           // persistent grid size
};
cudaError_t tc05_bwd_launch(const Tc05BwdArgs& a, cudaStream_t stream);

}  // namespace attn
