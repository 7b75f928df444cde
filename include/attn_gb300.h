/*
 * attn_gb300.h -- C ABI of a GB300 (sm_103a) library for fused causal
 * multi-head / grouped-query self-attention over a packed QKV activation,
 * forward and backward.
 *
 * Method.  For batch row b, query head h, position t, with hd = C/NH,
 * grp = NH/NKV and kv head kh = h / grp (integer division):
 *   q = R_t Q[b,t,h], k_s = R_s K[b,s,kh]     (NEOX RoPE, optional)
 *   s_ts = q . k_s / sqrt(hd)                  for s <= t (causal)
 *   P_ts = exp(s_ts - lse_t),  lse_t = ln sum_{s<=t} exp(s_ts)
 *   out[b,t,h] = sum_s P_ts V[b,s,kh]
 * Sources: "nanoeuler -- CUDA kernels" (nanoeuler_cuda.cu), section "Causal
 * multi-head attention with GQA" -- packed layout, 1/sqrt(hs) scale, GQA map
 * h/(NH/NKV), and the forward/backward kernel declarations with an `lse`
 * buffer of B*NH*T floats; "nx_f32_qwen2_train_gate.nx source", build_rope /
 * rope_node -- the NEOX rotation; "CUDA C microgpt" (microgpt.cu),
 * attention_backward_kernel -- the row-dot D_t = dO_t . O_t used by the
 * backward.
 *
 * Layouts (dense, row-major, device pointers unless stated):
 *   qkv, dqkv : [B, T, (NH + 2*NKV)*hd]; columns [0, C) hold Q (head h at
 *               h*hd), [C, C + NKV*hd) hold K (kv head kh at C + kh*hd),
 *               [C + NKV*hd, ...) hold V.
 *   out, dout : [B, T, C]; head h at columns h*hd.
 *   lse       : float32 [B, NH, T], index (b*NH + h)*T + t; natural log of
 *               the sum of exp of the scaled scores.
 * Element type of qkv/out/dout/dqkv is chosen by `dtype`; lse and every
 * accumulation are float32.
 *
 * RoPE: rope_theta <= 0 disables it.  Otherwise the NEOX rotation with base
 * rope_theta is applied inside the kernels to every Q and K head at position
 * t (0-based within each sequence): pair (i, i + hd/2) turns by angle
 * t * rope_theta^(-2i/hd).  qkv is never modified; dqkv is the gradient with
 * respect to the un-rotated qkv.
 *
 * Ownership and execution: the caller owns every buffer and the stream.  The
 * library allocates no device memory; scratch is the caller's `workspace`
 * (attn_bwd, attn_fwd_ws).  Every call validates its arguments on the host, then
 * enqueues kernels on `stream` (a cudaStream_t passed as void*; NULL is the
 * legacy default stream) and returns without synchronising.  Nothing is
 * launched when validation fails.
 *
 * Errors: every entry point returns ATTN_OK (0) or a negative attn_status.
 * The library never exits the process and never traps on the device.  A
 * kernel whose bounded wait on an on-chip barrier expires abandons its work,
 * records ATTN_ERR_DEVICE_TIMEOUT in a library-owned device status word and
 * returns; read it with attn_device_status() after synchronising.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  /* float32 tensors, exact float32 arithmetic on CUDA cores. */
  ATTN_DTYPE_F32 = 0,
  /* float32 tensors held to the same 1e-4 bar as ATTN_DTYPE_F32, computed on
     the tensor cores where it can be: with head size 64, attn_fwd_ws,
     attn_bwd and attn_bwd_rot split every float32 operand into bf16 parts
     hi + lo in the workspace and take each product as hi*hi + hi*lo + lo*hi
     on tcgen05 MMAs with float32 accumulation (~1e-5 of the float64 result;
     the softmax weights and dS are split the same way).  Elsewhere (attn_fwd,
     which has no workspace, and other head sizes) it runs the exact float32
     kernels, with results equal to ATTN_DTYPE_F32's. */
  ATTN_DTYPE_TF32 = 1,
  /* bf16 tensors, tcgen05 tensor-core MMAs with float32 accumulation. */
  ATTN_DTYPE_BF16 = 2
} attn_dtype_t;

/*
 * ATTN_FLAG_ROPE_INTERLEAVED -- OR-ed into the dtype argument of attn_fwd,
 * attn_fwd_ws, attn_fwd_fp8, attn_bwd, attn_bwd_rot and attn_bwd_noalloc to
 * use the interleaved (GPT-J) RoPE pairing of "nanoeuler -- CUDA
 * kernels", rope_kernel -- pair (2i, 2i+1) of each head turns by t*theta^(-2i/hd):
 *   y[2i] = x[2i] cos - x[2i+1] sin,   y[2i+1] = x[2i] sin + x[2i+1] cos
 * -- instead of the NEOX pairing (i, i + hd/2).  Ignored when rope_theta <= 0.
 * attn_fwd with ATTN_DTYPE_BF16 rotates inside its attention kernel, turning
 * each interleaved pair of the Q and K tiles in place.  The
 * *_workspace_bytes() functions accept and ignore the flag.
 * A forward and its backward must use the same pairing.
 */
#define ATTN_FLAG_ROPE_INTERLEAVED 0x100

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_NULL_POINTER = -1,    /* a required pointer is NULL */
  ATTN_ERR_BAD_SHAPE = -2,       /* B,T,NH,NKV < 1, C % NH, NH % NKV, odd hd with RoPE, overflow */
  ATTN_ERR_UNSUPPORTED = -3,     /* (dtype, head size) combination not implemented */
  ATTN_ERR_MISALIGNED = -4,      /* a pointer is not 16-byte aligned (bf16 path) */
  ATTN_ERR_WORKSPACE = -5,       /* workspace NULL or smaller than the *_workspace_bytes() size */
  ATTN_ERR_CUDA = -6,            /* a CUDA runtime call or kernel launch failed */
  ATTN_ERR_DEVICE_TIMEOUT = -7,  /* a device-side bounded wait expired (see attn_device_status) */
  ATTN_ERR_BAD_ARGUMENT = -8     /* any other invalid argument */
} attn_status_t;

/*
 * attn_fwd -- causal attention forward.
 *   out  : [B,T,C] of dtype, overwritten (every element).
 *   lse  : float32 [B,NH,T], overwritten.
 *   qkv  : [B,T,(NH+2*NKV)*hd] of dtype, read only.
 * Supported: dtype F32 with any hd <= 128 (even hd when RoPE is on);
 * dtype BF16 with hd in {64, 128}.  T >= 1, any NH divisible by NKV.
 * bf16 pointers must be 16-byte aligned.
 */
ATTN_API int attn_fwd(void* out, float* lse, const void* qkv,
             int B, int T, int C, int NH, int NKV, float rope_theta,
             int dtype, void* stream);

/*
 * attn_fwd_workspace_bytes -- size in bytes of the scratch attn_fwd_ws
 * uses for this shape and dtype: room for a RoPE-rotated copy of Q and K,
 * [B,T,(NH+NKV)*hd] of dtype, for BF16; for TF32 with head size 64 the bf16
 * hi and lo parts of qkv (2 x [B,T,(NH+2*NKV)*hd] bf16, Q and K rotated);
 * 0 for F32 and other TF32 head sizes (which need none) and for invalid
 * arguments.
 *
 * attn_fwd_ws -- attn_fwd with caller-provided scratch.  Same arguments,
 * results and supported shapes as attn_fwd, plus
 *   workspace : device scratch of at least attn_fwd_workspace_bytes(...)
 *          bytes (may be NULL when that is 0), 256-byte aligned, owned by the
 *          caller; its contents on entry do not matter and are garbage on
 *          return.
 * With BF16 and rope_theta > 0 it first rotates every Q and K head once into
 * the workspace (one HBM-bound pass over Q and K, the rotation the source
 * pages apply to qkv in place before attention) and then runs the attention
 * kernel on the rotated copy; attn_fwd instead rotates Q and every K tile
 * inside the attention kernel, once per use, which costs more for long
 * sequences because each K tile is used by many query tiles.  Without RoPE,
 * or for F32, it is attn_fwd.  The two give the same results up to the
 * rounding of the rotated values to dtype (both round them once).  With TF32
 * and head size 64 it runs the tensor-core path (see ATTN_DTYPE_TF32) on the
 * parts it writes into the workspace; float32 tensors must then be 16-byte
 * aligned (ATTN_ERR_MISALIGNED otherwise).
 */
ATTN_API size_t attn_fwd_workspace_bytes(int B, int T, int C, int NH, int NKV, int dtype);
ATTN_API int attn_fwd_ws(void* out, float* lse, const void* qkv,
             int B, int T, int C, int NH, int NKV, float rope_theta,
             int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd_workspace_bytes -- size in bytes of the scratch attn_bwd needs
 * for this shape and dtype: the row dots D = rowsum(dO * O) (float32
 * [B,NH,T]; for BF16 stored next to the rescaled lse as two float tables of
 * T rounded up to 128 rows per (b, h)), plus, for BF16, room for a
 * RoPE-rotated bf16 copy of Q and K, 256 bytes for a work-item counter and a
 * float (cos, sin) table of the RoPE angles [hd/2][T] (the copy and the table
 * are used only when rope_theta > 0); for TF32 with head size 64 the
 * row tables over T rounded up to 128 rows and the bf16 hi/lo parts of qkv
 * and dout (the tensor-core path; 16-byte aligned tensors).  Returns 0 for invalid
 * arguments.
 */
ATTN_API size_t attn_bwd_workspace_bytes(int B, int T, int C, int NH, int NKV, int dtype);

/*
 * attn_bwd -- causal attention backward.
 *   dqkv : [B,T,(NH+2*NKV)*hd] of dtype, overwritten (every element; no need
 *          to clear it first).  dQ at Q's columns, dK/dV (summed over the
 *          grp query heads sharing each kv head) at K/V's columns.
 *   qkv  : the forward's input.   out, lse : the forward's outputs.
 *   dout : [B,T,C] of dtype, the gradient of the loss with respect to out.
 *   workspace : device scratch of at least attn_bwd_workspace_bytes(...)
 *          bytes, 256-byte aligned, owned by the caller; its contents on
 *          entry do not matter and are garbage on return.
 * Deterministic: identical inputs give bit-identical dqkv (no atomics).
 */
ATTN_API int attn_bwd(void* dqkv, const void* qkv, const void* out, const void* dout,
             const float* lse, int B, int T, int C, int NH, int NKV,
             float rope_theta, int dtype, void* workspace, size_t workspace_bytes,
             void* stream);

/*
 * attn_bwd_rot -- attn_bwd that reuses the rotated Q/K copy of the forward.
 * Same arguments, results and errors as attn_bwd, plus
 *   qk_rot : the workspace of the attn_fwd_ws call that produced out and lse
 *          from this qkv, left unchanged since (it holds Q and K rotated by
 *          RoPE, [B,T,(NH+NKV)*hd] of dtype; 256-byte aligned).
 * With BF16 and rope_theta > 0 the backward then reads Q and K from qk_rot
 * instead of rotating them again into its own workspace (one HBM pass fewer);
 * with TF32 at head size 64 it reads the bf16 hi/lo parts of qkv that
 * attn_fwd_ws left there instead of forming them again; otherwise qk_rot is
 * ignored and it is attn_bwd.  A qk_rot that does not
 * hold the rotation of this qkv gives wrong gradients: the library cannot
 * check it.
 */
ATTN_API int attn_bwd_rot(void* dqkv, const void* qkv, const void* out, const void* dout,
             const float* lse, int B, int T, int C, int NH, int NKV,
             float rope_theta, int dtype, const void* qk_rot, void* workspace,
             size_t workspace_bytes, void* stream);

/*
 * attn_bwd_noalloc -- attn_bwd for callers that cannot allocate device
 * memory.  (The source pages have no counterpart: this is a library
 * convenience, not part of the attention method.)
 *
 * Some callers cannot obtain scratch memory when they run the backward:
 * code running inside a custom allocator or memory-pool callback (calling
 * cudaMalloc there would re-enter the allocator), runtimes that forbid
 * device allocation after start-up so that memory use stays fixed, and
 * plugins that are handed only input and output pointers.  This entry point
 * takes the same arguments as attn_bwd minus the workspace, and uses a
 * built-in device buffer of ATTN_NOALLOC_SCRATCH_BYTES instead.  It calls no
 * allocating routine.
 *
 * Limits and behaviour:
 *  - The buffer is a fixed array in device memory: every GPU on which it is
 *    loaded holds ATTN_NOALLOC_SCRATCH_BYTES until the process exits.
 *  - Problems whose attn_bwd_workspace_bytes() exceeds that size are
 *    rejected with ATTN_ERR_WORKSPACE before anything is launched (e.g. the
 *    bf16 B=4, T=2048, NH=16, NKV=4, hd=128 case needs about 44 MB and
 *    fits; B=1, T=8192, NH=32, NKV=8, hd=128 needs about 90 MB and does not).
 *  - The first call on a device (with that device current) looks up the
 *    buffer's device address with cudaGetSymbolAddress.  The address is then
 *    kept for the life of the process: after cudaDeviceReset() on a device
 *    the buffer lives in a new
 *    context at an address this library does not look up again, so do not
 *    call attn_bwd_noalloc on that device after a reset.
 *  - All calls share the one buffer, which keeps the last call's contents.
 *    Nothing in it needs to start at zero.  Calls whose kernels overlap on
 *    the GPU (different streams, or different host threads) race on it and
 *    give wrong results: serialise them.
 * Other arguments, results and errors are those of attn_bwd.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
ATTN_API int attn_bwd_noalloc(void* dqkv, const void* qkv, const void* out, const void* dout,
                              const float* lse, int B, int T, int C, int NH, int NKV,
                              float rope_theta, int dtype, void* stream);

/*
 * attn_decode -- single-query (decode) attention over a KV cache: one new
 * token per batch row attends to the cached keys and values of its sequence.
 * It is the per-position form of the forward ("CUDA C microgpt",
 * attention_forward_kernel: one query at position pos_id against keys
 * 0 .. pos_id) with grouped heads ("nanoeuler -- CUDA kernels": query head h
 * reads kv head h / (NH/NKV)).  For every batch row b and query head h:
 *   s_j = q[b,h,:] . k_cache[b,j,kh,:] / sqrt(hd)  for j < seq_lens[b],
 *   out[b,h,:] = sum_j softmax(s)_j v_cache[b,j,kh,:],
 *   lse[b,h]  = ln sum_j exp(s_j).
 *
 * Layouts (dense, row-major, device pointers; element type float for
 * ATTN_DTYPE_F32 / ATTN_DTYPE_TF32, bf16 for ATTN_DTYPE_BF16; arithmetic in
 * float32 throughout):
 *   q        [B, NH, hd]          the new token's queries;
 *   k_cache  [B, max_len, NKV, hd] keys of positions 0 .. max_len-1;
 *   v_cache  [B, max_len, NKV, hd] values;
 *   seq_lens [B] int32, device     visible cache rows per batch row, the new
 *                                  token's own row included (1 .. max_len);
 *   out      [B, NH, hd]          written;
 *   lse      [B, NH] float32       written.
 * RoPE is the caller's: q is expected rotated at the new token's position and
 * the cached keys at theirs (a cache holds rotated keys; rotating every cached
 * key on each step would cost far more than reading it).
 *
 * hd must be 64 or 128 (else ATTN_ERR_UNSUPPORTED); NH % NKV == 0.  q, k_cache,
 * v_cache, out and the workspace must be 16-byte aligned, lse and seq_lens
 * 4-byte aligned (ATTN_ERR_MISALIGNED).  The workspace (attn_decode_workspace_
 * bytes(), owned by the caller, contents irrelevant) holds one partial result
 * per (b, h, chunk of cache rows; the chunk length depends only on the
 * arguments).  A seq_lens entry outside
 * [1, max_len] is clamped into it and ATTN_ERR_BAD_ARGUMENT is recorded in
 * the device status word (attn_device_status).  Asynchronous on `stream`;
 * deterministic (the chunks of a head are merged in a fixed order).
 */
ATTN_API size_t attn_decode_workspace_bytes(int B, int NH, int NKV, int hd, int max_len, int dtype);
ATTN_API int attn_decode(void* out, float* lse, const void* q, const void* k_cache,
                         const void* v_cache, const int* seq_lens, int B, int NH, int NKV,
                         int hd, int max_len, int dtype, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * attn_qkv_proj -- the QKV projection that feeds the attention, with the RoPE
 * rotation fused into its epilogue.  The trainers on the pages project the
 * layer input into the packed Q | K | V activation with a GEMM and then run
 * separate RoPE passes over the Q and K column blocks ("nanoeuler -- CUDA
 * kernels": the qkv matmul, then rope_kernel over the query and kv heads);
 * here both come out of one kernel:
 *   qkv[m, n] = sum_k x[m, k] * w[n, k]     m < B*T, n < (NH + 2*NKV)*hd, k < Cm
 * (bf16 in and out, float32 accumulation; row m is position m % T of
 * sequence m / T), and, when rope_theta > 0 and qk_rot != NULL, the rotated
 * copy of its Q and K heads [B*T, (NH+NKV)*hd] bf16, rotated from the float32
 * accumulators, in the layout attn_fwd_rot / attn_bwd_rot read (the copy the
 * rotation pass of attn_fwd_ws makes).  `flags` may be
 * ATTN_FLAG_ROPE_INTERLEAVED (then pass it to the attention calls as well).
 *   x   [B*T, Cm] bf16, row-major (Cm a multiple of 8);
 *   w   [(NH+2*NKV)*hd, Cm] bf16, row-major (row n produces output column n);
 *   qkv [B*T, (NH+2*NKV)*hd] bf16, written.
 * hd must be 64 or 128 (ATTN_ERR_UNSUPPORTED otherwise).  All pointers
 * 16-byte aligned; a copy handed to attn_fwd_rot / attn_bwd_rot must be
 * 256-byte aligned.  Asynchronous on `stream`; deterministic.  The kernel
 * runs on clusters of two CTAs (one per SM); ATTN_ERR_CUDA if the device
 * cannot hold such a cluster.
 *
 * attn_fwd_rot -- attn_fwd (bf16 with RoPE) reading the rotated Q/K from
 * qk_rot (made by attn_qkv_proj or attn_fwd_ws on the same qkv) instead of
 * rotating them: no rotation pass.  Other dtypes, or rope_theta <= 0, behave
 * as attn_fwd and ignore qk_rot.  The library cannot check that qk_rot holds
 * the rotation of this qkv.
 */
ATTN_API int attn_qkv_proj(void* qkv, void* qk_rot, const void* x, const void* w, int B, int T,
                           int Cm, int NH, int NKV, int hd, float rope_theta, int flags,
                           void* stream);
ATTN_API int attn_fwd_rot(void* out, float* lse, const void* qkv, const void* qk_rot, int B,
                          int T, int C, int NH, int NKV, float rope_theta, int dtype, void* stream);

/*
 * attn_fwd_fp8 -- the forward with e4m3 (FP8) tensor-core operands (an
 * adjacent GB300 capability, not on the source pages): same inputs, outputs
 * and RoPE handling as attn_fwd_ws with ATTN_DTYPE_BF16, but Q and K are
 * rotated and rounded to e4m3 with one scale per (batch row, head, 128-row
 * tile) (x8 = rn(x * 448 / amax)), V to e4m3 with one scale per (batch row, kv
 * head), and the softmax weights P = exp(s - m) to e4m3 (as 112 P, with the
 * running row maximum m renewed only when exceeded by more than 2 log2 units,
 * so 112 P <= 448) before the P V product; scores, sums, O, out (bf16) and lse
 * (float32) are accumulated in float32.  Expect
 * errors of a few 1e-2 of max|out| (3 mantissa bits), not the bf16 path's
 * 2e-2.  Head size 128 and an even number of query heads per kv head only
 * (ATTN_ERR_UNSUPPORTED otherwise).  The workspace (attn_fwd_fp8_workspace_
 * bytes(), 256-byte aligned) holds the e4m3 copies and their scales.  There
 * is no FP8 backward.
 */
ATTN_API size_t attn_fwd_fp8_workspace_bytes(int B, int T, int C, int NH, int NKV, int dtype);
ATTN_API int attn_fwd_fp8(void* out, float* lse, const void* qkv, int B, int T, int C, int NH,
                          int NKV, float rope_theta, int dtype, void* workspace,
                          size_t workspace_bytes, void* stream);

/* attn_strerror -- static description of a status code; never NULL. */
ATTN_API const char* attn_strerror(int status);

/*
 * attn_device_status -- synchronise the current device, then store in
 * *status the first error a kernel of this library recorded on it since the
 * last reset (ATTN_OK if none); when `reset` is non-zero clear it.
 * Returns ATTN_OK, or ATTN_ERR_CUDA if the synchronisation failed.
 */
ATTN_API int attn_device_status(int* status, int reset);

/*
 * attn_selftest_wait_timeout -- failure-detection self test: launches one
 * block that waits on an on-chip barrier nothing will ever complete, with a
 * wait limit of `limit_ns` nanoseconds (clamped to [1e3, 1e9]).  The kernel
 * must give up, record ATTN_ERR_DEVICE_TIMEOUT and exit; the device stays
 * usable.  *status receives what the kernel recorded.  Synchronous.
 */
ATTN_API int attn_selftest_wait_timeout(long long limit_ns, int* status);

/*
 * Per-kernel timing (tracing aid; not part of the attention method).
 * attn_profile_start -- from now on, bracket every kernel this library
 *   launches (any thread, any stream) with a pair of CUDA events recorded on
 *   the launching stream.  Clears earlier records.
 * attn_profile_stop -- stop recording, wait for the recorded events, and for
 *   kernel ids 0..n-1 store the summed elapsed milliseconds in total_ms[id]
 *   and the launch count in launches[id] (either array may be NULL).
 * attn_kernel_name -- short name of kernel id (see attn_profile.h ids:
 *   0 fwd_tc05, 1 bwd_dkdv_tc05, 2 bwd_dq_tc05, 3 bwd_row_dot, 4 rope_qk,
 *   5 fwd_simt, 6 bwd_dkdv_simt, 7 bwd_dq_simt, 8 bwd_prologue, 9 decode (both
 *   of its kernels), 10 qkv_proj, 11 fp8_prep, 12 fwd_fp8); "unknown" otherwise.
 */
ATTN_API int attn_profile_start(void);
ATTN_API int attn_profile_stop(double* total_ms, int* launches, int n);
ATTN_API const char* attn_kernel_name(int id);

/* attn_abi_version -- ABI version of this header (currently 1). */
ATTN_API int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
