// Optional per-kernel timing: while enabled (attn_profile_start), every
// kernel launch of the library is bracketed by a pair of CUDA events on the
// launching stream; attn_profile_stop sums their elapsed times per kernel.
#pragma once

#include <cuda_runtime.h>

namespace attn {

enum KernelId {
  kKernelFwdTc05 = 0,
  kKernelBwdDkdvTc05 = 1,
  kKernelBwdDqTc05 = 2,
  kKernelBwdRowDot = 3,
  kKernelRopeQK = 4,
  kKernelFwdSimt = 5,
  kKernelBwdDkdvSimt = 6,
  kKernelBwdDqSimt = 7,
  kKernelBwdPrologue = 8,
  kKernelDecode = 9,
  kKernelProj = 10,
  kKernelFp8Prep = 11,
  kKernelFwdFp8 = 12,
  kKernelSplitPrep = 13,
  kKernelFwdSplit = 14,
  kKernelBwdDkdvSplit = 15,
  kKernelBwdDqSplit = 16,
  kKernelCount = 17
};

// Record the start / end of a launch of kernel `id` on `stream` (no-ops while
// profiling is off).
void prof_begin(int id, cudaStream_t stream);
void prof_end(int id, cudaStream_t stream);

}  // namespace attn
