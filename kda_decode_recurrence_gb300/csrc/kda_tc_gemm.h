// kda_tc_gemm.h -- the tcgen05 weight-streaming GEMM used by the fused block.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Ypart[ks][r][n] = sum over contraction split ks of (X2[r][k] + X2[R + r][k]) * W[k][n],
// or, with `accumulate`, every split added into Ypart[r][n] (fp32 atomics;
// Ypart [R, N] must hold the starting value, e.g. zeros).
// X2 bf16 [2R, Kdim] (hi rows then lo rows), W bf16 [Kdim, N] (row k contiguous),
// Ypart fp32 [KS, R, N].  Kdim % 64 == 0, N % 8 == 0, 1 <= KS <= Kdim / 64,
// 16-byte aligned pointers.  On an internal pipeline timeout the kernel ORs
// bit 1 into *err (a device int32) and leaves Ypart incomplete.  With `pdl`
// the kernel is a programmatic dependent of the previous kernel in the stream
// (it requests its first weight tiles before waiting for that kernel).
// With `tail` (fp32 [R, N - tail_col], holding the starting value, e.g.
// zeros; tail_col a multiple of 128), the columns n >= tail_col are summed
// over the splits into tail[r][n - tail_col] with fp32 atomics instead of
// being written to Ypart.
// With x_parts == 3, X2 is [3R, Kdim]: a third part (rows 2R..3R-1, the bf16
// rounding of x - hi - lo) whose product the tail CTAs add as well, which
// brings the tail columns to fp32 activation precision.
// Up to three device ranges that the GEMM's CTAs bring into L2 once their
// own MMAs are done (each CTA an equal slice): data the next kernels read
// right after the weight stream, which would otherwise be evicted by it if
// requested earlier.
struct L2Prefetch {
  const void* ptr[3];
  size_t bytes[3];
};

cudaError_t launch_tc_gemm(const kda_bf16* X2, int R, int Kdim, const kda_bf16* W, int N, int KS,
                           float* Ypart, bool accumulate, int32_t* err, cudaStream_t stream,
                           bool pdl, float* tail = nullptr, int tail_col = 0,
                           const L2Prefetch* prefetch = nullptr, int x_parts = 2);

size_t tc_gemm_smem_bytes(int R);

}  // namespace kda
