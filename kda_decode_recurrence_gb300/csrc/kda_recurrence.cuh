// kda_recurrence.cuh -- the register-resident delta-rule step on one fp32
// [128, 128] state tile, shared by the decode kernel and the block's head
// kernel.
//
// Tile ownership inside a 256-thread CTA: warp w owns value columns
// [16w, 16w + 16); lane = 4 * rg + cg holds rows rg, rg + 8, ..., rg + 120 of
// the four columns 16w + 4cg .. 16w + 4cg + 3, i.e. 16 float4 registers.  A
// warp's load/store instruction i covers rows 8i .. 8i + 7 x 64 contiguous
// bytes.
//
// One token ("Delta-rule write", naive recurrent loop; decay, delta write,
// read after the write):
//   S <- diag(exp(g)) S;  u = v - kh^T S;  S <- S + beta kh u^T;  o = qh^T S.
// The read is taken as qh^T S = qh^T (D S_old) + beta (qh . kh) u, the same
// quantity with a single pass over the tile.
//
// The transposed (V-first) step's arithmetic uses the packed fp32x2
// instructions of sm_100 and later (__fmul2_rn, __ffma2_rn, __fadd2_rn: two
// lanes per instruction, each rounded exactly like the scalar fmul/fma/add),
// which halves its floating-point instruction count.  The row-major step
// keeps scalar arithmetic: there a pair would be two columns of one row, each
// row coefficient has to be broadcast into both halves, and those moves plus
// the extra live registers made it slower (536 against 505 us per launch on
// the grouped workload).
#pragma once

#include "kda_common.cuh"

namespace kda {

struct __align__(16) RowCoef {
  float decay;  // exp(g[k])
  float kh;     // normalised key
  float qh;     // normalised, scaled query
  float bkh;    // beta * kh
};

// Per-token vectors in shared memory.
struct __align__(16) TokenStage {
  RowCoef row[kHeadDim];
  float v[kHeadDim];
  float bqk;  // beta * (qh . kh)
  float pad[3];
};

struct TileLane {
  int rg;   // row group 0..7
  int col;  // first of the lane's four value columns
};

__device__ __forceinline__ TileLane tile_lane() {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  return TileLane{lane >> 2, warp * 16 + (lane & 3) * 4};
}

__device__ __forceinline__ void tile_load(float4 (&s)[16], const float* tile, TileLane tl) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    s[i] = __ldcs(reinterpret_cast<const float4*>(tile + (tl.rg + 8 * i) * kHeadDim + tl.col));
}

__device__ __forceinline__ void tile_store(float* tile, const float4 (&s)[16], TileLane tl) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    __stcs(reinterpret_cast<float4*>(tile + (tl.rg + 8 * i) * kHeadDim + tl.col), s[i]);
}

// Advance the tile by one token; returns the read o for the lane's columns
// (identical in the 8 lanes of a column quad).
__device__ __forceinline__ float4 tile_token_step(float4 (&s)[16], const TokenStage& ts,
                                                  TileLane tl) {
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    // A compiler-only fence halfway: it keeps the compiler from hoisting all
    // sixteen 16-byte row loads ahead of the arithmetic, which with the 64
    // tile registers live exceeds the 128-register budget and spills.
    if (i == 8) asm volatile("" ::: "memory");
    const RowCoef rc = ts.row[tl.rg + 8 * i];
    s[i].x *= rc.decay; s[i].y *= rc.decay; s[i].z *= rc.decay; s[i].w *= rc.decay;
    a.x = fmaf(rc.kh, s[i].x, a.x); a.y = fmaf(rc.kh, s[i].y, a.y);
    a.z = fmaf(rc.kh, s[i].z, a.z); a.w = fmaf(rc.kh, s[i].w, a.w);
    c.x = fmaf(rc.qh, s[i].x, c.x); c.y = fmaf(rc.qh, s[i].y, c.y);
    c.z = fmaf(rc.qh, s[i].z, c.z); c.w = fmaf(rc.qh, s[i].w, c.w);
  }
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    a.x += __shfl_xor_sync(0xffffffffu, a.x, m); a.y += __shfl_xor_sync(0xffffffffu, a.y, m);
    a.z += __shfl_xor_sync(0xffffffffu, a.z, m); a.w += __shfl_xor_sync(0xffffffffu, a.w, m);
    c.x += __shfl_xor_sync(0xffffffffu, c.x, m); c.y += __shfl_xor_sync(0xffffffffu, c.y, m);
    c.z += __shfl_xor_sync(0xffffffffu, c.z, m); c.w += __shfl_xor_sync(0xffffffffu, c.w, m);
  }
  const float4 vv = *reinterpret_cast<const float4*>(&ts.v[tl.col]);
  const float4 u = make_float4(vv.x - a.x, vv.y - a.y, vv.z - a.z, vv.w - a.w);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (i == 8) asm volatile("" ::: "memory");  // as above
    const float bkh = ts.row[tl.rg + 8 * i].bkh;
    s[i].x = fmaf(bkh, u.x, s[i].x); s[i].y = fmaf(bkh, u.y, s[i].y);
    s[i].z = fmaf(bkh, u.z, s[i].z); s[i].w = fmaf(bkh, u.w, s[i].w);
  }
  const float bqk = ts.bqk;
  return make_float4(fmaf(bqk, u.x, c.x), fmaf(bqk, u.y, c.y), fmaf(bqk, u.z, c.z),
                     fmaf(bqk, u.w, c.w));
}

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }
__device__ __forceinline__ float2 bcast2(float x) { return make_float2(x, x); }

// x += the value of x in lane (this lane ^ m), both halves.
__device__ __forceinline__ float2 xor_add2(float2 x, int m) {
  return __fadd2_rn(x, f2(__shfl_xor_sync(0xffffffffu, x.x, m), __shfl_xor_sync(0xffffffffu, x.y, m)));
}

// ---------------------------------------------------------------------------
// Transposed (V-first) tiles: element (k, v) sits at v * 128 + k, so the
// contiguous direction is k.  Warp w still owns value columns [16w, 16w + 16),
// but lane = 8 * cq + kq holds, for each of its four columns 16w + 4cq + c,
// the rows 4kq + 32m .. 4kq + 32m + 3 (m = 0..3) as one float4: register
// s[4m + c].  Eight lanes of a column then cover 128 contiguous bytes, so a
// quarter-warp's 128-bit shared-memory load is conflict-free and a warp's
// 128-bit global store writes four full 128-byte lines.  The k-contractions
// are in-thread sums over 16 rows followed by three xor-shuffles across the
// 8 kq lanes, as in the row-major form.

// The token record for the transposed step: entry j of each array holds rows
// 4j .. 4j + 3 (the same 2576 bytes as TokenStage, laid out by field).
struct __align__(16) TokenStageT {
  float4 decay[kHeadDim / 4];
  float4 kh[kHeadDim / 4];
  float4 qh[kHeadDim / 4];
  float4 bkh[kHeadDim / 4];
  float v[kHeadDim];
  float bqk;
  float pad[3];
};
static_assert(sizeof(TokenStageT) == sizeof(TokenStage), "records share their storage");

struct TileLaneT {
  int kq;   // row quad 0..7 within each 32-row block
  int col;  // first of the lane's four value columns
};

__device__ __forceinline__ TileLaneT tile_lane_t() {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  return TileLaneT{lane & 7, warp * 16 + (lane >> 3) * 4};
}

// Offset of register s[4m + c] in a transposed tile.
__device__ __forceinline__ int tile_t_offset(TileLaneT tl, int m, int c) {
  return (tl.col + c) * kHeadDim + 4 * tl.kq + 32 * m;
}

__device__ __forceinline__ void tile_t_store(float* tile, const float4 (&s)[16], TileLaneT tl) {
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      __stcs(reinterpret_cast<float4*>(tile + tile_t_offset(tl, m, c)), s[4 * m + c]);
}

// Decay the four rows x (one column) and add their products with kh and qh
// into the even-row / odd-row halves of a and c.
__device__ __forceinline__ void decay_dot(float4& x, float4 d, float4 kh, float4 qh, float2& a,
                                          float2& c) {
  const float2 lo = __fmul2_rn(f2(x.x, x.y), f2(d.x, d.y));
  const float2 hi = __fmul2_rn(f2(x.z, x.w), f2(d.z, d.w));
  x = make_float4(lo.x, lo.y, hi.x, hi.y);
  a = __ffma2_rn(f2(kh.x, kh.y), lo, a);
  a = __ffma2_rn(f2(kh.z, kh.w), hi, a);
  c = __ffma2_rn(f2(qh.x, qh.y), lo, c);
  c = __ffma2_rn(f2(qh.z, qh.w), hi, c);
}

__device__ __forceinline__ void rank1(float4& x, float4 bkh, float u) {
  const float2 uu = bcast2(u);
  const float2 lo = __ffma2_rn(f2(bkh.x, bkh.y), uu, f2(x.x, x.y));
  const float2 hi = __ffma2_rn(f2(bkh.z, bkh.w), uu, f2(x.z, x.w));
  x = make_float4(lo.x, lo.y, hi.x, hi.y);
}

// One token on a transposed tile (same arithmetic as tile_token_step; here a
// pair is two consecutive rows of one column, so the row sums run in two
// halves, even and odd rows, added at the end); returns the read o for the
// lane's four columns (identical in the 8 lanes of a column quad).
__device__ __forceinline__ float4 tile_t_token_step(float4 (&s)[16], const TokenStageT& ts,
                                                    TileLaneT tl) {
  float2 a[4], c[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) a[q] = c[q] = f2(0.f, 0.f);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    if (m == 2) asm volatile("" ::: "memory");  // bounds the hoisting of the row loads
    const int j = tl.kq + 8 * m;
    const float4 d = ts.decay[j], kh = ts.kh[j], qh = ts.qh[j];
#pragma unroll
    for (int q = 0; q < 4; ++q) decay_dot(s[4 * m + q], d, kh, qh, a[q], c[q]);
  }
  // Fold the halves, then sum over the 8 kq lanes of each column.
  float2 a01 = f2(a[0].x, a[1].x), a23 = f2(a[2].x, a[3].x);
  float2 c01 = f2(c[0].x, c[1].x), c23 = f2(c[2].x, c[3].x);
  a01 = __fadd2_rn(a01, f2(a[0].y, a[1].y)); a23 = __fadd2_rn(a23, f2(a[2].y, a[3].y));
  c01 = __fadd2_rn(c01, f2(c[0].y, c[1].y)); c23 = __fadd2_rn(c23, f2(c[2].y, c[3].y));
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {
    a01 = xor_add2(a01, m); a23 = xor_add2(a23, m);
    c01 = xor_add2(c01, m); c23 = xor_add2(c23, m);
  }
  const float4 vv = *reinterpret_cast<const float4*>(&ts.v[tl.col]);
  const float4 u = make_float4(vv.x - a01.x, vv.y - a01.y, vv.z - a23.x, vv.w - a23.y);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float4 bkh = ts.bkh[tl.kq + 8 * m];
    rank1(s[4 * m + 0], bkh, u.x);
    rank1(s[4 * m + 1], bkh, u.y);
    rank1(s[4 * m + 2], bkh, u.z);
    rank1(s[4 * m + 3], bkh, u.w);
  }
  const float2 bq = bcast2(ts.bqk);
  const float2 o01 = __ffma2_rn(bq, f2(u.x, u.y), c01), o23 = __ffma2_rn(bq, f2(u.z, u.w), c23);
  return make_float4(o01.x, o01.y, o23.x, o23.y);
}

}  // namespace kda
