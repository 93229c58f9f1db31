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

__device__ __forceinline__ void decay_dot(float4& x, float4 d, float4 kh, float4 qh, float& a,
                                          float& c) {
  x.x *= d.x; x.y *= d.y; x.z *= d.z; x.w *= d.w;
  a = fmaf(kh.x, x.x, a); a = fmaf(kh.y, x.y, a); a = fmaf(kh.z, x.z, a); a = fmaf(kh.w, x.w, a);
  c = fmaf(qh.x, x.x, c); c = fmaf(qh.y, x.y, c); c = fmaf(qh.z, x.z, c); c = fmaf(qh.w, x.w, c);
}

__device__ __forceinline__ void rank1(float4& x, float4 bkh, float u) {
  x.x = fmaf(bkh.x, u, x.x); x.y = fmaf(bkh.y, u, x.y);
  x.z = fmaf(bkh.z, u, x.z); x.w = fmaf(bkh.w, u, x.w);
}

// One token on a transposed tile (same arithmetic as tile_token_step);
// returns the read o for the lane's four columns (identical in the 8 lanes of
// a column quad).
__device__ __forceinline__ float4 tile_t_token_step(float4 (&s)[16], const TokenStageT& ts,
                                                    TileLaneT tl) {
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    if (m == 2) asm volatile("" ::: "memory");  // bounds the hoisting of the row loads
    const int j = tl.kq + 8 * m;
    const float4 d = ts.decay[j], kh = ts.kh[j], qh = ts.qh[j];
    decay_dot(s[4 * m + 0], d, kh, qh, a.x, c.x);
    decay_dot(s[4 * m + 1], d, kh, qh, a.y, c.y);
    decay_dot(s[4 * m + 2], d, kh, qh, a.z, c.z);
    decay_dot(s[4 * m + 3], d, kh, qh, a.w, c.w);
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {
    a.x += __shfl_xor_sync(0xffffffffu, a.x, m); a.y += __shfl_xor_sync(0xffffffffu, a.y, m);
    a.z += __shfl_xor_sync(0xffffffffu, a.z, m); a.w += __shfl_xor_sync(0xffffffffu, a.w, m);
    c.x += __shfl_xor_sync(0xffffffffu, c.x, m); c.y += __shfl_xor_sync(0xffffffffu, c.y, m);
    c.z += __shfl_xor_sync(0xffffffffu, c.z, m); c.w += __shfl_xor_sync(0xffffffffu, c.w, m);
  }
  const float4 vv = *reinterpret_cast<const float4*>(&ts.v[tl.col]);
  const float4 u = make_float4(vv.x - a.x, vv.y - a.y, vv.z - a.z, vv.w - a.w);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float4 bkh = ts.bkh[tl.kq + 8 * m];
    rank1(s[4 * m + 0], bkh, u.x);
    rank1(s[4 * m + 1], bkh, u.y);
    rank1(s[4 * m + 2], bkh, u.z);
    rank1(s[4 * m + 3], bkh, u.w);
  }
  const float bqk = ts.bqk;
  return make_float4(fmaf(bqk, u.x, c.x), fmaf(bqk, u.y, c.y), fmaf(bqk, u.z, c.z),
                     fmaf(bqk, u.w, c.w));
}

}  // namespace kda
