// kda_tc_gemm.cu -- weight-streaming GEMM on the 5th-generation tensor cores
// (tcgen05 + TMEM, operands staged by TMA) for the fused block's two dense
// projections (the fused input projection W_in and the output projection W_o
// of "KDA Block TKG Kernel API Reference").
//
//   Ypart[ks][r][n] = sum_{k in split ks} (Xhi[r][k] + Xlo[r][k]) * W[k][n]
//
// W is bf16 [Kdim, N] stored contraction-first (row k contiguous over n);
// X2 is bf16 [2R, Kdim]: rows 0..R-1 hold the bf16 rounding of the fp32
// activations, rows R..2R-1 the bf16 rounding of the remainder, so the sum of
// the two products carries ~16 significant bits of the activation instead of
// 8 (the weights are exactly bf16).  The path is bound by streaming W from
// HBM; the doubled MMA work is free.  Optionally X2 has a third part, rows
// 2R..3R-1, the bf16 rounding of what hi + lo still misses: the CTAs of the
// tail columns (tail_col and up) then add that part's product into the lo
// accumulator too, which carries the activation to fp32 precision there.
//
// Mapping (swap-AB): MMA M = 128 weight columns (A = W^T tile, MN-major in
// shared memory), MMA N = the hi and lo copies of up to 128 tokens (B = X2
// tile, K-major), MMA K = 16 per instruction, 64 per pipeline stage.  The
// accumulator D[128, N] lives in TMEM.  One CTA per (one or two 128-column
// tiles, contraction split, 128-token block); with two tiles both
// accumulators share each activation tile.  4 warps: warp 0 allocates TMEM
// and its lane 0 issues the weight loads (the weight ring, from HBM), warp 2
// lane 0 the activation loads (their own ring, L2 hits), warp 1 lane 0 the
// MMAs; then all four warps drain TMEM (warp w owns TMEM lanes 32w..32w+31)
// and write the split's partial sums; warp 3 lane 0 first issues this CTA's
// slice of the optional L2 prefetch ranges.  Every wait on an mbarrier is bounded
// by a 1 s timer; on expiry the CTA records an error bit and returns cleanly.
#include <cuda.h>

#include "kda_async.cuh"
#include "kda_common.cuh"
#include "kda_launch.h"
#include "kda_tc_gemm.h"
#include "kda_tcgen05.cuh"
#include "kda_tmap.h"

namespace kda {
namespace {

constexpr int kMaxWStages = 8;           // weight ring depth (chosen per launch)
constexpr int kMaxXStages = 4;           // activation ring depth (chosen per launch)
constexpr int kBK = 64;                  // contraction rows per stage
constexpr int kTileN = 128;              // weight columns per CTA (MMA M)
constexpr int kABytes = kBK * kTileN * 2;  // 16 KiB: two 64x64 swizzled boxes
constexpr int kBoxRows = 32;             // token rows per TMA box of X2

// Instruction descriptor of the swap-AB GEMM: A (weights) MN-major, B
// (activations) K-major.
__device__ __forceinline__ uint32_t instr_desc_bf16(int n, int m) {
  return idesc_bf16(n, m, /*a_mn_major=*/true, /*b_mn_major=*/false);
}

struct GemmShape {
  int R;           // tokens
  int Kdim;        // contraction length (multiple of 64)
  int N;           // output columns (multiple of 8)
  int KS;          // contraction splits
  int accumulate;  // add each split into Y[r][n] instead of writing Ypart[ks]
  int wstages;     // weight ring depth, 2..kMaxWStages
  int xstages;     // activation ring depth, 2..kMaxXStages
  float* tail;     // optional: columns >= tail_col are added (fp32 atomics)
  int tail_col;    // into tail[r][n - tail_col] (row stride tail_n) instead
  int tail_n;      // of being written per split
  int x_parts;     // 2 (hi, lo) or 3 (hi, lo, lo2: the tail CTAs use lo2)
  int xstages_tail;  // activation ring depth of the tail CTAs when x_parts == 3
  L2Prefetch pf;   // ranges to bring into L2 after the MMAs (bytes 0: none)
};

// Dynamic shared memory, 1024-aligned: the weight ring (wstages x mtiles x
// 16 KiB A tiles), the activation ring (xstages x 2*RB*128 B B tiles), then the
// mbarriers and the TMEM base address word.  The two rings have their own
// producers and barriers, so the weight stream (HBM) runs as far ahead as
// its ring allows while the activation tiles (L2 hits) follow their own.
template <int MT>  // 128-column weight tiles per CTA
__global__ void __launch_bounds__(128, 1) tc_gemm_kernel(
    const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
    float* __restrict__ Ypart, const GemmShape sh, int32_t* __restrict__ err) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kTileN * MT;
  const int ks = blockIdx.y;
  const int r0 = blockIdx.z * 128;
  const int rows = min(128, sh.R - r0);
  const int RB = (rows + 31) & ~31;        // token rows per hi/lo half (32..128)
  const int NM = 2 * RB;                   // MMA N
  uint32_t tmem_cols = 64;                 // a power of two >= MT accumulators of NM columns
  while (tmem_cols < (uint32_t)(MT * NM)) tmem_cols *= 2;
  // Tail CTAs (whole tiles at tail_col and up) also stream the lo2 part.
  const bool x3 = sh.x_parts == 3 && sh.tail != nullptr && n0 >= sh.tail_col;
  const int b_bytes = (x3 ? 3 : 2) * RB * 128;  // hi, lo (and lo2) boxes, 128 B per token row
  const int a_bytes = kABytes * MT;        // one weight stage
  const int nW = sh.wstages, nX = x3 ? sh.xstages_tail : sh.xstages;
  const int nkb = sh.Kdim / kBK;
  const int kb0 = (int)((long long)ks * nkb / sh.KS);
  const int kb1 = (int)((long long)(ks + 1) * nkb / sh.KS);

  unsigned char* wring = smem;
  unsigned char* xring = smem + nW * a_bytes;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(xring + nX * b_bytes);
  uint64_t* wempty = wfull + kMaxWStages;
  uint64_t* xfull = wempty + kMaxWStages;
  uint64_t* xempty = xfull + kMaxXStages;
  uint64_t* done = xempty + kMaxXStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  // Progress of the three roles (k-blocks): weights and activations
  // requested, k-blocks whose operands the MMA issuer saw arrive.
  int* prog = reinterpret_cast<int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < nW; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 1);
    }
    for (int s = 0; s < nX; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], 1);
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The weights do not depend on the preceding kernel: the whole weight ring
  // is requested before waiting for it.
  const int pre = min(nW, kb1 - kb0);
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < pre; ++i) {
      unsigned char* a_s = wring + i * a_bytes;
      mbar_expect_tx(&wfull[i], a_bytes);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        tma_load_2d(a_s + mt * kABytes, &tmW, &wfull[i], n0 + mt * kTileN, (kb0 + i) * kBK);
        tma_load_2d(a_s + mt * kABytes + kABytes / 2, &tmW, &wfull[i], n0 + mt * kTileN + 64,
                    (kb0 + i) * kBK);
      }
    }
  }
  pdl_wait();
  pdl_trigger();

  bool ok = true;
  if (warp == 0 && lane == 0) {
    // weight producer
    int kb = kb0 + pre;
    for (; kb < kb1; ++kb) {
      const int i = kb - kb0, s = i % nW, round = i / nW;
      if (!mbar_wait(&wempty[s], (round - 1) & 1)) { ok = false; break; }
      unsigned char* a_s = wring + s * a_bytes;
      mbar_expect_tx(&wfull[s], a_bytes);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        tma_load_2d(a_s + mt * kABytes, &tmW, &wfull[s], n0 + mt * kTileN, kb * kBK);
        tma_load_2d(a_s + mt * kABytes + kABytes / 2, &tmW, &wfull[s], n0 + mt * kTileN + 64,
                    kb * kBK);
      }
    }
    prog[0] = kb - kb0;
  } else if (warp == 2 && lane == 0) {
    // activation producer
    int kb = kb0;
    for (; kb < kb1; ++kb) {
      const int i = kb - kb0, s = i % nX, round = i / nX;
      if (i >= nX && !mbar_wait(&xempty[s], (round - 1) & 1)) { ok = false; break; }
      unsigned char* b_s = xring + s * b_bytes;
      const int k0 = kb * kBK;
      mbar_expect_tx(&xfull[s], b_bytes);
      for (int j = 0; j < RB / kBoxRows; ++j) {
        tma_load_2d(b_s + j * kBoxRows * 128, &tmX, &xfull[s], k0, r0 + j * kBoxRows);
        tma_load_2d(b_s + (RB + j * kBoxRows) * 128, &tmX, &xfull[s], k0, sh.R + r0 + j * kBoxRows);
        if (x3)
          tma_load_2d(b_s + (2 * RB + j * kBoxRows) * 128, &tmX, &xfull[s], k0,
                      2 * sh.R + r0 + j * kBoxRows);
      }
    }
    prog[1] = kb - kb0;
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    const uint32_t idesc = instr_desc_bf16(NM, kTileN);
    const uint32_t idesc3 = instr_desc_bf16(RB, kTileN);  // the lo2 part alone
    int kb = kb0;
    for (; kb < kb1; ++kb) {
      const int i = kb - kb0, sw = i % nW, sx = i % nX;
      if (!mbar_wait(&wfull[sw], (i / nW) & 1) || !mbar_wait(&xfull[sx], (i / nX) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_addr = smem_u32(wring + sw * a_bytes);
      const uint32_t b_addr = smem_u32(xring + sx * b_bytes);
#pragma unroll
      for (int j = 0; j < kBK / 16; ++j) {
        // B: K-major, 128-byte rows, 8-row groups 1 KiB apart; 32 B per step.
        const uint64_t bdesc = smem_desc_sw128(b_addr + j * 32, 16, 1024);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          // A: MN-major, atoms of 64 columns x 8 rows; next column atom 8 KiB
          // away (LBO), next 8-row group 1 KiB away (SBO); 16 rows per step.
          const uint64_t adesc = smem_desc_sw128(a_addr + mt * kABytes + j * 2048, 8192, 1024);
          mma_bf16(tmem + mt * NM, adesc, bdesc, idesc, (kb > kb0 || j > 0) ? 1u : 0u);
          // lo2 rows follow the lo rows in the stage (2*RB*128 bytes in, a
          // multiple of 1 KiB, so the swizzle pattern lines up); their
          // product goes into the lo accumulator, after the MMA above.
          if (x3)
            mma_bf16(tmem + mt * NM + RB, adesc,
                     smem_desc_sw128(b_addr + 2 * RB * 128 + j * 32, 16, 1024), idesc3, 1u);
        }
      }
      mma_commit(&wempty[sw]);
      mma_commit(&xempty[sx]);
    }
    prog[2] = kb - kb0;
    mma_commit(done);  // arrives once every MMA issued above has completed
  }
  __syncwarp();

  // Epilogue: all four warps.  tcgen05.ld is warp-collective, so a warp
  // reads TMEM only if all of its lanes saw the accumulator complete.
  const bool have = __all_sync(0xffffffffu, mbar_wait(done, 0)) != 0;
  if (!have || !ok) {
    if (lane == 0) atomicOr(err, KDA_DEV_TIMEOUT);
  }
  if (have && warp == 3 && lane == 0) {
    // This CTA's slice of each prefetch range (16-byte pieces).
    const size_t ctas = (size_t)gridDim.x * gridDim.y * gridDim.z;
    const size_t cta = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      const size_t nb = sh.pf.bytes[r] & ~(size_t)15;
      if (nb == 0) continue;
      const size_t share = ((nb + ctas - 1) / ctas + 15) & ~(size_t)15;
      const size_t lo = min(cta * share, nb), hi = min(lo + share, nb);
      if (hi > lo)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                         static_cast<const char*>(sh.pf.ptr[r]) + lo),
                     "r"((uint32_t)(hi - lo))
                     : "memory");
    }
  }
  tc_fence_after();
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    if (!have) break;
    const int m = n0 + mt * kTileN + warp * 32 + lane;
    const bool to_tail = sh.tail != nullptr && n0 + mt * kTileN >= sh.tail_col;  // whole tiles
    const uint32_t lane_base = tmem + mt * NM + ((uint32_t)(warp * 32) << 16);
    for (int c = 0; c < RB / 32; ++c) {
      float hi[32], lo[32];
      tmem_ld_32cols(lane_base + c * 32, hi);
      tmem_ld_32cols(lane_base + RB + c * 32, lo);
      tmem_ld_wait();
      if (m < sh.N) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int r = r0 + c * 32 + j;
          if (r < sh.R) {
            if (to_tail)
              atomicAdd(sh.tail + (size_t)r * sh.tail_n + (m - sh.tail_col), hi[j] + lo[j]);
            else if (sh.accumulate)
              atomicAdd(Ypart + (size_t)r * sh.N + m, hi[j] + lo[j]);
            else
              Ypart[((size_t)ks * sh.R + r) * sh.N + m] = hi[j] + lo[j];
          }
        }
      }
    }
  }
  tc_fence_before();
  if (__syncthreads_or(!have || !ok) && threadIdx.x == 0) {
    // A wait gave up.  Let every copy this CTA requested land before its
    // shared memory is released (bounded again): the weight and activation
    // stages the MMA issuer had not yet seen arrive.  (The MMAs it issued
    // are covered by the wait on `done` above.)
    for (int i = prog[2]; i < prog[0]; ++i) mbar_wait(&wfull[i % nW], (uint32_t)(i / nW) & 1u);
    for (int i = prog[2]; i < prog[1]; ++i) mbar_wait(&xfull[i % nX], (uint32_t)(i / nX) & 1u);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// 2-D bf16 tensor map: inner extent `inner` (contiguous), outer extent
// `outer`, box 64 x box_rows, 128-byte swizzle, out-of-range reads as zero.
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
              uint32_t box_rows) {
  return make_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, 64, box_rows);
}

}  // namespace

// Ring depths and tile width for R token rows.  Every CTA streams its weight
// slice once from HBM but re-reads the activations of its contraction range
// from L2, 2*RB*128 bytes per 64-row stage.  For up to 32 rows (8 KiB per
// stage) a CTA takes one 128-column weight tile, two activation stages and the
// deepest weight ring that lets two CTAs share an SM (113 KiB each).  Larger
// row blocks take one CTA per SM (227 KiB) with two 128-column weight tiles
// per activation tile, which halves the activation re-reads, and 3-4
// activation stages.
// With three activation parts the tail CTAs stream 3*RB*128 bytes per stage:
// they take two stages (fewer than the others above 32 rows, so that their
// ring fits in the same shared memory).
struct GemmRings {
  int wstages, xstages, xstages_tail, mtiles;
  size_t smem;
};

static GemmRings gemm_rings(int R, bool x3) {
  const int rows = R < 128 ? R : 128;
  const int RB = (rows + 31) & ~31;
  const size_t b_bytes = (size_t)2 * RB * 128;
  const size_t b3_bytes = (size_t)3 * RB * 128;
  const size_t extra = 1024 + (2 * kMaxWStages + 2 * kMaxXStages + 1) * 8 + 32;
  GemmRings g;
  g.mtiles = RB <= 32 ? 1 : 2;
  const size_t budget = RB <= 32 ? 113 * 1024 : 227 * 1024;
  g.xstages = RB <= 32 ? 2 : (RB == 128 ? 3 : kMaxXStages);
  g.xstages_tail = x3 ? (2 * g.xstages / 3 > 2 ? 2 * g.xstages / 3 : 2) : g.xstages;
  size_t xbytes = g.xstages * b_bytes;
  if (x3 && g.xstages_tail * b3_bytes > xbytes) xbytes = g.xstages_tail * b3_bytes;
  const size_t a_bytes = (size_t)kABytes * g.mtiles;
  int w = (int)((budget - extra - xbytes) / a_bytes);
  if (w > kMaxWStages) w = kMaxWStages;
  g.wstages = w;
  g.smem = extra + xbytes + (size_t)w * a_bytes;
  return g;
}

size_t tc_gemm_smem_bytes(int R) { return gemm_rings(R, false).smem; }

cudaError_t launch_tc_gemm(const kda_bf16* X2, int R, int Kdim, const kda_bf16* W, int N, int KS,
                           float* Ypart, bool accumulate, int32_t* err, cudaStream_t stream,
                           bool pdl, float* tail, int tail_col, const L2Prefetch* prefetch,
                           int x_parts) {
  if (R < 1 || Kdim % kBK != 0 || N % 8 != 0 || KS < 1 || KS > Kdim / kBK ||
      (tail && (tail_col % kTileN != 0 || tail_col < 0 || tail_col >= N)) ||
      (x_parts != 2 && x_parts != 3))
    return cudaErrorInvalidValue;
  const bool x3 = x_parts == 3 && tail != nullptr;
  const GemmRings g = gemm_rings(R, x3);
  // Tail CTAs must hold whole column tiles of their own (tail_col a multiple
  // of the CTA's column span).
  if (x3 && tail_col % (kTileN * g.mtiles) != 0) return cudaErrorInvalidValue;
  CUtensorMap tmW, tmX;
  if (!make_map(&tmW, W, (uint64_t)N, (uint64_t)Kdim, kBK)) return cudaErrorInvalidValue;
  if (!make_map(&tmX, X2, (uint64_t)Kdim, (uint64_t)x_parts * R, kBoxRows))
    return cudaErrorInvalidValue;
  void (*kernel)(CUtensorMap, CUtensorMap, float*, GemmShape, int32_t*) =
      g.mtiles == 2 ? tc_gemm_kernel<2> : tc_gemm_kernel<1>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)g.smem);
  if (e != cudaSuccess) return e;
  GemmShape sh{R, Kdim, N, KS, accumulate ? 1 : 0, g.wstages, g.xstages, tail, tail_col,
               N - tail_col, x_parts, g.xstages_tail,
               L2Prefetch{{nullptr, nullptr, nullptr}, {0, 0, 0}}};
  if (prefetch)
    for (int r = 0; r < 3; ++r)
      if (prefetch->ptr[r] && (reinterpret_cast<uintptr_t>(prefetch->ptr[r]) & 15) == 0) {
        sh.pf.ptr[r] = prefetch->ptr[r];
        sh.pf.bytes[r] = prefetch->bytes[r];
      }
  const int cols = kTileN * g.mtiles;
  dim3 grid((N + cols - 1) / cols, KS, (R + 127) / 128);
  return launch(kernel, grid, dim3(128), g.smem, stream, pdl, tmW, tmX, Ypart, sh, err);
}

}  // namespace kda
