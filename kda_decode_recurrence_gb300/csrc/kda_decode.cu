// kda_decode.cu -- the KDA decode recurrence over a slot-indexed state pool.
//
// Operation ("KdaDecode": Tensor Shapes, Default parameters; "Delta-rule
// write": the naive recurrent loop): for each request b and value head hv the
// fp32 [128, 128] state tile state_pool[state_indices[b], hv] is advanced over
// the request's tokens by decay -> delta write -> read, and written back.
//
// GB300 design (HBM-bound: 64 KiB in + 64 KiB out per tile, ~1 flop/byte):
//   * one 256-thread CTA per (request, value head) tile; two CTAs per SM so one
//     tile's loads are in flight while the other computes;
//   * the tile is loaded once, straight into registers, with 128-bit streaming
//     loads (each warp instruction covers 8 rows x 64 contiguous bytes), held
//     on chip across all of the request's tokens, and stored once;
//   * warp w owns value columns [16w, 16w + 16); lane = (row group rg 0..7,
//     column quad cg 0..3) and holds rows rg, rg + 8, ..., rg + 120 of its four
//     columns (16 float4 = 64 registers);
//   * the k- and q-contractions over the 128 key rows are in-thread sums over
//     16 rows followed by three xor-shuffles across the 8 row groups, so warps
//     never wait for each other inside a token;
//   * per-token vectors (normalised q and k, exp(g), beta * k, v, beta, q.k)
//     are prepared once per CTA, one warp per token, in shared memory, up to 8
//     tokens per staging round.
//
// The read uses q^T S_new = q^T (D S) + beta (q.k) u with u = v - k^T (D S),
// which is the same quantity as reading after the write, with one pass over
// the tile per token instead of two.
#include "kda_recurrence.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 8;  // tokens staged per round (one warp each)
constexpr float kL2Eps = 1e-6f;

__device__ __forceinline__ void stage_token(const DecodeArgs& p, int t, int h, int hv,
                                            float a_exp, float q_scale, TokenStage& ts,
                                            int lane) {
  const int r0 = lane * 4;
  const uint2 qraw = *reinterpret_cast<const uint2*>(p.q + ((size_t)t * p.H + h) * kHeadDim + r0);
  const uint2 kraw = *reinterpret_cast<const uint2*>(p.k + ((size_t)t * p.H + h) * kHeadDim + r0);
  const uint2 vraw = *reinterpret_cast<const uint2*>(p.v + ((size_t)t * p.HV + hv) * kHeadDim + r0);
  const float4 raw = *reinterpret_cast<const float4*>(p.raw_gate + ((size_t)t * p.HV + hv) * kHeadDim + r0);
  const float4 bias = *reinterpret_cast<const float4*>(p.dt_bias + (size_t)hv * kHeadDim + r0);
  const float beta_logit = p.beta_logits[(size_t)t * p.HV + hv];

  const float q[4] = {bf16_lo(qraw.x), bf16_hi(qraw.x), bf16_lo(qraw.y), bf16_hi(qraw.y)};
  const float k[4] = {bf16_lo(kraw.x), bf16_hi(kraw.x), bf16_lo(kraw.y), bf16_hi(kraw.y)};
  float qq = 0.f, kk = 0.f, qk = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    qq = fmaf(q[i], q[i], qq);
    kk = fmaf(k[i], k[i], kk);
    qk = fmaf(q[i], k[i], qk);
  }
  qq = warp_sum(qq);
  kk = warp_sum(kk);
  qk = warp_sum(qk);
  const float qs = q_scale * rsqrtf(qq + kL2Eps);
  const float ks = rsqrtf(kk + kL2Eps);
  const float beta = sigmoidf_(beta_logit);
  const float xr[4] = {raw.x + bias.x, raw.y + bias.y, raw.z + bias.z, raw.w + bias.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float g = (p.gate_mode == KDA_GATE_SOFTPLUS) ? -a_exp * softplusf_(xr[i])
                                                        : p.lower_bound * sigmoidf_(a_exp * xr[i]);
    const float kh = k[i] * ks;
    ts.row[r0 + i] = RowCoef{expf(g), kh, q[i] * qs, beta * kh};
  }
  ts.v[r0 + 0] = bf16_lo(vraw.x);
  ts.v[r0 + 1] = bf16_hi(vraw.x);
  ts.v[r0 + 2] = bf16_lo(vraw.y);
  ts.v[r0 + 3] = bf16_hi(vraw.y);
  if (lane == 0) ts.bqk = beta * qk * qs * ks;
}

__global__ void __launch_bounds__(kThreads, 2) kda_decode_kernel(const DecodeArgs p) {
  __shared__ TokenStage stage[kChunk];

  const int item = blockIdx.x;
  const int b = item / p.HV;
  const int hv = item - b * p.HV;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int slot = p.state_indices[b];
  const int t0 = p.cu_seqlens[b];
  const int t1 = p.cu_seqlens[b + 1];

  if (item == 0 && threadIdx.x == 0 && (p.cu_seqlens[0] != 0 || p.cu_seqlens[p.B] != p.T))
    raise_status(p.dev_status, KDA_DEV_BAD_SEQLEN);
  if (t0 < 0 || t1 < t0 || t1 > p.T) {
    if (hv == 0 && threadIdx.x == 0) raise_status(p.dev_status, KDA_DEV_BAD_SEQLEN);
    return;
  }
  if (slot < 0 || slot >= p.max_slots) {
    if (slot >= p.max_slots && hv == 0 && threadIdx.x == 0)
      raise_status(p.dev_status, KDA_DEV_BAD_SLOT);
    const int quads = (t1 - t0) * (kHeadDim / 4);
    for (int i = threadIdx.x; i < quads; i += kThreads) {
      const int t = t0 + i / (kHeadDim / 4);
      const int c = (i % (kHeadDim / 4)) * 4;
      *reinterpret_cast<float4*>(p.output + ((size_t)t * p.HV + hv) * kHeadDim + c) =
          make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  if (t1 == t0) return;  // nothing to advance: state left bit-identical

  const TileLane tl = tile_lane();
  float* tile = p.state_pool + ((size_t)slot * p.HV + hv) * (size_t)(kHeadDim * kHeadDim);
  float4 s[16];
  tile_load(s, tile, tl);

  const int h = hv / p.G;
  const float a_exp = expf(p.a_log[hv]);

  for (int c0 = t0; c0 < t1; c0 += kChunk) {
    const int nc = min(kChunk, t1 - c0);
    if (c0 != t0) __syncthreads();  // the previous round's stage is consumed
    if (warp < nc) stage_token(p, c0 + warp, h, hv, a_exp, p.q_scale, stage[warp], lane);
    __syncthreads();
    for (int j = 0; j < nc; ++j) {
      const float4 o = tile_token_step(s, stage[j], tl);
      if (tl.rg == 0)
        __stcs(reinterpret_cast<float4*>(p.output + ((size_t)(c0 + j) * p.HV + hv) * kHeadDim + tl.col), o);
    }
  }
  tile_store(tile, s, tl);
}

}  // namespace

cudaError_t launch_kda_decode(const DecodeArgs& args, cudaStream_t stream) {
  const long long items = (long long)args.B * args.HV;
  if (items == 0) return cudaSuccess;
  kda_decode_kernel<<<(unsigned)items, kThreads, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace kda
