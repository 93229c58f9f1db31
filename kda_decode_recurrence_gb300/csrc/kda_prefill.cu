// kda_prefill.cu -- whole-prompt prefill of the KDA recurrence in chunk form.
//
// Operation: the same recurrence as kda_decode ("Delta-rule write": decay,
// delta write, read after the write; the model runs it over a whole sequence
// with chunk_kda), computed 16 tokens at a time.  Within a chunk, with the
// chunk-start state S0, per-channel cumulative log-decays G_t = g_1 + .. + g_t
// and D_t = diag(exp(G_t)):
//
//   S_t = D_t S0 + sum_{s <= t} D_t D_s^-1 kh_s u_s^T            (state)
//   u_t = beta_t (v_t - (D_t kh_t)^T S0 - sum_{s < t} A_ts u_s)  (values the
//          delta rule actually writes), A_ts = (D_t kh_t) . (D_s^-1 kh_s)
//   o_t = (D_t qh_t)^T S0 + sum_{s <= t} Q_ts u_s,   Q_ts = (D_t qh_t) . (D_s^-1 kh_s)
//   S_end = D_C S0 + sum_s (D_C D_s^-1 kh_s) u_s^T
//
// which is the token-by-token recurrence rearranged (no approximation): u
// comes from one 16 x 16 lower-triangular solve, everything else from dense
// products against the register-resident state.  The factors exp(-G_s) are
// bounded because the lower-bound gate keeps every g >= lower_bound >= -5, so
// |G| <= 80 inside a chunk ("KDA Block TKG Kernel API Reference", :param
// lower_bound: the bound the chunkwise prefill relies on); the softplus gate
// has no such bound and is served by kda_decode.
//
// One 256-thread CTA per (request, value head); the [128, 128] state tile is
// held in registers in the layout of kda_decode (warp w: value columns
// 16w .. 16w + 15; lane = (row group rg, column quad cg); rows rg + 8i).
#include <cstddef>

#include "kda_async.cuh"
#include "kda_recurrence.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kC = 16;     // tokens per chunk
constexpr int kTS = 20;    // row stride of the [channel][token] arrays: 16-byte aligned, and
                           // the 8 row groups of a warp read 8 disjoint bank quads
constexpr float kL2Eps = 1e-6f;

struct PrefillSmem {
  float qh[kC][kHeadDim];    // normalised, scaled queries   [token][channel]
  float kh[kC][kHeadDim];    // normalised keys
  float gg[kC][kHeadDim];    // log-decays
  float vv[kC][kHeadDim];    // values
  __align__(16) float ktT[kHeadDim][kTS];  // kh_t * exp(G_t)     [channel][token]
  __align__(16) float qtT[kHeadDim][kTS];  // qh_t * exp(G_t)
  __align__(16) float kbT[kHeadDim][kTS];  // kh_t * exp(-G_t)
  __align__(16) float keT[kHeadDim][kTS];  // kh_t * exp(G_end - G_t)
  float eGC[kHeadDim];       // exp(G_end)
  float A[kC][kC];           // A_ts, s < t
  float Q[kC][kC];           // Q_ts, s <= t
  __align__(16) float ws[kC][kHeadDim];  // (D_t kh_t)^T S0
  __align__(16) float qs[kC][kHeadDim];  // (D_t qh_t)^T S0
  __align__(16) float u[kC][kHeadDim];
  float beta[kC];
};

// Token inputs a lane stages: entries 4 lane .. 4 lane + 3.
struct ChunkIn {
  uint2 q, k, v;
  float4 raw, bias;
  float beta_logit;
};


// A chunk's raw token inputs are copied asynchronously (cp.async) into the
// region of qh, kh and gg, which is free from the end of phase 2 until the
// next chunk's staging: q, k, v rows (bf16, 8-byte copies: the C ABI
// guarantees 8-byte alignment for them), the raw gate rows (16-byte copies)
// and beta.  Byte offsets in the region:
constexpr int kRawQ = 0, kRawK = kC * kHeadDim * 2, kRawV = 2 * kC * kHeadDim * 2;
constexpr int kRawG = 3 * kC * kHeadDim * 2, kRawB = kRawG + kC * kHeadDim * 4;
constexpr int kRawBytes = kRawB + kC * 4;

static_assert(kRawBytes <= 3 * kC * kHeadDim * (int)sizeof(float), "raw inputs fit in qh, kh, gg");
static_assert(offsetof(PrefillSmem, kh) == offsetof(PrefillSmem, qh) + sizeof(float) * kC * kHeadDim &&
                  offsetof(PrefillSmem, gg) == offsetof(PrefillSmem, kh) + sizeof(float) * kC * kHeadDim,
              "qh, kh, gg are contiguous");

__device__ __forceinline__ void cp_async(void* dst, const void* src, int bytes) {
  if (bytes == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
  else if (bytes == 8)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Issue the copies of tokens c0 .. c0 + 15 (those before t1): the q, k, v
// rows in PB-byte pieces (16 when all three are 16-byte aligned, else 8),
// the gate rows in 16-byte pieces, and the 16 betas.
template <int PB>
__device__ __forceinline__ void issue_raw(const DecodeArgs& p, unsigned char* raw, int c0, int t1,
                                          int h, int hv, int tid) {
  constexpr int kPieces = kHeadDim * 2 / PB;  // per bf16 row
  constexpr int kQKV = 3 * kC * kPieces;
  constexpr int kGate = kC * (kHeadDim * 4 / 16);
  for (int i = tid; i < kQKV + kGate + kC; i += kThreads) {
    if (i < kQKV) {
      const int a = i / (kC * kPieces), j = i - a * (kC * kPieces), tt = j / kPieces;
      const int part = j - tt * kPieces;
      if (c0 + tt >= t1) continue;
      const kda_bf16* base = a == 0 ? p.q : (a == 1 ? p.k : p.v);
      const size_t row = a < 2 ? (size_t)(c0 + tt) * p.H + h : (size_t)(c0 + tt) * p.HV + hv;
      cp_async(raw + a * kC * kHeadDim * 2 + tt * kHeadDim * 2 + part * PB,
               base + row * kHeadDim + part * (PB / 2), PB);
    } else if (i < kQKV + kGate) {
      const int j = i - kQKV, tt = j >> 5, part = j & 31;
      if (c0 + tt >= t1) continue;
      cp_async(raw + kRawG + tt * kHeadDim * 4 + part * 16,
               p.raw_gate + ((size_t)(c0 + tt) * p.HV + hv) * kHeadDim + part * 4, 16);
    } else {
      const int tt = i - kQKV - kGate;
      if (c0 + tt >= t1) continue;
      cp_async(raw + kRawB + tt * 4, p.beta_logits + (size_t)(c0 + tt) * p.HV + hv, 4);
    }
  }
  cp_async_commit();
}


// Token slot tt's inputs for lane `lane` (entries 4 lane .. 4 lane + 3) from the raw region.
__device__ __forceinline__ ChunkIn read_raw(const unsigned char* raw, float4 bias, int tt, int lane) {
  ChunkIn in;
  in.q = *reinterpret_cast<const uint2*>(raw + kRawQ + tt * kHeadDim * 2 + lane * 8);
  in.k = *reinterpret_cast<const uint2*>(raw + kRawK + tt * kHeadDim * 2 + lane * 8);
  in.v = *reinterpret_cast<const uint2*>(raw + kRawV + tt * kHeadDim * 2 + lane * 8);
  in.raw = *reinterpret_cast<const float4*>(raw + kRawG + tt * kHeadDim * 4 + lane * 16);
  in.bias = bias;
  in.beta_logit = *reinterpret_cast<const float*>(raw + kRawB + tt * 4);
  return in;
}

// Phase 1 for one token slot: norms, gate, beta into the [token][channel]
// arrays (zeros for slots past the end of the request).
__device__ __forceinline__ void stage(const DecodeArgs& p, const ChunkIn& in, bool valid, float a_exp,
                                     PrefillSmem& sm, int tt, int lane) {
  const int r0 = lane * 4;
  float4 qv = make_float4(0.f, 0.f, 0.f, 0.f), kv = qv, gv = qv, vv = qv;
  float beta = 0.f;
  if (valid) {
    const float q[4] = {bf16_lo(in.q.x), bf16_hi(in.q.x), bf16_lo(in.q.y), bf16_hi(in.q.y)};
    const float k[4] = {bf16_lo(in.k.x), bf16_hi(in.k.x), bf16_lo(in.k.y), bf16_hi(in.k.y)};
    float qq = 0.f, kk = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qq = fmaf(q[i], q[i], qq);
      kk = fmaf(k[i], k[i], kk);
    }
    const float qsc = p.q_scale * rsqrtf(warp_sum(qq) + kL2Eps);
    const float ksc = rsqrtf(warp_sum(kk) + kL2Eps);
    qv = make_float4(q[0] * qsc, q[1] * qsc, q[2] * qsc, q[3] * qsc);
    kv = make_float4(k[0] * ksc, k[1] * ksc, k[2] * ksc, k[3] * ksc);
    gv = make_float4(p.lower_bound * sigmoidf_(a_exp * (in.raw.x + in.bias.x)),
                     p.lower_bound * sigmoidf_(a_exp * (in.raw.y + in.bias.y)),
                     p.lower_bound * sigmoidf_(a_exp * (in.raw.z + in.bias.z)),
                     p.lower_bound * sigmoidf_(a_exp * (in.raw.w + in.bias.w)));
    vv = make_float4(bf16_lo(in.v.x), bf16_hi(in.v.x), bf16_lo(in.v.y), bf16_hi(in.v.y));
    beta = sigmoidf_(in.beta_logit);
  }
  *reinterpret_cast<float4*>(&sm.qh[tt][r0]) = qv;
  *reinterpret_cast<float4*>(&sm.kh[tt][r0]) = kv;
  *reinterpret_cast<float4*>(&sm.gg[tt][r0]) = gv;
  *reinterpret_cast<float4*>(&sm.vv[tt][r0]) = vv;
  if (lane == 0) sm.beta[tt] = beta;
}

// (x_t)^T S0 for tokens t0 .. t0 + 7 of a chunk, x given as xT[channel][token]:
// in-thread partial sums over the lane's 16 rows, then a butterfly
// reduce-scatter over the 8 row groups (lane bits 16, 8, 4).  Each lane ends
// with one token x 4 columns fully summed and writes it to out[token][col].
__device__ __forceinline__ void project8(const float4 (&s)[16], const float (*xT)[kTS], int t0,
                                         float (*out)[kHeadDim], TileLane tl, int lane) {
  float acc[8][4];
#pragma unroll
  for (int t = 0; t < 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float* xr = xT[tl.rg + 8 * i] + t0;
#pragma unroll
    for (int t4 = 0; t4 < 8; t4 += 4) {
      const float4 x4 = *reinterpret_cast<const float4*>(xr + t4);
      const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int t = t4 + q;
        acc[t][0] = fmaf(xs[q], s[i].x, acc[t][0]);
        acc[t][1] = fmaf(xs[q], s[i].y, acc[t][1]);
        acc[t][2] = fmaf(xs[q], s[i].z, acc[t][2]);
        acc[t][3] = fmaf(xs[q], s[i].w, acc[t][3]);
      }
    }
  }
  // each round keeps the upper half of the remaining tokens where the lane
  // bit is set and adds the partner's copy of them
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4;
#pragma unroll
  for (int t = 0; t < 4; ++t)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float send = u16 ? acc[t][j] : acc[t + 4][j];
      const float keep = u16 ? acc[t + 4][j] : acc[t][j];
      acc[t][j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float send = u8 ? acc[t][j] : acc[t + 2][j];
      const float keep = u8 ? acc[t + 2][j] : acc[t][j];
      acc[t][j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float send = u4 ? acc[0][j] : acc[1][j];
    const float keep = u4 ? acc[1][j] : acc[0][j];
    acc[0][j] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  const int t = t0 + (u16 ? 4 : 0) + (u8 ? 2 : 0) + (u4 ? 1 : 0);
  *reinterpret_cast<float4*>(&out[t][tl.col]) = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
}

// Two CTAs per SM (128 registers, ~100 KB of shared memory each) so that a
// batch of (request, head) items twice the SM count runs in one wave.
// kPB: the piece size of the q, k, v copies (16 when all three pointers are
// 16-byte aligned, else 8).
template <int kPB>
__global__ void __launch_bounds__(kThreads, 2) kda_prefill_kernel(const DecodeArgs p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(smem_raw);

  const int item = blockIdx.x;
  const int b = item / p.HV;
  const int hv = item - b * p.HV;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int slot = p.state_indices[b];
  const int t0 = p.cu_seqlens[b];
  const int t1 = p.cu_seqlens[b + 1];

  if (item == 0 && tid == 0 && (p.cu_seqlens[0] != 0 || p.cu_seqlens[p.B] != p.T))
    raise_status(p.dev_status, KDA_DEV_BAD_SEQLEN);
  if (t0 < 0 || t1 < t0 || t1 > p.T) {
    if (hv == 0 && tid == 0) raise_status(p.dev_status, KDA_DEV_BAD_SEQLEN);
    return;
  }
  if (slot < 0 || slot >= p.max_slots) {
    if (slot >= p.max_slots && hv == 0 && tid == 0) raise_status(p.dev_status, KDA_DEV_BAD_SLOT);
    float* out = static_cast<float*>(p.output);
    for (int i = tid; i < (t1 - t0) * (kHeadDim / 4); i += kThreads)
      *reinterpret_cast<float4*>(out + ((size_t)(t0 + i / (kHeadDim / 4)) * p.HV + hv) * kHeadDim +
                                 (i % (kHeadDim / 4)) * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  if (t1 == t0) return;

  const TileLane tl = tile_lane();
  float* tile = p.state_pool + ((size_t)slot * p.HV + hv) * (size_t)(kHeadDim * kHeadDim);
  float4 s[16];
  tile_load(s, tile, tl);
  const int h = hv / p.G;
  const float a_exp = expf(p.a_log[hv]);
  float* out = static_cast<float*>(p.output);

  unsigned char* raw = reinterpret_cast<unsigned char*>(&sm.qh[0][0]);
  const float4 bias = __ldg(reinterpret_cast<const float4*>(p.dt_bias + (size_t)hv * kHeadDim + lane * 4));
  issue_raw<kPB>(p, raw, t0, t1, h, hv, tid);
  for (int c0 = t0; c0 < t1; c0 += kC) {
    const int nc = min(kC, t1 - c0);
    // ---- phase 1: stage the chunk's tokens, warp w takes slots w and w + 8
    {
      cp_async_wait_all();
      __syncthreads();  // every thread's copies of this chunk have landed
      ChunkIn in0 = {}, in1 = {};
      if (warp < nc) in0 = read_raw(raw, bias, warp, lane);
      if (warp + 8 < nc) in1 = read_raw(raw, bias, warp + 8, lane);
      __syncthreads();  // the raw region is read: staging overwrites it
      stage(p, in0, warp < nc, a_exp, sm, warp, lane);
      stage(p, in1, warp + 8 < nc, a_exp, sm, warp + 8, lane);
    }
    __syncthreads();
    // ---- phase 2: cumulative decays and the decayed key/query forms.
    // Thread c (and c + 128 for the other half of the tokens) owns channel c.
    {
      const int c = tid & (kHeadDim - 1), half = tid >> 7;
      float Gt[kC];
      float G = 0.f;
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        G += sm.gg[t][c];
        Gt[t] = G;
      }
#pragma unroll
      for (int tt = 0; tt < kC; ++tt) {
        if ((tt >> 3) != half) continue;  // static index into Gt, half of the tokens each
        const float k = sm.kh[tt][c], q = sm.qh[tt][c];
        const float e = expf(Gt[tt]);
        sm.ktT[c][tt] = k * e;
        sm.qtT[c][tt] = q * e;
        sm.kbT[c][tt] = k * expf(-Gt[tt]);
        sm.keT[c][tt] = k * expf(G - Gt[tt]);
      }
      if (half == 0) sm.eGC[c] = expf(G);
    }
    __syncthreads();
    // qh, kh and gg are consumed: the next chunk's raw inputs start arriving there.
    if (c0 + kC < t1) issue_raw<kPB>(p, raw, c0 + kC, t1, h, hv, tid);
    // ---- phase 3: the 16 x 16 products A (s < t) and Q (s <= t).  Thread
    // (block of tokens t in {2tp, 2tp + 1} x s in {2sp, 2sp + 1}, channel
    // phase cq) sums the 32 channels c = 4 cc + cq; the 4 phases (lanes
    // 4k .. 4k + 3) are added with two xor-shuffles.  Blocks above the
    // diagonal are zero.
    {
      const int cq = tid & 3, blk = tid >> 2, tp = blk >> 3, sp = blk & 7;
      float a[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, q[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      if (sp <= tp) {
#pragma unroll 8
        for (int cc = 0; cc < kHeadDim / 4; ++cc) {
          const int c = 4 * cc + cq;
          const float2 kt = *reinterpret_cast<const float2*>(&sm.ktT[c][2 * tp]);
          const float2 qt = *reinterpret_cast<const float2*>(&sm.qtT[c][2 * tp]);
          const float2 kb = *reinterpret_cast<const float2*>(&sm.kbT[c][2 * sp]);
          a[0][0] = fmaf(kt.x, kb.x, a[0][0]); a[0][1] = fmaf(kt.x, kb.y, a[0][1]);
          a[1][0] = fmaf(kt.y, kb.x, a[1][0]); a[1][1] = fmaf(kt.y, kb.y, a[1][1]);
          q[0][0] = fmaf(qt.x, kb.x, q[0][0]); q[0][1] = fmaf(qt.x, kb.y, q[0][1]);
          q[1][0] = fmaf(qt.y, kb.x, q[1][0]); q[1][1] = fmaf(qt.y, kb.y, q[1][1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j2 = 0; j2 < 2; ++j2) {
          a[i][j2] += __shfl_xor_sync(0xffffffffu, a[i][j2], 1);
          a[i][j2] += __shfl_xor_sync(0xffffffffu, a[i][j2], 2);
          q[i][j2] += __shfl_xor_sync(0xffffffffu, q[i][j2], 1);
          q[i][j2] += __shfl_xor_sync(0xffffffffu, q[i][j2], 2);
        }
      if (cq == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int j2 = 0; j2 < 2; ++j2) {
            const int t = 2 * tp + i, s2 = 2 * sp + j2;
            sm.A[t][s2] = s2 < t ? a[i][j2] : 0.f;
            sm.Q[t][s2] = s2 <= t ? q[i][j2] : 0.f;
          }
      }
    }
    // ---- phase 4: (D_t kh_t)^T S0 and (D_t qh_t)^T S0 for the chunk
    project8(s, sm.ktT, 0, sm.ws, tl, lane);
    project8(s, sm.ktT, 8, sm.ws, tl, lane);
    project8(s, sm.qtT, 0, sm.qs, tl, lane);
    project8(s, sm.qtT, 8, sm.qs, tl, lane);
    __syncthreads();
    // ---- phase 5: the triangular solve for u, one value column per thread
    if (tid < kHeadDim) {
      const int v = tid;
      float uc[kC];
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        float x = sm.vv[t][v] - sm.ws[t][v];
#pragma unroll
        for (int s2 = 0; s2 < t; ++s2) x = fmaf(-sm.A[t][s2], uc[s2], x);
        uc[t] = sm.beta[t] * x;
        sm.u[t][v] = uc[t];
      }
    }
    __syncthreads();
    // ---- phase 6: outputs and the chunk-end state
    {
      const int v = tid & (kHeadDim - 1), half = tid >> 7;
#pragma unroll
      for (int t = 0; t < kC / 2; ++t) {
        const int tt = half * (kC / 2) + t;
        if (tt < nc) {
          float o = sm.qs[tt][v];
#pragma unroll
          for (int s2 = 0; s2 <= tt; ++s2) o = fmaf(sm.Q[tt][s2], sm.u[s2][v], o);
          __stcs(out + ((size_t)(c0 + tt) * p.HV + hv) * kHeadDim + v, o);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float e = sm.eGC[tl.rg + 8 * i];
      s[i].x *= e; s[i].y *= e; s[i].z *= e; s[i].w *= e;
    }
#pragma unroll
    for (int t4 = 0; t4 < kC; t4 += 4) {
      float4 ut[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) ut[q] = *reinterpret_cast<const float4*>(&sm.u[t4 + q][tl.col]);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 k4 = *reinterpret_cast<const float4*>(&sm.keT[tl.rg + 8 * i][t4]);
        const float ks[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          s[i].x = fmaf(ks[q], ut[q].x, s[i].x); s[i].y = fmaf(ks[q], ut[q].y, s[i].y);
          s[i].z = fmaf(ks[q], ut[q].z, s[i].z); s[i].w = fmaf(ks[q], ut[q].w, s[i].w);
        }
      }
    }
    __syncthreads();  // the chunk's shared arrays are consumed
  }
  tile_store(tile, s, tl);
}

}  // namespace

cudaError_t launch_kda_prefill(const DecodeArgs& args, cudaStream_t stream) {
  const long long items = (long long)args.B * args.HV;
  if (items == 0) return cudaSuccess;
  const size_t smem = sizeof(PrefillSmem);
  const bool a16 = ((reinterpret_cast<uintptr_t>(args.q) | reinterpret_cast<uintptr_t>(args.k) |
                     reinterpret_cast<uintptr_t>(args.v)) & 15) == 0;
  void (*kernel)(DecodeArgs) = a16 ? kda_prefill_kernel<16> : kda_prefill_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<(unsigned)items, kThreads, smem, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace kda
