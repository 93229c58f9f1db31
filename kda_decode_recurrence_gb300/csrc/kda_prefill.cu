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
// held in registers in the accumulator layout of the tensor-core products
// (warp w: value columns 16w .. 16w + 15; see the FragLane comment), and the
// three products against it per chunk run on mma.sync with split-tf32
// operands.
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
  __align__(16) float eGC[kHeadDim];  // exp(G_end)
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

// ---- The state on the tensor cores (mma.sync m16n8k8, tf32 inputs, fp32
// accumulation).  Warp w owns value columns v in [16w, 16w + 16); with
// g = lane / 4 and q = lane % 4, register sf[j][e] holds S[c][v] for
//   c = 8j + 2q + (e & 1),  v = 16w + g + 8 (e >> 1),   j = 0..15,
// which is the accumulator fragment of S^T (rows v, columns c) for the update
// S^T += u^T keT^T, and -- reading positions q and q + 4 of each 8-wide
// k block as c = 8j + 2q and 8j + 2q + 1 -- the A fragment of S^T for the
// reads ws^T = S^T kt and qs^T = S^T qt, with no data movement.  Every fp32
// operand is split into a tf32 part and a tf32 remainder; the three products
// hi*hi + hi*lo + lo*hi carry about 22 significant bits (the dropped lo*lo
// term is below 2^-22 relative).
struct FragLane {
  int g, q, v0;  // v0 = 16w + g
};

__device__ __forceinline__ FragLane frag_lane() {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  return FragLane{lane >> 2, lane & 3, 16 * warp + (lane >> 2)};
}

__device__ __forceinline__ void frag_tile_load(float (&sf)[16][4], const float* tile, FragLane f) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float* r = tile + (8 * j + 2 * f.q) * kHeadDim + f.v0;
    sf[j][0] = __ldcs(r);
    sf[j][1] = __ldcs(r + kHeadDim);
    sf[j][2] = __ldcs(r + 8);
    sf[j][3] = __ldcs(r + kHeadDim + 8);
  }
}

__device__ __forceinline__ void frag_tile_store(float* tile, const float (&sf)[16][4], FragLane f) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float* r = tile + (8 * j + 2 * f.q) * kHeadDim + f.v0;
    __stcs(r, sf[j][0]);
    __stcs(r + kHeadDim, sf[j][1]);
    __stcs(r + 8, sf[j][2]);
    __stcs(r + kHeadDim + 8, sf[j][3]);
  }
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = to_tf32(x);
  lo = to_tf32(x - __uint_as_float(hi));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d += (ahi + alo)(bhi + blo) without the lo * lo term, small terms first.
__device__ __forceinline__ void mma3(float (&d)[4], const uint32_t (&ahi)[4],
                                     const uint32_t (&alo)[4], uint32_t bh0, uint32_t bh1,
                                     uint32_t bl0, uint32_t bl1) {
  mma_tf32(d, alo, bh0, bh1);
  mma_tf32(d, ahi, bl0, bl1);
  mma_tf32(d, ahi, bh0, bh1);
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

  const FragLane fl = frag_lane();
  float* tile = p.state_pool + ((size_t)slot * p.HV + hv) * (size_t)(kHeadDim * kHeadDim);
  float sf[16][4];
  frag_tile_load(sf, tile, fl);
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
    // ---- phase 4: (D_t kh_t)^T S0 and (D_t qh_t)^T S0 for the chunk, as
    // ws^T = S0^T kt and qs^T = S0^T qt (M = the warp's 16 values, N = 16
    // tokens in two tiles, K = the 128 channels in 16 steps of 8).
    {
      float aw[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float aq[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        uint32_t ahi[4], alo[4];
        split_tf32(sf[j][0], ahi[0], alo[0]);  // (row g,     k q)     = S[8j + 2q][v0]
        split_tf32(sf[j][2], ahi[1], alo[1]);  // (row g + 8, k q)
        split_tf32(sf[j][1], ahi[2], alo[2]);  // (row g,     k q + 4) = S[8j + 2q + 1][v0]
        split_tf32(sf[j][3], ahi[3], alo[3]);  // (row g + 8, k q + 4)
        const int c = 8 * j + 2 * fl.q;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          const int t = 8 * n + fl.g;  // B (k q, col g) = x[c][t], (k q + 4, col g) = x[c + 1][t]
          uint32_t bh0, bl0, bh1, bl1;
          split_tf32(sm.ktT[c][t], bh0, bl0);
          split_tf32(sm.ktT[c + 1][t], bh1, bl1);
          mma3(aw[n], ahi, alo, bh0, bh1, bl0, bl1);
          split_tf32(sm.qtT[c][t], bh0, bl0);
          split_tf32(sm.qtT[c + 1][t], bh1, bl1);
          mma3(aq[n], ahi, alo, bh0, bh1, bl0, bl1);
        }
      }
      // accumulator (row v, col t): (g, 2q), (g, 2q + 1), (g + 8, 2q), (g + 8, 2q + 1)
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const int t = 8 * n + 2 * fl.q;
        sm.ws[t][fl.v0] = aw[n][0];
        sm.ws[t + 1][fl.v0] = aw[n][1];
        sm.ws[t][fl.v0 + 8] = aw[n][2];
        sm.ws[t + 1][fl.v0 + 8] = aw[n][3];
        sm.qs[t][fl.v0] = aq[n][0];
        sm.qs[t + 1][fl.v0] = aq[n][1];
        sm.qs[t][fl.v0 + 8] = aq[n][2];
        sm.qs[t + 1][fl.v0 + 8] = aq[n][3];
      }
    }
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
    // The chunk-end state: S <- D_C S0, then S^T += u^T keT^T (M = the warp's
    // 16 values, N = the 128 channels in 16 tiles, K = the 16 tokens in 2
    // steps), accumulated into the state registers.
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float2 e = *reinterpret_cast<const float2*>(&sm.eGC[8 * j + 2 * fl.q]);
      sf[j][0] *= e.x; sf[j][1] *= e.y; sf[j][2] *= e.x; sf[j][3] *= e.y;
    }
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int t = 8 * kk + fl.q;
      uint32_t ahi[4], alo[4];
      split_tf32(sm.u[t][fl.v0], ahi[0], alo[0]);          // (row g,     k q)
      split_tf32(sm.u[t][fl.v0 + 8], ahi[1], alo[1]);      // (row g + 8, k q)
      split_tf32(sm.u[t + 4][fl.v0], ahi[2], alo[2]);      // (row g,     k q + 4)
      split_tf32(sm.u[t + 4][fl.v0 + 8], ahi[3], alo[3]);  // (row g + 8, k q + 4)
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = 8 * j + fl.g;  // B (k q, col g) = keT[c][t], (k q + 4, col g) = keT[c][t + 4]
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(sm.keT[c][t], bh0, bl0);
        split_tf32(sm.keT[c][t + 4], bh1, bl1);
        mma3(sf[j], ahi, alo, bh0, bh1, bl0, bl1);
      }
    }
    __syncthreads();  // the chunk's shared arrays are consumed
  }
  frag_tile_store(tile, sf, fl);
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
