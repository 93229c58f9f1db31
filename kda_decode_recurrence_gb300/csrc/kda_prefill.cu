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
// One 256-thread CTA per (request, value head), two per SM.  The fp32
// [128, 128] state tile stays in registers (thread (w, i) holds value column
// v = 32 (w % 4) + i for the 64 channels of half w / 4).  The products against
// it run on the 5th-generation tensor cores (tcgen05, accumulators in tensor
// memory), with every fp32 operand split into three bf16 parts p0 + p1 + p2
// (each difference exact in fp32) and the six part-products whose order is
// at most 2 summed, which carries fp32 precision:
//   reads   [ws | qs]^T = S0^T [kt | qt]   M = 128 values, N = 32 tokens,
//           K = 128 channels; A = the state's parts, written to tensor memory
//           by the threads that hold them (tcgen05.st), B = the decayed keys
//           and queries in shared memory (K-major, 128-byte swizzle);
//   update  S^T += u^T ke^T                M = 128 values, N = 128 channels,
//           K = 16 tokens; A = u's parts in tensor memory, B = ke in shared
//           memory (N-major, 128-byte swizzle); the result is read back and
//           added to the decayed registers;
//   outputs O^T = qs + u^T Q^T             M = 128 values, N = 16 tokens,
//           K = 16 tokens; A = u's parts, B = Q's parts in shared memory
//           (K-major, 32-byte swizzle), accumulated onto the reads' qs.
// Each tcgen05.mma of these shapes costs its issuing thread about 90 cycles,
// so the reads are issued by two threads into two accumulators (three
// part-products each, summed when read back), and the update and the outputs
// by one thread each.  The A and Q products and the triangular solve stay on
// the CUDA cores: A and Q beside the reads' issue, and the next chunk's
// staging beside the update and output MMAs.
#include <cstddef>

#include "kda_async.cuh"
#include "kda_recurrence.cuh"
#include "kda_tcgen05.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kC = 16;     // tokens per chunk
constexpr int kTS = 20;    // row stride of the [channel][token] arrays (16-byte aligned rows)
constexpr float kL2Eps = 1e-6f;

// Tensor memory: 256 columns per CTA (two CTAs per SM use all 512).
constexpr uint32_t kTmemCols = 256;
constexpr int kColSParts = 0;   // 3 x 64 columns: the state's bf16 parts (A of the reads)
constexpr int kColReads = 192;  // 2 x 32 columns: the reads' two accumulators [ws | qs]
constexpr int kColUParts = 0;   // 3 x 8 columns: u's bf16 parts (A of the update), after the reads
constexpr int kColUpd = 32;     // 128 columns: the update's accumulator, after the reads

struct PrefillSmem {
  // B operands, 128-byte rows of 64 bf16 in the 128-byte swizzle, 1024-aligned:
  // reads: part, channel panel (64 channels), 32 token rows (kt then qt);
  // update: part, channel atom (64 channels), 16 token rows (ke).
  unsigned char readsB[3][2][2 * kC * 128];
  unsigned char updB[3][2][kC * 128];
  // outputs: part, 16 token rows t of Q[t][0..15] (32 bytes), 32-byte swizzle
  __align__(256) unsigned char outB[3][kC * 32];
  float qh[kC][kHeadDim];    // normalised, scaled queries   [token][channel]
  float kh[kC][kHeadDim];    // normalised keys
  float gg[kC][kHeadDim];    // log-decays
  float vv[kC][kHeadDim];    // values
  __align__(16) float ktT[kHeadDim][kTS];  // kh_t * exp(G_t)     [channel][token]
  __align__(16) float qtT[kHeadDim][kTS];  // qh_t * exp(G_t)
  __align__(16) float kbT[kHeadDim][kTS];  // kh_t * exp(-G_t)
  __align__(16) float eGC[kHeadDim];  // exp(G_end)
  __align__(16) float A[kC][kC];  // A_ts, s < t
  float beta[kC];
  uint64_t bar_reads;        // the reads' MMAs are complete (two issuers)
  uint64_t bar_upd;          // the update's and the outputs' MMAs are complete (two issuers)
  uint32_t tmem_base;
};
// Two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per
// CTA, and 1 KB of alignment slack per CTA for the 1024-byte operands.
static_assert(2 * (sizeof(PrefillSmem) + 1024 + 1024) <= 228 * 1024, "two prefill CTAs fit an SM");

// Token inputs a lane stages: entries 4 lane .. 4 lane + 3.
struct ChunkIn {
  uint2 q, k, v;
  float4 raw;
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
// the gate rows in 16-byte pieces, and the 16 betas.  Thread tid takes
// pieces tid, tid + 256, ...; with 256 threads that fixes its token and piece
// within each row, so the loop is written out per round.
template <int PB>
__device__ __forceinline__ void issue_raw(const DecodeArgs& p, unsigned char* raw, int c0, int t1,
                                          int h, int hv, int tid) {
  static_assert(kThreads == 256 && kC == 16, "the piece assignment below assumes these");
  constexpr int kRowsPerRound = kThreads * PB / (kHeadDim * 2);  // rows of one tensor per round
  constexpr int kRounds = kC / kRowsPerRound;                     // rounds per tensor
  const int part = tid % (kHeadDim * 2 / PB);
  const int tq = tid / (kHeadDim * 2 / PB);
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    const kda_bf16* base = a == 0 ? p.q : (a == 1 ? p.k : p.v);
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int tt = tq + kRowsPerRound * r;
      if (c0 + tt < t1 && kda_in_bounds(c0 + tt < p.T, p.dev_status)) {
        const size_t row = a < 2 ? (size_t)(c0 + tt) * p.H + h : (size_t)(c0 + tt) * p.HV + hv;
        cp_async(raw + a * kC * kHeadDim * 2 + tt * kHeadDim * 2 + part * PB,
                 base + row * kHeadDim + part * (PB / 2), PB);
      }
    }
  }
  // gate rows: 32 pieces of 16 bytes, 8 rows per round
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int tt = (tid >> 5) + 8 * r, gp = tid & 31;
    if (c0 + tt < t1)
      cp_async(raw + kRawG + tt * kHeadDim * 4 + gp * 16,
               p.raw_gate + ((size_t)(c0 + tt) * p.HV + hv) * kHeadDim + gp * 4, 16);
  }
  if (tid < kC && c0 + tid < t1)
    cp_async(raw + kRawB + tid * 4, p.beta_logits + (size_t)(c0 + tid) * p.HV + hv, 4);
  cp_async_commit();
}


// Token slot tt's inputs for lane `lane` (entries 4 lane .. 4 lane + 3) from the raw region.
__device__ __forceinline__ ChunkIn read_raw(const unsigned char* raw, int tt, int lane) {
  ChunkIn in;
  in.q = *reinterpret_cast<const uint2*>(raw + kRawQ + tt * kHeadDim * 2 + lane * 8);
  in.k = *reinterpret_cast<const uint2*>(raw + kRawK + tt * kHeadDim * 2 + lane * 8);
  in.v = *reinterpret_cast<const uint2*>(raw + kRawV + tt * kHeadDim * 2 + lane * 8);
  in.raw = *reinterpret_cast<const float4*>(raw + kRawG + tt * kHeadDim * 4 + lane * 16);
  in.beta_logit = *reinterpret_cast<const float*>(raw + kRawB + tt * 4);
  return in;
}

// Phase 1 for the two token slots tt and tt + 8 of a warp: norms, gate,
// beta into the [token][channel] arrays (zeros for slots past the end of the
// request).  The two slots' four norm reductions are interleaved.
__device__ __forceinline__ void stage_pair(const DecodeArgs& p, const ChunkIn& in0, const ChunkIn& in1,
                                           bool valid0, bool valid1, int hv, PrefillSmem& sm,
                                           int tt, int lane) {
  const int r0 = lane * 4;
  // per-head gate parameters, read here (cache hits) rather than held in
  // registers across the chunk loop
  const float a_exp = expf(__ldg(p.a_log + hv));
  const float4 bias = __ldg(reinterpret_cast<const float4*>(p.dt_bias + (size_t)hv * kHeadDim + r0));
  const ChunkIn* ins[2] = {&in0, &in1};
  float q[2][4], k[2][4], ss[4];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const ChunkIn& in = *ins[j];
    q[j][0] = bf16_lo(in.q.x); q[j][1] = bf16_hi(in.q.x); q[j][2] = bf16_lo(in.q.y); q[j][3] = bf16_hi(in.q.y);
    k[j][0] = bf16_lo(in.k.x); k[j][1] = bf16_hi(in.k.x); k[j][2] = bf16_lo(in.k.y); k[j][3] = bf16_hi(in.k.y);
    float qq = 0.f, kk = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qq = fmaf(q[j][i], q[j][i], qq);
      kk = fmaf(k[j][i], k[j][i], kk);
    }
    ss[2 * j] = qq;
    ss[2 * j + 1] = kk;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int i = 0; i < 4; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], o);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const ChunkIn& in = *ins[j];
    const bool valid = j == 0 ? valid0 : valid1;
    float4 qv = make_float4(0.f, 0.f, 0.f, 0.f), kv = qv, gv = qv, vv = qv;
    float beta = 0.f;
    if (valid) {
      const float qsc = p.q_scale * rsqrtf(ss[2 * j] + kL2Eps);
      const float ksc = rsqrtf(ss[2 * j + 1] + kL2Eps);
      qv = make_float4(q[j][0] * qsc, q[j][1] * qsc, q[j][2] * qsc, q[j][3] * qsc);
      kv = make_float4(k[j][0] * ksc, k[j][1] * ksc, k[j][2] * ksc, k[j][3] * ksc);
      gv = make_float4(p.lower_bound * sigmoidf_(a_exp * (in.raw.x + bias.x)),
                       p.lower_bound * sigmoidf_(a_exp * (in.raw.y + bias.y)),
                       p.lower_bound * sigmoidf_(a_exp * (in.raw.z + bias.z)),
                       p.lower_bound * sigmoidf_(a_exp * (in.raw.w + bias.w)));
      vv = make_float4(bf16_lo(in.v.x), bf16_hi(in.v.x), bf16_lo(in.v.y), bf16_hi(in.v.y));
      beta = sigmoidf_(in.beta_logit);
    }
    const int t = tt + 8 * j;
    *reinterpret_cast<float4*>(&sm.qh[t][r0]) = qv;
    *reinterpret_cast<float4*>(&sm.kh[t][r0]) = kv;
    *reinterpret_cast<float4*>(&sm.gg[t][r0]) = gv;
    *reinterpret_cast<float4*>(&sm.vv[t][r0]) = vv;
    if (lane == 0) sm.beta[t] = beta;
  }
}

// ---- bf16 parts and the 128-byte swizzle

// x = p0 + p1 + p2 as bf16 bit patterns (round to nearest; both residuals are
// exact in fp32, so the three parts carry x to fp32 precision).
__device__ __forceinline__ void split3(float x, uint32_t (&pt)[3]) {
  const __nv_bfloat16 b0 = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(b0);
  const __nv_bfloat16 b1 = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(b1);
  pt[0] = __bfloat16_as_ushort(b0);
  pt[1] = __bfloat16_as_ushort(b1);
  pt[2] = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
}

// The same for a pair: word k holds part k of x0 (low half) and of x1
// (high half), the packing the tensor cores read along K.
__device__ __forceinline__ void split3_pair(float x0, float x1, uint32_t& w0, uint32_t& w1,
                                            uint32_t& w2) {
  const float2 m1 = make_float2(-1.f, -1.f);
  __nv_bfloat162 b = __floats2bfloat162_rn(x0, x1);
  w0 = *reinterpret_cast<uint32_t*>(&b);
  float2 r = __ffma2_rn(m1, make_float2(__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xffff0000u)),
                        make_float2(x0, x1));
  b = __floats2bfloat162_rn(r.x, r.y);
  w1 = *reinterpret_cast<uint32_t*>(&b);
  r = __ffma2_rn(m1, make_float2(__uint_as_float(w1 << 16), __uint_as_float(w1 & 0xffff0000u)), r);
  b = __floats2bfloat162_rn(r.x, r.y);
  w2 = *reinterpret_cast<uint32_t*>(&b);
}

// Byte offset of element `col` (0..63, bf16) of row `row` in a panel of
// 128-byte rows stored in the 128-byte swizzle (16-byte chunk index XOR row
// mod 8; the panel is 1024-byte aligned), the layout the tensor cores read.
__device__ __forceinline__ int sw128(int row, int col) {
  const int byte = col * 2;
  return row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15));
}

// The same in 32-byte rows (elements 0..15) and the 32-byte swizzle (16-byte
// chunk index XOR bit 2 of the row; the panel is 256-byte aligned).
__device__ __forceinline__ int sw32(int row, int col) {
  const int byte = col * 2;
  return row * 32 + ((((byte >> 4) ^ ((row >> 2) & 1)) << 4) | (byte & 15));
}

// The part-products summed, smallest first: (A part, B part) with
// part(A) + part(B) <= 2.
// Pair pr (0..5): (2, 0), (1, 1), (0, 2), (1, 0), (0, 1), (0, 0).
__host__ __device__ constexpr int part_a(int pr) { return pr == 0 ? 2 : (pr == 1 || pr == 3) ? 1 : 0; }
__host__ __device__ constexpr int part_b(int pr) { return pr == 2 ? 2 : (pr == 1 || pr == 4) ? 1 : 0; }

// The reads' MMAs of issuer Q (part-products 3Q .. 3Q + 2, into accumulator
// Q), written out so that every descriptor is a constant offset from one base.
template <int Q>
__device__ __forceinline__ void issue_reads(uint32_t readsB_addr, uint32_t tmem, uint32_t idesc) {
  const uint64_t base = smem_desc_sw128(readsB_addr, 16, 1024);
#pragma unroll
  for (int i = 0; i < 3; ++i) {
#pragma unroll
    for (int j = 0; j < kHeadDim / 16; ++j) {
      const int pr = 3 * Q + i;
      // readsB[part][channel panel] is 4096 bytes; a K step of 16 is 32 bytes
      const uint32_t off = (uint32_t)((part_b(pr) * 2 + (j >> 2)) * (2 * kC * 128) + (j & 3) * 32);
      mma_bf16_tmem_a(tmem + kColReads + 32 * Q, tmem + kColSParts + 64 * part_a(pr) + 8 * j,
                      base + (off >> 4), idesc, (i > 0 || j > 0) ? 1u : 0u);
    }
  }
}

// Two CTAs per SM (128 registers, about 110 KB of shared memory and 256
// tensor-memory columns each), so that a batch of (request, head) items
// twice the SM count runs in one wave.  kPB: the piece size of the q, k, v
// copies (16 when all three pointers are 16-byte aligned, else 8).
template <int kPB>
__global__ void __launch_bounds__(kThreads, 2) kda_prefill_kernel(const DecodeArgs p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

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
  // debug builds: the item's request, heads and slot lie in their tensors
  if (!kda_in_bounds(b < p.B && hv < p.HV && hv / p.G < p.H && slot < p.max_slots, p.dev_status))
    return;

  // Tensor memory and the MMA completion barrier.
  if (warp == 0) tmem_alloc(&sm.tmem_base, kTmemCols);
  if (tid == 0) {
    mbar_init(&sm.bar_reads, 2);
    mbar_init(&sm.bar_upd, 2);
    mbar_fence_init();
  }
  // A and Q's parts above the diagonal blocks stay zero (the products write
  // only the blocks on and below it).
  for (int i = tid; i < kC * kC; i += kThreads) (&sm.A[0][0])[i] = 0.f;
  for (int i = tid; i < 3 * kC * 32 / 4; i += kThreads) reinterpret_cast<uint32_t*>(&sm.outB[0][0])[i] = 0u;
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int lq = warp & 3, half = warp >> 2;
  const int v = 32 * lq + lane;         // this thread's value column (its TMEM lane)
  const int cbase = 64 * half;          // its channels cbase .. cbase + 63
  const uint32_t tlane = tmem + ((uint32_t)(32 * lq) << 16);
  const uint32_t idesc_reads = idesc_bf16(2 * kC, kHeadDim, false, false);
  const uint32_t idesc_upd = idesc_bf16(kHeadDim, kHeadDim, false, true);
  const uint32_t idesc_out = idesc_bf16(kC, kHeadDim, false, false);

  float* tile = p.state_pool + ((size_t)slot * p.HV + hv) * (size_t)(kHeadDim * kHeadDim);
  float st[64];  // S[cbase + c][v]
#pragma unroll
  for (int c = 0; c < 64; ++c) st[c] = __ldcs(tile + (size_t)(cbase + c) * kHeadDim + v);
  const int h = hv / p.G;
  float* out = static_cast<float*>(p.output);

  unsigned char* raw = reinterpret_cast<unsigned char*>(&sm.qh[0][0]);
  uint32_t ph = 0;                // parity of this chunk's phase of both MMA barriers
#if KDA_TEST_HOOKS
  const unsigned long long wait_ns = p.wait_ns;  // test-only: a shorter limit
#else
  constexpr unsigned long long wait_ns = kWaitLimitNs;
#endif
  uint64_t* failed = nullptr;     // uniform: the MMA barrier whose wait gave up
  // Phase 1, staging a chunk's tokens (warp w takes slots w and w + 8): the
  // first chunk here, every later one while the previous chunk's update and
  // output MMAs run.
  auto stage_chunk = [&](int cs) {
    const int ns = min(kC, t1 - cs);
    cp_async_wait_all();
    __syncthreads();  // every thread's copies of this chunk have landed
    ChunkIn in0 = {}, in1 = {};
    if (warp < ns) in0 = read_raw(raw, warp, lane);
    if (warp + 8 < ns) in1 = read_raw(raw, warp + 8, lane);
    __syncthreads();  // the raw region is read: staging overwrites it
    stage_pair(p, in0, in1, warp < ns, warp + 8 < ns, hv, sm, warp, lane);
  };
  issue_raw<kPB>(p, raw, t0, t1, h, hv, tid);
  stage_chunk(t0);
  __syncthreads();
  for (int c0 = t0; c0 < t1; c0 += kC) {
    const int nc = min(kC, t1 - c0);
    // ---- phase 2: cumulative decays, the decayed key/query forms (fp32 for
    // the A and Q products, bf16 parts for the tensor cores), and the
    // chunk-start state's parts into tensor memory.  Thread c (and c + 128
    // for the other half of the tokens) owns channel c.
    {
      const int c = tid & (kHeadDim - 1), th = tid >> 7;
      float Gt[kC];
      float G = 0.f;
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        G += sm.gg[t][c];
        Gt[t] = G;
      }
      const int pc = c >> 6, cc = c & 63;
      const float eG = expf(G);  // exp(G_end): ke = kb exp(G_end)
#pragma unroll
      for (int tt = 0; tt < kC; ++tt) {
        if ((tt >> 3) != th) continue;  // static index into Gt, half of the tokens each
        const float k = sm.kh[tt][c], q = sm.qh[tt][c];
        const float e = expf(Gt[tt]);
        const float kb = k * expf(-Gt[tt]);
        const float kt = k * e, qt = q * e, ke = kb * eG;
        sm.ktT[c][tt] = kt;
        sm.qtT[c][tt] = qt;
        sm.kbT[c][tt] = kb;
        uint32_t pk[3], pq[3], pe[3];
        split3(kt, pk);
        split3(qt, pq);
        split3(ke, pe);
#pragma unroll
        for (int pp = 0; pp < 3; ++pp) {
          *reinterpret_cast<unsigned short*>(&sm.readsB[pp][pc][sw128(tt, cc)]) = (unsigned short)pk[pp];
          *reinterpret_cast<unsigned short*>(&sm.readsB[pp][pc][sw128(kC + tt, cc)]) = (unsigned short)pq[pp];
          *reinterpret_cast<unsigned short*>(&sm.updB[pp][pc][sw128(tt, cc)]) = (unsigned short)pe[pp];
        }
      }
      if (th == 0) sm.eGC[c] = eG;
      // The state's parts: column 64 part + 32 half + m of lane v holds
      // channels cbase + 2m, cbase + 2m + 1 (K pairs, low half first).
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t r0[8], r1[8], r2[8];
#pragma unroll
        for (int m = 0; m < 8; ++m)
          split3_pair(st[16 * q4 + 2 * m], st[16 * q4 + 2 * m + 1], r0[m], r1[m], r2[m]);
        const uint32_t col = kColSParts + 32 * half + 8 * q4;
        tmem_st_8cols(tlane + col, r0);
        tmem_st_8cols(tlane + col + 64, r1);
        tmem_st_8cols(tlane + col + 128, r2);
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // this thread's B-operand writes, for the tensor cores
    }
    tc_fence_before();
    __syncthreads();
    // ---- phase 3a: the reads [ws | qs]^T = S0^T [kt | qt] on the tensor cores.
    // Two issuers (lane 0 of warps 0 and 1), three part-products each into
    // an accumulator of its own: issuing is what limits these small MMAs.
    if (tid == 0 || tid == 32) {
      tc_fence_after();
      const int q = tid >> 5;
      if (q == 0)
        issue_reads<0>(smem_u32(&sm.readsB[0][0][0]), tmem, idesc_reads);
      else
        issue_reads<1>(smem_u32(&sm.readsB[0][0][0]), tmem, idesc_reads);
#if KDA_TEST_HOOKS
      // test-only: this item's second issuer never commits its first reads,
      // so that phase never completes and the wait below gives up
      if (!(q == 1 && item == p.withhold_item && c0 == t0))
#endif
      mma_commit(&sm.bar_reads);
    }
    // qh, kh and gg are consumed: the next chunk's raw inputs start arriving there.
    if (c0 + kC < t1) issue_raw<kPB>(p, raw, c0 + kC, t1, h, hv, tid);
    // ---- phase 3b: the 16 x 16 products A (s < t) and Q (s <= t) on the CUDA
    // cores while the reads run, in warps 2..7 (warps 0 and 1 issue).  Thread
    // (block of tokens t in {2tp, 2tp + 1} x s in {2sp, 2sp + 1}, sp <= tp:
    // the 36 blocks on and below the diagonal; channel phase cq) sums the 32
    // channels c = 4 cc + cq; the 4 phases (lanes 4k .. 4k + 3) are added
    // with two xor-shuffles.
    if (warp >= 2 && warp < 7) {  // whole warps: the shuffles below take every lane
      const int cq = tid & 3, blk = (tid - 64) >> 2;
      const bool active = blk < 36;
      int tp = 0;
      while ((tp + 1) * (tp + 2) / 2 <= blk) ++tp;
      const int sp = blk - tp * (tp + 1) / 2;
      float a[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, q[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      if (active) {
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
      if (active && cq == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int j2 = 0; j2 < 2; ++j2) {
            const int t = 2 * tp + i, s2 = 2 * sp + j2;
            sm.A[t][s2] = s2 < t ? a[i][j2] : 0.f;
          }
        // Q's parts, the B operand of the outputs (K-major: row t holds Q[t][s])
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int t = 2 * tp + i, s2 = 2 * sp;
          uint32_t w0, w1, w2;
          split3_pair(s2 <= t ? q[i][0] : 0.f, s2 + 1 <= t ? q[i][1] : 0.f, w0, w1, w2);
          *reinterpret_cast<uint32_t*>(&sm.outB[0][sw32(t, s2)]) = w0;
          *reinterpret_cast<uint32_t*>(&sm.outB[1][sw32(t, s2)]) = w1;
          *reinterpret_cast<uint32_t*>(&sm.outB[2][sw32(t, s2)]) = w2;
        }
        fence_proxy_async_smem();
      }
    }
    {
      const bool ok = mbar_wait(&sm.bar_reads, ph, wait_ns);  // the reads are done
      if (__syncthreads_or(!ok)) {  // (also: A and Q are in shared memory)
        failed = &sm.bar_reads;
        break;
      }
    }
    tc_fence_after();
    // ---- phase 4: the triangular solve for u, one value column per thread
    // (threads 0..127: TMEM lane v = tid), reading ws straight from the
    // reads' accumulator; u goes to shared memory (outputs) and, as bf16
    // parts, to tensor memory (A of the update: column 8 part + m holds
    // tokens 2m, 2m + 1).
    if (tid < kHeadDim) {
      float ws[kC], ws1[kC];
      tmem_ld_16cols(tlane + kColReads, ws);
      tmem_ld_16cols(tlane + kColReads + 32, ws1);
      tmem_ld_wait();
      float uc[kC];
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        float x = sm.vv[t][v] - (ws[t] + ws1[t]);
#pragma unroll
        for (int s4 = 0; s4 < t; s4 += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(&sm.A[t][s4]);
          x = fmaf(-a4.x, uc[s4], x);
          if (s4 + 1 < t) x = fmaf(-a4.y, uc[s4 + 1], x);
          if (s4 + 2 < t) x = fmaf(-a4.z, uc[s4 + 2], x);
          if (s4 + 3 < t) x = fmaf(-a4.w, uc[s4 + 3], x);
        }
        uc[t] = sm.beta[t] * x;
      }
      uint32_t r0[8], r1[8], r2[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) split3_pair(uc[2 * m], uc[2 * m + 1], r0[m], r1[m], r2[m]);
      tmem_st_8cols(tlane + kColUParts, r0);
      tmem_st_8cols(tlane + kColUParts + 8, r1);
      tmem_st_8cols(tlane + kColUParts + 16, r2);
      tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    // ---- phase 5: the update S^T += u^T ke^T (lane 0 of warp 0) and the
    // outputs' intra-chunk term O^T += u^T Q^T, added into the first reads
    // accumulator's qs columns (lane 0 of warp 1), on the tensor cores
    if (tid == 0) {
      tc_fence_after();
      const uint64_t base = smem_desc_sw128(smem_u32(&sm.updB[0][0][0]), kC * 128, 1024);
#pragma unroll
      for (int pr = 0; pr < 6; ++pr)  // updB[part] is 4096 bytes
        mma_bf16_tmem_a(tmem + kColUpd, tmem + kColUParts + 8 * part_a(pr),
                        base + ((part_b(pr) * 2 * kC * 128) >> 4), idesc_upd, pr > 0 ? 1u : 0u);
      mma_commit(&sm.bar_upd);
    } else if (tid == 32) {
      tc_fence_after();
      const uint64_t base = smem_desc_sw32(smem_u32(&sm.outB[0][0]), 16, 256);
#pragma unroll
      for (int pr = 0; pr < 6; ++pr)  // outB[part] is 512 bytes
        mma_bf16_tmem_a(tmem + kColReads + kC, tmem + kColUParts + 8 * part_a(pr),
                        base + ((part_b(pr) * kC * 32) >> 4), idesc_out, 1u);
      mma_commit(&sm.bar_upd);
    }
    // The next chunk's staging while those MMAs run (its copies were issued
    // in phase 3; vv and beta of this chunk were last read by the solve).
    if (c0 + kC < t1) stage_chunk(c0 + kC);
    {
      const bool ok = mbar_wait(&sm.bar_upd, ph, wait_ns);
      if (__syncthreads_or(!ok)) {
        failed = &sm.bar_upd;
        break;
      }
    }
    tc_fence_after();
    // ---- phase 6: outputs o_t = (both qs accumulators) for tokens
    // 8 h2 .. 8 h2 + 7 of value column v (TMEM lane v), then the chunk-end
    // state S <- D_C S0 + the update
    {
      const int h2 = tid >> 7;
      float qa[kC / 2], qb[kC / 2];
      tmem_ld_8cols(tlane + kColReads + kC + (kC / 2) * h2, qa);
      tmem_ld_8cols(tlane + kColReads + 32 + kC + (kC / 2) * h2, qb);
      tmem_ld_wait();
#pragma unroll
      for (int t = 0; t < kC / 2; ++t) {
        const int tt = (kC / 2) * h2 + t;
        if (tt < nc && kda_in_bounds(c0 + tt < p.T, p.dev_status))
          __stcs(out + ((size_t)(c0 + tt) * p.HV + hv) * kHeadDim + v, qa[t] + qb[t]);
      }
    }
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) {
      float up[32];
      tmem_ld_32cols(tlane + kColUpd + cbase + 32 * q2, up);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i)
        st[32 * q2 + i] = fmaf(st[32 * q2 + i], sm.eGC[cbase + 32 * q2 + i], up[i]);
    }
    tc_fence_before();
    __syncthreads();  // the chunk's shared arrays and tensor-memory columns are free
    ph ^= 1u;
  }
  if (failed) {
    // A wait on the tensor cores gave up: report it, let the copies and the
    // MMAs issued finish (the latter bounded), and leave the state tile as it was.
    cp_async_wait_all();
    if (tid == 0) {
      raise_status(p.dev_status, KDA_DEV_TIMEOUT);
      mbar_wait(failed, ph, wait_ns);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 64; ++c) __stcs(tile + (size_t)(cbase + c) * kHeadDim + v, st[c]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

#if KDA_TEST_HOOKS
// Test-only build: the wait limit and the (request, head) item whose first
// reads are never committed, for the launches that follow.
unsigned long long g_test_prefill_wait_ns = kWaitLimitNs;
long long g_test_prefill_withhold_item = -1;
#endif

cudaError_t launch_kda_prefill(const DecodeArgs& in, cudaStream_t stream) {
  DecodeArgs args = in;
  args.wait_ns = kWaitLimitNs;
  args.withhold_item = -1;
#if KDA_TEST_HOOKS
  args.wait_ns = g_test_prefill_wait_ns;
  args.withhold_item = g_test_prefill_withhold_item;
#endif
  const long long items = (long long)args.B * args.HV;
  if (items == 0) return cudaSuccess;
  const size_t smem = sizeof(PrefillSmem) + 1024;  // + alignment of the 1024-byte operands
  const bool a16 = ((reinterpret_cast<uintptr_t>(args.q) | reinterpret_cast<uintptr_t>(args.k) |
                     reinterpret_cast<uintptr_t>(args.v)) & 15) == 0;
  void (*kernel)(DecodeArgs) = a16 ? kda_prefill_kernel<16> : kda_prefill_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<(unsigned)items, kThreads, smem, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace kda

#if KDA_TEST_HOOKS
// Exported by the test-only build (libkda_testhooks.so), not declared in
// kda.h: set the prefill kernel's wait limit and the work item (request * HV
// + value head) whose first reads are never committed.
extern "C" void kda_test_set_prefill_hooks(long long withhold_item, unsigned long long wait_ns) {
  kda::g_test_prefill_withhold_item = withhold_item;
  kda::g_test_prefill_wait_ns = wait_ns;
}
#endif
