// kda_block.cu -- the fused KDA block for token generation (n >= 1 tokens per
// request).
//
// Operation: "KDA Block TKG Kernel API Reference" (Background; :param hidden:,
// gamma_in, W_in, W_fb, W_gb, conv_w, A_log, dt_bias, gamma_o, W_o, out, S,
// conv_state, scale, rms_norm_eps, lower_bound), the recurrence of "Delta-rule
// write".
//
// Kernel chain on the caller's stream (rows r = b * n + j for token j of request
// b, R = B * n):
//   1. rmsnorm      x = hidden * rsqrt(mean(hidden^2) + eps) * gamma_in, written
//                   as three bf16 parts X3 [3R, Hd] (hi, lo, lo2) for the
//                   tensor cores; out and the projection tail zeroed
//   2. proj GEMM    tcgen05, P_part[ks] = x[:, split ks] . W_in[split ks, :]   [KS1, R, I]
//                   (split-K so every SM streams a slice of the 103 MB W_in;
//                   consumers add the KS1 partial sums of q, k, v from hi + lo;
//                   the g_a, beta, f_a columns take hi + lo + lo2, i.e. fp32
//                   activations, because the forget gate amplifies their
//                   error up to |lower_bound| exp(A_log) / 4 times, and are
//                   summed in place into `tail`); as
//                   its CTAs finish they bring conv_state, W_fb and W_gb
//                   into L2 for kernels 3 and 4
//   3. latent       graw = f_a . W_fb, z = g_a . W_gb (CUDA cores)            [R, CQ + CV]
//   4. prep         one CTA per (b, 8 heads), channels read coalesced: short
//                   conv + SiLU + conv_state update of the q, k, v channels,
//                   forget gate, beta, L2 norms -> the per-head token vectors
//                   (the same staging record kda_decode builds) and the output
//                   gate gamma_o * output_gate(z)
//   5. recurrence   one CTA per (b, h): the register-tile delta-rule step on
//                   S[b, h] (shared with kda_decode), gated output RMSNorm ->
//                   bf16 hi/lo on2
//   6. out GEMM     tcgen05, out += on[:, split ks] . W_o[split ks, :] for each
//                   split (fp32 atomics into the rows the RMSNorm kernel zeroed)
// Kernels 2, 4, 5 and 6 are programmatic dependents of the kernel before them
// (each requests what does not depend on it -- weights, state tiles, conv
// windows -- before waiting); the latent kernel is launched in plain stream
// order so that its CTAs spread over every SM.
// Intermediates live in the caller's workspace (a few MB: L2-resident).
//
// Output-gate activation (the page calls the output RMSNorm "gated" and names
// no activation): sigmoid by default; building with
// -DKDA_BLOCK_OUTPUT_GATE_SWISH=1 selects swish, z * sigmoid(z).
#include "kda_recurrence.cuh"
#include "kda_launch.h"
#include "kda_tc_gemm.h"

namespace kda {
namespace {

#ifndef KDA_BLOCK_OUTPUT_GATE_SWISH
#define KDA_BLOCK_OUTPUT_GATE_SWISH 0
#endif

__device__ __forceinline__ float output_gate(float z) {
#if KDA_BLOCK_OUTPUT_GATE_SWISH
  return z * sigmoidf_(z);
#else
  return sigmoidf_(z);
#endif
}

constexpr int kThreads = 256;
constexpr int kKS1 = 3;        // contraction splits of the W_in GEMM (99 tiles x 3 = 297 CTAs: one wave at 2 per SM)
constexpr int kKS2 = 9;        // contraction splits of the W_o GEMM (32 tiles x 9 = 288 CTAs)

struct Layout {
  int R, I, CQ, CV, KS1, KS2;
  int TC, TN;  // projection columns >= TC (g_a, beta, f_a): TN of them, summed in place
  size_t x2, ppart, tail, gz, stage, zgate, on2, err, total;
};

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

bool make_layout(int B, int n, int Hd, int nh, int K, int V, int Kc, Layout* L) {
  if (B < 1 || n < 1 || K != kHeadDim || V != kHeadDim || Kc < 2 || Kc > 4 || Hd < 128 ||
      Hd % 128 != 0 || nh < 8 || nh % 8 != 0)
    return false;
  L->R = B * n;
  L->CQ = K * nh;
  L->CV = V * nh;
  L->I = 2 * L->CQ + L->CV + 2 * K + nh;
  L->TC = 2 * L->CQ + L->CV;  // a multiple of 128
  L->TN = L->I - L->TC;
  L->KS1 = Hd / 64 < kKS1 ? Hd / 64 : kKS1;        // splits <= 64-row contraction blocks
  L->KS2 = L->CV / 64 < kKS2 ? L->CV / 64 : kKS2;
  size_t off = 0;
  L->x2 = off;    off = align_up(off + 3 * sizeof(kda_bf16) * (size_t)L->R * Hd);
  L->ppart = off; off = align_up(off + sizeof(float) * (size_t)L->KS1 * L->R * L->I);
  L->tail = off;  off = align_up(off + sizeof(float) * (size_t)L->R * L->TN);
  L->gz = off;    off = align_up(off + sizeof(float) * (size_t)L->R * (L->CQ + L->CV));
  L->stage = off; off = align_up(off + sizeof(TokenStage) * (size_t)L->R * nh);
  L->zgate = off; off = align_up(off + sizeof(float) * (size_t)L->R * L->CV);
  L->on2 = off;   off = align_up(off + 2 * sizeof(kda_bf16) * (size_t)L->R * L->CV);
  L->err = off;   off = align_up(off + sizeof(int32_t));
  L->total = off;
  return true;
}

// fp32 -> bf16 hi + bf16 lo with hi + lo == x to ~2^-16 relative.
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16* hi, __nv_bfloat16* lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  *hi = h;
  *lo = __float2bfloat16_rn(x - __bfloat162float(h));
}

// Four consecutive values as three bf16 parts hi + lo + lo2, each stored as
// one 8-byte word: hi = bf16(x), lo = bf16(x - hi), lo2 = bf16(x - hi - lo).
// Both differences are exact in fp32, so hi + lo keeps ~16 significant bits
// of x and hi + lo + lo2 all of them (to within the last bit or two).
__device__ __forceinline__ uint2 pack_bf16x4(float a, float b, float c, float d, float4* back) {
  const __nv_bfloat162 p01 = __floats2bfloat162_rn(a, b);
  const __nv_bfloat162 p23 = __floats2bfloat162_rn(c, d);
  const float2 f01 = __bfloat1622float2(p01), f23 = __bfloat1622float2(p23);
  *back = make_float4(f01.x, f01.y, f23.x, f23.y);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&p01);
  w.y = *reinterpret_cast<const uint32_t*>(&p23);
  return w;
}

__device__ __forceinline__ void split_bf16x4_3(float4 x, __nv_bfloat16* hi, __nv_bfloat16* lo,
                                               __nv_bfloat16* lo2) {
  float4 h, l, l2;
  *reinterpret_cast<uint2*>(hi) = pack_bf16x4(x.x, x.y, x.z, x.w, &h);
  const float4 r = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
  *reinterpret_cast<uint2*>(lo) = pack_bf16x4(r.x, r.y, r.z, r.w, &l);
  *reinterpret_cast<uint2*>(lo2) = pack_bf16x4(r.x - l.x, r.y - l.y, r.z - l.z, r.w - l.w, &l2);
}

__device__ __forceinline__ float block_sum(float x, float* red /* [kThreads/32] */) {
  x = warp_sum(x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) t += red[w];
  return t;
}

constexpr int kNormThreads = 1024;
constexpr int kNormCache = 4;  // float4 per thread held in registers (Hd <= 16384)

// 1. input RMSNorm, one CTA per row: the row is read once into registers,
// reduced, and written as three bf16 parts (rows r, R + r, 2R + r of X3).
// The CTA also zeroes its row of `out`, which the output projection
// accumulates into, and its row of the projection tail.
__global__ void __launch_bounds__(kNormThreads) rmsnorm_split_kernel(
    const float* __restrict__ hidden, const float* __restrict__ gamma,
    __nv_bfloat16* __restrict__ X3, float* __restrict__ out, float* __restrict__ tail, int TN,
    int R, int Hd, float eps) {
  __shared__ float red[kNormThreads / 32];
  pdl_trigger();
  const float* x = hidden + (size_t)blockIdx.x * Hd;
  float4 xv[kNormCache];  // gamma is read again at the end (an L1 / L2 hit)
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < kNormCache; ++c) {
    const int i = (threadIdx.x + c * kNormThreads) * 4;
    const bool in = i < Hd;
    xv[c] = in ? *reinterpret_cast<const float4*>(x + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += xv[c].x * xv[c].x + xv[c].y * xv[c].y + xv[c].z * xv[c].z + xv[c].w * xv[c].w;
  }
  for (int i = (threadIdx.x + kNormCache * kNormThreads) * 4; i < Hd; i += kNormThreads * 4) {
    const float4 v = *reinterpret_cast<const float4*>(x + i);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float inv = rsqrtf(tot / (float)Hd + eps);
  __nv_bfloat16* hi = X3 + (size_t)blockIdx.x * Hd;
  __nv_bfloat16* lo = X3 + ((size_t)R + blockIdx.x) * Hd;
  __nv_bfloat16* lo2 = X3 + ((size_t)2 * R + blockIdx.x) * Hd;
  float* orow = out + (size_t)blockIdx.x * Hd;
  for (int i = threadIdx.x; i < TN; i += kNormThreads) tail[(size_t)blockIdx.x * TN + i] = 0.f;
  auto emit = [&](int i, float4 v, float4 g) {
    split_bf16x4_3(make_float4(v.x * inv * g.x, v.y * inv * g.y, v.z * inv * g.z, v.w * inv * g.w),
                   hi + i, lo + i, lo2 + i);
    *reinterpret_cast<float4*>(orow + i) = make_float4(0.f, 0.f, 0.f, 0.f);
  };
#pragma unroll
  for (int c = 0; c < kNormCache; ++c) {
    const int i = (threadIdx.x + c * kNormThreads) * 4;
    if (i < Hd) emit(i, xv[c], *reinterpret_cast<const float4*>(gamma + i));
  }
  for (int i = (threadIdx.x + kNormCache * kNormThreads) * 4; i < Hd; i += kNormThreads * 4)
    emit(i, *reinterpret_cast<const float4*>(x + i), *reinterpret_cast<const float4*>(gamma + i));
}

// 3. gate latents on the CUDA cores: gz[r][c] = f_a[r] . W_fb[:, c] for
// c < CQ and g_a[r] . W_gb[:, c - CQ] after, with f_a and g_a read from the
// projection (Ppart holds KS1 partial sums to add; the block passes the
// in-place tail with KS1 = 1).  Grid ((CQ + CV) / 32, ceil(R / 32)), 256
// threads; a CTA computes a 32-row x 32-column block.  Its weight tile
// (128 x 32) is converted to fp32 in shared memory; the activation panel is
// stored k-major.  Warp w takes contraction rows
// [16w, 16w + 16) and lane (rb, cb) a 4-row x 8-column register block, so
// each k costs three 16-byte shared loads for 32 FMAs; the eight warps'
// partial blocks are then added through shared memory.
constexpr int kLatTile = 32;                 // rows and columns per CTA
constexpr int kLatKPerWarp = kHeadDim / 8;   // contraction rows per warp

__global__ void __launch_bounds__(256) latent_kernel(
    const float* __restrict__ Ppart, int KS1, int R, int I, int off_fa, int off_ga,
    const kda_bf16* __restrict__ W_fb, int CQ, const kda_bf16* __restrict__ W_gb, int CV,
    float* __restrict__ gz) {
  // Operands (xT 16 KiB + w 16 KiB), then reused for the partial sums.
  __shared__ __align__(16) float buf[8 * kLatTile * kLatTile];
  float (*xT)[kLatTile] = reinterpret_cast<float (*)[kLatTile]>(buf);                        // [k][r]
  float (*wf)[kLatTile] = reinterpret_cast<float (*)[kLatTile]>(buf + kHeadDim * kLatTile);  // [k][c]
  float (*part)[kLatTile * kLatTile] = reinterpret_cast<float (*)[kLatTile * kLatTile]>(buf);

  const int t = threadIdx.x;
  const int c0 = blockIdx.x * kLatTile;
  const bool is_fb = c0 < CQ;  // CQ is a multiple of 32
  const kda_bf16* W = is_fb ? W_fb : W_gb;
  const int N = is_fb ? CQ : CV;
  const int cbase = is_fb ? c0 : c0 - CQ;
  const int off = is_fb ? off_fa : off_ga;
  const int r0 = blockIdx.y * kLatTile;

  {  // weight tile: 128 rows x 32 bf16 = 4 x 16 bytes per row; 2 chunks per thread
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int e = t + 256 * i, k = e >> 2, q = e & 3;
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(W + (size_t)k * N + cbase) + q);
      float* dst = &wf[k][8 * q];
      *reinterpret_cast<float4*>(dst) = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
      *reinterpret_cast<float4*>(dst + 4) =
          make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
    }
  }
  pdl_wait();  // (a no-op: the kernel is launched in plain stream order)
  pdl_trigger();
  {  // activation panel, transposed: lane = row, so each k-row store is conflict-free
    const int r = t & 31, kq0 = t >> 5;  // kq = 4-column group of k
    const bool valid = r0 + r < R;
    // All of the thread's partial-sum loads are issued before any is used:
    // one L2 round trip instead of one per split and column group.
    float4 v[4][kKS1];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int ks = 0; ks < kKS1; ++ks)
        v[i][ks] = (valid && ks < KS1)
                       ? __ldg(reinterpret_cast<const float4*>(
                                   Ppart + ((size_t)ks * R + r0 + r) * I + off) + kq0 + 8 * i)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int kq = kq0 + 8 * i;
      float4 acc = v[i][0];
#pragma unroll
      for (int ks = 1; ks < kKS1; ++ks) {
        acc.x += v[i][ks].x; acc.y += v[i][ks].y; acc.z += v[i][ks].z; acc.w += v[i][ks].w;
      }
      xT[4 * kq + 0][r] = acc.x;
      xT[4 * kq + 1][r] = acc.y;
      xT[4 * kq + 2][r] = acc.z;
      xT[4 * kq + 3][r] = acc.w;
    }
  }
  __syncthreads();
  const int warp = t >> 5, lane = t & 31;
  const int rb = lane >> 2, cb = lane & 3;  // rows 4rb..4rb+3, columns 8cb..8cb+7
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
#pragma unroll 4
  for (int kk = 0; kk < kLatKPerWarp; ++kk) {
    const int k = warp * kLatKPerWarp + kk;
    const float4 x = *reinterpret_cast<const float4*>(&xT[k][4 * rb]);
    const float4 wa = *reinterpret_cast<const float4*>(&wf[k][8 * cb]);
    const float4 wb = *reinterpret_cast<const float4*>(&wf[k][8 * cb + 4]);
    const float xv[4] = {x.x, x.y, x.z, x.w};
    const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
  }
  __syncthreads();  // every warp is done with xT and wf: reuse them for the partials
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float* dst = &part[warp][(4 * rb + i) * kLatTile + 8 * cb];
    *reinterpret_cast<float4*>(dst) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
  __syncthreads();
  {  // thread t: row t / 8, columns 4 (t % 8) .. + 3, summed over the warps in order
    const int r = t >> 3, c4 = (t & 7) * 4;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const float4 v = *reinterpret_cast<const float4*>(&part[w][r * kLatTile + c4]);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    if (r0 + r < R) *reinterpret_cast<float4*>(gz + (size_t)(r0 + r) * (CQ + CV) + c0 + c4) = s;
  }
}

struct PrepArgs {
  const float* Ppart;
  const float* tail;  // [R, TN]: g_a, beta, f_a summed over the splits
  const float* gz;
  const kda_bf16* conv_w;
  float* conv_state;
  const float* A_log;
  const float* dt_bias;
  const float* gamma_o;
  TokenStage* stage;  // [R, nh]
  float* zgate;       // [R, nh, V]: gamma_o[d] * output_gate(z)
  int32_t* status;    // device status word (debug builds' index checks)
  float scale, lower_bound, l2_eps;
  int R, n, I, KS1, nh, Kc, CQ, CV, TN;
};

// One channel of the depthwise causal conv: the window is conv_state[b, s, c,
// 0..Kc-2] (oldest first) followed by the new projection value; taps
// conv_w[s, 0..Kc-1, c] (tap 0 oldest).
struct ConvChannel {
  float* state;  // &conv_state[b, s, c, 0]
  float win[3];  // previous Kc-1 inputs
  float tap[4];
};

__device__ __forceinline__ void conv_fetch(const PrepArgs& p, int b, int s, int c, ConvChannel& ch) {
  const int CS = p.CQ;  // channels per stream (K * nh == V * nh)
  ch.state = p.conv_state + (((size_t)b * 3 + s) * CS + c) * (p.Kc - 1);
  const unsigned short* w = reinterpret_cast<const unsigned short*>(p.conv_w) + (size_t)s * p.Kc * CS + c;
  ch.win[0] = ch.state[0];
  ch.win[1] = p.Kc > 2 ? ch.state[1] : 0.f;
  ch.win[2] = p.Kc > 3 ? ch.state[2] : 0.f;
  ch.tap[0] = __uint_as_float((uint32_t)w[0] << 16);
  ch.tap[1] = __uint_as_float((uint32_t)w[(size_t)CS] << 16);
  ch.tap[2] = p.Kc > 2 ? __uint_as_float((uint32_t)w[(size_t)2 * CS] << 16) : 0.f;
  ch.tap[3] = p.Kc > 3 ? __uint_as_float((uint32_t)w[(size_t)3 * CS] << 16) : 0.f;
}

// y = SiLU(sum_j tap[j] * window[j]) for the window ending at x_new, then
// slide the window (in registers) to end at x_new.  Kc is 2, 3 or 4.
__device__ __forceinline__ float conv_step(const PrepArgs& p, ConvChannel& ch, float x_new) {
  float y;
  if (p.Kc == 4) {
    y = fmaf(ch.tap[0], ch.win[0], fmaf(ch.tap[1], ch.win[1], fmaf(ch.tap[2], ch.win[2], ch.tap[3] * x_new)));
    ch.win[0] = ch.win[1];
    ch.win[1] = ch.win[2];
    ch.win[2] = x_new;
  } else if (p.Kc == 3) {
    y = fmaf(ch.tap[0], ch.win[0], fmaf(ch.tap[1], ch.win[1], ch.tap[2] * x_new));
    ch.win[0] = ch.win[1];
    ch.win[1] = x_new;
  } else {
    y = fmaf(ch.tap[0], ch.win[0], ch.tap[1] * x_new);
    ch.win[0] = x_new;
  }
  return y * sigmoidf_(y);
}

// conv_state keeps the last Kc-1 pre-convolution inputs.
__device__ __forceinline__ void conv_save(const PrepArgs& p, const ConvChannel& ch) {
  ch.state[0] = ch.win[0];
  if (p.Kc > 2) ch.state[1] = ch.win[1];
  if (p.Kc > 3) ch.state[2] = ch.win[2];
}

constexpr int kPrepHeads = 8;
constexpr int kPrepThreads = kPrepHeads * kHeadDim;  // 1024

// 4. per (request b, group of 8 heads), the request's n tokens in order.
// q/k channels are channel-outer (d * nh + h): thread t takes channel
// (t / 8) * nh + h0 + t % 8, so a warp reads 4 runs of 8 consecutive
// channels.  v channels and everything per (head, d) use hl = t / 128,
// d = t % 128 (v is head-outer, so contiguous).  Each channel's conv window
// slides across the tokens in registers and is written back once.  The work
// that does not need the gate latents (loads, convolutions, norms, most of
// the token record) runs before the wait for the latent kernel; the forget
// gate and the output gate after it.
__global__ void __launch_bounds__(kPrepThreads, 1) block_prep_kernel(const PrepArgs p) {
  __shared__ float qs_[kPrepHeads][kHeadDim];
  __shared__ float ks_[kPrepHeads][kHeadDim];
  __shared__ float red[3][kPrepThreads / 32];
  const int h0 = blockIdx.x * kPrepHeads;
  const int b = blockIdx.y;
  const int t = threadIdx.x;
  const int dq = t / kPrepHeads, hq = t % kPrepHeads;
  const int cq = dq * p.nh + h0 + hq;
  const int hl = t / kHeadDim, d = t % kHeadDim;
  const int h = h0 + hl;
  const int cv = h * kHeadDim + d;
  const size_t pstride = (size_t)p.R * p.I;

  const int w = t >> 5;
  const int w0 = hl * (kHeadDim / 32);  // the 4 warps of head hl

  // Before waiting for the latent kernel: everything that does not need its
  // gate latents.  The projection partial sums and the tail come from the
  // W_in GEMM, which completed before the latent kernel (launched in plain
  // stream order) began, and so before this kernel's CTAs were launched.
  ConvChannel chq, chk, chv;
  conv_fetch(p, b, 0, cq, chq);
  conv_fetch(p, b, 1, cq, chk);
  conv_fetch(p, b, 2, cv, chv);
  const float dtb = p.dt_bias[(size_t)d * p.nh + h];
  const float aexp = expf(p.A_log[h]);
  const float gam = p.gamma_o[d];

#pragma unroll 1
  for (int j = 0; j < p.n; ++j) {
    const int r = b * p.n + j;
    const float* prow = p.Ppart + (size_t)r * p.I;
    // Every load of the token is issued before any is used (one round trip).
    float pq[kKS1], pk[kKS1], pv[kKS1];
#pragma unroll
    for (int ks = 0; ks < kKS1; ++ks) {
      const float* pr = prow + ks * pstride;
      const bool on = ks < p.KS1;
      pq[ks] = on ? pr[cq] : 0.f;
      pk[ks] = on ? pr[p.CQ + cq] : 0.f;
      pv[ks] = on ? pr[2 * p.CQ + cv] : 0.f;
    }
    const float bl = p.tail[(size_t)r * p.TN + kHeadDim + h];
    float xq = pq[0], xk = pk[0], xv = pv[0];
#pragma unroll
    for (int ks = 1; ks < kKS1; ++ks) {
      xq += pq[ks];
      xk += pk[ks];
      xv += pv[ks];
    }

    if (j > 0) __syncthreads();  // the previous token's qs_, ks_ and red are consumed
    qs_[hq][dq] = conv_step(p, chq, xq);
    ks_[hq][dq] = conv_step(p, chk, xk);
    const float yv = conv_step(p, chv, xv);
    __syncthreads();
    const float qv = qs_[hl][d], kv = ks_[hl][d];
    const float qq = warp_sum(qv * qv), kk = warp_sum(kv * kv), qk = warp_sum(qv * kv);
    if ((t & 31) == 0) {
      red[0][w] = qq;
      red[1][w] = kk;
      red[2][w] = qk;
    }
    __syncthreads();
    float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
    for (int i = 0; i < kHeadDim / 32; ++i) {
      sq += red[0][w0 + i];
      sk += red[1][w0 + i];
      sqk += red[2][w0 + i];
    }
    const float qsc = p.scale * rsqrtf(sq + p.l2_eps);
    const float ksc = rsqrtf(sk + p.l2_eps);
    const float beta = sigmoidf_(bl);
    if (!kda_in_bounds(r < p.R && h < p.nh && cq < p.CQ && cv < p.CV, p.status)) continue;
    TokenStage& st = p.stage[(size_t)r * p.nh + h];
    const float kh = kv * ksc;
    st.row[d].kh = kh;
    st.row[d].qh = qv * qsc;
    st.row[d].bkh = beta * kh;
    st.v[d] = yv;
    if (d == 0) st.bqk = beta * sqk * qsc * ksc;
  }
  // The gates need the latent kernel's output.
  pdl_wait();
  pdl_trigger();
#pragma unroll 1
  for (int j = 0; j < p.n; ++j) {
    const int r = b * p.n + j;
    if (!kda_in_bounds(r < p.R && h < p.nh, p.status)) continue;
    const size_t gzrow = (size_t)r * (p.CQ + p.CV);
    const float graw = p.gz[gzrow + (size_t)h * kHeadDim + d];   // W_fb head-outer
    const float zz = p.gz[gzrow + p.CQ + (size_t)d * p.nh + h];  // W_gb channel-outer
    p.stage[(size_t)r * p.nh + h].row[d].decay =
        expf(p.lower_bound * sigmoidf_(aexp * (graw + dtb)));
    p.zgate[((size_t)r * p.nh + h) * kHeadDim + d] = gam * output_gate(zz);
  }
  conv_save(p, chq);
  conv_save(p, chk);
  conv_save(p, chv);
}

struct RecArgs {
  const TokenStage* stage;
  const float* zgate;
  float* S;
  __nv_bfloat16* on2;  // [2R, CV] bf16 hi rows then lo rows
  int32_t* status;     // device status word (debug builds' index checks)
  float rms_norm_eps;
  int R, n, nh, CV;
};

// 5. one CTA per (request b, head h): the state tile is fetched once and held
// in registers across the request's n tokens; per token the staged vectors
// are read, one delta-rule step is taken and the gated output RMSNorm is
// written as bf16 hi/lo for the output projection.
// kMulti: the n > 1 form (the token loop); both forms fit two CTAs per SM.
template <bool kMulti>
__global__ void __launch_bounds__(kThreads, 2) block_recurrence_kernel(const RecArgs p) {
  // Two record buffers: token j + 1's record and output gate are fetched while
  // token j is stepped.
  __shared__ TokenStage ts[2];
  __shared__ __align__(16) float zg[2][kHeadDim];
  __shared__ __align__(16) float o_s[kHeadDim];
  __shared__ float red[kThreads / 32];
  const int bh = blockIdx.x;
  const int b = bh / p.nh, h = bh - b * p.nh;
  const int tid = threadIdx.x;
  const TileLane tl = tile_lane();
  // debug builds: the CTA's request and head lie in the block's rows
  if (!kda_in_bounds(b * (kMulti ? p.n : 1) < p.R && h < p.nh, p.status)) return;

  float* tile = p.S + (size_t)bh * (size_t)(kHeadDim * kHeadDim);
  float4 s[16];
  tile_load(s, tile, tl);  // S is not written by the preceding kernels
  pdl_wait();
  pdl_trigger();
  // A token's record and gate as 16-byte vectors, one per thread.
  constexpr int kStageVec = (int)(sizeof(TokenStage) / sizeof(uint4));
  constexpr int kRecVec = kStageVec + kHeadDim / 4;
  static_assert(kRecVec <= kThreads, "one vector per thread");
  auto fetch = [&](size_t r) -> uint4 {
    if (tid < kStageVec) return reinterpret_cast<const uint4*>(p.stage + r * p.nh + h)[tid];
    if (tid < kRecVec)
      return reinterpret_cast<const uint4*>(p.zgate + (r * p.nh + h) * kHeadDim)[tid - kStageVec];
    return make_uint4(0u, 0u, 0u, 0u);
  };
  auto put = [&](int buf, uint4 v) {
    if (tid < kStageVec)
      reinterpret_cast<uint4*>(&ts[buf])[tid] = v;
    else if (tid < kRecVec)
      reinterpret_cast<uint4*>(zg[buf])[tid - kStageVec] = v;
  };
  const int n = kMulti ? p.n : 1;
  put(0, fetch((size_t)b * n));
#pragma unroll 1
  for (int j = 0; j < n; ++j) {
    const size_t r = (size_t)b * n + j;
    const int buf = j & 1;
    const bool more = kMulti && j + 1 < n;
    const uint4 next = more ? fetch(r + 1) : make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();  // record j is in place; token j - 1's o_s is consumed
    const float4 o = tile_token_step(s, ts[buf], tl);
    if (tl.rg == 0) *reinterpret_cast<float4*>(&o_s[tl.col]) = o;
    __syncthreads();
    const float od = tid < kHeadDim ? o_s[tid] : 0.f;
    const float m2 = block_sum(od * od, red);
    if (tid < kHeadDim) {
      const float inv = rsqrtf(m2 / (float)kHeadDim + p.rms_norm_eps);
      const size_t col = (size_t)h * kHeadDim + tid;  // W_o rows are head-outer
      split_bf16(od * inv * zg[buf][tid], p.on2 + r * p.CV + col,
                 p.on2 + ((size_t)p.R + r) * p.CV + col);
    }
    // The other buffer was last read by token j - 1, before this token's barriers.
    if (more) put(buf ^ 1, next);
  }
  tile_store(tile, s, tl);
}

}  // namespace

size_t block_workspace_bytes(int B, int n, int Hd, int nh, int K, int V, int Kc) {
  Layout L;
  if (!make_layout(B, n, Hd, nh, K, V, Kc, &L)) return 0;
  return L.total;
}

cudaError_t launch_kda_block(const BlockArgs& a, cudaStream_t stream) {
  Layout L;
  if (!make_layout(a.B, a.n, a.Hd, a.nh, a.K, a.V, a.Kc, &L)) return cudaErrorInvalidValue;
  char* ws = static_cast<char*>(a.workspace);
  __nv_bfloat16* x2 = reinterpret_cast<__nv_bfloat16*>(ws + L.x2);
  float* ppart = reinterpret_cast<float*>(ws + L.ppart);
  float* tail = reinterpret_cast<float*>(ws + L.tail);
  float* gz = reinterpret_cast<float*>(ws + L.gz);
  __nv_bfloat16* on2 = reinterpret_cast<__nv_bfloat16*>(ws + L.on2);
  int32_t* err = a.dev_status ? a.dev_status : reinterpret_cast<int32_t*>(ws + L.err);
  cudaError_t e;

  // The first kernel waits for everything before it in the stream; each later
  // kernel is a programmatic dependent of the one before it.
  e = launch(rmsnorm_split_kernel, dim3(L.R), dim3(kNormThreads), 0, stream, false, a.hidden,
             a.gamma_in, x2, a.out, tail, L.TN, L.R, a.Hd, a.rms_norm_eps);
  if (e != cudaSuccess) return e;
  // g_a, beta and f_a (the last TN columns) are summed over the splits in
  // place (into `tail`, zeroed by the RMSNorm kernel): every latent CTA reads
  // the f_a / g_a panel, so it is kept at one copy.
  // As their MMAs finish, the W_in CTAs bring into L2 what the next two
  // kernels read first: conv_state (prep) and the gate latent weights.
  const L2Prefetch pf{{a.conv_state, a.W_fb, a.W_gb},
                      {(size_t)a.B * 3 * L.CQ * (a.Kc - 1) * sizeof(float),
                       (size_t)a.K * L.CQ * sizeof(kda_bf16), (size_t)a.K * L.CV * sizeof(kda_bf16)}};
  e = launch_tc_gemm(reinterpret_cast<const kda_bf16*>(x2), L.R, a.Hd, a.W_in, L.I, L.KS1, ppart,
                     false, err, stream, true, tail, L.TC, &pf, /*x_parts=*/3);
  if (e != cudaSuccess) return e;
  // Within the tail: g_a at 0, beta at K, f_a at K + nh.
  const int off_ga = 0;
  const int off_fa = kHeadDim + a.nh;
  // Not a programmatic dependent: launched early, its CTAs would be packed
  // onto the first SMs the projection GEMM frees (several per SM, the other
  // SMs idle); launched after the GEMM they spread over every SM.
  e = launch(latent_kernel, dim3((L.CQ + L.CV) / kLatTile, (L.R + kLatTile - 1) / kLatTile),
             dim3(256), 0, stream, false, (const float*)tail, 1, L.R, L.TN, off_fa, off_ga,
             a.W_fb, L.CQ, a.W_gb, L.CV, gz);
  if (e != cudaSuccess) return e;
  TokenStage* stage = reinterpret_cast<TokenStage*>(ws + L.stage);
  float* zgate = reinterpret_cast<float*>(ws + L.zgate);
  PrepArgs pa;
  pa.Ppart = ppart;
  pa.tail = tail;
  pa.TN = L.TN;
  pa.gz = gz;
  pa.conv_w = a.conv_w;
  pa.conv_state = a.conv_state;
  pa.A_log = a.A_log;
  pa.dt_bias = a.dt_bias;
  pa.gamma_o = a.gamma_o;
  pa.stage = stage;
  pa.zgate = zgate;
  pa.status = err;
  pa.scale = a.scale;
  pa.lower_bound = a.lower_bound;
  pa.l2_eps = a.l2_eps;
  pa.R = L.R;
  pa.n = a.n;
  pa.I = L.I;
  pa.KS1 = L.KS1;
  pa.nh = a.nh;
  pa.Kc = a.Kc;
  pa.CQ = L.CQ;
  pa.CV = L.CV;
  e = launch(block_prep_kernel, dim3(a.nh / kPrepHeads, a.B), dim3(kPrepThreads), 0, stream, true,
             pa);
  if (e != cudaSuccess) return e;
  RecArgs ra;
  ra.stage = stage;
  ra.zgate = zgate;
  ra.S = a.S;
  ra.on2 = on2;
  ra.status = err;
  ra.rms_norm_eps = a.rms_norm_eps;
  ra.R = L.R;
  ra.n = a.n;
  ra.nh = a.nh;
  ra.CV = L.CV;
  e = launch(a.n > 1 ? block_recurrence_kernel<true> : block_recurrence_kernel<false>,
             dim3(a.B * a.nh), dim3(kThreads), 0, stream, true, ra);
  if (e != cudaSuccess) return e;
  // The output projection adds its contraction splits straight into `out`
  // (zeroed by the RMSNorm kernel).
  return launch_tc_gemm(reinterpret_cast<const kda_bf16*>(on2), L.R, L.CV, a.W_o, a.Hd, L.KS2,
                        a.out, true, err, stream, true);
}

}  // namespace kda
