// kda_block.cu -- the fused KDA block for token generation (n = 1).
//
// Operation: "KDA Block TKG Kernel API Reference" (Background; :param hidden:,
// gamma_in, W_in, W_fb, W_gb, conv_w, A_log, dt_bias, gamma_o, W_o, out, S,
// conv_state, scale, rms_norm_eps, lower_bound), the recurrence of "Delta-rule
// write".
//
// Kernel chain on the caller's stream (rows r = b, R = B):
//   1. rmsnorm      x = hidden * rsqrt(mean(hidden^2) + eps) * gamma_in, written
//                   as bf16 hi/lo halves X2 [2R, Hd] for the tensor cores
//   2. proj GEMM    tcgen05, P_part[ks] = x[:, split ks] . W_in[split ks, :]   [KS1, R, I]
//                   (split-K so every SM streams a slice of the 103 MB W_in;
//                   consumers add the KS1 partial sums)
//   3. latent       graw = f_a . W_fb, z = g_a . W_gb (CUDA cores)            [R, CQ + CV]
//   4. head         one CTA per (b, h): short conv + SiLU + conv_state update
//                   for the head's q, k, v channels, forget gate, beta, L2
//                   norms, the register-tile delta-rule step on S[b, h] (shared
//                   with kda_decode), gated output RMSNorm -> bf16 hi/lo on2
//   5. out GEMM     tcgen05, O_part[ks] = on[:, split ks] . W_o[split ks, :]   [KS2, R, Hd]
//   6. reduce       out = sum_ks O_part[ks]
// Intermediates live in the caller's workspace (a few MB: L2-resident).
#include "kda_recurrence.cuh"
#include "kda_tc_gemm.h"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kLatCols = 64;   // latent GEMM: output columns per CTA
constexpr int kLatRows = 32;   // latent GEMM: rows per CTA
constexpr int kKS1 = 4;        // contraction splits of the W_in GEMM
constexpr int kKS2 = 8;        // contraction splits of the W_o GEMM

struct Layout {
  int R, I, CQ, CV, KS1, KS2;
  size_t x2, ppart, gz, on2, opart, err, total;
};

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

bool make_layout(int B, int n, int Hd, int nh, int K, int V, int Kc, Layout* L) {
  if (B < 1 || n != 1 || K != kHeadDim || V != kHeadDim || Kc < 2 || Kc > 4 || Hd < 128 ||
      Hd % 128 != 0 || nh < 8 || nh % 8 != 0)
    return false;
  L->R = B * n;
  L->CQ = K * nh;
  L->CV = V * nh;
  L->I = 2 * L->CQ + L->CV + 2 * K + nh;
  L->KS1 = Hd / 64 < kKS1 ? Hd / 64 : kKS1;        // splits <= 64-row contraction blocks
  L->KS2 = L->CV / 64 < kKS2 ? L->CV / 64 : kKS2;
  size_t off = 0;
  L->x2 = off;    off = align_up(off + 2 * sizeof(kda_bf16) * (size_t)L->R * Hd);
  L->ppart = off; off = align_up(off + sizeof(float) * (size_t)L->KS1 * L->R * L->I);
  L->gz = off;    off = align_up(off + sizeof(float) * (size_t)L->R * (L->CQ + L->CV));
  L->on2 = off;   off = align_up(off + 2 * sizeof(kda_bf16) * (size_t)L->R * L->CV);
  L->opart = off; off = align_up(off + sizeof(float) * (size_t)L->KS2 * L->R * Hd);
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

// 1. input RMSNorm, one CTA per row, written as bf16 hi/lo halves.
__global__ void __launch_bounds__(kThreads) rmsnorm_split_kernel(const float* __restrict__ hidden,
                                                                 const float* __restrict__ gamma,
                                                                 __nv_bfloat16* __restrict__ X2,
                                                                 int R, int Hd, float eps) {
  __shared__ float red[kThreads / 32];
  const float* x = hidden + (size_t)blockIdx.x * Hd;
  float ss = 0.f;
  for (int i = threadIdx.x * 4; i < Hd; i += kThreads * 4) {
    const float4 v = *reinterpret_cast<const float4*>(x + i);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (float)Hd + eps);
  __nv_bfloat16* hi = X2 + (size_t)blockIdx.x * Hd;
  __nv_bfloat16* lo = X2 + ((size_t)R + blockIdx.x) * Hd;
  for (int i = threadIdx.x; i < Hd; i += kThreads) split_bf16(x[i] * inv * gamma[i], hi + i, lo + i);
}

// 3. gate latents on the CUDA cores: gz[r][c] = f_a[r] . W_fb[:, c] for
// c < CQ and g_a[r] . W_gb[:, c - CQ] after, with f_a and g_a summed from the
// projection's split-K partials.  Grid ((CQ + CV) / 64, ceil(R / 32)), 128
// threads: thread t owns columns 2 (t % 32) .. + 1 and rows 8 (t / 32) .. + 7.
__global__ void __launch_bounds__(128) latent_kernel(
    const float* __restrict__ Ppart, int KS1, int R, int I, int off_fa, int off_ga,
    const kda_bf16* __restrict__ W_fb, int CQ, const kda_bf16* __restrict__ W_gb, int CV,
    float* __restrict__ gz) {
  __shared__ __align__(16) float xs[kLatRows][kHeadDim];
  const int c0 = blockIdx.x * kLatCols;
  const bool is_fb = c0 < CQ;  // CQ is a multiple of 64
  const kda_bf16* W = is_fb ? W_fb : W_gb;
  const int N = is_fb ? CQ : CV;
  const int cl = (is_fb ? c0 : c0 - CQ) + 2 * (threadIdx.x & 31);
  const int off = is_fb ? off_fa : off_ga;
  const int r0 = blockIdx.y * kLatRows;
  const int rg = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < kLatRows * kHeadDim; e += 128) {
    const int r = e / kHeadDim, i = e % kHeadDim;
    float v = 0.f;
    if (r0 + r < R)
      for (int ks = 0; ks < KS1; ++ks) v += Ppart[((size_t)ks * R + r0 + r) * I + off + i];
    xs[r][i] = v;
  }
  __syncthreads();
  float acc[8][2];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = 0.f;
  const kda_bf16* wp = W + cl;
#pragma unroll 4
  for (int k = 0; k < kHeadDim; ++k) {
    const uint32_t w2 = __ldg(reinterpret_cast<const unsigned int*>(wp + (size_t)k * N));
    const float w0 = bf16_lo(w2), w1 = bf16_hi(w2);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float xv = xs[rg * 8 + j][k];
      acc[j][0] = fmaf(xv, w0, acc[j][0]);
      acc[j][1] = fmaf(xv, w1, acc[j][1]);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = r0 + rg * 8 + j;
    if (r < R)
      *reinterpret_cast<float2*>(gz + (size_t)r * (CQ + CV) + c0 + 2 * (threadIdx.x & 31)) =
          make_float2(acc[j][0], acc[j][1]);
  }
}

struct HeadArgs {
  const float* Ppart;
  const float* gz;
  const kda_bf16* conv_w;
  float* conv_state;
  const float* A_log;
  const float* dt_bias;
  const float* gamma_o;
  float* S;
  __nv_bfloat16* on2;  // [2R, CV] bf16 hi rows then lo rows
  float scale, lower_bound, rms_norm_eps, l2_eps;
  int R, I, KS1, nh, Kc, CQ, CV;
};

__device__ __forceinline__ float sum_partials(const float* Ppart, int KS1, size_t stride,
                                              size_t idx) {
  float v = 0.f;
  for (int ks = 0; ks < KS1; ++ks) v += Ppart[ks * stride + idx];
  return v;
}

// Causal depthwise conv over [conv_state (oldest first), x_new] with taps
// conv_w[s, 0..Kc-1, c] (tap 0 oldest), SiLU, and the window shift.
__device__ __forceinline__ float conv_silu_shift(const HeadArgs& p, int b, int s, int c,
                                                 float x_new) {
  const int CS = p.CQ;  // channels per stream (K * nh == V * nh)
  float* cs = p.conv_state + (((size_t)b * 3 + s) * CS + c) * (p.Kc - 1);
  float win[4];
  for (int j = 0; j < p.Kc - 1; ++j) win[j] = cs[j];
  win[p.Kc - 1] = x_new;
  float y = 0.f;
  for (int j = 0; j < p.Kc; ++j) {
    const unsigned short wb = reinterpret_cast<const unsigned short*>(p.conv_w)[((size_t)s * p.Kc + j) * CS + c];
    y = fmaf(__uint_as_float((uint32_t)wb << 16), win[j], y);
  }
  for (int j = 0; j < p.Kc - 1; ++j) cs[j] = win[j + 1];
  return y * sigmoidf_(y);
}

// 4. one CTA per (request b, head h).
__global__ void __launch_bounds__(kThreads, 2) block_head_kernel(const HeadArgs p) {
  __shared__ TokenStage ts;
  __shared__ float qk_s[2][kHeadDim];
  __shared__ float o_s[kHeadDim];
  __shared__ float red[kThreads / 32];

  const int h = blockIdx.x % p.nh;
  const int b = blockIdx.x / p.nh;
  const int r = b;  // n == 1
  const int tid = threadIdx.x;
  const TileLane tl = tile_lane();

  float* tile = p.S + ((size_t)b * p.nh + h) * (size_t)(kHeadDim * kHeadDim);
  float4 s[16];
  tile_load(s, tile, tl);

  const size_t pstride = (size_t)p.R * p.I;
  const float* prow = p.Ppart + (size_t)r * p.I;
  // q (threads 0..127) and k (128..255): channel-outer d * nh + h
  {
    const int sidx = tid >> 7, d = tid & 127;
    const int c = d * p.nh + h;
    const float x = sum_partials(prow, p.KS1, pstride, (size_t)sidx * p.CQ + c);
    qk_s[sidx][d] = conv_silu_shift(p, b, sidx, c, x);
  }
  float vval = 0.f;
  if (tid < kHeadDim) {  // v: head-outer h * V + d
    const int c = h * kHeadDim + tid;
    const float x = sum_partials(prow, p.KS1, pstride, (size_t)2 * p.CQ + c);
    vval = conv_silu_shift(p, b, 2, c, x);
  }
  const float beta = sigmoidf_(sum_partials(prow, p.KS1, pstride, (size_t)2 * p.CQ + p.CV + kHeadDim + h));
  __syncthreads();
  float qq = 0.f, kk = 0.f, qk = 0.f;
  if (tid < kHeadDim) {
    const float qv = qk_s[0][tid], kv = qk_s[1][tid];
    qq = qv * qv;
    kk = kv * kv;
    qk = qv * kv;
  }
  qq = block_sum(qq, red);
  kk = block_sum(kk, red);
  qk = block_sum(qk, red);
  const float qs = p.scale * rsqrtf(qq + p.l2_eps);
  const float ksc = rsqrtf(kk + p.l2_eps);
  if (tid < kHeadDim) {
    const int d = tid;
    const float graw = p.gz[(size_t)r * (p.CQ + p.CV) + h * kHeadDim + d];  // W_fb head-outer
    const float g = p.lower_bound * sigmoidf_(expf(p.A_log[h]) * (graw + p.dt_bias[(size_t)d * p.nh + h]));
    RowCoef rc;
    rc.decay = expf(g);
    rc.kh = qk_s[1][d] * ksc;
    rc.qh = qk_s[0][d] * qs;
    rc.bkh = beta * rc.kh;
    ts.row[d] = rc;
    ts.v[d] = vval;
    if (d == 0) ts.bqk = beta * qk * qs * ksc;
  }
  __syncthreads();
  const float4 o = tile_token_step(s, ts, tl);
  if (tl.rg == 0) *reinterpret_cast<float4*>(&o_s[tl.col]) = o;
  tile_store(tile, s, tl);
  __syncthreads();
  const float od = tid < kHeadDim ? o_s[tid] : 0.f;
  const float m2 = block_sum(od * od, red);
  if (tid < kHeadDim) {
    const int d = tid;
    const float inv = rsqrtf(m2 / (float)kHeadDim + p.rms_norm_eps);
    const float z = p.gz[(size_t)r * (p.CQ + p.CV) + p.CQ + d * p.nh + h];  // W_gb channel-outer
    const size_t col = (size_t)h * kHeadDim + d;  // W_o rows are head-outer
    split_bf16(od * inv * p.gamma_o[d] * sigmoidf_(z), p.on2 + (size_t)r * p.CV + col,
               p.on2 + ((size_t)p.R + r) * p.CV + col);
  }
}

// 6. out = sum of the split-K partials (float4 granularity).
__global__ void reduce_partials_kernel(const float* __restrict__ part, int KS, size_t count4,
                                       float* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count4;
       i += (size_t)gridDim.x * blockDim.x) {
    float4 acc = reinterpret_cast<const float4*>(part)[i];
    for (int ks = 1; ks < KS; ++ks) {
      const float4 v = reinterpret_cast<const float4*>(part)[(size_t)ks * count4 + i];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    reinterpret_cast<float4*>(out)[i] = acc;
  }
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
  float* gz = reinterpret_cast<float*>(ws + L.gz);
  __nv_bfloat16* on2 = reinterpret_cast<__nv_bfloat16*>(ws + L.on2);
  float* opart = reinterpret_cast<float*>(ws + L.opart);
  int32_t* err = a.dev_status ? a.dev_status : reinterpret_cast<int32_t*>(ws + L.err);
  cudaError_t e;

  rmsnorm_split_kernel<<<L.R, kThreads, 0, stream>>>(a.hidden, a.gamma_in, x2, L.R, a.Hd,
                                                      a.rms_norm_eps);
  e = launch_tc_gemm(reinterpret_cast<const kda_bf16*>(x2), L.R, a.Hd, a.W_in, L.I, L.KS1, ppart,
                     err, stream);
  if (e != cudaSuccess) return e;
  const int off_ga = 2 * L.CQ + L.CV;
  const int off_fa = off_ga + kHeadDim + a.nh;
  latent_kernel<<<dim3((L.CQ + L.CV) / kLatCols, (L.R + kLatRows - 1) / kLatRows), 128, 0, stream>>>(
      ppart, L.KS1, L.R, L.I, off_fa, off_ga, a.W_fb, L.CQ, a.W_gb, L.CV, gz);
  HeadArgs h;
  h.Ppart = ppart;
  h.gz = gz;
  h.conv_w = a.conv_w;
  h.conv_state = a.conv_state;
  h.A_log = a.A_log;
  h.dt_bias = a.dt_bias;
  h.gamma_o = a.gamma_o;
  h.S = a.S;
  h.on2 = on2;
  h.scale = a.scale;
  h.lower_bound = a.lower_bound;
  h.rms_norm_eps = a.rms_norm_eps;
  h.l2_eps = a.l2_eps;
  h.R = L.R;
  h.I = L.I;
  h.KS1 = L.KS1;
  h.nh = a.nh;
  h.Kc = a.Kc;
  h.CQ = L.CQ;
  h.CV = L.CV;
  block_head_kernel<<<L.R * a.nh, kThreads, 0, stream>>>(h);
  e = launch_tc_gemm(reinterpret_cast<const kda_bf16*>(on2), L.R, L.CV, a.W_o, a.Hd, L.KS2, opart,
                     err, stream);
  if (e != cudaSuccess) return e;
  const size_t count4 = (size_t)L.R * a.Hd / 4;
  const int rblk = (int)((count4 + kThreads - 1) / kThreads);
  reduce_partials_kernel<<<rblk, kThreads, 0, stream>>>(opart, L.KS2, count4, a.out);
  return cudaGetLastError();
}

}  // namespace kda
