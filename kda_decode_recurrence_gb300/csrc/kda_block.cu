// kda_block.cu -- the fused KDA block for token generation (n = 1).
//
// Operation: "KDA Block TKG Kernel API Reference" (Background; :param hidden:,
// gamma_in, W_in, W_fb, W_gb, conv_w, A_log, dt_bias, gamma_o, W_o, out, S,
// conv_state, scale, rms_norm_eps, lower_bound), the recurrence of "Delta-rule
// write".
//
// Kernel chain on the caller's stream (rows r = b, R = B):
//   1. rmsnorm      x = hidden * rsqrt(mean(hidden^2) + eps) * gamma_in      [R, Hd]
//   2. proj GEMM    P_part[ks] = x[:, chunk ks] . W_in[chunk ks, :]         [KS1, R, I]
//                   (split-K over the hidden dimension so every SM streams a
//                   slice of W_in; the partial sums are added by consumers)
//   3. latent GEMM  graw = f_a . W_fb, z = g_a . W_gb                        [R, CQ + CV]
//   4. head         one CTA per (b, h): short conv + SiLU + conv_state update
//                   for the head's q, k, v channels, forget gate, beta, L2
//                   norms, the register-tile delta-rule step on S[b, h] (shared
//                   with kda_decode), gated output RMSNorm -> on [R, nh*V]
//   5. out GEMM     O_part[ks] = on[:, chunk ks] . W_o[chunk ks, :]          [KS2, R, Hd]
//   6. reduce       out = sum_ks O_part[ks]
// Intermediates live in the caller's workspace (a few tens of MB: they stay
// L2-resident on GB300).  The GEMMs accumulate in fp32 from fp32 activations
// and exact bf16 weights on the CUDA cores.
#include "kda_recurrence.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kGemmCols = 2 * kThreads;  // output columns per GEMM CTA (2 per thread)
constexpr int kGemmRows = 32;            // rows (requests) per GEMM CTA
constexpr int kGemmKSub = 16;            // contraction rows staged per sub-step

struct Layout {
  int R, I, CQ, CV, KS1, KS2, kchunk1, kchunk2;
  size_t xhat, ppart, gz, on, opart, total;
};

int largest_divisor_at_most(int n, int cap) {
  for (int d = cap; d > 1; --d)
    if (n % d == 0) return d;
  return 1;
}

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

bool make_layout(int B, int n, int Hd, int nh, int K, int V, int Kc, Layout* L) {
  if (B < 1 || n != 1 || K != kHeadDim || V != kHeadDim || Kc < 2 || Kc > 4 || Hd < 128 ||
      Hd % 128 != 0 || nh < 8 || nh % 8 != 0)
    return false;
  L->R = B * n;
  L->CQ = K * nh;
  L->CV = V * nh;
  L->I = 2 * L->CQ + L->CV + 2 * K + nh;
  L->KS1 = largest_divisor_at_most(Hd / 128, 16);
  L->kchunk1 = Hd / L->KS1;
  L->KS2 = largest_divisor_at_most(L->CV / 128, 32);
  L->kchunk2 = L->CV / L->KS2;
  size_t off = 0;
  L->xhat = off;  off = align_up(off + sizeof(float) * (size_t)L->R * Hd);
  L->ppart = off; off = align_up(off + sizeof(float) * (size_t)L->KS1 * L->R * L->I);
  L->gz = off;    off = align_up(off + sizeof(float) * (size_t)L->R * (L->CQ + L->CV));
  L->on = off;    off = align_up(off + sizeof(float) * (size_t)L->R * L->CV);
  L->opart = off; off = align_up(off + sizeof(float) * (size_t)L->KS2 * L->R * Hd);
  L->total = off;
  return true;
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

// 1. input RMSNorm, one CTA per row.
__global__ void __launch_bounds__(kThreads) rmsnorm_kernel(const float* __restrict__ hidden,
                                                           const float* __restrict__ gamma,
                                                           float* __restrict__ xhat, int Hd,
                                                           float eps) {
  __shared__ float red[kThreads / 32];
  const float* x = hidden + (size_t)blockIdx.x * Hd;
  float ss = 0.f;
  for (int i = threadIdx.x * 4; i < Hd; i += kThreads * 4) {
    const float4 v = *reinterpret_cast<const float4*>(x + i);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (float)Hd + eps);
  float* y = xhat + (size_t)blockIdx.x * Hd;
  for (int i = threadIdx.x * 4; i < Hd; i += kThreads * 4) {
    const float4 v = *reinterpret_cast<const float4*>(x + i);
    const float4 g = *reinterpret_cast<const float4*>(gamma + i);
    *reinterpret_cast<float4*>(y + i) =
        make_float4(v.x * inv * g.x, v.y * inv * g.y, v.z * inv * g.z, v.w * inv * g.w);
  }
}

// Accumulate acc[r][0..1] += sum_{i < kGemmKSub} xs[r][i] * W[i][c .. c+1].
__device__ __forceinline__ void gemm_substep(float (&acc)[kGemmRows][2],
                                             const float (*xs)[kGemmKSub + 4],
                                             const kda_bf16* __restrict__ wp, int N) {
  uint32_t w[kGemmKSub];
#pragma unroll
  for (int i = 0; i < kGemmKSub; ++i) w[i] = __ldg(reinterpret_cast<const unsigned int*>(wp + (size_t)i * N));
#pragma unroll
  for (int i = 0; i < kGemmKSub; i += 4) {
#pragma unroll
    for (int r = 0; r < kGemmRows; ++r) {
      const float4 x = *reinterpret_cast<const float4*>(&xs[r][i]);
      acc[r][0] = fmaf(x.x, bf16_lo(w[i + 0]), acc[r][0]);
      acc[r][1] = fmaf(x.x, bf16_hi(w[i + 0]), acc[r][1]);
      acc[r][0] = fmaf(x.y, bf16_lo(w[i + 1]), acc[r][0]);
      acc[r][1] = fmaf(x.y, bf16_hi(w[i + 1]), acc[r][1]);
      acc[r][0] = fmaf(x.z, bf16_lo(w[i + 2]), acc[r][0]);
      acc[r][1] = fmaf(x.z, bf16_hi(w[i + 2]), acc[r][1]);
      acc[r][0] = fmaf(x.w, bf16_lo(w[i + 3]), acc[r][0]);
      acc[r][1] = fmaf(x.w, bf16_hi(w[i + 3]), acc[r][1]);
    }
  }
}

// 2./5. skinny split-K GEMM: Ypart[ks][r][c] = sum over the ks-th contraction
// chunk of X[r][i] * W[i][c].  X fp32 [R, ldx], W bf16 [*, N] (N even).
// Grid: (ceil(N / 512), KS, ceil(R / 32)).
__global__ void __launch_bounds__(kThreads, 2) skinny_gemm_kernel(
    const float* __restrict__ X, int R, int ldx, const kda_bf16* __restrict__ W, int N,
    int kchunk, float* __restrict__ Ypart) {
  __shared__ __align__(16) float xs[kGemmRows][kGemmKSub + 4];
  const int c = (blockIdx.x * kThreads + threadIdx.x) * 2;
  const int ks = blockIdx.y;
  const int r0 = blockIdx.z * kGemmRows;
  const int nrows = min(kGemmRows, R - r0);
  const int kbeg = ks * kchunk;
  float acc[kGemmRows][2];
#pragma unroll
  for (int r = 0; r < kGemmRows; ++r) acc[r][0] = acc[r][1] = 0.f;
  for (int kk = 0; kk < kchunk; kk += kGemmKSub) {
    __syncthreads();
    for (int e = threadIdx.x; e < kGemmRows * kGemmKSub; e += kThreads) {
      const int r = e / kGemmKSub, i = e % kGemmKSub;
      xs[r][i] = (r < nrows) ? X[(size_t)(r0 + r) * ldx + kbeg + kk + i] : 0.f;
    }
    __syncthreads();
    if (c < N) gemm_substep(acc, xs, W + (size_t)(kbeg + kk) * N + c, N);
  }
  if (c < N) {
#pragma unroll
    for (int r = 0; r < kGemmRows; ++r)
      if (r < nrows)
        *reinterpret_cast<float2*>(Ypart + ((size_t)ks * R + r0 + r) * N + c) =
            make_float2(acc[r][0], acc[r][1]);
  }
}

// 3. gate latents: gz[r][c] = f_a[r] . W_fb[:, c] for c < CQ and
// g_a[r] . W_gb[:, c - CQ] after, f_a and g_a summed from the projection's
// split-K partials.  Grid: ((CQ + CV) / 512, 1, ceil(R / 32)).
__global__ void __launch_bounds__(kThreads, 2) latent_gemm_kernel(
    const float* __restrict__ Ppart, int KS1, int R, int I, int off_fa, int off_ga,
    const kda_bf16* __restrict__ W_fb, int CQ, const kda_bf16* __restrict__ W_gb, int CV,
    float* __restrict__ gz) {
  __shared__ __align__(16) float xs[kGemmRows][kGemmKSub + 4];
  const int cglob = (blockIdx.x * kThreads + threadIdx.x) * 2;
  const bool is_fb = blockIdx.x * kGemmCols < CQ;  // CQ is a multiple of 512
  const kda_bf16* W = is_fb ? W_fb : W_gb;
  const int N = is_fb ? CQ : CV;
  const int c = is_fb ? cglob : cglob - CQ;
  const int off = is_fb ? off_fa : off_ga;
  const int r0 = blockIdx.z * kGemmRows;
  const int nrows = min(kGemmRows, R - r0);
  float acc[kGemmRows][2];
#pragma unroll
  for (int r = 0; r < kGemmRows; ++r) acc[r][0] = acc[r][1] = 0.f;
  for (int kk = 0; kk < kHeadDim; kk += kGemmKSub) {
    __syncthreads();
    for (int e = threadIdx.x; e < kGemmRows * kGemmKSub; e += kThreads) {
      const int r = e / kGemmKSub, i = e % kGemmKSub;
      float v = 0.f;
      if (r < nrows)
        for (int ks = 0; ks < KS1; ++ks) v += Ppart[((size_t)ks * R + r0 + r) * I + off + kk + i];
      xs[r][i] = v;
    }
    __syncthreads();
    if (c < N) gemm_substep(acc, xs, W + (size_t)kk * N + c, N);
  }
  if (c < N) {
#pragma unroll
    for (int r = 0; r < kGemmRows; ++r)
      if (r < nrows)
        *reinterpret_cast<float2*>(gz + (size_t)(r0 + r) * (CQ + CV) + cglob) =
            make_float2(acc[r][0], acc[r][1]);
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
  float* on;
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
    p.on[(size_t)r * p.CV + h * kHeadDim + d] = od * inv * p.gamma_o[d] * sigmoidf_(z);
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
  float* xhat = reinterpret_cast<float*>(ws + L.xhat);
  float* ppart = reinterpret_cast<float*>(ws + L.ppart);
  float* gz = reinterpret_cast<float*>(ws + L.gz);
  float* on = reinterpret_cast<float*>(ws + L.on);
  float* opart = reinterpret_cast<float*>(ws + L.opart);
  const int rblocks = (L.R + kGemmRows - 1) / kGemmRows;

  rmsnorm_kernel<<<L.R, kThreads, 0, stream>>>(a.hidden, a.gamma_in, xhat, a.Hd, a.rms_norm_eps);
  skinny_gemm_kernel<<<dim3((L.I + kGemmCols - 1) / kGemmCols, L.KS1, rblocks), kThreads, 0, stream>>>(
      xhat, L.R, a.Hd, a.W_in, L.I, L.kchunk1, ppart);
  const int off_ga = 2 * L.CQ + L.CV;
  const int off_fa = off_ga + kHeadDim + a.nh;
  latent_gemm_kernel<<<dim3((L.CQ + L.CV) / kGemmCols, 1, rblocks), kThreads, 0, stream>>>(
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
  h.on = on;
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
  skinny_gemm_kernel<<<dim3((a.Hd + kGemmCols - 1) / kGemmCols, L.KS2, rblocks), kThreads, 0, stream>>>(
      on, L.R, L.CV, a.W_o, a.Hd, L.kchunk2, opart);
  const size_t count4 = (size_t)L.R * a.Hd / 4;
  const int rblk = (int)((count4 + kThreads - 1) / kThreads);
  reduce_partials_kernel<<<rblk, kThreads, 0, stream>>>(opart, L.KS2, count4, a.out);
  return cudaGetLastError();
}

}  // namespace kda
