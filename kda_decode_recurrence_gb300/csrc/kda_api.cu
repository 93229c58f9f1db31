// kda_api.cu -- the extern "C" boundary of libkda: host-side argument
// validation, then kernel launches on the caller's stream.  No allocation.
#include <cmath>
#include <cstdint>

#include "kda.h"
#include "kda_internal.h"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" {

const char* kda_status_string(kda_status status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_NULL: return "a required pointer is NULL";
    case KDA_ERR_SHAPE: return "a size is out of range or sizes are inconsistent";
    case KDA_ERR_UNSUPPORTED: return "sizes not implemented by this build";
    case KDA_ERR_ENUM: return "unknown gate_mode, state_layout or output_dtype";
    case KDA_ERR_CUDA: return "a CUDA runtime call failed";
    case KDA_ERR_ALIGN: return "a pointer is not aligned as documented";
    case KDA_ERR_VALUE: return "a scalar argument is not finite or out of range";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char* kda_version(void) { return "kda-gb300 0.1"; }

}  // extern "C"

namespace {

kda_status decode_impl(void* output, const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                       const float* raw_gate, const float* beta_logits, const float* a_log,
                       const float* dt_bias, const int32_t* cu_seqlens, float* state_pool,
                       const int32_t* state_indices, int gate_mode, float lower_bound,
                       int state_layout, int output_dtype, int B, int T, int H, int HV, int K,
                       int V, int max_slots, int32_t* dev_status, void* stream,
                       bool prefill = false) {
  if (B < 0 || T < 0 || H < 1 || HV < 1 || K < 1 || V < 1 || max_slots < 1) return KDA_ERR_SHAPE;
  if (HV % H != 0) return KDA_ERR_SHAPE;
  if (gate_mode != KDA_GATE_SOFTPLUS && gate_mode != KDA_GATE_LOWER_BOUND) return KDA_ERR_ENUM;
  if (state_layout != KDA_STATE_K_FIRST && state_layout != KDA_STATE_V_FIRST) return KDA_ERR_ENUM;
  if (output_dtype != KDA_OUTPUT_F32 && output_dtype != KDA_OUTPUT_BF16) return KDA_ERR_ENUM;
  if (gate_mode == KDA_GATE_LOWER_BOUND && !(std::isfinite(lower_bound) && lower_bound <= 0.0f))
    return KDA_ERR_VALUE;
  if (K != kda::kHeadDim || V != kda::kHeadDim) return KDA_ERR_UNSUPPORTED;
  if ((long long)B * HV > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
  if (B == 0) return KDA_OK;
  if (!cu_seqlens || !state_pool || !state_indices || !a_log || !dt_bias) return KDA_ERR_NULL;
  if (T > 0 && (!output || !q || !k || !v || !raw_gate || !beta_logits)) return KDA_ERR_NULL;
  if (!aligned(state_pool, 16) || !aligned(dt_bias, 16) || !aligned(cu_seqlens, 4) ||
      !aligned(state_indices, 4) || !aligned(a_log, 4))
    return KDA_ERR_ALIGN;
  const uintptr_t out_align = output_dtype == KDA_OUTPUT_F32 ? 16 : 8;
  if (T > 0 && (!aligned(output, out_align) || !aligned(raw_gate, 16) || !aligned(q, 8) ||
                !aligned(k, 8) || !aligned(v, 8) || !aligned(beta_logits, 4)))
    return KDA_ERR_ALIGN;

  kda::DecodeArgs a;
  a.output = output;
  a.q = q;
  a.k = k;
  a.v = v;
  a.raw_gate = raw_gate;
  a.beta_logits = beta_logits;
  a.a_log = a_log;
  a.dt_bias = dt_bias;
  a.cu_seqlens = cu_seqlens;
  a.state_pool = state_pool;
  a.state_indices = state_indices;
  a.dev_status = dev_status;
  a.gate_mode = gate_mode;
  a.lower_bound = lower_bound;
  a.q_scale = 1.0f / std::sqrt((float)K);
  a.v_first = state_layout == KDA_STATE_V_FIRST;
  a.out_bf16 = output_dtype == KDA_OUTPUT_BF16;
  a.B = B;
  a.T = T;
  a.H = H;
  a.HV = HV;
  a.G = HV / H;
  a.max_slots = max_slots;
  const cudaError_t e = prefill ? kda::launch_kda_prefill(a, static_cast<cudaStream_t>(stream))
                                : kda::launch_kda_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

extern "C" {

kda_status kda_decode(float* output, const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                      const float* raw_gate, const float* beta_logits, const float* a_log,
                      const float* dt_bias, const int32_t* cu_seqlens, float* state_pool,
                      const int32_t* state_indices, int gate_mode, float lower_bound, int B,
                      int T, int H, int HV, int K, int V, int max_slots, int32_t* dev_status,
                      void* stream) {
  return decode_impl(output, q, k, v, raw_gate, beta_logits, a_log, dt_bias, cu_seqlens,
                     state_pool, state_indices, gate_mode, lower_bound, KDA_STATE_K_FIRST,
                     KDA_OUTPUT_F32, B, T, H, HV, K, V, max_slots, dev_status, stream);
}

kda_status kda_decode_ex(void* output, const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                         const float* raw_gate, const float* beta_logits, const float* a_log,
                         const float* dt_bias, const int32_t* cu_seqlens, float* state_pool,
                         const int32_t* state_indices, int gate_mode, float lower_bound,
                         int state_layout, int output_dtype, int B, int T, int H, int HV, int K,
                         int V, int max_slots, int32_t* dev_status, void* stream) {
  return decode_impl(output, q, k, v, raw_gate, beta_logits, a_log, dt_bias, cu_seqlens,
                     state_pool, state_indices, gate_mode, lower_bound, state_layout,
                     output_dtype, B, T, H, HV, K, V, max_slots, dev_status, stream);
}

kda_status kda_prefill(float* output, const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                       const float* raw_gate, const float* beta_logits, const float* a_log,
                       const float* dt_bias, const int32_t* cu_seqlens, float* state_pool,
                       const int32_t* state_indices, int gate_mode, float lower_bound, int B,
                       int T, int H, int HV, int K, int V, int max_slots, int32_t* dev_status,
                       void* stream) {
  // The chunk form needs the decay accumulated over a chunk bounded: the
  // lower-bound gate with lower_bound >= -5 keeps |G| <= 80, so every
  // e^(+-G) factor is a normal fp32 number.  The softplus gate (unbounded
  // decay) and lower bounds below -5 run the token-by-token kernel instead,
  // which computes the same recurrence.
  const bool chunked = !(gate_mode == KDA_GATE_SOFTPLUS ||
                         (gate_mode == KDA_GATE_LOWER_BOUND && std::isfinite(lower_bound) &&
                          lower_bound < -5.0f));
  return decode_impl(output, q, k, v, raw_gate, beta_logits, a_log, dt_bias, cu_seqlens,
                     state_pool, state_indices, gate_mode, lower_bound, KDA_STATE_K_FIRST,
                     KDA_OUTPUT_F32, B, T, H, HV, K, V, max_slots, dev_status, stream, chunked);
}

size_t kda_block_tkg_workspace_size(int B, int n, int Hd, int nh, int K, int V, int Kc) {
  return kda::block_workspace_bytes(B, n, Hd, nh, K, V, Kc);
}

kda_status kda_block_tkg(float* out, const float* hidden, const float* gamma_in,
                         const kda_bf16* W_in, const kda_bf16* W_fb, const kda_bf16* W_gb,
                         const kda_bf16* conv_w, const float* A_log, const float* dt_bias,
                         const float* gamma_o, const kda_bf16* W_o, float* S, float* conv_state,
                         float scale, float lower_bound, float rms_norm_eps, float l2_eps, int B,
                         int n, int Hd, int nh, int K, int V, int Kc, void* workspace,
                         size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (B < 0 || n < 1 || Hd < 1 || nh < 1 || K < 1 || V < 1 || Kc < 1) return KDA_ERR_SHAPE;
  if (!(std::isfinite(scale) && std::isfinite(lower_bound) && lower_bound <= 0.0f &&
        std::isfinite(rms_norm_eps) && rms_norm_eps >= 0.0f && std::isfinite(l2_eps) &&
        l2_eps >= 0.0f))
    return KDA_ERR_VALUE;
  if (K != kda::kHeadDim || V != kda::kHeadDim || Kc < 2 ||
      Kc > 4 || Hd % 128 != 0)
    return KDA_ERR_UNSUPPORTED;
  if (B == 0) return KDA_OK;
  if (!out || !hidden || !gamma_in || !W_in || !W_fb || !W_gb || !conv_w || !A_log ||
      !dt_bias || !gamma_o || !W_o || !S || !conv_state)
    return KDA_ERR_NULL;
  const void* ptrs[] = {out, hidden, gamma_in, W_in, W_fb, W_gb, conv_w, A_log,
                        dt_bias, gamma_o, W_o, S, conv_state};
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return KDA_ERR_ALIGN;
  const size_t need = kda::block_workspace_bytes(B, n, Hd, nh, K, V, Kc);
  if (need == 0) return KDA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KDA_ERR_ALIGN;

  kda::BlockArgs a;
  a.out = out;
  a.hidden = hidden;
  a.gamma_in = gamma_in;
  a.W_in = W_in;
  a.W_fb = W_fb;
  a.W_gb = W_gb;
  a.conv_w = conv_w;
  a.A_log = A_log;
  a.dt_bias = dt_bias;
  a.gamma_o = gamma_o;
  a.W_o = W_o;
  a.S = S;
  a.conv_state = conv_state;
  a.scale = scale;
  a.lower_bound = lower_bound;
  a.rms_norm_eps = rms_norm_eps;
  a.l2_eps = l2_eps;
  a.B = B;
  a.n = n;
  a.Hd = Hd;
  a.nh = nh;
  a.K = K;
  a.V = V;
  a.Kc = Kc;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.dev_status = dev_status;
  if (kda::launch_kda_block(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KDA_ERR_CUDA;
  return KDA_OK;
}

}  // extern "C"
