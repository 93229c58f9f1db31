/*
 * kda.h -- C ABI of libkda, the GB300 (sm_103a) KDA token-generation library.
 *
 * Two operations, each with variants:
 *   kda_decode     the Kimi Delta Attention decode recurrence over a
 *                  slot-indexed fp32 state pool, varlen tokens per request;
 *                  kda_decode_ex chooses the state layout (K-first or V-first)
 *                  and the output dtype (fp32 or bf16), kda_prefill computes
 *                  the same recurrence over whole prompts in 16-token chunks.
 *   kda_block_tkg  the fused KDA block for token generation (input RMSNorm,
 *                  fused projection, short convolutions, gates, recurrence,
 *                  gated output RMSNorm, output projection), n >= 1 tokens per
 *                  request; kda_block_tkg_static needs no caller workspace.
 *
 * Conventions shared by every call:
 *   - Every tensor pointer is a DEVICE pointer (cudaMalloc'd or equivalent),
 *     allocated, owned and freed by the caller.  The library keeps no pointer
 *     after a call returns and allocates no device memory.
 *   - Tensors are dense and row-major (last dimension contiguous) in the
 *     shapes given below.  bf16 tensors are passed as their 16-bit patterns
 *     (kda_bf16).
 *   - Calls are asynchronous: kernels are enqueued on `stream` (a cudaStream_t
 *     passed as void*; NULL means the legacy default stream) and the call
 *     returns without synchronising.
 *   - A host-detected problem returns a negative kda_status and launches
 *     nothing; no memory is touched.
 *   - A problem that only the device can see (a slot index out of range, a
 *     malformed cu_seqlens, an internal wait that gave up) never traps: the
 *     kernel skips the affected work and ORs a KDA_DEV_* bit into *dev_status
 *     (a device int32 the caller zeroes beforehand).  dev_status may be NULL,
 *     but then those reports are lost: a call can leave the state partly
 *     advanced (some requests skipped, or after KDA_DEV_TIMEOUT some tiles not
 *     written back) with no sign of it.  Pass a status word wherever the
 *     inputs are not known to be valid.
 *   - Calls that write the same state slots must not overlap in time.
 *
 * Page citations name the page title and the section it falls in:
 *   "KdaDecode"                       MAX Mojo builtin kernel, struct KdaDecode:
 *                                     Default parameters, Tensor Shapes, execute
 *   "KDA Block TKG Kernel API Reference"  AWS Neuron NKI kda_block_tkg:
 *                                     Background, signature, :param: entries,
 *                                     Dimensions
 *   "Delta-rule write"                Kimi K3 model atlas: prose, naive
 *                                     recurrent loop, attention forward code
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kda_bf16; /* bfloat16 bit pattern */

typedef enum kda_status {
  KDA_OK = 0,
  KDA_ERR_NULL = -1,        /* a required pointer is NULL                         */
  KDA_ERR_SHAPE = -2,       /* a size is out of range or sizes are inconsistent  */
  KDA_ERR_UNSUPPORTED = -3, /* valid sizes this build does not implement         */
  KDA_ERR_ENUM = -4,        /* unknown gate_mode, state_layout or output_dtype   */
  KDA_ERR_CUDA = -5,        /* a CUDA runtime call (launch) failed                */
  KDA_ERR_ALIGN = -6,       /* a pointer is not aligned as documented             */
  KDA_ERR_VALUE = -7,       /* a scalar argument is not finite / out of range     */
  KDA_ERR_WORKSPACE = -8    /* workspace missing or smaller than required         */
} kda_status;

/* gate_mode values.  "KdaDecode", Default parameters: gate_mode "original" is
 * the stable-softplus gate; "KDA Block TKG Kernel API Reference", :param
 * lower_bound: the activated gate is lower_bound * sigmoid(...). */
#define KDA_GATE_SOFTPLUS 0    /* g = -exp(a_log) * softplus(raw + dt_bias)              */
#define KDA_GATE_LOWER_BOUND 1 /* g = lower_bound * sigmoid(exp(a_log) * (raw + dt_bias)) */

/* Bits ORed into *dev_status by the kernels. */
#define KDA_DEV_BAD_SLOT 1   /* state_indices[b] >= max_slots: request b skipped, rows zeroed */
#define KDA_DEV_BAD_SEQLEN 2 /* cu_seqlens not 0 <= cu[b] <= cu[b+1] <= T, or cu[0] != 0, or
                                cu[B] != T: a request with a bad range is skipped              */
#define KDA_DEV_TIMEOUT 4    /* an internal copy/tensor-core pipeline wait exceeded its 1 s limit;
                                the kernel stopped early and its results are incomplete          */
#define KDA_DEV_BOUNDS 8     /* debug builds only (libkda_debugbounds.so, compiled with
                                KDA_DEBUG_BOUNDS=1): an index the kernels derived fell outside
                                its tensor; that access was skipped.  Never set by libkda.so,
                                whose kernels carry no such checks.                              */

/*
 * kda_decode -- advance each request's recurrent state over its new tokens.
 *
 * Defined by "KdaDecode" (Tensor Shapes; Default parameters gate_mode
 * original / beta_mode logits / state_layout K_FIRST) and "Delta-rule write"
 * (the naive recurrent loop: decay, delta write, read).  For every request b
 * and value head hv, with G = HV / H and key head h = hv / G:
 *
 *   S = state_pool[state_indices[b], hv]                         [K, V] fp32
 *   for t in cu_seqlens[b] .. cu_seqlens[b+1]-1:
 *     qh = q[t,h] / sqrt(|q[t,h]|^2 + 1e-6) * K^-1/2
 *     kh = k[t,h] / sqrt(|k[t,h]|^2 + 1e-6)
 *     g  = gate(raw_gate[t,hv] + dt_bias[hv], a_log[hv])   (per key channel)
 *     beta = sigmoid(beta_logits[t,hv])
 *     S  = diag(exp(g)) S                                     decay
 *     S  = S + beta * kh (v[t,hv] - kh^T S)^T                 delta write
 *     output[t,hv] = qh^T S                                   read after write
 *   state_pool[state_indices[b], hv] = S                      in place
 *
 * Arguments (shapes without the pages' leading batch axis of 1):
 *   output        [T, HV, V]  fp32, written.  Rows of padded (slot < 0) or
 *                 bad-slot requests are written as 0.  Alignment 16 B.
 *   q, k          [T, H, K]   bf16.  Alignment 8 B.
 *   v             [T, HV, V]  bf16.  Alignment 8 B.
 *   raw_gate      [T, HV, K]  fp32 gate pre-activation.  Alignment 16 B.
 *   beta_logits   [T, HV]     fp32.
 *   a_log         [HV]        fp32 log-gate parameter (exp(a_log) scales the
 *                 gate pre-activation).
 *   dt_bias       [HV, K]     fp32 per-channel gate bias.  Alignment 16 B.
 *   cu_seqlens    [B + 1]     int32, request b owns tokens cu[b] .. cu[b+1]-1;
 *                 cu[0] = 0, non-decreasing, cu[B] = T (checked on device).
 *   state_pool    [max_slots, HV, K, V] fp32, K_FIRST (row k contiguous over
 *                 v), read and written in place.  Alignment 16 B.  Slots not
 *                 named by state_indices are never touched.
 *   state_indices [B] int32 slot per request; < 0 marks a padded request
 *                 (skipped, no error); >= max_slots sets KDA_DEV_BAD_SLOT.
 *                 Slots must be distinct among non-padded requests.
 *   gate_mode     KDA_GATE_SOFTPLUS or KDA_GATE_LOWER_BOUND.
 *   lower_bound   used by KDA_GATE_LOWER_BOUND only; finite and <= 0
 *                 ("expected in [-5, 0]").
 *   B, T, H, HV, K, V, max_slots  sizes; B = 0 or T = 0 is a no-op apart from
 *                 device checks.  HV % H == 0.  This build implements
 *                 K == V == 128 (the pages allow <= 128).
 *   dev_status    device int32*, nullable (see conventions).
 *   stream        cudaStream_t as void*.
 *
 * An empty request (cu[b] == cu[b+1]) leaves its state bit-identical.
 * Returns KDA_OK after enqueuing, or a negative status without launching.
 */
kda_status kda_decode(float* output, const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                      const float* raw_gate, const float* beta_logits, const float* a_log,
                      const float* dt_bias, const int32_t* cu_seqlens, float* state_pool,
                      const int32_t* state_indices, int gate_mode, float lower_bound, int B,
                      int T, int H, int HV, int K, int V, int max_slots, int32_t* dev_status,
                      void* stream);

/* state_layout and output_dtype values of kda_decode_ex.  "KdaDecode", execute:
 * the state_layout and output_dtype template parameters; "Delta-rule write",
 * attention forward: the model keeps its state transposed
 * (transpose_state_layout=True). */
#define KDA_STATE_K_FIRST 0 /* tile [K, V], row k contiguous over v (kda_decode) */
#define KDA_STATE_V_FIRST 1 /* tile [V, K], row v contiguous over k (the transposed state) */
#define KDA_OUTPUT_F32 0
#define KDA_OUTPUT_BF16 1

/*
 * kda_decode_ex -- kda_decode with the state layout and output dtype chosen
 * at run time.  Same operation, arguments and error behaviour as kda_decode,
 * except:
 *   output        [T, HV, V] fp32 (KDA_OUTPUT_F32, alignment 16 B) or bf16
 *                 (KDA_OUTPUT_BF16, round to nearest even, alignment 8 B).
 *   state_pool    [max_slots, HV, K, V] (KDA_STATE_K_FIRST) or
 *                 [max_slots, HV, V, K] (KDA_STATE_V_FIRST) fp32.
 *   state_layout, output_dtype  the enums above; anything else returns
 *                 KDA_ERR_ENUM.
 * kda_decode(...) is kda_decode_ex(..., KDA_STATE_K_FIRST, KDA_OUTPUT_F32, ...).
 */
kda_status kda_decode_ex(void* output, const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                         const float* raw_gate, const float* beta_logits, const float* a_log,
                         const float* dt_bias, const int32_t* cu_seqlens, float* state_pool,
                         const int32_t* state_indices, int gate_mode, float lower_bound,
                         int state_layout, int output_dtype, int B, int T, int H, int HV, int K,
                         int V, int max_slots, int32_t* dev_status, void* stream);

/*
 * kda_prefill -- the same recurrence as kda_decode, computed in chunks of 16
 * tokens: the whole-sequence form ("Delta-rule write": the model runs
 * chunk_kda over a full sequence and fused_recurrent_kda for one new token
 * with a cache).  Arguments, layouts, outputs, state handling and device
 * status bits are those of kda_decode (K_FIRST state, fp32 output); the
 * result equals the token-by-token recurrence up to rounding (the products
 * against the state run on the tensor cores with every fp32 operand split
 * into three bf16 parts, about as accurate as fp32).  The device status bit
 * KDA_DEV_TIMEOUT reports a bounded wait on the tensor cores that gave up;
 * that request's state tile is then left unwritten.  Meant for
 * long prompts: each request's tokens are processed 16 at a time by one CTA
 * per (request, value head).
 *
 * The chunk form needs gate_mode == KDA_GATE_LOWER_BOUND with
 * -5 <= lower_bound <= 0 ("KDA Block TKG Kernel API Reference", :param
 * lower_bound:, the bound on the cumulative decay that the chunkwise prefill
 * depends on).  With the softplus gate or a lower bound below -5 the call runs
 * kda_decode's token-by-token kernel instead: same arguments, same results as
 * kda_decode bit for bit.
 */
kda_status kda_prefill(float* output, const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                       const float* raw_gate, const float* beta_logits, const float* a_log,
                       const float* dt_bias, const int32_t* cu_seqlens, float* state_pool,
                       const int32_t* state_indices, int gate_mode, float lower_bound, int B,
                       int T, int H, int HV, int K, int V, int max_slots, int32_t* dev_status,
                       void* stream);

/*
 * kda_block_tkg -- the fused KDA block for token generation.
 *
 * Defined by "KDA Block TKG Kernel API Reference" (Background; signature;
 * :param hidden:, gamma_in, W_in, W_fb, W_gb, conv_w, A_log, dt_bias, gamma_o,
 * W_o, out, S, conv_state, scale, rms_norm_eps, lower_bound; Dimensions), with
 * the recurrence of "Delta-rule write".  Per request b (nh = num_head heads,
 * here key heads = value heads; I = 2*K*nh + V*nh + 2*K + nh):
 *   x  = hidden[b] * rsqrt(mean(hidden[b]^2) + rms_norm_eps) * gamma_in
 *   P  = x . W_in       columns q | k | v | g_a | beta | f_a, widths
 *                       K*nh, K*nh, V*nh, K, nh, K; q, k channel-outer
 *                       (column d*nh + h), v head-outer (h*V + d)
 *   q, k, v: depthwise causal conv over [conv_state (oldest first), P],
 *            tap 0 oldest, then SiLU; conv_state keeps the last Kc-1
 *            PRE-convolution inputs
 *   g  = lower_bound * sigmoid(exp(A_log[h]) * (f_a . W_fb[:, h*K + d] + dt_bias[d, h]))
 *   beta = sigmoid(P_beta[h]); q, k L2-normalised (l2_eps), q * scale
 *   S[b, h] advanced by the delta rule (as kda_decode), o = q^T S
 *   on = o * rsqrt(mean_d(o^2) + rms_norm_eps) * gamma_o * sigmoid(g_a . W_gb[:, d*nh + h])
 *        (the page calls this RMSNorm "gated" without naming the activation:
 *        sigmoid here; the library built with KDA_BLOCK_OUTPUT_GATE_SWISH=1,
 *        shipped as libkda_outgate_swish.so, uses z * sigmoid(z) instead)
 *   out[b] = on (flattened h*V + d) . W_o
 *
 * Arguments:
 *   out        [B, n, Hd] fp32, written: the output projection (with one
 *              tensor-parallel rank this is the complete activation).
 *   hidden     [B, n, Hd] fp32 block input (before the RMSNorm).
 *   gamma_in   [Hd] fp32.            W_in  [Hd, I] bf16, contraction-first.
 *   W_fb       [K, K*nh] bf16 (head-outer).  W_gb [K, V*nh] bf16 (channel-outer).
 *   conv_w     [3, Kc, K*nh] bf16, tap-major, stream channel order as in W_in.
 *   A_log      [nh] fp32.            dt_bias [K, nh] fp32.
 *   gamma_o    [V] fp32.             W_o   [V*nh, Hd] bf16, contraction-first.
 *   S          [B, nh, K, V] fp32, read and advanced in place.
 *   conv_state [B, 3, K*nh, Kc-1] fp32, read and advanced in place.
 *   scale, lower_bound, rms_norm_eps, l2_eps  scalars (finite; lower_bound <= 0,
 *              eps >= 0).
 *   B, n, Hd, nh, K, V, Kc  sizes.  n >= 1 tokens per request (the page
 *              fixes n = 1 "today" and keeps the axis for a speculative
 *              verify/replay window; here the n tokens of a request are taken
 *              in order, each convolution window ending at its own token and
 *              the state carried from token to token; out[b, j] is token j's
 *              output).  This build implements K == V == 128, Kc in 2..4, Hd a
 *              multiple of 128 and nh a multiple of 8.
 *   workspace  device scratch of at least kda_block_tkg_workspace_size(...)
 *              bytes, 256-byte aligned; contents need not be initialised and
 *              are clobbered.
 *   dev_status nullable device int32; KDA_DEV_TIMEOUT is the only bit the
 *              block can set.
 * All pointers 16-byte aligned.
 */
kda_status kda_block_tkg(float* out, const float* hidden, const float* gamma_in,
                         const kda_bf16* W_in, const kda_bf16* W_fb, const kda_bf16* W_gb,
                         const kda_bf16* conv_w, const float* A_log, const float* dt_bias,
                         const float* gamma_o, const kda_bf16* W_o, float* S, float* conv_state,
                         float scale, float lower_bound, float rms_norm_eps, float l2_eps, int B,
                         int n, int Hd, int nh, int K, int V, int Kc, void* workspace,
                         size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * kda_block_tkg_static -- kda_block_tkg that allocates nothing and takes no
 * workspace argument.  The pages have no counterpart to this call: it exists
 * for callers that cannot hand the block a workspace because their host owns
 * all device memory (an inference server's memory pool, a plugin interface
 * that passes a kernel library only its input and output buffers).
 *
 * The intermediates live in one fixed 16 MiB device array inside the library
 * (held on every GPU that loads the library until the process exits), which
 * serves the Kimi K3 block with B = 32 requests, Hd = 4096, num_head = 32.
 * Arguments and results are those of kda_block_tkg without workspace and
 * workspace_bytes.
 *   - Sizes that need more than 16 MiB of workspace (see
 *     kda_block_tkg_workspace_size) return KDA_ERR_WORKSPACE before any CUDA
 *     call.  Invalid sizes and B = 0 return what kda_block_tkg returns for
 *     them, also without a CUDA call.
 *   - The first call made with a given device current looks up the array's
 *     device address on that device (cudaGetSymbolAddress) and caches it;
 *     make that first call before any stream capture.
 *   - Every call uses the same array and leaves its last contents there, so
 *     two calls that can run on the GPU at the same time (different streams,
 *     no ordering between them) race and corrupt each other's results.
 * No cudaMalloc, cudaFree or other allocating routine is called.
 */
kda_status kda_block_tkg_static(float* out, const float* hidden, const float* gamma_in,
                                const kda_bf16* W_in, const kda_bf16* W_fb, const kda_bf16* W_gb,
                                const kda_bf16* conv_w, const float* A_log, const float* dt_bias,
                                const float* gamma_o, const kda_bf16* W_o, float* S,
                                float* conv_state, float scale, float lower_bound,
                                float rms_norm_eps, float l2_eps, int B, int n, int Hd, int nh,
                                int K, int V, int Kc, int32_t* dev_status, void* stream);

/* Bytes of device workspace kda_block_tkg needs for these sizes (0 when the
 * sizes are invalid).  Host-only, no CUDA call. */
size_t kda_block_tkg_workspace_size(int B, int n, int Hd, int nh, int K, int V, int Kc);

/* Static description of a status code.  Host-only. */
const char* kda_status_string(kda_status status);

/* Library version string ("kda-gb300 <major>.<minor>").  Host-only. */
const char* kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
