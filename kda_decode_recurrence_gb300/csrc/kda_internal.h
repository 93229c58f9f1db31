// kda_internal.h -- argument bundles passed from the C ABI layer to the
// kernel launchers (host and device visible; no allocation, no ownership).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Head dimension this build implements (the block API page allows dk, dv <=
// 128; the Kimi K3 atlas page gives 128).
constexpr int kHeadDim = 128;

struct DecodeArgs {
  void* output;  // fp32 or bf16 [T, HV, V] (out_bf16)
  const kda_bf16* q;
  const kda_bf16* k;
  const kda_bf16* v;
  const float* raw_gate;
  const float* beta_logits;
  const float* a_log;
  const float* dt_bias;
  const int32_t* cu_seqlens;
  float* state_pool;
  const int32_t* state_indices;
  int32_t* dev_status;
  int gate_mode;
  float lower_bound;
  float q_scale;  // K^-1/2
  int v_first;    // state tiles stored [V, K] instead of [K, V]
  int out_bf16;   // output written as bf16
  int B, T, H, HV, G, max_slots;
  // Limit of every wait of the decode kernel on a copy (ns).  A test-only
  // build of the library can shorten it and name one work item whose tile
  // copy is never issued (withhold_item; -1: none), to exercise the path that
  // reports KDA_DEV_TIMEOUT; the product build always runs with the full
  // limit and no withheld item.
  unsigned long long wait_ns;
  long long withhold_item;
};

cudaError_t launch_kda_decode(const DecodeArgs& args, cudaStream_t stream);
cudaError_t launch_kda_prefill(const DecodeArgs& args, cudaStream_t stream);

struct BlockArgs {
  float* out;
  const float* hidden;
  const float* gamma_in;
  const kda_bf16* W_in;
  const kda_bf16* W_fb;
  const kda_bf16* W_gb;
  const kda_bf16* conv_w;
  const float* A_log;
  const float* dt_bias;
  const float* gamma_o;
  const kda_bf16* W_o;
  float* S;
  float* conv_state;
  float scale, lower_bound, rms_norm_eps, l2_eps;
  int B, n, Hd, nh, K, V, Kc;
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;
};

size_t block_workspace_bytes(int B, int n, int Hd, int nh, int K, int V, int Kc);
cudaError_t launch_kda_block(const BlockArgs& args, cudaStream_t stream);

}  // namespace kda
