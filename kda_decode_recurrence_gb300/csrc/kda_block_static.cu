// kda_block_static.cu -- kda_block_tkg for callers that cannot allocate.
//
// Some hosts own every byte of device memory themselves: an inference
// server's memory pool, or a plugin interface that hands a kernel library
// only its input and output buffers.  Such a caller cannot give the block its
// intermediate workspace.  This entry point takes that workspace from a fixed
// array compiled into the library instead, so it makes no allocation at all.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it for the life of the process.  Host code must not use the
// array's name as a device address (on the host it is only a stand-in), so
// the address is looked up once per device with cudaGetSymbolAddress, on the
// first call made with that device current, and cached.
#include <mutex>

#include "kda.h"
#include "kda_internal.h"

namespace {

// Largest workspace this entry point can serve: 16 MiB covers the Kimi K3
// block with B = 32 requests, Hd = 4096, num_head = 32 (about 12.5 MiB).
constexpr size_t kScratchBytes = (size_t)16 << 20;

static __device__ __align__(256) unsigned char g_block_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_block_scratch on the current device (looked up once).
kda_status scratch_on_current_device(void** ptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_block_scratch) != cudaSuccess || p == nullptr)
      return KDA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_block_tkg_static(
    float* out, const float* hidden, const float* gamma_in, const kda_bf16* W_in,
    const kda_bf16* W_fb, const kda_bf16* W_gb, const kda_bf16* conv_w, const float* A_log,
    const float* dt_bias, const float* gamma_o, const kda_bf16* W_o, float* S, float* conv_state,
    float scale, float lower_bound, float rms_norm_eps, float l2_eps, int B, int n, int Hd, int nh,
    int K, int V, int Kc, int32_t* dev_status, void* stream) {
  // Sizes that need no workspace -- invalid ones (size 0) and B == 0 -- go
  // straight to kda_block_tkg, whose checks answer them exactly as for a
  // caller with a workspace and make no CUDA call.  Sizes that need more
  // scratch than the fixed array are refused, also before any CUDA call.
  const size_t need = kda_block_tkg_workspace_size(B, n, Hd, nh, K, V, Kc);
  if (need == 0 || B == 0)
    return kda_block_tkg(out, hidden, gamma_in, W_in, W_fb, W_gb, conv_w, A_log, dt_bias,
                         gamma_o, W_o, S, conv_state, scale, lower_bound, rms_norm_eps, l2_eps, B,
                         n, Hd, nh, K, V, Kc, nullptr, 0, dev_status, stream);
  if (need > kScratchBytes) return KDA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const kda_status st = scratch_on_current_device(&scratch);
  if (st != KDA_OK) return st;
  // Nothing in the workspace has to start at zero: every intermediate is
  // written before it is read within one call.
  return kda_block_tkg(out, hidden, gamma_in, W_in, W_fb, W_gb, conv_w, A_log, dt_bias, gamma_o,
                       W_o, S, conv_state, scale, lower_bound, rms_norm_eps, l2_eps, B, n, Hd, nh,
                       K, V, Kc, scratch, kScratchBytes, dev_status, stream);
}
