// ra_attention_bwd_noalloc: the attention backward for callers that cannot allocate
// device memory.
//
// ra_attention_bwd needs a device workspace of ra_attention_bwd_workspace_size() bytes,
// which its caller allocates.  Some callers cannot do that: code running inside a
// framework that owns the allocator and exposes no hook for temporary buffers, and
// hosts that have to avoid cudaMalloc because it synchronises the device or is not
// allowed on their path.  For them this entry point takes the workspace from a
// fixed-size array that the library itself places in device memory, so nothing is
// allocated per call.
//
// The array is a file-scope __device__ variable: every GPU that loads this library
// holds RA_NOALLOC_SCRATCH_BYTES of device memory for it until the process exits.  On
// the host its name is only a stand-in, so the device address is taken once per device
// with cudaGetSymbolAddress and cached.
#include <mutex>

#include "kernels.cuh"

namespace raattn {
namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[RA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
void* g_scratch_ptr[kMaxScratchDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up on first use).
// Device ordinals from kMaxScratchDevices on are beyond what the cache holds.
ra_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return RA_ERR_LAUNCH;
  if (dev >= kMaxScratchDevices) return RA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return RA_ERR_LAUNCH;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return RA_OK;
}

}  // namespace
}  // namespace raattn

extern "C" ra_status_t ra_attention_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                                const void* dout, const float* row_m, const float* row_s,
                                                const int32_t* row_arg, void* dq, void* dk, void* dv, int B,
                                                int H, int N_Q, int N_K, int D, float scale, int causal,
                                                ra_dtype_t in_dtype, ra_dtype_t o_dtype, ra_dtype_t grad_dtype,
                                                void* stream) {
  // the workspace this call's path uses: fp32 inputs need far less than bf16 ones
  const size_t need = raattn::bwd_workspace_bytes(B, H, N_Q, N_K, D, in_dtype == RA_F32);
  if (need == 0) return RA_ERR_ARG;
  if (need > RA_NOALLOC_SCRATCH_BYTES) return RA_ERR_UNSUPPORTED;   // use ra_attention_bwd with a workspace
  void* scratch = nullptr;
  const ra_status_t got = raattn::scratch_for_current_device(&scratch);
  if (got != RA_OK) return got;
  // Nothing in the workspace has to start at zero: every entry the kernels read is
  // written earlier in the same call, so the previous call's contents do no harm.
  return ra_attention_bwd(q, k, v, o, dout, row_m, row_s, row_arg, dq, dk, dv, scratch, B, H, N_Q, N_K, D, scale,
                          causal, in_dtype, o_dtype, grad_dtype, stream);
}
