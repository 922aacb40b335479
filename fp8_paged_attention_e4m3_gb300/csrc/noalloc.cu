// verify_attn_e4m3_noalloc: the verify step with library-owned scratch, for
// callers that cannot allocate device memory (see the header for who they
// are).  The scratch is a file-scope __device__ array; its device address is
// looked up once per device and handed to the regular entry point as the
// workspace, so the kernels and their launch path are exactly the ones
// verify_attn_e4m3_ex uses.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"
#include "verify_attn_e4m3.h"

namespace {

// The scratch array.  In host code `g_scratch` names a host-side shadow, not
// device memory: only the address returned by cudaGetSymbolAddress may be
// given to a kernel.
static __device__ __align__(256) unsigned char g_scratch[VAE4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {nullptr};
unsigned long long g_ctx[kMaxDevices] = {0};  // context the address belongs to

// Device address of the scratch on the current device, looked up on first
// use (with that device current) and cached for the device's context; a
// new context (after cudaDeviceReset) gets a fresh lookup.
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VAE4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long ctx = vae4::current_context_id();
  if (!g_addr[dev] || ctx == 0 || ctx != g_ctx[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return VAE4_ERR_CUDA;
    g_addr[dev] = p;
    g_ctx[dev] = vae4::current_context_id();  // the lookup made the context current
  }
  *out = g_addr[dev];
  return VAE4_OK;
}

}  // namespace

extern "C" int verify_attn_e4m3_noalloc(const vae4_tensor *q, const vae4_tensor *kv_pages,
                                        const vae4_tensor *block_table,
                                        const vae4_tensor *seq_lens,
                                        const vae4_tensor *kv_scales, const vae4_tensor *out,
                                        vae4_stream stream, const vae4_options *opt) {
  if (!q || !kv_pages || !block_table || !seq_lens || !kv_scales || !out) return VAE4_ERR_NULL;
  void *scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  vae4_tensor ws = {};
  ws.data = scratch;
  ws.dtype = VAE4_U8;
  ws.ndim = 1;
  ws.shape[0] = VAE4_NOALLOC_SCRATCH_BYTES;
  ws.stride[0] = 1;
  // Nothing in the scratch has to start at zero: every live partition writes
  // its FP32 slots before the combine kernel of the same call reads them,
  // and the status word is only ever OR-ed into (it cannot be read through
  // this entry point), so the previous call's contents are harmless.
  // Validation (including "needs more scratch than the array holds", which
  // returns VAE4_ERR_WORKSPACE) happens before anything else is launched.
  return verify_attn_e4m3_ex(q, kv_pages, block_table, seq_lens, kv_scales, out, &ws, stream,
                             opt);
}
