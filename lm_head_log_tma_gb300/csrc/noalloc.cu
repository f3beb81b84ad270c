// Loss stage for callers that cannot allocate device memory.
//
// Some callers have no allocator to hand: code running while a CUDA graph is
// being captured by someone else, plugins that receive only the tensors they
// read and write, and runtimes whose memory pool is fully reserved up front
// for weights and activations.  For them this entry point runs the same loss
// stage as rlloss_loss_from_logp, but its scratch lives in a file-scope
// device array of fixed size instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "status.h"

namespace {

constexpr size_t kScratchBytes = RLLOSS_NOALLOC_SCRATCH_BYTES;   // 4 MiB, held by every GPU that loads the library
static_assert(kScratchBytes == (size_t(4) << 20), "scratch size is part of the ABI");

static __device__ __align__(256) unsigned char g_loss_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_loss_scratch on the current device, looked up once per
// device.  (In host code the array's name is only a host-side stand-in.)
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RLLOSS_ECUDA;
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_loss_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return RLLOSS_ECUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return RLLOSS_OK;
}

// Forget the cached address of the current device, so that the next call looks
// it up again (after a CUDA error, which a device reset would also produce).
void forget_scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
  std::lock_guard<std::mutex> g(g_mu);
  g_scratch_ptr[dev] = nullptr;
}

}  // namespace

extern "C" int rlloss_loss_from_logp_noalloc(const rlloss_cfg* cfg, const float* logp, const float* entropy,
                                             const float* old_logp, const float* ref_logp, const float* adv,
                                             const uint8_t* mask, float* out_loss, float* out_metrics,
                                             float* out_dlogp, uint8_t* out_entropy_mask,
                                             int32_t* out_device_status, void* stream) {
  const size_t need = rlloss_loss_workspace_bytes(cfg);
  if (need == 0) {
    // The configuration failed validation: let the workspace entry, which
    // validates before anything else, name the reason, so both entries return
    // the same code for the same cfg.  No workspace is passed, so nothing runs.
    const int v = rlloss_loss_from_logp(cfg, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                        nullptr, nullptr, nullptr, nullptr, 0, stream);
    return v != RLLOSS_OK ? v : RLLOSS_EINVAL;
  }
  if (need > kScratchBytes) return RLLOSS_ETOOLARGE;
  void* scratch = nullptr;
  const int e = scratch_address(&scratch);
  if (e != RLLOSS_OK) return e;
  const int rc = rlloss_loss_from_logp(cfg, logp, entropy, old_logp, ref_logp, adv, mask, out_loss, out_metrics,
                                       out_dlogp, out_entropy_mask, scratch, kScratchBytes, stream);
  if (rc == RLLOSS_ECUDA) forget_scratch_address();
  if (rc != RLLOSS_OK) return rc;
  if (out_device_status) {
    // the status word sits at the start of the scratch
    if (cudaMemcpyAsync(out_device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess) {
      forget_scratch_address();
      return RLLOSS_ECUDA;
    }
  }
  return RLLOSS_OK;
}
