// mhc_seam_noalloc: the split-path seam with its scratch in a static device
// array, for callers that cannot allocate device memory.
//
// Who needs it: callers that may not call cudaMalloc -- a plug-in loaded into
// a host program that owns every device allocation and gives the plug-in none
// of its own, code that runs inside an allocator or memory-pool callback where
// re-entering the allocator would deadlock, and latency-critical loops that
// must never block in the driver's allocator.  Such a caller still passes its
// inputs and outputs, but cannot hand this library a workspace.  The split path needs scratch (per-CTA partial sums, arrival
// counters, a status word), so this entry point keeps it in a file-scope
// __device__ array of kNoAllocScratchBytes that every GPU which loads the
// library holds until the process exits.
//
// Set-up: the first call on a device (with that device current) resolves the
// array's device address with cudaGetSymbolAddress; that first call should be
// made before any stream capture.  Every call clears the part of the array it
// uses for partial sums and arrival counters (cudaMemsetAsync on the caller's
// stream: no allocation) and then runs the ordinary split path with the array
// as its workspace.  The status word at the start of the array is not cleared
// by a call: a bounded wait that ran out in any call stays recorded until
// mhc_noalloc_check_status() reads and clears it.  All calls share the one
// array, so calls that can overlap on the GPU (different streams, or
// concurrent graphs) race on it and must be serialised by the caller.

#include <mutex>
#include <string>

#include "mhc_common.cuh"
#include "../../include/mhc_seam.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr size_t kStatusBytes = 256;  // the status word's header at the start of every workspace
constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

}  // namespace

namespace mhc {
void set_last_error(const std::string& msg);  // mhc_api.cu: the text mhc_last_error_string() returns
}

namespace {
int noalloc_fail(int code, const std::string& msg) {
  mhc::set_last_error(msg);
  return code;
}

// Device address of the static scratch on the current device, resolved once
// per device (with that device current); MHC_OK or an error status.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return noalloc_fail(MHC_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(MHC_ERR_CUDA, "device index out of range");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess)
      return noalloc_fail(MHC_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MHC_OK;
}
}  // namespace

extern "C" {

int mhc_seam_noalloc(const void* R, const void* Y, const float* post_prev, const float* comb_prev,
                     const float* pre_prev, const float* fn, const float* bias, const float* alpha,
                     const void* gamma, float eps, int64_t T, int H, mhc_out_mode out_mode, void* residual_out,
                     void* norm, uint8_t* fp8_codes, uint8_t* e8m0_scales, float* pre_out, float* post_out,
                     float* comb_out, const mhc_config* cfg, void* stream) {
  mhc_config c = {};
  if (cfg) c = *cfg;
  if (c.path == 2 || c.path == 3)
    return noalloc_fail(MHC_ERR_CONFIG, "mhc_seam_noalloc runs the split path only (cfg.path 0 or 1)");
  c.path = 1;
  if (T < 0 || H <= 0) return mhc_seam(R, Y, post_prev, comb_prev, pre_prev, fn, nullptr, bias, alpha, gamma, eps, T,
                                       H, out_mode, residual_out, norm, fp8_codes, e8m0_scales, pre_out, post_out,
                                       comb_out, nullptr, 0, &c, stream);
  const size_t need = mhc_workspace_bytes(T, H, &c);
  if (need > kNoAllocScratchBytes)
    return noalloc_fail(MHC_ERR_WORKSPACE, "mhc_seam_noalloc: this call needs " + std::to_string(need) +
                                               " bytes of scratch, above the fixed " +
                                               std::to_string(kNoAllocScratchBytes) + "-byte array");
  if (T == 0)
    return mhc_seam(R, Y, post_prev, comb_prev, pre_prev, fn, nullptr, bias, alpha, gamma, eps, T, H, out_mode,
                    residual_out, norm, fp8_codes, e8m0_scales, pre_out, post_out, comb_out, nullptr, 0, &c, stream);

  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != MHC_OK) return rc;
  // clear the partial sums and arrival counters; the status word stays
  cudaError_t e = cudaSuccess;
  if (need > kStatusBytes)
    e = cudaMemsetAsync(static_cast<char*>(scratch) + kStatusBytes, 0, need - kStatusBytes,
                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return noalloc_fail(MHC_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
  return mhc_seam(R, Y, post_prev, comb_prev, pre_prev, fn, nullptr, bias, alpha, gamma, eps, T, H, out_mode,
                  residual_out, norm, fp8_codes, e8m0_scales, pre_out, post_out, comb_out, scratch, need, &c, stream);
}

int mhc_noalloc_check_status(void* stream) {
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != MHC_OK) return rc;
  return mhc_check_status(scratch, stream);
}

}  // extern "C"
