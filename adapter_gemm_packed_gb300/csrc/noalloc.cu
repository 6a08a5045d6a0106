// mlora_forward_static_ws: the forward pass without a caller-provided workspace.
//
// Who needs it: code that may not allocate device memory at the point where it runs the
// layer -- for example a host runtime that forbids cudaMalloc after start-up, a framework that
// hands out memory only from its own pools and cannot size an extra scratch buffer, or a
// caller that must not touch the allocator while another thread is capturing work.  For
// them the library keeps its own scratch: one file-scope device array of STATIC_WS_BYTES that
// exists on every GPU the library's device code is loaded on, until the process exits.
//
// The kernels are exactly those of mlora_forward; only the scratch pointer differs.
#include <mutex>
#include <string>

#include "common.cuh"
#include "mlora.h"

namespace {

constexpr size_t STATIC_WS_BYTES = size_t(64) << 20;   // 64 MiB on every device that loads the library

// The scratch.  In host code this name is only a stand-in for the device array; its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_ws[STATIC_WS_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_ws_ptr[MAX_DEVICES] = {};

}  // namespace

namespace mlora {
void set_last_error(const std::string& msg);                            // api.cu
void forget_workspace(const mlora_plan_t* plan, const void* workspace);   // api.cu
bool plan_is_w4(const mlora_plan_t* plan);                              // api.cu
}

extern "C" {

mlora_status mlora_forward_static_ws(const mlora_plan_t* plan, const void* X, const void* Wt, void* Y, float* H,
                                     void* stream) {
  if (!plan) {
    mlora::set_last_error("null plan");
    return MLORA_ERR_INVALID;
  }
  if (mlora::plan_is_w4(plan)) {
    // a 4-bit base would also need its bf16 expansion (2 d_in d_out bytes) in the scratch
    mlora::set_last_error("mlora_forward_static_ws: plans with a 4-bit base (MLORA_BF16_W4) are not supported; "
                          "use mlora_forward_w4 with a caller workspace");
    return MLORA_ERR_UNSUPPORTED;
  }
  // The forward needs the plan's workspace minus the backward-only image set.
  int64_t summ[12] = {0};
  int64_t count = 0;
  mlora_status st = mlora_plan_describe(plan, MLORA_Q_SUMMARY, summ, 12, &count);
  if (st != MLORA_OK) return st;
  const int64_t ws_bytes = summ[11], n_images = summ[7];
  const size_t need = ws_bytes == 0 ? 0 : static_cast<size_t>(ws_bytes - n_images * mlora::IMG_BYTES);
  if (need > STATIC_WS_BYTES) {
    mlora::set_last_error("mlora_forward_static_ws: this plan needs " + std::to_string(need) +
                          " bytes of scratch, more than the library's static " + std::to_string(STATIC_WS_BYTES) +
                          "; use mlora_forward with a caller workspace");
    return MLORA_ERR_UNSUPPORTED;
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    mlora::set_last_error("mlora_forward_static_ws: no usable current device");
    return MLORA_ERR_CUDA;
  }
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ws_ptr[dev]) {
      // One-time set-up on this device (it is current here): look up the device address of
      // the scratch array.  This calls no allocator; the array belongs to the library's module.
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_ws);
      if (e != cudaSuccess || !p) {
        mlora::set_last_error(std::string("mlora_forward_static_ws: cudaGetSymbolAddress failed: ") +
                              cudaGetErrorString(e));
        return MLORA_ERR_CUDA;
      }
      g_ws_ptr[dev] = p;
    }
    ws = g_ws_ptr[dev];
  }
  // Every plan on this device writes the same array, so what this plan left there may have been
  // overwritten since: make the forward rebuild its bf16 shadows instead of trusting its record
  // (MLORA_REUSE_STAGING would otherwise skip the pack and read another plan's adapters).  With
  // that, nothing in the scratch needs to start at zero: every byte the forward reads was
  // written earlier in the same call.
  mlora::forget_workspace(plan, ws);
  return mlora_forward(plan, X, Wt, Y, H, ws, stream);
}

}  // extern "C"
