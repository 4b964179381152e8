// w4a8_moe_forward_noalloc: the whole MoE layer without any device allocation.
//
// w4a8_moe_forward needs a workspace for its intermediates (routing ids and
// weights, the permutation, the FP8 copies of the activations, Y13, Y2).  Some
// callers cannot provide one: a plugin inside a host application whose
// allocator owns all device memory and hands the plugin nothing but its input
// and output buffers, or a C program that must not allocate after start-up.
// This entry point takes the same inputs and outputs and keeps the
// intermediates in a fixed array in the library's own device memory instead.
//
// The array is a file-scope __device__ variable of kScratchBytes (64 MiB).  Every
// GPU that loads this library holds it until the process exits.  Host code can
// not use the variable's name as a device address, so the first call on each
// device looks the address up with cudaGetSymbolAddress while that device is
// current, and later calls reuse it.  Under CUDA's lazy module loading that
// lookup can be the moment the driver loads this file's module and places the
// array in the device's memory, so a caller that must not see any allocation
// later makes its first call at start-up.
#include <mutex>

#include "common.cuh"

namespace w4a8 {
namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return set_error(W4A8_ERR_CUDA, "no usable current CUDA device");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(W4A8_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed: %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return W4A8_OK;
}

}  // namespace
}  // namespace w4a8

extern "C" size_t w4a8_moe_noalloc_scratch_bytes(void) { return w4a8::kScratchBytes; }

extern "C" int w4a8_moe_forward_noalloc(const uint16_t* x, const float* logits, int64_t T, int64_t H, int64_t I,
                                        int64_t E, int k, int renormalize, const uint8_t* w13, const float* w13_s,
                                        const uint8_t* w2, const float* w2_s, uint16_t* out, void* stream) {
  using namespace w4a8;
  const size_t need = w4a8_moe_workspace_bytes(T, H, I, E, k);
  W4A8_REQUIRE(need > 0, "bad layer shape");
  W4A8_REQUIRE(need <= kScratchBytes,
               "layer needs %zu bytes of intermediates; w4a8_moe_forward_noalloc holds at most %zu "
               "(use w4a8_moe_forward with a caller-provided workspace)",
               need, kScratchBytes);
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  return w4a8_moe_forward(x, logits, T, H, I, E, k, renormalize, w13, w13_s, w2, w2_s, out, scratch, kScratchBytes,
                          stream);
}
