// Forward pass for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory for a workspace: a plug-in inside
// a host framework that owns every device allocation and hands its plug-ins only the
// tensors they work on, or a latency-critical caller that must not call cudaMalloc
// because cudaMalloc may synchronise the whole device. lwm_attn_fwd_noalloc serves
// them: its workspace is a file-scope device array that this library holds for as
// long as it is loaded, on every GPU where it is used.
//
// The array is a host-side stand-in in host code: its address on a device is fetched
// with cudaGetSymbolAddress once per device (with that device current) and passed to
// the kernels like any caller-provided workspace. The cached address belongs to the
// runtime's primary context of that device: it assumes that context lives as long as
// the process (no cudaDeviceReset in between, no other context made current).
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace lwm {
namespace {

constexpr size_t NOALLOC_BYTES = LWM_NOALLOC_SCRATCH_BYTES;
constexpr int NOALLOC_MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};

// Device address of the scratch array on the current device (looked up once per device).
lwm_status noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES) return LWM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return LWM_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return LWM_OK;
}

}  // namespace
}  // namespace lwm

extern "C" lwm_status lwm_attn_fwd_noalloc(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v,
                                           const int32_t *seg_ids, const int32_t *pos, lwm_bf16 *out,
                                           float *lse, int B, int S, int H, int D, lwm_stream stream) {
  using namespace lwm;
  const lwm_status sz = check_sizes(B, S, H, D);
  if (sz != LWM_OK) return sz;
  // The forward pass uses only the part of the workspace in front of the backward
  // rows; its size does not depend on H, and the layout with H = 1 up to the dK/dV
  // kernel's offset rows covers it.
  if (Workspace::layout(B, S, 1).off_qx > NOALLOC_BYTES) return LWM_ERR_INVALID_ARG;
  if (!q || !k || !v || !out || !lse) return LWM_ERR_INVALID_ARG;
  const auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const auto a4 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!a16(q) || !a16(k) || !a16(v) || !a16(out) || !a4(lse)) return LWM_ERR_ALIGNMENT;
  if ((seg_ids && !a4(seg_ids)) || (pos && !a4(pos))) return LWM_ERR_ALIGNMENT;
  // an unsupported device is reported as such before the array is looked up
  const lwm_status dev = check_device();
  if (dev != LWM_OK) return dev;
  void *scratch = nullptr;
  const lwm_status st = noalloc_scratch(&scratch);
  if (st != LWM_OK) return st;
  // Header words (error word, scheduler tickets) must start at zero on every call.
  if (cudaMemsetAsync(scratch, 0, HDR_WORDS * sizeof(int), stream) != cudaSuccess) {
    cudaGetLastError();
    return LWM_ERR_CUDA;
  }
  return fwd_with_forward_workspace(q, k, v, seg_ids, pos, out, lse, B, S, H, scratch, stream);
}
