// Internal launchers of the attention kernels (host side; not part of the C ABI).
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace lwm {

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current device, once
// per device (the attribute belongs to the kernel in each device's context, so a process
// that drives several GPUs needs it on each). `done` holds one bit per device ordinal.
inline cudaError_t smem_attr_once(const void *kernel, int bytes, std::atomic<uint64_t> &done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

struct Problem {
  int B, S, H;
  int num_sms;
};

cudaError_t launch_meta(const int *seg, const int *pos, int B, int S, int kv_chunk, void *workspace,
                        cudaStream_t stream);

cudaError_t launch_fwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, void *out,
                       float *lse, const Problem &p, void *workspace, cudaStream_t stream);

cudaError_t launch_delta(const void *out, const void *dout, const float *lse, const Problem &p, void *workspace,
                         cudaStream_t stream);

cudaError_t launch_dkdv(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const CUtensorMap &tdo, void *dk, void *dv, const Problem &p,
                        void *workspace, cudaStream_t stream);

// tdqacc: the workspace's fp32 dQ accumulator as a 2-D tensor map of
// [B * H * S_pad rows, 128 dims], boxes of 8 rows x 32 dims, no swizzle.
cudaError_t launch_dkdvq(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tdo,
                         const CUtensorMap &tdqacc, void *dq, void *dk, void *dv, const Problem &p, void *workspace,
                         cudaStream_t stream);

cudaError_t launch_dq(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                      const CUtensorMap &tdo, void *dq, const Problem &p, void *workspace,
                      cudaStream_t stream);

}  // namespace lwm

#include "lwm_attn.h"

namespace lwm {

// Host-side argument checks shared by the entry points (api.cu).
lwm_status check_sizes(int B, int S, int H, int D);
// LWM_OK when the current device is one the kernels are built for (sm_103),
// LWM_ERR_UNSUPPORTED when it is not, LWM_ERR_CUDA when it cannot be queried.
lwm_status check_device();

lwm_status fwd_with_forward_workspace(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const int32_t *seg,
                                      const int32_t *pos, lwm_bf16 *out, float *lse, int B, int S, int H, void *ws,
                                      cudaStream_t stream);

}  // namespace lwm
