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

// RoPE rotation of q and/or k (either may be null), in place when y == x.
cudaError_t launch_rope(const void *x0, const void *x1, const int *pos, double theta, void *y0, void *y1, int B,
                        int S, int H, bool inverse, int num_sms, cudaStream_t stream);

// Decoding against a key/value cache: workspace layout (header words, then the
// per-split (m, l) pairs and unnormalised outputs) and the two launches (splits, merge).
struct DecodeLayout {
  int split_len, n_split;
  size_t off_ml, off_o, total;
};
DecodeLayout decode_layout(int B, int T, int S_max, int H);
cudaError_t launch_decode(const void *q, const void *k, const void *v, const int *kv_len, void *out, float *lse,
                          int B, int T, int S_max, int H, void *workspace, cudaStream_t stream);

// Document starts lo[b, i] (the first pass of the metadata pre-pass, from seg alone);
// blk_last holds B * ceil(S_pad / 1024) ints of carries.
cudaError_t launch_doc_starts(const int *seg, int B, int S, int S_pad, int *lo, int *blk_last, int *err,
                              cudaStream_t stream);

// Packed-loss re-weighting: workspace layout and the launches.
struct LossLayout {
  int S_pad, n_blk, n_cta;
  size_t off_lo, off_blk, off_docsum, off_part, total;
};
LossLayout loss_layout(int B, int S);
cudaError_t launch_packed_loss(const void *logits, const int *targets, const float *weight, const int *seg,
                               double *loss, void *dlogits, int B, int S, int V, void *workspace, int num_sms,
                               cudaStream_t stream);

}  // namespace lwm

#include "lwm_attn.h"

namespace lwm {

// The bound of the kernels' pipeline waits for the next launches (process-wide,
// lwm_attn_set_wait_limit; WAIT_LIMIT_NS unless a test shortened it). api.cu.
struct WaitBound;
WaitBound wait_bound();

// Host-side argument checks shared by the entry points (api.cu).
lwm_status check_sizes(int B, int S, int H, int D);
// LWM_OK when the current device is one the kernels are built for (sm_103),
// LWM_ERR_UNSUPPORTED when it is not, LWM_ERR_CUDA when it cannot be queried.
lwm_status check_device();

lwm_status fwd_with_forward_workspace(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const int32_t *seg,
                                      const int32_t *pos, lwm_bf16 *out, float *lse, int B, int S, int H, void *ws,
                                      cudaStream_t stream);

}  // namespace lwm
