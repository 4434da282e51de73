// Internal launchers of the attention kernels (host side; not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace lwm {

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

lwm_status fwd_with_forward_workspace(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const int32_t *seg,
                                      const int32_t *pos, lwm_bf16 *out, float *lse, int B, int S, int H, void *ws,
                                      cudaStream_t stream);

}  // namespace lwm
