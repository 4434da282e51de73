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

cudaError_t launch_dq(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                      const CUtensorMap &tdo, void *dq, const Problem &p, void *workspace,
                      cudaStream_t stream);

}  // namespace lwm
