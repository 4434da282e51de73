// Backward pass kernels.
//
// Gradients of exact softmax attention recomputed block by block from the saved
// log-sum-exp (the blockwise method of the LWM pages: "World Model on Million-Length
// Video And Language With Blockwise RingAttention", deep-dive page, section
// "RingAttention 为什么必要"; the backward pass re-circulates the same blocks):
//   delta_i = dout_i . out_i                       (row-dot pre-pass, this file)
//   p_ij    = exp(s_ij - lse_i),  dp_ij = dout_i . v_j
//   ds_ij   = p_ij (dp_ij - delta_i)
//   dv_j    = sum_i p_ij dout_i,  dk_j = sum_i ds_ij q_i / sqrt(D),  dq_i = sum_j ds_ij k_j / sqrt(D)
#include "common.cuh"
#include "kernels.h"

namespace lwm {
namespace {

constexpr int DELTA_THREADS = 256;

// delta[b,h,i] = sum_d dout[b,i,h,d] * out[b,i,h,d] (fp32), and lse2[b,h,i] =
// lse * log2(e) on a row stride padded to a multiple of 128, with +inf for rows that
// see no key (padding) and for the pad tail, so that exp2(s - lse2) is 0 there.
// One warp handles 32 consecutive rows of one head: two rows per load step, 16 lanes
// per 256-byte row, fully coalesced; the 32 results are written as one 128-byte line.
__global__ void __launch_bounds__(DELTA_THREADS) delta_kernel(const uint4 *__restrict__ out,
                                                              const uint4 *__restrict__ dout,
                                                              const float *__restrict__ lse,
                                                              float *__restrict__ delta, float *__restrict__ lse2,
                                                              int B, int S, int H, int S_pad) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (DELTA_THREADS / 32);
  const int nI = (S_pad + 31) / 32;
  const long long tasks = (long long)B * nI * H;
  for (long long t = (long long)blockIdx.x * (DELTA_THREADS / 32) + (threadIdx.x >> 5); t < tasks; t += warps) {
    const int h = int(t % H);
    const int ib = int((t / H) % nI);
    const int b = int(t / ((long long)H * nI));
    const int i0 = ib * 32;
    float mine = 0.f;
#pragma unroll 4
    for (int r = 0; r < 32; r += 2) {
      const int row = i0 + r + (lane >> 4);
      float acc = 0.f;
      if (row < S) {
        const size_t idx = ((size_t(b) * S + row) * H + h) * (HD / 8) + (lane & 15);
        const uint4 a = __ldg(out + idx), d = __ldg(dout + idx);
        const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
        const __nv_bfloat162 *pd = reinterpret_cast<const __nv_bfloat162 *>(&d);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = __bfloat1622float2(pa[e]), fd = __bfloat1622float2(pd[e]);
          acc = fmaf(fa.x, fd.x, acc);
          acc = fmaf(fa.y, fd.y, acc);
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 8);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      const float v0 = __shfl_sync(0xffffffffu, acc, 0), v1 = __shfl_sync(0xffffffffu, acc, 16);
      if (lane == r) mine = v0;
      if (lane == r + 1) mine = v1;
    }
    const int i = i0 + lane;
    const size_t o = (size_t(b) * H + h) * S_pad + i;
    if (i < S_pad) {
      float l2 = __int_as_float(0x7f800000);
      if (i < S) {
        const float L = lse[(size_t(b) * H + h) * S + i];
        if (L != -__int_as_float(0x7f800000)) l2 = L * 1.4426950408889634f;
      }
      delta[o] = mine;
      lse2[o] = l2;
    }
  }
}

}  // namespace

cudaError_t launch_delta(const void *out, const void *dout, const float *lse, const Problem &p, void *workspace,
                         cudaStream_t stream) {
  const Workspace w = Workspace::layout(p.B, p.S, p.H);
  char *base = static_cast<char *>(workspace);
  float *delta = reinterpret_cast<float *>(base + w.off_delta);
  float *lse2 = reinterpret_cast<float *>(base + w.off_lse2);
  const int S_pad = w.nT * BM;
  const long long tasks = (long long)p.B * ((S_pad + 31) / 32) * p.H;
  long long blocks = (tasks + DELTA_THREADS / 32 - 1) / (DELTA_THREADS / 32);
  const long long cap = (long long)p.num_sms * 8;
  if (blocks > cap) blocks = cap;
  delta_kernel<<<int(blocks), DELTA_THREADS, 0, stream>>>(static_cast<const uint4 *>(out),
                                                           static_cast<const uint4 *>(dout), lse, delta, lse2, p.B,
                                                           p.S, p.H, S_pad);
  return cudaGetLastError();
}

cudaError_t launch_dkdv(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                        void *, void *, const Problem &, void *, cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t launch_dq(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, void *,
                      const Problem &, void *, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace lwm
