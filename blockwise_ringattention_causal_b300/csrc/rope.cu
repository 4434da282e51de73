// Rotary position embedding (RoPE) of q and k, and its inverse for the gradients.
//
// LWM raises RoPE's base theta as the context grows ("World Model on Million-Length
// Video And Language With Blockwise RingAttention", deep-dive page, section
// "Stage I：长上下文语言模型", Tables 11 and 13: theta = 1M at 32K tokens up to 50M at
// 1M). RoPE rotates each adjacent pair (2m, 2m+1) of a head vector of the token at
// position p by the angle p * theta^(-2m/D); the inverse rotates by the negative angle
// (the transpose, which maps gradients with respect to the rotated q, k back to the
// unrotated ones).
//
// Memory-bound: each element is read once and written once. A CTA takes a block of
// tokens: first the (cos, sin) of every (token, pair) -- the angle is formed and
// reduced to [-pi, pi] in fp64 (at theta^0 and p up to 2^20 the angle is 1e6 rad, far
// beyond what an fp32 angle resolves), then sin/cos in fp32 -- into shared memory;
// then every head of q and of k of those tokens is rotated with that table, 16-byte
// vectors, several loads in flight per thread.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace lwm {
namespace {

constexpr int ROPE_THREADS = 256;
constexpr int ROPE_TOKENS = 8;        // tokens per CTA step
constexpr int NPAIR = HD / 2;         // 64 pairs per head vector
constexpr int ROPE_BATCH = 4;         // 16-byte vectors loaded before any is stored

struct RopeArgs {
  const uint4 *x0, *x1;   // q, k (either may be null)
  uint4 *y0, *y1;
  const int *pos;         // [B, S] or null (position = index in the row)
  double inv_freq[NPAIR]; // theta^(-2m/D)
  long long ntok;         // B * S
  int S, H;
  float sign;             // +1 rotate, -1 inverse rotation
};

__device__ __forceinline__ uint32_t rot_pair(uint32_t w, float c, float s) {
  const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&w);
  const float2 f = __bfloat1622float2(v);
  return pack_bf16x2(fmaf(f.x, c, -f.y * s), fmaf(f.x, s, f.y * c));
}

__device__ __forceinline__ uint4 rot_vec(uint4 u, const float4 &cs01, const float4 &cs23) {
  uint4 r;
  r.x = rot_pair(u.x, cs01.x, cs01.y);
  r.y = rot_pair(u.y, cs01.z, cs01.w);
  r.z = rot_pair(u.z, cs23.x, cs23.y);
  r.w = rot_pair(u.w, cs23.z, cs23.w);
  return r;
}

__global__ void __launch_bounds__(ROPE_THREADS, 4) rope_kernel(const __grid_constant__ RopeArgs a) {
  __shared__ __align__(16) float2 cs[ROPE_TOKENS][NPAIR];   // (cos, sign * sin)
  constexpr double TWO_PI = 6.283185307179586476925286766559;
  constexpr double INV_TWO_PI = 0.15915494309189533576888376337251;
  const int vec_per_tok = a.H * (HD / 8);   // 16-byte vectors per token and tensor
  for (long long t0 = (long long)blockIdx.x * ROPE_TOKENS; t0 < a.ntok; t0 += (long long)gridDim.x * ROPE_TOKENS) {
    const int nt = int(min((long long)ROPE_TOKENS, a.ntok - t0));
    __syncthreads();   // the previous step is done with the table
    for (int e = threadIdx.x; e < nt * NPAIR; e += ROPE_THREADS) {
      const int tt = e / NPAIR, m = e % NPAIR;
      const long long tok = t0 + tt;
      const int p = a.pos ? a.pos[tok] : int(tok % a.S);
      const double ang = double(p) * a.inv_freq[m];
      const double r = ang - rint(ang * INV_TWO_PI) * TWO_PI;
      float s, c;
      sincosf(float(r), &s, &c);
      cs[tt][m] = make_float2(c, a.sign * s);
    }
    __syncthreads();
    const int n = nt * vec_per_tok;
    const size_t base = size_t(t0) * vec_per_tok;
    for (int e0 = threadIdx.x; e0 < n; e0 += ROPE_THREADS * ROPE_BATCH) {
      uint4 u0[ROPE_BATCH], u1[ROPE_BATCH];
#pragma unroll
      for (int r = 0; r < ROPE_BATCH; ++r) {
        const int e = e0 + r * ROPE_THREADS;
        if (e < n) {
          if (a.x0) u0[r] = a.x0[base + e];   // plain loads: y may alias x (in place)
          if (a.x1) u1[r] = a.x1[base + e];
        }
      }
#pragma unroll
      for (int r = 0; r < ROPE_BATCH; ++r) {
        const int e = e0 + r * ROPE_THREADS;
        if (e < n) {
          const int tt = e / vec_per_tok;
          const int v16 = (e % vec_per_tok) & 15;   // dims 8 v16 .. 8 v16 + 7: pairs 4 v16 .. 4 v16 + 3
          const float4 *t = reinterpret_cast<const float4 *>(&cs[tt][4 * v16]);
          const float4 cs01 = t[0], cs23 = t[1];
          if (a.x0) a.y0[base + e] = rot_vec(u0[r], cs01, cs23);
          if (a.x1) a.y1[base + e] = rot_vec(u1[r], cs01, cs23);
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_rope(const void *x0, const void *x1, const int *pos, double theta, void *y0, void *y1, int B,
                        int S, int H, bool inverse, int num_sms, cudaStream_t stream) {
  RopeArgs a;
  a.x0 = static_cast<const uint4 *>(x0);
  a.x1 = static_cast<const uint4 *>(x1);
  a.y0 = static_cast<uint4 *>(y0);
  a.y1 = static_cast<uint4 *>(y1);
  a.pos = pos;
  for (int m = 0; m < NPAIR; ++m) a.inv_freq[m] = std::pow(theta, -2.0 * m / HD);
  a.ntok = (long long)B * S;
  a.S = S;
  a.H = H;
  a.sign = inverse ? -1.f : 1.f;
  const long long steps = (a.ntok + ROPE_TOKENS - 1) / ROPE_TOKENS;
  const long long cap = (long long)num_sms * 4;   // 4 resident CTAs of 256 threads per SM
  const int grid = int(steps < cap ? steps : cap);
  rope_kernel<<<grid, ROPE_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace lwm
