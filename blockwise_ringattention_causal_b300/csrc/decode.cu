// Decoding: attention of the T newest tokens of each row against its key/value cache
// (the inference side of the 1M-token context of "World Model on Million-Length Video
// And Language With Blockwise RingAttention", deep-dive page, section
// "RingAttention 为什么必要"), split over the cache and merged by log-sum-exp.
//
// Memory-bound: each cache byte is read once, and a token's head vectors carry only
// 2 T FLOPs per byte. Kernel 1 gives every (split of the cache, group of 16 heads,
// batch row) a CTA: one producer thread stages the split's K and V rows into shared
// memory with bulk copies (three stages of 8 tokens x 16 heads x 2 tensors, 192 KB, so
// the SM keeps up to 128 KB of loads in flight), and 16 half-warps, one per head,
// run the online softmax over the staged tokens: lane l of a half-warp owns dims
// 8 l .. 8 l + 7, a score is the sum of the 16 lanes' partial dot products (an xor
// all-reduce for T = 1, 3; a halving reduce-scatter for T = 2, 4, where the shuffles of
// the all-reduce, not HBM, set the pace). Each CTA
// leaves, per (head, query), the running max m, the sum l and the unnormalised output
// of its split. Kernel 2 merges the splits of each (row, head, query):
//   M = max m_s,  L = sum_s l_s 2^(m_s - M),  out = sum_s o_s 2^(m_s - M) / L,
//   lse = (M + log2 L) ln 2   (scores in log2 units).
#include "common.cuh"
#include "kernels.h"

namespace lwm {
namespace {

constexpr int DEC_HEADS = 16;                       // heads per CTA (one per half-warp)
constexpr int DEC_CWARPS = 8;                       // consumer warps
constexpr int DEC_THREADS = (DEC_CWARPS + 1) * 32;  // + producer warp
constexpr int DEC_TB = 8;                           // tokens per stage
constexpr int DEC_NST = 3;                          // stages
constexpr int DEC_TOK_BYTES = DEC_HEADS * HD * 2;   // one token's 16 head vectors: 4 KB
constexpr int DEC_STAGE_BYTES = 2 * DEC_TB * DEC_TOK_BYTES;   // K then V: 64 KB
constexpr int DEC_SM_BAR = DEC_NST * DEC_STAGE_BYTES;

struct DecBars {
  uint64_t full[DEC_NST], empty[DEC_NST];
  uint64_t never;   // the failure test's wait (nothing arrives)
  WaitCtl ctl;
  int fill, seen;
};
constexpr int DEC_SMEM = DEC_SM_BAR + int(sizeof(DecBars)) + 128;
static_assert(DEC_SMEM <= 232448, "shared memory budget of one CTA");

struct DecArgs {
  const uint4 *q;            // [B, T, H, D]
  const __nv_bfloat16 *k, *v;   // [B, S_max, H, D]
  const int *kv_len;         // [B] or null
  float *part_o;             // [B, H, T, n_split, D]
  float2 *part_ml;           // [B, H, T, n_split]
  int *hdr;
  int B, T, S_max, H, n_split, split_len;
  float scale_log2;          // log2(e) / sqrt(D)
  WaitBound wait;
};

__device__ __forceinline__ int row_len(const DecArgs &a, int b, bool &bad) {
  const int len = a.kv_len ? a.kv_len[b] : a.S_max;
  bad = len < a.T || len > a.S_max;
  return bad ? 0 : len;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float *f) {
  const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __bfloat1622float2(p[e]);
    f[2 * e] = x.x;
    f[2 * e + 1] = x.y;
  }
}

template <int T, bool TEST>
__global__ void __launch_bounds__(DEC_THREADS, 1) decode_split_kernel(const __grid_constant__ DecArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  DecBars *bars = reinterpret_cast<DecBars *>(smem + DEC_SM_BAR);
  const int split = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h0 = hg * DEC_HEADS;
  const int nh = min(DEC_HEADS, a.H - h0);
  bool bad;
  const int len = row_len(a, b, bad);
  if (bad && split == 0 && hg == 0 && threadIdx.x == 0) raise_error(a.hdr + HDR_ERR, ERRBIT_LENGTHS);
  const int s0 = split * a.split_len;
  const int s1 = min(s0 + a.split_len, len);
  const int n_steps = s1 > s0 ? (s1 - s0 + DEC_TB - 1) / DEC_TB : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < DEC_NST; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], DEC_CWARPS);
    }
    if (TEST) mbar_init(&bars->never, 1);
    bars->ctl.init(a.wait);
    bars->fill = bars->seen = 0;
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtl *ctl = &bars->ctl;
  bool ok = true;

  if (warp == DEC_CWARPS) {
    // ---- producer: K rows then V rows of up to DEC_TB tokens per stage
    if (lane == 0) {
      const uint32_t row_bytes = uint32_t(nh) * HD * 2;
      int fill = 0;
      for (int st = 0; st < n_steps; ++st) {
        const int slot = st % DEC_NST;
        if (!(ok = mbar_wait(&bars->empty[slot], ((st / DEC_NST) & 1) ^ 1, ctl))) break;
        const int j0 = s0 + st * DEC_TB;
        const int nt = min(DEC_TB, s1 - j0);
        mbar_arrive_expect_tx(&bars->full[slot], 2u * uint32_t(nt) * row_bytes);
        uint8_t *dst = smem + slot * DEC_STAGE_BYTES;
        for (int u = 0; u < nt; ++u) {
          const size_t src = ((size_t(b) * a.S_max + j0 + u) * a.H + h0) * HD;
          bulk_load(dst + u * DEC_TOK_BYTES, a.k + src, row_bytes, &bars->full[slot]);
          bulk_load(dst + (DEC_TB + u) * DEC_TOK_BYTES, a.v + src, row_bytes, &bars->full[slot]);
        }
        ++fill;
        // failure test only: a phase that never completes, with this stage's copies in flight
        if constexpr (TEST) {
          if (st == 0 && !(ok = test_expiry_wait(&bars->never, ctl))) break;
        }
      }
      bars->fill = fill;
    }
    __syncwarp();
  } else {
    // ---- consumers: half-warp hw = head h0 + hw; lane l16 owns dims 8 l16 .. 8 l16 + 7
    if constexpr (T % 2 == 0) {
      // T = 2, 4: the 8 T partial scores of a stage are reduce-scattered over the 16 lanes
      // (halving exchanges: after the xor-8, -4, -2, -1 steps lane l16 holds the complete
      // scores of columns VPL l16 .. VPL l16 + VPL - 1, all of query t_l), 30 shuffles
      // instead of the 4 x 8 T of an all-reduce; each lane takes the softmax of its own
      // scores, and the P.V step fetches every p from its lane by index.
      const int hw = threadIdx.x >> 4, l16 = threadIdx.x & 15;
      const int h = h0 + min(hw, nh - 1);   // half-warps past the last head shadow it and store nothing
      const int hbase = lane & 16;          // first lane of this half-warp
      constexpr int N = 8 * T, VPL = N / 16, LPT = 8 / VPL;
      const int c0 = VPL * l16, t_l = c0 / 8, u_l = c0 % 8;
      float qf[T][8], o[T][8];
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const uint4 u = a.q[((size_t(b) * a.T + t) * a.H + h) * (HD / 8) + l16];
        bf16x8_to_f32(u, qf[t]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          qf[t][e] *= a.scale_log2;
          o[t][e] = 0.f;
        }
      }
      float m_l = -__builtin_huge_valf(), l_l = 0.f;   // query t_l: running max, this lane's share of the sum
      int seen = 0;
      for (int st = 0; st < n_steps; ++st) {
        const int slot = st % DEC_NST;
        if (!(ok = mbar_wait(&bars->full[slot], (st / DEC_NST) & 1, ctl))) break;
        seen = st + 1;
        const uint8_t *stage = smem + slot * DEC_STAGE_BYTES + hw * (HD * 2) + l16 * 16;
        const int j0 = s0 + st * DEC_TB;
        float v[N];
#pragma unroll
        for (int u = 0; u < DEC_TB; ++u) {
          float kf[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4 *>(stage + u * DEC_TOK_BYTES), kf);
#pragma unroll
          for (int t = 0; t < T; ++t) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc = fmaf(qf[t][e], kf[e], acc);
            v[t * 8 + u] = acc;
          }
        }
#pragma unroll
        for (int m = 8, n = N / 2; m >= 1; m >>= 1, n >>= 1) {
          const bool upper = (l16 & m) != 0;   // keeps the upper half of the remaining columns
#pragma unroll
          for (int i = 0; i < n; ++i) {
            const float send = upper ? v[i] : v[i + n];
            const float keep = upper ? v[i + n] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
        }
        // mask: keys past the split's end, or after the query's position len - T + t
        float mx = -__builtin_huge_valf();
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int j = j0 + u_l + i;
          if (j >= s1 || j > len - T + t_l) v[i] = -__builtin_huge_valf();
          mx = fmaxf(mx, v[i]);
        }
#pragma unroll
        for (int d = 1; d < LPT; d <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
        const float m_new = fmaxf(m_l, mx);
        const float m_use = m_new == -__builtin_huge_valf() ? 0.f : m_new;
        const float alpha = ex2_approx(m_l - m_use);   // 0 while nothing was visible
        m_l = m_new;
        float pl[VPL], psum = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          pl[i] = ex2_approx(v[i] - m_use);
          psum += pl[i];
        }
        l_l = l_l * alpha + psum;
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const float al = __shfl_sync(0xffffffffu, alpha, hbase + t * LPT);
#pragma unroll
          for (int e = 0; e < 8; ++e) o[t][e] *= al;
        }
#pragma unroll
        for (int u = 0; u < DEC_TB; ++u) {
          // slots past a partial last stage hold stale bytes (possibly NaN patterns): skip
          // them rather than multiply them by p = 0 (j0 and s1 are the same for the whole CTA)
          if (j0 + u >= s1) continue;
          float vf[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4 *>(stage + (DEC_TB + u) * DEC_TOK_BYTES), vf);
#pragma unroll
          for (int t = 0; t < T; ++t) {
            const int c = t * 8 + u;
            const float pc = __shfl_sync(0xffffffffu, pl[c % VPL], hbase + c / VPL);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[t][e] = fmaf(pc, vf[e], o[t][e]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->empty[slot]);
      }
      if (warp == 0 && lane == 0) bars->seen = seen;
#pragma unroll
      for (int d = 1; d < LPT; d <<= 1) l_l += __shfl_xor_sync(0xffffffffu, l_l, d);
      if (ok && hw < nh) {
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const size_t pi = ((size_t(b) * a.H + h) * a.T + t) * a.n_split + split;
          float4 *dst = reinterpret_cast<float4 *>(a.part_o + pi * HD + 8 * l16);
          dst[0] = make_float4(o[t][0], o[t][1], o[t][2], o[t][3]);
          dst[1] = make_float4(o[t][4], o[t][5], o[t][6], o[t][7]);
        }
        if (u_l == 0) a.part_ml[((size_t(b) * a.H + h) * a.T + t_l) * a.n_split + split] = make_float2(m_l, l_l);
      }
    } else {
      const int hw = threadIdx.x >> 4, l16 = threadIdx.x & 15;
      const int h = h0 + min(hw, nh - 1);   // half-warps past the last head shadow it and store nothing
      float qf[T][8], o[T][8], m[T], l[T];
  #pragma unroll
      for (int t = 0; t < T; ++t) {
        const uint4 u = a.q[((size_t(b) * a.T + t) * a.H + h) * (HD / 8) + l16];
        bf16x8_to_f32(u, qf[t]);
  #pragma unroll
        for (int e = 0; e < 8; ++e) {
          qf[t][e] *= a.scale_log2;
          o[t][e] = 0.f;
        }
        m[t] = -__builtin_huge_valf();
        l[t] = 0.f;
      }
      int seen = 0;
      for (int st = 0; st < n_steps; ++st) {
        const int slot = st % DEC_NST;
        if (!(ok = mbar_wait(&bars->full[slot], (st / DEC_NST) & 1, ctl))) break;
        seen = st + 1;
        const uint8_t *stage = smem + slot * DEC_STAGE_BYTES + hw * (HD * 2) + l16 * 16;
        const int j0 = s0 + st * DEC_TB;
        float s[T][DEC_TB];
  #pragma unroll
        for (int u = 0; u < DEC_TB; ++u) {
          float kf[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4 *>(stage + u * DEC_TOK_BYTES), kf);
  #pragma unroll
          for (int t = 0; t < T; ++t) {
            float acc = 0.f;
  #pragma unroll
            for (int e = 0; e < 8; ++e) acc = fmaf(qf[t][e], kf[e], acc);
            s[t][u] = acc;
          }
        }
  #pragma unroll
        for (int u = 0; u < DEC_TB; ++u)
  #pragma unroll
          for (int t = 0; t < T; ++t) {
            float x = s[t][u];
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            x += __shfl_xor_sync(0xffffffffu, x, 2);
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            // query t sits at position len - T + t and sees keys up to it; keys past the
            // split's end (a partial last stage) are not there
            const int j = j0 + u;
            s[t][u] = (j < s1 && j <= len - T + t) ? x : -__builtin_huge_valf();
          }
        float p[T][DEC_TB];
  #pragma unroll
        for (int t = 0; t < T; ++t) {
          float mx = s[t][0];
  #pragma unroll
          for (int u = 1; u < DEC_TB; ++u) mx = fmaxf(mx, s[t][u]);
          const float m_new = fmaxf(m[t], mx);
          const float m_use = m_new == -__builtin_huge_valf() ? 0.f : m_new;
          const float alpha = ex2_approx(m[t] - m_use);   // 0 while nothing was visible
          float sum = 0.f;
  #pragma unroll
          for (int u = 0; u < DEC_TB; ++u) {
            p[t][u] = ex2_approx(s[t][u] - m_use);
            sum += p[t][u];
          }
          l[t] = l[t] * alpha + sum;
          m[t] = m_new;
  #pragma unroll
          for (int e = 0; e < 8; ++e) o[t][e] *= alpha;
        }
  #pragma unroll
        for (int u = 0; u < DEC_TB; ++u) {
          // slots past a partial last stage hold stale bytes (possibly NaN patterns): skip
          // them rather than multiply them by p = 0
          if (j0 + u >= s1) continue;
          float vf[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4 *>(stage + (DEC_TB + u) * DEC_TOK_BYTES), vf);
  #pragma unroll
          for (int t = 0; t < T; ++t)
  #pragma unroll
            for (int e = 0; e < 8; ++e) o[t][e] = fmaf(p[t][u], vf[e], o[t][e]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->empty[slot]);
      }
      if (warp == 0 && lane == 0) bars->seen = seen;
      if (ok && hw < nh) {
  #pragma unroll
        for (int t = 0; t < T; ++t) {
          const size_t pi = ((size_t(b) * a.H + h) * a.T + t) * a.n_split + split;
          float4 *dst = reinterpret_cast<float4 *>(a.part_o + pi * HD + 8 * l16);
          dst[0] = make_float4(o[t][0], o[t][1], o[t][2], o[t][3]);
          dst[1] = make_float4(o[t][4], o[t][5], o[t][6], o[t][7]);
          if (l16 == 0) a.part_ml[pi] = make_float2(m[t], l[t]);
        }
      }
    }
  }

  if (!ok) {
    bars->ctl.abort = 1;
    raise_error(a.hdr + HDR_ERR, ERRBIT_TIMEOUT);
  }
  __syncthreads();
  if (bars->ctl.abort && threadIdx.x == DEC_CWARPS * 32) {
    // copies no consumer has observed must land before the CTA's shared memory goes away
    for (int k = bars->seen; k < bars->fill; ++k) bounded_wait_plain(&bars->full[k % DEC_NST], (k / DEC_NST) & 1);
  }
  __syncthreads();
}

// One warp per (row, head, query): merges the splits that hold any key of the row.
__global__ void __launch_bounds__(256) decode_merge_kernel(const __grid_constant__ DecArgs a, __nv_bfloat16 *out,
                                                           float *lse) {
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wid >= (long long)a.B * a.H * a.T) return;
  const int t = int(wid % a.T);
  const int h = int((wid / a.T) % a.H);
  const int b = int(wid / ((long long)a.T * a.H));
  bool bad;
  const int len = row_len(a, b, bad);
  const int n_used = (len + a.split_len - 1) / a.split_len;
  const size_t p0 = ((size_t(b) * a.H + h) * a.T + t) * a.n_split;
  float M = -__builtin_huge_valf();
  for (int s = lane; s < n_used; s += 32) M = fmaxf(M, a.part_ml[p0 + s].x);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, d));
  __nv_bfloat16 *dst = out + ((size_t(b) * a.T + t) * a.H + h) * HD + 4 * lane;
  float *lse_dst = lse + (size_t(b) * a.H + h) * a.T + t;
  if (M == -__builtin_huge_valf()) {
    reinterpret_cast<uint2 *>(dst)[0] = make_uint2(0, 0);
    if (lane == 0) *lse_dst = -__builtin_huge_valf();
    return;
  }
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < n_used; ++s) {
    const float2 ml = a.part_ml[p0 + s];
    const float w = ex2_approx(ml.x - M);   // 0 for an empty split (m = -inf)
    L = fmaf(ml.y, w, L);
    const float4 v = reinterpret_cast<const float4 *>(a.part_o + (p0 + s) * HD)[lane];
    acc.x = fmaf(v.x, w, acc.x);
    acc.y = fmaf(v.y, w, acc.y);
    acc.z = fmaf(v.z, w, acc.z);
    acc.w = fmaf(v.w, w, acc.w);
  }
  const float inv = 1.f / L;
  reinterpret_cast<uint2 *>(dst)[0] = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (lane == 0) *lse_dst = (M + __log2f(L)) * 0.69314718055994531f;
}

}  // namespace

DecodeLayout decode_layout(int B, int T, int S_max, int H) {
  DecodeLayout d;
  int want = (S_max + 511) / 512;   // about 512 splits of a long cache
  int sl = 256;
  while (sl < want && sl < 4096) sl <<= 1;
  d.split_len = sl;
  d.n_split = (S_max + sl - 1) / sl;
  size_t o = Workspace::align256(HDR_WORDS * 4);
  d.off_ml = o;
  o += Workspace::align256(size_t(B) * H * T * d.n_split * sizeof(float2));
  d.off_o = o;
  o += Workspace::align256(size_t(B) * H * T * d.n_split * HD * sizeof(float));
  d.total = o;
  return d;
}

cudaError_t launch_decode(const void *q, const void *k, const void *v, const int *kv_len, void *out, float *lse,
                          int B, int T, int S_max, int H, void *workspace, cudaStream_t stream) {
  const DecodeLayout d = decode_layout(B, T, S_max, H);
  char *base = static_cast<char *>(workspace);
  DecArgs a;
  a.q = static_cast<const uint4 *>(q);
  a.k = static_cast<const __nv_bfloat16 *>(k);
  a.v = static_cast<const __nv_bfloat16 *>(v);
  a.kv_len = kv_len;
  a.part_ml = reinterpret_cast<float2 *>(base + d.off_ml);
  a.part_o = reinterpret_cast<float *>(base + d.off_o);
  a.hdr = reinterpret_cast<int *>(base);
  a.B = B;
  a.T = T;
  a.S_max = S_max;
  a.H = H;
  a.n_split = d.n_split;
  a.split_len = d.split_len;
  a.scale_log2 = 1.4426950408889634f / sqrtf(float(HD));
  a.wait = wait_bound();
  const dim3 grid(d.n_split, (H + DEC_HEADS - 1) / DEC_HEADS, B);
  cudaError_t e = cudaSuccess;
  switch (T) {
#define LWM_DECODE_CASE(TT)                                                                                     \
  case TT: {                                                                                                    \
    static std::atomic<uint64_t> attr_done[2] = {{0}, {0}};                                                     \
    const void *kern = a.wait.test ? reinterpret_cast<const void *>(decode_split_kernel<TT, true>)              \
                                   : reinterpret_cast<const void *>(decode_split_kernel<TT, false>);            \
    e = smem_attr_once(kern, DEC_SMEM, attr_done[a.wait.test ? 1 : 0]);                                         \
    if (e != cudaSuccess) return e;                                                                             \
    if (a.wait.test) decode_split_kernel<TT, true><<<grid, DEC_THREADS, DEC_SMEM, stream>>>(a);                 \
    else decode_split_kernel<TT, false><<<grid, DEC_THREADS, DEC_SMEM, stream>>>(a);                            \
    break;                                                                                                      \
  }
    LWM_DECODE_CASE(1)
    LWM_DECODE_CASE(2)
    LWM_DECODE_CASE(3)
    LWM_DECODE_CASE(4)
#undef LWM_DECODE_CASE
    default:
      return cudaErrorInvalidValue;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long warps = (long long)B * H * T;
  decode_merge_kernel<<<int((warps + 7) / 8), 256, 0, stream>>>(a, static_cast<__nv_bfloat16 *>(out), lse);
  return cudaGetLastError();
}

}  // namespace lwm
