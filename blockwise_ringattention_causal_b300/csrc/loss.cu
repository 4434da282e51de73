// Packed-loss re-weighting: cross-entropy over the vocabulary with per-document
// weights, so that a packed batch trains like the same documents non-packed, one per
// padded row ("World Model on Million-Length Video And Language With Blockwise
// RingAttention", deep-dive page, section "Masked sequence packing": the loss is
// re-weighted to be equivalent to non-packed + padding training, because in a packed
// row the token count of long video samples would drown short answers).
//
// Each document's weighted mean token loss counts once:
//   loss = (1/N) sum_d sum_{t in d} w_t l_t / n_d,   n_d = sum_{t in d} w_t,
//   N = documents with n_d > 0,   l_t = logsumexp(z_t) - z_t[y_t],
//   dloss/dz_t = w_t / (N n_d) (softmax(z_t) - onehot(y_t)).
//
// Kernels (all memory-bound): document starts from seg (the metadata pre-pass's first
// pass), per-document weight sums (fp64; one atomic per document and CTA), the count
// N, then the rows: for vocabularies up to 48K, one CTA per row with the row staged
// once in shared memory by a bulk copy (an online max / sum pass and the gradient pass
// both read it there); beyond that, one warp per row reading the logits twice. The loss
// is summed per CTA and the CTA sums in a fixed order: deterministic for a given input.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace lwm {
namespace {

constexpr int LOSS_THREADS = 1024;
constexpr int CE_WARPS = 8;
constexpr int CE_UNROLL = 4;
constexpr int LHDR_NDOCS = 16;   // header word: number of documents with any weight

__device__ __forceinline__ float token_weight(const int *seg, const float *weight, size_t i) {
  if (seg && seg[i] < 0) return 0.f;
  const float w = weight ? weight[i] : 1.f;
  return (w > 0.f && w < __int_as_float(0x7f800000)) ? w : 0.f;   // negative / NaN / inf: no loss
}

// Sum of the weights of each document, at the slot of its first token. lo is
// non-decreasing, so a block whose first and last token share lo holds one document.
__global__ void __launch_bounds__(LOSS_THREADS) docsum_kernel(const int *__restrict__ seg,
                                                              const float *__restrict__ weight,
                                                              const int *__restrict__ lo, double *__restrict__ doc_sum,
                                                              int S, int S_pad) {
  __shared__ double red[LOSS_THREADS / 32];
  const int b = blockIdx.y;
  const int i0 = blockIdx.x * LOSS_THREADS;
  const int i = i0 + threadIdx.x;
  const int last = min(i0 + LOSS_THREADS, S) - 1;
  const int *lr = lo + size_t(b) * S_pad;
  const double w = i < S ? double(token_weight(seg, weight, size_t(b) * S + i)) : 0.0;
  const int key = i < S ? lr[i] : -1;
  const bool uniform = lr[i0] == lr[last] && lr[i0] <= i0;   // one document (not padding: lo = i + 1)
  if (uniform) {
    double v = w;
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
      for (int k = 0; k < LOSS_THREADS / 32; ++k) t += red[k];
      if (t != 0.0) atomicAdd(doc_sum + size_t(b) * S_pad + lr[i0], t);
    }
    return;
  }
  // several documents: per warp when the warp's tokens share one, else per token
  const int k0 = __shfl_sync(0xffffffffu, key, 0);
  if (__all_sync(0xffffffffu, key == k0)) {
    double v = w;
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    if ((threadIdx.x & 31) == 0 && v != 0.0 && k0 >= 0 && k0 < S) atomicAdd(doc_sum + size_t(b) * S_pad + k0, v);
  } else if (w != 0.0 && key >= 0 && key < S) {
    atomicAdd(doc_sum + size_t(b) * S_pad + key, w);
  }
}

// N: documents (first token: lo[i] == i, not padding) with a positive weight sum.
__global__ void __launch_bounds__(LOSS_THREADS) ndocs_kernel(const int *__restrict__ lo,
                                                             const double *__restrict__ doc_sum, int S, int S_pad,
                                                             int *__restrict__ ndocs) {
  __shared__ int red[LOSS_THREADS / 32];
  const int b = blockIdx.y;
  const int i = blockIdx.x * LOSS_THREADS + threadIdx.x;
  const size_t o = size_t(b) * S_pad + i;
  int c = (i < S && lo[o] == i && doc_sum[o] > 0.0) ? 1 : 0;
  for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(0xffffffffu, c, d);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int k = 0; k < LOSS_THREADS / 32; ++k) t += red[k];
    if (t) atomicAdd(ndocs, t);
  }
}

struct CeArgs {
  const uint4 *logits;       // [B * S, V] bf16, V / 8 vectors per row
  const __nv_bfloat16 *logits_e;
  const int *targets, *seg;
  const float *weight;
  const int *lo;
  const double *doc_sum;
  const int *ndocs;
  uint4 *dlogits;            // or null
  double *part;              // one loss term per CTA
  int *err;
  int B, S, S_pad, V;
  WaitBound wait;
};

__device__ __forceinline__ void bf16x8(const uint4 &u, float *f) {
  const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __bfloat1622float2(p[e]);
    f[2 * e] = x.x;
    f[2 * e + 1] = x.y;
  }
}

__global__ void __launch_bounds__(CE_WARPS * 32) ce_kernel(const __grid_constant__ CeArgs a) {
  __shared__ double red[CE_WARPS];
  constexpr float LOG2E = 1.4426950408889634f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * CE_WARPS + warp;
  const long long N = (long long)a.B * a.S;
  double contrib = 0.0;
  if (row < N) {
    const int b = int(row / a.S), t = int(row % a.S);
    const int nv = a.V / 8;
    const uint4 *zr = a.logits + size_t(row) * nv;
    uint4 *gr = a.dlogits ? a.dlogits + size_t(row) * nv : nullptr;
    double wp = 0.0;
    const float w = token_weight(a.seg, a.weight, size_t(row));
    const int y = a.targets[row];
    if (w > 0.f) {
      const double nd = a.doc_sum[size_t(b) * a.S_pad + a.lo[size_t(b) * a.S_pad + t]];
      const int nds = *a.ndocs;
      if (y < 0 || y >= a.V) {
        if (lane == 0) raise_error(a.err, ERRBIT_TARGETS);
      } else if (nd > 0.0 && nds > 0) {
        wp = double(w) / (nd * double(nds));
      }
    }
    if (wp == 0.0) {
      if (gr)
        for (int v = lane; v < nv; v += 32) gr[v] = make_uint4(0, 0, 0, 0);
    } else {
      // pass 1: running max and sum of 2^(z log2 e), per lane, then across the warp
      float m = -__builtin_huge_valf(), s = 0.f;
      for (int v0 = lane; v0 < nv; v0 += 32 * CE_UNROLL) {
        uint4 u[CE_UNROLL];
#pragma unroll
        for (int r = 0; r < CE_UNROLL; ++r)
          if (v0 + 32 * r < nv) u[r] = zr[v0 + 32 * r];
#pragma unroll
        for (int r = 0; r < CE_UNROLL; ++r) {
          if (v0 + 32 * r >= nv) break;
          float f[8];
          bf16x8(u[r], f);
          float mx = f[0];
#pragma unroll
          for (int e = 1; e < 8; ++e) mx = fmaxf(mx, f[e]);
          mx *= LOG2E;
          if (mx > m) {
            s *= ex2_approx(m - mx);
            m = mx;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) s += ex2_approx(fmaf(f[e], LOG2E, -m));
        }
      }
      float M = m;
      for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, d));
      s = (m == -__builtin_huge_valf()) ? 0.f : s * ex2_approx(m - M);
      for (int d = 16; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
      const float lse2 = M + __log2f(s);   // log2 units
      const float zy = __bfloat162float(a.logits_e[size_t(row) * a.V + y]);
      contrib = wp * (double(lse2) * 0.6931471805599453 - double(zy));
      if (gr) {
        // pass 2: dloss/dz = wp (softmax - onehot)
        const float g = float(wp);
        for (int v0 = lane; v0 < nv; v0 += 32 * CE_UNROLL) {
          uint4 u[CE_UNROLL];
#pragma unroll
          for (int r = 0; r < CE_UNROLL; ++r)
            if (v0 + 32 * r < nv) u[r] = zr[v0 + 32 * r];
#pragma unroll
          for (int r = 0; r < CE_UNROLL; ++r) {
            const int v = v0 + 32 * r;
            if (v >= nv) break;
            float f[8];
            bf16x8(u[r], f);
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              float p0 = ex2_approx(fmaf(f[e], LOG2E, -lse2));
              float p1 = ex2_approx(fmaf(f[e + 1], LOG2E, -lse2));
              if (8 * v + e == y) p0 -= 1.f;
              if (8 * v + e + 1 == y) p1 -= 1.f;
              o[e / 2] = pack_bf16x2(g * p0, g * p1);
            }
            gr[v] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    }
  }
  if (lane == 0) red[warp] = contrib;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tsum = 0.0;
    for (int k = 0; k < CE_WARPS; ++k) tsum += red[k];
    a.part[blockIdx.x] = tsum;
  }
}

// One CTA per token row (persistent over rows r = blockIdx.x + k gridDim.x), for
// vocabularies whose row fits shared memory: the row is bulk-copied once, then the max /
// sum pass and the gradient pass both read it from shared memory, so HBM sees each logit
// read once (the warp-per-row kernel above re-reads its row, from HBM once the rows in
// flight outgrow L2).
constexpr int CE_ROW_THREADS = 256;
constexpr int CE_ROW_MAX_BYTES = 96 * 1024;   // at least two CTAs per SM

__device__ __forceinline__ float block_sum_256(float v, float *red) {
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int k = 0; k < CE_ROW_THREADS / 32; ++k) t += red[k];
  __syncthreads();
  return t;
}

__device__ __forceinline__ float block_max_256(float v, float *red) {
  for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = red[0];
#pragma unroll
  for (int k = 1; k < CE_ROW_THREADS / 32; ++k) t = fmaxf(t, red[k]);
  __syncthreads();
  return t;
}

__global__ void __launch_bounds__(CE_ROW_THREADS, 3) ce_row_kernel(const __grid_constant__ CeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint4 *row = reinterpret_cast<uint4 *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  __shared__ uint64_t full;
  __shared__ WaitCtl ctl;
  __shared__ float red[CE_ROW_THREADS / 32];
  __shared__ double wp_s;
  __shared__ bool ok_s;
  constexpr float LOG2E = 1.4426950408889634f;
  const long long N = (long long)a.B * a.S;
  const int nv = a.V / 8;
  if (threadIdx.x == 0) {
    mbar_init(&full, 1);
    ctl.init(a.wait);
    fence_mbar_init();
  }
  __syncthreads();
  double contrib = 0.0;   // thread 0's running sum of this CTA's rows
  uint32_t phase = 0;
  bool ok = true;
  for (long long r = blockIdx.x; r < N; r += gridDim.x) {
    if (threadIdx.x == 0) {
      const int b = int(r / a.S), t = int(r % a.S);
      double wp = 0.0;
      const float w = token_weight(a.seg, a.weight, size_t(r));
      if (w > 0.f) {
        const int y = a.targets[r];
        const double nd = a.doc_sum[size_t(b) * a.S_pad + a.lo[size_t(b) * a.S_pad + t]];
        const int nds = *a.ndocs;
        if (y < 0 || y >= a.V) raise_error(a.err, ERRBIT_TARGETS);
        else if (nd > 0.0 && nds > 0) wp = double(w) / (nd * double(nds));
      }
      wp_s = wp;
      if (wp != 0.0) {
        mbar_arrive_expect_tx(&full, uint32_t(a.V) * 2u);
        bulk_load(row, a.logits + size_t(r) * nv, uint32_t(a.V) * 2u, &full);
      }
    }
    __syncthreads();
    const double wp = wp_s;
    uint4 *gr = a.dlogits ? a.dlogits + size_t(r) * nv : nullptr;
    if (wp == 0.0) {
      if (gr)
        for (int v = threadIdx.x; v < nv; v += CE_ROW_THREADS) gr[v] = make_uint4(0, 0, 0, 0);
      __syncthreads();
      continue;
    }
    // thread 0 waits for the row (and, if the wait ran out, lets the copy land before the
    // CTA leaves); the block barrier then orders the row before every thread's reads
    if (threadIdx.x == 0) {
      ok_s = mbar_wait(&full, phase, &ctl);
      if (!ok_s) bounded_wait_plain(&full, phase);
    }
    __syncthreads();
    if (!(ok = ok_s)) break;
    phase ^= 1;
    float m = -__builtin_huge_valf(), sum = 0.f;
    for (int v = threadIdx.x; v < nv; v += CE_ROW_THREADS) {
      float f[8];
      bf16x8(row[v], f);
      float mx = f[0];
#pragma unroll
      for (int e = 1; e < 8; ++e) mx = fmaxf(mx, f[e]);
      mx *= LOG2E;
      if (mx > m) {
        sum *= ex2_approx(m - mx);
        m = mx;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += ex2_approx(fmaf(f[e], LOG2E, -m));
    }
    const float M = block_max_256(m, red);
    const float tot = block_sum_256(m == -__builtin_huge_valf() ? 0.f : sum * ex2_approx(m - M), red);
    const float lse2 = M + __log2f(tot);
    const int y = a.targets[r];
    if (threadIdx.x == 0) {
      const float zy = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(row)[y]);
      contrib += wp * (double(lse2) * 0.6931471805599453 - double(zy));
    }
    if (gr) {
      const float g = float(wp);
      for (int v = threadIdx.x; v < nv; v += CE_ROW_THREADS) {
        float f[8];
        bf16x8(row[v], f);
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          float p0 = ex2_approx(fmaf(f[e], LOG2E, -lse2));
          float p1 = ex2_approx(fmaf(f[e + 1], LOG2E, -lse2));
          if (8 * v + e == y) p0 -= 1.f;
          if (8 * v + e + 1 == y) p1 -= 1.f;
          o[e / 2] = pack_bf16x2(g * p0, g * p1);
        }
        gr[v] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    __syncthreads();   // the row buffer is reused by the next row's copy
  }
  if (!ok && threadIdx.x == 0) raise_error(a.err, ERRBIT_TIMEOUT);
  if (threadIdx.x == 0) a.part[blockIdx.x] = contrib;
}

// The loss: the CTAs' terms summed in a fixed order.
__global__ void __launch_bounds__(LOSS_THREADS) loss_sum_kernel(const double *__restrict__ part, int n,
                                                                double *__restrict__ loss) {
  __shared__ double red[LOSS_THREADS];
  double v = 0.0;
  for (int i = threadIdx.x; i < n; i += LOSS_THREADS) v += part[i];
  red[threadIdx.x] = v;
  __syncthreads();
  for (int w = LOSS_THREADS / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = red[0];
}

}  // namespace

LossLayout loss_layout(int B, int S) {
  LossLayout l;
  l.S_pad = ((S + BM - 1) / BM) * BM;
  l.n_blk = (l.S_pad + LOSS_THREADS - 1) / LOSS_THREADS;
  l.n_cta = int(((long long)B * S + CE_WARPS - 1) / CE_WARPS);
  size_t o = Workspace::align256(HDR_WORDS * 4);
  l.off_lo = o;
  o += Workspace::align256(size_t(B) * l.S_pad * 4);
  l.off_blk = o;
  o += Workspace::align256(size_t(B) * l.n_blk * 4);
  l.off_docsum = o;
  o += Workspace::align256(size_t(B) * l.S_pad * 8);
  l.off_part = o;
  o += Workspace::align256(size_t(l.n_cta) * 8);
  l.total = o;
  return l;
}

cudaError_t launch_packed_loss(const void *logits, const int *targets, const float *weight, const int *seg,
                               double *loss, void *dlogits, int B, int S, int V, void *workspace, int num_sms,
                               cudaStream_t stream) {
  const LossLayout l = loss_layout(B, S);
  char *base = static_cast<char *>(workspace);
  int *hdr = reinterpret_cast<int *>(base);
  int *lo = reinterpret_cast<int *>(base + l.off_lo);
  double *doc_sum = reinterpret_cast<double *>(base + l.off_docsum);
  cudaError_t e = launch_doc_starts(seg, B, S, l.S_pad, lo, reinterpret_cast<int *>(base + l.off_blk), hdr + HDR_ERR,
                                    stream);
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(doc_sum, 0, size_t(B) * l.S_pad * 8, stream)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(hdr + LHDR_NDOCS, 0, sizeof(int), stream)) != cudaSuccess) return e;
  const dim3 g((S + LOSS_THREADS - 1) / LOSS_THREADS, B);
  docsum_kernel<<<g, LOSS_THREADS, 0, stream>>>(seg, weight, lo, doc_sum, S, l.S_pad);
  ndocs_kernel<<<g, LOSS_THREADS, 0, stream>>>(lo, doc_sum, S, l.S_pad, hdr + LHDR_NDOCS);
  CeArgs a;
  a.logits = static_cast<const uint4 *>(logits);
  a.logits_e = static_cast<const __nv_bfloat16 *>(logits);
  a.targets = targets;
  a.seg = seg;
  a.weight = weight;
  a.lo = lo;
  a.doc_sum = doc_sum;
  a.ndocs = hdr + LHDR_NDOCS;
  a.dlogits = static_cast<uint4 *>(dlogits);
  a.part = reinterpret_cast<double *>(base + l.off_part);
  a.err = hdr + HDR_ERR;
  a.B = B;
  a.S = S;
  a.S_pad = l.S_pad;
  a.V = V;
  a.wait = wait_bound();
  int n_part = l.n_cta;
  if (V * 2 <= CE_ROW_MAX_BYTES) {
    static std::atomic<uint64_t> attr_done{0};
    // the row buffer decides how many CTAs share an SM (up to 3: one loads while others compute)
    const int smem = V * 2 + 128;
    if ((e = smem_attr_once(reinterpret_cast<const void *>(ce_row_kernel), CE_ROW_MAX_BYTES + 128, attr_done)) !=
        cudaSuccess)
      return e;
    const int per_sm = std::max(1, std::min(3, (227 * 1024) / (smem + 1024)));
    const long long rows = (long long)B * S;
    long long grid = (long long)num_sms * per_sm;
    if (grid > rows) grid = rows;
    if (grid > l.n_cta) grid = l.n_cta;
    n_part = int(grid);
    ce_row_kernel<<<n_part, CE_ROW_THREADS, smem, stream>>>(a);
  } else {
    ce_kernel<<<l.n_cta, CE_WARPS * 32, 0, stream>>>(a);
  }
  loss_sum_kernel<<<1, LOSS_THREADS, 0, stream>>>(a.part, n_part, loss);
  return cudaGetLastError();
}

}  // namespace lwm
