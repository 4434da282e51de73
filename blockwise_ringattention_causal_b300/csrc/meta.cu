// Metadata pre-pass: per-token document starts, per-tile key/query ranges and the
// longest-first work lists of the persistent kernels.
//
// The packing mask of LWM's masked sequence packing (each packed document attends
// only to itself; LWM deep-dive page, section "Masked sequence packing") together
// with causality reduces, for contiguous documents, to one number per query: the
// first visible key lo[i] = i - pos[i] (the start of i's document). Query i then
// sees exactly the keys lo[i] <= j <= i. Padding tokens (negative ids) get
// lo[i] = i + 1, i.e. nothing visible.
#include "common.cuh"
#include "kernels.h"

namespace lwm {

namespace {

constexpr int META_THREADS = 1024;

__device__ __forceinline__ int warp_incl_max(int v) {
  const unsigned lane = threadIdx.x & 31u;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= unsigned(d)) v = max(v, o);
  }
  return v;
}

// Block-wide inclusive prefix max over META_THREADS values.
__device__ int block_incl_max(int v, int *scratch /* 32 ints */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_incl_max(v);
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
    w = warp_incl_max(w);
    scratch[lane] = w;
  }
  __syncthreads();
  if (warp > 0) v = max(v, scratch[warp - 1]);
  __syncthreads();
  return v;
}

// Pass 1: validate seg/pos and compute lo. With pos given, lo is local; without it,
// lo is the prefix max of document starts, finished by pass 2 across blocks.
__global__ void __launch_bounds__(META_THREADS) meta_lo_kernel(const int *__restrict__ seg,
                                                               const int *__restrict__ pos, int S, int S_pad,
                                                               int *__restrict__ lo, int *__restrict__ blk_last,
                                                               int *__restrict__ err) {
  __shared__ int scratch[32];
  const int b = blockIdx.y;
  const int i = blockIdx.x * META_THREADS + threadIdx.x;
  const bool in = i < S;
  const size_t row = size_t(b) * S;
  const int si = (in && seg) ? seg[row + i] : 0;
  const int sp = (in && seg && i > 0) ? seg[row + i - 1] : si;
  const bool start = in && (i == 0 || si != sp);
  const bool pad = si < 0;
  bool bad = false;
  if (in && i > 0 && seg) {
    if (sp < 0 && si >= 0) bad = true;              // a document after padding
    if (sp >= 0 && si >= 0 && si < sp) bad = true;  // ids must not decrease
  }
  int my_lo = 0;
  if (pos) {
    if (in && !pad) {
      const int p = pos[row + i];
      if (start) {
        if (p != 0) bad = true;
      } else if (p != pos[row + i - 1] + 1) {
        bad = true;
      }
      my_lo = i - p;
    }
  } else {
    const int v = block_incl_max(start ? i : -1, scratch);
    my_lo = v;   // -1: the document started in an earlier block (pass 2)
    if (threadIdx.x == META_THREADS - 1) blk_last[size_t(b) * gridDim.x + blockIdx.x] = v;
  }
  if (in) lo[size_t(b) * S_pad + i] = pad ? i + 1 : my_lo;
  else if (i < S_pad) lo[size_t(b) * S_pad + i] = i + 1;   // rows past the end see nothing
  if (bad) raise_error(err, ERRBIT_SEGMENTS);
}

// Pass 2 (pos == NULL only): carry the last document start of earlier blocks.
__global__ void __launch_bounds__(META_THREADS) meta_lo_carry_kernel(const int *__restrict__ seg, int S,
                                                                     int S_pad, int *__restrict__ lo,
                                                                     const int *__restrict__ blk_last) {
  __shared__ int red[32];
  const int b = blockIdx.y;
  int carry = -1;
  for (int k = threadIdx.x; k < int(blockIdx.x); k += META_THREADS)
    carry = max(carry, blk_last[size_t(b) * gridDim.x + k]);
  for (int d = 16; d > 0; d >>= 1) carry = max(carry, __shfl_xor_sync(0xffffffffu, carry, d));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = carry;
  __syncthreads();
  carry = red[0];
  for (int k = 1; k < 32; ++k) carry = max(carry, red[k]);
  const int i = blockIdx.x * META_THREADS + threadIdx.x;
  if (i < S) {
    const int si = seg ? seg[size_t(b) * S + i] : 0;
    int &l = lo[size_t(b) * S_pad + i];
    if (si >= 0 && l < 0) l = carry;
  }
}

// Per key tile: end (exclusive) of the query rows that see any of its keys. The rows
// that see key tile [k0, k1) are i >= k0 with lo[i] <= k1 - 1; lo is non-decreasing,
// so they form [k0, kend) with kend the first i >= k0 with lo[i] >= k1.
__global__ void meta_kend_kernel(const int *__restrict__ lo, int B, int S, int S_pad, int nT,
                                 int *__restrict__ kend) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= B * nT) return;
  const int b = t / nT, kt = t % nT;
  const int *lr = lo + size_t(b) * S_pad;
  const int k0 = kt * BN, k1 = min(k0 + BN, S);
  int a = k0, z = S;   // first index in [a, z) with lr[idx] >= k1
  while (a < z) {
    const int mid = (a + z) >> 1;
    if (lr[mid] >= k1) z = mid; else a = mid + 1;
  }
  kend[t] = a;
}

__device__ __forceinline__ int range_size(const int *lr, int S, int q0) {
  if (q0 >= S) return 0;
  const int qb = min(q0 + BM, S) - 1;
  const int la = lr[q0];
  if (la > qb) return 0;
  return qb / BN - la / BN + 1;
}

// Longest-first work lists by counting sort over integer costs, one block per list:
//   list 0: forward query-tile pairs (b, p)  - cost = key tiles of both tiles;
//   list 1: key tiles (b, kt) for dK/dV     - cost = query tiles that see the tile;
//   list 2: query tiles (b, qt) for dQ      - cost = key tiles the tile needs.
// Items of equal cost (or, for costs above NBINS, of costs that share a bin) keep no
// particular order. The block also resets the tickets.
__global__ void __launch_bounds__(META_THREADS) meta_sort_kernel(const int *__restrict__ lo,
                                                                 const int *__restrict__ kend, int B, int S,
                                                                 int S_pad, int nT, int nP, int *__restrict__ hdr,
                                                                 int *__restrict__ list_fwd,
                                                                 int *__restrict__ list_kv,
                                                                 int *__restrict__ list_q, int kv_chunk) {
  __shared__ int hist[NBINS];
  __shared__ int scratch[32];
  const int which = blockIdx.x;
  const int n = which == 0 ? B * nP : B * nT;
  int *list = which == 0 ? list_fwd : (which == 1 ? list_kv : list_q);

  if (which == 0 && threadIdx.x == 0) {
    hdr[HDR_KV_CHUNK] = kv_chunk;
    for (int w = HDR_TICKET_FWD; w <= HDR_DONE_FUSED; ++w) hdr[w] = 0;
  }
  for (int k = threadIdx.x; k < NBINS; k += META_THREADS) hist[k] = 0;
  __syncthreads();

  auto cost_of = [&](int idx) -> int {
    if (which == 0) {
      const int b = idx / nP, p = idx % nP;
      const int *lr = lo + size_t(b) * S_pad;
      return range_size(lr, S, (2 * p) * BM) + range_size(lr, S, (2 * p + 1) * BM);
    } else if (which == 1) {
      const int kt = idx % nT;
      const int k0 = kt * BN, e = kend[idx];
      return e > k0 ? (e - 1) / BM - k0 / BM + 1 : 0;
    } else {
      return range_size(lo + size_t(idx / nT) * S_pad, S, (idx % nT) * BM);
    }
  };
  // Costs reach 2 * nT (16384 key tiles for a forward pair at S = 1M), more than there
  // are bins: scale them by the smallest integer that maps the largest onto the bins,
  // so that the list stays longest first (items within one bin: any order).
  int cmax = 0;
  for (int idx = threadIdx.x; idx < n; idx += META_THREADS) cmax = max(cmax, cost_of(idx));
  for (int d = 16; d > 0; d >>= 1) cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, d));
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = cmax;
  __syncthreads();
  cmax = 0;
  for (int k = 0; k < META_THREADS / 32; ++k) cmax = max(cmax, scratch[k]);
  __syncthreads();
  const int div = cmax / NBINS + 1;   // cmax / div <= NBINS - 1
  // bins in descending cost order: bin 0 holds the largest costs
  auto bin_of = [&](int c) -> int { return NBINS - 1 - c / div; };

  for (int idx = threadIdx.x; idx < n; idx += META_THREADS) atomicAdd(&hist[bin_of(cost_of(idx))], 1);
  __syncthreads();

  // exclusive scan over the bins (each thread owns NBINS / META_THREADS consecutive bins)
  constexpr int PER = NBINS / META_THREADS;
  int local[PER];
  int sum = 0;
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    local[r] = hist[threadIdx.x * PER + r];
    sum += local[r];
  }
  // block inclusive sum scan
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int o = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += o;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  int excl = v - sum + (warp > 0 ? scratch[warp - 1] : 0);
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    hist[threadIdx.x * PER + r] = excl;
    excl += local[r];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < n; idx += META_THREADS) {
    const int slot = atomicAdd(&hist[bin_of(cost_of(idx))], 1);
    list[slot] = idx;
  }
}

}  // namespace

cudaError_t launch_doc_starts(const int *seg, int B, int S, int S_pad, int *lo, int *blk_last, int *err,
                              cudaStream_t stream) {
  const dim3 g1((S_pad + META_THREADS - 1) / META_THREADS, B);
  meta_lo_kernel<<<g1, META_THREADS, 0, stream>>>(seg, nullptr, S, S_pad, lo, blk_last, err);
  meta_lo_carry_kernel<<<g1, META_THREADS, 0, stream>>>(seg, S, S_pad, lo, blk_last);
  return cudaGetLastError();
}

cudaError_t launch_meta(const int *seg, const int *pos, int B, int S, int kv_chunk, void *workspace,
                        cudaStream_t stream) {
  const Workspace w = Workspace::layout(B, S, 1);
  char *base = static_cast<char *>(workspace);
  int *hdr = reinterpret_cast<int *>(base + w.off_hdr);
  int *lo = reinterpret_cast<int *>(base + w.off_lo);
  int *kend = reinterpret_cast<int *>(base + w.off_kend);
  int *lf = reinterpret_cast<int *>(base + w.off_list_fwd);
  int *lk = reinterpret_cast<int *>(base + w.off_list_kv);
  int *lq = reinterpret_cast<int *>(base + w.off_list_q);
  // the delta region (>= B*S*4 bytes, unused until the backward pass) holds the
  // per-block carries of pass 1
  int *blk_last = reinterpret_cast<int *>(base + w.off_delta);

  const dim3 g1((w.S_pad + META_THREADS - 1) / META_THREADS, B);
  meta_lo_kernel<<<g1, META_THREADS, 0, stream>>>(seg, pos, S, w.S_pad, lo, blk_last, hdr + HDR_ERR);
  if (!pos) meta_lo_carry_kernel<<<g1, META_THREADS, 0, stream>>>(seg, S, w.S_pad, lo, blk_last);
  const int nk = B * w.nT;
  meta_kend_kernel<<<(nk + 255) / 256, 256, 0, stream>>>(lo, B, S, w.S_pad, w.nT, kend);
  meta_sort_kernel<<<3, META_THREADS, 0, stream>>>(lo, kend, B, S, w.S_pad, w.nT, w.nP, hdr, lf, lk, lq,
                                                   kv_chunk);
  return cudaGetLastError();
}

}  // namespace lwm
