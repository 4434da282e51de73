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
  const int S_pad = w.S_pad;
  const long long tasks = (long long)p.B * ((S_pad + 31) / 32) * p.H;
  long long blocks = (tasks + DELTA_THREADS / 32 - 1) / (DELTA_THREADS / 32);
  const long long cap = (long long)p.num_sms * 8;
  if (blocks > cap) blocks = cap;
  delta_kernel<<<int(blocks), DELTA_THREADS, 0, stream>>>(static_cast<const uint4 *>(out),
                                                           static_cast<const uint4 *>(dout), lse, delta, lse2, p.B,
                                                           p.S, p.H, S_pad);
  return cudaGetLastError();
}

namespace {

// ----------------------------------------------------------------------------- shared pieces
// Both backward kernels keep one 128-row tile of their "own" rows resident (key rows
// for dK/dV, query rows for dQ) and stream 128-row tiles of the other side. Each
// streamed tile is processed as two 64-row halves h = 0, 1, one per softmax
// warpgroup, so that warpgroup h works on half h while the tensor core computes the
// other half's products. TMEM columns (fp32):
//   0-63 S_0 | 64-127 dP_0 | 128-191 S_1 | 192-255 dP_1 | 256-383 acc0 | 384-511 acc1
// The bf16 operands written back by the softmax warps (P, dS) overwrite the first 32
// columns of the S / dP block they were computed from.
constexpr int BW_WARPS = 12;
constexpr int BW_THREADS = BW_WARPS * 32;
constexpr int BW_PRODUCER = 8;
constexpr int BW_MMA = 9;
constexpr int HALF_ROWS = 64;
constexpr int HALF_ROW_BYTES = HALF_ROWS * 128;   // 64 rows of one 64-dim swizzled box
constexpr uint32_t COL_ACC0 = 256, COL_ACC1 = 384;
constexpr uint32_t IDESC_HALF = idesc_bf16(BM, HALF_ROWS, false, false);   // [128 x 64] = A . B_half^T
constexpr uint32_t IDESC_ACC = idesc_bf16(BM, HD, false, true);            // acc += X(tmem) . Y_half

__device__ __forceinline__ uint32_t col_s(int h) { return uint32_t(h) * 128u; }
__device__ __forceinline__ uint32_t col_dp(int h) { return uint32_t(h) * 128u + 64u; }

// D[128 x 64] = A[128 rows x 128 dims] . B[64 rows x 128 dims]^T, both K-major tiles
// (two 64-dim 128B-swizzled boxes, HALF_BYTES apart); `b_half` points at the first of
// the 64 B rows inside the tile.
__device__ __forceinline__ void issue_half(uint32_t d_tmem, uint32_t a_s, uint32_t b_half) {
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const uint32_t off = uint32_t(kk >> 2) * HALF_BYTES + uint32_t(kk & 3) * 32;
    mma_ss(d_tmem, sdesc_sw128(a_s + off, 16, 1024), sdesc_sw128(b_half + off, 16, 1024), IDESC_HALF, kk > 0);
  }
}

// acc[128 x 128] (+)= X[128 x 64] (bf16 in TMEM) . Y[64 rows x 128 dims] with Y read
// MN-major (dims contiguous): 16 rows = two 8-row groups of 1024 bytes.
__device__ __forceinline__ void issue_acc(uint32_t acc, uint32_t x_tmem, uint32_t y_half, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < HALF_ROWS / 16; ++kk)
    mma_ts(acc, x_tmem + uint32_t(kk) * 8, sdesc_sw128(y_half + uint32_t(kk) * 2048, HALF_BYTES, 1024), IDESC_ACC,
           (accumulate || kk > 0) ? 1u : 0u);
}

__device__ __forceinline__ void load_tile(const CUtensorMap *m, uint64_t *bar, uint8_t *dst, int h, int row0, int b) {
  tma_load_4d(m, bar, dst, 0, h, row0, b);
  tma_load_4d(m, bar, dst + HALF_BYTES, 64, h, row0, b);
}

__device__ bool bounded_wait_plain_bw(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
  return true;
}

// Writes one 128-value fp32 TMEM row (this thread's lane, columns c0..c0+n) scaled by
// `f` as bf16 to dst (n multiple of 32).
__device__ __forceinline__ void store_row_bf16(uint32_t t_addr, int n, float f, __nv_bfloat16 *dst, bool valid) {
  for (int cc = 0; cc < n; cc += 32) {
    uint32_t o[32];
    tmem_ld32(t_addr + cc, o);
    tmem_ld_wait();
    uint4 w[4];
    uint32_t *wp = reinterpret_cast<uint32_t *>(w);
#pragma unroll
    for (int e = 0; e < 16; ++e) wp[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * f, __uint_as_float(o[2 * e + 1]) * f);
    if (valid) {
      uint4 *d = reinterpret_cast<uint4 *>(dst + cc);
#pragma unroll
      for (int e = 0; e < 4; ++e) d[e] = w[e];
    }
  }
}

__device__ __forceinline__ void zero_row_bf16(__nv_bfloat16 *dst, int n) {
  uint4 *d = reinterpret_cast<uint4 *>(dst);
  for (int e = 0; e < n / 8; ++e) d[e] = make_uint4(0, 0, 0, 0);
}

struct BwArgs {
  const int *lo;       // [B, S_pad]
  const int *kend;     // [B, nT]
  const int *list;     // work list (b * nT + tile)
  const float *delta;  // [B, H, S_pad]
  const float *lse2;   // [B, H, S_pad], lse * log2(e), +inf where nothing is visible
  int *hdr;
  __nv_bfloat16 *out0, *out1;   // dK/dV kernel: dv, dk; dQ kernel: dq
  int B, S, H, nT, S_pad, n_items;
  float scale_log2;   // log2(e) / sqrt(D)
  float inv_sqrt_d;
};

struct BwItem {
  int b, h, tile;
};

__device__ __forceinline__ BwItem bw_decode(const BwArgs &a, int item) {
  const int e = a.list[item / a.H];
  return {e / a.nT, item % a.H, e % a.nT};
}

// Streamed-tile range of an item: dQ -> key tiles the query tile needs; dK/dV ->
// query tiles that see the key tile ([kt, (kend - 1) / BM]).
__device__ __forceinline__ TileRange dq_range(const BwArgs &a, const BwItem &I) {
  return q_tile_kv_range(a.lo + size_t(I.b) * a.S_pad, a.S, I.tile * BM);
}
__device__ __forceinline__ TileRange dkdv_range(const BwArgs &a, const BwItem &I) {
  const int k0 = I.tile * BN;
  const int e = a.kend[I.b * a.nT + I.tile];
  TileRange r{1, 0};
  if (e > k0) {
    r.first = k0 / BM;
    r.last = (e - 1) / BM;
  }
  return r;
}

// A tile pair is "full" when every (query, key) pair in it is visible: no masking.
__device__ __forceinline__ bool pair_full(const int *lo_row, int q0, int k0) {
  return lo_row[q0 + BM - 1] <= k0 && k0 + BN - 1 <= q0;
}

// ============================================================================= dQ
// Item: (b, h, query tile). Resident: Q and dO tiles. Streamed: K_j, V_j tiles.
//   S_h  = Q . K_h^T,  dP_h = dO . V_h^T            (h = 64-key half of tile j)
//   P    = exp2(S c - lse2_i) (masked),  dS = P (dP - delta_i)
//   dQ  += dS_h . K_h          (acc0; scaled by 1/sqrt(D) in the epilogue)
constexpr int DQ_STAGES = 2;
constexpr int DQ_SM_Q = 0, DQ_SM_DO = TILE_BYTES, DQ_SM_KV = 2 * TILE_BYTES;
constexpr int DQ_SM_BAR = DQ_SM_KV + DQ_STAGES * 2 * TILE_BYTES;

struct DqBars {
  uint64_t kv_full[DQ_STAGES], kv_empty[DQ_STAGES];
  uint64_t own_full, own_empty;
  uint64_t s_full[2], p_full[2];
  uint64_t acc_full, acc_empty;
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item[2];
  uint32_t tmem_base;
  int abort;
  int fill, use, own_issued, own_used;
};
constexpr int DQ_SMEM = DQ_SM_BAR + int(sizeof(DqBars)) + 1024;

__global__ void __launch_bounds__(BW_THREADS, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo, const BwArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DqBars *bars = reinterpret_cast<DqBars *>(smem + DQ_SM_BAR);
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < DQ_STAGES; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->own_full, 1);
    mbar_init(&bars->own_empty, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&bars->s_full[h], 1);
      mbar_init(&bars->p_full[h], 4);
      mbar_init(&bars->item_full[h], 1);
      mbar_init(&bars->item_empty[h], 9);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->fill = bars->use = bars->own_issued = bars->own_used = 0;
    fence_mbar_init();
  }
  if (warp == BW_MMA) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool ok = true;

  if (warp == BW_PRODUCER) {
    if (lane == 0) {
      int fill = 0, own = 0;
      for (int it = 0;; ++it) {
        const int slot = it & 1;
        if (!(ok = mbar_wait(&bars->item_empty[slot], ((it >> 1) & 1) ^ 1, abort))) break;
        const int t = atomicAdd(a.hdr + HDR_TICKET_DQ, 1);
        const int item = t < a.n_items ? t : -1;
        bars->item[slot] = item;
        mbar_arrive(&bars->item_full[slot]);
        if (item < 0) break;
        const BwItem I = bw_decode(a, item);
        const TileRange R = dq_range(a, I);
        if (!(ok = mbar_wait(&bars->own_empty, (it & 1) ^ 1, abort))) break;
        mbar_arrive_expect_tx(&bars->own_full, 2 * TILE_BYTES);
        load_tile(&tq, &bars->own_full, smem + DQ_SM_Q, I.h, I.tile * BM, I.b);
        load_tile(&tdo, &bars->own_full, smem + DQ_SM_DO, I.h, I.tile * BM, I.b);
        ++own;
        for (int j = R.first; j <= R.last && ok; ++j) {
          const int st = fill % DQ_STAGES;
          if (!(ok = mbar_wait(&bars->kv_empty[st], ((fill / DQ_STAGES) & 1) ^ 1, abort))) break;
          mbar_arrive_expect_tx(&bars->kv_full[st], 2 * TILE_BYTES);
          uint8_t *dst = smem + DQ_SM_KV + st * 2 * TILE_BYTES;
          load_tile(&tk, &bars->kv_full[st], dst, I.h, j * BN, I.b);
          load_tile(&tv, &bars->kv_full[st], dst + TILE_BYTES, I.h, j * BN, I.b);
          ++fill;
        }
        if (!ok) break;
      }
      bars->fill = fill;
      bars->own_issued = own;
    }
    __syncwarp();
  } else if (warp == BW_MMA) {
    const uint32_t q_s = smem_u32(smem + DQ_SM_Q), do_s = smem_u32(smem + DQ_SM_DO);
    const uint32_t kv0 = smem_u32(smem + DQ_SM_KV);
    int use = 0, own = 0;
    uint32_t pf_par[2] = {0, 0}, ae_par = 1;
    for (int it = 0; ok; ++it) {
      const int slot = it & 1;
      if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
      const int item = bars->item[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
      if (item < 0) break;
      const BwItem I = bw_decode(a, item);
      const TileRange R = dq_range(a, I);
      if (!(ok = mbar_wait(&bars->own_full, it & 1, abort))) break;
      ++own;
      tc_fence_after();
      bool first = true;
      if (!R.empty()) {
        // prologue: S and dP of both halves of the first key tile
        int st = use % DQ_STAGES;
        if (!(ok = mbar_wait(&bars->kv_full[st], (use / DQ_STAGES) & 1, abort))) break;
        ++use;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t k_s = kv0 + st * 2 * TILE_BYTES, v_s = k_s + TILE_BYTES;
          for (int h = 0; h < 2; ++h) {
            issue_half(tmem + col_s(h), q_s, k_s + h * HALF_ROW_BYTES);
            issue_half(tmem + col_dp(h), do_s, v_s + h * HALF_ROW_BYTES);
            mma_commit(&bars->s_full[h]);
          }
        }
        __syncwarp();
        for (int j = R.first; j <= R.last && ok; ++j) {
          const bool has_next = j < R.last;
          const uint32_t k_s = kv0 + st * 2 * TILE_BYTES;
          int st2 = -1;
          if (first) {
            if (!(ok = mbar_wait(&bars->acc_empty, ae_par, abort))) break;
            ae_par ^= 1;
          }
          for (int h = 0; h < 2 && ok; ++h) {
            if (!(ok = mbar_wait(&bars->p_full[h], pf_par[h], abort))) break;
            pf_par[h] ^= 1;
            tc_fence_after();
            if (lane == 0) issue_acc(tmem + COL_ACC0, tmem + col_s(h), k_s + h * HALF_ROW_BYTES, !first);
            first = false;
            if (h == 1 && lane == 0) mma_commit(&bars->kv_empty[st]);
            if (has_next) {
              if (h == 0) {
                st2 = use % DQ_STAGES;
                if (!(ok = mbar_wait(&bars->kv_full[st2], (use / DQ_STAGES) & 1, abort))) break;
                ++use;
                tc_fence_after();
              }
              if (lane == 0) {
                const uint32_t k2 = kv0 + st2 * 2 * TILE_BYTES, v2 = k2 + TILE_BYTES;
                issue_half(tmem + col_s(h), q_s, k2 + h * HALF_ROW_BYTES);
                issue_half(tmem + col_dp(h), do_s, v2 + h * HALF_ROW_BYTES);
                mma_commit(&bars->s_full[h]);
              }
            }
          }
          __syncwarp();
          st = st2;
        }
        if (!ok) break;
      }
      if (lane == 0) {
        mma_commit(&bars->own_empty);
        if (!first) mma_commit(&bars->acc_full);
      }
      __syncwarp();
    }
    if (lane == 0) {
      bars->use = use;
      bars->own_used = own;
    }
  } else if (warp < 8) {
    const int h = warp >> 2;   // key half this warpgroup owns
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + col_s(h), tP = tmem + lane_off + col_dp(h);
    const float c = a.scale_log2;
    uint32_t sf_par = 0, af_par = 0;
    for (int it = 0; ok; ++it) {
      const int slot = it & 1;
      if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
      const int item = bars->item[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
      if (item < 0) break;
      const BwItem I = bw_decode(a, item);
      const TileRange R = dq_range(a, I);
      const int q0 = I.tile * BM, i = q0 + r;
      const int *lr = a.lo + size_t(I.b) * a.S_pad;
      const int lo_i = lr[i];
      const size_t rowterm = (size_t(I.b) * a.H + I.h) * a.S_pad + i;
      const float l2 = a.lse2[rowterm], dl = a.delta[rowterm];
      for (int j = R.first; j <= R.last; ++j) {
        if (!(ok = mbar_wait(&bars->s_full[h], sf_par, abort))) break;
        sf_par ^= 1;
        tc_fence_after();
        const int k0 = j * BN;
        const bool full = pair_full(lr, q0, k0);
        const int kb = k0 + h * HALF_ROWS;   // first key of this half
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t sv[32], dv[32];
          tmem_ld32(tS + ch * 32, sv);
          tmem_ld32(tP + ch * 32, dv);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float ds2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int cidx = 2 * e + u;
              float p = ex2_approx(fmaf(__uint_as_float(sv[cidx]), c, -l2));
              if (!full) {
                const int kj = kb + ch * 32 + cidx;
                if (kj < lo_i || kj > i) p = 0.f;
              }
              ds2[u] = p * (__uint_as_float(dv[cidx]) - dl);
            }
            pk[e] = pack_bf16x2(ds2[0], ds2[1]);
          }
          tmem_st16(tS + ch * 16, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[h]);
      }
      if (!ok) break;
      __nv_bfloat16 *dst = a.out0 + ((size_t(I.b) * a.S + i) * a.H + I.h) * HD + h * 64;
      if (!R.empty()) {
        if (!(ok = mbar_wait(&bars->acc_full, af_par, abort))) break;
        af_par ^= 1;
        tc_fence_after();
        store_row_bf16(tmem + lane_off + COL_ACC0 + h * 64, 64, a.inv_sqrt_d, dst, i < a.S);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->acc_empty);
      } else if (i < a.S) {
        zero_row_bf16(dst, 64);
      }
    }
  }

  if (!ok) {
    bars->abort = 1;
    raise_error(a.hdr + HDR_ERR, ERRBIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (bars->abort) {
    if (warp == BW_PRODUCER && lane == 0) {
      for (int n = bars->use; n < bars->fill; ++n)
        bounded_wait_plain_bw(&bars->kv_full[n % DQ_STAGES], (n / DQ_STAGES) & 1);
      if (bars->own_issued > bars->own_used) bounded_wait_plain_bw(&bars->own_full, (bars->own_issued - 1) & 1);
    }
    if (warp == BW_MMA && lane == 0) {
      mma_commit(&bars->drain);
      bounded_wait_plain_bw(&bars->drain, 0);
    }
    __syncthreads();
  }
  if (warp == BW_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.hdr + HDR_DONE_DQ, 1) == int(gridDim.x) - 1) {
      a.hdr[HDR_TICKET_DQ] = 0;
      a.hdr[HDR_DONE_DQ] = 0;
      __threadfence();
    }
  }
}

// ============================================================================= dK/dV
// Item: (b, h, key tile). Resident: K and V tiles. Streamed: Q_i, dO_i tiles plus the
// tile's lo / lse2 / delta rows (bulk copies). Per 64-query half h of tile i:
//   S^T_h = K . Q_h^T,  dP^T_h = V . dO_h^T       (rows = keys, columns = queries)
//   P^T = exp2(S^T c - lse2) (masked), dS^T = P^T (dP^T - delta)
//   dV += P^T_h . dO_h (acc0),  dK += dS^T_h . Q_h (acc1; scaled by 1/sqrt(D) at the end)
constexpr int KV_STAGES_BW = 2;
constexpr int ROWTERM_BYTES = BM * 4;   // 128 fp32 / int32 values
constexpr int KVB_SM_K = 0, KVB_SM_V = TILE_BYTES, KVB_SM_ST = 2 * TILE_BYTES;
constexpr int KVB_STAGE_BYTES = 2 * TILE_BYTES + 3 * ROWTERM_BYTES;   // Q, dO, lo, lse2, delta
constexpr int KVB_SM_BAR = KVB_SM_ST + KV_STAGES_BW * ((KVB_STAGE_BYTES + 1023) & ~1023);
constexpr int KVB_STAGE_STRIDE = (KVB_STAGE_BYTES + 1023) & ~1023;

struct KvbBars {
  uint64_t st_full[KV_STAGES_BW], st_empty[KV_STAGES_BW];
  uint64_t own_full, own_empty;
  uint64_t s_full[2], p_full[2];
  uint64_t acc_full, acc_empty;
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item[2];
  uint32_t tmem_base;
  int abort;
  int fill, use, own_issued, own_used;
};
constexpr int KVB_SMEM = KVB_SM_BAR + int(sizeof(KvbBars)) + 1024;

__global__ void __launch_bounds__(BW_THREADS, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo, const BwArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  KvbBars *bars = reinterpret_cast<KvbBars *>(smem + KVB_SM_BAR);
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < KV_STAGES_BW; ++s) {
      mbar_init(&bars->st_full[s], 1);
      mbar_init(&bars->st_empty[s], 1);
    }
    mbar_init(&bars->own_full, 1);
    mbar_init(&bars->own_empty, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&bars->s_full[h], 1);
      mbar_init(&bars->p_full[h], 4);
      mbar_init(&bars->item_full[h], 1);
      mbar_init(&bars->item_empty[h], 9);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->fill = bars->use = bars->own_issued = bars->own_used = 0;
    fence_mbar_init();
  }
  if (warp == BW_MMA) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool ok = true;

  if (warp == BW_PRODUCER) {
    if (lane == 0) {
      int fill = 0, own = 0;
      for (int it = 0;; ++it) {
        const int slot = it & 1;
        if (!(ok = mbar_wait(&bars->item_empty[slot], ((it >> 1) & 1) ^ 1, abort))) break;
        const int t = atomicAdd(a.hdr + HDR_TICKET_DKDV, 1);
        const int item = t < a.n_items ? t : -1;
        bars->item[slot] = item;
        mbar_arrive(&bars->item_full[slot]);
        if (item < 0) break;
        const BwItem I = bw_decode(a, item);
        const TileRange R = dkdv_range(a, I);
        if (!(ok = mbar_wait(&bars->own_empty, (it & 1) ^ 1, abort))) break;
        mbar_arrive_expect_tx(&bars->own_full, 2 * TILE_BYTES);
        load_tile(&tk, &bars->own_full, smem + KVB_SM_K, I.h, I.tile * BN, I.b);
        load_tile(&tv, &bars->own_full, smem + KVB_SM_V, I.h, I.tile * BN, I.b);
        ++own;
        const size_t rowbase = (size_t(I.b) * a.H + I.h) * a.S_pad;
        for (int qi = R.first; qi <= R.last && ok; ++qi) {
          const int st = fill % KV_STAGES_BW;
          if (!(ok = mbar_wait(&bars->st_empty[st], ((fill / KV_STAGES_BW) & 1) ^ 1, abort))) break;
          mbar_arrive_expect_tx(&bars->st_full[st], 2 * TILE_BYTES + 3 * ROWTERM_BYTES);
          uint8_t *dst = smem + KVB_SM_ST + st * KVB_STAGE_STRIDE;
          load_tile(&tq, &bars->st_full[st], dst, I.h, qi * BM, I.b);
          load_tile(&tdo, &bars->st_full[st], dst + TILE_BYTES, I.h, qi * BM, I.b);
          bulk_load(dst + 2 * TILE_BYTES, a.lo + size_t(I.b) * a.S_pad + qi * BM, ROWTERM_BYTES, &bars->st_full[st]);
          bulk_load(dst + 2 * TILE_BYTES + ROWTERM_BYTES, a.lse2 + rowbase + qi * BM, ROWTERM_BYTES,
                    &bars->st_full[st]);
          bulk_load(dst + 2 * TILE_BYTES + 2 * ROWTERM_BYTES, a.delta + rowbase + qi * BM, ROWTERM_BYTES,
                    &bars->st_full[st]);
          ++fill;
        }
        if (!ok) break;
      }
      bars->fill = fill;
      bars->own_issued = own;
    }
    __syncwarp();
  } else if (warp == BW_MMA) {
    const uint32_t k_s = smem_u32(smem + KVB_SM_K), v_s = smem_u32(smem + KVB_SM_V);
    const uint32_t st0 = smem_u32(smem + KVB_SM_ST);
    int use = 0, own = 0;
    uint32_t pf_par[2] = {0, 0}, ae_par = 1;
    for (int it = 0; ok; ++it) {
      const int slot = it & 1;
      if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
      const int item = bars->item[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
      if (item < 0) break;
      const BwItem I = bw_decode(a, item);
      const TileRange R = dkdv_range(a, I);
      if (!(ok = mbar_wait(&bars->own_full, it & 1, abort))) break;
      ++own;
      tc_fence_after();
      bool first = true;
      if (!R.empty()) {
        int st = use % KV_STAGES_BW;
        if (!(ok = mbar_wait(&bars->st_full[st], (use / KV_STAGES_BW) & 1, abort))) break;
        ++use;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t q_s = st0 + st * KVB_STAGE_STRIDE, do_s = q_s + TILE_BYTES;
          for (int h = 0; h < 2; ++h) {
            issue_half(tmem + col_s(h), k_s, q_s + h * HALF_ROW_BYTES);
            issue_half(tmem + col_dp(h), v_s, do_s + h * HALF_ROW_BYTES);
            mma_commit(&bars->s_full[h]);
          }
        }
        __syncwarp();
        for (int qi = R.first; qi <= R.last && ok; ++qi) {
          const bool has_next = qi < R.last;
          const uint32_t q_s = st0 + st * KVB_STAGE_STRIDE, do_s = q_s + TILE_BYTES;
          int st2 = -1;
          if (first) {
            if (!(ok = mbar_wait(&bars->acc_empty, ae_par, abort))) break;
            ae_par ^= 1;
          }
          for (int h = 0; h < 2 && ok; ++h) {
            if (!(ok = mbar_wait(&bars->p_full[h], pf_par[h], abort))) break;
            pf_par[h] ^= 1;
            tc_fence_after();
            if (lane == 0) {
              issue_acc(tmem + COL_ACC0, tmem + col_s(h), do_s + h * HALF_ROW_BYTES, !first);   // dV
              issue_acc(tmem + COL_ACC1, tmem + col_dp(h), q_s + h * HALF_ROW_BYTES, !first);   // dK
            }
            first = false;
            if (h == 1 && lane == 0) mma_commit(&bars->st_empty[st]);
            if (has_next) {
              if (h == 0) {
                st2 = use % KV_STAGES_BW;
                if (!(ok = mbar_wait(&bars->st_full[st2], (use / KV_STAGES_BW) & 1, abort))) break;
                ++use;
                tc_fence_after();
              }
              if (lane == 0) {
                const uint32_t q2 = st0 + st2 * KVB_STAGE_STRIDE, do2 = q2 + TILE_BYTES;
                issue_half(tmem + col_s(h), k_s, q2 + h * HALF_ROW_BYTES);
                issue_half(tmem + col_dp(h), v_s, do2 + h * HALF_ROW_BYTES);
                mma_commit(&bars->s_full[h]);
              }
            }
          }
          __syncwarp();
          st = st2;
        }
        if (!ok) break;
      }
      if (lane == 0) {
        mma_commit(&bars->own_empty);
        if (!first) mma_commit(&bars->acc_full);
      }
      __syncwarp();
    }
    if (lane == 0) {
      bars->use = use;
      bars->own_used = own;
    }
  } else if (warp < 8) {
    const int h = warp >> 2;   // query half this warpgroup owns
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + col_s(h), tP = tmem + lane_off + col_dp(h);
    const float c = a.scale_log2;
    uint32_t sf_par = 0, af_par = 0;
    int use = 0;
    for (int it = 0; ok; ++it) {
      const int slot = it & 1;
      if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
      const int item = bars->item[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
      if (item < 0) break;
      const BwItem I = bw_decode(a, item);
      const TileRange R = dkdv_range(a, I);
      const int k0 = I.tile * BN, j = k0 + r;
      const int *lr = a.lo + size_t(I.b) * a.S_pad;
      for (int qi = R.first; qi <= R.last; ++qi) {
        const int st = use % KV_STAGES_BW;
        const uint32_t st_par = (use / KV_STAGES_BW) & 1;
        ++use;
        if (!(ok = mbar_wait(&bars->s_full[h], sf_par, abort))) break;
        sf_par ^= 1;
        // the stage's lo / lse2 / delta rows arrived by bulk copy: observe their barrier
        if (!(ok = mbar_wait(&bars->st_full[st], st_par, abort))) break;
        tc_fence_after();
        const uint8_t *stage = smem + KVB_SM_ST + st * KVB_STAGE_STRIDE;
        const int *lo_q = reinterpret_cast<const int *>(stage + 2 * TILE_BYTES) + h * HALF_ROWS;
        const float *l2_q = reinterpret_cast<const float *>(stage + 2 * TILE_BYTES + ROWTERM_BYTES) + h * HALF_ROWS;
        const float *dl_q = reinterpret_cast<const float *>(stage + 2 * TILE_BYTES + 2 * ROWTERM_BYTES) + h * HALF_ROWS;
        const int q0 = qi * BM;
        const bool full = pair_full(lr, q0, k0);
        const int qb = q0 + h * HALF_ROWS;   // first query of this half
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t sv[32], dv[32];
          tmem_ld32(tS + ch * 32, sv);
          tmem_ld32(tP + ch * 32, dv);
          tmem_ld_wait();
          uint32_t pk[16], dk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float pp[2], dd[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int cidx = ch * 32 + 2 * e + u;
              float p = ex2_approx(fmaf(__uint_as_float(sv[2 * e + u]), c, -l2_q[cidx]));
              if (!full) {
                const int qq = qb + cidx;
                if (j < lo_q[cidx] || j > qq) p = 0.f;
              }
              pp[u] = p;
              dd[u] = p * (__uint_as_float(dv[2 * e + u]) - dl_q[cidx]);
            }
            pk[e] = pack_bf16x2(pp[0], pp[1]);
            dk[e] = pack_bf16x2(dd[0], dd[1]);
          }
          tmem_st16(tS + ch * 16, pk);
          tmem_st16(tP + ch * 16, dk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[h]);
      }
      if (!ok) break;
      // epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (scaled by 1/sqrt(D))
      __nv_bfloat16 *dst = (h == 0 ? a.out0 : a.out1) + ((size_t(I.b) * a.S + j) * a.H + I.h) * HD;
      if (!R.empty()) {
        if (!(ok = mbar_wait(&bars->acc_full, af_par, abort))) break;
        af_par ^= 1;
        tc_fence_after();
        store_row_bf16(tmem + lane_off + (h == 0 ? COL_ACC0 : COL_ACC1), HD, h == 0 ? 1.f : a.inv_sqrt_d, dst,
                       j < a.S);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->acc_empty);
      } else if (j < a.S) {
        zero_row_bf16(dst, HD);
      }
    }
  }

  if (!ok) {
    bars->abort = 1;
    raise_error(a.hdr + HDR_ERR, ERRBIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (bars->abort) {
    if (warp == BW_PRODUCER && lane == 0) {
      for (int n = bars->use; n < bars->fill; ++n)
        bounded_wait_plain_bw(&bars->st_full[n % KV_STAGES_BW], (n / KV_STAGES_BW) & 1);
      if (bars->own_issued > bars->own_used) bounded_wait_plain_bw(&bars->own_full, (bars->own_issued - 1) & 1);
    }
    if (warp == BW_MMA && lane == 0) {
      mma_commit(&bars->drain);
      bounded_wait_plain_bw(&bars->drain, 0);
    }
    __syncthreads();
  }
  if (warp == BW_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.hdr + HDR_DONE_DKDV, 1) == int(gridDim.x) - 1) {
      a.hdr[HDR_TICKET_DKDV] = 0;
      a.hdr[HDR_DONE_DKDV] = 0;
      __threadfence();
    }
  }
}

BwArgs bw_args(const Problem &p, void *workspace, const int *list) {
  const Workspace w = Workspace::layout(p.B, p.S, p.H);
  char *base = static_cast<char *>(workspace);
  BwArgs a;
  a.lo = reinterpret_cast<const int *>(base + w.off_lo);
  a.kend = reinterpret_cast<const int *>(base + w.off_kend);
  a.list = list;
  a.delta = reinterpret_cast<const float *>(base + w.off_delta);
  a.lse2 = reinterpret_cast<const float *>(base + w.off_lse2);
  a.hdr = reinterpret_cast<int *>(base + w.off_hdr);
  a.out0 = a.out1 = nullptr;
  a.B = p.B;
  a.S = p.S;
  a.H = p.H;
  a.nT = w.nT;
  a.S_pad = w.S_pad;
  a.n_items = p.B * w.nT * p.H;
  a.scale_log2 = 1.4426950408889634f / sqrtf(float(HD));
  a.inv_sqrt_d = 1.f / sqrtf(float(HD));
  return a;
}

}  // namespace

cudaError_t launch_dkdv(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tdo,
                        void *dk, void *dv, const Problem &p, void *workspace, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KVB_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const Workspace w = Workspace::layout(p.B, p.S, p.H);
  BwArgs a = bw_args(p, workspace, reinterpret_cast<const int *>(static_cast<char *>(workspace) + w.off_list_kv));
  a.out0 = static_cast<__nv_bfloat16 *>(dv);
  a.out1 = static_cast<__nv_bfloat16 *>(dk);
  const int grid = a.n_items < p.num_sms ? a.n_items : p.num_sms;
  dkdv_kernel<<<grid, BW_THREADS, KVB_SMEM, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

cudaError_t launch_dq(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tdo,
                      void *dq, const Problem &p, void *workspace, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const Workspace w = Workspace::layout(p.B, p.S, p.H);
  BwArgs a = bw_args(p, workspace, reinterpret_cast<const int *>(static_cast<char *>(workspace) + w.off_list_q));
  a.out0 = static_cast<__nv_bfloat16 *>(dq);
  const int grid = a.n_items < p.num_sms ? a.n_items : p.num_sms;
  dq_kernel<<<grid, BW_THREADS, DQ_SMEM, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}
}  // namespace lwm
