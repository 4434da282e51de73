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

// x as hi + mid + lo in bf16 (each the rounding of what is left): the sum carries about
// 24 bits, as an fp32 value does; products with 1 are exact in the tensor core.
__device__ __forceinline__ uint4 bf16_split_row(float x) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  __nv_bfloat162 a, b;
  a.x = hi;
  a.y = mid;
  b.x = lo;
  b.y = __float2bfloat16_rn(0.f);
  return make_uint4(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&b), 0u, 0u);
}

// delta[b,h,i] = sum_d dout[b,i,h,d] * out[b,i,h,d] (fp32), and lse2[b,h,i] =
// lse * log2(e) on a row stride padded to a multiple of 128, with +inf for rows that
// see no key (padding) and for the pad tail, so that exp2(s - lse2) is 0 there. Also,
// for the dK/dV kernel, the offset rows qx = -lse * sqrt(D) (so that (S^T + qx) * c =
// S^T c - lse2 with c = log2(e) / sqrt(D); -1e30 where nothing is visible) and dox =
// -delta, each as three bf16 parts in a 16-byte row (see the dK/dV kernel).
// One warp handles 32 consecutive rows of one head: two rows per load step, 16 lanes
// per 256-byte row, fully coalesced; the 32 results are written as one 128-byte line.
__global__ void __launch_bounds__(DELTA_THREADS) delta_kernel(const uint4 *__restrict__ out,
                                                              const uint4 *__restrict__ dout,
                                                              const float *__restrict__ lse,
                                                              float *__restrict__ delta, float *__restrict__ lse2,
                                                              uint4 *__restrict__ qx, uint4 *__restrict__ dox,
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
      float xq = -1e30f;
      if (i < S) {
        const float L = lse[(size_t(b) * H + h) * S + i];
        if (L != -__int_as_float(0x7f800000)) {
          l2 = L * 1.4426950408889634f;
          xq = -L * 11.313708498984761f;   // sqrt(128)
        }
      }
      delta[o] = mine;
      lse2[o] = l2;
      qx[o] = bf16_split_row(xq);
      dox[o] = bf16_split_row(-mine);
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
  uint4 *qx = reinterpret_cast<uint4 *>(base + w.off_qx);
  uint4 *dox = reinterpret_cast<uint4 *>(base + w.off_dox);
  const int S_pad = w.S_pad;
  const long long tasks = (long long)p.B * ((S_pad + 31) / 32) * p.H;
  long long blocks = (tasks + DELTA_THREADS / 32 - 1) / (DELTA_THREADS / 32);
  const long long cap = (long long)p.num_sms * 8;
  if (blocks > cap) blocks = cap;
  delta_kernel<<<int(blocks), DELTA_THREADS, 0, stream>>>(static_cast<const uint4 *>(out),
                                                           static_cast<const uint4 *>(dout), lse, delta, lse2, qx,
                                                           dox, p.B, p.S, p.H, S_pad);
  return cudaGetLastError();
}

namespace {

// ----------------------------------------------------------------------------- shared pieces
// Both kernels keep one 128-row tile of their "own" rows resident (key rows for dK/dV,
// query rows for dQ) and stream 128-row tiles of the other side; every product is
// 128 x 128 x 128 (K = 16 per instruction). Warp roles: 0-3 and 4-7 two softmax
// warpgroups, warpgroup w owning columns [64 w, 64 w + 64) of every 128 x 128 score
// tile (thread = row of the tile = TMEM lane); 8 TMA producer; 9 and 10 two MMA issuers
// (one thread issuing back to back cannot keep the tensor core busy while the softmax
// warps load the SM: each tcgen05.mma issue costs that thread about as long as the
// product takes to run); 11 idle (3 warps per SM sub-partition: up to 168 registers per
// thread).
constexpr int BW_WARPS = 12;
constexpr int BW_THREADS = BW_WARPS * 32;
constexpr int BW_PRODUCER = 8;
constexpr int BW_MMA = 9;       // MMA issuer (owns TMEM)
constexpr int BW_MMA2 = 10;     // second MMA issuer
constexpr int BW_MMA3 = 11;     // third MMA issuer (dQ kernel: the S products)
constexpr int RT_BYTES = BM * 4;   // 128 row terms (int32 / fp32)

__device__ __forceinline__ void load_tile(const CUtensorMap *m, uint64_t *bar, uint8_t *dst, int h, int row0, int b) {
  tma_load_4d(m, bar, dst, 0, h, row0, b);
  tma_load_4d(m, bar, dst + HALF_BYTES, 64, h, row0, b);
}

// Writes 64 fp32 TMEM columns of this thread's lane, scaled by f, as bf16 to dst.
__device__ __forceinline__ void store_cols_bf16(uint32_t t_addr, float f, __nv_bfloat16 *dst, bool valid) {
#pragma unroll 1
  for (int cc = 0; cc < 64; cc += 32) {
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

__device__ __forceinline__ void zero_cols_bf16(__nv_bfloat16 *dst, int n) {
  uint4 *d = reinterpret_cast<uint4 *>(dst);
  for (int e = 0; e < n / 8; ++e) d[e] = make_uint4(0, 0, 0, 0);
}

struct BwArgs {
  const int *lo;       // [B, S_pad]
  const int *kend;     // [B, nT]
  const int *list;     // (b * nT + tile), longest first
  const float *delta;  // [B, H, S_pad]
  const float *lse2;   // [B, H, S_pad], lse * log2(e), +inf where nothing is visible
  const uint4 *qx;     // [B, H, S_pad] offset rows -lse * sqrt(D) (bf16 hi, mid, lo, 0 x 5)
  const uint4 *dox;    // [B, H, S_pad] offset rows -delta (the same form)
  int *hdr;
  __nv_bfloat16 *out0, *out1;   // dK/dV kernel: dv, dk; dQ kernel: dq
  int B, S, H, nT, S_pad, n_list, n_items;
  float scale_log2;   // log2(e) / sqrt(D)
  float inv_sqrt_d;
  WaitBound wait;
};

struct BwItem {
  int b, h, tile;
};

// Items of one head are consecutive (head-major), each head's tiles longest first, so
// that the CTAs running at the same time share the streamed tiles in L2.
__device__ __forceinline__ BwItem bw_decode(const BwArgs &a, int item) {
  const int e = a.list[item % a.n_list];
  return {e / a.nT, item / a.n_list, e % a.nT};
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
__device__ __forceinline__ int range_tiles(const TileRange &R) { return R.empty() ? 0 : R.last - R.first + 1; }

// ============================================================================= dK/dV
// Item: (b, h, key tile). Resident: K and V. Streamed: Q_j, dO_j, the rows' lo and their
// two offset rows (two stages). Per query tile j:
//   X    = K . Q_j^T - lse sqrt(D)  -> X     (dP^T - delta) = V . dO_j^T - delta -> X
//   P^T  = exp2(X c) (masked)                 -> bf16 in PT
//   dS^T = P^T (dP^T - delta)                 -> bf16 in DS
//   dV  += P^T . dO_j,  dK += dS^T . Q_j      (dK scaled by 1/sqrt(D) in the epilogue)
// The per-query terms are folded into the X products as one more K = 16 slice: a
// constant block of rows [1, 1, 1, 0, ...] times the query rows' [hi, mid, lo, 0, ...]
// (the term as three bf16 parts, exact products, fp32 sums), so the softmax warps read
// no per-query terms from shared memory (that cost about a tenth of the kernel's time).
// c = log2(e) / sqrt(D); rows that see no key carry -1e30 and give P = 0.
// TMEM: X [0, 128) fp32, taken by S^T and dP^T in turn | PT [128, 192) | DS [192, 256)
// (bf16 pairs) | dV [256, 384) | dK [384, 512). The softmax warps read X out first
// thing in each phase, so the next S^T or dP^T runs while they still work on this one;
// P^T and dS^T wait in columns of their own for their dV / dK products. Two MMA issuers:
// warp 9 the X products (S^T, dP^T, alternating), warp 10 the accumulating ones. Warp 11
// idles. (Measured slower, interleaved A/B: a third issuer for the dK products, 1.7 %,
// since they then interleave with the next S^T on the tensor core and delay it; and
// splitting every X product into two 64-query halves, one chain per softmax warpgroup,
// 13 %.)
// stage: Q, dO (128B-swizzled tiles), lo (int32), the offset rows of -lse sqrt(D) and of
// -delta (128 x 16 bytes each: core matrices of 8 rows, 128 bytes apart)
constexpr int KV_OFF_LO = 2 * TILE_BYTES;
constexpr int KV_OFF_QX = KV_OFF_LO + RT_BYTES;
constexpr int KV_OFF_DOX = KV_OFF_QX + BM * XROW_BYTES;
constexpr int KV_STAGE_BYTES = KV_OFF_DOX + BM * XROW_BYTES;
constexpr int KV_STAGE_STRIDE = (KV_STAGE_BYTES + 1023) & ~1023;
// the constant operand of the folded slice: 128 rows of [1, 1, 1, 0 x 5] (K elements
// 0-7), then 128 rows of zeros (K elements 8-15)
constexpr int KV_ONES_BYTES = 2 * BN * XROW_BYTES;
constexpr int KVB_SM_K = 0, KVB_SM_V = TILE_BYTES, KVB_SM_ONES = 2 * TILE_BYTES;
constexpr int KVB_SM_ST = KVB_SM_ONES + KV_ONES_BYTES;
constexpr int KVB_SM_BAR = KVB_SM_ST + 2 * KV_STAGE_STRIDE;
static_assert(KVB_SM_ST % 1024 == 0, "128B-swizzled tiles start on 1024-byte boundaries");
constexpr uint32_t KV_COL_X = 0, KV_COL_PT = 128, KV_COL_DS = 192, KV_COL_DV = 256, KV_COL_DK = 384;

struct KvbBars {
  uint64_t st_full[2], st_empty[2];
  uint64_t own_full, own_empty;
  uint64_t s_full, dp_full, x_free;   // X products and their read-out
  uint64_t p_full, ds_full;           // P^T / dS^T written
  uint64_t pt_free, ds_free;          // dV / dK product done with PT / DS
  uint64_t acc_full, acc_empty;
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item[2];
  uint32_t tmem_base;
  WaitCtl ctl;
  int fill, use, own_issued, own_used;
  uint64_t never;   // the failure test's wait (test instantiation only)
};
constexpr int KVB_SMEM = KVB_SM_BAR + int(sizeof(KvbBars)) + 1024;
static_assert(KVB_SMEM <= 232448, "shared memory budget of one CTA");

template <bool TEST>
__device__ __forceinline__ bool kv_producer(const CUtensorMap *tq, const CUtensorMap *tk, const CUtensorMap *tv,
                                            const CUtensorMap *tdo, const BwArgs &a, uint8_t *smem, KvbBars *bars) {
  WaitCtl *abort = &bars->ctl;
  int fill = 0, own = 0;
  bool ok = true;
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
    const int n = range_tiles(R);
    if (!(ok = mbar_wait(&bars->own_empty, (it & 1) ^ 1, abort))) break;
    mbar_arrive_expect_tx(&bars->own_full, 2 * TILE_BYTES);
    load_tile(tk, &bars->own_full, smem + KVB_SM_K, I.h, I.tile * BN, I.b);
    load_tile(tv, &bars->own_full, smem + KVB_SM_V, I.h, I.tile * BN, I.b);
    ++own;
    const size_t rowbase = (size_t(I.b) * a.H + I.h) * a.S_pad;
    for (int j = 0; j < n && ok; ++j) {
      const int st = fill & 1;
      if (!(ok = mbar_wait(&bars->st_empty[st], ((fill >> 1) & 1) ^ 1, abort))) break;
      mbar_arrive_expect_tx(&bars->st_full[st], KV_STAGE_BYTES);
      uint8_t *dst = smem + KVB_SM_ST + st * KV_STAGE_STRIDE;
      const int row0 = (R.first + j) * BM;
      load_tile(tq, &bars->st_full[st], dst, I.h, row0, I.b);
      load_tile(tdo, &bars->st_full[st], dst + TILE_BYTES, I.h, row0, I.b);
      bulk_load(dst + KV_OFF_LO, a.lo + size_t(I.b) * a.S_pad + row0, RT_BYTES, &bars->st_full[st]);
      bulk_load(dst + KV_OFF_QX, a.qx + rowbase + row0, BM * XROW_BYTES, &bars->st_full[st]);
      bulk_load(dst + KV_OFF_DOX, a.dox + rowbase + row0, BM * XROW_BYTES, &bars->st_full[st]);
      ++fill;
    }
    if (!ok) break;
    if constexpr (TEST) {
      if (it == 0 && !(ok = test_expiry_wait(&bars->never, abort))) break;
    }
  }
  bars->fill = fill;
  bars->own_issued = own;
  return ok;
}

// Issuer of the X products: S^T(j) - lse sqrt(D) = K Q_j^T + ones qx_j^T, then
// dP^T(j) - delta = V dO_j^T + ones dox_j^T, each once the softmax warps have read the
// previous X product out (x_free). Releases K and V after the item's last product.
__device__ __forceinline__ bool kv_x_issuer(const BwArgs &a, uint8_t *smem, KvbBars *bars, uint32_t tmem, int lane) {
  WaitCtl *abort = &bars->ctl;
  const uint32_t k_s = smem_u32(smem + KVB_SM_K), v_s = smem_u32(smem + KVB_SM_V);
  const uint32_t st0 = smem_u32(smem + KVB_SM_ST);
  // ones: K elements 8-15 are the zero rows behind the 128 rows of ones; the offset rows'
  // K elements 8-15 re-read elements 0-7 (lbo 0), which the zeros cancel exactly
  const uint64_t ones_desc = sdesc_plain(smem_u32(smem + KVB_SM_ONES), BN * XROW_BYTES, 8 * XROW_BYTES);
  int use = 0, own = 0, n_x = 0;
  int seen = 0;   // stages whose arrival this warp has observed (the abort path waits for the rest)
  bool ok = true;
  auto x_product = [&](uint32_t a_s, uint32_t b_s, uint32_t off_s, uint64_t *done) -> bool {
    if (n_x > 0 && !mbar_wait(&bars->x_free, (n_x - 1) & 1, abort)) return false;
    tc_fence_after();
    if (lane == 0) {
      mma_ss(tmem + KV_COL_X, ones_desc, sdesc_plain(off_s, 0, 8 * XROW_BYTES), IDESC_128_KK, 0u);
      mma_tile_kk(tmem + KV_COL_X, a_s, b_s, true);
      mma_commit(done);
    }
    __syncwarp();
    ++n_x;
    return true;
  };
  for (int it = 0; ok; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const BwItem I = bw_decode(a, item);
    const int n = range_tiles(dkdv_range(a, I));
    if (!(ok = mbar_wait(&bars->own_full, it & 1, abort))) break;
    ++own;
    for (int j = 0; j < n && ok; ++j) {
      const int k = use + j;
      if (!(ok = mbar_wait(&bars->st_full[k & 1], (k >> 1) & 1, abort))) break;
      seen = k + 1;
      const uint32_t q_s = st0 + uint32_t(k & 1) * KV_STAGE_STRIDE;
      if (!(ok = x_product(k_s, q_s, q_s + KV_OFF_QX, &bars->s_full))) break;                 // S^T(j)
      if (!(ok = x_product(v_s, q_s + TILE_BYTES, q_s + KV_OFF_DOX, &bars->dp_full))) break;  // dP^T(j)
    }
    if (!ok) break;
    use += n;
    if (lane == 0) mma_commit(&bars->own_empty);
    __syncwarp();
  }
  if (lane == 0) {
    bars->use = seen;
    bars->own_used = own;
  }
  return ok;
}

// Issuer of the accumulating products: dV += P^T(j) dO_j once P^T is written, dK +=
// dS^T(j) Q_j once dS^T is written; then releases the stage (its lo terms were read,
// and the X products that read its offset rows had completed, before dS^T was
// signalled). The first products of an item overwrite dV and dK once
// the previous item's have been read out.
__device__ __forceinline__ bool kv_acc_issuer(const BwArgs &a, uint8_t *smem, KvbBars *bars, uint32_t tmem,
                                              int lane) {
  WaitCtl *abort = &bars->ctl;
  const uint32_t st0 = smem_u32(smem + KVB_SM_ST);
  int use = 0;
  uint32_t pf_par = 0, dsf_par = 0, ae_par = 1;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const BwItem I = bw_decode(a, item);
    const int n = range_tiles(dkdv_range(a, I));
    for (int j = 0; j < n && ok; ++j) {
      const int k = use + j;
      if (!(ok = mbar_wait(&bars->st_full[k & 1], (k >> 1) & 1, abort))) break;
      const uint32_t q_s = st0 + uint32_t(k & 1) * KV_STAGE_STRIDE;
      if (!(ok = mbar_wait(&bars->p_full, pf_par, abort))) break;
      pf_par ^= 1;
      if (j == 0) {
        if (!(ok = mbar_wait(&bars->acc_empty, ae_par, abort))) break;
        ae_par ^= 1;
      }
      tc_fence_after();
      if (lane == 0) {
        mma_tile_ts_packed(tmem + KV_COL_DV, tmem + KV_COL_PT, q_s + TILE_BYTES, j > 0);   // dV += P^T dO
        mma_commit(&bars->pt_free);
      }
      __syncwarp();
      if (!(ok = mbar_wait(&bars->ds_full, dsf_par, abort))) break;
      dsf_par ^= 1;
      tc_fence_after();
      if (lane == 0) {
        mma_tile_ts_packed(tmem + KV_COL_DK, tmem + KV_COL_DS, q_s, j > 0);   // dK += dS^T Q
        mma_commit(&bars->ds_free);
        mma_commit(&bars->st_empty[k & 1]);
      }
      __syncwarp();
    }
    if (!ok) break;
    use += n;
    if (lane == 0 && n > 0) mma_commit(&bars->acc_full);
    __syncwarp();
  }
  return ok;
}

// Softmax warpgroup w of the dK/dV kernel: thread = key row `row`; query columns
// [64 w, 64 w + 64) of every streamed tile.
__device__ __forceinline__ bool kv_softmax(const BwArgs &a, uint8_t *smem, KvbBars *bars, uint32_t tmem, int w,
                                           int warp, int lane) {
  WaitCtl *abort = &bars->ctl;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = uint32_t(quarter * 32) << 16;
  const uint32_t tX = tmem + lane_off + KV_COL_X + 64 * w;
  const uint32_t tPT = tmem + lane_off + KV_COL_PT + 32 * w;
  const uint32_t tDS = tmem + lane_off + KV_COL_DS + 32 * w;
  const uint64_t c2 = f2_pack(a.scale_log2, a.scale_log2);
  uint32_t sf_par = 0, dpf_par = 0, af_par = 0;
  int use = 0, n_done = 0;   // n_done: query tiles finished (all items), = dV / dK products issued before
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const BwItem I = bw_decode(a, item);
    const TileRange R = dkdv_range(a, I);
    const int n = range_tiles(R);
    const int k0 = I.tile * BN, jk = k0 + row;   // this thread's key
    for (int j = 0; j < n; ++j, ++use, ++n_done) {
      const int st = use & 1;
      const uint8_t *stage = smem + KVB_SM_ST + st * KV_STAGE_STRIDE;
      const int *lo_q = reinterpret_cast<const int *>(stage + KV_OFF_LO);
      const int q0 = (R.first + j) * BM;

      // ---- P phase
      if (!(ok = mbar_wait(&bars->s_full, sf_par, abort))) break;
      sf_par ^= 1;
      // the stage's lo terms arrived by bulk copy: observe the stage's barrier
      if (!(ok = mbar_wait(&bars->st_full[st], (use >> 1) & 1, abort))) break;
      tc_fence_after();
      float p[64];
      {
        uint32_t sv[64];
        tmem_ld32(tX, sv);
        tmem_ld32(tX + 32, sv + 32);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->x_free);   // S^T is in registers: X may take dP^T
#pragma unroll
        for (int e = 0; e < 64; ++e) p[e] = __uint_as_float(sv[e]);
      }
      // Key jk is visible from query q0 + q iff lo[q0 + q] <= jk <= q0 + q; lo is
      // non-decreasing, so these q form one range [q_from, q_to).
      const bool full = lo_q[BM - 1] <= k0 && k0 + BN - 1 <= q0;
      int q_from = 0, q_to = BM;
      if (!full) {
        q_from = jk - q0;
        int lo_i = 0, hi_i = BM;
        while (lo_i < hi_i) {
          const int m = (lo_i + hi_i) >> 1;
          if (lo_q[m] <= jk) lo_i = m + 1; else hi_i = m;
        }
        q_to = lo_i;
      }
      q_from -= 64 * w;
      q_to -= 64 * w;
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        float x0, x1;
        f2_unpack(f2_mul(f2_pack(p[e], p[e + 1]), c2), x0, x1);
        p[e] = ex2_approx(x0);
        p[e + 1] = ex2_approx(x1);
      }
      if (!full) {
#pragma unroll
        for (int q = 0; q < 64; ++q)
          if (q < q_from || q >= q_to) p[q] = 0.f;
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = pack_bf16x2(p[2 * e], p[2 * e + 1]);
        // PT belongs to the previous dV product until it completes
        if (n_done > 0) {
          if (!(ok = mbar_wait(&bars->pt_free, (n_done - 1) & 1, abort))) break;
          tc_fence_after();
        }
        tmem_st16(tPT, pk);
        tmem_st16(tPT + 16, pk + 16);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);

      // ---- dS phase
      if (!(ok = mbar_wait(&bars->dp_full, dpf_par, abort))) break;
      dpf_par ^= 1;
      tc_fence_after();
      uint32_t dk[32];
      {
        uint32_t dv[64];
        tmem_ld32(tX, dv);
        tmem_ld32(tX + 32, dv + 32);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->x_free);   // dP^T is in registers: X may take S^T(j+1)
#pragma unroll
        for (int e = 0; e < 32; ++e)
        {
          float s0, s1;
          f2_unpack(f2_mul(f2_pack(p[2 * e], p[2 * e + 1]),
                           f2_pack(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1]))), s0, s1);
          dk[e] = pack_bf16x2(s0, s1);
        }
      }
      // DS belongs to the previous dK product until it completes
      if (n_done > 0) {
        if (!(ok = mbar_wait(&bars->ds_free, (n_done - 1) & 1, abort))) break;
        tc_fence_after();
      }
      tmem_st16(tDS, dk);
      tmem_st16(tDS + 16, dk + 16);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ds_full);
    }
    if (!ok) break;

    // epilogue: both warpgroups write half of the columns of dV and of dK (dK scaled by 1/sqrt(D))
    __nv_bfloat16 *dv_row = a.out0 + ((size_t(I.b) * a.S + jk) * a.H + I.h) * HD + 64 * w;
    __nv_bfloat16 *dk_row = a.out1 + ((size_t(I.b) * a.S + jk) * a.H + I.h) * HD + 64 * w;
    if (n > 0) {
      if (!(ok = mbar_wait(&bars->acc_full, af_par, abort))) break;
      af_par ^= 1;
      tc_fence_after();
      store_cols_bf16(tmem + lane_off + KV_COL_DV + 64 * w, 1.f, dv_row, jk < a.S);
      store_cols_bf16(tmem + lane_off + KV_COL_DK + 64 * w, a.inv_sqrt_d, dk_row, jk < a.S);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_empty);
    } else if (jk < a.S) {
      zero_cols_bf16(dv_row, 64);
      zero_cols_bf16(dk_row, 64);
    }
  }
  return ok;
}

template <bool TEST>
__global__ void __launch_bounds__(BW_THREADS, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo, const BwArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  KvbBars *bars = reinterpret_cast<KvbBars *>(smem + KVB_SM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->st_full[s], 1);
      mbar_init(&bars->st_empty[s], 1);
      mbar_init(&bars->item_full[s], 1);
      mbar_init(&bars->item_empty[s], 10);   // softmax 8 + MMA 2 warps
    }
    mbar_init(&bars->own_full, 1);
    mbar_init(&bars->own_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->x_free, 8);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->pt_free, 1);
    mbar_init(&bars->ds_free, 1);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->drain, 2);
    if (TEST) mbar_init(&bars->never, 1);
    bars->ctl.init(a.wait);
    bars->fill = bars->use = bars->own_issued = bars->own_used = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < KV_ONES_BYTES / 16) {   // the folded slice's constant operand
    const uint32_t one = 0x3F80u;           // bf16 1.0
    reinterpret_cast<uint4 *>(smem + KVB_SM_ONES)[threadIdx.x] =
        threadIdx.x < BN ? make_uint4(one | (one << 16), one, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (warp == BW_MMA) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == BW_PRODUCER && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool ok = true;
  if (warp < BW_PRODUCER) {
    ok = kv_softmax(a, smem, bars, tmem, warp >> 2, warp, lane);
  } else if (warp == BW_PRODUCER) {
    if (lane == 0) ok = kv_producer<TEST>(&tq, &tk, &tv, &tdo, a, smem, bars);
    __syncwarp();
  } else if (warp == BW_MMA) {
    ok = kv_x_issuer(a, smem, bars, tmem, lane);
  } else if (warp == BW_MMA2) {
    ok = kv_acc_issuer(a, smem, bars, tmem, lane);
  }

  if (!ok) {
    bars->ctl.abort = 1;
    raise_error(a.hdr + HDR_ERR, ERRBIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (bars->ctl.abort) {
    if (warp == BW_PRODUCER && lane == 0) {
      for (int k = bars->use; k < bars->fill; ++k) bounded_wait_plain(&bars->st_full[k & 1], (k >> 1) & 1);
      if (bars->own_issued > bars->own_used) bounded_wait_plain(&bars->own_full, (bars->own_issued - 1) & 1);
    }
    if ((warp == BW_MMA || warp == BW_MMA2) && lane == 0) {
      mma_commit(&bars->drain);
      bounded_wait_plain(&bars->drain, 0);
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

// ============================================================================= dQ
// Item: (b, h, query tile). Resident: Q and dO; the rows' lo / lse2 / delta live in
// registers (thread = query row). Streamed: K_j (ring of three) and V_j (ring of two).
// Per key tile g (counted over all items of the CTA):
//   S    = Q . K_g^T  -> X                 dP = dO . V_g^T -> Y_{g % 2}
//   P    = exp2(S c - lse2) (masked),  dS = P (dP - delta)  -> bf16 over its own dP
//   dQ  += dS . K_g   (C; scaled by 1/sqrt(D) in the epilogue)
// TMEM: X [0, 128), Y0 [128, 256), Y1 [256, 384), C [384, 512). X is free as soon as the
// softmax warps have read S out, so S(g + 1) runs while they work on tile g; the dP
// products are double-buffered, so dP(g + 1) runs before the dS phase of g ends (it
// waits only for dQ(g - 1), the last reader of its slot). Three MMA issuers: warp 9 runs
// dQ(g), warp 10 dP(g), warp 11 S(g). Deterministic: every dQ row is summed by one CTA
// in a fixed order.
constexpr int DQ_KSTAGES = 3, DQ_VSTAGES = 2;
constexpr int DQ_SM_Q = 0, DQ_SM_DO = TILE_BYTES, DQ_SM_K = 2 * TILE_BYTES;
constexpr int DQ_SM_V = DQ_SM_K + DQ_KSTAGES * TILE_BYTES;
constexpr int DQ_SM_BAR = DQ_SM_V + DQ_VSTAGES * TILE_BYTES;
constexpr uint32_t DQ_COL_X = 0, DQ_COL_Y = 128, DQ_COL_C = 384;

struct DqBars {
  uint64_t k_full[DQ_KSTAGES], k_empty[DQ_KSTAGES], v_full[DQ_VSTAGES], v_empty[DQ_VSTAGES];
  uint64_t own_full, own_empty;
  uint64_t s_full, x_free;   // S(g) written to X; the softmax warps have read it out
  // slot Y_{g % 2}: dP(g) written; dS(g) written over it; dQ(g), its last reader, done.
  // Every waiter's next phase on one of them needs an action the waiter takes after its
  // wait (S(g + 1) after x_free(g), dP(g + 2) after y_free(g), dQ(g) after ds_full(g)),
  // so no barrier can run two phases ahead of its waiter.
  uint64_t dp_full[2], ds_full[2], y_free[2];
  uint64_t acc_full, acc_empty;
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item[2];
  uint32_t tmem_base;
  WaitCtl ctl;
  int k_fill, k_use, v_fill, v_use, own_issued, own_used;
  uint64_t never;   // the failure test's wait (test instantiation only)
};
constexpr int DQ_SMEM = DQ_SM_BAR + int(sizeof(DqBars)) + 1024;
static_assert(DQ_SMEM <= 232448, "shared memory budget of one CTA");

template <bool TEST>
__device__ __forceinline__ bool dq_producer(const CUtensorMap *tq, const CUtensorMap *tk, const CUtensorMap *tv,
                                            const CUtensorMap *tdo, const BwArgs &a, uint8_t *smem, DqBars *bars) {
  WaitCtl *abort = &bars->ctl;
  int k_fill = 0, v_fill = 0, own = 0;
  bool ok = true;
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
    const int n = range_tiles(R);
    if (!(ok = mbar_wait(&bars->own_empty, (it & 1) ^ 1, abort))) break;
    mbar_arrive_expect_tx(&bars->own_full, 2 * TILE_BYTES);
    load_tile(tq, &bars->own_full, smem + DQ_SM_Q, I.h, I.tile * BM, I.b);
    load_tile(tdo, &bars->own_full, smem + DQ_SM_DO, I.h, I.tile * BM, I.b);
    ++own;
    // K_j, then V_j: each ring is refilled as soon as its oldest tile is released
    for (int j = 0; j < n && ok; ++j) {
      const int row0 = (R.first + j) * BN;
      const int ks = k_fill % DQ_KSTAGES;
      if (!(ok = mbar_wait(&bars->k_empty[ks], ((k_fill / DQ_KSTAGES) & 1) ^ 1, abort))) break;
      mbar_arrive_expect_tx(&bars->k_full[ks], TILE_BYTES);
      load_tile(tk, &bars->k_full[ks], smem + DQ_SM_K + ks * TILE_BYTES, I.h, row0, I.b);
      ++k_fill;
      const int vs = v_fill % DQ_VSTAGES;
      if (!(ok = mbar_wait(&bars->v_empty[vs], ((v_fill / DQ_VSTAGES) & 1) ^ 1, abort))) break;
      mbar_arrive_expect_tx(&bars->v_full[vs], TILE_BYTES);
      load_tile(tv, &bars->v_full[vs], smem + DQ_SM_V + vs * TILE_BYTES, I.h, row0, I.b);
      ++v_fill;
    }
    if (!ok) break;
    // failure test only: wait, with this item's copies and products in flight, for a
    // phase that never completes (the short test bound makes the wait run out)
    if constexpr (TEST) {
      if (it == 0 && !(ok = test_expiry_wait(&bars->never, abort))) break;
    }
  }
  bars->k_fill = k_fill;
  bars->v_fill = v_fill;
  bars->own_issued = own;
  return ok;
}

// MMA chains of the dQ kernel, one issuing warp each (g = the CTA's running key-tile
// count, slot s = g % 2):
//   chain 0 (warp 9):  dQ += dS(g) K_g once the softmax has written dS(g) over Y_s; then
//                      releases K_g and Y_s (on completion);
//   chain 1 (warp 10): dP(g) = dO V_g^T into Y_s once dQ(g - 2) has released it;
//   chain 2 (warp 11): S(g) = Q K_g^T into X once the softmax has read S(g - 1) out.
__device__ __forceinline__ bool dq_mma(const BwArgs &a, uint8_t *smem, DqBars *bars, uint32_t tmem, int chain,
                                       int lane) {
  WaitCtl *abort = &bars->ctl;
  const uint32_t q_s = smem_u32(smem + DQ_SM_Q), do_s = smem_u32(smem + DQ_SM_DO);
  const uint32_t k0_s = smem_u32(smem + DQ_SM_K), v0_s = smem_u32(smem + DQ_SM_V);
  int k_use = 0, v_use = 0, own = 0, g = 0;
  int k_seen = 0;   // K stages whose arrival chain 2 has observed (the abort path waits for the rest)
  uint32_t ae_par = 1;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const BwItem I = bw_decode(a, item);
    const int n = range_tiles(dq_range(a, I));
    if (chain != 0) {   // Q (S products) and dO (dP products) resident
      if (!(ok = mbar_wait(&bars->own_full, it & 1, abort))) break;
      ++own;
    }
    const int kb = k_use;
    auto k_stage = [&](int j) { return (kb + j) % DQ_KSTAGES; };
    auto k_par = [&](int j) { return uint32_t((kb + j) / DQ_KSTAGES) & 1u; };
    if (chain == 0) {
      for (int j = 0; j < n && ok; ++j) {
        const int gg = g + j, s = gg & 1;
        if (!(ok = mbar_wait(&bars->ds_full[s], uint32_t(gg >> 1) & 1u, abort))) break;
        if (j == 0) {
          if (!(ok = mbar_wait(&bars->acc_empty, ae_par, abort))) break;
          ae_par ^= 1;
        }
        // K_g arrived (chain 2 saw it before S(g)); the stage stays until this chain releases it
        if (!(ok = mbar_wait(&bars->k_full[k_stage(j)], k_par(j), abort))) break;
        tc_fence_after();
        if (lane == 0) {
          mma_tile_ts(tmem + DQ_COL_C, tmem + DQ_COL_Y + uint32_t(s) * 128,
                      k0_s + uint32_t(k_stage(j)) * TILE_BYTES, j > 0);   // dQ += dS K
          mma_commit(&bars->k_empty[k_stage(j)]);
          mma_commit(&bars->y_free[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0 && n > 0) mma_commit(&bars->acc_full);
      __syncwarp();
    } else if (chain == 2) {
      for (int j = 0; j < n && ok; ++j) {
        const int gg = g + j;
        if (!(ok = mbar_wait(&bars->k_full[k_stage(j)], k_par(j), abort))) break;
        k_seen = kb + j + 1;
        if (gg > 0 && !(ok = mbar_wait(&bars->x_free, uint32_t(gg - 1) & 1u, abort))) break;
        tc_fence_after();
        if (lane == 0) {
          mma_tile_kk(tmem + DQ_COL_X, q_s, k0_s + uint32_t(k_stage(j)) * TILE_BYTES, false);   // S = Q K^T
          mma_commit(&bars->s_full);
        }
        __syncwarp();
      }
      if (!ok) break;
    } else {
      for (int j = 0; j < n && ok; ++j, ++v_use) {
        const int gg = g + j, s = gg & 1;
        const int vs = v_use % DQ_VSTAGES;
        if (!(ok = mbar_wait(&bars->v_full[vs], (v_use / DQ_VSTAGES) & 1, abort))) break;
        if (gg >= 2 && !(ok = mbar_wait(&bars->y_free[s], uint32_t((gg - 2) >> 1) & 1u, abort))) break;
        tc_fence_after();
        if (lane == 0) {
          mma_tile_kk(tmem + DQ_COL_Y + uint32_t(s) * 128, do_s, v0_s + uint32_t(vs) * TILE_BYTES,
                      false);   // dP = dO V^T
          mma_commit(&bars->dp_full[s]);
          mma_commit(&bars->v_empty[vs]);
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    k_use = kb + n;
    g += n;
    if (chain != 0) {
      if (lane == 0) mma_commit(&bars->own_empty);
      __syncwarp();
    }
  }
  if (lane == 0 && chain == 2) {
    bars->k_use = k_seen;
    bars->own_used = own;
  }
  if (lane == 0 && chain == 1) bars->v_use = v_use;
  return ok;
}

// Softmax warpgroup w of the dQ kernel: thread = query row `row`; key columns
// [64 w, 64 w + 64) of every streamed tile.
__device__ __forceinline__ bool dq_softmax(const BwArgs &a, DqBars *bars, uint32_t tmem, int w, int warp, int lane) {
  WaitCtl *abort = &bars->ctl;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = uint32_t(quarter * 32) << 16;
  const uint32_t tX = tmem + lane_off + DQ_COL_X + 64 * w;
  const uint64_t c2 = f2_pack(a.scale_log2, a.scale_log2);
  uint32_t af_par = 0;
  int g = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const BwItem I = bw_decode(a, item);
    const TileRange R = dq_range(a, I);
    const int n = range_tiles(R);
    const int q0 = I.tile * BM, i = q0 + row;   // this thread's query
    const int *lr = a.lo + size_t(I.b) * a.S_pad;
    const size_t rowterm = (size_t(I.b) * a.H + I.h) * a.S_pad + i;
    const int lo_i = lr[i];
    const int lo_last = lr[q0 + BM - 1];
    const float l2 = a.lse2[rowterm], dl = a.delta[rowterm];
    const uint64_t nl2 = f2_pack(-l2, -l2), ndl2 = f2_pack(-dl, -dl);
    for (int j = 0; j < n; ++j, ++g) {
      const int k0 = (R.first + j) * BN;
      const uint32_t tY = tmem + lane_off + DQ_COL_Y + uint32_t(g & 1) * 128 + 64 * w;
      const bool full = lo_last <= k0 && k0 + BN - 1 <= q0;
      // visible keys of query i: lo_i <= key <= i, i.e. columns [c_from, c_to) here
      const int c_from = lo_i - k0 - 64 * w, c_to = i - k0 - 64 * w + 1;

      // ---- P phase: read S out of X (which then takes S(g + 1)), P in registers
      if (!(ok = mbar_wait(&bars->s_full, uint32_t(g) & 1u, abort))) break;
      tc_fence_after();
      float p[64];
      {
        uint32_t sv[64];
        tmem_ld16(tX, sv);
        tmem_ld16(tX + 16, sv + 16);
        tmem_ld16(tX + 32, sv + 32);
        tmem_ld16(tX + 48, sv + 48);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->x_free);
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2, nl2), x0, x1);
          p[e] = ex2_approx(x0);
          p[e + 1] = ex2_approx(x1);
        }
      }
      if (!full) {
#pragma unroll
        for (int cc = 0; cc < 64; ++cc)
          if (cc < c_from || cc >= c_to) p[cc] = 0.f;
      }

      // ---- dS phase: dS over the dP columns just read (each 16-column block's first 8
      // columns take its 16 bf16 values; no block is written before it has been read)
      if (!(ok = mbar_wait(&bars->dp_full[g & 1], uint32_t(g >> 1) & 1u, abort))) break;
      tc_fence_after();
      uint32_t dv[64];
      tmem_ld16(tY, dv);
      tmem_ld16(tY + 16, dv + 16);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        if (ch == 0 || ch == 2) {
          tmem_ld_wait();
          if (ch == 0) {
            tmem_ld16(tY + 32, dv + 32);
            tmem_ld16(tY + 48, dv + 48);
          }
        }
        uint32_t dk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int q = ch * 16 + 2 * e;
          float s0, s1;
          f2_unpack(f2_mul(f2_pack(p[q], p[q + 1]),
                           f2_add(f2_pack(__uint_as_float(dv[q]), __uint_as_float(dv[q + 1])), ndl2)), s0, s1);
          dk[e] = pack_bf16x2(s0, s1);
        }
        tmem_st8(tY + ch * 16, dk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ds_full[g & 1]);
    }
    if (!ok) break;

    __nv_bfloat16 *dst = a.out0 + ((size_t(I.b) * a.S + i) * a.H + I.h) * HD + 64 * w;
    if (n > 0) {
      if (!(ok = mbar_wait(&bars->acc_full, af_par, abort))) break;
      af_par ^= 1;
      tc_fence_after();
      store_cols_bf16(tmem + lane_off + DQ_COL_C + 64 * w, a.inv_sqrt_d, dst, i < a.S);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_empty);
    } else if (i < a.S) {
      zero_cols_bf16(dst, 64);
    }
  }
  return ok;
}

template <bool TEST>
__global__ void __launch_bounds__(BW_THREADS, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo, const BwArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DqBars *bars = reinterpret_cast<DqBars *>(smem + DQ_SM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < DQ_KSTAGES; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < DQ_VSTAGES; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->dp_full[s], 1);
      mbar_init(&bars->ds_full[s], 8);
      mbar_init(&bars->y_free[s], 1);
      mbar_init(&bars->item_full[s], 1);
      mbar_init(&bars->item_empty[s], 11);  // softmax 8 + MMA 3 warps
    }
    mbar_init(&bars->own_full, 1);
    mbar_init(&bars->own_empty, 2);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->x_free, 8);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->drain, 3);
    if (TEST) mbar_init(&bars->never, 1);
    bars->ctl.init(a.wait);
    bars->k_fill = bars->k_use = bars->v_fill = bars->v_use = bars->own_issued = bars->own_used = 0;
    fence_mbar_init();
  }
  if (warp == BW_MMA) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == BW_PRODUCER && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool ok = true;
  if (warp < BW_PRODUCER) {
    ok = dq_softmax(a, bars, tmem, warp >> 2, warp, lane);
  } else if (warp == BW_PRODUCER) {
    if (lane == 0) ok = dq_producer<TEST>(&tq, &tk, &tv, &tdo, a, smem, bars);
    __syncwarp();
  } else if (warp == BW_MMA || warp == BW_MMA2 || warp == BW_MMA3) {
    ok = dq_mma(a, smem, bars, tmem, warp - BW_MMA, lane);
  }

  if (!ok) {
    bars->ctl.abort = 1;
    raise_error(a.hdr + HDR_ERR, ERRBIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (bars->ctl.abort) {
    if (warp == BW_PRODUCER && lane == 0) {
      for (int k = bars->k_use; k < bars->k_fill; ++k)
        bounded_wait_plain(&bars->k_full[k % DQ_KSTAGES], (k / DQ_KSTAGES) & 1);
      for (int k = bars->v_use; k < bars->v_fill; ++k)
        bounded_wait_plain(&bars->v_full[k % DQ_VSTAGES], (k / DQ_VSTAGES) & 1);
      if (bars->own_issued > bars->own_used) bounded_wait_plain(&bars->own_full, (bars->own_issued - 1) & 1);
    }
    if ((warp == BW_MMA || warp == BW_MMA2 || warp == BW_MMA3) && lane == 0) {
      mma_commit(&bars->drain);
      bounded_wait_plain(&bars->drain, 0);
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

BwArgs bw_args(const Problem &p, void *workspace, const int *list) {
  const Workspace w = Workspace::layout(p.B, p.S, p.H);
  char *base = static_cast<char *>(workspace);
  BwArgs a;
  a.lo = reinterpret_cast<const int *>(base + w.off_lo);
  a.kend = reinterpret_cast<const int *>(base + w.off_kend);
  a.list = list;
  a.delta = reinterpret_cast<const float *>(base + w.off_delta);
  a.lse2 = reinterpret_cast<const float *>(base + w.off_lse2);
  a.qx = reinterpret_cast<const uint4 *>(base + w.off_qx);
  a.dox = reinterpret_cast<const uint4 *>(base + w.off_dox);
  a.hdr = reinterpret_cast<int *>(base + w.off_hdr);
  a.out0 = a.out1 = nullptr;
  a.B = p.B;
  a.S = p.S;
  a.H = p.H;
  a.nT = w.nT;
  a.S_pad = w.S_pad;
  a.n_list = p.B * w.nT;
  a.n_items = a.n_list * p.H;
  a.scale_log2 = 1.4426950408889634f / sqrtf(float(HD));
  a.inv_sqrt_d = 1.f / sqrtf(float(HD));
  a.wait = wait_bound();
  return a;
}

}  // namespace

cudaError_t launch_dkdv(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tdo,
                        void *dk, void *dv, const Problem &p, void *workspace, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done[2] = {{0}, {0}};
  const bool test = wait_bound().test != 0;
  {
    const void *kern = test ? reinterpret_cast<const void *>(dkdv_kernel<true>)
                            : reinterpret_cast<const void *>(dkdv_kernel<false>);
    const cudaError_t e = smem_attr_once(kern, KVB_SMEM, attr_done[test ? 1 : 0]);
    if (e != cudaSuccess) return e;
  }
  const Workspace w = Workspace::layout(p.B, p.S, p.H);
  BwArgs a = bw_args(p, workspace, reinterpret_cast<const int *>(static_cast<char *>(workspace) + w.off_list_kv));
  a.out0 = static_cast<__nv_bfloat16 *>(dv);
  a.out1 = static_cast<__nv_bfloat16 *>(dk);
  const int grid = a.n_items < p.num_sms ? a.n_items : p.num_sms;
  if (test) dkdv_kernel<true><<<grid, BW_THREADS, KVB_SMEM, stream>>>(tq, tk, tv, tdo, a);
  else dkdv_kernel<false><<<grid, BW_THREADS, KVB_SMEM, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

cudaError_t launch_dq(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tdo,
                      void *dq, const Problem &p, void *workspace, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done[2] = {{0}, {0}};
  const bool test = wait_bound().test != 0;
  {
    const void *kern = test ? reinterpret_cast<const void *>(dq_kernel<true>)
                            : reinterpret_cast<const void *>(dq_kernel<false>);
    const cudaError_t e = smem_attr_once(kern, DQ_SMEM, attr_done[test ? 1 : 0]);
    if (e != cudaSuccess) return e;
  }
  const Workspace w = Workspace::layout(p.B, p.S, p.H);
  BwArgs a = bw_args(p, workspace, reinterpret_cast<const int *>(static_cast<char *>(workspace) + w.off_list_q));
  a.out0 = static_cast<__nv_bfloat16 *>(dq);
  const int grid = a.n_items < p.num_sms ? a.n_items : p.num_sms;
  if (test) dq_kernel<true><<<grid, BW_THREADS, DQ_SMEM, stream>>>(tq, tk, tv, tdo, a);
  else dq_kernel<false><<<grid, BW_THREADS, DQ_SMEM, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}
}  // namespace lwm
