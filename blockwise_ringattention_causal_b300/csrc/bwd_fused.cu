// Backward pass in one kernel: dK, dV and dQ from a single recomputation of the
// probabilities (five tensor-core products per visible tile pair instead of the seven
// that separate dK/dV and dQ kernels need).
//
// Gradients of exact softmax attention, recomputed block by block from the saved
// log-sum-exp (the blockwise method of the LWM pages: "World Model on Million-Length
// Video And Language With Blockwise RingAttention", deep-dive page, section
// "RingAttention 为什么必要"):
//   p_ij = exp(s_ij - lse_i),  dp_ij = dout_i . v_j,  ds_ij = p_ij (dp_ij - delta_i)
//   dv_j = sum_i p_ij dout_i,  dk_j = sum_i ds_ij q_i / sqrt(D),  dq_i = sum_j ds_ij k_j / sqrt(D)
//
// Item: (b, h, 128-key tile), taken longest-first through an atomic ticket by one
// persistent CTA per SM. K and V of the tile stay resident in shared memory; the
// query rows that see the tile stream through in 64-row halves u = 0, 1, 2, ...
// (Q, dO and the rows' lo / lse / delta terms). Per half u, with region r = u & 1:
//   S^T_u  = K . Q_u^T, dP^T_u = V . dO_u^T          (128 keys x 64 queries, fp32 TMEM)
//   P^T, dS^T (softmax warpgroup r, one key row per thread) -> bf16 TMEM, and dS^T
//   also into shared memory
//   dV += P^T_u . dO_u,  dK += dS^T_u . Q_u           (TMEM accumulators)
//   dQ^T_u = K^T . dS^T_u                             (128 dims x 64 queries, fp32 TMEM)
// and four readout warps, each owning 32 of the head dims, stage dQ^T_u in shared
// memory as [16 queries x 32 dims] fp32 blocks that tensor bulk reduce-add copies add
// into an fp32 accumulator [B, H, S_pad, D] in global memory (the addition happens in
// L2). A final pass converts it to bf16 dq. The
// order of the fp32 additions depends on scheduling, so dq is not bitwise reproducible
// from run to run (dk and dv are).
//
// Warp roles: 0-3 softmax of region 0, 4-7 softmax of region 1, 8-11 dQ readout (warp
// w reads TMEM lanes 32 (w % 4) ...), 12 TMA producer, 13 MMA issuer (128 registers
// per thread: 14 warps put 4 warps on some SM sub-partitions).
// TMEM columns (fp32):
//   r*128 + [0, 64)   S^T_r, then P^T_r and dS^T_r (bf16, 8 columns per 16 queries,
//                     alternating: P^T q0-15, dS^T q0-15, P^T q16-31, ...)
//   r*128 + [64, 128) dP^T_r, then dQ^T_r
//   256 dV, 384 dK
#include "common.cuh"
#include "kernels.h"

namespace lwm {
namespace {

constexpr int FB_WARPS = 14;
constexpr int FB_THREADS = FB_WARPS * 32;
constexpr int FB_READ0 = 8;
constexpr int FB_PRODUCER = 12;
constexpr int FB_MMA = 13;
constexpr int QH = 64;                        // queries per streamed half tile
constexpr int QH_BOX = QH * 128;              // 64 rows x 64 dims, 128B-swizzled: 8 KiB
constexpr int QH_BYTES = 2 * QH_BOX;          // 64 rows x 128 dims: 16 KiB
constexpr int RT_BYTES = QH * 4;              // 64 row terms (int32 / fp32)
constexpr int FB_STAGES = 3;
constexpr int FB_STAGE_BYTES = 2 * QH_BYTES + 3 * RT_BYTES;   // Q, dO, lo, lse2, delta
constexpr int FB_STAGE_STRIDE = (FB_STAGE_BYTES + 1023) & ~1023;
constexpr int DS_BYTES = BN * QH * 2;         // dS^T: 128 keys x 64 queries bf16
constexpr int FB_SM_K = 0, FB_SM_V = TILE_BYTES, FB_SM_DS = 2 * TILE_BYTES;
constexpr int FB_SM_ST = FB_SM_DS + 2 * DS_BYTES;
constexpr int RED_Q = 16;                     // queries per dQ reduction block
constexpr int RED_BLOCK = RED_Q * 32 * 4;     // [16 queries x 32 dims] fp32 of one warp: 2 KiB
constexpr int FB_SM_RED = FB_SM_ST + FB_STAGES * FB_STAGE_STRIDE;   // 4 warps x 2 buffers
constexpr int FB_SM_BAR = FB_SM_RED + 4 * 2 * RED_BLOCK;

constexpr uint32_t COL_DV = 256, COL_DK = 384;
constexpr uint32_t IDESC_ST = idesc_bf16(BN, QH, false, false);   // [128 x 64] = A . B^T, both K-major
constexpr uint32_t IDESC_ACC = idesc_bf16(BN, HD, false, true);   // acc += X(tmem) . Y (Y MN-major)
constexpr uint32_t IDESC_DQ = idesc_bf16(HD, QH, true, true);     // dQ^T = K^T . dS^T, both MN-major

__device__ __forceinline__ uint32_t col_s(int r) { return uint32_t(r) * 128u; }
__device__ __forceinline__ uint32_t col_dp(int r) { return uint32_t(r) * 128u + 64u; }

struct FbBars {
  uint64_t st_full[FB_STAGES], st_empty[FB_STAGES];
  uint64_t own_full, own_empty;
  uint64_t s_full[2], p_full[2], dq_full[2], dq_empty[2];
  uint64_t acc_full, acc_empty;
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item[2];
  uint32_t tmem_base;
  int abort;
  int fill, use, own_issued, own_used;
};
constexpr int FB_SMEM = FB_SM_BAR + int(sizeof(FbBars)) + 1024;
static_assert(FB_SMEM <= 232448, "shared memory budget of one CTA");

struct FbArgs {
  const int *lo;       // [B, S_pad]
  const int *kend;     // [B, nT]
  const int *list;     // key-tile work list (b * nT + tile), longest first
  const float *delta;  // [B, H, S_pad]
  const float *lse2;   // [B, H, S_pad]: lse * log2(e), +inf where nothing is visible
  float *dqacc;        // [B, H, S_pad, D] fp32, zero on entry
  int *hdr;
  __nv_bfloat16 *dk, *dv;
  int B, S, H, nT, S_pad, n_items;
  float scale_log2;    // log2(e) / sqrt(D)
  float inv_sqrt_d;
};

struct FbItem {
  int b, h, tile;
};

__device__ __forceinline__ FbItem fb_decode(const FbArgs &a, int item) {
  const int e = a.list[item / a.H];
  return {e / a.nT, item % a.H, e % a.nT};
}

// Query tiles that see key tile `tile`: [tile, (kend - 1) / BM].
__device__ __forceinline__ TileRange fb_range(const FbArgs &a, const FbItem &I) {
  const int k0 = I.tile * BN;
  const int e = a.kend[I.b * a.nT + I.tile];
  TileRange r{1, 0};
  if (e > k0) {
    r.first = k0 / BM;
    r.last = (e - 1) / BM;
  }
  return r;
}

__device__ __forceinline__ int fb_halves(const TileRange &R) { return R.empty() ? 0 : 2 * (R.last - R.first + 1); }

// D[128 keys x 64 queries] = A[128 keys x 128 dims] . B[64 queries x 128 dims]^T.
// A is a resident tile (its two 64-dim boxes HALF_BYTES apart), B a streamed half
// tile (boxes QH_BOX apart); both K-major, 128B-swizzled.
__device__ __forceinline__ void issue_st(uint32_t d_tmem, uint32_t a_s, uint32_t b_s) {
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const uint32_t in_row = uint32_t(kk & 3) * 32;
    mma_ss(d_tmem, sdesc_sw128(a_s + uint32_t(kk >> 2) * HALF_BYTES + in_row, 16, 1024),
           sdesc_sw128(b_s + uint32_t(kk >> 2) * QH_BOX + in_row, 16, 1024), IDESC_ST, kk > 0);
  }
}

// acc[128 keys x 128 dims] (+)= X[128 keys x 64 queries] (bf16 in TMEM) . Y[64 x 128]
// with Y a streamed half tile read MN-major (dims contiguous; 16 rows = two 8-row
// groups of 1024 bytes; the 64-dim boxes QH_BOX apart). X's 16-query blocks (8 packed
// columns each) sit 16 columns apart: P^T and dS^T blocks alternate.
__device__ __forceinline__ void issue_acc(uint32_t acc, uint32_t x_tmem, uint32_t y_s, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < QH / 16; ++kk)
    mma_ts(acc, x_tmem + uint32_t(kk) * 16, sdesc_sw128(y_s + uint32_t(kk) * 2048, QH_BOX, 1024), IDESC_ACC,
           (accumulate || kk > 0) ? 1u : 0u);
}

// dQ^T[128 dims x 64 queries] = K^T[128 dims x 128 keys] . dS^T[128 keys x 64 queries].
// Both operands are read MN-major: K as stored (dims contiguous, 64-dim boxes
// HALF_BYTES apart), dS^T as written by the softmax warps (queries contiguous, one
// 128-byte swizzled row per key).
__device__ __forceinline__ void issue_dqt(uint32_t d_tmem, uint32_t k_s, uint32_t ds_s) {
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk)
    mma_ss(d_tmem, sdesc_sw128(k_s + uint32_t(kk) * 2048, HALF_BYTES, 1024),
           sdesc_sw128(ds_s + uint32_t(kk) * 2048, DS_BYTES, 1024), IDESC_DQ, kk > 0);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ bool fb_wait_plain(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
  return true;
}

__device__ __forceinline__ void fb_load_half(const CUtensorMap *m, uint64_t *bar, uint8_t *dst, int h, int row0,
                                             int b) {
  tma_load_4d(m, bar, dst, 0, h, row0, b);
  tma_load_4d(m, bar, dst + QH_BOX, 64, h, row0, b);
}

__device__ __forceinline__ void fb_load_tile(const CUtensorMap *m, uint64_t *bar, uint8_t *dst, int h, int row0,
                                             int b) {
  tma_load_4d(m, bar, dst, 0, h, row0, b);
  tma_load_4d(m, bar, dst + HALF_BYTES, 64, h, row0, b);
}

// ----------------------------------------------------------------------------- roles
__device__ __forceinline__ bool fb_producer(const CUtensorMap *tq, const CUtensorMap *tk, const CUtensorMap *tv,
                            const CUtensorMap *tdo, const FbArgs &a, uint8_t *smem, FbBars *bars) {
  volatile int *abort = &bars->abort;
  int fill = 0, own = 0;
  bool ok = true;
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_empty[slot], ((it >> 1) & 1) ^ 1, abort))) break;
    const int t = atomicAdd(a.hdr + HDR_TICKET_FUSED, 1);
    const int item = t < a.n_items ? t : -1;
    bars->item[slot] = item;
    mbar_arrive(&bars->item_full[slot]);
    if (item < 0) break;
    const FbItem I = fb_decode(a, item);
    const TileRange R = fb_range(a, I);
    const int n = fb_halves(R);
    if (!(ok = mbar_wait(&bars->own_empty, (it & 1) ^ 1, abort))) break;
    mbar_arrive_expect_tx(&bars->own_full, 2 * TILE_BYTES);
    fb_load_tile(tk, &bars->own_full, smem + FB_SM_K, I.h, I.tile * BN, I.b);
    fb_load_tile(tv, &bars->own_full, smem + FB_SM_V, I.h, I.tile * BN, I.b);
    ++own;
    const size_t rowbase = (size_t(I.b) * a.H + I.h) * a.S_pad;
    for (int u = 0; u < n && ok; ++u) {
      const int st = fill % FB_STAGES;
      if (!(ok = mbar_wait(&bars->st_empty[st], ((fill / FB_STAGES) & 1) ^ 1, abort))) break;
      mbar_arrive_expect_tx(&bars->st_full[st], FB_STAGE_BYTES);
      uint8_t *dst = smem + FB_SM_ST + st * FB_STAGE_STRIDE;
      const int row0 = (R.first + (u >> 1)) * BM + (u & 1) * QH;
      fb_load_half(tq, &bars->st_full[st], dst, I.h, row0, I.b);
      fb_load_half(tdo, &bars->st_full[st], dst + QH_BYTES, I.h, row0, I.b);
      bulk_load(dst + 2 * QH_BYTES, a.lo + size_t(I.b) * a.S_pad + row0, RT_BYTES, &bars->st_full[st]);
      bulk_load(dst + 2 * QH_BYTES + RT_BYTES, a.lse2 + rowbase + row0, RT_BYTES, &bars->st_full[st]);
      bulk_load(dst + 2 * QH_BYTES + 2 * RT_BYTES, a.delta + rowbase + row0, RT_BYTES, &bars->st_full[st]);
      ++fill;
    }
    if (!ok) break;
  }
  bars->fill = fill;
  bars->own_issued = own;
  return ok;
}

__device__ __forceinline__ bool fb_mma(const FbArgs &a, uint8_t *smem, FbBars *bars, uint32_t tmem, int lane) {
  volatile int *abort = &bars->abort;
  const uint32_t k_s = smem_u32(smem + FB_SM_K), v_s = smem_u32(smem + FB_SM_V);
  const uint32_t ds0 = smem_u32(smem + FB_SM_DS), st0 = smem_u32(smem + FB_SM_ST);
  int use = 0, own = 0;
  uint32_t pf_par[2] = {0, 0}, de_par[2] = {0, 0}, ae_par = 1;
  bool dq_pending[2] = {false, false};
  bool ok = true;

  for (int it = 0; ok; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const FbItem I = fb_decode(a, item);
    const int n = fb_halves(fb_range(a, I));
    if (!(ok = mbar_wait(&bars->own_full, it & 1, abort))) break;
    ++own;
    tc_fence_after();
    const int base = use;

    // S^T and dP^T of half u into region u & 1. dP^T overwrites the region's dQ^T of
    // two halves ago, so it waits until the readout warps have taken that out.
    auto issue_sdp = [&](int u) -> bool {
      const int r = u & 1, st = (base + u) % FB_STAGES;
      if (!mbar_wait(&bars->st_full[st], ((base + u) / FB_STAGES) & 1, abort)) return false;
      tc_fence_after();
      const uint32_t q_s = st0 + st * FB_STAGE_STRIDE, do_s = q_s + QH_BYTES;
      if (lane == 0) issue_st(tmem + col_s(r), k_s, q_s);
      __syncwarp();
      if (dq_pending[r]) {
        if (!mbar_wait(&bars->dq_empty[r], de_par[r], abort)) return false;
        de_par[r] ^= 1;
        dq_pending[r] = false;
        tc_fence_after();
      }
      if (lane == 0) {
        issue_st(tmem + col_dp(r), v_s, do_s);
        mma_commit(&bars->s_full[r]);
      }
      __syncwarp();
      return true;
    };

    for (int u = 0; u < n && u < 2 && ok; ++u) ok = issue_sdp(u);
    for (int u = 0; u < n && ok; ++u) {
      const int r = u & 1, st = (base + u) % FB_STAGES;
      const uint32_t q_s = st0 + st * FB_STAGE_STRIDE, do_s = q_s + QH_BYTES;
      if (!(ok = mbar_wait(&bars->p_full[r], pf_par[r], abort))) break;
      pf_par[r] ^= 1;
      if (u == 0) {
        if (!(ok = mbar_wait(&bars->acc_empty, ae_par, abort))) break;
        ae_par ^= 1;
      }
      tc_fence_after();
      if (lane == 0) {
        issue_acc(tmem + COL_DV, tmem + col_s(r), do_s, u > 0);          // dV += P^T dO
        issue_acc(tmem + COL_DK, tmem + col_s(r) + 8, q_s, u > 0);      // dK += dS^T Q
        issue_dqt(tmem + col_dp(r), k_s, ds0 + r * DS_BYTES);            // dQ^T = K^T dS^T
        mma_commit(&bars->dq_full[r]);
        mma_commit(&bars->st_empty[st]);
      }
      __syncwarp();
      dq_pending[r] = true;
      if (u + 2 < n) ok = issue_sdp(u + 2);
    }
    if (!ok) break;
    use = base + n;
    if (lane == 0) {
      if (n > 0) mma_commit(&bars->acc_full);
      mma_commit(&bars->own_empty);
    }
    __syncwarp();
  }
  if (lane == 0) {
    bars->use = use;
    bars->own_used = own;
  }
  return ok;
}

// Softmax warpgroup of region r: thread = key row j of the tile (TMEM lane).
__device__ __forceinline__ bool fb_softmax(const FbArgs &a, uint8_t *smem, FbBars *bars, uint32_t tmem, int r, int warp,
                           int lane) {
  volatile int *abort = &bars->abort;
  const int row = (warp & 3) * 32 + lane;
  const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_off + col_s(r), tP = tmem + lane_off + col_dp(r);
  uint8_t *ds_row = smem + FB_SM_DS + r * DS_BYTES + (row >> 3) * 1024 + (row & 7) * 128;
  const float c = a.scale_log2;
  uint32_t sf_par = 0, af_par = 0;
  int use = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const FbItem I = fb_decode(a, item);
    const TileRange R = fb_range(a, I);
    const int n = fb_halves(R);
    const int k0 = I.tile * BN, j = k0 + row;
    const int *lr = a.lo + size_t(I.b) * a.S_pad;
    for (int u = r; u < n; u += 2) {
      const int st = (use + u) % FB_STAGES;
      const uint32_t st_par = ((use + u) / FB_STAGES) & 1;
      if (!(ok = mbar_wait(&bars->s_full[r], sf_par, abort))) break;
      sf_par ^= 1;
      // the stage's lo / lse2 / delta rows arrived by bulk copy: observe their barrier
      if (!(ok = mbar_wait(&bars->st_full[st], st_par, abort))) break;
      tc_fence_after();
      const uint8_t *stage = smem + FB_SM_ST + st * FB_STAGE_STRIDE;
      const int *lo_q = reinterpret_cast<const int *>(stage + 2 * QH_BYTES);
      const float *l2_q = reinterpret_cast<const float *>(stage + 2 * QH_BYTES + RT_BYTES);
      const float *dl_q = reinterpret_cast<const float *>(stage + 2 * QH_BYTES + 2 * RT_BYTES);
      const int qb = (R.first + (u >> 1)) * BM + (u & 1) * QH;   // first query of the half
      // Key j is visible from query qb + q iff lo[qb + q] <= j <= qb + q. lo is
      // non-decreasing, so the visible q form one range [q_from, q_to): q_from = j - qb,
      // q_to = the number of q with lo <= j. Whole-visible pairs skip the search.
      int q_from = 0, q_to = QH;
      if (!(lr[qb + QH - 1] <= k0 && k0 + BN - 1 <= qb)) {
        q_from = j - qb;
        int lo_i = 0, hi_i = QH;
        while (lo_i < hi_i) {
          const int m = (lo_i + hi_i) >> 1;
          if (lo_q[m] <= j) lo_i = m + 1; else hi_i = m;
        }
        q_to = lo_i;
      }
      // 16 queries at a time: their S^T / dP^T columns, row terms and results stay in
      // registers together
#pragma unroll 1
      for (int ch = 0; ch < QH / 16; ++ch) {
        uint32_t sv[16], dv[16];
        tmem_ld16(tS + ch * 16, sv);
        tmem_ld16(tP + ch * 16, dv);
        tmem_ld_wait();
        uint32_t pk[8], dk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float pp[2], dd[2];
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            const int q = ch * 16 + 2 * e + w;
            float p = ex2_approx(fmaf(__uint_as_float(sv[2 * e + w]), c, -l2_q[q]));
            if (q < q_from || q >= q_to) p = 0.f;
            pp[w] = p;
            dd[w] = p * (__uint_as_float(dv[2 * e + w]) - dl_q[q]);
          }
          pk[e] = pack_bf16x2(pp[0], pp[1]);
          dk[e] = pack_bf16x2(dd[0], dd[1]);
        }
        // bf16 results over the 16 columns just read: P^T block, then dS^T block
        tmem_st8(tS + ch * 16, pk);
        tmem_st8(tS + ch * 16 + 8, dk);
        // dS^T row of this key into the 128B-swizzled staging tile: 16-byte chunk
        // c (queries 8c .. 8c+7) sits at chunk position c ^ (row & 7)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int chunk = ch * 2 + cc;
          *reinterpret_cast<uint4 *>(ds_row + ((chunk ^ (row & 7)) << 4)) =
              make_uint4(dk[4 * cc], dk[4 * cc + 1], dk[4 * cc + 2], dk[4 * cc + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[r]);
    }
    if (!ok) break;
    use += n;
    // epilogue: region 0's warpgroup writes dV, region 1's writes dK (scaled by 1/sqrt(D))
    __nv_bfloat16 *dst = (r == 0 ? a.dv : a.dk) + ((size_t(I.b) * a.S + j) * a.H + I.h) * HD;
    if (n > 0) {
      if (!(ok = mbar_wait(&bars->acc_full, af_par, abort))) break;
      af_par ^= 1;
      tc_fence_after();
      const uint32_t t_acc = tmem + lane_off + (r == 0 ? COL_DV : COL_DK);
      const float f = r == 0 ? 1.f : a.inv_sqrt_d;
      for (int cc = 0; cc < HD; cc += 32) {
        uint32_t o[32];
        tmem_ld32(t_acc + cc, o);
        tmem_ld_wait();
        uint4 w4[4];
        uint32_t *wp = reinterpret_cast<uint32_t *>(w4);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          wp[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * f, __uint_as_float(o[2 * e + 1]) * f);
        if (j < a.S) {
          uint4 *d = reinterpret_cast<uint4 *>(dst + cc);
#pragma unroll
          for (int e = 0; e < 4; ++e) d[e] = w4[e];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_empty);
    } else if (j < a.S) {
      uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
      for (int e = 0; e < HD / 8; ++e) d[e] = make_uint4(0, 0, 0, 0);
    }
  }
  return ok;
}

// Tensor bulk reduce-add of a shared-memory box into the fp32 dQ accumulator (the
// addition is performed in L2), tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *map, const void *src, int x, int y) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most one committed bulk group still reads its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Waits until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// dQ readout: warp w takes TMEM lanes 32 (w % 4) .. + 31 = head dims 32 (w % 4) .. + 31
// of dQ^T, and passes every 16-query block of them through one of its two shared
// staging buffers ([query][dim]) to a tensor bulk reduce-add into the accumulator.
__device__ __forceinline__ bool fb_readout(const CUtensorMap *tdq, const FbArgs &a, uint8_t *smem, FbBars *bars,
                                           uint32_t tmem, int warp, int lane) {
  volatile int *abort = &bars->abort;
  const int quarter = warp & 3;
  const uint32_t lane_off = uint32_t(quarter * 32) << 16;
  float *stage = reinterpret_cast<float *>(smem + FB_SM_RED + quarter * 2 * RED_BLOCK);
  uint32_t df_par[2] = {0, 0};
  int nblk = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const FbItem I = fb_decode(a, item);
    const TileRange R = fb_range(a, I);
    const int n = fb_halves(R);
    const int row_bh = (I.b * a.H + I.h) * a.S_pad;   // accumulator row of query 0
    for (int u = 0; u < n; ++u) {
      const int r = u & 1;
      if (!(ok = mbar_wait(&bars->dq_full[r], df_par[r], abort))) break;
      df_par[r] ^= 1;
      tc_fence_after();
      uint32_t v[QH];
      tmem_ld32(tmem + lane_off + col_dp(r), v);
      tmem_ld32(tmem + lane_off + col_dp(r) + 32, v + 32);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->dq_empty[r]);
      const int row0 = row_bh + (R.first + (u >> 1)) * BM + r * QH;
#pragma unroll
      for (int blk = 0; blk < QH / RED_Q; ++blk, ++nblk) {
        float *buf = stage + (nblk & 1) * (RED_BLOCK / 4);
        if (lane == 0) bulk_wait_read_1();   // this buffer's previous block has been read
        __syncwarp();
#pragma unroll
        for (int q = 0; q < RED_Q; ++q) buf[q * 32 + lane] = __uint_as_float(v[blk * RED_Q + q]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tma_reduce_add_2d(tdq, buf, quarter * 32, row0 + blk * RED_Q);
      }
    }
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
  return ok;
}

// Common exit of every warp: on a failed (timed-out) wait raise the abort flag and the
// error bit, let copies and MMAs still in flight land before shared memory and TMEM go
// away, free TMEM, and let the last CTA reset the scheduler ticket.
__device__ __forceinline__ void fb_finish(bool ok, const FbArgs &a, FbBars *bars, uint32_t tmem, int warp, int lane) {
  if (!ok) {
    bars->abort = 1;
    raise_error(a.hdr + HDR_ERR, ERRBIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (bars->abort) {
    if (warp == FB_PRODUCER && lane == 0) {
      for (int k = bars->use; k < bars->fill; ++k)
        fb_wait_plain(&bars->st_full[k % FB_STAGES], (k / FB_STAGES) & 1);
      if (bars->own_issued > bars->own_used) fb_wait_plain(&bars->own_full, (bars->own_issued - 1) & 1);
    }
    if (warp == FB_MMA && lane == 0) {
      mma_commit(&bars->drain);
      fb_wait_plain(&bars->drain, 0);
    }
    __syncthreads();
  }
  if (warp == FB_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.hdr + HDR_DONE_FUSED, 1) == int(gridDim.x) - 1) {
      a.hdr[HDR_TICKET_FUSED] = 0;
      a.hdr[HDR_DONE_FUSED] = 0;
      __threadfence();
    }
  }
}

__global__ void __launch_bounds__(FB_THREADS, 1)
    dkdvq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                 const __grid_constant__ CUtensorMap tdq, const FbArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FbBars *bars = reinterpret_cast<FbBars *>(smem + FB_SM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < FB_STAGES; ++s) {
      mbar_init(&bars->st_full[s], 1);
      mbar_init(&bars->st_empty[s], 1);
    }
    mbar_init(&bars->own_full, 1);
    mbar_init(&bars->own_empty, 1);
    for (int r = 0; r < 2; ++r) {
      mbar_init(&bars->s_full[r], 1);
      mbar_init(&bars->p_full[r], 4);
      mbar_init(&bars->dq_full[r], 1);
      mbar_init(&bars->dq_empty[r], 4);
      mbar_init(&bars->item_full[r], 1);
      mbar_init(&bars->item_empty[r], 13);   // softmax 8 + readout 4 + MMA 1 warps
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->fill = bars->use = bars->own_issued = bars->own_used = 0;
    fence_mbar_init();
  }
  if (warp == FB_MMA) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == FB_PRODUCER && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
  }
  if (warp == FB_READ0 && lane == 0) tma_prefetch_desc(&tdq);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < FB_READ0) {
    fb_finish(fb_softmax(a, smem, bars, tmem, warp >> 2, warp, lane), a, bars, tmem, warp, lane);
  } else if (warp < FB_PRODUCER) {
    fb_finish(fb_readout(&tdq, a, smem, bars, tmem, warp, lane), a, bars, tmem, warp, lane);
  } else {
    bool ok = true;
    if (warp == FB_PRODUCER) {
      if (lane == 0) ok = fb_producer(&tq, &tk, &tv, &tdo, a, smem, bars);
      __syncwarp();
    } else if (warp == FB_MMA) {
      ok = fb_mma(a, smem, bars, tmem, lane);
    }
    fb_finish(ok, a, bars, tmem, warp, lane);
  }
}

// dq[b, s, h, :] = bf16(dqacc[b, h, s, :] / sqrt(D)); one thread per 8 dims.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float4 *__restrict__ acc, uint4 *__restrict__ dq,
                                                         int B, int S, int H, int S_pad, float scale) {
  const long long total = (long long)B * S * H * (HD / 8);
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c8 = int(idx % (HD / 8));
    const long long row = idx / (HD / 8);   // (b, s, h) in dq order
    const int h = int(row % H);
    const long long bs = row / H;
    const int s = int(bs % S);
    const int b = int(bs / S);
    const size_t src = ((size_t(b) * H + h) * S_pad + s) * (HD / 4) + c8 * 2;
    const float4 x = __ldg(acc + src), y = __ldg(acc + src + 1);
    uint4 o;
    o.x = pack_bf16x2(x.x * scale, x.y * scale);
    o.y = pack_bf16x2(x.z * scale, x.w * scale);
    o.z = pack_bf16x2(y.x * scale, y.y * scale);
    o.w = pack_bf16x2(y.z * scale, y.w * scale);
    dq[idx] = o;
  }
}

}  // namespace

cudaError_t launch_dkdvq(const CUtensorMap &tq64, const CUtensorMap &tk, const CUtensorMap &tv,
                         const CUtensorMap &tdo64, const CUtensorMap &tdqacc, void *dq, void *dk, void *dv,
                         const Problem &p, void *workspace, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(dkdvq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FB_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const Workspace w = Workspace::layout(p.B, p.S, p.H);
  char *base = static_cast<char *>(workspace);
  FbArgs a;
  a.lo = reinterpret_cast<const int *>(base + w.off_lo);
  a.kend = reinterpret_cast<const int *>(base + w.off_kend);
  a.list = reinterpret_cast<const int *>(base + w.off_list_kv);
  a.delta = reinterpret_cast<const float *>(base + w.off_delta);
  a.lse2 = reinterpret_cast<const float *>(base + w.off_lse2);
  a.dqacc = reinterpret_cast<float *>(base + w.off_dqacc);
  a.hdr = reinterpret_cast<int *>(base + w.off_hdr);
  a.dk = static_cast<__nv_bfloat16 *>(dk);
  a.dv = static_cast<__nv_bfloat16 *>(dv);
  a.B = p.B;
  a.S = p.S;
  a.H = p.H;
  a.nT = w.nT;
  a.S_pad = w.S_pad;
  a.n_items = p.B * w.nT * p.H;
  a.scale_log2 = 1.4426950408889634f / sqrtf(float(HD));
  a.inv_sqrt_d = 1.f / sqrtf(float(HD));
  cudaError_t e = cudaMemsetAsync(a.dqacc, 0, w.dqacc_bytes, stream);
  if (e != cudaSuccess) return e;
  const int grid = a.n_items < p.num_sms ? a.n_items : p.num_sms;
  dkdvq_kernel<<<grid, FB_THREADS, FB_SMEM, stream>>>(tq64, tk, tv, tdo64, tdqacc, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long total = (long long)p.B * p.S * p.H * (HD / 8);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)p.num_sms * 16;
  if (blocks > cap) blocks = cap;
  dq_convert_kernel<<<int(blocks), 256, 0, stream>>>(reinterpret_cast<const float4 *>(a.dqacc),
                                                      static_cast<uint4 *>(dq), p.B, p.S, p.H, w.S_pad,
                                                      a.inv_sqrt_d);
  return cudaGetLastError();
}

}  // namespace lwm
