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
// Item: (b, h, 128-key tile), taken through an atomic ticket by one persistent CTA per
// SM (items of one head are consecutive, longest first, so that the CTAs running at
// the same time share their query-side tiles in L2). K and V of the tile stay
// resident in shared memory; the 128-row query tiles j that see it stream through
// (Q_j in a ring of two buffers with its rows' lo / lse / delta terms, dO_j in one
// buffer). Per tile j, every product is 128 x 128 x 128:
//   S^T  = K . Q_j^T   -> TMEM region A         dP^T = V . dO_j^T -> TMEM region B
//   P^T  = exp2(S^T c - lse2)  (softmax warps)  -> bf16 over region A
//   dV  += P^T . dO_j                           (needs only P: issued before dS is ready)
//   dS^T = P^T (dP^T - delta)  (softmax warps)  -> bf16 over region A, and into shared memory
//   dK  += dS^T . Q_j,   dQ^T = K^T . dS^T      -> dQ^T into region B
// and the softmax warps then move dQ^T out of TMEM and add it, through shared staging
// buffers and tensor bulk reduce-add copies (performed in L2), into an fp32
// accumulator [B, H, S_pad, D]. A final pass converts that to bf16 dq. The order of
// the fp32 additions depends on scheduling, so dq is not bitwise reproducible from run
// to run (dk and dv are).
//
// The tensor core runs S^T(j+1) while the softmax warps take dQ^T(j) out, dP^T(j+1)
// while they compute P(j+1), and dV(j+1) while they compute dS(j+1), so that it has
// work queued through each softmax phase.
//
// Warp roles: 0-3 and 4-7 two warpgroups, warpgroup w owning query columns
// [64 w, 64 w + 64) of every tile (thread = key row = TMEM lane); 8 TMA producer;
// 9 MMA issuer; 10-11 idle (3 warps per SM sub-partition: 168 registers per thread).
// TMEM columns: A [0, 128), B [128, 256), dV [256, 384), dK [384, 512). In region A,
// the 16-query chunk c (columns 16c .. 16c+15 of S^T) is overwritten by P^T of those
// queries (bf16, columns 16c .. 16c+7) and then dS^T (16c+8 .. 16c+15).
#include "common.cuh"
#include "kernels.h"

namespace lwm {
namespace {

constexpr int FB_WARPS = 12;
constexpr int FB_THREADS = FB_WARPS * 32;
constexpr int FB_PRODUCER = 8;
constexpr int FB_MMA = 9;
constexpr int RT_BYTES = BM * 4;                // 128 row terms (int32 / fp32)
constexpr int DS_BYTES = BN * BM * 2;           // dS^T staging: 128 keys x 128 queries bf16
constexpr int RED_Q = 8;                        // queries per dQ reduction block
constexpr int RED_BLOCK = RED_Q * 32 * 4;       // [8 queries x 32 dims] fp32: 1 KiB
// shared memory map (bytes; tiles 1024-aligned)
constexpr int FB_SM_K = 0;
constexpr int FB_SM_V = FB_SM_K + TILE_BYTES;
constexpr int FB_SM_Q = FB_SM_V + TILE_BYTES;             // 2 Q buffers
constexpr int FB_SM_DO = FB_SM_Q + 2 * TILE_BYTES;        // 1 dO buffer
constexpr int FB_SM_DS = FB_SM_DO + TILE_BYTES;           // dS^T, two 64-query halves of 16 KiB
constexpr int FB_SM_RED = FB_SM_DS + DS_BYTES;            // 8 warps x 2 reduction buffers
constexpr int FB_SM_RT = FB_SM_RED + 8 * 2 * RED_BLOCK;   // row terms of the 2 Q buffers
constexpr int FB_SM_BAR = FB_SM_RT + 2 * 3 * RT_BYTES;

constexpr uint32_t COL_A = 0, COL_B = 128, COL_DV = 256, COL_DK = 384;
constexpr uint32_t IDESC_KM = idesc_bf16(128, 128, false, false);   // D = A . B^T, both K-major
constexpr uint32_t IDESC_TS = idesc_bf16(128, 128, false, true);    // acc += X(tmem) . Y (Y MN-major)
constexpr uint32_t IDESC_MN = idesc_bf16(128, 128, true, true);     // dQ^T = K^T . dS^T, both MN-major

struct FbBars {
  uint64_t q_full[2], q_empty[2], do_full, do_empty;
  uint64_t own_full, own_empty;
  uint64_t s_full, dp_full, p_full, ds_full, dq_full, dq_empty;
  uint64_t acc_full, acc_empty;
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item[2];
  uint32_t tmem_base;
  WaitCtl ctl;
  int q_fill, q_use, do_fill, do_use, own_issued, own_used;
  uint64_t never;   // the failure test's wait (test instantiation only)
};
constexpr int FB_SMEM = FB_SM_BAR + int(sizeof(FbBars)) + 1024;
static_assert(FB_SMEM <= 232448, "shared memory budget of one CTA");

struct FbArgs {
  const int *lo;       // [B, S_pad]
  const int *kend;     // [B, nT]
  const int *list;     // key tiles (b * nT + tile), longest first
  const float *delta;  // [B, H, S_pad]
  const float *lse2;   // [B, H, S_pad]: lse * log2(e), +inf where nothing is visible
  int *hdr;
  __nv_bfloat16 *dk, *dv;
  int B, S, H, nT, S_pad, n_list, n_items;
  float scale_log2;    // log2(e) / sqrt(D)
  float inv_sqrt_d;
  WaitBound wait;
};

struct FbItem {
  int b, h, tile;
};

// Items of one head are consecutive (head-major), each head's key tiles longest first.
__device__ __forceinline__ FbItem fb_decode(const FbArgs &a, int item) {
  const int e = a.list[item % a.n_list];
  return {e / a.nT, item / a.n_list, e % a.nT};
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

__device__ __forceinline__ int fb_tiles(const TileRange &R) { return R.empty() ? 0 : R.last - R.first + 1; }

// D[128 x 128] = A[128 rows x 128 dims] . B[128 rows x 128 dims]^T; both operands are
// 128-row tiles stored as two 64-dim 128B-swizzled boxes HALF_BYTES apart (K-major).
__device__ __forceinline__ void issue_kmajor(uint32_t d_tmem, uint32_t a_s, uint32_t b_s) {
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const uint32_t off = uint32_t(kk >> 2) * HALF_BYTES + uint32_t(kk & 3) * 32;
    mma_ss(d_tmem, sdesc_sw128(a_s + off, 16, 1024), sdesc_sw128(b_s + off, 16, 1024), IDESC_KM, kk > 0);
  }
}

// acc[128 keys x 128 dims] (+)= X[128 keys x 128 queries] (bf16 in TMEM; the 16-query
// block kk at column 16 kk of x_tmem) . Y[128 queries x 128 dims] read MN-major (dims
// contiguous: 16 rows = two 8-row groups of 1024 bytes; the 64-dim boxes HALF_BYTES
// apart).
__device__ __forceinline__ void issue_ts(uint32_t acc, uint32_t x_tmem, uint32_t y_s, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < BM / 16; ++kk)
    mma_ts(acc, x_tmem + uint32_t(kk) * 16, sdesc_sw128(y_s + uint32_t(kk) * 2048, HALF_BYTES, 1024), IDESC_TS,
           (accumulate || kk > 0) ? 1u : 0u);
}

// dQ^T[128 dims x 128 queries] = K^T[128 dims x 128 keys] . dS^T[128 keys x 128 queries].
// Both operands are read MN-major: K as stored (dims contiguous, 64-dim boxes
// HALF_BYTES apart), dS^T as the softmax warps write it (queries contiguous, 128-byte
// swizzled rows, one per key; the 64-query halves DS_BYTES / 2 apart).
__device__ __forceinline__ void issue_dqt(uint32_t d_tmem, uint32_t k_s, uint32_t ds_s) {
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk)
    mma_ss(d_tmem, sdesc_sw128(k_s + uint32_t(kk) * 2048, HALF_BYTES, 1024),
           sdesc_sw128(ds_s + uint32_t(kk) * 2048, DS_BYTES / 2, 1024), IDESC_MN, kk > 0);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

__device__ __forceinline__ void fb_load_tile(const CUtensorMap *m, uint64_t *bar, uint8_t *dst, int h, int row0,
                                             int b) {
  tma_load_4d(m, bar, dst, 0, h, row0, b);
  tma_load_4d(m, bar, dst + HALF_BYTES, 64, h, row0, b);
}

// ----------------------------------------------------------------------------- producer
template <bool TEST>
__device__ __forceinline__ bool fb_producer(const CUtensorMap *tq, const CUtensorMap *tk, const CUtensorMap *tv,
                                            const CUtensorMap *tdo, const FbArgs &a, uint8_t *smem, FbBars *bars) {
  WaitCtl *abort = &bars->ctl;
  int q_fill = 0, do_fill = 0, own = 0;
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
    const int n = fb_tiles(R);
    if (!(ok = mbar_wait(&bars->own_empty, (it & 1) ^ 1, abort))) break;
    mbar_arrive_expect_tx(&bars->own_full, 2 * TILE_BYTES);
    fb_load_tile(tk, &bars->own_full, smem + FB_SM_K, I.h, I.tile * BN, I.b);
    fb_load_tile(tv, &bars->own_full, smem + FB_SM_V, I.h, I.tile * BN, I.b);
    ++own;
    const size_t rowbase = (size_t(I.b) * a.H + I.h) * a.S_pad;
    for (int j = 0; j < n && ok; ++j) {
      const int row0 = (R.first + j) * BM;
      const int qs = q_fill & 1;
      if (!(ok = mbar_wait(&bars->q_empty[qs], ((q_fill >> 1) & 1) ^ 1, abort))) break;
      mbar_arrive_expect_tx(&bars->q_full[qs], TILE_BYTES + 3 * RT_BYTES);
      fb_load_tile(tq, &bars->q_full[qs], smem + FB_SM_Q + qs * TILE_BYTES, I.h, row0, I.b);
      uint8_t *rt = smem + FB_SM_RT + qs * 3 * RT_BYTES;
      bulk_load(rt, a.lo + size_t(I.b) * a.S_pad + row0, RT_BYTES, &bars->q_full[qs]);
      bulk_load(rt + RT_BYTES, a.lse2 + rowbase + row0, RT_BYTES, &bars->q_full[qs]);
      bulk_load(rt + 2 * RT_BYTES, a.delta + rowbase + row0, RT_BYTES, &bars->q_full[qs]);
      ++q_fill;
      if (!(ok = mbar_wait(&bars->do_empty, (do_fill & 1) ^ 1, abort))) break;
      mbar_arrive_expect_tx(&bars->do_full, TILE_BYTES);
      fb_load_tile(tdo, &bars->do_full, smem + FB_SM_DO, I.h, row0, I.b);
      ++do_fill;
    }
    if (!ok) break;
    // failure test only: wait, with this item's copies and products in flight, for a
    // phase that never completes (the short test bound makes the wait run out)
    if constexpr (TEST) {
      if (it == 0 && !(ok = test_expiry_wait(&bars->never, abort))) break;
    }
  }
  bars->q_fill = q_fill;
  bars->do_fill = do_fill;
  bars->own_issued = own;
  return ok;
}

// ----------------------------------------------------------------------------- MMA issuer
__device__ __forceinline__ bool fb_mma(const FbArgs &a, uint8_t *smem, FbBars *bars, uint32_t tmem, int lane) {
  WaitCtl *abort = &bars->ctl;
  const uint32_t k_s = smem_u32(smem + FB_SM_K), v_s = smem_u32(smem + FB_SM_V);
  const uint32_t q0_s = smem_u32(smem + FB_SM_Q), do_s = smem_u32(smem + FB_SM_DO);
  const uint32_t ds_s = smem_u32(smem + FB_SM_DS);
  int q_use = 0, do_use = 0, own = 0;
  uint32_t pf_par = 0, dsf_par = 0, dqe_par = 0, ae_par = 1;
  bool dq_pending = false;
  bool ok = true;

  for (int it = 0; ok; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const FbItem I = fb_decode(a, item);
    const int n = fb_tiles(fb_range(a, I));
    if (!(ok = mbar_wait(&bars->own_full, it & 1, abort))) break;
    ++own;
    tc_fence_after();

    // S^T(j) into region A (free once the previous tile's dV and dK have been issued:
    // the tensor core runs them in order), then dP^T(j) into region B, which holds the
    // previous tile's dQ^T until the softmax warps have taken it out.
    auto issue_sdp = [&]() -> bool {
      const int qs = q_use & 1;
      if (!mbar_wait(&bars->q_full[qs], (q_use >> 1) & 1, abort)) return false;
      tc_fence_after();
      if (lane == 0) {
        issue_kmajor(tmem + COL_A, k_s, q0_s + qs * TILE_BYTES);
        mma_commit(&bars->s_full);
      }
      __syncwarp();
      if (dq_pending) {
        if (!mbar_wait(&bars->dq_empty, dqe_par, abort)) return false;
        dqe_par ^= 1;
        dq_pending = false;
      }
      if (!mbar_wait(&bars->do_full, do_use & 1, abort)) return false;
      tc_fence_after();
      if (lane == 0) {
        issue_kmajor(tmem + COL_B, v_s, do_s);
        mma_commit(&bars->dp_full);
      }
      __syncwarp();
      return true;
    };

    if (n > 0) ok = issue_sdp();
    for (int j = 0; j < n && ok; ++j) {
      const int qs = q_use & 1;
      if (!(ok = mbar_wait(&bars->p_full, pf_par, abort))) break;
      pf_par ^= 1;
      if (j == 0) {
        if (!(ok = mbar_wait(&bars->acc_empty, ae_par, abort))) break;
        ae_par ^= 1;
      }
      tc_fence_after();
      if (lane == 0) {
        issue_ts(tmem + COL_DV, tmem + COL_A, do_s, j > 0);   // dV += P^T dO
        mma_commit(&bars->do_empty);
      }
      __syncwarp();
      ++do_use;
      if (!(ok = mbar_wait(&bars->ds_full, dsf_par, abort))) break;
      dsf_par ^= 1;
      tc_fence_after();
      if (lane == 0) {
        issue_ts(tmem + COL_DK, tmem + COL_A + 8, q0_s + qs * TILE_BYTES, j > 0);   // dK += dS^T Q
        mma_commit(&bars->q_empty[qs]);
        issue_dqt(tmem + COL_B, k_s, ds_s);                                         // dQ^T = K^T dS^T
        mma_commit(&bars->dq_full);
      }
      __syncwarp();
      ++q_use;
      dq_pending = true;
      if (j + 1 < n) ok = issue_sdp();
    }
    if (!ok) break;
    if (lane == 0) {
      if (n > 0) mma_commit(&bars->acc_full);
      mma_commit(&bars->own_empty);
    }
    __syncwarp();
  }
  if (lane == 0) {
    bars->q_use = q_use;
    bars->do_use = do_use;
    bars->own_used = own;
  }
  return ok;
}

// ----------------------------------------------------------------------------- softmax
// Warpgroup w: thread = key row `row` of the tile (TMEM lane), query columns
// [64 w, 64 w + 64) of every streamed tile. Per tile: the P phase, the dS phase, then
// the readout of its columns of dQ^T.
__device__ __forceinline__ bool fb_softmax(const CUtensorMap *tdq, const FbArgs &a, uint8_t *smem, FbBars *bars,
                                           uint32_t tmem, int w, int warp, int lane) {
  WaitCtl *abort = &bars->ctl;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = uint32_t(quarter * 32) << 16;
  const uint32_t tA = tmem + lane_off + COL_A + 64 * w;   // this warpgroup's S^T / P^T / dS^T columns
  const uint32_t tB = tmem + lane_off + COL_B + 64 * w;   // dP^T, then dQ^T
  // dS^T staging: 64-query half w, row `row` (128 bytes, 16-byte chunks swizzled by row & 7)
  uint8_t *ds_row = smem + FB_SM_DS + w * (DS_BYTES / 2) + (row >> 3) * 1024 + (row & 7) * 128;
  float *red = reinterpret_cast<float *>(smem + FB_SM_RED + warp * 2 * RED_BLOCK);
  const float c = a.scale_log2;
  const bool red_leader = lane == 0;
  uint32_t sf_par = 0, dpf_par = 0, dqf_par = 0, af_par = 0;
  int q_use = 0, nred = 0;
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
    const int n = fb_tiles(R);
    const int k0 = I.tile * BN, jk = k0 + row;   // this thread's key
    const int row_bh = (I.b * a.H + I.h) * a.S_pad;
    for (int j = 0; j < n; ++j, ++q_use) {
      const int qs = q_use & 1;
      const int q0 = (R.first + j) * BM;
      const uint8_t *rt = smem + FB_SM_RT + qs * 3 * RT_BYTES;
      const int *lo_q = reinterpret_cast<const int *>(rt);
      const float4 *l2_q = reinterpret_cast<const float4 *>(rt + RT_BYTES) + 16 * w;
      const float4 *dl_q = reinterpret_cast<const float4 *>(rt + 2 * RT_BYTES) + 16 * w;

      // ---- P phase: P^T = exp2(S^T c - lse2) on the visible pairs
      if (!(ok = mbar_wait(&bars->s_full, sf_par, abort))) break;
      sf_par ^= 1;
      // the row terms arrived by bulk copy with Q_j: observe that buffer's barrier
      if (!(ok = mbar_wait(&bars->q_full[qs], (q_use >> 1) & 1, abort))) break;
      tc_fence_after();
      // Key jk is visible from query q0 + q iff lo[q0 + q] <= jk <= q0 + q; lo is
      // non-decreasing, so these q form one range [q_from, q_to).
      int q_from = 0, q_to = BM;
      if (!(lo_q[BM - 1] <= k0 && k0 + BN - 1 <= q0)) {
        q_from = jk - q0;
        int lo_i = 0, hi_i = BM;
        while (lo_i < hi_i) {
          const int m = (lo_i + hi_i) >> 1;
          if (lo_q[m] <= jk) lo_i = m + 1; else hi_i = m;
        }
        q_to = lo_i;
      }
      q_from -= 64 * w;   // relative to this warpgroup's first column
      q_to -= 64 * w;
      float p[64];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t sv[16];
        tmem_ld16(tA + ch * 16, sv);
        tmem_ld_wait();
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
          const float4 l2 = l2_q[ch * 4 + e4];
          const float l2v[4] = {l2.x, l2.y, l2.z, l2.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = ch * 16 + e4 * 4 + e;
            float pv = ex2_approx(fmaf(__uint_as_float(sv[e4 * 4 + e]), c, -l2v[e]));
            if (q < q_from || q >= q_to) pv = 0.f;
            p[q] = pv;
          }
        }
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) pk[e] = pack_bf16x2(p[ch * 16 + 2 * e], p[ch * 16 + 2 * e + 1]);
        tmem_st8(tA + ch * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);

      // ---- dS phase: dS^T = P^T (dP^T - delta) -> TMEM (for dK) and shared memory (for dQ)
      if (!(ok = mbar_wait(&bars->dp_full, dpf_par, abort))) break;
      dpf_par ^= 1;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t dv[16];
        tmem_ld16(tB + ch * 16, dv);
        tmem_ld_wait();
        float ds[16];
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
          const float4 dl = dl_q[ch * 4 + e4];
          const float dlv[4] = {dl.x, dl.y, dl.z, dl.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            ds[e4 * 4 + e] = p[ch * 16 + e4 * 4 + e] * (__uint_as_float(dv[e4 * 4 + e]) - dlv[e]);
        }
        uint32_t dk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) dk[e] = pack_bf16x2(ds[2 * e], ds[2 * e + 1]);
        tmem_st8(tA + ch * 16 + 8, dk);
        // 16-byte chunks 2 ch and 2 ch + 1 of this key's row (queries 16 ch .. 16 ch + 15)
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
      if (lane == 0) mbar_arrive(&bars->ds_full);

      // ---- dQ readout: this warpgroup's 64 query columns of dQ^T; lane = head dim
      if (!(ok = mbar_wait(&bars->dq_full, dqf_par, abort))) break;
      dqf_par ^= 1;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32(tB, v);
      tmem_ld32(tB + 32, v + 32);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->dq_empty);
      const int yq = row_bh + q0 + 64 * w;   // accumulator row of this warpgroup's first query
#pragma unroll
      for (int blk = 0; blk < 64 / RED_Q; ++blk, ++nred) {
        float *buf = red + (nred & 1) * (RED_BLOCK / 4);
        if (red_leader) bulk_wait_read_1();   // this buffer's previous block has been read
        __syncwarp();
#pragma unroll
        for (int q = 0; q < RED_Q; ++q) buf[q * 32 + lane] = __uint_as_float(v[blk * RED_Q + q]);
        fence_proxy_async_smem();
        __syncwarp();
        if (red_leader) tma_reduce_add_2d(tdq, buf, quarter * 32, yq + blk * RED_Q);
      }
    }
    if (!ok) break;

    // epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (scaled by 1/sqrt(D))
    __nv_bfloat16 *dst = (w == 0 ? a.dv : a.dk) + ((size_t(I.b) * a.S + jk) * a.H + I.h) * HD;
    if (n > 0) {
      if (!(ok = mbar_wait(&bars->acc_full, af_par, abort))) break;
      af_par ^= 1;
      tc_fence_after();
      const uint32_t t_acc = tmem + lane_off + (w == 0 ? COL_DV : COL_DK);
      const float f = w == 0 ? 1.f : a.inv_sqrt_d;
#pragma unroll 1
      for (int cc = 0; cc < HD; cc += 32) {
        uint32_t o[32];
        tmem_ld32(t_acc + cc, o);
        tmem_ld_wait();
        uint4 w4[4];
        uint32_t *wp = reinterpret_cast<uint32_t *>(w4);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          wp[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * f, __uint_as_float(o[2 * e + 1]) * f);
        if (jk < a.S) {
          uint4 *d = reinterpret_cast<uint4 *>(dst + cc);
#pragma unroll
          for (int e = 0; e < 4; ++e) d[e] = w4[e];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_empty);
    } else if (jk < a.S) {
      uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
      for (int e = 0; e < HD / 8; ++e) d[e] = make_uint4(0, 0, 0, 0);
    }
  }
  if (red_leader) bulk_wait_all();
  __syncwarp();
  return ok;
}

// Common exit of every warp: on a failed (timed-out) wait raise the abort flag and the
// error bit, let copies and MMAs still in flight land before shared memory and TMEM go
// away, free TMEM, and let the last CTA reset the scheduler ticket.
__device__ __forceinline__ void fb_finish(bool ok, const FbArgs &a, FbBars *bars, uint32_t tmem, int warp, int lane) {
  if (!ok) {
    bars->ctl.abort = 1;
    raise_error(a.hdr + HDR_ERR, ERRBIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (bars->ctl.abort) {
    if (warp == FB_PRODUCER && lane == 0) {
      for (int k = bars->q_use; k < bars->q_fill; ++k) bounded_wait_plain(&bars->q_full[k & 1], (k >> 1) & 1);
      for (int k = bars->do_use; k < bars->do_fill; ++k) bounded_wait_plain(&bars->do_full, k & 1);
      if (bars->own_issued > bars->own_used) bounded_wait_plain(&bars->own_full, (bars->own_issued - 1) & 1);
    }
    if (warp == FB_MMA && lane == 0) {
      mma_commit(&bars->drain);
      bounded_wait_plain(&bars->drain, 0);
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

template <bool TEST>
__global__ void __launch_bounds__(FB_THREADS, 1)
    dkdvq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                 const __grid_constant__ CUtensorMap tdq, const FbArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FbBars *bars = reinterpret_cast<FbBars *>(smem + FB_SM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
      mbar_init(&bars->item_full[s], 1);
      mbar_init(&bars->item_empty[s], 9);   // softmax 8 + MMA 1 warps
    }
    mbar_init(&bars->do_full, 1);
    mbar_init(&bars->do_empty, 1);
    mbar_init(&bars->own_full, 1);
    mbar_init(&bars->own_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, 8);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->drain, 1);
    if (TEST) mbar_init(&bars->never, 1);
    bars->ctl.init(a.wait);
    bars->q_fill = bars->q_use = bars->do_fill = bars->do_use = bars->own_issued = bars->own_used = 0;
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
    tma_prefetch_desc(&tdq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  bool ok = true;
  if (warp < FB_PRODUCER) {
    ok = fb_softmax(&tdq, a, smem, bars, tmem, warp >> 2, warp, lane);
  } else if (warp == FB_PRODUCER) {
    if (lane == 0) ok = fb_producer<TEST>(&tq, &tk, &tv, &tdo, a, smem, bars);
    __syncwarp();
  } else if (warp == FB_MMA) {
    ok = fb_mma(a, smem, bars, tmem, lane);
  }
  fb_finish(ok, a, bars, tmem, warp, lane);
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

cudaError_t launch_dkdvq(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tdo,
                         const CUtensorMap &tdqacc, void *dq, void *dk, void *dv, const Problem &p, void *workspace,
                         cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done[2] = {{0}, {0}};
  const bool test = wait_bound().test != 0;
  {
    const void *kern = test ? reinterpret_cast<const void *>(dkdvq_kernel<true>)
                            : reinterpret_cast<const void *>(dkdvq_kernel<false>);
    const cudaError_t e = smem_attr_once(kern, FB_SMEM, attr_done[test ? 1 : 0]);
    if (e != cudaSuccess) return e;
  }
  const Workspace w = Workspace::layout(p.B, p.S, p.H);
  char *base = static_cast<char *>(workspace);
  FbArgs a;
  a.lo = reinterpret_cast<const int *>(base + w.off_lo);
  a.kend = reinterpret_cast<const int *>(base + w.off_kend);
  a.list = reinterpret_cast<const int *>(base + w.off_list_kv);
  a.delta = reinterpret_cast<const float *>(base + w.off_delta);
  a.lse2 = reinterpret_cast<const float *>(base + w.off_lse2);
  a.hdr = reinterpret_cast<int *>(base + w.off_hdr);
  a.dk = static_cast<__nv_bfloat16 *>(dk);
  a.dv = static_cast<__nv_bfloat16 *>(dv);
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
  float *dqacc = reinterpret_cast<float *>(base + w.off_dqacc);
  cudaError_t e = cudaMemsetAsync(dqacc, 0, w.dqacc_bytes, stream);
  if (e != cudaSuccess) return e;
  const int grid = a.n_items < p.num_sms ? a.n_items : p.num_sms;
  if (test) dkdvq_kernel<true><<<grid, FB_THREADS, FB_SMEM, stream>>>(tq, tk, tv, tdo, tdqacc, a);
  else dkdvq_kernel<false><<<grid, FB_THREADS, FB_SMEM, stream>>>(tq, tk, tv, tdo, tdqacc, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long total = (long long)p.B * p.S * p.H * (HD / 8);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)p.num_sms * 16;
  if (blocks > cap) blocks = cap;
  dq_convert_kernel<<<int(blocks), 256, 0, stream>>>(reinterpret_cast<const float4 *>(dqacc),
                                                      static_cast<uint4 *>(dq), p.B, p.S, p.H, w.S_pad,
                                                      a.inv_sqrt_d);
  return cudaGetLastError();
}

}  // namespace lwm
