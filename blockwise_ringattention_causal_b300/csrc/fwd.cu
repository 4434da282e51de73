// Forward pass: exact causal, segment-masked softmax attention, block by block with an
// online softmax, on the sm_100-family tensor cores (tcgen05 + TMEM) with TMA-staged
// tiles.
//
// Method (LWM, "World Model on Million-Length Video And Language With Blockwise
// RingAttention"; deep-dive page, section "RingAttention 为什么必要"): exact attention
// computed block by block, so that memory stays linear in the sequence length. The
// per-block normaliser is the running max / running sum of the blockwise-transformer
// work the pages cite by title. On one GPU the ring of devices becomes the loop over
// key/value tiles below; kv_chunks > 1 visits the tiles in ring order.
//
// One persistent CTA per SM takes work items (b, h, pair of 128-row query tiles) from
// a head-major, longest-first list through an atomic ticket. Warp roles:
//   warps 0-3  softmax for query tile 0 (one TMEM lane = one query row per thread)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer (and the scheduler ticket)
//   warp  9    tcgen05 issuer of the S = Q K^T products (and TMEM owner)
//   warps 10, 11  tcgen05 issuers of the O_t += P_t V products of query tile 0, 1
// TMEM (512 columns): S (128 fp32 columns, shared by the two query tiles in turn) |
// P0 | P1 (64 columns each, bf16 pairs) | O0 | O1 (128 fp32 columns each). Because P
// has columns of its own, the S product of the next key tile does not wait for the P.V
// product of this one: it only needs the other tile's softmax to have read S out of
// TMEM, which it does first. So S(j+1) runs while the softmax still works on tile j,
// and the tensor core interleaves S0, S1, P0.V and P1.V products.
#include "common.cuh"
#include "kernels.h"

namespace lwm {
namespace {

constexpr int FWD_WARPS = 12;   // 3 warps per SM sub-partition: 168 registers each at launch
constexpr int FWD_THREADS = FWD_WARPS * 32;
constexpr int WARP_PRODUCER = 8;
constexpr int WARP_MMA = 9;    // issuer of the S products (and TMEM owner)
constexpr int WARP_PV0 = 10;   // issuers of the P.V products of query tiles 0 and 1
constexpr int WARP_PV1 = 11;
constexpr int KV_STAGES = 4;
// Register split (setmaxnreg): the block is launched with 168 registers per thread
// (384 threads, 64,512 in all); warpgroup 2 (producer and issuers) shrinks to
// FWD_REGS_OTHER and the two softmax warpgroups grow to FWD_REGS_SOFTMAX:
// 2 x 128 x 200 + 128 x 96 = 63,488 <= 64,512. At 168 the softmax, which holds a
// 128-column score row per thread, spilled about 11 values per warp and tile.
constexpr int FWD_REGS_SOFTMAX = 200, FWD_REGS_OTHER = 96;
static_assert(2 * 128 * FWD_REGS_SOFTMAX + 128 * FWD_REGS_OTHER <= 168 * FWD_THREADS,
              "register split must fit the launch's registers");
static_assert(KV_STAGES % 2 == 0, "K tiles take the even stages, V tiles the odd ones");

constexpr int SM_Q = 0;
constexpr int SM_KV = 2 * TILE_BYTES;
constexpr int SM_BAR = SM_KV + KV_STAGES * TILE_BYTES;

struct FwdBars {
  uint64_t kv_full[KV_STAGES], kv_empty[KV_STAGES];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], s_free, p_full[2], pv_done[2], o_empty[2];
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item[2];
  uint32_t tmem_base;
  WaitCtl ctl;
  int kv_fill, kv_use_k, kv_use_v[2], q_issued, q_used;
  int s_issued[2];   // S products of query tile t issued so far
  uint64_t never;    // the failure test's wait (test instantiation only)
};

constexpr int FWD_SMEM = SM_BAR + int(sizeof(FwdBars)) + 1024;   // + alignment slack

constexpr uint32_t COL_S = 0;                                                  // S (either tile)
__device__ __forceinline__ uint32_t col_p(int t) { return t ? 192u : 128u; }  // P_t
__device__ __forceinline__ uint32_t col_o(int t) { return t ? 384u : 256u; }  // O_t
constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, false, false);   // Q, K both K-major
constexpr uint32_t IDESC_PV = idesc_bf16(BM, HD, false, true);    // P from TMEM, V MN-major
constexpr float NEG_INF = -__builtin_huge_valf();

struct FwdArgs {
  const int *lo;
  const int *list;
  int *hdr;
  __nv_bfloat16 *out;
  float *lse;
  int B, S, H, nP, n_list, n_items, S_pad;
  float scale_log2;   // log2(e) / sqrt(D)
  WaitBound wait;
};

struct Item {
  int b, h, pair;
};

// Items of one head are consecutive (head-major), each head's query-tile pairs longest
// first, so that the CTAs running at the same time stream the same head's K and V
// through L2.
__device__ __forceinline__ Item decode(const FwdArgs &a, int item) {
  const int e = a.list[item % a.n_list];
  return {e / a.nP, item / a.n_list, e % a.nP};
}

// S = Q K^T over D = 128: 8 MMAs of K = 16; each 64-dim half of a tile is one
// 128B-swizzled K-major block (rows 128 bytes apart, 8-row groups 1024 bytes apart).
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_s, uint32_t k_s) {
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const uint32_t off = uint32_t(kk >> 2) * HALF_BYTES + uint32_t(kk & 3) * 32;
    mma_ss(d_tmem, sdesc_sw128(q_s + off, 16, 1024), sdesc_sw128(k_s + off, 16, 1024), IDESC_QK, kk > 0);
  }
}

// O (+)= P V over 128 keys: 8 MMAs of K = 16 keys; V is MN-major (dims contiguous):
// 16 keys = two 1024-byte 8-row groups; the two 64-dim halves are HALF_BYTES apart.
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_s, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    mma_ts(o_tmem, p_tmem + uint32_t(kk) * 8, sdesc_sw128(v_s + uint32_t(kk) * 2048, HALF_BYTES, 1024),
           IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
  }
}

struct Ranges {
  TileRange r[2];
  int first, last;
};

__device__ __forceinline__ Ranges item_ranges(const FwdArgs &a, const Item &I) {
  const int *lr = a.lo + size_t(I.b) * a.S_pad;
  Ranges R;
  R.r[0] = q_tile_kv_range(lr, a.S, (2 * I.pair) * BM);
  R.r[1] = q_tile_kv_range(lr, a.S, (2 * I.pair + 1) * BM);
  if (R.r[0].empty()) {
    R.first = R.r[1].first;
    R.last = R.r[1].last;
  } else if (R.r[1].empty()) {
    R.first = R.r[0].first;
    R.last = R.r[0].last;
  } else {
    R.first = min(R.r[0].first, R.r[1].first);
    R.last = max(R.r[0].last, R.r[1].last);
  }
  return R;
}

// ----------------------------------------------------------------------------- producer
template <bool TEST>
__device__ bool producer_role(const CUtensorMap *tq, const CUtensorMap *tk, const CUtensorMap *tv,
                              const FwdArgs &a, uint8_t *smem, FwdBars *bars, int kv_chunk) {
  WaitCtl *abort = &bars->ctl;
  int kv_fill = 0, q_issued = 0;
  bool ok = true;
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_empty[slot], ((it >> 1) & 1) ^ 1, abort))) break;
    const int t = atomicAdd(a.hdr + HDR_TICKET_FWD, 1);
    const int item = t < a.n_items ? t : -1;
    bars->item[slot] = item;
    mbar_arrive(&bars->item_full[slot]);
    if (item < 0) break;
    const Item I = decode(a, item);
    const Ranges R = item_ranges(a, I);
    if (!(ok = mbar_wait(&bars->q_empty, (it & 1) ^ 1, abort))) break;
    const int q0 = 2 * I.pair * BM;
    mbar_arrive_expect_tx(&bars->q_full, 2 * TILE_BYTES);
    tma_load_4d(tq, &bars->q_full, smem + SM_Q, 0, I.h, q0, I.b);
    tma_load_4d(tq, &bars->q_full, smem + SM_Q + HALF_BYTES, 64, I.h, q0, I.b);
    tma_load_4d(tq, &bars->q_full, smem + SM_Q + TILE_BYTES, 0, I.h, q0 + BM, I.b);
    tma_load_4d(tq, &bars->q_full, smem + SM_Q + TILE_BYTES + HALF_BYTES, 64, I.h, q0 + BM, I.b);
    ++q_issued;
    KvSeq seq;
    for (seq.init(R.first, R.last, kv_chunk); seq.valid() && ok; seq.next()) {
      for (int w = 0; w < 2; ++w) {
        const int st = kv_fill % KV_STAGES;
        if (!(ok = mbar_wait(&bars->kv_empty[st], ((kv_fill / KV_STAGES) & 1) ^ 1, abort))) break;
        mbar_arrive_expect_tx(&bars->kv_full[st], TILE_BYTES);
        const CUtensorMap *m = w ? tv : tk;
        uint8_t *dst = smem + SM_KV + st * TILE_BYTES;
        tma_load_4d(m, &bars->kv_full[st], dst, 0, I.h, seq.t * BN, I.b);
        tma_load_4d(m, &bars->kv_full[st], dst + HALF_BYTES, 64, I.h, seq.t * BN, I.b);
        ++kv_fill;
      }
    }
    if (!ok) break;
    // failure test only: wait, with this item's copies and products in flight, for a
    // phase that never completes (the short test bound makes the wait run out)
    if constexpr (TEST) {
      if (it == 0 && !(ok = test_expiry_wait(&bars->never, abort))) break;
    }
  }
  bars->kv_fill = kv_fill;
  bars->q_issued = q_issued;
  return ok;
}

// ----------------------------------------------------------------------------- MMA issuers
// Two issuing threads keep the tensor core busy where one could not: each tcgen05.mma
// issue costs the issuing thread about as long as the product takes to run.
//
// S issuer: per key tile in ring order, S_0 then S_1 (each only for a query tile that
// sees the key tile) into the shared S columns, each once the softmax that read the
// previous S has signalled s_free. Releases the K stage after its products and the Q
// tiles after the item's last product.
__device__ bool s_issuer_role(const FwdArgs &a, uint8_t *smem, FwdBars *bars, uint32_t tmem, int kv_chunk,
                              int lane) {
  WaitCtl *abort = &bars->ctl;
  const uint32_t kv_s0 = smem_u32(smem + SM_KV);
  int kv_use = 0, q_used = 0, n_s = 0, n_st[2] = {0, 0};
  bool ok = true;
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const Item I = decode(a, item);
    const Ranges R = item_ranges(a, I);
    if (!(ok = mbar_wait(&bars->q_full, it & 1, abort))) break;
    ++q_used;
    KvSeq seq;
    for (seq.init(R.first, R.last, kv_chunk); seq.valid() && ok; seq.next()) {
      const int stK = kv_use % KV_STAGES, parK = (kv_use / KV_STAGES) & 1;
      if (!(ok = mbar_wait(&bars->kv_full[stK], parK, abort))) break;
      kv_use += 2;
      bool used = false;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!R.r[t].has(seq.t)) continue;
        // the S columns are free once the softmax of the previous S has read them
        if (n_s > 0 && !(ok = mbar_wait(&bars->s_free, (n_s - 1) & 1, abort))) break;
        tc_fence_after();
        if (lane == 0) {
          issue_qk(tmem + COL_S, smem_u32(smem + SM_Q + t * TILE_BYTES), kv_s0 + stK * TILE_BYTES);
          mma_commit(&bars->s_full[t]);
          reinterpret_cast<volatile int *>(bars->s_issued)[t] = ++n_st[t];
        }
        __syncwarp();
        ++n_s;
        used = true;
      }
      if (!ok) break;
      if (lane == 0) {
        if (used) mma_commit(&bars->kv_empty[stK]);
        else mbar_arrive(&bars->kv_empty[stK]);
      }
      __syncwarp();
    }
    if (!ok) break;
    if (lane == 0) mma_commit(&bars->q_empty);
    __syncwarp();
  }
  if (lane == 0) {
    bars->kv_use_k = kv_use;
    bars->q_used = q_used;
  }
  return ok;
}

// P.V issuer of query tile t: per key tile in ring order, O_t += P_t V once the softmax
// has written P_t and rescaled O_t, then its share of the V stage's release. The first
// product of an item overwrites O_t once the previous item's O_t has been read out.
// P_t V of key tile j enters the tensor core's queue after S_t of key tile j + 1 (when
// the tile sees it): the softmax waits for that S, not for the P.V product. One issuer
// per tile, so that neither tile's P.V waits for the other's S.
__device__ bool pv_issuer_role(const FwdArgs &a, uint8_t *smem, FwdBars *bars, uint32_t tmem, int kv_chunk,
                               int t, int lane) {
  WaitCtl *abort = &bars->ctl;
  volatile int *s_issued = bars->s_issued + t;
  const uint32_t kv_s0 = smem_u32(smem + SM_KV);
  int kv_use = 0, n_pv = 0;
  uint32_t pf_par = 0, oe_par = 1;
  bool ok = true;
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const Item I = decode(a, item);
    const Ranges R = item_ranges(a, I);
    const TileRange my = R.r[t];
    bool first = true;
    KvSeq seq;
    for (seq.init(R.first, R.last, kv_chunk); seq.valid() && ok; seq.next()) {
      const int stV = (kv_use + 1) % KV_STAGES, parV = ((kv_use + 1) / KV_STAGES) & 1;
      if (!(ok = mbar_wait(&bars->kv_full[stV], parV, abort))) break;
      kv_use += 2;
      if (!my.has(seq.t)) {
        if (lane == 0) mbar_arrive(&bars->kv_empty[stV]);
        __syncwarp();
        continue;
      }
      if (first) {
        if (!(ok = mbar_wait(&bars->o_empty[t], oe_par, abort))) break;
        oe_par ^= 1;
      }
      if (!(ok = mbar_wait(&bars->p_full[t], pf_par, abort))) break;
      pf_par ^= 1;
      KvSeq nx = seq;
      nx.next();
      if (nx.valid() && my.has(nx.t) && !(ok = wait_count(s_issued, n_pv + 2, abort))) break;
      ++n_pv;
      tc_fence_after();
      if (lane == 0) {
        issue_pv(tmem + col_o(t), tmem + col_p(t), kv_s0 + stV * TILE_BYTES, !first);
        mma_commit(&bars->pv_done[t]);
        mma_commit(&bars->kv_empty[stV]);
      }
      __syncwarp();
      first = false;
    }
    if (!ok) break;
  }
  if (lane == 0) bars->kv_use_v[t] = kv_use;
  return ok;
}

// ----------------------------------------------------------------------------- softmax
__device__ bool softmax_role(const FwdArgs &a, FwdBars *bars, uint32_t tmem, int kv_chunk, int t, int warp,
                             int lane) {
  WaitCtl *abort = &bars->ctl;
  const int wq = warp & 3;
  const int r = wq * 32 + lane;
  const uint32_t lane_off = uint32_t(wq * 32) << 16;
  const uint32_t tS = tmem + lane_off + COL_S;
  const uint32_t tP = tmem + lane_off + col_p(t);
  const uint32_t tO = tmem + lane_off + col_o(t);
  const float c = a.scale_log2;
  uint32_t sf_par = 0, pd_par = 0;
  bool ok = true;

  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!(ok = mbar_wait(&bars->item_full[slot], (it >> 1) & 1, abort))) break;
    const int item = bars->item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
    if (item < 0) break;
    const Item I = decode(a, item);
    const Ranges R = item_ranges(a, I);
    const TileRange my = R.r[t];
    const int q0 = (2 * I.pair + t) * BM;
    const int i = q0 + r;
    const int *lr = a.lo + size_t(I.b) * a.S_pad;
    const int lo_i = i < a.S ? lr[i] : i + 1;
    const int qb = min(q0 + BM, a.S) - 1;
    const int lo_qb = q0 < a.S ? lr[qb] : 0;
    float m = NEG_INF, l = 0.f;
    bool had = false;

    KvSeq seq;
    for (seq.init(R.first, R.last, kv_chunk); seq.valid(); seq.next()) {
      const int kt = seq.t;
      if (!my.has(kt)) continue;
      if (!(ok = mbar_wait(&bars->s_full[t], sf_par, abort))) break;
      sf_par ^= 1;
      tc_fence_after();
      uint32_t s[BN];
      tmem_ld32(tS + 0, s);
      tmem_ld32(tS + 32, s + 32);
      tmem_ld32(tS + 64, s + 64);
      tmem_ld32(tS + 96, s + 96);
      tmem_ld_wait();
      // S is in registers: the S columns may take the next product
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free);
      const int k0 = kt * BN;
      const bool full = (lo_qb <= k0) && (k0 + BN - 1 <= q0);
      if (!full) {
#pragma unroll
        for (int cc = 0; cc < BN; ++cc) {
          const int j = k0 + cc;
          if (j < lo_i || j > i) s[cc] = 0xff800000u;   // -inf
        }
      }
      // row max: four independent chains of 3-input max
      float mq[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
      for (int cc = 0; cc < BN; cc += 8) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          mq[u] = max3f(mq[u], __uint_as_float(s[cc + 2 * u]), __uint_as_float(s[cc + 2 * u + 1]));
      }
      const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      const float m_new = fmaxf(m, mx * c);
      // Rescale only when the running max grew by more than 8 (log2 units); otherwise
      // keep the stale max: p <= 2^8 stays exact in fp32 and the final o = O / l uses
      // the same max for O and l.
      const bool resc = m_new > m + 8.f;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m - m_new);   // 0 when m = -inf
        m = m_new;
      }
      const bool fix_o = resc && had && l > 0.f;
      l *= alpha;
      const float m_use = (m == NEG_INF) ? 0.f : m;
      // p = exp2(s c - m) two at a time (paired fma and add), packed to bf16 pairs
      const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-m_use, -m_use);
      uint64_t acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
      uint32_t pk[BN / 2];
#pragma unroll
      for (int e = 0; e < BN / 2; ++e) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), c2, nm2), x0, x1);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        acc[e & 1] = f2_add(acc[e & 1], f2_pack(p0, p1));
        pk[e] = pack_bf16x2(p0, p1);
      }
      float a0, a1, b0, b1;
      f2_unpack(acc[0], a0, a1);
      f2_unpack(acc[1], b0, b1);
      l += (a0 + a1) + (b0 + b1);
      // P_t and O_t belong to the previous P.V product until it completes
      if (had) {
        if (!(ok = mbar_wait(&bars->pv_done[t], pd_par, abort))) break;
        pd_par ^= 1;
        tc_fence_after();
      }
#pragma unroll
      for (int cc = 0; cc < BN / 2; cc += 16) tmem_st16(tP + cc, pk + cc);
      // O rescale after the scores are dead (fewer live registers); it must land before
      // p_full lets the next P.V product accumulate into O.
      if (__any_sync(0xffffffffu, fix_o)) {
        const float f = fix_o ? alpha : 1.f;
#pragma unroll
        for (int cc = 0; cc < HD; cc += 16) {
          uint32_t o[16];
          tmem_ld16(tO + cc, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
          tmem_st16(tO + cc, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[t]);
      had = true;
    }
    if (!ok) break;

    const size_t orow = (size_t(I.b) * a.S + i) * a.H + I.h;
    if (had) {
      if (!(ok = mbar_wait(&bars->pv_done[t], pd_par, abort))) break;
      pd_par ^= 1;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int cc = 0; cc < HD; cc += 32) {
        uint32_t o[32];
        tmem_ld32(tO + cc, o);
        tmem_ld_wait();
        uint4 w[4];
        uint32_t *wp = reinterpret_cast<uint32_t *>(w);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          wp[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
        if (i < a.S) {
          uint4 *dst = reinterpret_cast<uint4 *>(a.out + orow * HD + cc);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = w[e];
        }
      }
      if (i < a.S) a.lse[(size_t(I.b) * a.H + I.h) * a.S + i] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : NEG_INF;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_empty[t]);
    } else if (i < a.S) {
      uint4 *dst = reinterpret_cast<uint4 *>(a.out + orow * HD);
#pragma unroll
      for (int e = 0; e < HD / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
      a.lse[(size_t(I.b) * a.H + I.h) * a.S + i] = NEG_INF;
    }
  }
  return ok;
}

template <bool TEST>
__global__ void __launch_bounds__(FWD_THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBars *bars = reinterpret_cast<FwdBars *>(smem + SM_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kv_chunk = a.hdr[HDR_KV_CHUNK];

  if (threadIdx.x == 0) {
    for (int s = 0; s < KV_STAGES; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], (s & 1) ? 2 : 1);   // K stages: the S issuer; V stages: both P.V issuers
    }
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->s_free, 4);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 4);
      mbar_init(&bars->pv_done[t], 1);
      mbar_init(&bars->o_empty[t], 4);
      mbar_init(&bars->item_full[t], 1);
      mbar_init(&bars->item_empty[t], 11);   // softmax 8 + MMA 3 warps
    }
    mbar_init(&bars->drain, 3);
    if (TEST) mbar_init(&bars->never, 1);
    bars->ctl.init(a.wait);
    bars->kv_fill = bars->kv_use_k = bars->kv_use_v[0] = bars->kv_use_v[1] = bars->q_issued = bars->q_used = 0;
    bars->s_issued[0] = bars->s_issued[1] = 0;
    fence_mbar_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == WARP_PRODUCER && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  bool ok = true;
  if (warp >= WARP_PRODUCER) {   // warpgroup 2: producer and MMA issuers, few registers each
    reg_shrink<FWD_REGS_OTHER>();
    if (warp == WARP_PRODUCER) {
      if (lane == 0) ok = producer_role<TEST>(&tq, &tk, &tv, a, smem, bars, kv_chunk);
      __syncwarp();
    } else if (warp == WARP_MMA) {
      ok = s_issuer_role(a, smem, bars, tmem, kv_chunk, lane);
    } else {
      ok = pv_issuer_role(a, smem, bars, tmem, kv_chunk, warp - WARP_PV0, lane);
    }
  } else {   // warpgroups 0, 1: softmax, a full 128-column score row per thread
    reg_grow<FWD_REGS_SOFTMAX>();
    ok = softmax_role(a, bars, tmem, kv_chunk, warp >> 2, warp, lane);
  }
  if (!ok) {
    bars->ctl.abort = 1;
    raise_error(a.hdr + HDR_ERR, ERRBIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (bars->ctl.abort) {
    // Let copies and MMAs still in flight land before shared memory and TMEM go away.
    if (warp == WARP_PRODUCER && lane == 0) {
      // loads no consumer has waited for: K (even n) from the S issuer's count, V (odd n)
      // from the further of the P.V issuers' counts
      const int use_v = max(bars->kv_use_v[0], bars->kv_use_v[1]);
      for (int n = min(bars->kv_use_k, use_v); n < bars->kv_fill; ++n)
        if (n >= ((n & 1) ? use_v : bars->kv_use_k))
          bounded_wait_plain(&bars->kv_full[n % KV_STAGES], (n / KV_STAGES) & 1);
      if (bars->q_issued > bars->q_used) bounded_wait_plain(&bars->q_full, (bars->q_issued - 1) & 1);
    }
    if ((warp == WARP_MMA || warp == WARP_PV0 || warp == WARP_PV1) && lane == 0) {
      mma_commit(&bars->drain);
      bounded_wait_plain(&bars->drain, 0);
    }
    __syncthreads();
  }
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    const int d = atomicAdd(a.hdr + HDR_DONE_FWD, 1);
    if (d == int(gridDim.x) - 1) {
      a.hdr[HDR_TICKET_FWD] = 0;
      a.hdr[HDR_DONE_FWD] = 0;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, void *out,
                       float *lse, const Problem &p, void *workspace, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done[2] = {{0}, {0}};
  const WaitBound wb = wait_bound();
  const void *kern = wb.test ? reinterpret_cast<const void *>(fwd_kernel<true>)
                             : reinterpret_cast<const void *>(fwd_kernel<false>);
  {
    const cudaError_t e = smem_attr_once(kern, FWD_SMEM, attr_done[wb.test ? 1 : 0]);
    if (e != cudaSuccess) return e;
  }
  const Workspace w = Workspace::layout(p.B, p.S, p.H);
  char *base = static_cast<char *>(workspace);
  FwdArgs a;
  a.lo = reinterpret_cast<const int *>(base + w.off_lo);
  a.list = reinterpret_cast<const int *>(base + w.off_list_fwd);
  a.hdr = reinterpret_cast<int *>(base + w.off_hdr);
  a.out = static_cast<__nv_bfloat16 *>(out);
  a.lse = lse;
  a.B = p.B;
  a.S = p.S;
  a.H = p.H;
  a.nP = w.nP;
  a.S_pad = w.S_pad;
  a.n_list = p.B * w.nP;
  a.n_items = a.n_list * p.H;
  a.scale_log2 = 1.4426950408889634f / sqrtf(float(HD));
  a.wait = wb;
  const int grid = a.n_items < p.num_sms ? a.n_items : p.num_sms;
  if (wb.test) fwd_kernel<true><<<grid, FWD_THREADS, FWD_SMEM, stream>>>(tq, tk, tv, a);
  else fwd_kernel<false><<<grid, FWD_THREADS, FWD_SMEM, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace lwm
