// Shared device helpers for the sm_103a attention kernels: inline-PTX wrappers for
// mbarriers, TMA tensor copies and the 5th-generation tensor core (tcgen05 / TMEM),
// bounded waits, and the workspace layout that the host launcher and every kernel
// agree on.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lwm_attn.h"

namespace lwm {

// ----------------------------------------------------------------------------- tiling
constexpr int HD = 128;            // head dimension (the only one supported)
constexpr int BM = 128;            // query rows per tile (one TMEM lane per row)
constexpr int BN = 128;            // keys per tile
constexpr int TILE_BYTES = BM * HD * 2;        // one 128 x 128 bf16 tile: 32 KiB
constexpr int HALF_BYTES = TILE_BYTES / 2;     // 128 rows x 64 dims, 128B-swizzled
constexpr int NBINS = 4096;                    // cost buckets of the longest-first sort

// Device error word values (a bit mask; lwm_attn_check maps it to a status).
constexpr int ERRBIT_SEGMENTS = 1;
constexpr int ERRBIT_TIMEOUT = 2;
constexpr int ERRBIT_LENGTHS = 4;   // decode: a kv_len outside [T, S_max]
constexpr int ERRBIT_TARGETS = 8;   // packed loss: a weighted token's target outside [0, V)

// ----------------------------------------------------------------------------- workspace
// Header words (int32) at the start of the workspace.
enum HeaderWord {
  HDR_ERR = 0,          // error bits
  HDR_KV_CHUNK = 1,     // ring chunk length in key tiles
  HDR_TICKET_FWD = 4,   // persistent-scheduler tickets and exit counters
  HDR_DONE_FWD = 5,
  HDR_TICKET_DKDV = 6,
  HDR_DONE_DKDV = 7,
  HDR_TICKET_DQ = 8,
  HDR_DONE_DQ = 9,
  HDR_TICKET_FUSED = 10,
  HDR_DONE_FUSED = 11,
  HDR_WORDS = 64
};

constexpr int XROW_BYTES = 16;     // one bf16 offset row of the dK/dV kernel (see Workspace)

struct Workspace {
  size_t off_hdr, off_lo, off_kend, off_list_fwd, off_list_kv, off_list_q, off_delta, off_lse2, off_qx, off_dox,
      off_dqacc, total;
  size_t dqacc_bytes;
  int nT, nP, S_pad;   // S_pad = nT * BM: per-row stride of lo, delta and lse2

  __host__ __device__ static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

  __host__ __device__ static Workspace layout(int B, int S, int H) {
    Workspace w;
    w.nT = (S + BM - 1) / BM;
    w.nP = (w.nT + 1) / 2;
    w.S_pad = w.nT * BM;
    size_t o = 0;
    w.off_hdr = o;      o += align256(HDR_WORDS * 4);
    w.off_lo = o;       o += align256(size_t(B) * w.S_pad * 4);
    w.off_kend = o;     o += align256(size_t(B) * w.nT * 4);
    w.off_list_fwd = o; o += align256(size_t(B) * w.nP * 4);
    w.off_list_kv = o;  o += align256(size_t(B) * w.nT * 4);
    w.off_list_q = o;   o += align256(size_t(B) * w.nT * 4);
    // backward row terms, fp32 [B, H, nT * BM] (rows padded to whole tiles)
    w.off_delta = o;    o += align256(size_t(B) * H * w.S_pad * 4);
    w.off_lse2 = o;     o += align256(size_t(B) * H * w.S_pad * 4);
    // the same two row terms as the dK/dV kernel's offset rows, bf16 [B, H, S_pad, 8]:
    // -lse * sqrt(D) and -delta, each as hi + mid + lo (see delta_kernel)
    w.off_qx = o;       o += align256(size_t(B) * H * w.S_pad * XROW_BYTES);
    w.off_dox = o;      o += align256(size_t(B) * H * w.S_pad * XROW_BYTES);
    // fp32 dQ accumulator of the single-kernel backward pass, [B, H, S_pad, D]
    w.dqacc_bytes = size_t(B) * H * w.S_pad * HD * 4;
    w.off_dqacc = o;    o += align256(w.dqacc_bytes);
    w.total = o;
    return w;
  }
};

// ----------------------------------------------------------------------------- PTX: misc
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Paired fp32 arithmetic (f32x2: two lanes per 64-bit register pair, one instruction).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);   // .x (low half) = lo
  return *reinterpret_cast<uint32_t *>(&v);
}

// ----------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded waiting. Every wait of a pipeline role gives up after `limit_ns` of wall
// time (a phase that never completes would otherwise hang the GPU) or as soon as
// another role of the CTA has raised `abort` after its own wait gave up. The kernels
// then let copies and products in flight land, free TMEM and return; the host reads
// the error word. The bound is a launch parameter (WaitBound, from the process-wide
// setting of lwm_attn_set_wait_limit), so that a test can shorten it and watch the
// waits run out; the fast path of a wait is a single try_wait on the barrier.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // 2 s: far above any legitimate wait

// Bounds below this are test settings (the failure test): the host then launches each
// kernel's test instantiation, whose producer waits once, with work in flight, for a
// phase that never completes (test_expiry_wait), so that the bound runs out for certain.
// A suspending try_wait usually sees a real phase complete before any clock check, so
// shortening the bound alone would not make waits run out. The production
// instantiations contain no test code at all (it would shift their code layout).
constexpr uint64_t SHORT_WAIT_LIMIT_NS = 1000000ull;

// The bound as a kernel launch parameter.
struct WaitBound {
  unsigned long long limit_ns;   // WAIT_LIMIT_NS unless a test shortened it
  int test;                      // limit_ns < SHORT_WAIT_LIMIT_NS: the failure test
};

struct WaitCtl {
  int abort;           // raised by the role whose wait ran out; the others poll it
  int unused;
  uint64_t limit_ns;   // bound of the pipeline waits

  __device__ __forceinline__ void init(const WaitBound &b) {
    abort = 0;
    limit_ns = b.limit_ns;
  }
};

// The fast path is one (suspending) try_wait; only after it fails are the abort flag and
// the clock consulted, every 64 polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, WaitCtl *ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  const uint64_t limit = ctl->limit_ns;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*reinterpret_cast<volatile int *>(&ctl->abort)) return false;
      if (global_timer_ns() - t0 > limit) return false;
    }
  }
}

// The failure test's wait, compiled only into the kernels' test instantiations: a phase
// that nothing ever completes (an mbarrier that no thread arrives on), waited for under
// the test's short bound, with the clock read on every poll, at a point where copies and
// products are in flight, so that the abort path has real work to let land.
__device__ __forceinline__ bool test_expiry_wait(uint64_t *never, WaitCtl *ctl) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(never, 0)) return true;
    if (global_timer_ns() - t0 > ctl->limit_ns) return false;
  }
}

// Spins (bounded like mbar_wait) until *count reaches target.
__device__ __forceinline__ bool wait_count(volatile int *count, int target, WaitCtl *ctl) {
  if (*count >= target) return true;
  const uint64_t t0 = global_timer_ns();
  const uint64_t limit = ctl->limit_ns;
  for (uint32_t it = 1; *count < target; ++it) {
    if ((it & 63u) == 0u) {
      if (*reinterpret_cast<volatile int *>(&ctl->abort)) return false;
      if (global_timer_ns() - t0 > limit) return false;
    }
  }
  return true;
}

// Waits of the abort path (copies and products in flight must land before shared
// memory and TMEM are released): always the full default bound, never the
// configurable one.
__device__ __forceinline__ bool bounded_wait_plain(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
  return true;
}

// ----------------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled load into shared memory; completion is signalled on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_4d(const CUtensorMap *map, uint64_t *bar, void *dst, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Plain (untiled) bulk copy global -> shared; both addresses 16-byte aligned and
// `bytes` a multiple of 16. Completion is signalled on `bar` (tx bytes).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ----------------------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// The same descriptor for a K-major operand stored without swizzle: core matrices of
// 8 rows x 16 bytes (128 contiguous bytes); lbo = byte offset between the two core
// matrices along K (a K = 16 bf16 slice), sbo = byte offset between 8-row groups.
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  return d;
}

// Register reconfiguration of a whole warpgroup (all four warps execute the same one).
// A shrink returns registers to the CTA's pool at once; a grow waits until the pool
// holds them, so the grows of a kernel must fit what its shrinks release plus what the
// launch left unused.
template <int N>
__device__ __forceinline__ void reg_shrink() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg count");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_grow() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg count");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Makes this thread's shared-memory stores visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Instruction descriptor for kind::f16 with bf16 inputs and an fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn_major) << 15) | (uint32_t(b_mn_major) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T-by-descriptor
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 32 columns of 32-bit: thread t of the warp gets lane (base + t), 32 values.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 16 columns of 32-bit.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t *v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ----------------------------------------------------------------------------- 128x128x128 products
// Instruction descriptors of the 128 x 128 (M x N) bf16 products with fp32 accumulation.
constexpr uint32_t IDESC_128_KK = idesc_bf16(128, 128, false, false);   // A, B both K-major
constexpr uint32_t IDESC_128_KM = idesc_bf16(128, 128, false, true);    // A K-major (or TMEM), B MN-major
constexpr uint32_t IDESC_128_MM = idesc_bf16(128, 128, true, true);     // A, B both MN-major

// D[128 x 128] (+)= A[128 rows x 128] . B[128 rows x 128]^T over the 128-wide inner
// dimension; both operands are 128-row tiles stored as two 64-column 128B-swizzled
// boxes HALF_BYTES apart (K-major: rows 128 bytes apart, 8-row groups 1024 bytes apart).
__device__ __forceinline__ void mma_tile_kk(uint32_t d_tmem, uint32_t a_s, uint32_t b_s, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = uint32_t(kk >> 2) * HALF_BYTES + uint32_t(kk & 3) * 32;
    mma_ss(d_tmem, sdesc_sw128(a_s + off, 16, 1024), sdesc_sw128(b_s + off, 16, 1024), IDESC_128_KK,
           (accumulate || kk > 0) ? 1u : 0u);
  }
}

// D[128 x 128] (+)= X[128 x 128] . Y[128 x 128] with X bf16 in TMEM (the inner block kk
// of 16 at column x_tmem + 16 kk, 8 packed columns) and Y a 128-row tile read MN-major
// (its rows are the inner dimension: 16 rows = two 8-row groups of 1024 bytes; the two
// 64-column boxes HALF_BYTES apart are the N halves).
__device__ __forceinline__ void mma_tile_ts(uint32_t d_tmem, uint32_t x_tmem, uint32_t y_s, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts(d_tmem, x_tmem + uint32_t(kk) * 16, sdesc_sw128(y_s + uint32_t(kk) * 2048, HALF_BYTES, 1024),
           IDESC_128_KM, (accumulate || kk > 0) ? 1u : 0u);
}

// The same product with X packed contiguously in TMEM: inner block kk at x_tmem + 8 kk.
__device__ __forceinline__ void mma_tile_ts_packed(uint32_t d_tmem, uint32_t x_tmem, uint32_t y_s, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts(d_tmem, x_tmem + uint32_t(kk) * 8, sdesc_sw128(y_s + uint32_t(kk) * 2048, HALF_BYTES, 1024),
           IDESC_128_KM, (accumulate || kk > 0) ? 1u : 0u);
}

// ----------------------------------------------------------------------------- tile ranges
// Inclusive range of key tiles that query tile [q0, q0+BM) of one batch row needs.
// `lo_row[i]` is the first key visible to query i (its document start; i+1 for
// padding and for the rows S..S_pad-1 past the end). Documents are contiguous, so lo is non-decreasing and the range is
// [lo[q0] / BN, last_row / BN]. Empty (first > last) when no row sees anything.
struct TileRange {
  int first, last;
  __device__ __forceinline__ bool has(int t) const { return t >= first && t <= last; }
  __device__ __forceinline__ bool empty() const { return first > last; }
};

__device__ __forceinline__ TileRange q_tile_kv_range(const int *lo_row, int S, int q0) {
  TileRange r{1, 0};
  if (q0 >= S) return r;
  const int qb = min(q0 + BM, S) - 1;
  const int la = lo_row[q0];
  if (la > qb) return r;
  r.first = la / BN;
  r.last = qb / BN;
  return r;
}

// Key-tile sequence in ring order: the key tiles are grouped into chunks of `cs`
// tiles; the chunk holding the last tile is visited first, then the chunks before it,
// each in ascending tile order, all clipped to [first, last].
struct KvSeq {
  int first, last, cs, c, t, tend;
  __device__ __forceinline__ void init(int first_, int last_, int cs_) {
    first = first_;
    last = last_;
    cs = cs_;
    if (first > last) {
      t = 1;
      tend = 0;
      return;
    }
    c = last / cs;
    t = max(first, c * cs);
    tend = last;
  }
  __device__ __forceinline__ bool valid() const { return t <= tend; }
  __device__ __forceinline__ void next() {
    if (t < tend) {
      ++t;
      return;
    }
    --c;
    if (c < 0 || c * cs + cs - 1 < first) {
      t = 1;
      tend = 0;
      return;
    }
    t = max(first, c * cs);
    tend = min(last, c * cs + cs - 1);
  }
};

__device__ __forceinline__ void raise_error(int *err_word, int bits) { atomicOr(err_word, bits); }

}  // namespace lwm
