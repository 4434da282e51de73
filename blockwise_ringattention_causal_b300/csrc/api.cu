// C ABI of the attention library: argument checks, TMA tensor maps and kernel
// launches. See include/lwm_attn.h for the contract of every entry point.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace lwm {
namespace {

constexpr int MAX_DEVICES = 64;

struct DeviceInfo {
  bool known = false;
  bool supported = false;
  int num_sms = 0;
};

std::mutex g_mu;
std::atomic<uint64_t> g_wait_limit_ns{0};   // lwm_attn_set_wait_limit (0 = WAIT_LIMIT_NS)
DeviceInfo g_dev[MAX_DEVICES];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

thread_local char g_last_error[512] = "";

lwm_status fail(const char *what, const char *detail) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, detail);
  return LWM_ERR_CUDA;
}

lwm_status cuda_check(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return LWM_OK;
  cudaGetLastError();   // clear the sticky-free error so later calls start clean
  return fail(what, cudaGetErrorString(e));
}

#define from_cuda(call) cuda_check((call), #call)

lwm_status device_info(DeviceInfo &out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return fail("cudaGetDevice", "no device");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo &d = g_dev[dev];
  if (!d.known) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return fail("cudaDeviceGetAttribute", "failed");
    d.supported = (major == 10 && minor == 3);   // the kernels are built for sm_103a
    d.num_sms = sms;
    d.known = true;
  }
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return fail("cudaGetDriverEntryPointByVersion", "cuTensorMapEncodeTiled not found");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  out = d;
  return d.supported ? LWM_OK : LWM_ERR_UNSUPPORTED;
}

// [B, S, H, 128] bf16, loaded as boxes of 64 dims x 1 head x `rows` rows x 1 batch row,
// 128-byte swizzled (the K-major / MN-major canonical layout of the MMA operands).
CUresult make_map_raw(CUtensorMap *m, const void *ptr, int B, int S, int H, int rows) {
  cuuint64_t dims[4] = {cuuint64_t(HD), cuuint64_t(H), cuuint64_t(S), cuuint64_t(B)};
  cuuint64_t strides[3] = {cuuint64_t(HD) * 2, cuuint64_t(H) * HD * 2, cuuint64_t(S) * H * HD * 2};
  cuuint32_t box[4] = {64, 1, cuuint32_t(rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

bool make_map(CUtensorMap *m, const void *ptr, int B, int S, int H, int rows = BM) {
  const CUresult r = make_map_raw(m, ptr, B, S, H, rows);
  if (r != CUDA_SUCCESS) {
    char buf[64];
    std::snprintf(buf, sizeof(buf), "CUresult %d", int(r));
    fail("cuTensorMapEncodeTiled", buf);
    return false;
  }
  return true;
}

// The fp32 dQ accumulator [B * H * S_pad rows, 128 dims] of the workspace, written by
// tensor reduce-add copies of 8-row x 32-dim boxes.
bool make_dqacc_map(CUtensorMap *m, void *ws, int B, int S, int H) {
  const Workspace w = Workspace::layout(B, S, H);
  cuuint64_t dims[2] = {cuuint64_t(HD), cuuint64_t(B) * H * w.S_pad};
  cuuint64_t strides[1] = {cuuint64_t(HD) * 4};
  cuuint32_t box[2] = {32, 8};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, static_cast<char *>(ws) + w.off_dqacc, dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[64];
    std::snprintf(buf, sizeof(buf), "CUresult %d", int(r));
    fail("cuTensorMapEncodeTiled (dQ accumulator)", buf);
    return false;
  }
  return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

lwm_status check_sizes(int B, int S, int H, int D) {
  if (B <= 0 || S <= 0 || H <= 0 || D <= 0) return LWM_ERR_INVALID_ARG;
  if (D != HD) return LWM_ERR_UNSUPPORTED;
  const long long nT = (S + BM - 1) / BM;
  if (static_cast<long long>(B) * S >= (1ll << 31)) return LWM_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * ((nT + 1) / 2) * H >= (1ll << 31)) return LWM_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * nT * H >= (1ll << 31)) return LWM_ERR_INVALID_ARG;
  return LWM_OK;
}

WaitBound wait_bound() {
  const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
  WaitBound b;
  b.limit_ns = v ? v : WAIT_LIMIT_NS;
  b.test = b.limit_ns < SHORT_WAIT_LIMIT_NS ? 1 : 0;
  return b;
}

lwm_status check_device() {
  DeviceInfo d;
  return device_info(d);
}

namespace {

// `with_dqacc`: the call runs the single-kernel backward pass, which needs the whole
// layout; every other call needs only the part in front of the dQ accumulator.
lwm_status check_workspace(const void *ws, size_t bytes, int B, int S, int H, bool with_dqacc) {
  if (!ws) return LWM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return LWM_ERR_WORKSPACE;
  const Workspace w = Workspace::layout(B, S, H);
  if (bytes < (with_dqacc ? w.total : w.off_dqacc)) return LWM_ERR_INVALID_ARG;
  return LWM_OK;
}



#define LWM_TRY(x)                 \
  do {                             \
    const lwm_status s_ = (x);     \
    if (s_ != LWM_OK) return s_;   \
  } while (0)

lwm_status prepare_impl(const int32_t *seg, const int32_t *pos, int B, int S, int H, int kv_chunks, void *ws,
                        cudaStream_t stream) {
  const int nT = (S + BM - 1) / BM;
  int chunk_tiles = (nT + kv_chunks - 1) / kv_chunks;
  if (chunk_tiles < 1) chunk_tiles = 1;
  return from_cuda(launch_meta(seg, pos, B, S, chunk_tiles, ws, stream));
}

lwm_status fwd_common(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, lwm_bf16 *out, float *lse,
                      int B, int S, int H, void *ws, cudaStream_t stream, const DeviceInfo &d) {
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, B, S, H) || !make_map(&tk, k, B, S, H) || !make_map(&tv, v, B, S, H))
    return LWM_ERR_CUDA;
  Problem p{B, S, H, d.num_sms};
  return from_cuda(launch_fwd(tq, tk, tv, out, lse, p, ws, stream));
}

lwm_status check_fwd_args(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, lwm_bf16 *out, float *lse,
                          int B, int S, int H, int D, void *ws, size_t ws_bytes) {
  LWM_TRY(check_sizes(B, S, H, D));
  if (!q || !k || !v || !out || !lse) return LWM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned4(lse))
    return LWM_ERR_ALIGNMENT;
  return check_workspace(ws, ws_bytes, B, S, H, false);
}

lwm_status check_seg_args(const int32_t *seg, const int32_t *pos) {
  if ((seg && !aligned4(seg)) || (pos && !aligned4(pos))) return LWM_ERR_ALIGNMENT;
  return LWM_OK;
}

lwm_status check_bwd_args(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const lwm_bf16 *out,
                          const lwm_bf16 *dout, const float *lse, lwm_bf16 *dq, lwm_bf16 *dk, lwm_bf16 *dv, int B,
                          int S, int H, int D, void *ws, size_t ws_bytes) {
  LWM_TRY(check_sizes(B, S, H, D));
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return LWM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned4(lse))
    return LWM_ERR_ALIGNMENT;
  return check_workspace(ws, ws_bytes, B, S, H, false);
}

lwm_status bwd_common(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const lwm_bf16 *out,
                      const lwm_bf16 *dout, const float *lse, lwm_bf16 *dq, lwm_bf16 *dk, lwm_bf16 *dv, int B,
                      int S, int H, unsigned stages, void *ws, cudaStream_t stream, const DeviceInfo &d) {
  Problem p{B, S, H, d.num_sms};
  if (stages & LWM_BWD_DELTA) LWM_TRY(from_cuda(launch_delta(out, dout, lse, p, ws, stream)));
  if (!(stages & (LWM_BWD_DKDV | LWM_BWD_DQ | LWM_BWD_FUSED))) return LWM_OK;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_map(&tq, q, B, S, H) || !make_map(&tk, k, B, S, H) || !make_map(&tv, v, B, S, H) ||
      !make_map(&tdo, dout, B, S, H))
    return LWM_ERR_CUDA;
  if (stages & LWM_BWD_FUSED) {
    CUtensorMap tacc;
    if (!make_dqacc_map(&tacc, ws, B, S, H)) return LWM_ERR_CUDA;
    LWM_TRY(from_cuda(launch_dkdvq(tq, tk, tv, tdo, tacc, dq, dk, dv, p, ws, stream)));
  }
  if (stages & LWM_BWD_DKDV) LWM_TRY(from_cuda(launch_dkdv(tq, tk, tv, tdo, dk, dv, p, ws, stream)));
  if (stages & LWM_BWD_DQ) LWM_TRY(from_cuda(launch_dq(tq, tk, tv, tdo, dq, p, ws, stream)));
  return LWM_OK;
}

// Argument checks for the selected backward stages only.
lwm_status check_stage_args(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const lwm_bf16 *out,
                            const lwm_bf16 *dout, const float *lse, lwm_bf16 *dq, lwm_bf16 *dk, lwm_bf16 *dv,
                            int B, int S, int H, int D, unsigned stages, void *ws, size_t ws_bytes) {
  LWM_TRY(check_sizes(B, S, H, D));
  if (stages == 0 || (stages & ~unsigned(LWM_BWD_ALL | LWM_BWD_FUSED))) return LWM_ERR_INVALID_ARG;
  if ((stages & LWM_BWD_FUSED) && (stages & (LWM_BWD_DKDV | LWM_BWD_DQ))) return LWM_ERR_INVALID_ARG;
  const void *need16[10];
  int n = 0;
  if (stages & LWM_BWD_DELTA) {
    if (!lse) return LWM_ERR_INVALID_ARG;
    if (!aligned4(lse)) return LWM_ERR_ALIGNMENT;
    need16[n++] = out;
    need16[n++] = dout;
  }
  if (stages & (LWM_BWD_DKDV | LWM_BWD_DQ | LWM_BWD_FUSED)) {
    need16[n++] = q;
    need16[n++] = k;
    need16[n++] = v;
    need16[n++] = dout;
  }
  if (stages & (LWM_BWD_DKDV | LWM_BWD_FUSED)) {
    need16[n++] = dk;
    need16[n++] = dv;
  }
  if (stages & (LWM_BWD_DQ | LWM_BWD_FUSED)) need16[n++] = dq;
  for (int i = 0; i < n; ++i) {
    if (!need16[i]) return LWM_ERR_INVALID_ARG;
    if (!aligned16(need16[i])) return LWM_ERR_ALIGNMENT;
  }
  return check_workspace(ws, ws_bytes, B, S, H, (stages & LWM_BWD_FUSED) != 0);
}

}  // namespace

// Forward pass (metadata pre-pass + forward kernel) into a workspace that holds at
// least the forward part of the layout (Workspace::layout(B, S, 1).total bytes).
// Arguments are checked by the caller.
lwm_status fwd_with_forward_workspace(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const int32_t *seg,
                                      const int32_t *pos, lwm_bf16 *out, float *lse, int B, int S, int H, void *ws,
                                      cudaStream_t stream) {
  DeviceInfo d;
  LWM_TRY(device_info(d));
  LWM_TRY(prepare_impl(seg, pos, B, S, H, 1, ws, stream));
  return fwd_common(q, k, v, out, lse, B, S, H, ws, stream, d);
}

}  // namespace lwm

using namespace lwm;

extern "C" {

size_t lwm_attn_workspace_size(int B, int S, int H, int D) {
  if (check_sizes(B, S, H, D) != LWM_OK) return 0;
  return Workspace::layout(B, S, H).total;
}

size_t lwm_attn_workspace_size_fwd(int B, int S, int H, int D) {
  if (check_sizes(B, S, H, D) != LWM_OK) return 0;
  return Workspace::layout(B, S, H).off_dqacc;
}

lwm_status lwm_attn_prepare(const int32_t *seg_ids, const int32_t *pos, int B, int S, int H, int D,
                            int kv_chunks, void *workspace, size_t workspace_bytes, lwm_stream stream) {
  LWM_TRY(check_sizes(B, S, H, D));
  if (kv_chunks < 1) return LWM_ERR_INVALID_ARG;
  LWM_TRY(check_seg_args(seg_ids, pos));
  LWM_TRY(check_workspace(workspace, workspace_bytes, B, S, H, false));
  DeviceInfo d;
  LWM_TRY(device_info(d));
  return prepare_impl(seg_ids, pos, B, S, H, kv_chunks, workspace, stream);
}

lwm_status lwm_attn_fwd_ring(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const int32_t *seg_ids,
                             const int32_t *pos, lwm_bf16 *out, float *lse, int B, int S, int H, int D,
                             int kv_chunks, void *workspace, size_t workspace_bytes, lwm_stream stream) {
  LWM_TRY(check_fwd_args(q, k, v, out, lse, B, S, H, D, workspace, workspace_bytes));
  if (kv_chunks < 1) return LWM_ERR_INVALID_ARG;
  LWM_TRY(check_seg_args(seg_ids, pos));
  DeviceInfo d;
  LWM_TRY(device_info(d));
  LWM_TRY(prepare_impl(seg_ids, pos, B, S, H, kv_chunks, workspace, stream));
  return fwd_common(q, k, v, out, lse, B, S, H, workspace, stream, d);
}

lwm_status lwm_attn_fwd(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const int32_t *seg_ids,
                        const int32_t *pos, lwm_bf16 *out, float *lse, int B, int S, int H, int D, void *workspace,
                        size_t workspace_bytes, lwm_stream stream) {
  return lwm_attn_fwd_ring(q, k, v, seg_ids, pos, out, lse, B, S, H, D, 1, workspace, workspace_bytes, stream);
}

lwm_status lwm_attn_fwd_prepared(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, lwm_bf16 *out,
                                 float *lse, int B, int S, int H, int D, void *workspace, size_t workspace_bytes,
                                 lwm_stream stream) {
  LWM_TRY(check_fwd_args(q, k, v, out, lse, B, S, H, D, workspace, workspace_bytes));
  DeviceInfo d;
  LWM_TRY(device_info(d));
  return fwd_common(q, k, v, out, lse, B, S, H, workspace, stream, d);
}

lwm_status lwm_attn_bwd(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const lwm_bf16 *out,
                        const lwm_bf16 *dout, const float *lse, const int32_t *seg_ids, const int32_t *pos,
                        lwm_bf16 *dq, lwm_bf16 *dk, lwm_bf16 *dv, int B, int S, int H, int D, void *workspace,
                        size_t workspace_bytes, lwm_stream stream) {
  LWM_TRY(check_bwd_args(q, k, v, out, dout, lse, dq, dk, dv, B, S, H, D, workspace, workspace_bytes));
  LWM_TRY(check_seg_args(seg_ids, pos));
  DeviceInfo d;
  LWM_TRY(device_info(d));
  LWM_TRY(prepare_impl(seg_ids, pos, B, S, H, 1, workspace, stream));
  return bwd_common(q, k, v, out, dout, lse, dq, dk, dv, B, S, H, LWM_BWD_ALL, workspace, stream, d);
}

lwm_status lwm_attn_bwd_prepared(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const lwm_bf16 *out,
                                 const lwm_bf16 *dout, const float *lse, lwm_bf16 *dq, lwm_bf16 *dk,
                                 lwm_bf16 *dv, int B, int S, int H, int D, void *workspace,
                                 size_t workspace_bytes, lwm_stream stream) {
  LWM_TRY(check_bwd_args(q, k, v, out, dout, lse, dq, dk, dv, B, S, H, D, workspace, workspace_bytes));
  DeviceInfo d;
  LWM_TRY(device_info(d));
  return bwd_common(q, k, v, out, dout, lse, dq, dk, dv, B, S, H, LWM_BWD_ALL, workspace, stream, d);
}

lwm_status lwm_attn_bwd_stages(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v, const lwm_bf16 *out,
                               const lwm_bf16 *dout, const float *lse, lwm_bf16 *dq, lwm_bf16 *dk, lwm_bf16 *dv,
                               int B, int S, int H, int D, unsigned stages, void *workspace,
                               size_t workspace_bytes, lwm_stream stream) {
  LWM_TRY(check_stage_args(q, k, v, out, dout, lse, dq, dk, dv, B, S, H, D, stages, workspace, workspace_bytes));
  DeviceInfo d;
  LWM_TRY(device_info(d));
  return bwd_common(q, k, v, out, dout, lse, dq, dk, dv, B, S, H, stages, workspace, stream, d);
}

lwm_status lwm_attn_check(void *workspace, lwm_stream stream) {
  if (!workspace) return LWM_ERR_INVALID_ARG;
  LWM_TRY(from_cuda(cudaStreamSynchronize(stream)));
  int word = 0;
  int *hdr = static_cast<int *>(workspace);
  LWM_TRY(from_cuda(cudaMemcpy(&word, hdr + HDR_ERR, sizeof(int), cudaMemcpyDeviceToHost)));
  if (word != 0) LWM_TRY(from_cuda(cudaMemset(hdr + HDR_ERR, 0, sizeof(int))));
  if (word & ERRBIT_SEGMENTS) return LWM_ERR_SEGMENTS;
  if (word & ERRBIT_LENGTHS) return LWM_ERR_LENGTHS;
  if (word & ERRBIT_TARGETS) return LWM_ERR_TARGETS;
  if (word & ERRBIT_TIMEOUT) return LWM_ERR_TIMEOUT;
  return LWM_OK;
}

lwm_status lwm_attn_rope(const lwm_bf16 *q, const lwm_bf16 *k, const int32_t *pos, double theta, lwm_bf16 *q_out,
                         lwm_bf16 *k_out, int B, int S, int H, int D, int inverse, lwm_stream stream) {
  LWM_TRY(check_sizes(B, S, H, D));
  if (!(theta > 0.0) || !std::isfinite(theta) || (inverse != 0 && inverse != 1)) return LWM_ERR_INVALID_ARG;
  if ((q == nullptr) != (q_out == nullptr) || (k == nullptr) != (k_out == nullptr) || (!q && !k))
    return LWM_ERR_INVALID_ARG;
  if ((q && (!aligned16(q) || !aligned16(q_out))) || (k && (!aligned16(k) || !aligned16(k_out))) ||
      (pos && !aligned4(pos)))
    return LWM_ERR_ALIGNMENT;
  DeviceInfo d;
  LWM_TRY(device_info(d));
  return from_cuda(launch_rope(q, k, pos, theta, q_out, k_out, B, S, H, inverse != 0, d.num_sms, stream));
}

size_t lwm_attn_decode_workspace_size(int B, int T, int S_max, int H, int D) {
  if (B <= 0 || B > 65535 || T < 1 || T > 4 || S_max < T || H <= 0 || D != HD) return 0;
  if (static_cast<long long>(B) * S_max * H >= (1ll << 31)) return 0;
  return decode_layout(B, T, S_max, H).total;
}

lwm_status lwm_attn_decode(const lwm_bf16 *q, const lwm_bf16 *k_cache, const lwm_bf16 *v_cache,
                           const int32_t *kv_len, lwm_bf16 *out, float *lse, int B, int T, int S_max, int H, int D,
                           void *workspace, size_t workspace_bytes, lwm_stream stream) {
  if (B <= 0 || T <= 0 || S_max <= 0 || H <= 0 || D <= 0) return LWM_ERR_INVALID_ARG;
  if (D != HD || T > 4) return LWM_ERR_UNSUPPORTED;
  const size_t need = lwm_attn_decode_workspace_size(B, T, S_max, H, D);
  if (need == 0) return LWM_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !out || !lse || !workspace) return LWM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned4(lse) ||
      (kv_len && !aligned4(kv_len)))
    return LWM_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LWM_ERR_WORKSPACE;
  if (workspace_bytes < need) return LWM_ERR_INVALID_ARG;
  DeviceInfo d;
  LWM_TRY(device_info(d));
  return from_cuda(launch_decode(q, k_cache, v_cache, kv_len, out, lse, B, T, S_max, H, workspace, stream));
}

size_t lwm_packed_loss_workspace_size(int B, int S) {
  if (B <= 0 || S <= 0 || B > 65535 || static_cast<long long>(B) * S >= (1ll << 31)) return 0;
  return loss_layout(B, S).total;
}

lwm_status lwm_packed_loss(const lwm_bf16 *logits, const int32_t *targets, const float *weight,
                           const int32_t *seg_ids, double *loss, lwm_bf16 *dlogits, int B, int S, int V,
                           void *workspace, size_t workspace_bytes, lwm_stream stream) {
  if (B <= 0 || S <= 0 || V <= 0) return LWM_ERR_INVALID_ARG;
  const size_t need = lwm_packed_loss_workspace_size(B, S);
  if (need == 0) return LWM_ERR_INVALID_ARG;
  if (V % 8 != 0) return LWM_ERR_UNSUPPORTED;
  if (!logits || !targets || !loss || !workspace) return LWM_ERR_INVALID_ARG;
  if (!aligned16(logits) || (dlogits && !aligned16(dlogits)) || !aligned4(targets) || (weight && !aligned4(weight)) ||
      (seg_ids && !aligned4(seg_ids)) || (reinterpret_cast<uintptr_t>(loss) & 7u) != 0)
    return LWM_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LWM_ERR_WORKSPACE;
  if (workspace_bytes < need) return LWM_ERR_INVALID_ARG;
  DeviceInfo d;
  LWM_TRY(device_info(d));
  return from_cuda(
      launch_packed_loss(logits, targets, weight, seg_ids, loss, dlogits, B, S, V, workspace, d.num_sms, stream));
}

lwm_status lwm_attn_set_wait_limit(uint64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
  return LWM_OK;
}

const char *lwm_last_error(void) { return g_last_error; }

const char *lwm_status_string(lwm_status status) {
  switch (status) {
    case LWM_OK: return "LWM_OK";
    case LWM_ERR_INVALID_ARG: return "LWM_ERR_INVALID_ARG: null pointer, bad size or too-small workspace";
    case LWM_ERR_UNSUPPORTED: return "LWM_ERR_UNSUPPORTED: only D == 128 on sm_103 devices";
    case LWM_ERR_ALIGNMENT: return "LWM_ERR_ALIGNMENT: tensors must be 16-byte aligned";
    case LWM_ERR_SEGMENTS: return "LWM_ERR_SEGMENTS: seg_ids/pos break the packing preconditions";
    case LWM_ERR_WORKSPACE: return "LWM_ERR_WORKSPACE: workspace must be 256-byte aligned";
    case LWM_ERR_CUDA: return "LWM_ERR_CUDA: a CUDA call failed";
    case LWM_ERR_TIMEOUT: return "LWM_ERR_TIMEOUT: a device pipeline wait exceeded its bound";
    case LWM_ERR_LENGTHS: return "LWM_ERR_LENGTHS: a decode kv_len is outside [T, S_max]";
    case LWM_ERR_TARGETS: return "LWM_ERR_TARGETS: a weighted token's target is outside [0, V)";
  }
  return "unknown lwm_status";
}

}  // extern "C"
