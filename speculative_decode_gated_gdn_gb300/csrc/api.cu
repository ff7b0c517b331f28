// api.cu -- the extern "C" boundary of libgdn_gb300.so: host-side validation,
// workspace sizing, dispatch to the kernels, and error reporting.
//
// Every check runs before anything is launched, so a rejected call leaves all
// device memory untouched ("Add request-owned eight-way MTP serving for Qwen
// 35B", Clean-install public launch verification: an incomplete launch
// contract fails before any work; "MTP inference: review and commit
// structure", Review fixes: grouped replay checks all inputs before combining
// layers).
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <cmath>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include "gdn_common.cuh"

using namespace gdn;

namespace {

thread_local std::string t_err;

// An NVTX range around each entry point (what a profiler timeline shows as
// the call's host-side extent; a no-op unless a tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}

int ok() {
  t_err.clear();
  return GDN_OK;
}

constexpr int kMaxPrefillLen = 1 << 20;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_dims(const gdn_dims *d) {
  if (!d) return fail(GDN_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 0 || d->B > 65535) return fail(GDN_ERR_UNSUPPORTED, "B=%d outside [0, 65535]", d->B);
  if (d->T < 1 || d->T > d->T_max || d->T_max > kMaxT)
    return fail(GDN_ERR_UNSUPPORTED, "need 1 <= T (%d) <= T_max (%d) <= %d", d->T, d->T_max, kMaxT);
  if (d->H_k < 1 || d->H_v < 1 || d->H_v % d->H_k != 0 || d->H_v > 65535)
    return fail(GDN_ERR_UNSUPPORTED, "need H_k >= 1 and H_v (%d) a multiple of H_k (%d), H_v <= 65535",
                d->H_v, d->H_k);
  if (d->d_k != d->d_v || (d->d_k != 32 && d->d_k != 64 && d->d_k != 128))
    return fail(GDN_ERR_UNSUPPORTED, "need d_k == d_v in {32, 64, 128} (got %d, %d)", d->d_k, d->d_v);
  if (d->width != kWidth) return fail(GDN_ERR_UNSUPPORTED, "conv width must be 4 (got %d)", d->width);
  if (d->act != GDN_ACT_NONE && d->act != GDN_ACT_SILU)
    return fail(GDN_ERR_INVALID_ARG, "act must be GDN_ACT_NONE or GDN_ACT_SILU (got %d)", d->act);
  const long long C = (2LL * d->H_k + d->H_v) * d->d_k;
  if (C > (1LL << 30)) return fail(GDN_ERR_UNSUPPORTED, "too many conv channels (%lld)", C);
  return GDN_OK;
}

int check_mode(int mode) {
  if (mode != GDN_COMMIT_RECOMPUTE && mode != GDN_COMMIT_SNAPSHOT && mode != GDN_COMMIT_DEFERRED)
    return fail(GDN_ERR_INVALID_ARG,
                "mode must be GDN_COMMIT_RECOMPUTE, GDN_COMMIT_SNAPSHOT or GDN_COMMIT_DEFERRED (got %d)", mode);
  return GDN_OK;
}

size_t layer_ws_bytes(const gdn_dims *d, int mode) {
  if (mode == GDN_COMMIT_RECOMPUTE) return recompute_ws(d->B, d->T, d->H_k, d->H_v, d->d_k).total;
  if (mode == GDN_COMMIT_DEFERRED) return deferred_ws(d->B, d->T, d->H_k, d->H_v, d->d_k).total;
  return snapshot_ws(d->B, d->T, d->H_v, d->d_k);
}

// Host arrays of per-layer device pointers for gdn_commit / gdn_flush.
int fill_layers(CommitParams &p, int n_layers, float *const *state, gdn_bf16 *const *ring, void *const *layer_ws) {
  if (n_layers < 1 || n_layers > kMaxLayers)
    return fail(GDN_ERR_INVALID_ARG, "n_layers=%d outside [1, %d]", n_layers, kMaxLayers);
  if (!state || !layer_ws) return fail(GDN_ERR_INVALID_ARG, "state / layer_ws host arrays are NULL");
  for (int l = 0; l < n_layers; ++l) {
    if (!state[l] || !layer_ws[l]) return fail(GDN_ERR_INVALID_ARG, "layer %d: NULL state or workspace", l);
    if (!aligned(state[l], 16)) return fail(GDN_ERR_MISALIGNED, "layer %d: state not 16-byte aligned", l);
    if (!aligned(layer_ws[l], 256))
      return fail(GDN_ERR_MISALIGNED, "layer %d: workspace not 256-byte aligned", l);
    p.state[l] = state[l];
    p.ws[l] = static_cast<float *>(layer_ws[l]);
    if (ring) {
      if (!ring[l]) return fail(GDN_ERR_INVALID_ARG, "layer %d: NULL ring", l);
      if (!aligned(ring[l], 16)) return fail(GDN_ERR_MISALIGNED, "layer %d: ring not 16-byte aligned", l);
      p.ring[l] = reinterpret_cast<uint16_t *>(ring[l]);
    }
  }
  p.n_layers = n_layers;
  return GDN_OK;
}

#define GDN_NEED_PTR(ptr, align)                                                             \
  do {                                                                                       \
    if (!(ptr)) return fail(GDN_ERR_INVALID_ARG, "%s is NULL", #ptr);                        \
    if (!aligned((ptr), (align)))                                                            \
      return fail(GDN_ERR_MISALIGNED, "%s is not %d-byte aligned", #ptr, int(align));        \
  } while (0)

int cuda_fail(cudaError_t e, const char *what) {
  return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static_assert(sizeof(CUtensorMap) == sizeof(TmaDesc), "TmaDesc holds one CUtensorMap");

// cuTensorMapEncodeTiled, looked up once through the runtime (thread-safe
// static initialisation); nullptr if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// The tensor map of one layer's state for the d = 128 tensor-core verify:
// fp32 [rows][128] (rows = B * H_v * d_v), boxes of 128 rows x 32 columns,
// 128-byte swizzle (the layout the kind::tf32 products read).
int encode_state_map(TmaDesc &m, const float *state, long long rows) {
  if (rows > (1LL << 31) - 1)
    return fail(GDN_ERR_UNSUPPORTED, "B * H_v * d_v = %lld state rows exceed the 2^31 - 1 a tensor map addresses", rows);
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return fail(GDN_ERR_CUDA, "the driver provides no cuTensorMapEncodeTiled");
  CUtensorMap map;
  const cuuint64_t dim[2] = {128, cuuint64_t(rows)};
  const cuuint64_t stride[1] = {128 * sizeof(float)};
  const cuuint32_t box[2] = {32, 128};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(state), dim, stride, box,
                         estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled of the state failed (CUresult %d)", int(r));
  std::memcpy(&m, &map, sizeof map);
  return GDN_OK;
}

}  // namespace

extern "C" {

__attribute__((visibility("default"))) const char *gdn_version(void) {
  return "gdn_gb300 1.0 (sm_103a)";
}

__attribute__((visibility("default"))) const char *gdn_last_error(void) { return t_err.c_str(); }

__attribute__((visibility("default"))) size_t gdn_layer_workspace_bytes(const gdn_dims *dims, int mode) {
  if (check_dims(dims) != GDN_OK || check_mode(mode) != GDN_OK) return 0;
  return layer_ws_bytes(dims, mode);
}

namespace {

int verify_impl(const gdn_dims *dims, int mode, const gdn_bf16 *x, const gdn_bf16 *conv_w, const float *g,
                const float *beta, const float *state, gdn_bf16 *ring, const int32_t *offsets,
                const uint8_t *active, const gdn_bf16 *gate_z, const gdn_bf16 *norm_w, float eps, gdn_bf16 *out,
                void *layer_ws, size_t layer_ws_bytes_given, void *stream, uint32_t test_extra_tx = 0,
                uint32_t wait_limit = kWaitLimit) {
  NvtxRange range(gate_z ? "gdn_conv_verify_gated" : "gdn_conv_verify");
  int rc = check_dims(dims);
  if (rc) return rc;
  if (mode & ~(GDN_VERIFY_OVERLAP | GDN_VERIFY_OVERLAP_STATE | 0xff))
    return fail(GDN_ERR_INVALID_ARG, "unknown flag bits in mode 0x%x", mode);
  if ((mode & GDN_VERIFY_OVERLAP) && (mode & GDN_VERIFY_OVERLAP_STATE))
    return fail(GDN_ERR_INVALID_ARG, "GDN_VERIFY_OVERLAP and GDN_VERIFY_OVERLAP_STATE exclude each other");
  int overlap = (mode & GDN_VERIFY_OVERLAP) ? 1 : (mode & GDN_VERIFY_OVERLAP_STATE) ? 2 : 0;
  mode &= 0xff;
  // the state-only level exists in the d = 128 tensor-core verify; elsewhere
  // it is the same as no flag
  if (overlap == 2 && (dims->d_k != 128 || mode == GDN_COMMIT_SNAPSHOT)) overlap = 0;
  if ((rc = check_mode(mode))) return rc;
  if (dims->B == 0) return ok();
  GDN_NEED_PTR(x, 16);
  GDN_NEED_PTR(conv_w, 16);
  GDN_NEED_PTR(g, 16);
  GDN_NEED_PTR(beta, 16);
  GDN_NEED_PTR(state, 16);
  GDN_NEED_PTR(ring, 16);
  GDN_NEED_PTR(active, 1);
  GDN_NEED_PTR(out, 16);
  GDN_NEED_PTR(layer_ws, 256);
  (void)offsets;  // the committed window lives at fixed ring slots
  const size_t need = layer_ws_bytes(dims, mode);
  if (layer_ws_bytes_given < need)
    return fail(GDN_ERR_WORKSPACE, "layer workspace has %zu bytes, needs %zu", layer_ws_bytes_given, need);

  VerifyParams p{};
  p.x = x;
  p.w = conv_w;
  p.g = g;
  p.beta = beta;
  p.state = state;
  p.ring = ring;
  p.active = active;
  p.out = out;
  p.B = dims->B;
  p.T = dims->T;
  p.H_k = dims->H_k;
  p.H_v = dims->H_v;
  p.C = (2 * dims->H_k + dims->H_v) * dims->d_k;
  p.R = kHist + dims->T_max;
  p.act = dims->act;
  p.overlap = overlap;
  p.gz = gate_z;
  p.gw = norm_w;
  p.geps = eps;
  p.status = status_word_address();
  if (!p.status) return fail(GDN_ERR_CUDA, "cannot resolve the device status word");
  p.wait_limit = wait_limit;
  p.test_extra_tx = test_extra_tx;
  if (dims->d_k == 128 && mode != GDN_COMMIT_SNAPSHOT &&
      (rc = encode_state_map(p.tmap_state, state, (long long)dims->B * dims->H_v * 128)))
    return rc;
  char *ws = static_cast<char *>(layer_ws);
  if (mode == GDN_COMMIT_RECOMPUTE) {
    const RecomputeWs w = recompute_ws(dims->B, dims->T, dims->H_k, dims->H_v, dims->d_k);
    p.ws_e = reinterpret_cast<float *>(ws + w.e);
    p.ws_k = reinterpret_cast<float *>(ws + w.k);
    p.ws_G = reinterpret_cast<float *>(ws + w.G);
  } else if (mode == GDN_COMMIT_SNAPSHOT) {
    p.ws_snap = reinterpret_cast<float *>(ws);
  } else {
    const DeferredWs w = deferred_ws(dims->B, dims->T, dims->H_k, dims->H_v, dims->d_k);
    const RecomputeWs r = recompute_ws(dims->B, dims->T, dims->H_v, dims->H_v, dims->d_k);
    p.ws_pend = reinterpret_cast<int *>(ws + w.pend);
    p.ws_e = reinterpret_cast<float *>(ws + w.cap + r.e);
    p.ws_k = reinterpret_cast<float *>(ws + w.cap + r.k);
    p.ws_G = reinterpret_cast<float *>(ws + w.cap + r.G);
    p.state_w = const_cast<float *>(state);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (dims->d_k) {
    case 32: e = launch_verify_32(p, dims->T, mode, s); break;
    case 64: e = launch_verify_64(p, dims->T, mode, s); break;
    default: e = launch_verify_128(p, dims->T, mode, s); break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "gdn_conv_verify launch");
  return ok();
}

}  // namespace

__attribute__((visibility("default"))) int gdn_conv_verify(
    const gdn_dims *dims, int mode, const gdn_bf16 *x, const gdn_bf16 *conv_w, const float *g,
    const float *beta, const float *state, gdn_bf16 *ring, const int32_t *offsets,
    const uint8_t *active, gdn_bf16 *out, void *layer_ws, size_t layer_ws_bytes_given, void *stream) {
  return verify_impl(dims, mode, x, conv_w, g, beta, state, ring, offsets, active, nullptr, nullptr, 0.f, out,
                     layer_ws, layer_ws_bytes_given, stream);
}

__attribute__((visibility("default"))) int gdn_test_verify_timeout(
    const gdn_dims *dims, int mode, const gdn_bf16 *x, const gdn_bf16 *conv_w, const float *g,
    const float *beta, const float *state, gdn_bf16 *ring, const int32_t *offsets,
    const uint8_t *active, gdn_bf16 *out, void *layer_ws, size_t layer_ws_bytes_given, uint32_t wait_limit,
    void *stream) {
  if (check_dims(dims) == GDN_OK && (dims->d_k != 128 || (mode & 0xff) == GDN_COMMIT_SNAPSHOT))
    return fail(GDN_ERR_UNSUPPORTED, "gdn_test_verify_timeout: d = 128, RECOMPUTE or DEFERRED only");
  if (wait_limit < 1) return fail(GDN_ERR_INVALID_ARG, "gdn_test_verify_timeout: wait_limit must be >= 1");
  return verify_impl(dims, mode, x, conv_w, g, beta, state, ring, offsets, active, nullptr, nullptr, 0.f, out,
                     layer_ws, layer_ws_bytes_given, stream, 16u, wait_limit);
}

__attribute__((visibility("default"))) int gdn_conv_verify_gated(
    const gdn_dims *dims, int mode, const gdn_bf16 *x, const gdn_bf16 *conv_w, const float *g,
    const float *beta, const float *state, gdn_bf16 *ring, const int32_t *offsets,
    const uint8_t *active, const gdn_bf16 *gate_z, const gdn_bf16 *norm_w, float eps, gdn_bf16 *out,
    void *layer_ws, size_t layer_ws_bytes_given, void *stream) {
  if (check_dims(dims) == GDN_OK && dims->B > 0) {
    GDN_NEED_PTR(gate_z, 16);
    GDN_NEED_PTR(norm_w, 16);
    if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(GDN_ERR_INVALID_ARG, "eps must be finite and >= 0");
  }
  return verify_impl(dims, mode, x, conv_w, g, beta, state, ring, offsets, active, gate_z, norm_w, eps, out,
                     layer_ws, layer_ws_bytes_given, stream);
}

__attribute__((visibility("default"))) int gdn_commit(const gdn_dims *dims, int mode, int n_layers,
                                                      float *const *state, gdn_bf16 *const *ring,
                                                      void *const *layer_ws, const int32_t *keep,
                                                      const uint8_t *active, int32_t *offsets, void *stream) {
  NvtxRange range("gdn_commit");
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_mode(mode))) return rc;
  if (!ring) return fail(GDN_ERR_INVALID_ARG, "ring host array is NULL");
  CommitParams p{};
  if ((rc = fill_layers(p, n_layers, state, ring, layer_ws))) return rc;
  if (dims->B == 0) return ok();
  GDN_NEED_PTR(keep, 4);
  GDN_NEED_PTR(active, 1);
  GDN_NEED_PTR(offsets, 4);
  p.keep = keep;
  p.active = active;
  p.offsets = offsets;
  p.B = dims->B;
  p.T = dims->T;
  p.H_k = dims->H_k;
  p.H_v = dims->H_v;
  p.C = (2 * dims->H_k + dims->H_v) * dims->d_k;
  p.R = kHist + dims->T_max;
  p.status = status_word_address();
  if (!p.status) return fail(GDN_ERR_CUDA, "cannot resolve the device status word");
  cudaError_t e = launch_commit(p, dims->d_k, mode, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gdn_commit launch");
  return ok();
}

__attribute__((visibility("default"))) int gdn_flush(const gdn_dims *dims, int mode, int n_layers,
                                                     float *const *state, void *const *layer_ws, void *stream) {
  NvtxRange range("gdn_flush");
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_mode(mode))) return rc;
  CommitParams p{};
  if ((rc = fill_layers(p, n_layers, state, nullptr, layer_ws))) return rc;
  if (dims->B == 0 || mode != GDN_COMMIT_DEFERRED) return ok();
  p.B = dims->B;
  p.T = dims->T;
  p.H_k = dims->H_k;
  p.H_v = dims->H_v;
  cudaError_t e = launch_flush(p, dims->d_k, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gdn_flush launch");
  return ok();
}

__attribute__((visibility("default"))) size_t gdn_prefill_workspace_bytes(const gdn_dims *dims, int L) {
  if (check_dims(dims) != GDN_OK || L < 1 || L > kMaxPrefillLen) return 0;
  return prefill_workspace_bytes(dims->B, L, dims->H_k, dims->H_v, dims->d_k);
}

__attribute__((visibility("default"))) int gdn_prefill_chunked(
    const gdn_dims *dims, int L, const gdn_bf16 *x, const gdn_bf16 *conv_w, const float *g,
    const float *beta, float *state, gdn_bf16 *ring, int32_t *offsets, gdn_bf16 *out, void *ws,
    size_t ws_bytes, void *stream) {
  NvtxRange range("gdn_prefill_chunked");
  int rc = check_dims(dims);
  if (rc) return rc;
  if (L < 0 || L > kMaxPrefillLen)
    return fail(GDN_ERR_UNSUPPORTED, "prompt length L=%d outside [0, %d]", L, kMaxPrefillLen);
  if (dims->B == 0 || L == 0) return ok();
  GDN_NEED_PTR(x, 16);
  GDN_NEED_PTR(conv_w, 16);
  GDN_NEED_PTR(g, 16);
  GDN_NEED_PTR(beta, 16);
  GDN_NEED_PTR(state, 16);
  GDN_NEED_PTR(ring, 16);
  GDN_NEED_PTR(offsets, 4);
  GDN_NEED_PTR(out, 16);
  GDN_NEED_PTR(ws, 256);
  const size_t need = prefill_workspace_bytes(dims->B, L, dims->H_k, dims->H_v, dims->d_k);
  if (ws_bytes < need) return fail(GDN_ERR_WORKSPACE, "prefill workspace has %zu bytes, needs %zu", ws_bytes, need);
  cudaError_t e = launch_prefill(x, conv_w, g, beta, state, ring, offsets, out, ws, dims->B, L, dims->H_k,
                                 dims->H_v, dims->d_k, kHist + dims->T_max, dims->act,
                                 static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gdn_prefill_chunked launch");
  return ok();
}

__attribute__((visibility("default"))) int gdn_get_status(int clear, uint32_t *status) {
  if (!status) return fail(GDN_ERR_INVALID_ARG, "status is NULL");
  uint32_t *dev = status_word_address();
  if (!dev) return fail(GDN_ERR_CUDA, "cannot resolve the device status word");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "gdn_get_status synchronize");
  e = cudaMemcpy(status, dev, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "gdn_get_status read");
  if (clear) {
    e = cudaMemset(dev, 0, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "gdn_get_status clear");
  }
  return ok();
}

__attribute__((visibility("default"))) size_t gdn_accept_workspace_bytes(int B, int T, int V) {
  if (B < 0 || T < 1 || T > kMaxAcceptT || V < 1) return 0;
  return accept_workspace_bytes(B, T, V);
}

__attribute__((visibility("default"))) int gdn_accept_greedy(int B, int T, int V, const gdn_bf16 *logits,
                                                             const int32_t *draft, const uint8_t *active,
                                                             int32_t *keep, int32_t *next, void *ws,
                                                             size_t ws_bytes, void *stream) {
  NvtxRange range("gdn_accept_greedy");
  if (B < 0 || T < 1 || V < 1) return fail(GDN_ERR_INVALID_ARG, "accept: B=%d T=%d V=%d", B, T, V);
  if (T > kMaxAcceptT) return fail(GDN_ERR_UNSUPPORTED, "accept: T=%d above %d", T, kMaxAcceptT);
  if ((long long)B * T > 65535) return fail(GDN_ERR_UNSUPPORTED, "accept: B*T=%lld above 65535", (long long)B * T);
  if (B == 0) return ok();
  GDN_NEED_PTR(logits, 16);
  GDN_NEED_PTR(draft, 16);
  GDN_NEED_PTR(active, 16);
  GDN_NEED_PTR(keep, 16);
  GDN_NEED_PTR(next, 16);
  GDN_NEED_PTR(ws, 256);
  const size_t need = accept_workspace_bytes(B, T, V);
  if (ws_bytes < need) return fail(GDN_ERR_WORKSPACE, "accept workspace has %zu bytes, needs %zu", ws_bytes, need);
  cudaError_t e = launch_accept(logits, draft, active, keep, next, ws, B, T, V, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gdn_accept_greedy launch");
  return ok();
}

__attribute__((visibility("default"))) int gdn_move_rows(
    const gdn_dims *src_dims, const gdn_dims *dst_dims, int mode, int n_layers, const float *const *src_state,
    const gdn_bf16 *const *src_ring, const int32_t *src_offsets, float *const *dst_state, gdn_bf16 *const *dst_ring,
    int32_t *dst_offsets, void *const *dst_layer_ws, const int32_t *src_rows, const int32_t *dst_rows, int n_rows,
    void *stream) {
  NvtxRange range("gdn_move_rows");
  int rc = check_dims(src_dims);
  if (rc) return rc;
  if ((rc = check_dims(dst_dims))) return rc;
  if ((rc = check_mode(mode))) return rc;
  if (src_dims->H_k != dst_dims->H_k || src_dims->H_v != dst_dims->H_v || src_dims->d_k != dst_dims->d_k ||
      src_dims->T_max != dst_dims->T_max || src_dims->width != dst_dims->width)
    return fail(GDN_ERR_INVALID_ARG, "move_rows: the cohorts differ in heads, head size or T_max");
  if (n_layers < 1 || n_layers > kMaxLayers)
    return fail(GDN_ERR_INVALID_ARG, "n_layers=%d outside [1, %d]", n_layers, kMaxLayers);
  if (n_rows < 0) return fail(GDN_ERR_INVALID_ARG, "n_rows=%d", n_rows);
  if (!src_state || !src_ring || !dst_state || !dst_ring) return fail(GDN_ERR_INVALID_ARG, "NULL layer array");
  if (mode == GDN_COMMIT_DEFERRED && !dst_layer_ws)
    return fail(GDN_ERR_INVALID_ARG, "DEFERRED: the destination layer workspaces are needed");
  if (n_rows == 0) return ok();
  GDN_NEED_PTR(src_offsets, 16);
  GDN_NEED_PTR(dst_offsets, 16);
  GDN_NEED_PTR(src_rows, 16);
  GDN_NEED_PTR(dst_rows, 16);
  MoveParams p{};
  for (int l = 0; l < n_layers; ++l) {
    if (!src_state[l] || !src_ring[l] || !dst_state[l] || !dst_ring[l])
      return fail(GDN_ERR_INVALID_ARG, "layer %d: NULL state or ring", l);
    if (!aligned(src_state[l], 16) || !aligned(src_ring[l], 16) || !aligned(dst_state[l], 16) ||
        !aligned(dst_ring[l], 16))
      return fail(GDN_ERR_MISALIGNED, "layer %d: state or ring not 16-byte aligned", l);
    p.src_state[l] = src_state[l];
    p.src_ring[l] = reinterpret_cast<const uint16_t *>(src_ring[l]);
    p.dst_state[l] = dst_state[l];
    p.dst_ring[l] = reinterpret_cast<uint16_t *>(dst_ring[l]);
    if (mode == GDN_COMMIT_DEFERRED) {
      if (!dst_layer_ws[l] || !aligned(dst_layer_ws[l], 256))
        return fail(GDN_ERR_MISALIGNED, "layer %d: NULL or misaligned destination workspace", l);
      p.dst_ws[l] = dst_layer_ws[l];
    }
  }
  const int C = (2 * src_dims->H_k + src_dims->H_v) * src_dims->d_k;
  p.src_offsets = src_offsets;
  p.dst_offsets = dst_offsets;
  p.src_rows = src_rows;
  p.dst_rows = dst_rows;
  p.state_bytes = size_t(src_dims->H_v) * src_dims->d_v * src_dims->d_k * sizeof(float);
  p.ring_bytes = size_t(kHist + src_dims->T_max) * C * sizeof(uint16_t);
  p.pend_bytes = mode == GDN_COMMIT_DEFERRED ? size_t(dst_dims->H_v) * sizeof(int) : 0;
  p.n_layers = n_layers;
  p.n_rows = n_rows;
  p.src_B = src_dims->B;
  p.dst_B = dst_dims->B;
  p.H_v = dst_dims->H_v;
  p.status = status_word_address();
  if (!p.status) return fail(GDN_ERR_CUDA, "cannot resolve the device status word");
  cudaError_t e = launch_move_rows(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gdn_move_rows launch");
  return ok();
}

// ---- verify without caller-provided workspace ---------------------------------
// Scratch for gdn_conv_verify_noalloc: one layer's verify captures.  It lives
// in the library's own device memory, so every GPU that loads the library
// holds these bytes until the process exits.  Host code may not use the name
// `g_noalloc_ws` as an address (on the host it is only a stand-in for the
// device symbol); the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_ws[GDN_NOALLOC_WS_BYTES];

namespace {

std::mutex g_noalloc_lock;
void *g_noalloc_ptr[64] = {nullptr};  // device address of g_noalloc_ws, per device

// Look up (once per device, with that device current) where the scratch
// array lives on the current device.
int noalloc_scratch(void **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "gdn_conv_verify_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(GDN_ERR_UNSUPPORTED, "device index %d above 63", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_lock);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_ws);
    if (e != cudaSuccess || !p) return cuda_fail(e, "gdn_conv_verify_noalloc: cudaGetSymbolAddress");
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return GDN_OK;
}

}  // namespace

__attribute__((visibility("default"))) int gdn_conv_verify_noalloc(
    const gdn_dims *dims, int mode, const gdn_bf16 *x, const gdn_bf16 *conv_w, const float *g,
    const float *beta, const float *state, gdn_bf16 *ring, const int32_t *offsets,
    const uint8_t *active, gdn_bf16 *out, void **layer_ws_used, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_mode(mode & 0xff))) return rc;
  if ((mode & 0xff) == GDN_COMMIT_DEFERRED)
    return fail(GDN_ERR_INVALID_ARG,
                "gdn_conv_verify_noalloc: DEFERRED mode needs a workspace that persists per layer");
  const size_t need = layer_ws_bytes(dims, mode & 0xff);
  if (need > GDN_NOALLOC_WS_BYTES)
    return fail(GDN_ERR_WORKSPACE,
                "gdn_conv_verify_noalloc: this shape and mode need %zu bytes of scratch, the library's "
                "built-in scratch holds %zu; use gdn_conv_verify with a caller-allocated workspace",
                need, size_t(GDN_NOALLOC_WS_BYTES));
  void *ws = nullptr;
  if ((rc = noalloc_scratch(&ws))) return rc;
  rc = gdn_conv_verify(dims, mode, x, conv_w, g, beta, state, ring, offsets, active, out, ws,
                       GDN_NOALLOC_WS_BYTES, stream);
  if (rc == GDN_OK && layer_ws_used) *layer_ws_used = ws;
  return rc;
}

}  // extern "C"
