// gdn_common.cuh -- shared device helpers and kernel parameter blocks for the
// GB300 GDN speculative-transaction library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kWidth = 4;        // conv width
constexpr int kHist = kWidth - 1; // inputs in the committed conv window
constexpr int kMaxT = 8;         // positions per verify
constexpr int kTileRows = 32;    // state rows (d_v) per verify CTA
constexpr int kVerifyThreads = 128;
constexpr float kNormEps = 1e-6f;

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ int ring_slot(int pos, int R) {
  int s = pos % R;
  return s < 0 ? s + R : s;
}

// SiLU with the fast exponential and division intrinsics (a few ulp; the
// conv output feeds an fp32 recurrence whose tolerance is far looser).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Streaming 128-bit load that does not allocate in L1 (each state byte is
// read once per call).
__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_f4(float *p, float4 v) {
  *reinterpret_cast<float4 *>(p) = v;
}

// ---- shared-memory barrier + bulk-copy (TMA) helpers ------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make an initialised mbarrier visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Contiguous global -> shared copy on the bulk-copy engine; completion is
// counted on `bar` in bytes.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` with an iteration limit (about a second in
// total); false if the limit ran out.
constexpr uint32_t kWaitLimit = 1u << 22;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i >= 32) __nanosleep(256);
  }
  return false;
}

// ---- programmatic dependent launch --------------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialization.  It waits for the preceding kernel on the stream
// (griddepcontrol.wait) before touching anything that kernel may write, and
// only then lets the next kernel start (launch_dependents), so a kernel's
// pre-wait section can overlap only its immediate predecessor.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename Kernel, typename Params>
inline cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, cudaStream_t stream, const Params &p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, a.x * b.x)));
}

// Lane geometry of a warp that owns 8 consecutive state rows of head size D:
// LPR lanes share one row (4 floats each), GPW row groups per warp, RPL rows
// per lane.  Lane l holds elements [4*(l % LPR), +4) of rows grp + GPW*i.
template <int D>
struct RowLanes {
  static constexpr int LPR = D / 4;
  static constexpr int GPW = 32 / LPR;
  static constexpr int RPL = 8 / GPW;
  static constexpr int LOG2_RPL = RPL == 8 ? 3 : RPL == 4 ? 2 : RPL == 2 ? 1 : 0;
  static_assert(LPR * GPW == 32 && RPL * GPW == 8, "D must be 32, 64 or 128");
};

// Sum each of the RPL per-lane partials over the LPR lanes sharing a row with
// a reduce-scatter butterfly: after the call the lane holds the full sum of
// row index row_of_lane(lane) (one of its RPL rows), using RPL-1 + log2(LPR/RPL)
// shuffles instead of RPL*log2(LPR).
template <int D>
__device__ __forceinline__ float reduce_rows(float (&a)[RowLanes<D>::RPL], int lane) {
  using G = RowLanes<D>;
#pragma unroll
  for (int step = 0; step < G::LOG2_RPL; ++step) {
    const int m = G::LPR >> (step + 1);
    const bool upper = (lane & m) != 0;
    const int half = G::RPL >> (step + 1);
#pragma unroll
    for (int i = 0; i < G::RPL / 2; ++i) {
      if (i < half) {
        const float send = upper ? a[i] : a[i + half];
        const float keep = upper ? a[i + half] : a[i];
        a[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
      }
    }
  }
  float v = a[0];
#pragma unroll
  for (int m = G::LPR >> (G::LOG2_RPL + 1); m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Which of the lane's RPL rows reduce_rows left in this lane.
template <int D>
__device__ __forceinline__ int row_of_lane(int lane) {
  using G = RowLanes<D>;
  int i = 0;
#pragma unroll
  for (int step = 0; step < G::LOG2_RPL; ++step)
    if (lane & (G::LPR >> (step + 1))) i += G::RPL >> (step + 1);
  return i;
}

// Lane offset (within its LPR-lane row group) that holds row index i after
// reduce_rows: the inverse of row_of_lane.
template <int D>
__device__ __forceinline__ int lane_of_row(int i) {
  using G = RowLanes<D>;
  int off = 0;
#pragma unroll
  for (int step = 0; step < G::LOG2_RPL; ++step)
    if ((i >> (G::LOG2_RPL - 1 - step)) & 1) off += G::LPR >> (step + 1);
  return off;
}

// Per-layer verify parameters.
struct VerifyParams {
  const uint16_t *x;
  const uint16_t *w;
  const float *g;
  const float *beta;
  const float *state;
  uint16_t *ring;
  const int32_t *offsets;
  const uint8_t *active;
  uint16_t *out;
  float *ws_e;    // RECOMPUTE: [B][T][H_v][D]
  float *ws_k;    // RECOMPUTE: [B][T][H_k][D]
  float *ws_G;    // RECOMPUTE: [B][T][H_v]
  float *ws_snap; // SNAPSHOT:  [T][B][H_v][D][D]
  uint32_t *status; // sticky device status word
  int B, H_k, H_v, C, R, act;
  int overlap;      // GDN_VERIFY_OVERLAP: stage the state tile before the PDL wait
};

constexpr int kMaxLayers = GDN_MAX_LAYERS;

struct CommitParams {
  float *state[kMaxLayers];
  const float *ws[kMaxLayers];
  const int32_t *keep;
  const uint8_t *active;
  int32_t *offsets;
  int n_layers, B, T, H_k, H_v;
};

// Byte offsets of the RECOMPUTE workspace regions (each 256-byte aligned).
struct RecomputeWs {
  size_t e, k, G, total;
};

__host__ __device__ inline size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

__host__ __device__ inline RecomputeWs recompute_ws(int B, int T, int H_k, int H_v, int D) {
  RecomputeWs w;
  w.e = 0;
  w.k = w.e + align256(sizeof(float) * size_t(B) * T * H_v * D);
  w.G = w.k + align256(sizeof(float) * size_t(B) * T * H_k * D);
  w.total = w.G + align256(sizeof(float) * size_t(B) * T * H_v);
  return w;
}

__host__ __device__ inline size_t snapshot_ws(int B, int T, int H_v, int D) {
  return sizeof(float) * size_t(T) * B * H_v * D * D;
}

// launchers (defined in the .cu files)
cudaError_t launch_verify_32(const VerifyParams &p, int T, int mode, cudaStream_t s);
cudaError_t launch_verify_64(const VerifyParams &p, int T, int mode, cudaStream_t s);
cudaError_t launch_verify_128(const VerifyParams &p, int T, int mode, cudaStream_t s);
cudaError_t launch_commit(const CommitParams &p, int D, int mode, cudaStream_t s);
size_t prefill_workspace_bytes(int B, int L, int H_k, int H_v, int D);
cudaError_t launch_prefill(const uint16_t *x, const uint16_t *w, const float *g, const float *beta, float *state,
                           uint16_t *ring, int32_t *offsets, uint16_t *out, void *ws, int B, int L, int H_k,
                           int H_v, int D, int R, int act, cudaStream_t stream);
uint32_t *status_word_address();  // device address of the sticky status word

}  // namespace gdn
