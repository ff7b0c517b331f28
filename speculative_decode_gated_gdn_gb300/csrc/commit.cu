// commit.cu -- accepted-prefix commit of the GDN state, grouped over layers.
//
// "Add request-owned eight-way MTP serving for Qwen 35B", section 4: the commit
// handles keep = 0, 1, 2 per row and keep=0 restores the real pre-verification
// state; section 2: inactive rows use keep=0, and committed offsets are kept
// per row.  "MTP inference: review and commit structure", Functional commits
// item 2: accepted-prefix state replay with grouped copies across layers.
//
// One launch covers every layer.  Work units are (layer, row b, head h, tile
// of 32 state rows); a persistent grid strides over them and skips every unit
// whose row has keep' = 0, so restored rows cost no state traffic at all and
// their bytes are never written.  A committed unit reads S_0 once and writes
// S_keep once (RECOMPUTE) or copies the verify-time snapshot (SNAPSHOT).
#include "gdn_common.cuh"

namespace gdn {

__device__ uint32_t g_status;  // sticky GDN_STATUS_* bits of this device

// Device address of g_status on the current device, looked up once per device
// (the launchers pass it to kernels in other translation units).
uint32_t *status_word_address() {
  static void *cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < 64 && cached[dev]) return static_cast<uint32_t *>(cached[dev]);
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < 64) cached[dev] = ptr;
  return static_cast<uint32_t *>(ptr);
}

__device__ __forceinline__ int effective_keep(const CommitParams &p, int b) {
  const int k = p.keep[b];
  if (!p.active[b]) return 0;
  return (k >= 0 && k <= p.T) ? k : 0;
}

template <int D, int MODE>
__global__ void __launch_bounds__(128) commit_kernel(const CommitParams p) {
  using G = RowLanes<D>;
  constexpr int RPL = G::RPL, GPW = G::GPW, LPR = G::LPR;
  constexpr int TILES = D / kTileRows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  pdl_wait();  // every state, workspace and offsets access follows the preceding kernel
  pdl_trigger();

  if (blockIdx.x == 0) {
    for (int b = tid; b < p.B; b += blockDim.x) {
      const int k = p.keep[b];
      int kp = 0;
      if (p.active[b]) {
        if (k >= 0 && k <= p.T) kp = k;
        else atomicOr(&g_status, GDN_STATUS_BAD_KEEP);
      }
      p.offsets[b] += kp;
    }
  }

  const int H_v = p.H_v, T = p.T;
  const int rep = H_v / p.H_k;
  const long long per_layer = (long long)p.B * H_v * TILES;
  const long long total = per_layer * p.n_layers;
  for (long long u = blockIdx.x; u < total; u += gridDim.x) {
    const int layer = int(u / per_layer);
    long long r = u - layer * per_layer;
    const int b = int(r / (H_v * TILES));
    r -= (long long)b * H_v * TILES;
    const int h = int(r / TILES);
    const int tile = int(r - (long long)h * TILES);
    const int K = effective_keep(p, b);
    if (K == 0) continue;

    float *S = p.state[layer] + ((size_t(b) * H_v + h) * D + tile * kTileRows + warp * 8) * D;
    if (MODE == GDN_COMMIT_SNAPSHOT) {
      const size_t plane = size_t(p.B) * H_v * D * D;
      const float *src = p.ws[layer] + size_t(K - 1) * plane +
                         ((size_t(b) * H_v + h) * D + tile * kTileRows + warp * 8) * D;
      float4 v[RPL];
#pragma unroll
      for (int i = 0; i < RPL; ++i) v[i] = ld_stream_f4(src + size_t(grp + GPW * i) * D + 4 * sub);
#pragma unroll
      for (int i = 0; i < RPL; ++i) st_f4(S + size_t(grp + GPW * i) * D + 4 * sub, v[i]);
    } else {
      const RecomputeWs wl = recompute_ws(p.B, T, p.H_k, H_v, D);
      const char *base = reinterpret_cast<const char *>(p.ws[layer]);
      const float *we = reinterpret_cast<const float *>(base + wl.e);
      const float *wk = reinterpret_cast<const float *>(base + wl.k);
      const float *wG = reinterpret_cast<const float *>(base + wl.G);
      const int hk = h / rep;
      float4 s[RPL];
#pragma unroll
      for (int i = 0; i < RPL; ++i) s[i] = ld_stream_f4(S + size_t(grp + GPW * i) * D + 4 * sub);
      const float GK = wG[(size_t(b) * T + (K - 1)) * H_v + h];
      const float gam = expf(GK);
      float4 acc[RPL];
#pragma unroll
      for (int i = 0; i < RPL; ++i)
        acc[i] = make_float4(gam * s[i].x, gam * s[i].y, gam * s[i].z, gam * s[i].w);
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) {
        if (t < K) {
          const float c = expf(GK - wG[(size_t(b) * T + t) * H_v + h]);
          const float4 kv = *reinterpret_cast<const float4 *>(
              wk + ((size_t(b) * T + t) * p.H_k + hk) * D + 4 * sub);
          const float *ert = we + ((size_t(b) * T + t) * H_v + h) * D + tile * kTileRows + warp * 8;
#pragma unroll
          for (int i = 0; i < RPL; ++i) {
            const float f = c * ert[grp + GPW * i];
            acc[i].x = fmaf(f, kv.x, acc[i].x);
            acc[i].y = fmaf(f, kv.y, acc[i].y);
            acc[i].z = fmaf(f, kv.z, acc[i].z);
            acc[i].w = fmaf(f, kv.w, acc[i].w);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < RPL; ++i) st_f4(S + size_t(grp + GPW * i) * D + 4 * sub, acc[i]);
    }
  }
}

static int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 152;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int D>
static cudaError_t launch_commit_d(const CommitParams &p, int mode, cudaStream_t stream) {
  const long long units = (long long)p.n_layers * p.B * p.H_v * (D / kTileRows);
  long long grid = (long long)sm_count() * 8;
  if (units < grid) grid = units;
  if (grid < 1) grid = 1;
  if (mode == GDN_COMMIT_RECOMPUTE)
    return launch_pdl(commit_kernel<D, GDN_COMMIT_RECOMPUTE>, dim3(unsigned(grid)), dim3(128), stream, p);
  return launch_pdl(commit_kernel<D, GDN_COMMIT_SNAPSHOT>, dim3(unsigned(grid)), dim3(128), stream, p);
}

cudaError_t launch_commit(const CommitParams &p, int D, int mode, cudaStream_t stream) {
  switch (D) {
    case 32: return launch_commit_d<32>(p, mode, stream);
    case 64: return launch_commit_d<64>(p, mode, stream);
    case 128: return launch_commit_d<128>(p, mode, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
