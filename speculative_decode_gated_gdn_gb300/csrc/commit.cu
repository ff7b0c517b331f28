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
// S_keep once (RECOMPUTE) or copies the verify-time snapshot (SNAPSHOT); in
// DEFERRED mode the commit only records keep' per layer, and the next verify
// of each (row, head) applies it.  Every mode also shifts the conv window of
// committed rows (the conv-cache mutation).
#include <atomic>

#include "gdn_common.cuh"

namespace gdn {

__device__ uint32_t g_status;  // sticky GDN_STATUS_* bits of this device

// Device address of g_status on the current device, looked up once per device
// (the launchers pass it to kernels in other translation units).
uint32_t *status_word_address() {
  static std::atomic<void *> cached[64];  // per device; host threads may race to fill it (same value)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < 64) {
    if (void *c = cached[dev].load(std::memory_order_acquire)) return static_cast<uint32_t *>(c);
  }
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < 64) cached[dev].store(ptr, std::memory_order_release);
  return static_cast<uint32_t *>(ptr);
}

__device__ __forceinline__ int effective_keep(const CommitParams &p, int b) {
  const int k = p.keep[b];
  if (!p.active[b]) return 0;
  return (k >= 0 && k <= p.T) ? k : 0;
}

// S_keep of 8 state rows (this warp's), in place on the lane's float4
// segments: S <- gamma_{K-1} S + sum_{t<K} exp(G_{K-1} - G_t) e_t k_t^T with the
// captures e [B][H_v][T][D], k [B][KH][T][D], G [B][H_v][kMaxT] of one verify;
// kh is the head's index among the KH copies of k.  Every capture load of the
// first kPre positions is issued before any arithmetic, so they are in flight
// together with the caller's state loads.
template <int D>
__device__ __forceinline__ void rebuild_rows(float4 (&s)[RowLanes<D>::RPL], const float *we, const float *wk,
                                             const float *wG, int b, int h, int kh, int KH, int row0, int K, int T,
                                             int H_v, int sub, int grp) {
  using G = RowLanes<D>;
  constexpr int kPre = 4;
  const size_t bh = size_t(b) * H_v + h, bk = size_t(b) * KH + kh;
  const float4 g0 = *reinterpret_cast<const float4 *>(wG + bh * kMaxT);
  const float4 g1 = *reinterpret_cast<const float4 *>(wG + bh * kMaxT + 4);
  float4 kv[kPre];
  float ev[kPre][G::RPL];
#pragma unroll
  for (int t = 0; t < kPre; ++t) {
    if (t < K) {
      kv[t] = *reinterpret_cast<const float4 *>(wk + (bk * T + t) * D + 4 * sub);
      const float *ert = we + (bh * T + t) * D + row0;
#pragma unroll
      for (int i = 0; i < G::RPL; ++i) ev[t][i] = ert[grp + G::GPW * i];
    }
  }
  const float gv[kMaxT] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  float GK = gv[0];
#pragma unroll
  for (int t = 1; t < kMaxT; ++t)
    if (t == K - 1) GK = gv[t];
  const float gam = expf(GK);
#pragma unroll
  for (int i = 0; i < G::RPL; ++i) s[i] = make_float4(gam * s[i].x, gam * s[i].y, gam * s[i].z, gam * s[i].w);
#pragma unroll
  for (int t = 0; t < kMaxT; ++t) {
    if (t < K) {
      const float c = expf(GK - gv[t]);
      float4 k4;
      float e8[G::RPL];
      if (t < kPre) {
        k4 = kv[t];
#pragma unroll
        for (int i = 0; i < G::RPL; ++i) e8[i] = ev[t][i];
      } else {
        k4 = *reinterpret_cast<const float4 *>(wk + (bk * T + t) * D + 4 * sub);
        const float *ert = we + (bh * T + t) * D + row0;
#pragma unroll
        for (int i = 0; i < G::RPL; ++i) e8[i] = ert[grp + G::GPW * i];
      }
#pragma unroll
      for (int i = 0; i < G::RPL; ++i) {
        const float f = c * e8[i];
        s[i].x = fmaf(f, k4.x, s[i].x);
        s[i].y = fmaf(f, k4.y, s[i].y);
        s[i].z = fmaf(f, k4.z, s[i].z);
        s[i].w = fmaf(f, k4.w, s[i].w);
      }
    }
  }
}

// Conv-cache mutation of the commit: for rows with keep' = K >= 1 the new
// committed window is ring slots K..K+2 (the last three raw inputs of
// window ++ x_0..x_{K-1}); it is written to slots 0..2.  Each thread moves 8
// channels; units are (layer, row, 1024-channel block) after `first_unit`.
__device__ __forceinline__ void shift_windows(const CommitParams &p, long long first_unit) {
  const int C8 = p.C / 8;
  const int blocks_per_row = (C8 + blockDim.x - 1) / blockDim.x;
  const long long units = (long long)p.n_layers * p.B * blocks_per_row;
  for (long long u = (long long)blockIdx.x - first_unit; u < units; u += gridDim.x) {
    if (u < 0) continue;
    const int layer = int(u / ((long long)p.B * blocks_per_row));
    const int r = int(u % ((long long)p.B * blocks_per_row));
    const int b = r / blocks_per_row, blk = r % blocks_per_row;
    const int K = effective_keep(p, b);
    const int c8 = blk * blockDim.x + threadIdx.x;
    if (K == 0 || c8 >= C8) continue;
    uint4 *ring = reinterpret_cast<uint4 *>(p.ring[layer] + size_t(b) * p.R * p.C) + c8;
    uint4 w[kHist];
#pragma unroll
    for (int i = 0; i < kHist; ++i) w[i] = ring[size_t(K + i) * C8];
#pragma unroll
    for (int i = 0; i < kHist; ++i) ring[size_t(kWinSlot + i) * C8] = w[i];
  }
}

template <int D, int MODE>
__global__ void __launch_bounds__(128) commit_kernel(const CommitParams p) {
  using G = RowLanes<D>;
  constexpr int RPL = G::RPL, GPW = G::GPW, LPR = G::LPR;
  constexpr int TILES = D / kTileRows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  pdl_wait();  // every state, ring, workspace and offsets access follows the preceding kernel
  pdl_trigger();

  if (blockIdx.x == 0) {
    for (int b = tid; b < p.B; b += blockDim.x) {
      const int k = p.keep[b];
      int kp = 0;
      if (p.active[b]) {
        if (k >= 0 && k <= p.T) kp = k;
        else atomicOr(p.status, GDN_STATUS_BAD_KEEP);
      }
      p.offsets[b] += kp;
    }
  }
  if (MODE == GDN_COMMIT_DEFERRED) {
    // record keep' for every (layer, row, head); the next verify of each
    // (or a flush) applies it and resets it to 0
    const DeferredWs dl = deferred_ws(p.B, p.T, p.H_k, p.H_v, D);
    const long long n = (long long)p.n_layers * p.B * p.H_v;
    for (long long i = (long long)blockIdx.x * blockDim.x + tid; i < n; i += (long long)gridDim.x * blockDim.x) {
      const int l = int(i / ((long long)p.B * p.H_v));
      const int bh = int(i % ((long long)p.B * p.H_v));
      reinterpret_cast<int *>(reinterpret_cast<char *>(p.ws[l]) + dl.pend)[bh] = effective_keep(p, bh / p.H_v);
    }
  }

  const int H_v = p.H_v, T = p.T;
  const long long per_layer = (long long)p.B * H_v * TILES;
  const long long total = MODE == GDN_COMMIT_DEFERRED ? 0 : per_layer * p.n_layers;
  for (long long u = blockIdx.x; u < total; u += gridDim.x) {
    const int layer = int(u / per_layer);
    long long r = u - layer * per_layer;
    const int b = int(r / (H_v * TILES));
    r -= (long long)b * H_v * TILES;
    const int h = int(r / TILES);
    const int tile = int(r - (long long)h * TILES);
    const int K = effective_keep(p, b);
    if (K == 0) continue;

    const int row0 = tile * kTileRows + warp * 8;
    float *S = p.state[layer] + ((size_t(b) * H_v + h) * D + row0) * D;
    float4 s[RPL];
    if (MODE == GDN_COMMIT_SNAPSHOT) {
      const size_t plane = size_t(p.B) * H_v * D * D;
      const float *src = p.ws[layer] + size_t(K - 1) * plane + ((size_t(b) * H_v + h) * D + row0) * D;
#pragma unroll
      for (int i = 0; i < RPL; ++i) s[i] = ld_stream_f4(src + size_t(grp + GPW * i) * D + 4 * sub);
    } else {
      const RecomputeWs wl = recompute_ws(p.B, T, p.H_k, H_v, D);
      const int rep = H_v / p.H_k;
      const char *base = reinterpret_cast<const char *>(p.ws[layer]);
#pragma unroll
      for (int i = 0; i < RPL; ++i) s[i] = ld_stream_f4(S + size_t(grp + GPW * i) * D + 4 * sub);
      rebuild_rows<D>(s, reinterpret_cast<const float *>(base + wl.e), reinterpret_cast<const float *>(base + wl.k),
                      reinterpret_cast<const float *>(base + wl.G), b, h, h / rep, p.H_k, row0, K, T, H_v, sub,
                      grp);
    }
#pragma unroll
    for (int i = 0; i < RPL; ++i) st_f4(S + size_t(grp + GPW * i) * D + 4 * sub, s[i]);
  }
  shift_windows(p, 0);
}

// Materialise the commits a DEFERRED cycle left pending: one CTA per
// (layer, row, head) unit at a time, so the unit's applied epoch is set by the
// only CTA that handles it.
template <int D>
__global__ void __launch_bounds__(128) flush_kernel(const CommitParams p) {
  using G = RowLanes<D>;
  constexpr int RPL = G::RPL, GPW = G::GPW, LPR = G::LPR;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  pdl_wait();
  pdl_trigger();
  const int H_v = p.H_v, T = p.T;
  const DeferredWs dl = deferred_ws(p.B, T, p.H_k, H_v, D);
  const RecomputeWs rl = recompute_ws(p.B, T, H_v, H_v, D);
  const long long total = (long long)p.n_layers * p.B * H_v;
  for (long long u = blockIdx.x; u < total; u += gridDim.x) {
    const int layer = int(u / ((long long)p.B * H_v));
    const int r = int(u % ((long long)p.B * H_v));
    const int b = r / H_v, h = r % H_v;
    char *ws = reinterpret_cast<char *>(p.ws[layer]);
    int *pend = reinterpret_cast<int *>(ws + dl.pend) + size_t(b) * H_v + h;
    const int K = min(*pend, T);
    if (K >= 1) {
      const char *cap = ws + dl.cap;
      for (int row0 = warp * 8; row0 < D; row0 += 32) {
        float *S = p.state[layer] + ((size_t(b) * H_v + h) * D + row0) * D;
        float4 s[RPL];
#pragma unroll
        for (int i = 0; i < RPL; ++i) s[i] = ld_stream_f4(S + size_t(grp + GPW * i) * D + 4 * sub);
        rebuild_rows<D>(s, reinterpret_cast<const float *>(cap + rl.e), reinterpret_cast<const float *>(cap + rl.k),
                        reinterpret_cast<const float *>(cap + rl.G), b, h, h, H_v, row0, K, T, H_v, sub, grp);
#pragma unroll
        for (int i = 0; i < RPL; ++i) st_f4(S + size_t(grp + GPW * i) * D + 4 * sub, s[i]);
      }
    }
    __syncthreads();  // every CTA thread has read the pending keep before it is reset
    if (K >= 1 && tid == 0) *pend = 0;
  }
}

static int sm_count() {
  static std::atomic<int> cached[64];  // per device, 0 until looked up
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 152;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <int D>
static cudaError_t launch_commit_d(const CommitParams &p, int mode, cudaStream_t stream) {
  long long units = (long long)p.n_layers * p.B * p.H_v * (D / kTileRows);
  long long grid = (long long)sm_count() * 8;
  if (mode == GDN_COMMIT_DEFERRED) {
    // only window shifts: small units, one wave of up to 16 CTAs per SM
    units = (long long)p.n_layers * p.B * ((p.C / 8 + 127) / 128);
    grid = (long long)sm_count() * 16;
  }
  if (units < grid) grid = units;
  if (grid < 1) grid = 1;
  if (mode == GDN_COMMIT_RECOMPUTE)
    return launch_pdl(commit_kernel<D, GDN_COMMIT_RECOMPUTE>, dim3(unsigned(grid)), dim3(128), stream, p);
  if (mode == GDN_COMMIT_SNAPSHOT)
    return launch_pdl(commit_kernel<D, GDN_COMMIT_SNAPSHOT>, dim3(unsigned(grid)), dim3(128), stream, p);
  return launch_pdl(commit_kernel<D, GDN_COMMIT_DEFERRED>, dim3(unsigned(grid)), dim3(128), stream, p);
}

template <int D>
static cudaError_t launch_flush_d(const CommitParams &p, cudaStream_t stream) {
  long long grid = (long long)p.n_layers * p.B * p.H_v;
  if (grid > (long long)sm_count() * 8) grid = (long long)sm_count() * 8;
  if (grid < 1) grid = 1;
  return launch_pdl(flush_kernel<D>, dim3(unsigned(grid)), dim3(128), stream, p);
}

cudaError_t launch_flush(const CommitParams &p, int D, cudaStream_t stream) {
  switch (D) {
    case 32: return launch_flush_d<32>(p, stream);
    case 64: return launch_flush_d<64>(p, stream);
    case 128: return launch_flush_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
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
