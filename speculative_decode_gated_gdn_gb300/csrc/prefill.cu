// prefill.cu -- state priming over a prompt: the chunked (WY / UT-transform)
// form of the gated delta rule.
//
// "MTP inference: review and commit structure", Verification and limits: the
// chunked recurrence used for the prompt differs from the sequential one only
// in its rounding boundaries.  The chunked form is the one of Yang et al.,
// "Parallelizing Linear Transformers with the Delta Rule over Sequence Length"
// (2024) with the gating of "Gated Delta Networks" (2025), restated here for
// the state layout S[d_v][d_k] (v ~ S k).  Within a chunk of n <= 64 tokens,
// with G_t the within-chunk cumulative log-decay and gamma_t = exp(G_t):
//   A[t][s]  = beta_t exp(G_t - G_s) (k_t . k_s)            (s < t)
//   Tm       = (I + A)^-1                                     (UT transform)
//   W        = Tm diag(beta gamma) K,   U = Tm diag(beta) V
//   E        = U - W S^T                                      (needs the state)
//   O        = diag(gamma) Q S^T + Pm E,  Pm[t][s] = exp(G_t - G_s) (q_t . k_s), s <= t
//   S       <- gamma_n S + sum_t exp(G_n - G_t) E[t] K[t]^T
// The first two lines and W, U, Pm depend only on the chunk's inputs and run
// in parallel over chunks; the last three run sequentially over chunks.
//
// Kernels (one stream, in order):
//   prefill_conv_kernel   conv + SiLU + L2 norm of every token  -> Q, K, V (fp32)
//   prefill_chunk_kernel  per (chunk, value head): G, A, Tm, W, U, Pm
//   prefill_state_kernel  per (value head, 32-row d_v slice): the chunk loop
//   prefill_ring_kernel   last three raw inputs into the ring
// The state kernel also advances offsets by L.
#include "gdn_common.cuh"

namespace gdn {

constexpr int kChunk = 64;

struct PrefillParams {
  const uint16_t *x;  // [B][L][C]
  const uint16_t *w;  // [C][4]
  const float *g;     // [B][L][H_v]
  const float *beta;  // [B][L][H_v]
  float *state;       // [B][H_v][D][D]
  uint16_t *ring;     // [B][R][C]
  int32_t *offsets;   // [B]
  uint16_t *out;      // [B][L][H_v][D]
  // workspace
  float *q;   // [B][H_k][L][D]  normalised q / sqrt(D)
  float *k;   // [B][H_k][L][D]  normalised k
  float *v;   // [B][H_v][L][D]
  float *W;   // [B][H_v][L][D]
  float *U;   // [B][H_v][L][D]
  float *Gc;  // [B][H_v][L]     within-chunk cumulative log-decay
  float *Pm;  // [B][H_v][NC][64][64]
  int B, L, NC, H_k, H_v, C, R, act;
};

struct PrefillWs {
  size_t q, k, v, W, U, Gc, Pm, total;
};

inline PrefillWs prefill_ws(int B, int L, int H_k, int H_v, int D) {
  const int NC = (L + kChunk - 1) / kChunk;
  const size_t Lp = size_t(NC) * kChunk;  // padded so every chunk tile is whole
  PrefillWs w;
  size_t o = 0;
  w.q = o, o += align256(sizeof(float) * size_t(B) * H_k * Lp * D);
  w.k = o, o += align256(sizeof(float) * size_t(B) * H_k * Lp * D);
  w.v = o, o += align256(sizeof(float) * size_t(B) * H_v * Lp * D);
  w.W = o, o += align256(sizeof(float) * size_t(B) * H_v * Lp * D);
  w.U = o, o += align256(sizeof(float) * size_t(B) * H_v * Lp * D);
  w.Gc = o, o += align256(sizeof(float) * size_t(B) * H_v * Lp);
  w.Pm = o, o += align256(sizeof(float) * size_t(B) * H_v * NC * kChunk * kChunk);
  w.total = o;
  return w;
}

// ---------------------------------------------------------------------------
// 1. conv + activation + L2 norm.  Block = D threads = the D channels of one
//    head (q, k or v) for one chunk of tokens of one row.  Tokens past L are
//    written as zeros so chunk tiles are whole.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(D) prefill_conv_kernel(const PrefillParams p) {
  const int chunk = blockIdx.x, head = blockIdx.y, b = blockIdx.z;  // head in [0, 2 H_k + H_v)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = D / 32;
  __shared__ float s_part[kChunk][NW];
  __shared__ float s_inv[kChunk];
  pdl_wait();
  pdl_trigger();
  const int H_k = p.H_k, C = p.C, R = p.R, L = p.L;
  const int c = head * D + tid;  // channel (q heads, then k heads, then v heads)
  const int kind = head < H_k ? 0 : head < 2 * H_k ? 1 : 2;
  const uint2 wr = *reinterpret_cast<const uint2 *>(p.w + size_t(c) * kWidth);
  const float w0 = bf2f(uint16_t(wr.x & 0xffff)), w1 = bf2f(uint16_t(wr.x >> 16));
  const float w2 = bf2f(uint16_t(wr.y & 0xffff)), w3 = bf2f(uint16_t(wr.y >> 16));
  const int t0 = chunk * kChunk;
  // the three inputs before t0: from the prompt, or the committed window
  float h0, h1, h2;
  {
    float hv[kHist];
    const int off = p.offsets[b];
#pragma unroll
    for (int i = 0; i < kHist; ++i) {
      const int t = t0 - kHist + i;
      hv[i] = t >= 0 ? bf2f(p.x[(size_t(b) * L + t) * C + c])
                     : bf2f(p.ring[(size_t(b) * R + ring_slot(off + t, R)) * C + c]);
    }
    h0 = hv[0], h1 = hv[1], h2 = hv[2];
  }
  float y[kChunk];
#pragma unroll
  for (int i = 0; i < kChunk; ++i) {
    const int t = t0 + i;
    const float xt = t < L ? bf2f(p.x[(size_t(b) * L + t) * C + c]) : 0.f;
    float acc = w0 * h0;
    acc = fmaf(w1, h1, acc);
    acc = fmaf(w2, h2, acc);
    acc = fmaf(w3, xt, acc);
    y[i] = t < L ? (p.act ? silu_fast(acc) : acc) : 0.f;
    h0 = h1, h1 = h2, h2 = xt;
  }
  const size_t Lp = size_t(p.NC) * kChunk;
  if (kind == 2) {
    float *dst = p.v + ((size_t(b) * p.H_v + (head - 2 * H_k)) * Lp + t0) * D + tid;
#pragma unroll
    for (int i = 0; i < kChunk; ++i) dst[size_t(i) * D] = y[i];
    return;
  }
#pragma unroll
  for (int i = 0; i < kChunk; ++i) {
    float ss = y[i] * y[i];
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    if (lane == 0) s_part[i][warp] = ss;
  }
  __syncthreads();
  for (int i = tid; i < kChunk; i += D) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NW; ++j) ss += s_part[i][j];
    float inv = rsqrtf(ss + kNormEps);
    if (kind == 0) inv *= rsqrtf(float(D));
    s_inv[i] = inv;
  }
  __syncthreads();
  const int hk = kind == 0 ? head : head - H_k;
  float *dst = (kind == 0 ? p.q : p.k) + ((size_t(b) * H_k + hk) * Lp + t0) * D + tid;
#pragma unroll
  for (int i = 0; i < kChunk; ++i) dst[size_t(i) * D] = y[i] * s_inv[i];
}

// ---------------------------------------------------------------------------
// 2. per (chunk, value head): G, A, the UT transform Tm = (I + A)^-1, W, U, Pm.
//    256 threads; K, Q, V tiles of the chunk in shared memory.
// ---------------------------------------------------------------------------
constexpr int kChunkThreads = 256;
constexpr int kPad = kChunk + 1;

template <int D>
struct ChunkSmem {
  float K[kChunk][D];
  float Q[kChunk][D];
  float V[kChunk][D];
  float A[kChunk][kPad];
  float Tm[kChunk][kPad];
  float G[kChunk];
  float bt[kChunk];
};

template <int D>
__global__ void __launch_bounds__(kChunkThreads) prefill_chunk_kernel(const PrefillParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ChunkSmem<D> &sm = *reinterpret_cast<ChunkSmem<D> *>(smem_raw);
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const int H_v = p.H_v, H_k = p.H_k, L = p.L;
  const int hk = h / (H_v / H_k);
  const size_t Lp = size_t(p.NC) * kChunk;
  const int t0 = chunk * kChunk;
  const int n = min(kChunk, L - t0);
  const float *Kg = p.k + ((size_t(b) * H_k + hk) * Lp + t0) * D;
  const float *Qg = p.q + ((size_t(b) * H_k + hk) * Lp + t0) * D;
  const float *Vg = p.v + ((size_t(b) * H_v + h) * Lp + t0) * D;
  for (int i = tid; i < kChunk * D / 4; i += kChunkThreads) {
    reinterpret_cast<float4 *>(&sm.K[0][0])[i] = reinterpret_cast<const float4 *>(Kg)[i];
    reinterpret_cast<float4 *>(&sm.Q[0][0])[i] = reinterpret_cast<const float4 *>(Qg)[i];
    reinterpret_cast<float4 *>(&sm.V[0][0])[i] = reinterpret_cast<const float4 *>(Vg)[i];
  }
  if (tid < 32) {
    // within-chunk cumulative log-decay (two tokens per lane, warp scan)
    float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
    const int ta = 2 * tid, tb = 2 * tid + 1;
    if (ta < n) g0 = p.g[(size_t(b) * L + t0 + ta) * H_v + h], b0 = p.beta[(size_t(b) * L + t0 + ta) * H_v + h];
    if (tb < n) g1 = p.g[(size_t(b) * L + t0 + tb) * H_v + h], b1 = p.beta[(size_t(b) * L + t0 + tb) * H_v + h];
    float pair = g0 + g1;
    float incl = pair;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, m);
      if (tid >= m) incl += o;
    }
    const float excl = incl - pair;
    sm.G[ta] = excl + g0;
    sm.G[tb] = excl + g0 + g1;
    sm.bt[ta] = b0;
    sm.bt[tb] = b1;
  }
  __syncthreads();

  // A (strictly lower, decay- and beta-weighted K K^T) and Pm (lower incl.
  // diagonal, decay-weighted Q K^T).  Each thread: a 4 x 4 block of (t, s).
  float *Pg = p.Pm + ((size_t(b) * H_v + h) * p.NC + chunk) * kChunk * kChunk;
  {
    const int tb = (tid / 16) * 4, sb = (tid % 16) * 4;
    float kk[4][4] = {}, qk[4][4] = {};
    for (int i = 0; i < D; i += 4) {
      float4 kt[4], qt[4], ks[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        kt[a] = *reinterpret_cast<const float4 *>(&sm.K[tb + a][i]);
        qt[a] = *reinterpret_cast<const float4 *>(&sm.Q[tb + a][i]);
        ks[a] = *reinterpret_cast<const float4 *>(&sm.K[sb + a][i]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          kk[a][c] += dot4(kt[a], ks[c]);
          qk[a][c] += dot4(qt[a], ks[c]);
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int t = tb + a, s = sb + c;
        const bool valid = t < n && s < n;
        const float decay = valid && s <= t ? expf(sm.G[t] - sm.G[s]) : 0.f;
        sm.A[t][s] = s < t ? sm.bt[t] * decay * kk[a][c] : 0.f;
        Pg[t * kChunk + s] = s <= t ? decay * qk[a][c] : 0.f;
      }
  }
  __syncthreads();

  // Tm = (I + A)^-1 by forward substitution, one row at a time:
  // Tm[t][s] = [t == s] - sum_{s <= r < t} A[t][r] Tm[r][s].
  for (int t = 0; t < kChunk; ++t) {
    if (tid < kChunk) {
      const int s = tid;
      float acc = s == t ? 1.f : 0.f;
      if (s < t)
        for (int r = s; r < t; ++r) acc = fmaf(-sm.A[t][r], sm.Tm[r][s], acc);
      sm.Tm[t][s] = s <= t ? acc : 0.f;
    }
    __syncthreads();
  }

  // W = Tm diag(beta gamma) K and U = Tm diag(beta) V.  Each thread: 2 rows
  // t and 16 columns.
  {
    float *Wg = p.W + ((size_t(b) * H_v + h) * Lp + t0) * D;
    float *Ug = p.U + ((size_t(b) * H_v + h) * Lp + t0) * D;
    constexpr int CPT = D * kChunk / kChunkThreads;  // outputs per thread per matrix
    const int col0 = (tid % (D / 4)) * 4;
    const int rowg = tid / (D / 4);
    constexpr int ROWS_PER = kChunk / (kChunkThreads / (D / 4));
    static_assert(ROWS_PER * 4 == CPT, "thread tiling");
#pragma unroll
    for (int rr = 0; rr < ROWS_PER; ++rr) {
      const int t = rowg * ROWS_PER + rr;
      float4 aw = make_float4(0.f, 0.f, 0.f, 0.f), au = aw;
      for (int s = 0; s <= t && s < n; ++s) {
        const float tm = sm.Tm[t][s] * sm.bt[s];
        const float tw = tm * expf(sm.G[s]);
        const float4 kv = *reinterpret_cast<const float4 *>(&sm.K[s][col0]);
        const float4 vv = *reinterpret_cast<const float4 *>(&sm.V[s][col0]);
        aw.x = fmaf(tw, kv.x, aw.x), aw.y = fmaf(tw, kv.y, aw.y), aw.z = fmaf(tw, kv.z, aw.z),
        aw.w = fmaf(tw, kv.w, aw.w);
        au.x = fmaf(tm, vv.x, au.x), au.y = fmaf(tm, vv.y, au.y), au.z = fmaf(tm, vv.z, au.z),
        au.w = fmaf(tm, vv.w, au.w);
      }
      if (t >= n) aw = au = make_float4(0.f, 0.f, 0.f, 0.f);
      st_f4(Wg + size_t(t) * D + col0, aw);
      st_f4(Ug + size_t(t) * D + col0, au);
    }
  }
  if (tid < kChunk) p.Gc[(size_t(b) * H_v + h) * Lp + t0 + tid] = tid < n ? sm.G[tid] : 0.f;
}

// ---------------------------------------------------------------------------
// 3. the sequential pass over chunks for one (row, value head, 32-row slice
//    of d_v).  256 threads; the state slice stays in shared memory.
// ---------------------------------------------------------------------------
constexpr int kStateThreads = 256;
constexpr int kSlice = 32;

template <int D>
struct StateSmem {
  float S[kSlice][D + 4];  // padded rows: conflict-free column access
  float W[kChunk][D];
  float Q[kChunk][D];
  float K[kChunk][D];
  float Pm[kChunk][kChunk];
  float U[kChunk][kSlice];
  float E[kChunk][kSlice + 1];
  float G[kChunk];
};

template <int D>
__global__ void __launch_bounds__(kStateThreads) prefill_state_kernel(const PrefillParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  StateSmem<D> &sm = *reinterpret_cast<StateSmem<D> *>(smem_raw);
  const int slice = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_trigger();
  const int H_v = p.H_v, H_k = p.H_k, L = p.L;
  const int hk = h / (H_v / H_k);
  const size_t Lp = size_t(p.NC) * kChunk;
  const int j0 = slice * kSlice;
  float *Sg = p.state + ((size_t(b) * H_v + h) * D + j0) * D;
  for (int i = tid; i < kSlice * D; i += kStateThreads) sm.S[i / D][i % D] = Sg[i];

  for (int chunk = 0; chunk < p.NC; ++chunk) {
    const int t0 = chunk * kChunk;
    const int n = min(kChunk, L - t0);
    __syncthreads();  // previous chunk's state update is done
    {
      const float4 *Wg = reinterpret_cast<const float4 *>(p.W + ((size_t(b) * H_v + h) * Lp + t0) * D);
      const float4 *Qg = reinterpret_cast<const float4 *>(p.q + ((size_t(b) * H_k + hk) * Lp + t0) * D);
      const float4 *Kg = reinterpret_cast<const float4 *>(p.k + ((size_t(b) * H_k + hk) * Lp + t0) * D);
      for (int i = tid; i < kChunk * D / 4; i += kStateThreads) {
        reinterpret_cast<float4 *>(&sm.W[0][0])[i] = Wg[i];
        reinterpret_cast<float4 *>(&sm.Q[0][0])[i] = Qg[i];
        reinterpret_cast<float4 *>(&sm.K[0][0])[i] = Kg[i];
      }
      const float4 *Pg = reinterpret_cast<const float4 *>(
          p.Pm + ((size_t(b) * H_v + h) * p.NC + chunk) * kChunk * kChunk);
      for (int i = tid; i < kChunk * kChunk / 4; i += kStateThreads)
        reinterpret_cast<float4 *>(&sm.Pm[0][0])[i] = Pg[i];
      const float *Ug = p.U + ((size_t(b) * H_v + h) * Lp + t0) * D + j0;
      for (int i = tid; i < kChunk * kSlice; i += kStateThreads) sm.U[i / kSlice][i % kSlice] = Ug[(i / kSlice) * D + i % kSlice];
      if (tid < kChunk) sm.G[tid] = p.Gc[(size_t(b) * H_v + h) * Lp + t0 + tid];
    }
    __syncthreads();

    // E[t][j] = U[t][j] - W[t] . S[j];  QS[t][j] = Q[t] . S[j]   (j = lane)
    float qs[kChunk / 8];
#pragma unroll
    for (int m = 0; m < kChunk / 8; ++m) {
      const int t = warp + 8 * m;
      float ew = 0.f, eq = 0.f;
      for (int i = 0; i < D; i += 4) {
        const float4 sv = *reinterpret_cast<const float4 *>(&sm.S[lane][i]);
        const float4 wv = *reinterpret_cast<const float4 *>(&sm.W[t][i]);
        const float4 qv = *reinterpret_cast<const float4 *>(&sm.Q[t][i]);
        ew += dot4(wv, sv);
        eq += dot4(qv, sv);
      }
      sm.E[t][lane] = t < n ? sm.U[t][lane] - ew : 0.f;
      qs[m] = eq;
    }
    __syncthreads();

    // O[t][j] = gamma_t QS[t][j] + sum_{s <= t} Pm[t][s] E[s][j]
#pragma unroll
    for (int m = 0; m < kChunk / 8; ++m) {
      const int t = warp + 8 * m;
      if (t < n) {
        float o = expf(sm.G[t]) * qs[m];
        for (int s = 0; s <= t; ++s) o = fmaf(sm.Pm[t][s], sm.E[s][lane], o);
        p.out[((size_t(b) * L + t0 + t) * H_v + h) * D + j0 + lane] = f2bf(o);
      }
    }

    // S[j][i] <- gamma_n S[j][i] + sum_t exp(G_n - G_t) E[t][j] K[t][i]
    // thread: row j = lane, columns i = warp*(D/8) .. +D/8
    {
      const float Gn = sm.G[n - 1];
      const float gn = expf(Gn);
      constexpr int CPW = D / 8;
      float acc[CPW];
#pragma unroll
      for (int c = 0; c < CPW; ++c) acc[c] = gn * sm.S[lane][warp * CPW + c];
      for (int t = 0; t < n; ++t) {
        const float f = expf(Gn - sm.G[t]) * sm.E[t][lane];
#pragma unroll
        for (int c = 0; c < CPW; c += 4) {
          const float4 kv = *reinterpret_cast<const float4 *>(&sm.K[t][warp * CPW + c]);
          acc[c] = fmaf(f, kv.x, acc[c]);
          acc[c + 1] = fmaf(f, kv.y, acc[c + 1]);
          acc[c + 2] = fmaf(f, kv.z, acc[c + 2]);
          acc[c + 3] = fmaf(f, kv.w, acc[c + 3]);
        }
      }
      __syncthreads();  // all reads of the old S (E, QS) finished above; S rows are private below
#pragma unroll
      for (int c = 0; c < CPW; ++c) sm.S[lane][warp * CPW + c] = acc[c];
    }
  }
  __syncthreads();
  for (int i = tid; i < kSlice * D; i += kStateThreads) Sg[i] = sm.S[i / D][i % D];
  if (slice == 0 && h == 0 && tid == 0) p.offsets[b] += L;
}

// ---------------------------------------------------------------------------
// 4. ring: the raw inputs of the last three positions of window ++ prompt.
//    Positions before the prompt already sit in their slots, so only prompt
//    tokens are written.  Runs after the conv kernel has read the old window.
// ---------------------------------------------------------------------------
__global__ void prefill_ring_kernel(const PrefillParams p) {
  const int b = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (c >= p.C) return;
  const int off = p.offsets[b];
#pragma unroll
  for (int i = 0; i < kHist; ++i) {
    const int t = p.L - kHist + i;
    if (t >= 0) p.ring[(size_t(b) * p.R + ring_slot(off + t, p.R)) * p.C + c] = p.x[(size_t(b) * p.L + t) * p.C + c];
  }
}

template <int D>
static cudaError_t launch_prefill_d(const PrefillParams &p, cudaStream_t stream) {
  cudaError_t e;
  e = launch_pdl(prefill_conv_kernel<D>, dim3(p.NC, 2 * p.H_k + p.H_v, p.B), dim3(D), stream, p);
  if (e != cudaSuccess) return e;
  // the ring update must follow the conv (which reads the old window) and
  // precede the state pass (which advances offsets)
  e = launch_pdl(prefill_ring_kernel, dim3((p.C + 255) / 256, p.B), dim3(256), stream, p);
  if (e != cudaSuccess) return e;
  const size_t chunk_smem = sizeof(ChunkSmem<D>);
  e = cudaFuncSetAttribute(prefill_chunk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(chunk_smem));
  if (e != cudaSuccess) return e;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.NC, p.H_v, p.B);
    cfg.blockDim = dim3(kChunkThreads);
    cfg.dynamicSmemBytes = chunk_smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, prefill_chunk_kernel<D>, p);
    if (e != cudaSuccess) return e;
  }
  const size_t state_smem = sizeof(StateSmem<D>);
  e = cudaFuncSetAttribute(prefill_state_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(state_smem));
  if (e != cudaSuccess) return e;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(D / kSlice, p.H_v, p.B);
    cfg.blockDim = dim3(kStateThreads);
    cfg.dynamicSmemBytes = state_smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, prefill_state_kernel<D>, p);
  }
  return e;
}

size_t prefill_workspace_bytes(int B, int L, int H_k, int H_v, int D) {
  return prefill_ws(B, L, H_k, H_v, D).total;
}

cudaError_t launch_prefill(const uint16_t *x, const uint16_t *w, const float *g, const float *beta, float *state,
                           uint16_t *ring, int32_t *offsets, uint16_t *out, void *ws, int B, int L, int H_k,
                           int H_v, int D, int R, int act, cudaStream_t stream) {
  PrefillParams p{};
  p.x = x, p.w = w, p.g = g, p.beta = beta, p.state = state, p.ring = ring, p.offsets = offsets, p.out = out;
  const PrefillWs l = prefill_ws(B, L, H_k, H_v, D);
  char *base = static_cast<char *>(ws);
  p.q = reinterpret_cast<float *>(base + l.q);
  p.k = reinterpret_cast<float *>(base + l.k);
  p.v = reinterpret_cast<float *>(base + l.v);
  p.W = reinterpret_cast<float *>(base + l.W);
  p.U = reinterpret_cast<float *>(base + l.U);
  p.Gc = reinterpret_cast<float *>(base + l.Gc);
  p.Pm = reinterpret_cast<float *>(base + l.Pm);
  p.B = B, p.L = L, p.NC = (L + kChunk - 1) / kChunk, p.H_k = H_k, p.H_v = H_v;
  p.C = (2 * H_k + H_v) * D, p.R = R, p.act = act;
  switch (D) {
    case 32: return launch_prefill_d<32>(p, stream);
    case 64: return launch_prefill_d<64>(p, stream);
    case 128: return launch_prefill_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
