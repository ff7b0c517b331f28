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
// Kernels, in order (at d = 128 and 24 or more chunks once per chunk range,
// the state passes and the later ranges' products on two streams; see the
// segmented schedule below):
//   prefill_conv_kernel      conv + SiLU + L2 norm of every token -> Q, K, V
//                            (fp32; at d = 128 prefill_conv128_kernel,
//                            straight into the operand tiles)
//   prefill_ring_kernel      last three raw inputs into the ring
//   prefill_chunk_tc_kernel  per (chunk pair, value head): G, A, Tm, W, U, Pm
//                            (the products on tcgen05)
//   prefill_state_tc_kernel  d = 128: per (row, value head, 64 value rows):
//                            the chunk loop on tcgen05
//   prefill_state_kernel     d < 128: per (value head, 32-row d_v slice): the
//                            chunk loop on the CUDA cores
// The (last) state pass also advances offsets by L.
#include <atomic>
#include <mutex>

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
  float *q;   // [B][H_k][L][D]  normalised q / sqrt(D)   (CUDA-core state pass only)
  float *k;   // [B][H_k][L][D]  normalised k             (CUDA-core state pass only)
  float *W;   // [B][H_v][L][D]
  float *U;   // [B][H_v][L][D]
  float *Gc;  // [B][H_v][L]     within-chunk cumulative log-decay
  float *Pm;  // [B][H_v][NC][64][64]
  // bf16 hi/lo operand tiles for the tensor-core chunk kernel, one 64-token
  // chunk per tile, in the tcgen05 K-major no-swizzle canonical layout
  // (8-row x 16-byte core matrices; K-direction stride 128 B).
  uint16_t *qn_hi;          // [B][H_k][NCp] tiles of q  as [t][i] (K dim = d), bf16
                            // only: q enters the outputs alone
  uint16_t *kn_hi, *kn_lo;  // [B][H_k][NCp] tiles of k  as [t][i]
  uint16_t *kt_hi, *kt_lo;  // [B][H_k][NCp] tiles of k^T as [i][t] (K dim = 64 tokens)
  uint16_t *vt_hi, *vt_lo;  // [B][H_v][NCp] tiles of v^T as [j][t]
  // d = 128: the chunk kernel hands W and Pm to the tensor-core state pass
  // as bf16 tiles instead of fp32 rows
  uint16_t *w_hi, *w_lo;    // [B][H_v][NCp] tiles of W as [t][i] (K dim = d)
  uint16_t *pm_hi;          // [B][H_v][NCp] tiles of Pm as [t][s] (K dim = 64)
  uint32_t *status;         // sticky device status word
  int B, L, NC, NCp, H_k, H_v, C, R, act;
  // the launch covers chunks [seg0, seg1) (seg0 even: whole pairs); the
  // state pass advances offsets only in the launch with `last` set
  int seg0, seg1, last;
};

struct PrefillWs {
  size_t q, k, W, U, Gc, Pm, qn_hi, kn_hi, kn_lo, kt_hi, kt_lo, vt_hi, vt_lo, w_hi, w_lo, pm_hi, total;
};

// The sequential pass runs on the tensor cores at d = 128 (one TMEM lane per
// state row) and on the CUDA cores at d = 32, 64.
__host__ __device__ constexpr bool state_pass_tc(int D) { return D == 128; }

inline PrefillWs prefill_ws(int B, int L, int H_k, int H_v, int D) {
  const int NC = (L + kChunk - 1) / kChunk;
  const size_t Lp = size_t(NC) * kChunk;  // padded so every chunk tile is whole
  const bool tc = state_pass_tc(D);
  const int NCp = (NC + 1) & ~1;  // the tensor-core kernels work on chunk pairs
  PrefillWs w;
  size_t o = 0;
  w.q = o, o += tc ? 0 : align256(sizeof(float) * size_t(B) * H_k * Lp * D);
  w.k = o, o += tc ? 0 : align256(sizeof(float) * size_t(B) * H_k * Lp * D);
  w.W = o, o += tc ? 0 : align256(sizeof(float) * size_t(B) * H_v * Lp * D);
  w.U = o, o += align256(sizeof(float) * size_t(B) * H_v * Lp * D);
  w.Gc = o, o += align256(sizeof(float) * size_t(B) * H_v * Lp);
  w.Pm = o, o += tc ? 0 : align256(sizeof(float) * size_t(B) * H_v * NC * kChunk * kChunk);
  const size_t tile = size_t(kChunk) * D * sizeof(uint16_t);
  size_t *hk_tiles[5] = {&w.qn_hi, &w.kn_hi, &w.kn_lo, &w.kt_hi, &w.kt_lo};
  for (size_t *f : hk_tiles) *f = o, o += align256(tile * B * H_k * NCp);
  w.vt_hi = o, o += align256(tile * B * H_v * NCp);
  w.vt_lo = o, o += align256(tile * B * H_v * NCp);
  w.w_hi = o, o += tc ? align256(tile * B * H_v * NCp) : 0;
  w.w_lo = o, o += tc ? align256(tile * B * H_v * NCp) : 0;
  w.pm_hi = o, o += tc ? align256(size_t(kChunk) * kChunk * sizeof(uint16_t) * B * H_v * NCp) : 0;
  w.total = o;
  return w;
}


// Write one channel's 64 values into a natural tile ([t][i], K dim D) and,
// when `transposed` is set, into a transposed tile ([i][t], K dim 64).
template <int D>
__device__ __forceinline__ void store_tiles(const float (&y)[kChunk], int ch, uint16_t *nat_hi, uint16_t *nat_lo,
                                            uint16_t *tr_hi, uint16_t *tr_lo) {
  if (nat_hi) {
#pragma unroll
    for (int t = 0; t < kChunk; ++t) {
      uint16_t hi, lo;
      split_bf16(y[t], hi, lo);
      const uint32_t o = canon_off(t, ch, D) / 2;
      nat_hi[o] = hi;
      nat_lo[o] = lo;
    }
  }
  if (tr_hi) {
#pragma unroll
    for (int t8 = 0; t8 < kChunk; t8 += 8) {
      uint32_t h[4], l[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint16_t h0, l0, h1, l1;
        split_bf16(y[t8 + 2 * q], h0, l0);
        split_bf16(y[t8 + 2 * q + 1], h1, l1);
        h[q] = uint32_t(h0) | (uint32_t(h1) << 16);
        l[q] = uint32_t(l0) | (uint32_t(l1) << 16);
      }
      const uint32_t o = canon_off(ch, t8, kChunk) / 2;  // 16-byte aligned: t8 % 8 == 0
      *reinterpret_cast<uint4 *>(tr_hi + o) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4 *>(tr_lo + o) = make_uint4(l[0], l[1], l[2], l[3]);
    }
  }
}

// ---------------------------------------------------------------------------
// 1. conv + activation + L2 norm.  Block = D threads = the D channels of one
//    head (q, k or v) for one chunk of tokens of one row.  Tokens past L are
//    written as zeros so chunk tiles are whole.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(D) prefill_conv_kernel(const PrefillParams p) {
  const int chunk = p.seg0 + blockIdx.x, head = blockIdx.y, b = blockIdx.z;  // head in [0, 2 H_k + H_v)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = D / 32;
  __shared__ float s_part[kChunk][NW];
  __shared__ float s_inv[kChunk];
  __shared__ __align__(16) float s_y[kChunk][D + 4];  // q/k of the chunk, to store the [t][i] tile 16 bytes at a time
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
  // (ring slots 0..2)
  float h0, h1, h2;
  {
    float hv[kHist];
#pragma unroll
    for (int i = 0; i < kHist; ++i) {
      const int t = t0 - kHist + i;
      hv[i] = t >= L ? 0.f  // the padding chunk past the prompt
              : t >= 0 ? bf2f(p.x[(size_t(b) * L + t) * C + c])
                       : bf2f(p.ring[(size_t(b) * R + kWinSlot + kHist + t) * C + c]);
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
  const size_t tile = size_t(kChunk) * D;  // elements per bf16 tile
  if (kind == 2) {
    const int hv = head - 2 * H_k;
    const size_t tbase = ((size_t(b) * p.H_v + hv) * p.NCp + chunk) * tile;
    store_tiles<D>(y, tid, nullptr, nullptr, p.vt_hi + tbase, p.vt_lo + tbase);
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
#pragma unroll
  for (int i = 0; i < kChunk; ++i) y[i] *= s_inv[i];
  const size_t tbase = ((size_t(b) * H_k + hk) * p.NCp + chunk) * tile;
  // the [t][i] tile: a 16-byte run is 8 channels of one token, so the chunk
  // goes through shared memory and every thread stores whole runs
#pragma unroll
  for (int i = 0; i < kChunk; ++i) s_y[i][tid] = y[i];
  if (kind == 1) store_tiles<D>(y, tid, nullptr, nullptr, p.kt_hi + tbase, p.kt_lo + tbase);
  __syncthreads();
  {
    uint16_t *nh = (kind == 0 ? p.qn_hi : p.kn_hi) + tbase, *nl = kind == 0 ? nullptr : p.kn_lo + tbase;
    for (int u = tid; u < kChunk * (D / 8); u += D) {
      const int t = u / (D / 8), i8 = (u % (D / 8)) * 8;
      const uint32_t o = canon_off(t, i8, D) / 2;
      store8_split(&s_y[t][i8], nh + o, nl ? nl + o : nullptr);
    }
  }
  if (state_pass_tc(D) || chunk >= p.NC) return;
  float *dst = (kind == 0 ? p.q : p.k) + ((size_t(b) * H_k + hk) * Lp + t0) * D + tid;
#pragma unroll
  for (int i = 0; i < kChunk; ++i) dst[size_t(i) * D] = y[i];
}

// ---------------------------------------------------------------------------
// 1b. conv + activation + L2 norm at d = 128, for the tensor-core passes.
//    Block = one chunk of 64 tokens of one head (q, k or v) of one row, 128
//    threads; thread (o, g) = (tid % 16, tid / 16) owns channels 8o..8o+7 of
//    tokens 8g..8g+7.  That 8 x 8 block is exactly one 128-byte core matrix
//    of every operand tile the chunk feeds (the [t][i] tiles of q and k, the
//    [i][t] tiles of k and v), so each thread reads its inputs as 16-byte
//    runs of one token row, and a token's squared norm is the sum over the
//    16 lanes of its half warp.  Each 16 KiB tile is staged in shared memory
//    (the 16-byte rows of a 128-byte line rotated by an XOR key, so that the
//    lanes of a warp hit distinct banks) and copied out by the block as
//    whole contiguous lines.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    f[2 * q] = __uint_as_float(w[q] << 16);
    f[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
  }
}

// Shared staging of one bf16 hi/lo tile pair (64 x 128 elements = 1024
// lines' worth of 16-byte rows each): row r of 128-byte line l sits at
// position r ^ key(l) of the line.
struct ConvStage {
  uint4 hi[kChunk * 128 / 8], lo[kChunk * 128 / 8];
};

// One core matrix (8 rows of 8 values) split into bf16 hi/lo into line
// `line` of the staging tiles.
__device__ __forceinline__ void stage_core_split(const float (&v)[8][8], ConvStage &st, int line, int key) {
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // the rounding of store8_split
      const __nv_bfloat162 hv = __floats2bfloat162_rn(v[r][2 * q], v[r][2 * q + 1]);
      const __nv_bfloat162 lv =
          __floats2bfloat162_rn(v[r][2 * q] - __low2float(hv), v[r][2 * q + 1] - __high2float(hv));
      h[q] = *reinterpret_cast<const uint32_t *>(&hv);
      l[q] = *reinterpret_cast<const uint32_t *>(&lv);
    }
    st.hi[line * 8 + (r ^ key)] = make_uint4(h[0], h[1], h[2], h[3]);
    st.lo[line * 8 + (r ^ key)] = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// The staged tile pair out to global memory, 16 contiguous bytes per thread
// per step.  `tkey` selects the key of a line: its index mod 8 ([t][i]
// tiles, 16 lines per token group) or its index / 8 mod 8 ([i][t] tiles, 8
// lines per channel group).
// `lo` may be null (the hi tile alone).
__device__ __forceinline__ void flush_stage(const ConvStage &st, uint16_t *hi, uint16_t *lo, bool tkey) {
  __syncthreads();
  uint4 *gh = reinterpret_cast<uint4 *>(hi), *gl = reinterpret_cast<uint4 *>(lo);
  for (int i = threadIdx.x; i < kChunk * 128 / 8; i += blockDim.x) {
    const int line = i >> 3, key = (tkey ? line >> 3 : line) & 7;
    const int src = line * 8 + ((i & 7) ^ key);
    gh[i] = st.hi[src];
    if (lo) gl[i] = st.lo[src];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(128, 5) prefill_conv128_kernel(const PrefillParams p) {
  constexpr int D = 128;
  const int chunk = p.seg0 + blockIdx.x, head = blockIdx.y, b = blockIdx.z;  // head in [0, 2 H_k + H_v)
  const int tid = threadIdx.x, o = tid & 15, g = tid >> 4;
  pdl_wait();
  pdl_trigger();
  const int H_k = p.H_k, C = p.C, R = p.R, L = p.L;
  const int kind = head < H_k ? 0 : head < 2 * H_k ? 1 : 2;
  const int c0 = head * D + 8 * o;  // first of this thread's channels
  // raw inputs of tokens t1-3 .. t1+7: from the prompt, the committed window
  // (ring slots 0..2) before it, zeros past it
  const int t1 = chunk * kChunk + 8 * g;
  uint4 xr[8 + kHist];
#pragma unroll
  for (int k = 0; k < 8 + kHist; ++k) {
    const int t = t1 - kHist + k;
    xr[k] = t >= L   ? make_uint4(0, 0, 0, 0)
            : t >= 0 ? *reinterpret_cast<const uint4 *>(p.x + (size_t(b) * L + t) * C + c0)
                     : *reinterpret_cast<const uint4 *>(p.ring + (size_t(b) * R + kWinSlot + kHist + t) * C + c0);
  }
  float y[8][8];  // [token][channel]
  const uint4 *wp = reinterpret_cast<const uint4 *>(p.w + size_t(c0) * kWidth);
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // channels 2q, 2q+1: their taps are 16 bytes
    float w[8];
    unpack8(wp[q], w);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int i = 0; i < kWidth; ++i) {
        const uint32_t word = q == 0 ? xr[r + i].x : q == 1 ? xr[r + i].y : q == 2 ? xr[r + i].z : xr[r + i].w;
        acc0 = fmaf(w[i], __uint_as_float(word << 16), acc0);
        acc1 = fmaf(w[kWidth + i], __uint_as_float(word & 0xffff0000u), acc1);
      }
      const bool live = t1 + r < L;
      y[r][2 * q] = live ? (p.act ? silu_fast(acc0) : acc0) : 0.f;
      y[r][2 * q + 1] = live ? (p.act ? silu_fast(acc1) : acc1) : 0.f;
    }
  }
  __shared__ ConvStage st;
  const size_t tile = size_t(kChunk) * D;  // elements per bf16 tile
  // this thread's core matrix: line g * 16 + o of a [t][i] tile (K = D),
  // line o * 8 + g of an [i][t] tile (K = 64); both keyed by o % 8
  const int nat = g * (D / 8) + o, tra = o * (kChunk / 8) + g, key = o & 7;
  if (kind == 2) {
    float yt[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) yt[c][r] = y[r][c];
    const size_t tb = ((size_t(b) * p.H_v + (head - 2 * H_k)) * p.NCp + chunk) * tile;
    stage_core_split(yt, st, tra, key);
    flush_stage(st, p.vt_hi + tb, p.vt_lo + tb, true);
    return;
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) ss = fmaf(y[r][c], y[r][c], ss);
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);  // the 16 lanes of this token
    float inv = rsqrtf(ss + kNormEps);
    if (kind == 0) inv *= rsqrtf(float(D));
#pragma unroll
    for (int c = 0; c < 8; ++c) y[r][c] *= inv;
  }
  const int hk = kind == 0 ? head : head - H_k;
  const size_t tb = ((size_t(b) * H_k + hk) * p.NCp + chunk) * tile;
  stage_core_split(y, st, nat, key);
  if (kind == 0) {
    flush_stage(st, p.qn_hi + tb, nullptr, false);
    return;
  }
  flush_stage(st, p.kn_hi + tb, p.kn_lo + tb, false);
  float yt[8][8];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int c = 0; c < 8; ++c) yt[c][r] = y[r][c];
  stage_core_split(yt, st, tra, key);
  flush_stage(st, p.kt_hi + tb, p.kt_lo + tb, true);
}

// ---------------------------------------------------------------------------
// 2. per (pair of chunks, value head): G, A, Tm = (I + A)^-1, W, U, Pm, with
//    the four products on the tensor cores (tcgen05, accumulators in TMEM).
//
//    Two consecutive 64-token chunks are stacked so every product has M = 128:
//      KK = K K^T and QK = Q K^T   (128 x 128, K dim d)   -> A and Pm of each
//                                   chunk are the diagonal 64 x 64 blocks
//      W  = (Tm diag(beta gamma)) K,  U = (Tm diag(beta)) V  (128 x d, K dim
//           128 tokens; Tm is block diagonal, so the chunks stay separate)
//    The products that reach the state (KK, W, U) are taken in three bf16
//    passes, x = x_hi + x_lo with x_hi = bf16(x), x_lo = bf16(x - x_hi):
//    a b ~ a_hi b_hi + a_hi b_lo + a_lo b_hi, which keeps about 16 bits of
//    the fp32 operands (a single pass sits near the 1e-3 relative state
//    tolerance once the decay is weak enough for the state to carry over many
//    chunks).  QK only forms Pm, which only enters the bf16 outputs: one pass.
//    The UT transform itself is a forward substitution on the CUDA cores:
//    each thread of the first warpgroup solves one column of one chunk's Tm,
//    without block barriers.  Four warpgroups read the accumulators: threads
//    t, t + 128, t + 256 and t + 384 share TMEM lane t (token t of the pair)
//    and take one quarter of each epilogue's columns.
// ---------------------------------------------------------------------------
constexpr int kPairRows = 2 * kChunk;  // M of every product
constexpr int kTcThreads = 512;        // thread t <-> TMEM lane t % 128 <-> token t % 128 of the pair
constexpr int kTcGroups = kTcThreads / kPairRows;  // warpgroups
constexpr uint32_t kTmemCols = 256;    // [0,128): KK then W; [128,256): QK then U

template <int D>
struct TcLayout {
  static constexpr uint32_t nat_pair = 2u * kChunk * D * 2;       // a [t][i] tile pair, one of hi/lo
  static constexpr uint32_t tr_tile = uint32_t(D) * kChunk * 2;    // one [i][t] tile
  static constexpr uint32_t sq_op = kPairRows * kPairRows * 2;     // a 128 x 128 bf16 operand
  static constexpr uint32_t R0 = 0, R1 = 65536, R2 = 131072, R3 = 196608;
  // the UT solve's columns, in the second half of R1 (q takes the first;
  // the U operand's lo tile reuses this half after the solve)
  static constexpr uint32_t xs_off = 32768;
  // A of each chunk stored transposed, At[u][r] = A[r][u]: the epilogue's
  // writes (thread r, one column u at a time) are consecutive, and the
  // solve reads 16 rows of a column as four broadcast 16-byte loads
  static constexpr uint32_t solve_bytes = 2 * kChunk * kChunk * 4;
  static constexpr uint32_t misc = R3 + solve_bytes;              // G[128], beta[128], beta gamma[128]
  static constexpr uint32_t total = misc + 3 * kPairRows * 4;
  static_assert(2 * nat_pair <= 65536 && 4 * tr_tile <= 65536 && 2 * sq_op <= 65536, "regions");
  static_assert(nat_pair <= xs_off && xs_off + 2 * kChunk * kChunk * 4 <= 65536, "solve columns");
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_chunk_tc_kernel(const PrefillParams p) {
  using Lay = TcLayout<D>;
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[6];
  __shared__ uint32_t s_tmem;
  __shared__ float s_wsum[kTcThreads / 32];
  float(*At)[kChunk][kChunk] = reinterpret_cast<float(*)[kChunk][kChunk]>(smem + Lay::R3);
  float *sG = reinterpret_cast<float *>(smem + Lay::misc);
  float *sBeta = sG + kPairRows;
  float *sColW = sBeta + kPairRows;  // beta_s gamma_s of column s of the pair

  const int pair = p.seg0 / 2 + blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & (kPairRows - 1), wg = tid / kPairRows;  // token of the pair, warpgroup
  const int H_v = p.H_v, H_k = p.H_k, L = p.L;
  const int hk = h / (H_v / H_k);
  const int c0 = 2 * pair;
  const size_t Lp = size_t(p.NC) * kChunk;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;  // this warp's TMEM lanes

  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 6; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  pdl_wait();
  pdl_trigger();
  // tensor memory is taken only after the wait: no CTA holds it while it
  // waits for another grid, so an allocation never waits on a CTA that is
  // itself waiting for the allocating grid
  if (warp == 0) tmem_alloc(&s_tmem, kTmemCols);

  const size_t tile_el = size_t(kChunk) * D;
  if (tid == 0) {
    const size_t kq = ((size_t(b) * H_k + hk) * p.NCp + c0) * tile_el;
    mbar_arrive_expect_tx(&bars[0], 3 * Lay::nat_pair);
    bulk_g2s(smem + Lay::R0, p.kn_hi + kq, Lay::nat_pair, &bars[0]);
    bulk_g2s(smem + Lay::R0 + Lay::nat_pair, p.kn_lo + kq, Lay::nat_pair, &bars[0]);
    bulk_g2s(smem + Lay::R1, p.qn_hi + kq, Lay::nat_pair, &bars[0]);
    mbar_arrive_expect_tx(&bars[1], 4 * Lay::tr_tile);
    bulk_g2s(smem + Lay::R2, p.kt_hi + kq, 2 * Lay::tr_tile, &bars[1]);
    bulk_g2s(smem + Lay::R2 + 2 * Lay::tr_tile, p.kt_lo + kq, 2 * Lay::tr_tile, &bars[1]);
  }

  // within-chunk cumulative log-decay: rows 0-63 scan chunk c0, 64-127 chunk
  // c0+1 (every warpgroup, the first one stores it)
  const int tok = c0 * kChunk + row;
  float gt = 0.f, bt = 0.f;
  if (tok < L) {
    gt = p.g[(size_t(b) * L + tok) * H_v + h];
    bt = p.beta[(size_t(b) * L + tok) * H_v + h];
  }
  float incl = gt;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, incl, m);
    if (lane >= m) incl += o;
  }
  if (lane == 31) s_wsum[warp] = incl;
  tc_fence_before();
  __syncthreads();  // barriers, TMEM address, warp sums
  tc_fence_after();
  if (warp & 1) incl += s_wsum[warp - 1];
  if (wg == 0) {
    sG[row] = incl;
    sBeta[row] = bt;
  }
  const uint32_t tmem = s_tmem;
  bool ok = true;

  // ---- phase 1: KK and QK ---------------------------------------------------
  constexpr int pa[3] = {0, 0, 1}, pb[3] = {0, 1, 0};  // (hi,hi), (hi,lo), (lo,hi)
  if (tid == 0) {
    if (!mbar_wait_bounded(&bars[0], 0)) {
      ok = false;
    } else {
      tc_fence_after();
      constexpr uint32_t idesc = umma_idesc_bf16(kPairRows, kPairRows);
      constexpr uint32_t sbo = (D / 8) * 128;
      const uint32_t aK[2] = {sbase + Lay::R0, sbase + Lay::R0 + Lay::nat_pair};
      const uint32_t aQ = sbase + Lay::R1;
#pragma unroll
      for (int ps = 0; ps < 3; ++ps)
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_bf16(tmem, umma_desc(aK[pa[ps]] + k * 256, 128, sbo), umma_desc(aK[pb[ps]] + k * 256, 128, sbo),
                    idesc, ps | k);
      // QK only feeds Pm, which only enters the bf16 outputs: one pass
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        umma_bf16(tmem + 128, umma_desc(aQ + k * 256, 128, sbo), umma_desc(aK[0] + k * 256, 128, sbo), idesc,
                  k > 0);
    }
    umma_commit(&bars[2]);  // also arrives when nothing was issued
  }
  ok = mbar_wait_bounded(&bars[2], 0) && ok;
  tc_fence_after();
  __syncthreads();  // sG / sBeta of every token are visible

  // ---- epilogue 1: A (strictly lower, beta- and decay-weighted KK) and Pm ---
  const int q = row >> 6, tl = row & (kChunk - 1);  // chunk in the pair, row in the chunk
  const int chunk = c0 + q;
  if (ok) {
    const float Gt = sG[row], bq = sBeta[row];
    const int cb = q * kChunk;
    float *Pg = p.Pm + (((size_t(b) * H_v + h) * p.NC + chunk) * kChunk + tl) * kChunk;
    uint16_t *Pt = p.pm_hi + ((size_t(b) * H_v + h) * p.NCp + chunk) * kChunk * kChunk;
    {  // this warpgroup's 16 of the chunk's 64 columns
      constexpr int kE1 = kChunk / kTcGroups;
      const int cc = kE1 * wg;
      float kk[kE1], qk[kE1], pm[kE1];
      tmem_ld16x2(tmem + lane_base + cb + cc, tmem + lane_base + 128 + cb + cc, kk, qk);
#pragma unroll
      for (int j = 0; j < kE1; ++j) {
        const int sl = cc + j;
        const float decay = sl <= tl ? expf(Gt - sG[cb + sl]) : 0.f;
        At[q][sl][tl] = sl < tl ? bq * decay * kk[j] : 0.f;
        pm[j] = decay * qk[j];
      }
      if (chunk < p.NC) {
        if constexpr (state_pass_tc(D)) {
#pragma unroll
          for (int s8 = 0; s8 < kE1; s8 += 8)
            store8_split(pm + s8, Pt + canon_off(tl, cc + s8, kChunk) / 2, nullptr);
        } else {
#pragma unroll
          for (int j = 0; j < kE1; ++j) Pg[cc + j] = pm[j];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- UT transform: column s of chunk q of Tm, by forward substitution ----
  // Thread s keeps its column x in shared memory (the free half of the q
  // region, Tm[u][s] of chunk q at xs[q][u][s ^ 8 (u % 8)]: conflict-free
  // across the warp, and row runs of 8 columns stay contiguous) and solves
  // it in blocks of 16 rows: first the block's right-hand side loses the
  // contribution of every row already solved (16 independent accumulators),
  // then a 16-step substitution inside the block.
  constexpr int kBlk = 16;
  const int s = tl;
  float *xq = reinterpret_cast<float *>(smem + Lay::R1 + Lay::xs_off) + q * kChunk * kChunk;
  auto xsw = [](int u, int col) { return u * kChunk + (col ^ ((u & 7) << 3)); };
  if (ok && wg == 0) {
#pragma unroll
    for (int ib = 0; ib < kChunk / kBlk; ++ib) {
      const int r0 = ib * kBlk;
      float y[kBlk];
#pragma unroll
      for (int rr = 0; rr < kBlk; ++rr) y[rr] = r0 + rr == s ? 1.f : 0.f;
#pragma unroll 4  // the loads of four solved rows in flight together
      for (int u = 0; u < r0; ++u) {
        const float xu = xq[xsw(u, s)];
        const float4 *ac = reinterpret_cast<const float4 *>(&At[q][u][r0]);
#pragma unroll
        for (int v = 0; v < kBlk / 4; ++v) {
          const float4 a = ac[v];
          y[4 * v] = fmaf(-a.x, xu, y[4 * v]);
          y[4 * v + 1] = fmaf(-a.y, xu, y[4 * v + 1]);
          y[4 * v + 2] = fmaf(-a.z, xu, y[4 * v + 2]);
          y[4 * v + 3] = fmaf(-a.w, xu, y[4 * v + 3]);
        }
      }
#pragma unroll
      for (int rr = 0; rr < kBlk; ++rr) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums: a short dependency chain
#pragma unroll
        for (int c = 0; c < rr; ++c) d[c & 3] = fmaf(At[q][r0 + c][r0 + rr], y[c], d[c & 3]);
        y[rr] -= (d[0] + d[1]) + (d[2] + d[3]);
        xq[xsw(r0 + rr, s)] = y[rr];
      }
    }
  }
  // operands of W and U: Tm scaled by beta_s gamma_s (resp. beta_s) per
  // column s, block diagonal over the pair, split into bf16 hi/lo.  Written
  // by rows: item (chunk, row t, columns 8 c8 .. 8 c8 + 7) is one 16-byte row
  // of a core matrix, and eight consecutive threads (rows t .. t+7) fill a
  // whole 128-byte core matrix.
  if (ok && wg == 0) sColW[row] = sBeta[row] * expf(sG[row]);  // column `row` of the pair
  __syncthreads();  // every column is solved (and the U lo tile may reuse its space below)
  constexpr int kItems = kPairRows * kChunk / 8 / kTcThreads;  // 2 per thread
  float rv[kItems][8];
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int idx = it * kTcThreads + tid, qq = idx / (kChunk * 8), t = idx % kChunk, c8 = (idx / kChunk) % 8;
    const float4 *src = reinterpret_cast<const float4 *>(
        reinterpret_cast<const float *>(smem + Lay::R1 + Lay::xs_off) + qq * kChunk * kChunk + xsw(t, 8 * c8));
    const float4 lo4 = src[0], hi4 = src[1];
    rv[it][0] = lo4.x, rv[it][1] = lo4.y, rv[it][2] = lo4.z, rv[it][3] = lo4.w;
    rv[it][4] = hi4.x, rv[it][5] = hi4.y, rv[it][6] = hi4.z, rv[it][7] = hi4.w;
  }
  __syncthreads();
  if (ok) {
    uint16_t *awh = reinterpret_cast<uint16_t *>(smem + Lay::R0), *awl = awh + kPairRows * kPairRows;
    uint16_t *auh = reinterpret_cast<uint16_t *>(smem + Lay::R1), *aul = auh + kPairRows * kPairRows;
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int idx = it * kTcThreads + tid, qq = idx / (kChunk * 8), t = idx % kChunk, c8 = (idx / kChunk) % 8;
      const int tr = qq * kChunk + t, ks0 = qq * kChunk + 8 * c8;
      float w[8], u[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        w[e] = rv[it][e] * sColW[ks0 + e];
        u[e] = rv[it][e] * sBeta[ks0 + e];
      }
      const uint32_t o = canon_off(tr, ks0, kPairRows) / 2;
      store8_split(w, awh + o, awl + o);
      store8_split(u, auh + o, aul + o);
    }
    // the off-diagonal 64 x 64 quadrants are zero: in the canonical layout
    // each 8-row group of a quadrant is one contiguous kilobyte
    const uint4 z = make_uint4(0, 0, 0, 0);
    constexpr int kQuadU4 = kChunk / 8 * 1024 / 16;  // uint4 per quadrant
#pragma unroll
    for (int i = tid; i < 2 * kQuadU4; i += kTcThreads) {
      const int quad = i / kQuadU4, w = i % kQuadU4;  // quad 0: rows 0..63 x cols 64..127; 1: the mirror
      const int g = w / 64, c16 = w % 64;             // 8-row group, 16-byte unit within its kilobyte
      const uint32_t byte = uint32_t((quad * 8 + g) * (kPairRows / 8) * 128 + (1 - quad) * 1024 + c16 * 16);
      *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(awh) + byte) = z;
      *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(awl) + byte) = z;
      *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(auh) + byte) = z;
      *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(aul) + byte) = z;
    }
  }
  fence_async_smem();  // generic-proxy writes above -> tensor-core reads below
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- phase 2: W = A_W K (via K^T tiles), U = A_U V (via V^T tiles) -------
  if (tid == 0) {
    bool issued = false;
    if (ok && mbar_wait_bounded(&bars[1], 0)) {
      tc_fence_after();
      constexpr uint32_t idesc = umma_idesc_bf16(kPairRows, D);
      constexpr uint32_t sbo_a = (kPairRows / 8) * 128, sbo_t = (kChunk / 8) * 128;
      const uint32_t aW[2] = {sbase + Lay::R0, sbase + Lay::R0 + Lay::sq_op};
      const uint32_t aU[2] = {sbase + Lay::R1, sbase + Lay::R1 + Lay::sq_op};
      const uint32_t bT[2] = {sbase + Lay::R2, sbase + Lay::R2 + 2 * Lay::tr_tile};
#pragma unroll
      for (int ps = 0; ps < 3; ++ps)
#pragma unroll
        for (int k = 0; k < kPairRows / 16; ++k)
          umma_bf16(tmem, umma_desc(aW[pa[ps]] + k * 256, 128, sbo_a),
                    umma_desc(bT[pb[ps]] + (k / 4) * Lay::tr_tile + (k % 4) * 256, 128, sbo_t), idesc, ps | k);
      umma_commit(&bars[3]);
      issued = true;
      // the K^T tiles are free once W is done: bring in V^T
      if (mbar_wait_bounded(&bars[3], 0)) {
        const size_t vq = ((size_t(b) * H_v + h) * p.NCp + c0) * tile_el;
        mbar_arrive_expect_tx(&bars[4], 4 * Lay::tr_tile);
        bulk_g2s(smem + Lay::R2, p.vt_hi + vq, 2 * Lay::tr_tile, &bars[4]);
        bulk_g2s(smem + Lay::R2 + 2 * Lay::tr_tile, p.vt_lo + vq, 2 * Lay::tr_tile, &bars[4]);
        if (mbar_wait_bounded(&bars[4], 0)) {
          tc_fence_after();
#pragma unroll
          for (int ps = 0; ps < 3; ++ps)
#pragma unroll
            for (int k = 0; k < kPairRows / 16; ++k)
              umma_bf16(tmem + 128, umma_desc(aU[pa[ps]] + k * 256, 128, sbo_a),
                        umma_desc(bT[pb[ps]] + (k / 4) * Lay::tr_tile + (k % 4) * 256, 128, sbo_t), idesc,
                        ps | k);
        }
      }
      umma_commit(&bars[5]);
    }
    if (!issued) {  // let the waiting threads through
      umma_commit(&bars[3]);
      umma_commit(&bars[5]);
    }
  }

  // ---- epilogue 2: W and U rows (fp32) for the state pass; decay -----------
  // (columns per warpgroup: a quarter of d, at least 32, the last warpgroups
  // idle when d < 128)
  constexpr int kEpCols = D / kTcGroups >= 32 ? D / kTcGroups : 32;
  const int ep0 = wg * kEpCols;
  const bool okw = mbar_wait_bounded(&bars[3], 0) && ok;
  tc_fence_after();
  if (okw && chunk < p.NC) {
    float *Wg = p.W + ((size_t(b) * H_v + h) * Lp + size_t(chunk) * kChunk + tl) * D;
    const size_t wt = ((size_t(b) * H_v + h) * p.NCp + chunk) * tile_el;
#pragma unroll
    for (int cc = ep0; cc < ep0 + kEpCols && cc < D; cc += 32) {  // this warpgroup's columns
      float v[32];
      tmem_ld32(tmem + lane_base + cc, v);
      if constexpr (state_pass_tc(D)) {
#pragma unroll
        for (int i8 = 0; i8 < 32; i8 += 8) {
          const uint32_t o = canon_off(tl, cc + i8, D) / 2;
          store8_split(v + i8, p.w_hi + wt + o, p.w_lo + wt + o);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; j += 4) st_f4(Wg + cc + j, make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]));
      }
    }
    if (wg == 0) p.Gc[(size_t(b) * H_v + h) * Lp + size_t(chunk) * kChunk + tl] = sG[row];
  }
  const bool oku = mbar_wait_bounded(&bars[5], 0) && okw;
  tc_fence_after();
  if (oku && chunk < p.NC) {
    float *Ug = p.U + ((size_t(b) * H_v + h) * Lp + size_t(chunk) * kChunk + tl) * D;
#pragma unroll
    for (int cc = ep0; cc < ep0 + kEpCols && cc < D; cc += 32) {  // this warpgroup's columns
      float v[32];
      tmem_ld32(tmem + lane_base + 128 + cc, v);
#pragma unroll
      for (int j = 0; j < 32; j += 4) st_f4(Ug + cc + j, make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]));
    }
  }
  if (!oku && lane == 0) atomicOr(p.status, GDN_STATUS_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
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
// 3b. the sequential pass over chunks on the tensor cores (d = 128).  The
//     value rows j of the state evolve independently (the delta rule mixes
//     only its key columns i), so two CTAs per (row, value head) each carry
//     64 of them, M = 64 in every product (row r of a half in TMEM lane
//     32 (r / 16) + r % 16).  The fp32 state stays in TMEM for the whole
//     prompt; per chunk of n tokens (t, s index tokens, i, j state columns
//     and rows):
//       E'^T = S W^T,   QS^T = S Q^T       M = 64 rows j, N = 64 tokens each, K = d
//       E = U - E',  E~_t = exp(G_n - G_t) E_t,  S <- gamma_n S   (epilogue)
//       O^T = E^T Pm^T                     N = 64 tokens, K = 64 tokens
//       S += E~^T K                        N = d columns, K = 64 tokens
//       o_t = gamma_t QS^T + O^T,  then the bf16 hi/lo tiles of the new S
//     The products that feed the state (E', S += ...) take three bf16 passes
//     (hi hi, hi lo, lo hi); those that only feed the bf16 outputs (QS^T,
//     O^T) take one (both operands rounded to bf16 once: about 2^-9 of each
//     term, far inside the output tolerance, and nothing of it flows back
//     into the state).  The first products stack [W_hi; Q_hi; W_lo] into one
//     N = 192 operand against S_hi, so E'^T arrives as two column ranges the
//     epilogue adds.  The chunk's [E' | QS | E'] columns alternate between two
//     TMEM ranges by chunk parity: the next chunk's first products run while
//     this chunk's outputs are read out, after the bf16 hi/lo tiles of the
//     new state (all the next products wait for) are written.  Operand tiles
//     of the next chunk are fetched as soon as the products of this chunk
//     that read them are done.  The epilogues are spread over 16 warps: warp
//     w reads the 16 rows of TMEM lane quarter w % 4 and takes column group
//     w / 4, its two half-warps one half of it each (8 tokens or 16 state
//     columns a thread); the per-token decay factors are computed once per
//     chunk.
// ---------------------------------------------------------------------------
constexpr uint32_t kStCols = 512;
// [E'a | QS | E'c] of a chunk at kColE (even chunks) or kColE1 (odd chunks);
// O^T later takes the E'c columns; the state at kColS
constexpr uint32_t kColE = 0, kColE1 = 192, kColS = 384;
constexpr int kStThreads = 512;

constexpr int kStRows = 64;  // value rows j of the state per CTA
struct StLayout {  // d = 128, byte offsets in dynamic shared memory
  static constexpr uint32_t S_hi = 0, S_lo = 16384;         // S [j][i] of the half, K = 128: A operand
  static constexpr uint32_t W_hi = 32768, Q_hi = 49152;     // W, Q [t][i], K = 128: B operands;
  static constexpr uint32_t W_lo = 65536;                   // [W_hi; Q_hi; W_lo] is one 192-row one
  static constexpr uint32_t Kt_hi = 81920, Kt_lo = 98304;   // K^T [i][t], K = 64: B operand
  static constexpr uint32_t Pm_hi = 114688;                 // Pm [t][s], K = 64: B operand
  static constexpr uint32_t E_hi = 122880;                  // E^T [j][s], K = 64: A operand (bf16)
  static constexpr uint32_t Et_hi = 131072, Et_lo = 139264;  // decayed E^T [j][t], K = 64: A operand
  static constexpr uint32_t G = 147456;                     // [2][64] within-chunk G, by chunk parity
  static constexpr uint32_t Dec = G + 2 * kChunk * 4;        // [2][64] exp(G_n - G_t), 0 past n
  static constexpr uint32_t Gam = Dec + 2 * kChunk * 4;      // [2][64] exp(G_t)
  static constexpr uint32_t total = Gam + 2 * kChunk * 4;
};

__global__ void __launch_bounds__(kStThreads, 1) prefill_state_tc_kernel(const PrefillParams p) {
  constexpr int D = 128;
  using Lay = StLayout;
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[4];  // W+Q tiles, K^T+Pm tiles, products 1, products 2
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  float *sG = reinterpret_cast<float *>(smem + Lay::G);
  float *sDec = reinterpret_cast<float *>(smem + Lay::Dec);
  float *sGam = reinterpret_cast<float *>(smem + Lay::Gam);
  const int h = blockIdx.x >> 1, half = blockIdx.x & 1, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, cg = warp >> 2;  // TMEM lane quarter, column group
  const int hl = lane >> 4;                      // half of the column group
  const int jr = 16 * quarter + (lane & 15);     // this thread's row of the CTA's 64
  const int j = kStRows * half + jr;             // ... and of the state
  const int H_v = p.H_v, H_k = p.H_k, L = p.L, NC = p.NC;
  const int hk = h / (H_v / H_k);
  const size_t Lp = size_t(NC) * kChunk;
  const size_t bh = size_t(b) * H_v + h;
  const uint32_t sbase = smem_u32(smem);
  constexpr uint32_t kT128 = kChunk * D * sizeof(uint16_t);     // a 64 x 128 bf16 tile
  constexpr uint32_t kT64 = kChunk * kChunk * sizeof(uint16_t);  // a 64 x 64 bf16 tile
  const int tc0 = 16 * cg + 8 * hl;   // this thread's 8 tokens of a chunk
  const int ic0 = 32 * cg + 16 * hl;  // this thread's 16 state columns

  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    s_fail = 0;
  }
  pdl_wait();
  pdl_trigger();
  // tensor memory is taken only after the wait: no CTA holds it while it
  // waits for another grid, so an allocation never waits on a CTA that is
  // itself waiting for the allocating grid
  if (warp == 0) tmem_alloc(&s_tmem, kStCols);

  auto load_wq = [&](int c) {
    const size_t wq = (bh * p.NCp + c) * (kChunk * D);
    const size_t qq = ((size_t(b) * H_k + hk) * p.NCp + c) * (kChunk * D);
    mbar_arrive_expect_tx(&bars[0], 3 * kT128);
    bulk_g2s(smem + Lay::W_hi, p.w_hi + wq, kT128, &bars[0]);
    bulk_g2s(smem + Lay::W_lo, p.w_lo + wq, kT128, &bars[0]);
    bulk_g2s(smem + Lay::Q_hi, p.qn_hi + qq, kT128, &bars[0]);
  };
  auto load_kp = [&](int c) {
    const size_t kq = ((size_t(b) * H_k + hk) * p.NCp + c) * (kChunk * D);
    const size_t pq = (bh * p.NCp + c) * (kChunk * kChunk);
    mbar_arrive_expect_tx(&bars[1], 2 * kT128 + kT64);
    bulk_g2s(smem + Lay::Kt_hi, p.kt_hi + kq, kT128, &bars[1]);
    bulk_g2s(smem + Lay::Kt_lo, p.kt_lo + kq, kT128, &bars[1]);
    bulk_g2s(smem + Lay::Pm_hi, p.pm_hi + pq, kT64, &bars[1]);
  };
  // bf16 hi/lo of this thread's 16 state columns of row j into the A tiles of S
  auto put_row = [&](const float (&v)[16]) {
#pragma unroll
    for (int i8 = 0; i8 < 16; i8 += 8) {
      const uint32_t o = canon_off(jr, ic0 + i8, D);
      store8_split(v + i8, reinterpret_cast<uint16_t *>(smem + Lay::S_hi + o),
                   reinterpret_cast<uint16_t *>(smem + Lay::S_lo + o));
    }
  };
  // this launch's chunks [c_beg, c_end); c_beg is even, so a chunk's parity
  // (buffers, barrier phases) is the same counted from here or from 0
  const int c_beg = p.seg0, c_end = p.seg1;
  int pend_wq = -1, pend_kp = -1;  // (thread 0) chunk whose operand copies are in flight
  if (tid == 0 && c_end > c_beg) {
    load_wq(c_beg);
    load_kp(c_beg);
    pend_wq = pend_kp = c_beg;
  }
  if (tid < kChunk) {
    const int t = c_beg * kChunk + tid;
    sG[tid] = t < L ? p.Gc[bh * Lp + t] : 0.f;
  }
  tc_fence_before();
  __syncthreads();  // barriers, TMEM address, first gates
  tc_fence_after();
  const uint32_t tm = s_tmem;
  const uint32_t trow = tm + (uint32_t(32 * quarter) << 16);
  // 16x32bx2 loads and stores: the second half-warp 8 tokens or 16 columns on
  const uint32_t ttok = trow + 16 * cg, tcol = trow + kColS + 32 * cg;

  // the initial state: this thread's columns of row j into TMEM and the A tiles
  float *Sg = p.state + (bh * D + j) * D + ic0;
  {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const float4 f = *reinterpret_cast<const float4 *>(Sg + i);
      v[i] = f.x, v[i + 1] = f.y, v[i + 2] = f.z, v[i + 3] = f.w;
    }
    put_row(v);
    // the TMEM state is kept pre-multiplied by the decay of the chunk about
    // to be accumulated onto it (S <- gamma_n S + E~^T K)
    if (c_end > c_beg) {
      const float g0 = expf(sG[min(kChunk, L - c_beg * kChunk) - 1]);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] *= g0;
    }
    tmem_st_h16_async<16>(tcol, v);
    tmem_wait_st();
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  constexpr int pa[3] = {0, 0, 1}, pb[3] = {0, 1, 0};  // (hi,hi), (hi,lo), (lo,hi)
  constexpr uint32_t sbo128 = (D / 8) * 128, sbo64 = (kChunk / 8) * 128;
  constexpr uint32_t idesc64 = umma_idesc_bf16(kStRows, kChunk), idesc128 = umma_idesc_bf16(kStRows, D);
  constexpr uint32_t idesc192 = umma_idesc_bf16(kStRows, 192);
  // [E'a | QS | E'c] of chunk c lives in the columns of its parity, so that
  // chunk c+1's products 1 can run while chunk c's outputs are read out
  auto col_e = [](int c) -> uint32_t { return (c & 1) ? kColE1 : kColE; };
  // ---- products 1 of chunk c (thread 0):
  //   [E'a | QS | E'c]^T = S_hi [W_hi; Q_hi; W_lo]^T     (N = 192)
  //   E'a^T += S_lo W_hi^T                                (N = 64)
  // so E'^T = E'a^T + E'c^T takes the three passes and QS^T (outputs only)
  // the one ----
  auto issue_p1 = [&](int c) -> bool {
    const bool ok = mbar_wait_bounded(&bars[0], uint32_t(c) & 1u);
    if (ok) {
      pend_wq = -1;
      tc_fence_after();
      static_assert(Lay::Q_hi == Lay::W_hi + kT128 && Lay::W_lo == Lay::Q_hi + kT128, "[W_hi; Q_hi; W_lo]");
      const uint32_t ce = col_e(c);
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        umma_bf16(tm + ce, umma_desc(sbase + Lay::S_hi + k * 256, 128, sbo128),
                  umma_desc(sbase + Lay::W_hi + k * 256, 128, sbo128), idesc192, k > 0);
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        umma_bf16(tm + ce, umma_desc(sbase + Lay::S_lo + k * 256, 128, sbo128),
                  umma_desc(sbase + Lay::W_hi + k * 256, 128, sbo128), idesc64, true);
    }
    umma_commit(&bars[2]);  // also arrives when nothing was issued
    return ok;
  };
  // per-token factors of chunk c (threads < 64), in the buffers of its parity
  auto factors = [&](int c) {
    if (tid < kChunk) {
      const int n = min(kChunk, L - c * kChunk);
      const float *Gs = sG + (c & 1) * kChunk;
      sDec[(c & 1) * kChunk + tid] = tid < n ? expf(Gs[n - 1] - Gs[tid]) : 0.f;
      sGam[(c & 1) * kChunk + tid] = expf(Gs[tid]);
    }
  };
  if (c_end > c_beg) {
    if (tid == 0 && !issue_p1(c_beg)) s_fail = 1;
    factors(c_beg);
  }
  __syncthreads();  // factors of the first chunk

  for (int c = c_beg; c < c_end; ++c) {
    const int t0 = c * kChunk, n = min(kChunk, L - t0);
    const uint32_t ph = uint32_t(c) & 1u;
    const int par = c & 1;
    const uint32_t ce = col_e(c);
    if (s_fail) break;
    // the next chunk's gates (threads < 64, into the buffer of its parity)
    // and this thread's U of the chunk, in flight while products 1 finish
    // (that buffer was last read by the factors of chunk c-1)
    if (tid < kChunk && c + 1 < c_end) {
      const int t = (c + 1) * kChunk + tid;
      sG[((c + 1) & 1) * kChunk + tid] = t < L ? p.Gc[bh * Lp + t] : 0.f;
    }
    float u[8];
    {
      const float *Ug = p.U + (bh * Lp + t0 + tc0) * D + j;
#pragma unroll
      for (int t = 0; t < 8; ++t) u[t] = Ug[size_t(t) * D];
    }
    const bool ok1 = mbar_wait_bounded(&bars[2], ph);
    tc_fence_after();
    if (!ok1) s_fail = 1;
    if (tid == 0 && ok1 && c + 1 < c_end) {  // W and Q tiles are free
      load_wq(c + 1);
      pend_wq = c + 1;
    }
    // ---- epilogue 1: E^T and decayed E^T tiles ----
    {
      const float *dec = sDec + par * kChunk;
      float ea[8], ec[8], ev[8], et[8];
      tmem_ld_h8x2<8>(ttok + ce, ttok + ce + 2 * kChunk, ea, ec);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = tc0 + k;
        ev[k] = t < n ? u[k] - (ea[k] + ec[k]) : 0.f;
        et[k] = ev[k] * dec[t];
      }
      {
        const uint32_t o = canon_off(jr, tc0, kChunk);
        store8_split(ev, reinterpret_cast<uint16_t *>(smem + Lay::E_hi + o), nullptr);
        store8_split(et, reinterpret_cast<uint16_t *>(smem + Lay::Et_hi + o),
                     reinterpret_cast<uint16_t *>(smem + Lay::Et_lo + o));
      }
      tmem_wait_st();  // the previous epilogue's decayed state is in place
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (s_fail) break;
    // ---- products 2: O^T = E^T Pm^T, S += E~^T K ----
    bool ok2 = true;
    if (tid == 0) {
      ok2 = mbar_wait_bounded(&bars[1], ph);
      if (ok2) {
        pend_kp = -1;
        tc_fence_after();
        const uint32_t aE = sbase + Lay::E_hi;
        const uint32_t aEt[2] = {sbase + Lay::Et_hi, sbase + Lay::Et_lo};
        const uint32_t bK[2] = {sbase + Lay::Kt_hi, sbase + Lay::Kt_lo};
        // O^T only enters the bf16 outputs: one pass
#pragma unroll
        for (int k = 0; k < kChunk / 16; ++k)
          umma_bf16(tm + ce + 2 * kChunk, umma_desc(aE + k * 256, 128, sbo64),
                    umma_desc(sbase + Lay::Pm_hi + k * 256, 128, sbo64), idesc64, k > 0);
#pragma unroll
        for (int ps = 0; ps < 3; ++ps)
#pragma unroll
          for (int k = 0; k < kChunk / 16; ++k)
            umma_bf16(tm + kColS, umma_desc(aEt[pa[ps]] + k * 256, 128, sbo64),
                      umma_desc(bK[pb[ps]] + k * 256, 128, sbo64), idesc128, true);
      }
      umma_commit(&bars[3]);
    }
    ok2 = mbar_wait_bounded(&bars[3], ph) && ok2;
    tc_fence_after();
    if (!ok2) s_fail = 1;
    if (tid == 0 && ok2 && c + 1 < c_end) {  // K^T and Pm tiles are free
      load_kp(c + 1);
      pend_kp = c + 1;
    }
    // ---- epilogue 2: the A tiles of the updated state (the next chunk's
    // products 1 wait for them); this chunk's QS^T and O^T into registers ----
    float qs[8], eo[8];
    tmem_ld_h8x2<8>(ttok + ce + kChunk, ttok + ce + 2 * kChunk, qs, eo);
    {
      float v[16];
      tmem_ld_h16<16>(tcol, v);
      put_row(v);
      if (c + 1 < c_end) {  // the TMEM state, decayed for the next chunk
        const float gn = expf(sG[((c + 1) & 1) * kChunk + min(kChunk, L - (c + 1) * kChunk) - 1]);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= gn;
        tmem_st_h16_async<16>(tcol, v);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (s_fail) break;
    // ---- the next chunk's products 1 run while this chunk's outputs go out ----
    if (c + 1 < c_end) {
      if (tid == 0 && !issue_p1(c + 1)) s_fail = 1;
      factors(c + 1);
    }
    {
      const float *gam = sGam + par * kChunk;
      uint16_t *o = p.out + ((size_t(b) * L + t0 + tc0) * H_v + h) * D + j;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (tc0 + k < n) o[size_t(k) * H_v * D] = f2bf(fmaf(gam[tc0 + k], qs[k], eo[k]));
    }
    __syncthreads();  // the next chunk's factors (and any failure) are visible
  }
  if (!s_fail) {
    float v[16];
    tmem_ld_h16<16>(tcol, v);
#pragma unroll
    for (int i = 0; i < 16; i += 4) st_f4(Sg + i, make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
  } else if (tid == 0) {
    atomicOr(p.status, GDN_STATUS_TIMEOUT);
    // copies still in flight must land before the CTA leaves
    if (pend_wq >= 0) mbar_wait_bounded(&bars[0], uint32_t(pend_wq) & 1u);
    if (pend_kp >= 0) mbar_wait_bounded(&bars[1], uint32_t(pend_kp) & 1u);
  }
  if (p.last && h == 0 && half == 0 && tid == 0) p.offsets[b] += L;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, kStCols);
}

// ---------------------------------------------------------------------------
// 4. ring: slots 0..2 become the raw inputs of the last three positions of
//    window ++ prompt (for L < 3 partly the old window, read before any
//    write by the same thread).  Runs after the conv kernel has read the old
//    window.
// ---------------------------------------------------------------------------
__global__ void prefill_ring_kernel(const PrefillParams p) {
  const int b = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (c >= p.C) return;
  uint16_t *ring = p.ring + size_t(b) * p.R * p.C + c;
  uint16_t w[kHist];
#pragma unroll
  for (int i = 0; i < kHist; ++i) {
    const int t = p.L - kHist + i;  // prompt index; negative reaches the old window
    w[i] = t >= 0 ? p.x[(size_t(b) * p.L + t) * p.C + c] : ring[size_t(kWinSlot + kHist + t) * p.C];
  }
#pragma unroll
  for (int i = 0; i < kHist; ++i) ring[size_t(kWinSlot + i) * p.C] = w[i];
}

// Launch with or without programmatic stream serialization, at the stream's
// priority or (priority != 0) at that launch priority.
template <typename K>
static cudaError_t launch_ex(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                             const PrefillParams &p, int priority = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n++].val.programmaticStreamSerializationAllowed = 1;
  }
  if (priority != 0) {
    attr[n].id = cudaLaunchAttributePriority;
    attr[n++].val.priority = priority;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Raise the kernels' dynamic shared-memory limits, once per device.
template <int D>
static cudaError_t set_prefill_smem() {
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && configured[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(prefill_chunk_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(TcLayout<D>::total));
  if (e == cudaSuccess && state_pass_tc(D))
    e = cudaFuncSetAttribute(prefill_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(StLayout::total));
  if (e == cudaSuccess && !state_pass_tc(D))
    e = cudaFuncSetAttribute(prefill_state_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(sizeof(StateSmem<D>)));
  if (e == cudaSuccess && dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  return e;
}

// conv and chunk products of chunks [p.seg0, p.seg1) on `stream`
template <int D>
static cudaError_t launch_chunk_stage(const PrefillParams &p, cudaStream_t stream, bool pdl) {
  const int nchunks = ((p.seg1 + 1) & ~1) - p.seg0;  // whole pairs (the padding chunk past an odd NC)
  cudaError_t e;
  if constexpr (state_pass_tc(D))
    e = launch_ex(prefill_conv128_kernel, dim3(nchunks, 2 * p.H_k + p.H_v, p.B), dim3(128), 0, stream, pdl, p);
  else
    e = launch_ex(prefill_conv_kernel<D>, dim3(nchunks, 2 * p.H_k + p.H_v, p.B), dim3(D), 0, stream, pdl, p);
  if (e != cudaSuccess) return e;
  // the ring update follows the conv of the first chunks, the only one that
  // reads the old window
  if (p.seg0 == 0) {
    e = launch_ex(prefill_ring_kernel, dim3((p.C + 255) / 256, p.B), dim3(256), 0, stream, pdl, p);
    if (e != cudaSuccess) return e;
  }
  return launch_ex(prefill_chunk_tc_kernel<D>, dim3(nchunks / 2, p.H_v, p.B), dim3(kTcThreads), TcLayout<D>::total,
                   stream, pdl, p);
}

template <int D>
static cudaError_t launch_state_stage(const PrefillParams &p, cudaStream_t stream, bool pdl, int priority = 0) {
  if constexpr (state_pass_tc(D))
    return launch_ex(prefill_state_tc_kernel, dim3(2 * p.H_v, p.B), dim3(kStThreads), StLayout::total, stream, pdl, p,
                     priority);
  else
    return launch_ex(prefill_state_kernel<D>, dim3(D / kSlice, p.H_v, p.B), dim3(kStateThreads),
                     sizeof(StateSmem<D>), stream, pdl, p);
}

// The segmented schedule: the sequential state pass of each range of chunks
// (two CTAs per (row, value head): 2 B H_v SMs) runs on the caller's stream
// at the highest launch priority, the first one chained to the first range's
// products by programmatic serialization; the conv and chunk products of the
// later ranges run on a side stream on the remaining SMs, forked once the
// first range's products are done.  Stream order and events carry every
// dependency (no kernel waits on another's flag), and the caller's stream
// ends behind the last state pass, which waited for the last products.
constexpr int kMaxSegments = 8;
struct PrefillSide {
  cudaStream_t side = nullptr;
  cudaEvent_t ev[kMaxSegments + 1] = {};
  int high = 0;  // the device's greatest stream priority
  bool ready = false, failed = false;
};

static std::mutex &prefill_side_mutex() {
  static std::mutex m;
  return m;
}

// (with prefill_side_mutex held) the current device's side stream and events
static PrefillSide *prefill_side() {
  static PrefillSide sides[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  PrefillSide &s = sides[dev];
  if (!s.ready && !s.failed) {
    int least = 0, greatest = 0;
    bool ok = cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess &&
              cudaStreamCreateWithPriority(&s.side, cudaStreamNonBlocking, least) == cudaSuccess;
    s.high = greatest;
    for (int i = 0; ok && i <= kMaxSegments; ++i)
      ok = cudaEventCreateWithFlags(&s.ev[i], cudaEventDisableTiming) == cudaSuccess;
    s.ready = ok;
    s.failed = !ok;
  }
  return s.ready ? &s : nullptr;
}

// SMs of the current device (cached per device; 0 if unknown).
static int prefill_sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 0) n = 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Chunk ranges: a short first range (so the state pass starts early), then
// the rest in up to kMaxSegments - 1 even-sized ranges of whole pairs.
static int prefill_segments(int NC, int (&bound)[kMaxSegments + 1]) {
  constexpr int kFirst = 8, kMinRest = 16;
  if (NC < kFirst + kMinRest) return 0;
  const int rest = NC - kFirst;
  int n = (rest + kMinRest - 1) / kMinRest;
  n = n < kMaxSegments - 1 ? n : kMaxSegments - 1;
  bound[0] = 0;
  bound[1] = kFirst;
  for (int i = 1; i <= n; ++i) {
    int c = kFirst + int((long(rest) * i) / n);
    c = i == n ? NC : (c & ~1);
    bound[i + 1] = c;
  }
  return n + 1;
}

template <int D>
static cudaError_t launch_prefill_d(const PrefillParams &p0, cudaStream_t stream) {
  cudaError_t e = set_prefill_smem<D>();
  if (e != cudaSuccess) return e;
  int bound[kMaxSegments + 1];
  // ranges only when a range's state pass (2 B H_v CTAs, one per SM) fits in
  // one wave beside the products of the next range
  const bool fits = 2 * p0.B * p0.H_v <= prefill_sm_count();
  const int nseg = state_pass_tc(D) && fits ? prefill_segments(p0.NC, bound) : 0;
  if (nseg > 1) {
    std::lock_guard<std::mutex> lock(prefill_side_mutex());
    PrefillSide *side = prefill_side();
    if (side) {
      for (int sgi = 0; sgi < nseg; ++sgi) {
        PrefillParams p = p0;
        p.seg0 = bound[sgi], p.seg1 = bound[sgi + 1], p.last = sgi == nseg - 1;
        if (sgi == 0) {  // products on the caller's stream, the side stream forked behind them
          if ((e = launch_chunk_stage<D>(p, stream, false)) != cudaSuccess) return e;
          if ((e = cudaEventRecord(side->ev[0], stream)) != cudaSuccess) return e;
          if ((e = cudaStreamWaitEvent(side->side, side->ev[0], 0)) != cudaSuccess) return e;
          if ((e = launch_state_stage<D>(p, stream, true, side->high)) != cudaSuccess) return e;
        } else {  // products on the side stream, the state pass behind them on the caller's
          if ((e = launch_chunk_stage<D>(p, side->side, false)) != cudaSuccess) return e;
          if ((e = cudaEventRecord(side->ev[sgi], side->side)) != cudaSuccess) return e;
          if ((e = cudaStreamWaitEvent(stream, side->ev[sgi], 0)) != cudaSuccess) return e;
          if ((e = launch_state_stage<D>(p, stream, false, side->high)) != cudaSuccess) return e;
        }
      }
      return cudaSuccess;
    }
  }
  // one range: every kernel on the caller's stream, chained by PDL
  PrefillParams p = p0;
  p.seg0 = 0, p.seg1 = p.NC, p.last = 1;
  if ((e = launch_chunk_stage<D>(p, stream, true)) != cudaSuccess) return e;
  return launch_state_stage<D>(p, stream, true);
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
  p.W = reinterpret_cast<float *>(base + l.W);
  p.U = reinterpret_cast<float *>(base + l.U);
  p.Gc = reinterpret_cast<float *>(base + l.Gc);
  p.Pm = reinterpret_cast<float *>(base + l.Pm);
  p.qn_hi = reinterpret_cast<uint16_t *>(base + l.qn_hi);
  p.kn_hi = reinterpret_cast<uint16_t *>(base + l.kn_hi);
  p.kn_lo = reinterpret_cast<uint16_t *>(base + l.kn_lo);
  p.kt_hi = reinterpret_cast<uint16_t *>(base + l.kt_hi);
  p.kt_lo = reinterpret_cast<uint16_t *>(base + l.kt_lo);
  p.vt_hi = reinterpret_cast<uint16_t *>(base + l.vt_hi);
  p.vt_lo = reinterpret_cast<uint16_t *>(base + l.vt_lo);
  p.w_hi = reinterpret_cast<uint16_t *>(base + l.w_hi);
  p.w_lo = reinterpret_cast<uint16_t *>(base + l.w_lo);
  p.pm_hi = reinterpret_cast<uint16_t *>(base + l.pm_hi);
  p.B = B, p.L = L, p.NC = (L + kChunk - 1) / kChunk, p.H_k = H_k, p.H_v = H_v;
  p.NCp = (p.NC + 1) & ~1;
  p.status = status_word_address();
  if (!p.status) return cudaErrorInvalidValue;
  p.C = (2 * H_k + H_v) * D, p.R = R, p.act = act;
  switch (D) {
    case 32: return launch_prefill_d<32>(p, stream);
    case 64: return launch_prefill_d<64>(p, stream);
    case 128: return launch_prefill_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
