// verify.cuh -- the fused conv + L2-norm + gated-delta-rule verify kernel.
//
// One CTA of 128 threads owns 32 state rows (d_v) of one (row b, value head h)
// and runs all T draft-plus-verify positions of that tile from the
// pre-verification state S_0, which it only reads ("MTP inference: review and
// commit structure", Functional commits item 2: speculative transactions with
// verifier buffers; "Add request-owned eight-way MTP serving for Qwen 35B",
// section 4: keep=0 must find the real base state).
//
// Arithmetic.  With gamma_t = exp(G_t), G_t = g_0 + ... + g_t, the gated delta
// rule S_t = a_t S_{t-1} + e_t k_t^T, e_t = b_t (v_t - a_t S_{t-1} k_t),
// o_t = S_t q_t unrolls, for state row j, into
//   e_t[j] = b_t v_t[j] - b_t gamma_t (S_0[j].k_t)
//            - sum_{s<t} b_t exp(G_t - G_s) (k_s.k_t) e_s[j]
//   o_t[j] = gamma_t (S_0[j].q_t) + sum_{s<=t} exp(G_t - G_s) (k_s.q_t) e_s[j]
// so a state row only needs its 2T dot products with S_0 (one batched warp
// reduction) plus per-head scalars that every CTA computes once in shared
// memory; the T sequential steps act on scalars, not on the 64 KiB state.
// This is the chunked (WY) form of the rule with one chunk of T positions
// (Yang et al., "Parallelizing Linear Transformers with the Delta Rule over
// Sequence Length", 2024), which differs from the step-by-step form only in
// rounding ("MTP inference: review and commit structure", Verification and
// limits).
//
// Captures for the commit (the "captured verification inputs" of "perf(qwen):
// full-context MTP draft prefill and replay-free rewind", Summary item 4):
//   RECOMPUTE: e_t[j] (fp32), the normalised k_t of the key head and the
//              cumulative log-decay G_t; commit rebuilds
//              S_K = gamma_{K-1} S_0 + sum_{s<K} exp(G_{K-1} - G_s) e_s k_s^T.
//   SNAPSHOT:  every S_t, written with the step-by-step update
//              S_t = a_t S_{t-1} + e_t k_t^T.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

template <int D, int T, int MODE>
__global__ void __launch_bounds__(kVerifyThreads) verify_kernel(const VerifyParams p) {
  using G = RowLanes<D>;
  constexpr int RPL = G::RPL, GPW = G::GPW, LPR = G::LPR;
  constexpr int NCH = 2 * D + kTileRows;  // q, k of the key head + this tile's v channels

  __shared__ __align__(16) float sq[T][D];
  __shared__ __align__(16) float sk[T][D];
  __shared__ float sv[T][kTileRows];
  __shared__ float s_inv[2 * T];
  __shared__ float s_dot[2][T][T];  // [0][s][t] = k_s.k_t, [1][s][t] = k_s.q_t
  __shared__ float sG[T], sBeta[T];
  __shared__ float sM[T][T], sN[T][T], sBg[T], sGam[T], sAlpha[T];

  const int tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  const int j0 = tile * kTileRows;
  const int H_v = p.H_v, H_k = p.H_k, C = p.C, R = p.R;
  const int rep = H_v / H_k;
  const int hk = h / rep;

  if (!p.active[b]) {
    // Inactive / padding / finished rows are inert: zero output, no state,
    // ring or workspace access.
    for (int i = tid; i < T * kTileRows; i += kVerifyThreads) {
      const int t = i / kTileRows, jj = i % kTileRows;
      p.out[((size_t(b) * T + t) * H_v + h) * D + j0 + jj] = 0;
    }
    return;
  }

  // 1. Issue the state loads first so the HBM reads overlap the conv prologue.
  const float *Sw = p.state + ((size_t(b) * H_v + h) * D + j0 + warp * 8) * D;
  float4 s[RPL];
#pragma unroll
  for (int i = 0; i < RPL; ++i) s[i] = ld_stream_f4(Sw + size_t(grp + GPW * i) * D + 4 * sub);

  // 2. Causal conv over window ++ x for the q/k channels of key head hk and the
  //    v channels of this tile; the raw inputs go to ring slots (off + t) mod R.
  const int off = p.offsets[b];
  const bool qk_writer = (tile == 0) && (h % rep == 0);
  for (int ci = tid; ci < NCH; ci += kVerifyThreads) {
    int c;
    float *dst;
    int dstride;
    bool write_ring;
    if (ci < D) {
      c = hk * D + ci;
      dst = &sq[0][ci];
      dstride = D;
      write_ring = qk_writer;
    } else if (ci < 2 * D) {
      c = H_k * D + hk * D + (ci - D);
      dst = &sk[0][ci - D];
      dstride = D;
      write_ring = qk_writer;
    } else {
      c = 2 * H_k * D + h * D + j0 + (ci - 2 * D);
      dst = &sv[0][ci - 2 * D];
      dstride = kTileRows;
      write_ring = true;
    }
    const uint2 wr = *reinterpret_cast<const uint2 *>(p.w + size_t(c) * kWidth);
    const float w0 = bf2f(uint16_t(wr.x & 0xffff)), w1 = bf2f(uint16_t(wr.x >> 16));
    const float w2 = bf2f(uint16_t(wr.y & 0xffff)), w3 = bf2f(uint16_t(wr.y >> 16));
    float xt[kHist + T];
    uint16_t xraw[T];
    const uint16_t *ringb = p.ring + size_t(b) * R * C + c;
#pragma unroll
    for (int i = 0; i < kHist; ++i) xt[i] = bf2f(ringb[size_t(ring_slot(off - kHist + i, R)) * C]);
#pragma unroll
    for (int t = 0; t < T; ++t) {
      xraw[t] = p.x[(size_t(b) * T + t) * C + c];
      xt[kHist + t] = bf2f(xraw[t]);
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float acc = w0 * xt[t];
      acc = fmaf(w1, xt[t + 1], acc);
      acc = fmaf(w2, xt[t + 2], acc);
      acc = fmaf(w3, xt[t + 3], acc);
      dst[t * dstride] = p.act ? silu(acc) : acc;
    }
    if (write_ring) {
      uint16_t *ringw = p.ring + size_t(b) * R * C + c;
#pragma unroll
      for (int t = 0; t < T; ++t) ringw[size_t(ring_slot(off + t, R)) * C] = xraw[t];
    }
  }
  if (tid < T) {
    sBeta[tid] = p.beta[(size_t(b) * T + tid) * H_v + h];
  }
  if (tid == 0) {
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const float gt = p.g[(size_t(b) * T + t) * H_v + h];
      acc += gt;
      sG[t] = acc;
      sAlpha[t] = expf(gt);
    }
  }
  __syncthreads();

  // 3. L2 norms of q_t and k_t (q also scaled by 1/sqrt(D)).
  for (int pr = warp; pr < 2 * T; pr += kVerifyThreads / 32) {
    const float *v = pr < T ? sq[pr] : sk[pr - T];
    float ss = 0.f;
    for (int i = lane; i < D; i += 32) ss = fmaf(v[i], v[i], ss);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    if (lane == 0) {
      const float inv = 1.0f / sqrtf(ss + kNormEps);
      s_inv[pr] = pr < T ? inv * (1.0f / sqrtf(float(D))) : inv;
    }
  }
  __syncthreads();
  for (int i = tid; i < 2 * T * D; i += kVerifyThreads) {
    const int pr = i / D, e = i % D;
    if (pr < T) sq[pr][e] *= s_inv[pr];
    else sk[pr - T][e] *= s_inv[pr];
  }
  __syncthreads();

  // 4. Per-head scalars: k_s.k_t, k_s.q_t and the decay/strength coefficients.
  for (int pr = warp; pr < 2 * T * T; pr += kVerifyThreads / 32) {
    const int which = pr / (T * T), st = pr % (T * T), s0 = st / T, t0 = st % T;
    const float *va = sk[s0];
    const float *vb = which ? sq[t0] : sk[t0];
    float d = 0.f;
    for (int i = lane; i < D; i += 32) d = fmaf(va[i], vb[i], d);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) d += __shfl_xor_sync(0xffffffffu, d, m);
    if (lane == 0) s_dot[which][s0][t0] = d;
  }
  __syncthreads();
  if (tid < T * T) {
    const int t = tid / T, s0 = tid % T;
    const float r = expf(sG[t] - sG[s0]);
    sM[t][s0] = s0 < t ? sBeta[t] * r * s_dot[0][s0][t] : 0.f;
    sN[t][s0] = s0 <= t ? r * s_dot[1][s0][t] : 0.f;
    if (s0 == 0) {
      sGam[t] = expf(sG[t]);
      sBg[t] = sBeta[t] * sGam[t];
    }
  }
  __syncthreads();

  // 5. The 2T dot products of every state row with S_0, one butterfly each.
  float red[2 * T];
#pragma unroll
  for (int m = 0; m < 2 * T; ++m) {
    const float4 vec = *reinterpret_cast<const float4 *>(m < T ? &sk[m][4 * sub] : &sq[m - T][4 * sub]);
    float acc[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) acc[i] = dot4(s[i], vec);
    red[m] = reduce_rows<D>(acc, lane);
  }

  // 6. Scalar recurrence for the row this lane now holds.
  const int istar = row_of_lane<D>(lane);
  const int jj = warp * 8 + grp + GPW * istar;  // row within the tile
  float e[T];
  float o[T];
#pragma unroll
  for (int t = 0; t < T; ++t) {
    float acc = fmaf(sBeta[t], sv[t][jj], -sBg[t] * red[t]);
#pragma unroll
    for (int s0 = 0; s0 < t; ++s0) acc = fmaf(-sM[t][s0], e[s0], acc);
    e[t] = acc;
    float ot = sGam[t] * red[T + t];
#pragma unroll
    for (int s0 = 0; s0 <= t; ++s0) ot = fmaf(sN[t][s0], e[s0], ot);
    o[t] = ot;
  }
  const bool row_leader = (lane & 3) == 0;  // four lanes hold each row after the butterfly
  if (row_leader) {
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const size_t idx = ((size_t(b) * T + t) * H_v + h) * D + j0 + jj;
      p.out[idx] = f2bf(o[t]);
      if (MODE == GDN_COMMIT_RECOMPUTE) p.ws_e[idx] = e[t];
    }
  }

  if (MODE == GDN_COMMIT_RECOMPUTE) {
    if (qk_writer)
      for (int i = tid; i < T * D; i += kVerifyThreads) {
        const int t = i / D, e2 = i % D;
        p.ws_k[((size_t(b) * T + t) * H_k + hk) * D + e2] = sk[t][e2];
      }
    if (tile == 0 && tid < T) p.ws_G[(size_t(b) * T + tid) * H_v + h] = sG[tid];
  } else {
    // SNAPSHOT: every lane needs e_t of each of its rows; fetch them from the
    // lane that computed them, then step the rows through S_t = a_t S_{t-1} + e_t k_t.
    const size_t plane = size_t(p.B) * H_v * D * D;
    float *snap = p.ws_snap + ((size_t(b) * H_v + h) * D + j0 + warp * 8) * D;
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
      const int src = grp * LPR + lane_of_row<D>(i);
      float4 st = s[i];
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const float et = __shfl_sync(0xffffffffu, e[t], src);
        const float4 kv = *reinterpret_cast<const float4 *>(&sk[t][4 * sub]);
        const float a = sAlpha[t];
        st.x = fmaf(et, kv.x, a * st.x);
        st.y = fmaf(et, kv.y, a * st.y);
        st.z = fmaf(et, kv.z, a * st.z);
        st.w = fmaf(et, kv.w, a * st.w);
        st_f4(snap + t * plane + size_t(grp + GPW * i) * D + 4 * sub, st);
      }
    }
  }
}

template <int D>
cudaError_t launch_verify_d(const VerifyParams &p, int T, int mode, cudaStream_t stream) {
  const dim3 grid(D / kTileRows, p.H_v, p.B), block(kVerifyThreads);
#define GDN_VERIFY_CASE(TT)                                                                   \
  case TT:                                                                                    \
    if (mode == GDN_COMMIT_RECOMPUTE)                                                         \
      verify_kernel<D, TT, GDN_COMMIT_RECOMPUTE><<<grid, block, 0, stream>>>(p);              \
    else                                                                                      \
      verify_kernel<D, TT, GDN_COMMIT_SNAPSHOT><<<grid, block, 0, stream>>>(p);               \
    break;
  switch (T) {
    GDN_VERIFY_CASE(1)
    GDN_VERIFY_CASE(2)
    GDN_VERIFY_CASE(3)
    GDN_VERIFY_CASE(4)
    GDN_VERIFY_CASE(5)
    GDN_VERIFY_CASE(6)
    GDN_VERIFY_CASE(7)
    GDN_VERIFY_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef GDN_VERIFY_CASE
  return cudaGetLastError();
}

}  // namespace gdn
