// verify.cuh -- the fused conv + L2-norm + gated-delta-rule verify kernel.
//
// Work decomposition.  One CTA of 2*d threads owns one (row b, value head h):
// its whole d_v x d_k state (64 KiB at d = 128) is staged in shared memory by
// d/32 bulk copies on the TMA engine, issued at entry, each completing on its
// own mbarrier.  Each thread convolves one q or k channel of the key head;
// the conv outputs are exchanged at the kernel's one block barrier, after
// which every warp owns 16 state rows (two groups of 8) and works alone.
// Lane l works on the d_k segment [4*(l % LPR), +4) of its rows.  A layer
// occupies about 1.3 CTAs per SM at B = 8, so with GDN_VERIFY_OVERLAP the next
// layer's CTAs fit beside it and stream their state while this one computes.
//
// The pre-verification state S_0 is only read ("MTP inference: review and
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
// reduction) plus per-head scalars, and the T sequential steps act on
// scalars, not on the 64 KiB state.  This is the chunked (WY) form of the rule
// with one chunk of T positions (Yang et al., "Parallelizing Linear
// Transformers with the Delta Rule over Sequence Length", 2024), equal to the
// step-by-step form up to rounding ("MTP inference: review and commit
// structure", Verification and limits).  The L2 norms are folded in as scale
// factors: every dot product is taken on the raw conv outputs and multiplied
// by 1/|k| (and 1/(|q| sqrt(d_k))) afterwards.
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

// Causal conv of one channel over T new positions: window xt[0..2] (oldest
// first) followed by the new inputs; taps w[0..3], w[3] on the current token.
template <int T>
__device__ __forceinline__ void conv1(const float (&w)[kWidth], const float (&xt)[kHist + T], int act,
                                      float (&y)[T]) {
#pragma unroll
  for (int t = 0; t < T; ++t) {
    float acc = w[0] * xt[t];
    acc = fmaf(w[1], xt[t + 1], acc);
    acc = fmaf(w[2], xt[t + 2], acc);
    acc = fmaf(w[3], xt[t + 3], acc);
    y[t] = act ? silu_fast(acc) : acc;
  }
}

// Load the taps, the committed window (ring slots 0..2) and the new inputs of
// channel c of row b and run its conv; optionally copy the new raw inputs into
// ring slots 3..2+T.
template <int T>
__device__ __forceinline__ void conv_channel(const VerifyParams &p, int b, int c, bool write_ring,
                                            float (&y)[T]) {
  const int C = p.C, R = p.R;
  const uint2 wr = *reinterpret_cast<const uint2 *>(p.w + size_t(c) * kWidth);
  const float w[kWidth] = {bf2f(uint16_t(wr.x & 0xffff)), bf2f(uint16_t(wr.x >> 16)),
                           bf2f(uint16_t(wr.y & 0xffff)), bf2f(uint16_t(wr.y >> 16))};
  uint16_t *ringb = p.ring + size_t(b) * R * C + c;
  const uint16_t *xb = p.x + size_t(b) * T * C + c;
  float xt[kHist + T];
  uint16_t xraw[T];
#pragma unroll
  for (int i = 0; i < kHist; ++i) xt[i] = bf2f(ringb[size_t(kWinSlot + i) * C]);
#pragma unroll
  for (int t = 0; t < T; ++t) {
    xraw[t] = xb[size_t(t) * C];
    xt[kHist + t] = bf2f(xraw[t]);
  }
  conv1<T>(w, xt, p.act, y);
  if (write_ring) {
#pragma unroll
    for (int t = 0; t < T; ++t) ringb[size_t(kNewSlot + t) * C] = xraw[t];
  }
}

// Shared memory of one verify CTA: the (row, head) state tile and the conv
// outputs of its key head.
template <int D, int T>
struct VerifySmem {
  float S[D * D];
  float q[T][D];
  float k[T][D];
  uint64_t bar[D / kTileRows];
};

template <int D, int T, int MODE>
__global__ void __launch_bounds__(2 * D, T <= 4 ? 2 : 1) verify_kernel(const VerifyParams p) {
  using G = RowLanes<D>;
  constexpr int RPL = G::RPL, GPW = G::GPW, LPR = G::LPR;
  constexpr int NT = D / kTileRows;   // 32-row tiles, one bulk copy and barrier each
  // per-head reductions: |q_t|^2, |k_t|^2, k_s.k_t (s<t), k_s.q_t (s<=t)
  constexpr int NKK = T * (T - 1) / 2, NKQ = T * (T + 1) / 2, NV = 2 * T + NKK + NKQ;

  extern __shared__ __align__(128) unsigned char vsm_raw[];
  VerifySmem<D, T> &sm = *reinterpret_cast<VerifySmem<D, T> *>(vsm_raw);

  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  const int H_v = p.H_v, H_k = p.H_k, R = p.R;
  const int rep = H_v / H_k;
  const int hk = h / rep;
  const int istar = row_of_lane<D>(lane);  // row (within a group of 8) this lane holds after a reduction
  const bool leader = (lane & 3) == 0;     // four lanes share a row after the reduction

  // With GDN_VERIFY_OVERLAP the caller guarantees that nothing issued since
  // the last call without the flag writes this call's state or active mask:
  // the kernel lets the next kernel start at once and stages its state tiles
  // before waiting for the preceding one.  Without the flag it waits first
  // and only then lets the next kernel start, so a chain of flagged verifies
  // can never run ahead of the last unflagged call.
  if (p.overlap) {
    pdl_trigger();
  } else {
    pdl_wait();
    pdl_trigger();
  }
  const bool active = p.active[b] != 0;
  constexpr uint32_t kTileBytes = kTileRows * D * sizeof(float);
  const float *Sg = p.state + (size_t(b) * H_v + h) * D * D;
  auto stage_state = [&]() {
    if (tid == 0) {
#pragma unroll
      for (int i = 0; i < NT; ++i) mbar_init(&sm.bar[i], 1);
      fence_mbar_init();
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        mbar_arrive_expect_tx(&sm.bar[i], kTileBytes);
        bulk_g2s(sm.S + i * kTileRows * D, Sg + size_t(i) * kTileRows * D, kTileBytes, &sm.bar[i]);
      }
    }
  };
  // ---- 1. stage the (row, head) state, 32 rows per bulk copy ----------------
  if (active) stage_state();
  if (p.overlap) pdl_wait();

  // DEFERRED: is a commit of this (row, head) still to be applied?
  int E = 0, K = 0;
  bool pending = false, mark = false;
  if (MODE == GDN_COMMIT_DEFERRED) {
    E = *p.ws_epoch;
    const int A = p.ws_applied[size_t(b) * H_v + h];
    K = p.ws_pend[b];
    mark = E > A;
    pending = mark && K >= 1;
  }
  if (!active) {
    // Inactive / padding / finished rows are inert: zero output, no ring
    // access.  A commit still pending from an earlier cycle is applied.
    for (int i = tid; i < T * D; i += 2 * D) p.out[((size_t(b) * T + i / D) * H_v + h) * D + i % D] = 0;
    if (!pending) {
      if (mark && tid == 0) p.ws_applied[size_t(b) * H_v + h] = E;
      return;
    }
    stage_state();
    __syncthreads();
  }

  const bool qk_writer = (h % rep) == 0;  // one CTA per key head writes its q/k ring slots
  constexpr int ROWS_W = 16;              // state rows per warp: two groups of 8
  const int jw0 = warp * ROWS_W;
  float q[T][4], k[T][4], vrow[ROWS_W / 8][T];
  float gt[T], bt[T];
  if (active) {
    // ---- 2. conv + activation: one q or k channel of the key head per thread
    {
      const bool is_k = tid >= D;
      const int ch = is_k ? tid - D : tid;
      float y[T];
      conv_channel<T>(p, b, (is_k ? H_k * D : 0) + hk * D + ch, qk_writer, y);
#pragma unroll
      for (int t = 0; t < T; ++t) (is_k ? sm.k : sm.q)[t][ch] = y[t];
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
      gt[t] = p.g[(size_t(b) * T + t) * H_v + h];
      bt[t] = p.beta[(size_t(b) * T + t) * H_v + h];
    }
    // the v channels of the rows this lane will hold, also before the barrier
#pragma unroll
    for (int grp8 = 0; grp8 < ROWS_W / 8; ++grp8)
      conv_channel<T>(p, b, 2 * H_k * D + h * D + jw0 + 8 * grp8 + grp + GPW * istar, leader, vrow[grp8]);
    __syncthreads();  // conv outputs and the initialised barriers are visible
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const float4 qv = *reinterpret_cast<const float4 *>(&sm.q[t][4 * sub]);
      const float4 kv = *reinterpret_cast<const float4 *>(&sm.k[t][4 * sub]);
      q[t][0] = qv.x, q[t][1] = qv.y, q[t][2] = qv.z, q[t][3] = qv.w;
      k[t][0] = kv.x, k[t][1] = kv.y, k[t][2] = kv.z, k[t][3] = kv.w;
    }
  }

  // ---- 3. per-head sums over the LPR lanes of a row group ------------------
  float red_h[NV];
  float inv_q[T], inv_k[T], Gc[T], gam[T];
  float decay[T][T];  // exp(G_t - G_s), s < t
  if (active) {
    int n = 0;
#pragma unroll
    for (int t = 0; t < T; ++t) {
      red_h[n++] = q[t][0] * q[t][0] + q[t][1] * q[t][1] + q[t][2] * q[t][2] + q[t][3] * q[t][3];
      red_h[n++] = k[t][0] * k[t][0] + k[t][1] * k[t][1] + k[t][2] * k[t][2] + k[t][3] * k[t][3];
    }
#pragma unroll
    for (int t = 0; t < T; ++t)
#pragma unroll
      for (int s0 = 0; s0 < t; ++s0)
        red_h[n++] = k[s0][0] * k[t][0] + k[s0][1] * k[t][1] + k[s0][2] * k[t][2] + k[s0][3] * k[t][3];
#pragma unroll
    for (int t = 0; t < T; ++t)
#pragma unroll
      for (int s0 = 0; s0 <= t; ++s0)
        red_h[n++] = k[s0][0] * q[t][0] + k[s0][1] * q[t][1] + k[s0][2] * q[t][2] + k[s0][3] * q[t][3];
#pragma unroll
    for (int m = LPR / 2; m >= 1; m >>= 1)
#pragma unroll
      for (int i = 0; i < NV; ++i) red_h[i] += __shfl_xor_sync(0xffffffffu, red_h[i], m);

    // ---- 4. per-head coefficients (every lane, in registers) ---------------
    const float qs = 1.0f / sqrtf(float(D));
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < T; ++t) {
      inv_q[t] = rsqrtf(red_h[2 * t] + kNormEps) * qs;
      inv_k[t] = rsqrtf(red_h[2 * t + 1] + kNormEps);
      acc += gt[t];
      Gc[t] = acc;
      gam[t] = expf(acc);
    }
#pragma unroll
    for (int t = 0; t < T; ++t)
#pragma unroll
      for (int s0 = 0; s0 < t; ++s0) decay[t][s0] = expf(Gc[t] - Gc[s0]);
  }

  // DEFERRED: coefficients of the pending commit, S <- gamma S + sum_s c_s e_s k_s^T
  // with the captures of the verify that preceded it
  const int old = (E - 1) & 1, cur = E & 1;
  float pc_gam = 0.f;
  if (MODE == GDN_COMMIT_DEFERRED && pending) pc_gam = expf(p.dh_G[old][(size_t(b) * T + (K - 1)) * H_v + h]);

  // ---- 5. this warp's 16 rows, in two groups of 8 ---------------------------
  if (!mbar_wait_bounded(&sm.bar[jw0 / kTileRows], 0)) {
    // The staged tile never arrived: flag it, give the copies one more bounded
    // wait so they do not land in a retired CTA's shared memory, and write
    // nothing for these rows.
    if (lane == 0) atomicOr(p.status, GDN_STATUS_TIMEOUT);
#pragma unroll
    for (int i = 0; i < NT; ++i) mbar_wait_bounded(&sm.bar[i], 0);
    return;
  }
  const size_t plane = size_t(p.B) * H_v * D * D;
#pragma unroll
  for (int grp8 = 0; grp8 < ROWS_W / 8; ++grp8) {
    const int jw = jw0 + 8 * grp8;  // first state row of this group
    const int jrow = jw + grp + GPW * istar;
    float4 s[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i)
      s[i] = *reinterpret_cast<const float4 *>(&sm.S[(jw + grp + GPW * i) * D + 4 * sub]);
    if (MODE == GDN_COMMIT_DEFERRED && pending) {
      // apply the pending commit to these rows (same arithmetic as the eager
      // RECOMPUTE commit) and write them back as the committed state
      const float GK = p.dh_G[old][(size_t(b) * T + (K - 1)) * H_v + h];
#pragma unroll
      for (int i = 0; i < RPL; ++i)
        s[i] = make_float4(pc_gam * s[i].x, pc_gam * s[i].y, pc_gam * s[i].z, pc_gam * s[i].w);
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) {
        if (t < K) {
          const float c = expf(GK - p.dh_G[old][(size_t(b) * T + t) * H_v + h]);
          const float4 kv =
              *reinterpret_cast<const float4 *>(p.dh_k[old] + ((size_t(b) * T + t) * H_k + hk) * D + 4 * sub);
          const float *ert = p.dh_e[old] + ((size_t(b) * T + t) * H_v + h) * D + jw;
#pragma unroll
          for (int i = 0; i < RPL; ++i) {
            const float f = c * ert[grp + GPW * i];
            s[i].x = fmaf(f, kv.x, s[i].x);
            s[i].y = fmaf(f, kv.y, s[i].y);
            s[i].z = fmaf(f, kv.z, s[i].z);
            s[i].w = fmaf(f, kv.w, s[i].w);
          }
        }
      }
      float *Sw = p.state_w + ((size_t(b) * H_v + h) * D + jw) * D;
#pragma unroll
      for (int i = 0; i < RPL; ++i) st_f4(Sw + size_t(grp + GPW * i) * D + 4 * sub, s[i]);
    }
    if (!active) continue;

    float red[2 * T];
#pragma unroll
    for (int mvec = 0; mvec < 2 * T; ++mvec) {
      const float *vv = mvec < T ? k[mvec] : q[mvec - T];
      const float4 vec = make_float4(vv[0], vv[1], vv[2], vv[3]);
      float acc[RPL];
#pragma unroll
      for (int i = 0; i < RPL; ++i) acc[i] = dot4(s[i], vec);
      red[mvec] = reduce_rows<D>(acc, lane);
    }
    const float *v = vrow[grp8];

    // scalar recurrence for the row this lane holds
    float e[T], o[T];
    {
      int nkk = 2 * T, nkq = 2 * T + NKK;
#pragma unroll
      for (int t = 0; t < T; ++t) {
        float acc = fmaf(bt[t], v[t], -(bt[t] * gam[t]) * (red[t] * inv_k[t]));
#pragma unroll
        for (int s0 = 0; s0 < t; ++s0) {
          const float kk = red_h[nkk++] * inv_k[s0] * inv_k[t];
          acc = fmaf(-(bt[t] * decay[t][s0] * kk), e[s0], acc);
        }
        e[t] = acc;
        float ot = gam[t] * (red[T + t] * inv_q[t]);
#pragma unroll
        for (int s0 = 0; s0 <= t; ++s0) {
          const float kq = red_h[nkq++] * inv_k[s0] * inv_q[t];
          ot = fmaf((s0 == t ? 1.0f : decay[t][s0]) * kq, e[s0], ot);
        }
        o[t] = ot;
      }
    }
    if (leader) {
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const size_t idx = ((size_t(b) * T + t) * H_v + h) * D + jrow;
        p.out[idx] = f2bf(o[t]);
        if (MODE == GDN_COMMIT_RECOMPUTE) p.ws_e[idx] = e[t];
        if (MODE == GDN_COMMIT_DEFERRED) p.dh_e[cur][idx] = e[t];
      }
    }
    if (MODE == GDN_COMMIT_SNAPSHOT) {
      // every lane needs e_t of each of its rows; fetch them from the lane
      // that computed them, then step the rows through S_t = a_t S_{t-1} + e_t k_t
      float *snap = p.ws_snap + ((size_t(b) * H_v + h) * D + jw) * D;
#pragma unroll
      for (int i = 0; i < RPL; ++i) {
        const int src = grp * LPR + lane_of_row<D>(i);
        float4 st = s[i];
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const float et = __shfl_sync(0xffffffffu, e[t], src);
          const float a = expf(gt[t]);
          st.x = fmaf(et, k[t][0] * inv_k[t], a * st.x);
          st.y = fmaf(et, k[t][1] * inv_k[t], a * st.y);
          st.z = fmaf(et, k[t][2] * inv_k[t], a * st.z);
          st.w = fmaf(et, k[t][3] * inv_k[t], a * st.w);
          st_f4(snap + t * plane + size_t(grp + GPW * i) * D + 4 * sub, st);
        }
      }
    }
  }
  if (MODE == GDN_COMMIT_DEFERRED && mark && tid == 0) p.ws_applied[size_t(b) * H_v + h] = E;
  if (!active) return;

  // ---- 6. captures of the key head and decay --------------------------------
  if (MODE == GDN_COMMIT_RECOMPUTE || MODE == GDN_COMMIT_DEFERRED) {
    float *wk = MODE == GDN_COMMIT_RECOMPUTE ? p.ws_k : p.dh_k[cur];
    float *wG = MODE == GDN_COMMIT_RECOMPUTE ? p.ws_G : p.dh_G[cur];
    if (qk_writer && warp == 0 && grp == 0)
#pragma unroll
      for (int t = 0; t < T; ++t)
        st_f4(wk + ((size_t(b) * T + t) * H_k + hk) * D + 4 * sub,
              make_float4(k[t][0] * inv_k[t], k[t][1] * inv_k[t], k[t][2] * inv_k[t], k[t][3] * inv_k[t]));
    if (warp == 0 && lane < T) {
#pragma unroll
      for (int t = 0; t < T; ++t)
        if (lane == t) wG[(size_t(b) * T + t) * H_v + h] = Gc[t];
    }
  }
}

// Launch one verify instantiation, raising its dynamic shared-memory limit on
// the first launch of that instantiation on each device.
template <int D, int T, int MODE>
cudaError_t launch_verify_kernel(dim3 grid, dim3 block, cudaStream_t stream, const VerifyParams &p) {
  static bool configured[64] = {false};  // one flag set per instantiation
  constexpr int smem = int(sizeof(VerifySmem<D, T>));
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(verify_kernel<D, T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  return launch_pdl_smem(verify_kernel<D, T, MODE>, grid, block, smem, stream, p);
}

template <int D>
cudaError_t launch_verify_d(const VerifyParams &p, int T, int mode, cudaStream_t stream) {
  const dim3 grid(p.H_v, p.B), block(2 * D);
#define GDN_VERIFY_CASE(TT)                                                                   \
  case TT:                                                                                    \
    return mode == GDN_COMMIT_RECOMPUTE                                                       \
               ? launch_verify_kernel<D, TT, GDN_COMMIT_RECOMPUTE>(grid, block, stream, p)    \
               : mode == GDN_COMMIT_SNAPSHOT                                                  \
                     ? launch_verify_kernel<D, TT, GDN_COMMIT_SNAPSHOT>(grid, block, stream, p) \
                     : launch_verify_kernel<D, TT, GDN_COMMIT_DEFERRED>(grid, block, stream, p);
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
}

}  // namespace gdn
