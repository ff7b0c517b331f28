// verify.cuh -- the fused conv + L2-norm + gated-delta-rule verify kernel.
//
// Work decomposition.  One CTA of 2d threads owns one (row b, value head h):
// its whole d_v x d_k state (64 KiB at d = 128) is staged in shared memory by
// d/32 bulk copies on the TMA engine, issued at entry, each completing on its
// own mbarrier.  The threads convolve the q and k channels of the key head
// (one per thread); the conv outputs are exchanged at the kernel's one block
// barrier, after which every warp owns 16 state rows (two groups of 8) and
// works alone.  Lane l works on the d_k segment [4*(l % LPR), +4) of its
// rows.  A layer occupies about 1.3 CTAs per SM at B = 8, so with
// GDN_VERIFY_OVERLAP part of the next layer's CTAs fit beside it and stream
// their state while this one computes.
//
// (d = 128 in RECOMPUTE and DEFERRED mode runs the tensor-core verify of
// verify_tc.cuh; this CUDA-core kernel serves d = 32, 64 and SNAPSHOT mode.)
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

#include <atomic>

#include "gdn_common.cuh"

namespace gdn {

// Raw conv inputs of one channel of one row: taps w[0..3] (w[3] on the
// current token), the committed window (ring slots 0..2, oldest first) and
// the T new inputs, all as bf16 bit patterns.  Loading every channel a
// thread needs before any arithmetic or store keeps the conv to a single
// round trip to memory.
template <int T>
struct ConvIn {
  uint2 w;
  uint16_t win[kHist];
  uint16_t x[T];
};

template <int T>
__device__ __forceinline__ void conv_load(const VerifyParams &p, int b, int c, ConvIn<T> &in) {
  const int C = p.C;
  in.w = *reinterpret_cast<const uint2 *>(p.w + size_t(c) * kWidth);
  const uint16_t *ringb = p.ring + size_t(b) * p.R * C + c;
  const uint16_t *xb = p.x + size_t(b) * T * C + c;
#pragma unroll
  for (int i = 0; i < kHist; ++i) in.win[i] = ringb[size_t(kWinSlot + i) * C];
#pragma unroll
  for (int t = 0; t < T; ++t) in.x[t] = xb[size_t(t) * C];
}

// Causal conv over the T new positions, then the activation.
template <int T>
__device__ __forceinline__ void conv_eval(const ConvIn<T> &in, int act, float (&y)[T]) {
  const float w0 = bf2f(uint16_t(in.w.x & 0xffff)), w1 = bf2f(uint16_t(in.w.x >> 16));
  const float w2 = bf2f(uint16_t(in.w.y & 0xffff)), w3 = bf2f(uint16_t(in.w.y >> 16));
  float xt[kHist + T];
#pragma unroll
  for (int i = 0; i < kHist; ++i) xt[i] = bf2f(in.win[i]);
#pragma unroll
  for (int t = 0; t < T; ++t) xt[kHist + t] = bf2f(in.x[t]);
#pragma unroll
  for (int t = 0; t < T; ++t) {
    float acc = w0 * xt[t];
    acc = fmaf(w1, xt[t + 1], acc);
    acc = fmaf(w2, xt[t + 2], acc);
    acc = fmaf(w3, xt[t + 3], acc);
    y[t] = act ? silu_fast(acc) : acc;
  }
}

// The new raw inputs of channel c go to ring slots 3..2+T.
template <int T>
__device__ __forceinline__ void conv_store_ring(const VerifyParams &p, int b, int c, const ConvIn<T> &in) {
  uint16_t *ringb = p.ring + size_t(b) * p.R * p.C + c;
#pragma unroll
  for (int t = 0; t < T; ++t) ringb[size_t(kNewSlot + t) * p.C] = in.x[t];
}

// Shared memory of one verify CTA: the (row, head) state tile, the conv
// outputs of its key head and, in DEFERRED mode, the captures of the previous
// verify (e_t, normalised k_t, G_t) for the commit that may still be pending.
template <int D, int T>
struct VerifySmem {
  alignas(128) float S[D * D];  // fp32 state tile
  float q[T][D];
  float k[T][D];
  float ce[T][D];
  float ck[T][D];
  float cG[kMaxT];
  // T >= 4: the per-head scalars, computed once per CTA
  float hraw[T * T + 2 * T];  // |q_t|^2, |k_t|^2, k_s.k_t (s<t), k_s.q_t (s<=t) of the raw conv outputs
  float cA[T][T];             // beta_t e^{G_t-G_s} (k^_s.k^_t), s < t: weight of e_s in e_t
  float cQ[T][T];             // e^{G_t-G_s} (k^_s.q^_t), s <= t: weight of e_s in o_t
  float cbk[T], cgq[T], cinvk[T], cGc[T];
  float gsq[T][8];  // gated RMSNorm: per-warp sums of o_t^2 (at most 8 warps)
  uint64_t bar[D / kTileRows];
  uint64_t cbar;
};

// Threads per verify CTA: 2d (8 warps at d = 128, 16 state rows per warp).
// Measured at B = 8, T = 2: d threads (3 CTAs per SM, 32 rows per warp) make
// a layer about 1 us slower, the longer per-warp row loop costing more than
// the deeper residency gains.
// Two CTAs per SM for T <= 4; at T > 4 the row loop needs more registers
// than that leaves (spills measured).
template <int D, int T, int MODE>
struct VerifyShape {
  static constexpr int kThreads = 2 * D;
  static constexpr int kMinBlocks = T <= 4 ? 2 : 1;
};

template <int D, int T, int MODE>
__global__ void __launch_bounds__(VerifyShape<D, T, MODE>::kThreads, VerifyShape<D, T, MODE>::kMinBlocks)
    verify_kernel(const VerifyParams p) {
  using G = RowLanes<D>;
  constexpr int RPL = G::RPL, GPW = G::GPW, LPR = G::LPR;
  constexpr int NTHR = VerifyShape<D, T, MODE>::kThreads, NWARP = NTHR / 32;
  constexpr int ROWS_W = D / NWARP;   // state rows per warp, in groups of 8
  constexpr int NGRP = ROWS_W / 8;
  static_assert(ROWS_W % 8 == 0 && NWARP * ROWS_W == D, "rows must split evenly over warps");
  static_assert(NWARP <= 8, "the gated-norm partial sums hold 8 warps");
  constexpr int NT = D / kTileRows;   // 32-row tiles, one bulk copy and barrier each
  // per-head reductions: |q_t|^2, |k_t|^2, k_s.k_t (s<t), k_s.q_t (s<=t)
  constexpr int NKK = T * (T - 1) / 2, NKQ = T * (T + 1) / 2, NV = 2 * T + NKK + NKQ;

  extern __shared__ __align__(128) unsigned char vsm_raw[];
  VerifySmem<D, T> &sm = *reinterpret_cast<VerifySmem<D, T> *>(vsm_raw);

  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  const int H_v = p.H_v, H_k = p.H_k;
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
  const size_t bh = size_t(b) * H_v + h;
  // DEFERRED: this (row, head)'s captures of the previous verify, one bulk
  // copy per region.  Only this CTA writes them (at its end), and the
  // previous verify of the layer finished before the last unflagged call, so
  // they may be fetched before the PDL wait like the state.
  auto stage_state = [&]() {
    if (tid == 0) {
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        mbar_arrive_expect_tx(&sm.bar[i], kTileBytes);
        bulk_g2s(sm.S + i * kTileRows * D, Sg + size_t(i) * kTileRows * D, kTileBytes, &sm.bar[i]);
      }
      if (MODE == GDN_COMMIT_DEFERRED) {
        constexpr uint32_t kCap = T * D * sizeof(float);
        mbar_arrive_expect_tx(&sm.cbar, 2 * kCap + kMaxT * sizeof(float));
        bulk_g2s(&sm.ce[0][0], p.ws_e + bh * T * D, kCap, &sm.cbar);
        bulk_g2s(&sm.ck[0][0], p.ws_k + bh * T * D, kCap, &sm.cbar);
        bulk_g2s(sm.cG, p.ws_G + bh * kMaxT, kMaxT * sizeof(float), &sm.cbar);
      }
    }
  };
  // ---- 1. stage the (row, head) state, 32 rows per bulk copy ----------------
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < NT; ++i) mbar_init(&sm.bar[i], 1);
    mbar_init(&sm.cbar, 1);
    fence_mbar_init();
  }
  if (active) stage_state();
  __syncthreads();  // initialised barriers are visible to every waiter

  // DEFERRED: K = keep' of a commit of this (row, head) not yet applied.
  int K = 0;
  bool pending = false, applied = false;
  auto give_up = [&]() {
    // A staged copy never arrived: flag it, give the copies one more bounded
    // wait so they do not land in a retired CTA's shared memory, and write
    // nothing more.
    if (lane == 0) atomicOr(p.status, GDN_STATUS_TIMEOUT);
#pragma unroll
    for (int i = 0; i < NT; ++i) mbar_wait_bounded(&sm.bar[i], 0);
    if (MODE == GDN_COMMIT_DEFERRED && (active || pending)) mbar_wait_bounded(&sm.cbar, 0);
    if (MODE == GDN_COMMIT_DEFERRED && applied && tid == 0) bulk_wait_read_all();
  };
  const int jw0 = warp * ROWS_W;
  // DEFERRED: S <- gamma S + sum_{s<K} c_s e_s k_s^T on this warp's rows (the
  // arithmetic of the eager RECOMPUTE commit), in place in shared memory;
  // write_back() then stores the tile as the committed state.  Returns false
  // if a staged copy timed out.
  auto apply_pending = [&]() -> bool {
    if (!mbar_wait_bounded(&sm.cbar, 0)) return false;
    const float GK = sm.cG[K - 1];
    const float pc_gam = expf(GK);
    float pc_c[T];
#pragma unroll
    for (int t = 0; t < T; ++t) pc_c[t] = t < K ? expf(GK - sm.cG[t]) : 0.f;
#pragma unroll
    for (int grp8 = 0; grp8 < NGRP; ++grp8) {
      const int jw = jw0 + 8 * grp8;
      if ((grp8 * 8) % kTileRows == 0 && !mbar_wait_bounded(&sm.bar[jw / kTileRows], 0)) return false;
      float4 sv[RPL];
#pragma unroll
      for (int i = 0; i < RPL; ++i) {
        const float4 s0 = *reinterpret_cast<const float4 *>(&sm.S[(jw + grp + GPW * i) * D + 4 * sub]);
        sv[i] = make_float4(pc_gam * s0.x, pc_gam * s0.y, pc_gam * s0.z, pc_gam * s0.w);
      }
#pragma unroll
      for (int t = 0; t < T; ++t) {
        if (t < K) {
          const float4 kv = *reinterpret_cast<const float4 *>(&sm.ck[t][4 * sub]);
          const float *ert = &sm.ce[t][jw];
#pragma unroll
          for (int i = 0; i < RPL; ++i) {
            const float f = pc_c[t] * ert[grp + GPW * i];
            sv[i].x = fmaf(f, kv.x, sv[i].x);
            sv[i].y = fmaf(f, kv.y, sv[i].y);
            sv[i].z = fmaf(f, kv.z, sv[i].z);
            sv[i].w = fmaf(f, kv.w, sv[i].w);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < RPL; ++i) *reinterpret_cast<float4 *>(&sm.S[(jw + grp + GPW * i) * D + 4 * sub]) = sv[i];
    }
    fence_proxy_async_shared();  // the bulk copies of write_back read these rows
    return true;
  };
  // After a barrier that follows every warp's apply: the updated tile goes
  // back to the state buffer on the bulk-copy engine while the warps carry
  // on; the issuing thread waits for the reads of shared memory before it
  // leaves.
  auto write_back = [&]() {
    if (tid == 0) {
      float *Sw = p.state_w + bh * D * D;
#pragma unroll
      for (int i = 0; i < NT; ++i)
        bulk_s2g(Sw + size_t(i) * kTileRows * D, sm.S + i * kTileRows * D, kTileBytes);
      bulk_commit_group();
    }
  };
  // Stage (if the row is inactive), apply, write back and retire a pending
  // commit; CTA-uniform, so its barrier is safe.  False if a copy timed out.
  auto apply_and_write = [&]() -> bool {
    if (!active) stage_state();
    const bool failed = !apply_pending();
    // every warp has applied (or given up) before the write-back and the
    // reset; no thread leaves before this barrier
    if (__syncthreads_or(failed)) return false;
    write_back();
    if (tid == 0) p.ws_pend[bh] = 0;
    applied = true;
    return true;
  };
  // DEFERRED with GDN_VERIFY_OVERLAP: nothing issued since the last call
  // without the flag wrote this layer's workspace (a commit is followed by an
  // unflagged call), so the pending keep is final before the PDL wait and the
  // commit is applied and written back while the preceding kernel still runs.
  // Without the flag it is read after the wait and applied while the conv
  // inputs are in flight.
  if (MODE == GDN_COMMIT_DEFERRED && p.overlap) {
    K = min(p.ws_pend[bh], T);
    pending = K >= 1;
    if (pending && !apply_and_write()) {
      give_up();
      return;
    }
  }
  if (p.overlap) pdl_wait();
  if (MODE == GDN_COMMIT_DEFERRED && !p.overlap) {
    K = min(p.ws_pend[bh], T);
    pending = K >= 1;
  }
  if (!active) {
    // Inactive / padding / finished rows are inert: zero output, no ring
    // access.  A commit still pending from an earlier cycle is applied.
    for (int i = tid; i < T * D; i += NTHR) p.out[((size_t(b) * T + i / D) * H_v + h) * D + i % D] = 0;
    if (MODE == GDN_COMMIT_DEFERRED && pending && !applied && !apply_and_write()) {
      give_up();
      return;
    }
    if (MODE == GDN_COMMIT_DEFERRED && applied && tid == 0) bulk_wait_read_all();
    return;
  }

  const bool qk_writer = (h % rep) == 0;  // one CTA per key head writes its q/k ring slots
  // T >= 4: the per-head scalars are shared through shared memory and q, k
  // are read from it per row group, instead of every lane reducing all
  // T^2 + 2T of them and holding 2T vectors in registers
  constexpr bool kSC = T >= 4;
  float q[T][4], k[T][4], vrow[NGRP][T];
  float gt[T], bt[T];
  {
    // ---- 2. conv + activation: the key head's q and k channels (spread over
    // the CTA) and the v channels of the rows this lane will hold; every load
    // is issued before the first use
    constexpr int NQK = (2 * D + NTHR - 1) / NTHR;
    ConvIn<T> inqk[NQK], inv[NGRP];
#pragma unroll
    for (int r = 0; r < NQK; ++r) {
      const int c2 = tid + r * NTHR;
      if (c2 < 2 * D) conv_load<T>(p, b, (c2 >= D ? H_k * D + c2 - D : c2) + hk * D, inqk[r]);
    }
#pragma unroll
    for (int grp8 = 0; grp8 < NGRP; ++grp8)
      conv_load<T>(p, b, 2 * H_k * D + h * D + jw0 + 8 * grp8 + grp + GPW * istar, inv[grp8]);
#pragma unroll
    for (int t = 0; t < T; ++t) {
      gt[t] = p.g[(size_t(b) * T + t) * H_v + h];
      bt[t] = p.beta[(size_t(b) * T + t) * H_v + h];
    }
    // (DEFERRED: the staged captures are waited for even when nothing is
    // pending, so no copy lands after the CTA has left)
    const bool failed = MODE == GDN_COMMIT_DEFERRED &&
                        (pending && !applied ? !apply_pending() : !mbar_wait_bounded(&sm.cbar, 0));
#pragma unroll
    for (int r = 0; r < NQK; ++r) {
      const int c2 = tid + r * NTHR;
      if (c2 < 2 * D) {
        float y[T];
        conv_eval<T>(inqk[r], p.act, y);
#pragma unroll
        for (int t = 0; t < T; ++t) (c2 >= D ? sm.k : sm.q)[t][c2 >= D ? c2 - D : c2] = y[t];
      }
    }
#pragma unroll
    for (int grp8 = 0; grp8 < NGRP; ++grp8) conv_eval<T>(inv[grp8], p.act, vrow[grp8]);
    // new raw inputs into the ring: q/k channels by one CTA of the key head,
    // v channels by one lane of the four sharing a row
#pragma unroll
    for (int r = 0; r < NQK; ++r) {
      const int c2 = tid + r * NTHR;
      if (qk_writer && c2 < 2 * D) conv_store_ring<T>(p, b, (c2 >= D ? H_k * D + c2 - D : c2) + hk * D, inqk[r]);
    }
    if (leader) {
#pragma unroll
      for (int grp8 = 0; grp8 < NGRP; ++grp8)
        conv_store_ring<T>(p, b, 2 * H_k * D + h * D + jw0 + 8 * grp8 + grp + GPW * istar, inv[grp8]);
    }
    // conv outputs (and applied state rows) are visible; a timed-out staged
    // copy stops the CTA here, where no thread has left yet
    if (__syncthreads_or(failed)) {
      give_up();
      return;
    }
    if (MODE == GDN_COMMIT_DEFERRED && pending && !applied) {
      write_back();
      applied = true;
    }
    if constexpr (!kSC) {
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const float4 qv = *reinterpret_cast<const float4 *>(&sm.q[t][4 * sub]);
        const float4 kv = *reinterpret_cast<const float4 *>(&sm.k[t][4 * sub]);
        q[t][0] = qv.x, q[t][1] = qv.y, q[t][2] = qv.z, q[t][3] = qv.w;
        k[t][0] = kv.x, k[t][1] = kv.y, k[t][2] = kv.z, k[t][3] = kv.w;
      }
    }
  }

  // ---- 3. per-head sums over the LPR lanes of a row group ------------------
  float red_h[NV];
  float inv_q[T], inv_k[T], Gc[T], gam[T];
  float decay[T][T];  // exp(G_t - G_s), s < t
  if constexpr (kSC) {
    // ---- 3'. the T^2 + 2T dot products, four lanes each ----------------------
    // Lane l of quad qd sums float4 columns l, l+4, ... of its pair, starting
    // 4*qd columns in, so the two quads of a quarter-warp read different banks.
    constexpr int NQ4 = NTHR / 4, F4 = D / 4;
    {
      const int qd = tid >> 2, ql = tid & 3;
      for (int r0 = 0; r0 < NV; r0 += NQ4) {  // the same trip count in every lane
        const int n = r0 + qd;
        float part = 0.f;
        if (n < NV) {
          const float *u, *w;
          if (n < 2 * T) {
            u = w = (n & 1) ? sm.k[n >> 1] : sm.q[n >> 1];
          } else if (n < 2 * T + NKK) {  // k_s . k_t, s < t, t-major
            int r = n - 2 * T, t = 1;
            while (r >= t) r -= t, ++t;
            u = sm.k[r], w = sm.k[t];
          } else {                        // k_s . q_t, s <= t, t-major
            int r = n - 2 * T - NKK, t = 0;
            while (r > t) r -= t + 1, ++t;
            u = sm.k[r], w = sm.q[t];
          }
#pragma unroll
          for (int j = 0; j < F4 / 4; ++j) {
            const int f = (ql + 4 * (j + qd)) % F4;
            part += dot4(*reinterpret_cast<const float4 *>(u + 4 * f), *reinterpret_cast<const float4 *>(w + 4 * f));
          }
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (n < NV && ql == 0) sm.hraw[n] = part;
      }
      // cumulative log-decay G_t = g_0 + ... + g_t, in order
      if (tid < T) {
        float a = 0.f;
#pragma unroll
        for (int u = 0; u < T; ++u)
          if (u <= tid) a += gt[u];
        sm.cGc[tid] = a;
      }
    }
    __syncthreads();
    // ---- 4'. coefficients of the recurrence, one thread each -----------------
    const float qs = 1.0f / sqrtf(float(D));
    for (int i = tid; i < T + T * T; i += NTHR) {  // (T + T^2 can exceed the CTA at d = 32)
      if (i < T) {
        const int t = i;
        const float iq = rsqrtf(sm.hraw[2 * t] + kNormEps) * qs, ik = rsqrtf(sm.hraw[2 * t + 1] + kNormEps);
        const float gm = expf(sm.cGc[t]);
        sm.cbk[t] = (bt[t] * gm) * ik;
        sm.cgq[t] = gm * iq;
        sm.cinvk[t] = ik;
        continue;
      }
      const int t = (i - T) / T, s0 = (i - T) % T;
      if (s0 <= t) {
        const float ik_s = rsqrtf(sm.hraw[2 * s0 + 1] + kNormEps), ik_t = rsqrtf(sm.hraw[2 * t + 1] + kNormEps);
        const float iq_t = rsqrtf(sm.hraw[2 * t] + kNormEps) * qs;
        const float dec = s0 == t ? 1.0f : expf(sm.cGc[t] - sm.cGc[s0]);
        if (s0 < t) sm.cA[t][s0] = bt[t] * dec * (sm.hraw[2 * T + t * (t - 1) / 2 + s0] * ik_s * ik_t);
        sm.cQ[t][s0] = dec * (sm.hraw[2 * T + NKK + t * (t + 1) / 2 + s0] * ik_s * iq_t);
      }
    }
    __syncthreads();
  } else {
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

  // ---- 5. this warp's rows, in groups of 8 (the state is already staged,
  // and in DEFERRED mode already brought up to date) -------------------------
  const size_t plane = size_t(p.B) * H_v * D * D;
  const bool gated = p.gz != nullptr;
  {
  float og[NGRP][T];           // gated: o of the rows this lane leads, until the norm is known
  uint16_t zg[NGRP][T], wg[NGRP];
  if (gated && leader) {       // the gate and weight of those rows, loaded now
#pragma unroll
    for (int grp8 = 0; grp8 < NGRP; ++grp8) {
      const int jrow = jw0 + 8 * grp8 + grp + GPW * istar;
      wg[grp8] = p.gw[jrow];
#pragma unroll
      for (int t = 0; t < T; ++t) zg[grp8][t] = p.gz[((size_t(b) * T + t) * H_v + h) * D + jrow];
    }
  }
  bool bad = false;
#pragma unroll
  for (int grp8 = 0; grp8 < NGRP; ++grp8) {
    const int jw = jw0 + 8 * grp8;  // first state row of this group
    const int jrow = jw + grp + GPW * istar;
    if ((grp8 * 8) % kTileRows == 0 && !mbar_wait_bounded(&sm.bar[jw / kTileRows], 0)) {
      bad = true;
      break;
    }
    float4 s[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i)
      s[i] = *reinterpret_cast<const float4 *>(&sm.S[(jw + grp + GPW * i) * D + 4 * sub]);
    float red[2 * T];
#pragma unroll
    for (int mvec = 0; mvec < 2 * T; ++mvec) {
      float4 vec;
      if constexpr (kSC) {
        vec = *reinterpret_cast<const float4 *>(&(mvec < T ? sm.k[mvec] : sm.q[mvec - T])[4 * sub]);
      } else {
        const float *vv = mvec < T ? k[mvec] : q[mvec - T];
        vec = make_float4(vv[0], vv[1], vv[2], vv[3]);
      }
      float acc[RPL];
#pragma unroll
      for (int i = 0; i < RPL; ++i) acc[i] = dot4(s[i], vec);
      red[mvec] = reduce_rows<D>(acc, lane);
    }
    const float *v = vrow[grp8];

    // scalar recurrence for the row this lane holds
    float e[T], o[T];
    if constexpr (kSC) {
#pragma unroll
      for (int t = 0; t < T; ++t) {
        float acc = fmaf(bt[t], v[t], -sm.cbk[t] * red[t]);
#pragma unroll
        for (int s0 = 0; s0 < t; ++s0) acc = fmaf(-sm.cA[t][s0], e[s0], acc);
        e[t] = acc;
        float ot = sm.cgq[t] * red[T + t];
#pragma unroll
        for (int s0 = 0; s0 <= t; ++s0) ot = fmaf(sm.cQ[t][s0], e[s0], ot);
        o[t] = ot;
      }
    } else {
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
        if (gated)
          og[grp8][t] = o[t];
        else
          p.out[((size_t(b) * T + t) * H_v + h) * D + jrow] = f2bf(o[t]);
        if (MODE != GDN_COMMIT_SNAPSHOT) p.ws_e[(bh * T + t) * D + jrow] = e[t];
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
          float4 kh;
          if constexpr (kSC) {
            const float4 kr = *reinterpret_cast<const float4 *>(&sm.k[t][4 * sub]);
            const float ik = sm.cinvk[t];
            kh = make_float4(kr.x * ik, kr.y * ik, kr.z * ik, kr.w * ik);
          } else {
            kh = make_float4(k[t][0] * inv_k[t], k[t][1] * inv_k[t], k[t][2] * inv_k[t], k[t][3] * inv_k[t]);
          }
          st.x = fmaf(et, kh.x, a * st.x);
          st.y = fmaf(et, kh.y, a * st.y);
          st.z = fmaf(et, kh.z, a * st.z);
          st.w = fmaf(et, kh.w, a * st.w);
          st_f4(snap + t * plane + size_t(grp + GPW * i) * D + 4 * sub, st);
        }
      }
    }
  }
  if (gated) {
    // out = o_t / sqrt(mean_j o_t[j]^2 + eps) * w[j] * silu(z_t[j]) over the
    // head's d_v rows, which the CTA's warps share: one more block barrier
    // (reached by every thread; a timed-out warp leaves after it)
    if (__syncthreads_or(bad)) {
      if (bad) give_up();
      return;
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float q2 = 0.f;
      if (leader)
#pragma unroll
        for (int grp8 = 0; grp8 < NGRP; ++grp8) q2 = fmaf(og[grp8][t], og[grp8][t], q2);
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) q2 += __shfl_xor_sync(0xffffffffu, q2, m);
      if (lane == 0) sm.gsq[t][warp] = q2;
    }
    __syncthreads();
    if (leader) {
#pragma unroll
      for (int t = 0; t < T; ++t) {
        float ss = 0.f;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) ss += sm.gsq[t][w];
        const float rstd = rsqrtf(ss / float(D) + p.geps);
#pragma unroll
        for (int grp8 = 0; grp8 < NGRP; ++grp8) {
          const int jrow = jw0 + 8 * grp8 + grp + GPW * istar;
          const float z = bf2f(zg[grp8][t]);
          p.out[((size_t(b) * T + t) * H_v + h) * D + jrow] =
              f2bf(og[grp8][t] * rstd * bf2f(wg[grp8]) * silu_fast(z));
        }
      }
    }
  } else if (bad) {
    give_up();
    return;
  }
  }  // row loop
  // every warp applied its rows before the conv barrier
  if (MODE == GDN_COMMIT_DEFERRED && pending && tid == 0) p.ws_pend[bh] = 0;  // (a repeat if applied before the wait)

  // ---- 6. captures of the key head and decay --------------------------------
  if (MODE != GDN_COMMIT_SNAPSHOT) {
    // k: one copy per key head in RECOMPUTE mode, one per (row, value head)
    // in DEFERRED mode
    const size_t bk = MODE == GDN_COMMIT_DEFERRED ? bh : size_t(b) * H_k + hk;
    if ((MODE == GDN_COMMIT_DEFERRED || qk_writer) && warp == 0 && grp == 0)
#pragma unroll
      for (int t = 0; t < T; ++t) {
        if constexpr (kSC) {
          const float4 kr = *reinterpret_cast<const float4 *>(&sm.k[t][4 * sub]);
          const float ik = sm.cinvk[t];
          st_f4(p.ws_k + (bk * T + t) * D + 4 * sub, make_float4(kr.x * ik, kr.y * ik, kr.z * ik, kr.w * ik));
        } else {
          st_f4(p.ws_k + (bk * T + t) * D + 4 * sub,
                make_float4(k[t][0] * inv_k[t], k[t][1] * inv_k[t], k[t][2] * inv_k[t], k[t][3] * inv_k[t]));
        }
      }
    if (warp == 0 && lane < T) {
#pragma unroll
      for (int t = 0; t < T; ++t)
        if (lane == t) p.ws_G[bh * kMaxT + t] = kSC ? sm.cGc[t] : Gc[t];
    }
  }
  if (MODE == GDN_COMMIT_DEFERRED && applied && tid == 0) bulk_wait_read_all();
}

// Launch one verify instantiation, raising its dynamic shared-memory limit on
// the first launch of that instantiation on each device.
template <int D, int T, int MODE>
cudaError_t launch_verify_kernel(dim3 grid, cudaStream_t stream, const VerifyParams &p) {
  const dim3 block(VerifyShape<D, T, MODE>::kThreads);
  static std::atomic<bool> configured[64];  // one flag set per instantiation
  constexpr int smem = int(sizeof(VerifySmem<D, T>));
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(verify_kernel<D, T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  return launch_pdl_smem(verify_kernel<D, T, MODE>, grid, block, smem, stream, p);
}

// One commit mode, every T.
template <int D, int MODE>
cudaError_t launch_verify_m(const VerifyParams &p, int T, cudaStream_t stream) {
  const dim3 grid(p.H_v, p.B);
  switch (T) {
    case 1: return launch_verify_kernel<D, 1, MODE>(grid, stream, p);
    case 2: return launch_verify_kernel<D, 2, MODE>(grid, stream, p);
    case 3: return launch_verify_kernel<D, 3, MODE>(grid, stream, p);
    case 4: return launch_verify_kernel<D, 4, MODE>(grid, stream, p);
    case 5: return launch_verify_kernel<D, 5, MODE>(grid, stream, p);
    case 6: return launch_verify_kernel<D, 6, MODE>(grid, stream, p);
    case 7: return launch_verify_kernel<D, 7, MODE>(grid, stream, p);
    case 8: return launch_verify_kernel<D, 8, MODE>(grid, stream, p);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
cudaError_t launch_verify_d(const VerifyParams &p, int T, int mode, cudaStream_t stream) {
  if (mode == GDN_COMMIT_RECOMPUTE) return launch_verify_m<D, GDN_COMMIT_RECOMPUTE>(p, T, stream);
  if (mode == GDN_COMMIT_SNAPSHOT) return launch_verify_m<D, GDN_COMMIT_SNAPSHOT>(p, T, stream);
  return launch_verify_m<D, GDN_COMMIT_DEFERRED>(p, T, stream);
}

}  // namespace gdn
