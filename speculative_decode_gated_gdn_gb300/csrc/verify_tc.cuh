// verify_tc.cuh -- the d = 128 verify (RECOMPUTE and DEFERRED commits) with
// the state dot products on the tensor cores.
//
// Work decomposition.  One CTA owns one (row b, value head h): warps 0-3
// (128 threads, thread j = state row j, the d_v index) convolve and run the
// recurrence; warp 4 owns the tensor memory and issues the products.  At
// entry one thread stages the head's 64 KiB fp32 state with four bulk tensor
// copies (boxes of 128 rows x 32 columns, 128-byte swizzle), each completing
// on its own mbarrier.  The staged tile is directly the A operand of a
// kind::tf32 tcgen05 product: the 2T dot products of every state row with the
// raw conv outputs k_t, q_t are
//   D[j][n] = sum_i S_0[j][i] B[n][i],   B = [k_0 .. k_{T-1}; q_0 .. q_{T-1}],
// one M = 128, N = 16, K = 128 product (16 MMAs of K = 8) accumulated in
// TMEM, so no thread reduces anything across lanes and no pass converts the
// state.  The tensor cores read the fp32 state truncated to tf32 (and B
// rounded to tf32): about 2^-11 of each term; the products only enter e_t and
// o_t through per-head coefficients, and every state update, conv, norm, gate
// and recurrence step stays in fp32.  (Measured: bf16 products need half the
// instructions, but converting the tile costs the SM more than they save.)
//
// Thread i also convolves channel i of the key head's q and k and of the
// value head's v (so the v channel it convolves is its own state row).  The
// conv taps and the committed window are loaded before the wait on the
// preceding kernel when the call carries GDN_VERIFY_OVERLAP; only x, g and
// beta are read after it.
//
// Arithmetic: the single-chunk WY form of the gated delta rule ("MTP
// inference: review and commit structure", Verification and limits: the
// chunked form equals the sequential one up to rounding).  With
// gamma_t = exp(G_t), G_t = g_0 + ... + g_t:
//   e_t[j] = b_t v_t[j] - b_t gamma_t (S_0[j].k^_t) - sum_{s<t} b_t e^{G_t-G_s} (k^_s.k^_t) e_s[j]
//   o_t[j] = gamma_t (S_0[j].q^_t) + sum_{s<=t} e^{G_t-G_s} (k^_s.q^_t) e_s[j]
// with the L2 norms (and 1/sqrt(d_k)) folded into per-head coefficients.
//
// DEFERRED: a commit the last gdn_commit left pending for this (row, head)
// is applied to the staged tile in shared memory (thread j, row j, the eager
// commit's arithmetic and order) and written back with bulk tensor stores
// before the products read the tile.
#pragma once

#include <atomic>
#include <cstddef>

#include "gdn_common.cuh"

namespace gdn {

constexpr int kVtD = 128;          // head size of this kernel
constexpr int kVtRowThreads = 128; // warps 0-3: one thread per state row
constexpr int kVtThreads = 160;    // + warp 4: tensor memory and the products
constexpr int kVtBoxCols = 32;     // columns per swizzled box (128 bytes of fp32)
constexpr int kVtBoxes = kVtD / kVtBoxCols;
constexpr uint32_t kVtBoxBytes = kVtD * kVtBoxCols * sizeof(float);  // 16 KiB
constexpr int kVtN = 16;           // N of the product: rows 0..2T-1 of B used
constexpr uint32_t kVtTmemCols = 32;

// Per-CTA scalars of the recurrence and the barriers.
template <int T>
struct VtScalars {
  static constexpr int NV = 2 * T + T * (T - 1) / 2 + T * (T + 1) / 2;
  alignas(16) float cG[kMaxT];  // DEFERRED: G of the verify whose commit is pending (one bulk copy)
  // per-warp partial sums of the per-head dot products of the raw conv
  // outputs: |q_t|^2, |k_t|^2, k_s.k_t (s<t), k_s.q_t (s<=t)
  float hpart[kVtRowThreads / 32][NV];
  float cA[T][T];     // beta_t e^{G_t-G_s} (k^_s.k^_t), s < t
  float cQ[T][T];     // e^{G_t-G_s} (k^_s.q^_t), s <= t
  float cbk[T], cgq[T], cinvk[T], cGc[T];
  float gsq[T][kVtRowThreads / 32];
  uint64_t bar[kVtBoxes];  // the four state boxes
  uint64_t cbar;           // DEFERRED captures
  uint64_t bready;         // every row thread has written its B column
  uint64_t mbar;           // products done (never completes if they were not all issued)
  uint64_t fbar;           // products issued before a failed wait have drained
  uint32_t tmem;
};

// Shared memory.  S is the fp32 state tile as the swizzled copies leave it.
// B holds the first 8-row group of the product's B operand (tf32, K-major, no
// swizzle: 8-row x 16-byte core matrices of 4 elements, 128 bytes apart along
// K, 8-row groups 4 KiB apart).  The descriptor's second group (rows 8..15)
// is the memory after B, the DEFERRED k captures (padded to 8 rows when
// 2T > 8): for 2T <= 8 its rows are never read back, and for 2T > 8 rows
// 8..2T-1 are written there once the captures are dead (applied, or waited
// for and unused).  The e captures, which each thread reads only for its own
// row, are staged with the k captures for T <= 4 and come straight from
// global memory above that.  That keeps every T at three CTAs per SM.
template <int T, bool kStaged>
struct VtCe {
  float ce[T][kVtD];  // DEFERRED: e_t of the verify whose commit is pending
};
template <int T>
struct VtCe<T, false> {};

template <int T>
struct VtSmem {
  static constexpr int kCkRows = 2 * T > 8 ? 8 : T;
  static constexpr bool kCeStaged = T <= 4;
  alignas(1024) float S[kVtD * kVtD];
  alignas(1024) uint32_t B[8 * kVtD];
  float ck[kCkRows][kVtD];  // DEFERRED: normalised k_t of the verify whose commit is pending
  VtCe<T, kCeStaged> cep;
  VtScalars<T> sc;
};

// every bulk-copy destination is 16-byte aligned, the tile 1024-byte aligned
template <int T>
constexpr bool vt_layout_ok() {
  // the second 8-row group of B overlays the captures: contiguous, and whole when used
  static_assert(offsetof(VtSmem<T>, ck) == offsetof(VtSmem<T>, B) + 8 * kVtD * 4, "B's second group");
  static_assert(2 * T <= 8 || sizeof(VtSmem<T>::ck) >= 8 * kVtD * 4, "ck covers B's second group");
  static_assert(!VtSmem<T>::kCeStaged || offsetof(VtSmem<T>, cep) % 16 == 0, "ce copy alignment");
  return offsetof(VtSmem<T>, S) % 1024 == 0 && offsetof(VtSmem<T>, B) % 1024 == 0 &&
         offsetof(VtSmem<T>, ck) % 16 == 0 && (offsetof(VtSmem<T>, sc) + offsetof(VtScalars<T>, cG)) % 16 == 0 &&
         (offsetof(VtSmem<T>, sc) + offsetof(VtScalars<T>, bar)) % 8 == 0;
}

template <int T>
constexpr size_t vt_smem_bytes() {
  static_assert(vt_layout_ok<T>(), "shared-memory layout alignment");
  // the descriptors read two 8-row groups of B whatever T is
  constexpr size_t need = offsetof(VtSmem<T>, B) + 2 * 4096;
  return sizeof(VtSmem<T>) > need ? sizeof(VtSmem<T>) : need;
}

// Byte offset of tf32 element (row n, column i) of the B operand (K = 128:
// 8-row groups 4 KiB apart, core matrices of 4 elements 128 bytes apart
// along K, 16 bytes per row of a core matrix).
__device__ __forceinline__ uint32_t vt_canon32(int n, int i) {
  return uint32_t((n / 8) * 4096 + (i / 4) * 128 + (n % 8) * 16 + (i % 4) * 4);
}

// Float index of state element (row j, columns 4u..4u+3 of box c) in the
// swizzled tile: the 16-byte chunk u of a 128-byte row moves to u ^ (j % 8).
__device__ __forceinline__ int vt_s_idx(int c, int j, int u) {
  return c * (kVtD * kVtBoxCols) + j * kVtBoxCols + ((u ^ (j & 7)) << 2);
}

// Conv taps and committed window of one channel (raw bf16 patterns).
struct VtTaps {
  uint2 w;
  uint16_t win[kHist];
};

__device__ __forceinline__ void vt_load_w(const VerifyParams &p, int c, VtTaps &t) {
  t.w = *reinterpret_cast<const uint2 *>(p.w + size_t(c) * kWidth);
}

__device__ __forceinline__ void vt_load_win(const VerifyParams &p, int b, int c, VtTaps &t) {
  const uint16_t *rb = p.ring + size_t(b) * p.R * p.C + c;
#pragma unroll
  for (int i = 0; i < kHist; ++i) t.win[i] = rb[size_t(kWinSlot + i) * p.C];
}

template <int T>
__device__ __forceinline__ void vt_load_x(const VerifyParams &p, int b, int c, uint16_t (&x)[T]) {
  const uint16_t *xb = p.x + size_t(b) * T * p.C + c;
#pragma unroll
  for (int t = 0; t < T; ++t) x[t] = xb[size_t(t) * p.C];
}

// Causal width-4 conv over the T new positions, then the activation (the
// arithmetic of the CUDA-core verify, term for term).
template <int T>
__device__ __forceinline__ void vt_conv(const VtTaps &tp, const uint16_t (&x)[T], int act, float (&y)[T]) {
  const float w0 = bf2f(uint16_t(tp.w.x & 0xffff)), w1 = bf2f(uint16_t(tp.w.x >> 16));
  const float w2 = bf2f(uint16_t(tp.w.y & 0xffff)), w3 = bf2f(uint16_t(tp.w.y >> 16));
  float xt[kHist + T];
#pragma unroll
  for (int i = 0; i < kHist; ++i) xt[i] = bf2f(tp.win[i]);
#pragma unroll
  for (int t = 0; t < T; ++t) xt[kHist + t] = bf2f(x[t]);
#pragma unroll
  for (int t = 0; t < T; ++t) {
    float acc = w0 * xt[t];
    acc = fmaf(w1, xt[t + 1], acc);
    acc = fmaf(w2, xt[t + 2], acc);
    acc = fmaf(w3, xt[t + 3], acc);
    y[t] = act ? silu_fast(acc) : acc;
  }
}

template <int T>
__device__ __forceinline__ void vt_store_ring(const VerifyParams &p, int b, int c, const uint16_t (&x)[T]) {
  uint16_t *rb = p.ring + size_t(b) * p.R * p.C + c;
#pragma unroll
  for (int t = 0; t < T; ++t) rb[size_t(kNewSlot + t) * p.C] = x[t];
}

// The products of one round (r0 .. r0+W-1) of the per-head dot products for
// one channel's conv outputs, in the order n: |q_t|^2, |k_t|^2 (t = 0..T-1,
// interleaved); k_s.k_t (s < t, t-major); k_s.q_t (s <= t, t-major).  Every
// loop is unrolled, so n is a compile-time constant and yq, yk stay in
// registers.
template <int T, int W>
__device__ __forceinline__ void vt_head_round(int r0, const float (&yq)[T], const float (&yk)[T], float (&v)[W]) {
  int n = 0;
#pragma unroll
  for (int t = 0; t < T; ++t) {
    if (n >= r0 && n < r0 + W) v[n - r0] = yq[t] * yq[t];
    ++n;
    if (n >= r0 && n < r0 + W) v[n - r0] = yk[t] * yk[t];
    ++n;
  }
#pragma unroll
  for (int t = 1; t < T; ++t)
#pragma unroll
    for (int s0 = 0; s0 < t; ++s0) {
      if (n >= r0 && n < r0 + W) v[n - r0] = yk[s0] * yk[t];
      ++n;
    }
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int s0 = 0; s0 <= t; ++s0) {
      if (n >= r0 && n < r0 + W) v[n - r0] = yk[s0] * yq[t];
      ++n;
    }
}

// Sums of the per-head products over the warp's 32 channels: rounds of W <= 32
// products, a reduce-scatter butterfly (masks 16, 8, .., 32/W) then plain
// butterfly sums; afterwards lane l holds product r0 + (l >> log2(32/W)),
// and the first lane of each such group writes it to part[].
template <int T>
__device__ __forceinline__ void vt_head_partials(const float (&yq)[T], const float (&yk)[T], int lane, float *part) {
  constexpr int NV = 2 * T + T * (T - 1) / 2 + T * (T + 1) / 2;
  constexpr int W = NV > 16 ? 32 : NV > 8 ? 16 : NV > 4 ? 8 : NV > 2 ? 4 : 2;
  constexpr int SH = W == 32 ? 0 : W == 16 ? 1 : W == 8 ? 2 : W == 4 ? 3 : 4;  // log2(32 / W)
#pragma unroll
  for (int r0 = 0; r0 < NV; r0 += W) {
    float v[W];
#pragma unroll
    for (int m = 0; m < W; ++m) v[m] = 0.f;
    vt_head_round<T, W>(r0, yq, yk, v);
#pragma unroll
    for (int half = W / 2, mask = 16; half >= 1; half >>= 1, mask >>= 1) {
      const bool upper = (lane & mask) != 0;
#pragma unroll
      for (int m = 0; m < half; ++m) {
        const float send = upper ? v[m] : v[m + half];
        const float keep = upper ? v[m + half] : v[m];
        v[m] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
      }
    }
    float x = v[0];
#pragma unroll
    for (int mask = (1 << SH) >> 1; mask >= 1; mask >>= 1) x += __shfl_xor_sync(0xffffffffu, x, mask);
    const int n = r0 + (lane >> SH);
    if ((lane & ((1 << SH) - 1)) == 0 && n < NV) part[n] = x;
  }
}

template <int T, int MODE>
__global__ void __launch_bounds__(kVtThreads, 3)
    verify_tc_kernel(const __grid_constant__ VerifyParams p) {
  constexpr int D = kVtD, NROW = kVtRowThreads;
  constexpr int NKK = T * (T - 1) / 2;
  constexpr bool kDef = MODE == GDN_COMMIT_DEFERRED;
  static_assert(2 * T <= kVtN, "the product holds 2T <= 16 vectors");
  static_assert(NROW == D, "one row thread per state row");
  extern __shared__ __align__(1024) unsigned char tsm_raw[];
  VtSmem<T> &sm = *reinterpret_cast<VtSmem<T> *>(tsm_raw);
  VtScalars<T> &sc = sm.sc;

  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool row = tid < NROW;           // warps 0-3: conv channel i = state row j = tid
  const bool issuer = warp == NROW / 32;  // warp 4
  const int H_v = p.H_v, H_k = p.H_k;
  const int hk = h / (H_v / H_k);
  const size_t bh = size_t(b) * H_v + h;
  const int row0 = int(bh) * D;  // first row of this tile in the state map
  const uint32_t wl = p.wait_limit;
  const bool gated = p.gz != nullptr;

  // With GDN_VERIFY_OVERLAP (level 1) the next kernel may start at once and
  // this one stages its state (and reads its taps, window and pending keep)
  // before waiting for the preceding kernel.  Without it the next kernel
  // starts only after this one's wait, so a chain of level-1 calls can never
  // run ahead of the last call below level 1 (whose own reads of the pending
  // keep and the window may not run ahead of the preceding commit); at level
  // 2 (GDN_VERIFY_OVERLAP_STATE) this one still stages its state before its
  // wait, and lets the next kernel start right after it.
  if (p.overlap == 1) {
    pdl_trigger();
  } else if (p.overlap == 0) {
    pdl_wait();
    pdl_trigger();
  }
  // the swizzled copies and the products need a 1024-byte aligned tile; a
  // misaligned window (never seen) is reported, not used
  if (smem_u32(tsm_raw) & 1023u) {
    if (tid == 0) atomicOr(p.status, GDN_STATUS_TIMEOUT);
    return;
  }
  const bool active = p.active[b] != 0;
  // Tensor memory (active rows): taken at once by warp 4, before the wait
  // when the call is flagged.  Allocating gives up the allocation permit, and
  // an SM admits one CTA still holding the permit of a kernel that allocates
  // tensor memory, so this is what lets further CTAs of this and the next
  // layer start beside a waiting one.  The 32 columns cannot starve the
  // preceding kernel: at most three verify CTAs fit on an SM (96 of 512
  // columns), and the library's prefill kernels, the only others that take
  // tensor memory, need more shared memory than can sit beside a verify CTA.
  // An unflagged call has already waited, whatever the preceding kernel is.
  if (active && issuer) tmem_alloc(&sc.tmem, kVtTmemCols);
  if (tid == 0) {
#pragma unroll
    for (int c = 0; c < kVtBoxes; ++c) mbar_init(&sc.bar[c], 1);
    mbar_init(&sc.cbar, 1);
    mbar_init(&sc.bready, NROW);
    mbar_init(&sc.mbar, 1);
    mbar_init(&sc.fbar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();  // initialised barriers and the TMEM address are visible
  tc_fence_after();

  // Overlap level: 0 none; 1 (GDN_VERIFY_OVERLAP) state, captures, taps,
  // window, active and pending keep before the wait; 2
  // (GDN_VERIFY_OVERLAP_STATE) state, captures, taps and active before it,
  // the pending keep and the window after it.
  const int ov = p.overlap;
  // DEFERRED: K = keep' of a commit of this (row, head) not yet applied.  It
  // is final before the wait at level 1 (a commit is followed by a call
  // without that flag), otherwise read after it.
  int K = 0;
  bool applied = false;
  if (kDef && ov == 1) K = min(p.ws_pend[bh], T);
  bool staged = false, cap_staged = false;
  auto stage = [&](bool captures) {
    staged = true;
    cap_staged = captures;
    if (tid == 0) {
      const uint32_t extra = (b == 0 && h == 0) ? p.test_extra_tx : 0u;
#pragma unroll
      for (int c = 0; c < kVtBoxes; ++c) {
        mbar_arrive_expect_tx(&sc.bar[c], kVtBoxBytes + (c == 0 ? extra : 0u));
        tma_load_2d(&sm.S[c * D * kVtBoxCols], &p.tmap_state, c * kVtBoxCols, row0, &sc.bar[c]);
      }
      if (captures) {
        constexpr uint32_t kCap = T * D * sizeof(float);
        constexpr bool kCe = VtSmem<T>::kCeStaged;
        mbar_arrive_expect_tx(&sc.cbar, (kCe ? 2 : 1) * kCap + kMaxT * sizeof(float));
        if constexpr (kCe) bulk_g2s(&sm.cep.ce[0][0], p.ws_e + bh * T * D, kCap, &sc.cbar);
        bulk_g2s(&sm.ck[0][0], p.ws_k + bh * T * D, kCap, &sc.cbar);
        bulk_g2s(sc.cG, p.ws_G + bh * kMaxT, kMaxT * sizeof(float), &sc.cbar);
      }
    }
  };
  // A bounded wait ran out: flag it, wait (bounded) for every copy this CTA
  // issued so none lands after it has left, and write nothing more.
  auto give_up = [&]() {
    if (tid == 0) {
      atomicOr(p.status, GDN_STATUS_TIMEOUT);
      if (staged) {
#pragma unroll
        for (int c = 0; c < kVtBoxes; ++c) mbar_wait_limit(&sc.bar[c], 0, wl);
        if (cap_staged) mbar_wait_limit(&sc.cbar, 0, wl);
      }
      if (applied) bulk_wait_read_all();
    }
  };
  // DEFERRED: S <- gamma_{K-1} S + sum_{s<K} e^{G_{K-1}-G_s} e_s k^_s^T on row
  // j = tid of the staged tile (the eager commit's arithmetic and order), then
  // the updated tile goes back to the state buffer on the bulk-copy engine.
  // Reached by every thread of the CTA (its barrier); false on a timeout.
  auto apply_and_write = [&]() -> bool {
    bool ok = true;
    if (row) {
      // this row's e_t: staged with the k captures, or (T > 4) straight from
      // the workspace, in flight while the k captures land
      const int j = tid;
      float ej[T];
      if constexpr (!VtSmem<T>::kCeStaged) {
#pragma unroll
        for (int t = 0; t < T; ++t) ej[t] = t < K ? p.ws_e[(bh * T + t) * D + j] : 0.f;
      }
      ok = mbar_wait_limit(&sc.cbar, 0, wl);
      if constexpr (VtSmem<T>::kCeStaged) {
#pragma unroll
        for (int t = 0; t < T; ++t) ej[t] = sm.cep.ce[t][j];
      }
      if (ok) {
        const float GK = sc.cG[K - 1];
        const float gam = expf(GK);
        float f[T];
#pragma unroll
        for (int t = 0; t < T; ++t) f[t] = t < K ? expf(GK - sc.cG[t]) * ej[t] : 0.f;
        // drafts past T = 2 roll the box and chunk loops (the token loop stays
        // unrolled, so the arithmetic and its order are unchanged): the fully
        // unrolled body grows with T and costs instruction fetch
        constexpr int kApplyUnroll = T >= 3 ? 1 : kVtBoxCols / 4, kApplyUnrollBoxes = T >= 3 ? 1 : kVtBoxes;
#pragma unroll kApplyUnrollBoxes
        for (int c = 0; c < kVtBoxes; ++c) {
          if (!mbar_wait_limit(&sc.bar[c], 0, wl)) {
            ok = false;
            break;
          }
#pragma unroll kApplyUnroll
          for (int u = 0; u < kVtBoxCols / 4; ++u) {
            float4 *sp = reinterpret_cast<float4 *>(&sm.S[vt_s_idx(c, j, u)]);
            float4 s4 = *sp;
            s4 = make_float4(gam * s4.x, gam * s4.y, gam * s4.z, gam * s4.w);
#pragma unroll
            for (int t = 0; t < T; ++t) {
              if (t < K) {
                const float4 kv = *reinterpret_cast<const float4 *>(&sm.ck[t][c * kVtBoxCols + 4 * u]);
                s4.x = fmaf(f[t], kv.x, s4.x);
                s4.y = fmaf(f[t], kv.y, s4.y);
                s4.z = fmaf(f[t], kv.z, s4.z);
                s4.w = fmaf(f[t], kv.w, s4.w);
              }
            }
            *sp = s4;
          }
        }
      }
      fence_proxy_async_shared();  // the bulk stores below read these rows
    }
    if (__syncthreads_or(!ok)) return false;
    if (tid == 0) {
#pragma unroll
      for (int c = 0; c < kVtBoxes; ++c) tma_store_2d(&p.tmap_state, c * kVtBoxCols, row0, &sm.S[c * D * kVtBoxCols]);
      bulk_commit_group();
      p.ws_pend[bh] = 0;
    }
    applied = true;
    return true;
  };

  // ---- inactive rows: no ring access and no output of their own (the CTA of
  // an active row zero-fills them after its wait, so these CTAs do not hold a
  // slot while the preceding kernel runs); a pending commit is applied, before
  // the wait when the call is flagged, like the state staging
  if (!active) {
    if (kDef && ov != 1) {
      if (ov == 2) {  // the pending keep may be written by the preceding kernel
        pdl_wait();
        pdl_trigger();
      }
      K = min(p.ws_pend[bh], T);
    }
    if (kDef && K >= 1) {
      stage(true);
      if (!apply_and_write()) {
        give_up();
        return;
      }
    }
    if (b == 0) {  // no active row at all: row 0's CTA zero-fills every row of head h
      bool any = false;
      for (int r = tid; r < p.B; r += kVtThreads) any |= p.active[r] != 0;
      if (!__syncthreads_or(any)) {
        if (ov) pdl_wait();
        if (row)
          for (int r = 0; r < p.B; ++r)
#pragma unroll
            for (int t = 0; t < T; ++t) p.out[((size_t(r) * T + t) * H_v + h) * D + tid] = 0;
      }
    }
    if (applied && tid == 0) bulk_wait_read_all();
    return;
  }

  // the inactive rows this CTA zero-fills: those after b up to the next
  // active row (rows b+1 .. r_hi-1) and, when no row below b is active
  // (r_lo < 0), every row below b; a chain of dependent loads, so a flagged
  // call finds them before its wait
  int r_hi = b + 1, r_lo = b - 1;
  auto find_inactive_neighbours = [&]() {
    while (r_hi < p.B && !p.active[r_hi]) ++r_hi;
    while (r_lo >= 0 && !p.active[r_lo]) --r_lo;
  };
  const int i = tid;  // conv channel i of q, k, v; state row i
  const int cq = hk * D + i, ck = H_k * D + hk * D + i, cv = 2 * H_k * D + h * D + i;
  VtTaps tq, tk, tv;
  if (ov) {
    // flagged: state, captures, taps (and at level 1 the window) before the
    // wait; at level 1 a pending commit is applied and written back while the
    // preceding kernel runs.  At level 2 the pending keep is not known yet, so
    // the captures are fetched whether or not a commit is pending.
    stage(kDef && (ov == 2 || K >= 1));
    if (row) {
      vt_load_w(p, cq, tq);
      vt_load_w(p, ck, tk);
      vt_load_w(p, cv, tv);
      if (ov == 1) {
        vt_load_win(p, b, cq, tq);
        vt_load_win(p, b, ck, tk);
        vt_load_win(p, b, cv, tv);
      }
      // warm L2 with this call's x, g and beta lines (a prefetch only: the
      // values are read after the wait, so a later write by the preceding
      // kernel is still what they see)
      if (tid < 6 * T) {
        const int t = tid / 6, r = tid % 6;  // slabs q, k, v of 128 channels (two 128-byte lines each)
        const int c0 = (r < 2 ? hk * D : r < 4 ? H_k * D + hk * D : 2 * H_k * D + h * D) + (r & 1) * 64;
        prefetch_l2(p.x + (size_t(b) * T + t) * p.C + c0);
      } else if (tid < 8 * T) {
        const int t = (tid - 6 * T) >> 1;
        prefetch_l2(((tid & 1) ? p.beta : p.g) + (size_t(b) * T + t) * H_v + h);
      }
      find_inactive_neighbours();
    }
    if (ov == 1 && kDef && K >= 1 && !apply_and_write()) {
      if (issuer) tmem_dealloc(sc.tmem, kVtTmemCols);
      give_up();
      return;
    }
    pdl_wait();
    if (ov == 2) {
      pdl_trigger();
      if (kDef) K = min(p.ws_pend[bh], T);
      if (row) {
        vt_load_win(p, b, cq, tq);
        vt_load_win(p, b, ck, tk);
        vt_load_win(p, b, cv, tv);
      }
    }
  } else {
    if (kDef) K = min(p.ws_pend[bh], T);
    stage(kDef && K >= 1);
    if (row) {
      vt_load_w(p, cq, tq);
      vt_load_w(p, ck, tk);
      vt_load_w(p, cv, tv);
      vt_load_win(p, b, cq, tq);
      vt_load_win(p, b, ck, tk);
      vt_load_win(p, b, cv, tv);
    }
  }

  // ---- conv inputs of this call ------------------------------------------------
  uint16_t xq[T], xk[T], xv[T];
  float gt[T], bt[T];
  if (row) {
    vt_load_x<T>(p, b, cq, xq);
    vt_load_x<T>(p, b, ck, xk);
    vt_load_x<T>(p, b, cv, xv);
#pragma unroll
    for (int t = 0; t < T; ++t) {
      gt[t] = p.g[(size_t(b) * T + t) * H_v + h];
      bt[t] = p.beta[(size_t(b) * T + t) * H_v + h];
    }
    // zero-fill of the inactive rows found above
    if (!ov) find_inactive_neighbours();
    for (int r = b + 1; r < r_hi; ++r)
#pragma unroll
      for (int t = 0; t < T; ++t) p.out[((size_t(r) * T + t) * H_v + h) * D + tid] = 0;
    if (r_lo < 0)
      for (int r = 0; r < b; ++r)
#pragma unroll
        for (int t = 0; t < T; ++t) p.out[((size_t(r) * T + t) * H_v + h) * D + tid] = 0;
  }
  // DEFERRED below level 1: the pending commit is applied while the inputs load
  if (ov != 1 && kDef && K >= 1 && !apply_and_write()) {
    if (issuer) tmem_dealloc(sc.tmem, kVtTmemCols);
    give_up();
    return;
  }

  if (issuer) {
    // ---- warp 4: the products D[j][n] = S_0[j] . B[n], as soon as every row
    // thread has written its B column; then, once every row thread has read
    // its accumulators, the tensor memory goes back --------------------------
    const uint32_t tmem = sc.tmem;
    if (lane == 0) {
      const uint32_t sB = smem_u32(sm.B);
      // tf32 straight from the swizzled fp32 tile, box by box as it lands
      bool ok = mbar_wait_spin(&sc.bready, 0, wl);
      constexpr uint32_t idesc = umma_idesc_tf32(D, kVtN);
      const uint32_t sS = smem_u32(sm.S);
      int issued = 0;
#pragma unroll
      for (int c = 0; c < kVtBoxes; ++c) {
        if (!ok || !mbar_wait_limit(&sc.bar[c], 0, wl)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kVtBoxCols / 8; ++kk) {
          const int ks = c * (kVtBoxCols / 8) + kk;  // K step of 8 columns
          umma_tf32(tmem, umma_desc_sw128(sS + c * kVtBoxBytes + kk * 32), umma_desc(sB + ks * 256, 128, 4096),
                    idesc, ks > 0);
          ++issued;
        }
      }
      if (ok) {
        umma_commit(&sc.mbar);
      } else if (issued) {  // products in flight finish before the columns go back
        umma_commit(&sc.fbar);
        mbar_wait_limit(&sc.fbar, 0, wl);
      }
    }
    __syncwarp();
    asm volatile("bar.sync 2, %0;" ::"n"(kVtThreads) : "memory");  // the row threads' TMEM reads are done
    tc_fence_after();
    tmem_dealloc(tmem, kVtTmemCols);
    if (applied && tid == 0) bulk_wait_read_all();
    return;
  }

  // ---- warps 0-3: conv, B column, head partial sums, ring -----------------------
  float yq[T], yk[T], yv[T];
  vt_conv<T>(tq, xq, p.act, yq);
  vt_conv<T>(tk, xk, p.act, yk);
  vt_conv<T>(tv, xv, p.act, yv);
  // new raw inputs into ring slots 3..2+T: q/k channels by one CTA of the key
  // head.  Past T = 2 they go out at once, so that the raw inputs are dead
  // before the per-head sums (whose butterfly then fits the register budget);
  // at T <= 2 after the sums, which measured slightly faster there.
  constexpr bool kRingEarly = T >= 3;
  auto store_ring = [&]() {
    if (h % (H_v / H_k) == 0) {
      vt_store_ring<T>(p, b, cq, xq);
      vt_store_ring<T>(p, b, ck, xk);
    }
    vt_store_ring<T>(p, b, cv, xv);
  };
  if constexpr (kRingEarly) store_ring();
  // B rows 8..2T-1 overlay the capture arrays: when captures were staged
  // but no commit applied them (level 2 with nothing pending), their copies
  // must have landed before these writes
  bool cap_late = false;
  if constexpr (2 * T > 8) {
    if (cap_staged && !applied) cap_late = !mbar_wait_limit(&sc.cbar, 0, wl);
  }
  unsigned char *bsm = reinterpret_cast<unsigned char *>(&sm) + offsetof(VtSmem<T>, B);
#pragma unroll
  for (int t = 0; t < T; ++t) {
    *reinterpret_cast<uint32_t *>(bsm + vt_canon32(t, i)) = f2tf32(yk[t]);
    *reinterpret_cast<uint32_t *>(bsm + vt_canon32(T + t, i)) = f2tf32(yq[t]);
  }
  fence_async_smem();  // B is read by the tensor cores
  mbar_arrive(&sc.bready);
  // the per-head dot products as each warp's partial sums
  vt_head_partials<T>(yq, yk, lane, sc.hpart[warp]);
  if constexpr (!kRingEarly) store_ring();
  asm volatile("bar.sync 1, %0;" ::"n"(NROW) : "memory");  // the partial sums are visible

  // ---- coefficients of the recurrence, one thread each --------------------------
  {
    // the head sums (the four warps' partials, in warp order) and the
    // cumulative log-decays G_t = g_0 + ... + g_t (in order)
    auto H = [&](int n) { return ((sc.hpart[0][n] + sc.hpart[1][n]) + sc.hpart[2][n]) + sc.hpart[3][n]; };
    auto Gcum = [&](int t) {
      float a = 0.f;
#pragma unroll
      for (int u = 0; u < T; ++u)
        if (u <= t) a += gt[u];
      return a;
    };
    auto beta_of = [&](int t) {  // bt[t] for a run-time t, kept in registers
      float r = 0.f;
#pragma unroll
      for (int u = 0; u < T; ++u)
        if (u == t) r = bt[u];
      return r;
    };
    const float qs = 1.0f / sqrtf(float(D));
    for (int n = tid; n < T + T * T; n += NROW) {
      if (n < T) {
        const int t = n;
        const float iq = rsqrtf(H(2 * t) + kNormEps) * qs, ik = rsqrtf(H(2 * t + 1) + kNormEps);
        const float Gt = Gcum(t);
        const float gm = expf(Gt);
        sc.cbk[t] = (beta_of(t) * gm) * ik;
        sc.cgq[t] = gm * iq;
        sc.cinvk[t] = ik;
        sc.cGc[t] = Gt;
        continue;
      }
      const int t = (n - T) / T, s0 = (n - T) % T;
      if (s0 <= t) {
        const float ik_s = rsqrtf(H(2 * s0 + 1) + kNormEps), ik_t = rsqrtf(H(2 * t + 1) + kNormEps);
        const float iq_t = rsqrtf(H(2 * t) + kNormEps) * qs;
        const float dec = s0 == t ? 1.0f : expf(Gcum(t) - Gcum(s0));
        if (s0 < t) sc.cA[t][s0] = beta_of(t) * dec * (H(2 * T + t * (t - 1) / 2 + s0) * ik_s * ik_t);
        sc.cQ[t][s0] = dec * (H(2 * T + NKK + t * (t + 1) / 2 + s0) * ik_s * iq_t);
      }
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(NROW) : "memory");  // the coefficients are visible

  // ---- row j = tid: its 2T products from TMEM lane j, then the recurrence ------
  const int j = tid;
  uint16_t zt[T], wj = 0;
  if (gated) {
    wj = p.gw[j];
#pragma unroll
    for (int t = 0; t < T; ++t) zt[t] = p.gz[((size_t(b) * T + t) * H_v + h) * D + j];
  }
  // (the products barrier completes only when all products were issued)
  const bool late = !mbar_wait_spin(&sc.mbar, 0, wl);
  tc_fence_after();
  float red[kVtN];
  if (!late) tmem_ld16(sc.tmem + (uint32_t(32 * warp) << 16), red);
  tc_fence_before();
  asm volatile("bar.arrive 2, %0;" ::"n"(kVtThreads) : "memory");  // this thread's TMEM reads are done
  float o[T], e[T];
  if (!late) {
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float acc = fmaf(bt[t], yv[t], -sc.cbk[t] * red[t]);
#pragma unroll
      for (int s0 = 0; s0 < t; ++s0) acc = fmaf(-sc.cA[t][s0], e[s0], acc);
      e[t] = acc;
      float ot = sc.cgq[t] * red[T + t];
#pragma unroll
      for (int s0 = 0; s0 <= t; ++s0) ot = fmaf(sc.cQ[t][s0], e[s0], ot);
      o[t] = ot;
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
      if (!gated) p.out[((size_t(b) * T + t) * H_v + h) * D + j] = f2bf(o[t]);
      p.ws_e[(bh * T + t) * D + j] = e[t];
    }
    // captures of the key head: normalised k (one copy per key head in
    // RECOMPUTE mode, per (row, value head) in DEFERRED mode) and G
    const size_t bk = kDef ? bh : size_t(b) * H_k + hk;
    if (kDef || h % (H_v / H_k) == 0) {
#pragma unroll
      for (int t = 0; t < T; ++t) p.ws_k[(bk * T + t) * D + i] = yk[t] * sc.cinvk[t];
    }
    if (tid < T) p.ws_G[bh * kMaxT + tid] = sc.cGc[tid];
  }
  if (gated) {
    // out = o_t / sqrt(mean_j o_t[j]^2 + eps) * w[j] * silu(z_t[j]) over the
    // head's rows, which the four row warps share
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float q2 = late ? 0.f : o[t] * o[t];
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) q2 += __shfl_xor_sync(0xffffffffu, q2, m);
      if (lane == 0) sc.gsq[t][warp] = q2;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NROW) : "memory");
    if (!late) {
#pragma unroll
      for (int t = 0; t < T; ++t) {
        float ss = 0.f;
#pragma unroll
        for (int w = 0; w < NROW / 32; ++w) ss += sc.gsq[t][w];
        const float rstd = rsqrtf(ss / float(D) + p.geps);
        p.out[((size_t(b) * T + t) * H_v + h) * D + j] = f2bf(o[t] * rstd * bf2f(wj) * silu_fast(bf2f(zt[t])));
      }
    }
  }
  if (late || cap_late) give_up();  // (thread 0 flags it and drains the copies)
  else if (applied && tid == 0) bulk_wait_read_all();
}

// Launch one instantiation, raising its dynamic shared-memory limit once per
// device.
template <int T, int MODE>
cudaError_t launch_verify_tc_kernel(const VerifyParams &p, cudaStream_t stream) {
  constexpr int smem = int(vt_smem_bytes<T>());
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(verify_tc_kernel<T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // the whole unified L1 / shared array as shared memory: three CTAs per SM
    // (a layer and most of the next one resident together)
    e = cudaFuncSetAttribute(verify_tc_kernel<T, MODE>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             int(cudaSharedmemCarveoutMaxShared));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  return launch_pdl_smem(verify_tc_kernel<T, MODE>, dim3(p.H_v, p.B), dim3(kVtThreads), smem, stream, p);
}

inline cudaError_t launch_verify_tc(const VerifyParams &p, int T, int mode, cudaStream_t stream) {
#define GDN_VERIFY_TC_CASE(TT)                                                             \
  case TT:                                                                                 \
    return mode == GDN_COMMIT_RECOMPUTE ? launch_verify_tc_kernel<TT, GDN_COMMIT_RECOMPUTE>(p, stream) \
                                        : launch_verify_tc_kernel<TT, GDN_COMMIT_DEFERRED>(p, stream);
  switch (T) {
    GDN_VERIFY_TC_CASE(1)
    GDN_VERIFY_TC_CASE(2)
    GDN_VERIFY_TC_CASE(3)
    GDN_VERIFY_TC_CASE(4)
    GDN_VERIFY_TC_CASE(5)
    GDN_VERIFY_TC_CASE(6)
    GDN_VERIFY_TC_CASE(7)
    GDN_VERIFY_TC_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef GDN_VERIFY_TC_CASE
}

}  // namespace gdn
