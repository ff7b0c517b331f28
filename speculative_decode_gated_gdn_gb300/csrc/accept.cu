// accept.cu -- greedy acceptance of one verify cycle, on the device.
//
// "Add request-owned eight-way MTP serving for Qwen 35B" moves the acceptance
// decision of the batched decode cycle off the host, so that a cycle needs no
// host synchronisation.  Position 0 of a row's verify holds the last accepted
// token and positions 1..T-1 the draft tokens.  For an active row b:
//   target_t = argmax_v logits[b][t][v]   (first index of the maximum; NaN
//                                          never wins; an all-NaN row gives 0)
//   keep[b]  = 1 + the number of leading t in 1..T-1 with draft[b][t] == target_{t-1}
//   next[b]  = target_{keep[b]-1}
// Inactive rows get keep 0 and next -1.  keep feeds gdn_commit directly.
//
// One launch.  CTA (c, b*T + t) scans vocabulary slice c of row (b, t) with
// 16-byte loads and writes its best (value, index) to the workspace; the last
// CTA of a row to finish (a per-row atomic count) reduces the slices of every
// position of that row and writes keep and next, then returns the count to 0.
// No CTA waits for another.  The work is one read of the logits: HBM-bound.
#include "gdn_common.cuh"

namespace gdn {

constexpr int kAccThreads = 256;
constexpr int kAccSlice = 8192;  // vocabulary entries per CTA

struct AcceptParams {
  const uint16_t *logits;  // [B][T][V] bf16
  const int32_t *draft;    // [B][T]
  const uint8_t *active;   // [B]
  int32_t *keep, *next;    // [B]
  float *pmax;             // [B][T][NB] best value of each slice
  int32_t *pidx;           // [B][T][NB] its index (-1: the slice had no number)
  uint32_t *count;         // [B] CTAs of the row finished
  int B, T, V, NB;
};

struct AccBest {
  float v;
  int i;  // -1: none
};

// a better than b: a larger value, or an equal value at a smaller index
__device__ __forceinline__ bool acc_better(const AccBest &a, const AccBest &b) {
  if (a.i < 0) return false;
  if (b.i < 0) return true;
  return a.v > b.v || (a.v == b.v && a.i < b.i);
}

__device__ __forceinline__ void acc_take(AccBest &best, float x, int i) {
  if (x == x && (best.i < 0 || x > best.v)) best = AccBest{x, i};  // indices arrive in increasing order
}

__device__ __forceinline__ AccBest acc_warp_reduce(AccBest b) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    AccBest o;
    o.v = __shfl_xor_sync(0xffffffffu, b.v, m);
    o.i = __shfl_xor_sync(0xffffffffu, b.i, m);
    if (acc_better(o, b)) b = o;
  }
  return b;
}

__global__ void __launch_bounds__(kAccThreads) accept_kernel(const AcceptParams p) {
  const int c = blockIdx.x, bt = blockIdx.y;
  const int b = bt / p.T;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ AccBest s_part[kAccThreads / 32];
  __shared__ int s_last;
  __shared__ int s_target[kMaxAcceptT];
  pdl_wait();
  pdl_trigger();
  const bool active = p.active[b] != 0;

  // ---- this CTA's slice of the row --------------------------------------------
  if (active) {
    const int v0 = c * kAccSlice, v1 = min(p.V, v0 + kAccSlice);
    const uint16_t *row = p.logits + size_t(bt) * p.V;
    AccBest best{0.f, -1};
    if ((p.V & 7) == 0) {
      // 8 entries per 16-byte load, all of a thread's loads issued before
      // any comparison; its entries arrive in increasing order
      constexpr int kLoads = kAccSlice / (8 * kAccThreads);
      uint4 q[kLoads];
#pragma unroll
      for (int r = 0; r < kLoads; ++r) {
        const int v = v0 + 8 * (tid + r * kAccThreads);
        q[r] = v < v1 ? *reinterpret_cast<const uint4 *>(row + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int r = 0; r < kLoads; ++r) {
        const int v = v0 + 8 * (tid + r * kAccThreads);
        if (v < v1) {
          const uint32_t w[4] = {q[r].x, q[r].y, q[r].z, q[r].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc_take(best, bf2f(uint16_t(w[j] & 0xffff)), v + 2 * j);
            acc_take(best, bf2f(uint16_t(w[j] >> 16)), v + 2 * j + 1);
          }
        }
      }
    } else {
      for (int v = v0 + tid; v < v1; v += kAccThreads) acc_take(best, bf2f(row[v]), v);
    }
    best = acc_warp_reduce(best);
    if (lane == 0) s_part[warp] = best;
    __syncthreads();
    if (tid == 0) {
      AccBest r = s_part[0];
      for (int w = 1; w < kAccThreads / 32; ++w)
        if (acc_better(s_part[w], r)) r = s_part[w];
      p.pmax[size_t(bt) * p.NB + c] = r.v;
      p.pidx[size_t(bt) * p.NB + c] = r.i;
    }
  }

  // ---- the row's last CTA decides -------------------------------------------
  if (tid == 0) {
    __threadfence();  // this CTA's partial is visible before it is counted
    const uint32_t done = atomicAdd(&p.count[b], 1u) + 1u;
    s_last = done == uint32_t(p.NB) * uint32_t(p.T);
    if (s_last) __threadfence();  // every other CTA's partial is visible from here
  }
  __syncthreads();
  if (!s_last) return;
  if (!active) {
    if (tid == 0) {
      p.keep[b] = 0;
      p.next[b] = -1;
      p.count[b] = 0;
    }
    return;
  }
  // one warp per position: the lanes read the slices' results in parallel
  for (int t = warp; t < p.T; t += kAccThreads / 32) {
    AccBest r{0.f, -1};
    const size_t base = (size_t(b) * p.T + t) * p.NB;
    for (int s = lane; s < p.NB; s += 32) {
      const AccBest o{__ldcg(p.pmax + base + s), __ldcg(p.pidx + base + s)};
      if (acc_better(o, r)) r = o;
    }
    r = acc_warp_reduce(r);
    if (lane == 0) s_target[t] = r.i < 0 ? 0 : r.i;
  }
  __syncthreads();
  if (tid == 0) {
    int k = 1;
    while (k < p.T && p.draft[size_t(b) * p.T + k] == s_target[k - 1]) ++k;
    p.keep[b] = k;
    p.next[b] = s_target[k - 1];
    p.count[b] = 0;  // ready for the next call
  }
}

size_t accept_workspace_bytes(int B, int T, int V) {
  const size_t NB = (size_t(V) + kAccSlice - 1) / kAccSlice;
  const size_t n = size_t(B) * T * NB;
  return align256(n * sizeof(float)) + align256(n * sizeof(int32_t)) + align256(size_t(B) * sizeof(uint32_t));
}

cudaError_t launch_accept(const uint16_t *logits, const int32_t *draft, const uint8_t *active, int32_t *keep,
                          int32_t *next, void *ws, int B, int T, int V, cudaStream_t stream) {
  AcceptParams p{};
  p.logits = logits, p.draft = draft, p.active = active, p.keep = keep, p.next = next;
  p.B = B, p.T = T, p.V = V, p.NB = (V + kAccSlice - 1) / kAccSlice;
  const size_t n = size_t(B) * T * p.NB;
  char *w = static_cast<char *>(ws);
  p.pmax = reinterpret_cast<float *>(w);
  p.pidx = reinterpret_cast<int32_t *>(w + align256(n * sizeof(float)));
  p.count = reinterpret_cast<uint32_t *>(w + align256(n * sizeof(float)) + align256(n * sizeof(int32_t)));
  return launch_pdl(accept_kernel, dim3(p.NB, B * T), dim3(kAccThreads), stream, p);
}

}  // namespace gdn
