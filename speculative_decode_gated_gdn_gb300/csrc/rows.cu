// rows.cu -- move per-row decode state between cohorts.
//
// A row primed over its prompt (gdn_prefill_chunked, usually B = 1) joins a
// verify cohort by copying its recurrent state, its conv cache and its
// committed offset into a free row of the cohort, for every layer ("Add
// request-owned eight-way MTP serving for Qwen 35B", sections 2 and 3: rows
// are admitted into the eight-way cohort with their own committed offsets).
// Pure copies: 16-byte loads and stores, units of 64 KiB of one row of one
// layer striding over a grid of CTAs.  Indices are read on the device; a pair
// with a row outside its cohort sets GDN_STATUS_BAD_ROW and is skipped.
#include "gdn_common.cuh"

namespace gdn {

constexpr int kMoveThreads = 256;
constexpr size_t kMoveUnit = 64 * 1024;  // bytes per work unit

__device__ __forceinline__ void copy16(void *dst, const void *src, size_t bytes, size_t off, size_t len) {
  const uint4 *s = reinterpret_cast<const uint4 *>(static_cast<const char *>(src) + off);
  uint4 *d = reinterpret_cast<uint4 *>(static_cast<char *>(dst) + off);
  const size_t n = min(len, bytes - off) / 16;
  for (size_t i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
}

__global__ void __launch_bounds__(kMoveThreads) move_rows_kernel(const MoveParams p) {
  pdl_wait();
  pdl_trigger();
  const size_t s_units = (p.state_bytes + kMoveUnit - 1) / kMoveUnit;
  const size_t r_units = (p.ring_bytes + kMoveUnit - 1) / kMoveUnit;
  const size_t per_pair = s_units + r_units;
  const size_t total = size_t(p.n_layers) * p.n_rows * per_pair;
  for (size_t u = blockIdx.x; u < total; u += gridDim.x) {
    const int layer = int(u / (size_t(p.n_rows) * per_pair));
    const size_t r = u % (size_t(p.n_rows) * per_pair);
    const int i = int(r / per_pair);
    const size_t w = r % per_pair;
    const int sr = p.src_rows[i], dr = p.dst_rows[i];
    if (sr < 0 || sr >= p.src_B || dr < 0 || dr >= p.dst_B) continue;  // flagged below, once
    if (w < s_units) {
      copy16(p.dst_state[layer] + size_t(dr) * p.state_bytes / 4, p.src_state[layer] + size_t(sr) * p.state_bytes / 4,
             p.state_bytes, w * kMoveUnit, kMoveUnit);
    } else {
      const size_t off = (w - s_units) * kMoveUnit;
      copy16(p.dst_ring[layer] + size_t(dr) * p.ring_bytes / 2, p.src_ring[layer] + size_t(sr) * p.ring_bytes / 2,
             p.ring_bytes, off, kMoveUnit);
    }
  }
  // per pair: the offset, the destination's pending DEFERRED keep, the status
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < p.n_rows; i += blockDim.x) {
      const int sr = p.src_rows[i], dr = p.dst_rows[i];
      if (sr < 0 || sr >= p.src_B || dr < 0 || dr >= p.dst_B) {
        atomicOr(p.status, GDN_STATUS_BAD_ROW);
        continue;
      }
      p.dst_offsets[dr] = p.src_offsets[sr];
      if (p.pend_bytes)
        for (int l = 0; l < p.n_layers; ++l)
          for (int hh = 0; hh < p.H_v; ++hh) reinterpret_cast<int *>(p.dst_ws[l])[size_t(dr) * p.H_v + hh] = 0;
    }
  }
}

cudaError_t launch_move_rows(const MoveParams &p, cudaStream_t stream) {
  const size_t s_units = (p.state_bytes + kMoveUnit - 1) / kMoveUnit;
  const size_t r_units = (p.ring_bytes + kMoveUnit - 1) / kMoveUnit;
  long long units = (long long)p.n_layers * p.n_rows * (long long)(s_units + r_units);
  long long grid = units < 1 ? 1 : units;
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (grid > 8LL * sms) grid = 8LL * sms;
  return launch_pdl(move_rows_kernel, dim3(unsigned(grid)), dim3(kMoveThreads), stream, p);
}

}  // namespace gdn
