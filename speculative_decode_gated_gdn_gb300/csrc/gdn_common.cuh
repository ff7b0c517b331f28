// gdn_common.cuh -- shared device helpers and kernel parameter blocks for the
// GB300 GDN speculative-transaction library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kWidth = 4;        // conv width
constexpr int kHist = kWidth - 1; // inputs in the committed conv window
constexpr int kMaxT = 8;         // positions per verify
constexpr int kTileRows = 32;    // state rows (d_v) per verify CTA
constexpr int kVerifyThreads = 128;
constexpr float kNormEps = 1e-6f;

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Conv cache layout: ring slots 0..2 hold the committed window (oldest first),
// slots 3..2+T the raw inputs of the latest verify.
constexpr int kWinSlot = 0;
constexpr int kNewSlot = kHist;

// SiLU with the fast exponential and division intrinsics (a few ulp; the
// conv output feeds an fp32 recurrence whose tolerance is far looser).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Streaming 128-bit load that does not allocate in L1 (each state byte is
// read once per call).
__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Hint: bring the 128-byte line holding p into L2.
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void st_f4(float *p, float4 v) {
  *reinterpret_cast<float4 *>(p) = v;
}

// ---- shared-memory barrier + bulk-copy (TMA) helpers ------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make an initialised mbarrier visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Plain arrival (count 1) of the executing thread.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Contiguous global -> shared copy on the bulk-copy engine; completion is
// counted on `bar` in bytes.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Contiguous shared -> global copy on the bulk-copy engine, tracked as a bulk
// group of the issuing thread.  src, dst 16-byte aligned; bytes a multiple of
// 16.  Writes of the generic proxy to `src` must be fenced with
// fence_proxy_async_shared() and a barrier before the copy is issued.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every bulk group of this thread has finished reading shared
// memory (the global writes complete on their own; kernel completion makes
// them visible).
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` with an iteration limit (about a second in
// total); false if the limit ran out.
constexpr uint32_t kWaitLimit = 1u << 22;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i >= 32) __nanosleep(256);
  }
  return false;
}

// As mbar_wait_bounded, with the iteration limit passed in.
__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i >= 32) __nanosleep(256);
  }
  return false;
}

// As mbar_wait_limit without the sleep between polls, for waits on the
// critical path: each try_wait suspends the thread until the phase completes
// or at most ~1 us passes (its suspend-time hint), so a poll is cheap, the
// wake-up immediate and the whole wait bounded by `limit` polls.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t *bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000u)
        : "memory");
    if (ok) return true;
  }
  return false;
}

// ---- bulk tensor copies (tensor maps) -------------------------------------------
// A tensor map (CUtensorMap) for the bulk tensor copies, encoded on the host
// by cuTensorMapEncodeTiled and passed to kernels as a __grid_constant__
// parameter so that its address is valid for cp.async.bulk.tensor.
struct alignas(64) TmaDesc {
  unsigned long long raw[16];
};

// One 2-D box of `map` at column x, row y into shared memory (complete_tx on
// `bar`); x times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const TmaDesc *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// One 2-D box from shared memory to `map` at column x, row y (x, y >= 0),
// tracked as a bulk group of the issuing thread.
__device__ __forceinline__ void tma_store_2d(const TmaDesc *map, int x, int y, const void *src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}

// ---- programmatic dependent launch --------------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialization.  It waits for the preceding kernel on the stream
// (griddepcontrol.wait) before touching anything that kernel may write, and
// only then lets the next kernel start (launch_dependents), so a kernel's
// pre-wait section can overlap only its immediate predecessor.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename Kernel, typename Params>
inline cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, cudaStream_t stream, const Params &p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// ---- tcgen05 (5th-generation tensor cores, TMEM accumulators) -----------------
// Operand tiles live in shared memory in the K-major no-swizzle canonical
// layout: 8-row x 16-byte core matrices, adjacent along K at `lbo` bytes and
// adjacent 8-row groups at `sbo` bytes.  Descriptor fields: start address,
// leading and stride byte offsets (all >> 4), version 1 at bit 46, no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((saddr >> 4) & 0x3FFF) | (uint64_t((lbo >> 4) & 0x3FFF) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}

// Byte offset of element (row, k) in a K-major no-swizzle canonical tile whose
// K extent is Kd bf16 elements: core matrix (row/8, k/8) at
// (row/8) * (Kd/8)*128 + (k/8) * 128, then row%8 * 16 + k%8 * 2 inside it.
__host__ __device__ constexpr uint32_t canon_off(int row, int k, int Kd) {
  return uint32_t((row / 8) * (Kd / 8) * 128 + (k / 8) * 128 + (row % 8) * 16 + (k % 8) * 2);
}

__device__ __forceinline__ void split_bf16(float y, uint16_t &hi, uint16_t &lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(y);
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(__float2bfloat16_rn(y - __bfloat162float(h)));
}

// Split 8 fp32 values into bf16 hi/lo (x_hi = bf16(x), x_lo = bf16(x - x_hi),
// the same rounding as split_bf16, two values per conversion) and store them
// as two 16-byte runs.
__device__ __forceinline__ void store8_split(const float *v, uint16_t *hi, uint16_t *lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162 hv = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
    h[q] = *reinterpret_cast<const uint32_t *>(&hv);
    if (lo) {
      const __nv_bfloat162 lv = __floats2bfloat162_rn(v[2 * q] - __low2float(hv), v[2 * q + 1] - __high2float(hv));
      l[q] = *reinterpret_cast<const uint32_t *>(&lv);
    }
  }
  *reinterpret_cast<uint4 *>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
  if (lo) *reinterpret_cast<uint4 *>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

// fp32 -> tf32 (round to nearest, ties away from zero), as the 32-bit pattern
// the tensor cores read.
__device__ __forceinline__ uint32_t f2tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// Shared-memory descriptor of a K-major operand stored with the 128-byte
// swizzle (as a bulk tensor copy with that swizzle leaves it): 8-row groups
// of 128-byte rows, 1024 bytes apart; layout type 2 at bits 61-63.  A K step
// inside the 128-byte row advances the start address by its bytes.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  return uint64_t((saddr >> 4) & 0x3FFF) | (uint64_t(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::tf32 (A and B tf32, fp32 accumulator, both
// K-major), shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// D[tmem] (+)= A * B^T for one K step of 8 tf32 elements; issued by one thread.
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(uint32_t(acc))
      : "memory");
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulator,
// both operands K-major, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// D[tmem] (+)= A * B^T for one K step of 16 bf16 elements; issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(uint32_t(acc))
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {  // one full warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // one full warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Warp-collective load of 32 consecutive fp32 columns of the warp's 32 TMEM
// lanes (lane i of the warp gets row 32*(warp%4) + i), then wait for it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Warp-collective load of 16 consecutive fp32 columns of the warp's 32 TMEM
// lanes, then wait for it.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Two warp-collective 16-column loads (any two column offsets), then one
// wait for both: one TMEM round trip instead of two.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float (&va)[16], float (&vb)[16]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
      "[%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) va[i] = __uint_as_float(r[i]), vb[i] = __uint_as_float(r[16 + i]);
}

// Warp-collective store of 32 consecutive fp32 columns of the warp's 32 TMEM
// lanes without waiting for it; tmem_wait_st() completes it.
__device__ __forceinline__ void tmem_st32_async(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
      "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
      "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// An M = 64 accumulator (cta_group::1) holds row r in lane 32 (r / 16) + r % 16:
// the first 16 lanes of each warp's quarter.  The 16x32bx2 shape reads those
// 16 lanes with the whole warp: threads 0-15 get their lane's columns
// [c, c + N), threads 16-31 the same lanes' columns [c + OFF, c + OFF + N).
// Two such 8-column loads (any two base columns), then one wait.
template <int OFF>
__device__ __forceinline__ void tmem_ld_h8x2(uint32_t ta, uint32_t tb, float (&va)[8], float (&vb)[8]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16], %18;\n\t"
      "tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17], %18;\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(ta), "r"(tb), "n"(OFF)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) va[i] = __uint_as_float(r[i]), vb[i] = __uint_as_float(r[8 + i]);
}

// As tmem_ld_h8x2, one load of 16 columns per half.
template <int OFF>
__device__ __forceinline__ void tmem_ld_h16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], %17;\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr), "n"(OFF)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// The mirror store of tmem_ld_h16, without waiting for it (tmem_wait_st()).
template <int OFF>
__device__ __forceinline__ void tmem_st_h16_async(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %17, {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
      "n"(OFF)
      : "memory");
}

// Warp-collective store of 32 consecutive fp32 columns of the warp's 32 TMEM
// lanes (the mirror of tmem_ld32), then wait until the store is done.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
      "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
      "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <typename Kernel, typename Params>
inline cudaError_t launch_pdl_smem(Kernel kernel, dim3 grid, dim3 block, int smem, cudaStream_t stream,
                                   const Params &p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, a.x * b.x)));
}

// Lane geometry of a warp that owns 8 consecutive state rows of head size D:
// LPR lanes share one row (4 floats each), GPW row groups per warp, RPL rows
// per lane.  Lane l holds elements [4*(l % LPR), +4) of rows grp + GPW*i.
template <int D>
struct RowLanes {
  static constexpr int LPR = D / 4;
  static constexpr int GPW = 32 / LPR;
  static constexpr int RPL = 8 / GPW;
  static constexpr int LOG2_RPL = RPL == 8 ? 3 : RPL == 4 ? 2 : RPL == 2 ? 1 : 0;
  static_assert(LPR * GPW == 32 && RPL * GPW == 8, "D must be 32, 64 or 128");
};

// Sum each of the RPL per-lane partials over the LPR lanes sharing a row with
// a reduce-scatter butterfly: after the call the lane holds the full sum of
// row index row_of_lane(lane) (one of its RPL rows), using RPL-1 + log2(LPR/RPL)
// shuffles instead of RPL*log2(LPR).
template <int D>
__device__ __forceinline__ float reduce_rows(float (&a)[RowLanes<D>::RPL], int lane) {
  using G = RowLanes<D>;
#pragma unroll
  for (int step = 0; step < G::LOG2_RPL; ++step) {
    const int m = G::LPR >> (step + 1);
    const bool upper = (lane & m) != 0;
    const int half = G::RPL >> (step + 1);
#pragma unroll
    for (int i = 0; i < G::RPL / 2; ++i) {
      if (i < half) {
        const float send = upper ? a[i] : a[i + half];
        const float keep = upper ? a[i + half] : a[i];
        a[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
      }
    }
  }
  float v = a[0];
#pragma unroll
  for (int m = G::LPR >> (G::LOG2_RPL + 1); m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Which of the lane's RPL rows reduce_rows left in this lane.
template <int D>
__device__ __forceinline__ int row_of_lane(int lane) {
  using G = RowLanes<D>;
  int i = 0;
#pragma unroll
  for (int step = 0; step < G::LOG2_RPL; ++step)
    if (lane & (G::LPR >> (step + 1))) i += G::RPL >> (step + 1);
  return i;
}

// Lane offset (within its LPR-lane row group) that holds row index i after
// reduce_rows: the inverse of row_of_lane.
template <int D>
__device__ __forceinline__ int lane_of_row(int i) {
  using G = RowLanes<D>;
  int off = 0;
#pragma unroll
  for (int step = 0; step < G::LOG2_RPL; ++step)
    if ((i >> (G::LOG2_RPL - 1 - step)) & 1) off += G::LPR >> (step + 1);
  return off;
}

// Per-layer verify parameters.
struct VerifyParams {
  // d = 128 tensor-core verify: the layer's state viewed as a 2-D fp32 array
  // [B * H_v * d_v rows][d_k columns], boxes of 128 rows x 32 columns with the
  // 128-byte swizzle
  TmaDesc tmap_state;
  const uint16_t *x;
  const uint16_t *w;
  const float *g;
  const float *beta;
  const float *state;
  uint16_t *ring;
  const uint8_t *active;
  uint16_t *out;
  // captures of this verify for the commit (RECOMPUTE and DEFERRED)
  float *ws_e;    // [B][H_v][T][D]   e_t of each state row
  float *ws_k;    // [B][H_v][T][D]   normalised k_t of the head's key head
  float *ws_G;    // [B][H_v][kMaxT]  cumulative log-decay G_t
  float *ws_snap; // SNAPSHOT:  [T][B][H_v][D][D]
  // DEFERRED: the captures above still hold the previous verify's until this
  // verify has applied them
  int *ws_pend;         // [B][H_v] keep' of a commit not yet applied (0: none)
  float *state_w;       // DEFERRED: the state, written where a commit is applied
  uint32_t *status; // sticky device status word
  int B, T, H_k, H_v, C, R, act;
  int overlap;      // GDN_VERIFY_OVERLAP: stage the state tile before the PDL wait
  // optional gated RMSNorm of the output: out = o / rms(o) * w * silu(z)
  const uint16_t *gz;  // [B][T][H_v][d_v] bf16 gate, or nullptr (plain o)
  const uint16_t *gw;  // [d_v] bf16 weight
  float geps;
  uint32_t wait_limit;  // iterations of a bounded mbarrier wait (kWaitLimit)
  // tests only (0 in every library call): extra bytes announced on the first
  // state-tile barrier of CTA (row 0, head 0), so that its bounded wait runs out
  uint32_t test_extra_tx;
};

constexpr int kMaxLayers = GDN_MAX_LAYERS;

struct CommitParams {
  float *state[kMaxLayers];
  uint16_t *ring[kMaxLayers];  // nullptr in a flush
  float *ws[kMaxLayers];
  const int32_t *keep;
  const uint8_t *active;
  int32_t *offsets;
  uint32_t *status;
  int n_layers, B, T, H_k, H_v, C, R;
};

// Byte offsets of the capture regions of a verify (each 256-byte aligned):
// e [B][H_v][T][D], normalised k [B][KH][T][D], G [B][H_v][kMaxT].  KH = H_k
// (one copy per key head, written by one CTA of the key head) in RECOMPUTE
// mode; KH = H_v in DEFERRED mode, where every (row, value head) owns its
// copy so that it can fetch its captures before the PDL wait.  A (row, head)'s
// captures are contiguous per region, one bulk copy each.
struct RecomputeWs {
  size_t e, k, G, total;
};

__host__ __device__ inline size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

__host__ __device__ inline RecomputeWs recompute_ws(int B, int T, int KH, int H_v, int D) {
  RecomputeWs w;
  w.e = 0;
  w.k = w.e + align256(sizeof(float) * size_t(B) * H_v * T * D);
  w.G = w.k + align256(sizeof(float) * size_t(B) * KH * T * D);
  w.total = w.G + align256(sizeof(float) * size_t(B) * H_v * kMaxT);
  return w;
}

__host__ __device__ inline size_t snapshot_ws(int B, int T, int H_v, int D) {
  return sizeof(float) * size_t(T) * B * H_v * D * D;
}

// DEFERRED workspace: the pending keep' [B][H_v] of each (row, head) (set by
// the commit, reset to 0 by whichever verify or flush applies it), then the
// captures in the RECOMPUTE layout.
struct DeferredWs {
  size_t pend, cap, total;
};

__host__ __device__ inline DeferredWs deferred_ws(int B, int T, int H_k, int H_v, int D) {
  DeferredWs w;
  w.pend = 0;
  w.cap = w.pend + align256(sizeof(int) * size_t(B) * H_v);
  (void)H_k;
  w.total = w.cap + recompute_ws(B, T, H_v, H_v, D).total;
  return w;
}

// launchers (defined in the .cu files)
cudaError_t launch_verify_32(const VerifyParams &p, int T, int mode, cudaStream_t s);
cudaError_t launch_verify_64(const VerifyParams &p, int T, int mode, cudaStream_t s);
cudaError_t launch_verify_128(const VerifyParams &p, int T, int mode, cudaStream_t s);
cudaError_t launch_commit(const CommitParams &p, int D, int mode, cudaStream_t s);
cudaError_t launch_flush(const CommitParams &p, int D, cudaStream_t s);
size_t prefill_workspace_bytes(int B, int L, int H_k, int H_v, int D);
cudaError_t launch_prefill(const uint16_t *x, const uint16_t *w, const float *g, const float *beta, float *state,
                           uint16_t *ring, int32_t *offsets, uint16_t *out, void *ws, int B, int L, int H_k,
                           int H_v, int D, int R, int act, cudaStream_t stream);
uint32_t *status_word_address();  // device address of the sticky status word
struct MoveParams {
  const float *src_state[kMaxLayers];
  const uint16_t *src_ring[kMaxLayers];
  float *dst_state[kMaxLayers];
  uint16_t *dst_ring[kMaxLayers];
  void *dst_ws[kMaxLayers];     // DEFERRED: pending keep [B][H_v] at the start
  const int32_t *src_offsets;
  int32_t *dst_offsets;
  const int32_t *src_rows, *dst_rows;
  uint32_t *status;
  size_t state_bytes, ring_bytes, pend_bytes;  // per row
  int n_layers, n_rows, src_B, dst_B, H_v;
};
cudaError_t launch_move_rows(const MoveParams &p, cudaStream_t stream);
constexpr int kMaxAcceptT = 64;   // positions per row the acceptance kernel handles
size_t accept_workspace_bytes(int B, int T, int V);
cudaError_t launch_accept(const uint16_t *logits, const int32_t *draft, const uint8_t *active, int32_t *keep,
                          int32_t *next, void *ws, int B, int T, int V, cudaStream_t stream);

}  // namespace gdn
