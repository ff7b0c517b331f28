// verify_d128.cu -- verify kernels for head size 128 (one translation unit per
// head size so the T variants of each compile in parallel).  RECOMPUTE and
// DEFERRED run the tensor-core verify; SNAPSHOT, which writes every
// intermediate state, runs the CUDA-core one.
#include "verify.cuh"
#include "verify_tc.cuh"

namespace gdn {

cudaError_t launch_verify_128(const VerifyParams &p, int T, int mode, cudaStream_t stream) {
  if (mode == GDN_COMMIT_SNAPSHOT) return launch_verify_m<128, GDN_COMMIT_SNAPSHOT>(p, T, stream);
  return launch_verify_tc(p, T, mode, stream);
}

}  // namespace gdn
