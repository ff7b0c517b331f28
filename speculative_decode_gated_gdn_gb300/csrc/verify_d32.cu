// verify_d32.cu -- verify kernels for head size 32 (one translation unit per
// head size so the eight T variants of each compile in parallel).
#include "verify.cuh"

namespace gdn {

cudaError_t launch_verify_32(const VerifyParams &p, int T, int mode, cudaStream_t stream) {
  return launch_verify_d<32>(p, T, mode, stream);
}

}  // namespace gdn
