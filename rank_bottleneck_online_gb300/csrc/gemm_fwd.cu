// gemm_fwd.cu -- instantiations of the tensor-core GEMM for the forward path:
// the grouped down-projection with deferred 1/rms + activation (EPI_ACT) and plain
// bf16 stores (EPI_BF16: batched up-projection, unsplit dB).
#include "gemm_launch.inc"

namespace boost_gb300 {

cudaError_t launch_gemm_fwd_modes(int bn, int mode, const GemmParams& p, int num_sms,
                                  cudaStream_t stream) {
  if (mode == EPI_ACT) {
    if (bn == 64) return launch_one<64, EPI_ACT>(p, num_sms, stream);
    if (bn == 128) return launch_one<128, EPI_ACT>(p, num_sms, stream);
    if (bn == 256) return launch_one<256, EPI_ACT>(p, num_sms, stream);
  } else if (mode == EPI_BF16) {
    if (bn == 64) return launch_one<64, EPI_BF16>(p, num_sms, stream);
    if (bn == 128) return launch_one<128, EPI_BF16>(p, num_sms, stream);
    if (bn == 256) return launch_one<256, EPI_BF16>(p, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace boost_gb300
