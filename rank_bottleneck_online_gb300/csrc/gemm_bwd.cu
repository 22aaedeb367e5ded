// gemm_bwd.cu -- instantiations of the tensor-core GEMM for the backward path:
// recompute + dgrad with two TMEM accumulators (EPI_DUAL), dgrad of x with the
// RMSNorm-backward epilogue (EPI_DX), wgrad of A with gamma scaling and dgamma
// partials (EPI_DA), and fp32 split-K partials (EPI_F32).
#include "gemm_launch.inc"

namespace boost_gb300 {

cudaError_t launch_gemm_bwd_modes(int bn, int mode, const GemmParams& p, int num_sms,
                                  cudaStream_t stream) {
  if (mode == EPI_DUAL) {
    if (bn == 64) return launch_one<64, EPI_DUAL>(p, num_sms, stream);
    if (bn == 128) return launch_one<128, EPI_DUAL>(p, num_sms, stream);
    if (bn == 256) return launch_one<256, EPI_DUAL>(p, num_sms, stream);
  } else if (mode == EPI_DX) {
    if (bn == 64) return launch_one<64, EPI_DX>(p, num_sms, stream);
    if (bn == 128) return launch_one<128, EPI_DX>(p, num_sms, stream);
    if (bn == 256) return launch_one<256, EPI_DX>(p, num_sms, stream);
  } else if (mode == EPI_DA) {
    if (bn == 64) return launch_one<64, EPI_DA>(p, num_sms, stream);
    if (bn == 128) return launch_one<128, EPI_DA>(p, num_sms, stream);
    if (bn == 256) return launch_one<256, EPI_DA>(p, num_sms, stream);
  } else if (mode == EPI_F32) {
    if (bn == 64) return launch_one<64, EPI_F32>(p, num_sms, stream);
    if (bn == 128) return launch_one<128, EPI_F32>(p, num_sms, stream);
    if (bn == 256) return launch_one<256, EPI_F32>(p, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace boost_gb300
