// gemm_fwd.cu -- instantiations of the tensor-core GEMM for the forward path:
// the grouped down-projection with deferred 1/rms + activation (EPI_ACT) and plain
// bf16 stores (EPI_BF16: batched up-projection, unsplit dB; EPI_BF16T: the same through
// TMA stores), and the gate/up up-projection with the SwiGLU forward in its epilogue
// (EPI_UPGLU).
#include "gemm_launch.inc"

namespace boost_gb300 {

cudaError_t launch_gemm_fwd_modes(int bn, int mode, int cg, int mcm, int mcn, const GemmParams& p,
                                  int num_sms, cudaStream_t stream) {
  if (mode == EPI_ACT) return launch_mode<EPI_ACT>(bn, cg, mcm, mcn, p, num_sms, stream);
  if (mode == EPI_BF16) return launch_mode<EPI_BF16>(bn, cg, mcm, mcn, p, num_sms, stream);
  if (mode == EPI_UPGLU) return launch_mode<EPI_UPGLU>(bn, cg, mcm, mcn, p, num_sms, stream);
  if (mode == EPI_BF16T) return launch_mode<EPI_BF16T>(bn, cg, mcm, mcn, p, num_sms, stream);
  return cudaErrorInvalidValue;
}

int gemm_resident_fwd(int bn, int mode, int cg, int mcm, int mcn, int num_sms) {
  if (mode == EPI_ACT) return resident_mode<EPI_ACT>(bn, cg, mcm, mcn, num_sms);
  if (mode == EPI_BF16) return resident_mode<EPI_BF16>(bn, cg, mcm, mcn, num_sms);
  if (mode == EPI_UPGLU) return resident_mode<EPI_UPGLU>(bn, cg, mcm, mcn, num_sms);
  if (mode == EPI_BF16T) return resident_mode<EPI_BF16T>(bn, cg, mcm, mcn, num_sms);
  return num_sms / cg;
}

}  // namespace boost_gb300
