// gemm_bwd.cu -- instantiations of the tensor-core GEMM for the backward path:
// recompute + dgrad with two TMEM accumulators (EPI_DUAL; EPI_DUALT stores through TMA),
// dgrad of x with the RMSNorm-backward epilogue (EPI_DX), wgrad of A with gamma scaling
// and dgamma partials (EPI_DA), fp32 split-K partials (EPI_F32), and the
// down-projection's dgrad with the SwiGLU backward in its epilogue (EPI_GLU).
#include "gemm_launch.inc"

namespace boost_gb300 {

cudaError_t launch_gemm_bwd_modes(int bn, int mode, int cg, int mcm, int mcn, const GemmParams& p,
                                  int num_sms, cudaStream_t stream) {
  if (mode == EPI_DUAL) return launch_mode<EPI_DUAL>(bn, cg, mcm, mcn, p, num_sms, stream);
  if (mode == EPI_DUALT) return launch_mode<EPI_DUALT>(bn, cg, mcm, mcn, p, num_sms, stream);
  if (mode == EPI_DX) return launch_mode<EPI_DX>(bn, cg, mcm, mcn, p, num_sms, stream);
  if (mode == EPI_DA) return launch_mode<EPI_DA>(bn, cg, mcm, mcn, p, num_sms, stream);
  if (mode == EPI_F32) return launch_mode<EPI_F32>(bn, cg, mcm, mcn, p, num_sms, stream);
  if (mode == EPI_GLU) return launch_mode<EPI_GLU>(bn, cg, mcm, mcn, p, num_sms, stream);
  return cudaErrorInvalidValue;
}

int gemm_resident_bwd(int bn, int mode, int cg, int mcm, int mcn, int num_sms) {
  if (mode == EPI_DUAL) return resident_mode<EPI_DUAL>(bn, cg, mcm, mcn, num_sms);
  if (mode == EPI_DUALT) return resident_mode<EPI_DUALT>(bn, cg, mcm, mcn, num_sms);
  if (mode == EPI_DX) return resident_mode<EPI_DX>(bn, cg, mcm, mcn, num_sms);
  if (mode == EPI_DA) return resident_mode<EPI_DA>(bn, cg, mcm, mcn, num_sms);
  if (mode == EPI_F32) return resident_mode<EPI_F32>(bn, cg, mcm, mcn, num_sms);
  if (mode == EPI_GLU) return resident_mode<EPI_GLU>(bn, cg, mcm, mcn, num_sms);
  return num_sms / cg;
}

}  // namespace boost_gb300
