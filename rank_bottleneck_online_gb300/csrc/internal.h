// internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "gemm.cuh"

namespace boost_gb300 {

// ----------------------------------------------------------- GEMM launches
// Launch gemm_kernel<BN, MODE, CG, MCM, MCN> persistently (CG = 2: CTA pairs, 256-row
// tiles; MCM x MCN pairs per cluster sharing B along M and A along N by multicast).
// p.m_tiles is derived from p.M and the super-tile height; p.n_tiles must count
// super-tile columns (BN * MCN wide).
cudaError_t launch_gemm(int bn, int mode, int cg, int mcm, int mcn, const GemmParams& p,
                        int num_sms, cudaStream_t stream);
// Clusters of that configuration resident at once (the persistent grid size).
int gemm_resident(int bn, int mode, int cg, int mcm, int mcn, int num_sms);

// Launches carry the programmatic-stream-serialisation attribute (the next kernel's
// prologue overlaps this one's tail; every kernel waits in griddep_wait before it
// touches global memory) unless the environment sets BOOST_PDL=0.
bool pdl_enabled();

// ------------------------------------------------------ CUDA-core kernels
cudaError_t launch_rmsnorm_stats(const void* x, int64_t T, int64_t d, int S, float eps,
                                 float* ssq, float* rstd, cudaStream_t stream);
cudaError_t launch_fold_gamma(const void* gamma, const void* A, void* Ap, int64_t d, int64_t kr,
                              cudaStream_t stream);
// the statistics and the gamma fold of a normed block in one launch
cudaError_t launch_stats_fold(const void* x, int64_t T, int64_t d, int S, float eps, float* ssq,
                              float* rstd, const void* gamma, const void* A, void* Ap, int64_t kr,
                              cudaStream_t stream);
cudaError_t launch_btp_reduce(const float* zpart, const float* ssq, int S, int64_t T,
                              int64_t kr, int64_t d, float eps, int act, void* a, float* rstd,
                              cudaStream_t stream);
cudaError_t launch_swiglu_fwd(const void* g, const void* u, void* h, int64_t count,
                              cudaStream_t stream);
cudaError_t launch_swiglu_bwd(const void* g, const void* u, const void* dh, void* dg, void* du,
                              int64_t count, cudaStream_t stream);
cudaError_t launch_add(const void* a, const void* b, void* out, int64_t count,
                       cudaStream_t stream);
cudaError_t launch_splitk_sum_bf16(const float* part, int splits, int64_t count, void* out,
                                   cudaStream_t stream);
cudaError_t launch_splitk_finalize_dA(const float* part, int splits, int64_t d, int64_t kr,
                                      const void* gamma, const void* A, void* dA, void* dgamma,
                                      cudaStream_t stream);
cudaError_t launch_dgamma_reduce(const float* dgpart, int ntiles, int64_t d, void* dgamma,
                                 cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(DeviceError* err, uint64_t limit_ns, cudaStream_t stream);

}  // namespace boost_gb300
