// internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "gemm.cuh"

namespace boost_gb300 {

// ----------------------------------------------------------- GEMM launches
// Launch gemm_kernel<BN, MODE, CG, MC> persistently (CG = 2: CTA pairs, 256-row tiles;
// MC = 2: two pairs per cluster sharing B by multicast). p.m_tiles is derived from p.M
// and the tile height.
cudaError_t launch_gemm(int bn, int mode, int cg, int mc, const GemmParams& p, int num_sms,
                        cudaStream_t stream);

// ------------------------------------------------------ CUDA-core kernels
cudaError_t launch_rmsnorm_stats(const void* x, int64_t T, int64_t d, int S, float eps,
                                 float* ssq, float* rstd, cudaStream_t stream);
cudaError_t launch_fold_gamma(const void* gamma, const void* A, void* Ap, int64_t d, int64_t kr,
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
