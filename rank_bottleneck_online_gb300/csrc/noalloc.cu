// noalloc.cu -- RMSNorm row scales for callers that cannot allocate device memory.
//
// Some callers can't call cudaMalloc: code that runs inside a host framework whose
// caching allocator owns all device memory (a direct cudaMalloc there bypasses its
// accounting, or fails under its memory cap), and plugins that are handed only their
// input and output buffers. For them, boost_rmsnorm_rstd_noalloc computes the row
// scales rstd [T] with the per-shard sums of squares kept in a fixed array compiled
// into this library (g_shard_ssq below): the CUDA runtime reserves it on every GPU
// that loads the library's device code and it stays there until the process exits.
// The caller passes only x and rstd; nothing is allocated per call.
//
// Structure: one kernel writes ssq[s, t] for every (row, shard) into the array, a
// second reads each row's S partials back in shard order and writes rstd[t]. Every
// partial a call reads is written earlier by the same call, so the array needs no
// clearing; it keeps the last call's values. All calls share the one array, so calls
// whose kernels overlap on the GPU race.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "boost_block.h"
#include "ptx.cuh"

namespace {

// Capacity of the shared partials array: S * T floats (4 MiB).
constexpr int64_t kNoAllocMaxPartials = int64_t{1} << 20;

static __device__ __align__(256) float g_shard_ssq[kNoAllocMaxPartials];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch[kMaxDevices] = {};

// Device address of g_shard_ssq on the current device. The name g_shard_ssq in host
// code is only a host-side stand-in; the address comes from cudaGetSymbolAddress,
// looked up once per device with that device current (on the first call there).
cudaError_t scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_shard_ssq);
    if (e != cudaSuccess) return e;
    g_scratch[dev] = static_cast<float*>(p);
  }
  *out = g_scratch[dev];
  return cudaSuccess;
}

constexpr int kThreads = 256;

// One warp per (row, shard): sum of squares of the shard's w = d / S columns.
__global__ void __launch_bounds__(kThreads) shard_ssq_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t T, int64_t d, int S, float* __restrict__ ssq) {
  const int64_t item = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (item >= T * S) return;
  const int64_t row = item / S;
  const int s = static_cast<int>(item - row * S);
  const int64_t w = d / S;
  const __nv_bfloat16* xs = x + row * d + s * w;
  float acc = 0.0f;
  if ((w & 7) == 0) {
    const uint4* v = reinterpret_cast<const uint4*>(xs);
    for (int64_t i = lane; i < (w >> 3); i += 32) {
      const uint4 u = __ldg(v + i);
      const float f[8] = {boost_gb300::bf16_lo(u.x), boost_gb300::bf16_hi(u.x),
                          boost_gb300::bf16_lo(u.y), boost_gb300::bf16_hi(u.y),
                          boost_gb300::bf16_lo(u.z), boost_gb300::bf16_hi(u.z),
                          boost_gb300::bf16_lo(u.w), boost_gb300::bf16_hi(u.w)};
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(f[e], f[e], acc);
    }
  } else {
    for (int64_t i = lane; i < w; i += 32) {
      const float f = __bfloat162float(xs[i]);
      acc = fmaf(f, f, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) ssq[static_cast<int64_t>(s) * T + row] = acc;
}

// One thread per row: the single combine of the S partials, in shard order.
__global__ void __launch_bounds__(kThreads) combine_rstd_kernel(
    const float* __restrict__ ssq, int64_t T, int64_t d, int S, float eps,
    float* __restrict__ rstd) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (row >= T) return;
  float total = 0.0f;
  for (int s = 0; s < S; ++s) total += ssq[static_cast<int64_t>(s) * T + row];
  rstd[row] = 1.0f / sqrtf(total / static_cast<float>(d) + eps);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" boost_status boost_rmsnorm_rstd_noalloc(const boost_block_desc* desc, const void* x,
                                                   float* rstd, void* stream) {
  if (desc == nullptr) return BOOST_ERR_INVALID_ARG;
  const boost_block_desc& D = *desc;
  if (D.has_norm != 1 || D.T < 0 || D.d < 1 || D.S < 1) return BOOST_ERR_INVALID_ARG;
  if (!(D.eps >= 0.0f) || !std::isfinite(D.eps)) return BOOST_ERR_INVALID_ARG;
  if (D.d % 8 != 0 || D.d % D.S != 0 || D.d > (int64_t{1} << 31) - 1)
    return BOOST_ERR_UNSUPPORTED_SHAPE;
  if (D.T > kNoAllocMaxPartials || D.T * D.S > kNoAllocMaxPartials)
    return BOOST_ERR_UNSUPPORTED_SHAPE;   // partials would not fit the fixed array
  if (D.T == 0) return BOOST_OK;
  if (x == nullptr || rstd == nullptr) return BOOST_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(rstd)) return BOOST_ERR_ALIGNMENT;
  float* ssq = nullptr;
  if (scratch_for_current_device(&ssq) != cudaSuccess) {
    cudaGetLastError();
    return BOOST_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t items = D.T * D.S;
  const int64_t warps_per_block = kThreads / 32;
  shard_ssq_kernel<<<static_cast<unsigned>((items + warps_per_block - 1) / warps_per_block),
                     kThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(x), D.T, D.d, D.S, ssq);
  if (cudaGetLastError() != cudaSuccess) return BOOST_ERR_CUDA;
  combine_rstd_kernel<<<static_cast<unsigned>((D.T + kThreads - 1) / kThreads), kThreads, 0, s>>>(
      ssq, D.T, D.d, D.S, D.eps, rstd);
  if (cudaGetLastError() != cudaSuccess) return BOOST_ERR_CUDA;
  return BOOST_OK;
}
