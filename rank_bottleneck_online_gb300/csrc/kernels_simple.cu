// kernels_simple.cu -- the block's HBM-bound CUDA-core kernels: Online-RMSNorm
// statistics, the gamma fold, SwiGLU forward/backward, residual add, split-K
// finalisation, the dgamma reduction and the bounded-wait self-test.
// All bf16 traffic moves in 16-byte vectors (8 elements per thread access).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <utility>

#include "internal.h"

namespace boost_gb300 {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
  f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
  f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The first statement of every kernel here: wait for the kernel before it on the
// stream (a no-op unless the launch carried a programmatic dependency), then let the
// next one be scheduled. Both precede any global memory access.
__device__ __forceinline__ void pdl_enter() {
  griddep_wait();
  griddep_launch_dependents();
}

// Launch `kern` on `stream`, with the programmatic-stream-serialisation attribute
// when enabled.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), int64_t grid, cudaStream_t stream,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// logistic(z) with the hardware exp2 and a fast reciprocal divide, the same expression
// as the GEMM epilogues', so that the fused and the stand-alone SwiGLU passes agree bit
// for bit.
__device__ __forceinline__ float sigmoid_fast(float z) {
  return __fdividef(1.0f, 1.0f + __expf(-z));
}

__device__ __forceinline__ float silu_f(float z) { return z * sigmoid_fast(z); }

__device__ __forceinline__ float silu_grad_f(float z) {
  const float g = sigmoid_fast(z);
  return g * (1.0f + z * (1.0f - g));
}

// Online-RMSNorm statistics (BOOST technical summary §2.2): one warp per row.
// ssq[s, t] is the fp32 sum of squares over shard s = columns [s*w, (s+1)*w);
// the shards are then combined once, in index order, into rstd[t].
__device__ __forceinline__ void stats_row(const __nv_bfloat16* __restrict__ x, int64_t T,
                                          int64_t d, int S, float eps, float* __restrict__ ssq,
                                          float* __restrict__ rstd, int64_t row, int lane) {
  const __nv_bfloat16* xr = x + row * d;
  const int64_t w = d / S;
  float total = 0.0f;
  for (int s = 0; s < S; ++s) {
    const __nv_bfloat16* xs = xr + s * w;
    float acc0 = 0.0f, acc1 = 0.0f;
    if ((w & 7) == 0) {
      const uint4* v = reinterpret_cast<const uint4*>(xs);
      const int64_t nv = w >> 3;
      int64_t i = lane;
      for (; i + 32 < nv; i += 64) {
        float f[8], g[8];
        unpack8(__ldg(v + i), f);
        unpack8(__ldg(v + i + 32), g);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc0 = fmaf(f[e], f[e], acc0);
          acc1 = fmaf(g[e], g[e], acc1);
        }
      }
      for (; i < nv; i += 32) {
        float f[8];
        unpack8(__ldg(v + i), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc0 = fmaf(f[e], f[e], acc0);
      }
    } else {
      for (int64_t i = lane; i < w; i += 32) {
        const float f = __bfloat162float(xs[i]);
        acc0 = fmaf(f, f, acc0);
      }
    }
    const float part = warp_sum(acc0 + acc1);
    if (lane == 0 && ssq != nullptr) ssq[static_cast<int64_t>(s) * T + row] = part;
    total += part;  // the single combine, in shard order
  }
  if (lane == 0) rstd[row] = 1.0f / sqrtf(total / static_cast<float>(d) + eps);
}

__global__ void __launch_bounds__(kThreads) rmsnorm_stats_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t T, int64_t d, int S, float eps,
    float* __restrict__ ssq, float* __restrict__ rstd) {
  pdl_enter();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
  if (row < T) stats_row(x, T, d, S, eps, ssq, rstd, row, threadIdx.x & 31);
}

// The reduction standing in for the bottleneck-aware TP all-reduce (BOOST technical
// summary §2.1, statistics fused per §2.2): z = sum over shards of the partial products
// zpart [S, T, kr] (shard order), the row scale from the summed sums of squares
// ssq [S, T] (full-d mean, the same expression and order as rmsnorm_stats_kernel), and
// a = bf16(act(s * z)) with the GEMM epilogue's activation. One thread per 8 columns.
__global__ void __launch_bounds__(kThreads) btp_reduce_kernel(
    const float* __restrict__ zpart, const float* __restrict__ ssq, int S, int64_t T,
    int64_t kr, int64_t d, float eps, int act, uint4* __restrict__ a, float* __restrict__ rstd) {
  pdl_enter();
  const int64_t nv = kr / 8;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < T * nv;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t t = i / nv;
    const int64_t v = i - t * nv;
    float srow = 1.0f;
    if (ssq != nullptr) {
      float total = 0.0f;
      for (int s = 0; s < S; ++s) total += ssq[static_cast<int64_t>(s) * T + t];
      srow = 1.0f / sqrtf(total / static_cast<float>(d) + eps);
      if (v == 0 && rstd != nullptr) rstd[t] = srow;
    }
    float z[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    for (int s = 0; s < S; ++s) {
      const float4* src =
          reinterpret_cast<const float4*>(zpart + (static_cast<int64_t>(s) * T + t) * kr) + 2 * v;
      const float4 p0 = src[0], p1 = src[1];
      z[0] += p0.x; z[1] += p0.y; z[2] += p0.z; z[3] += p0.w;
      z[4] += p1.x; z[5] += p1.y; z[6] += p1.z; z[7] += p1.w;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float f = srow * z[e];
      z[e] = act == 1 ? silu_f(f) : f;
    }
    a[i] = pack8(z);
  }
}

// The same statistics when every shard spans a multiple of 256 columns (32 lanes x 8
// values): each lane's 16-byte pieces lane + 32 j of a row then fall, for every j, into
// one shard for the whole warp, so a lane can issue eight loads before it reduces (a
// row's loads in flight instead of two pieces per shard) and the shard boundaries stay
// warp-uniform. Shards are reduced and combined in index order.
__device__ __forceinline__ void stats_row_wide(const __nv_bfloat16* __restrict__ x, int64_t T,
                                               int64_t d, int S, float eps,
                                               float* __restrict__ ssq, float* __restrict__ rstd,
                                               int64_t row, int lane) {
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * d) + lane;
  const int nj = static_cast<int>(d / 256);          // pieces per lane
  const int jps = static_cast<int>(d / S / 256);     // pieces per lane per shard
  float total = 0.0f, run = 0.0f;
  int cur = 0;
  for (int j0 = 0; j0 < nj; j0 += 8) {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (j0 + k < nj) v[k] = __ldg(xr + 32 * (j0 + k));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (j0 + k >= nj) break;
      const int sh = (j0 + k) / jps;               // warp-uniform
      if (sh != cur) {
        const float part = warp_sum(run);
        if (lane == 0 && ssq != nullptr) ssq[static_cast<int64_t>(cur) * T + row] = part;
        total += part;
        run = 0.0f;
        cur = sh;
      }
      float f[8];
      unpack8(v[k], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) run = fmaf(f[e], f[e], run);
    }
  }
  const float part = warp_sum(run);
  if (lane == 0 && ssq != nullptr) ssq[static_cast<int64_t>(cur) * T + row] = part;
  total += part;
  if (lane == 0) rstd[row] = 1.0f / sqrtf(total / static_cast<float>(d) + eps);
}

__global__ void __launch_bounds__(kThreads) rmsnorm_stats_wide_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t T, int64_t d, int S, float eps,
    float* __restrict__ ssq, float* __restrict__ rstd) {
  pdl_enter();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
  if (row < T) stats_row_wide(x, T, d, S, eps, ssq, rstd, row, threadIdx.x & 31);
}

// A'[j, m] = bf16(gamma_j * A[j, m]); the product of two bf16 values is exact in fp32.
// A grid-stride loop over the 16-byte pieces of A; each thread has kFoldUnroll pieces
// (kThreads pieces apart) in flight before it scales and stores them.
constexpr int kFoldUnroll = 4;

// (block `blk` of `nblk` blocks taking part in the fold)
__device__ __forceinline__ void fold_part(const __nv_bfloat16* __restrict__ gamma,
                                          const uint4* __restrict__ A, uint4* __restrict__ Ap,
                                          int64_t nvec, int64_t row_vecs, int64_t blk,
                                          int64_t nblk) {
  const int64_t stride = nblk * kThreads * kFoldUnroll;
  for (int64_t base = blk * kThreads * kFoldUnroll + threadIdx.x; base < nvec; base += stride) {
    uint4 u[kFoldUnroll];
#pragma unroll
    for (int k = 0; k < kFoldUnroll; ++k) {
      const int64_t i = base + k * kThreads;
      if (i < nvec) u[k] = __ldg(A + i);
    }
#pragma unroll
    for (int k = 0; k < kFoldUnroll; ++k) {
      const int64_t i = base + k * kThreads;
      if (i >= nvec) break;
      const float g = __bfloat162float(gamma[i / row_vecs]);
      float f[8];
      unpack8(u[k], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] *= g;
      Ap[i] = pack8(f);
    }
  }
}

__global__ void __launch_bounds__(kThreads) fold_gamma_kernel(
    const __nv_bfloat16* __restrict__ gamma, const uint4* __restrict__ A, uint4* __restrict__ Ap,
    int64_t nvec, int64_t row_vecs) {
  pdl_enter();
  fold_part(gamma, A, Ap, nvec, row_vecs, blockIdx.x, gridDim.x);
}

// The statistics and the gamma fold of a normed block in one launch: they are
// independent and both bandwidth-bound, so the fold's blocks fill the statistics' tail
// and one launch replaces two. Blocks [0, stat_blocks) take rows of x (one warp per row),
// the rest take pieces of A.
__global__ void __launch_bounds__(kThreads) stats_fold_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t T, int64_t d, int S, float eps,
    float* __restrict__ ssq, float* __restrict__ rstd, int wide, int64_t stat_blocks,
    const __nv_bfloat16* __restrict__ gamma, const uint4* __restrict__ A, uint4* __restrict__ Ap,
    int64_t nvec, int64_t row_vecs) {
  pdl_enter();
  const int64_t b = blockIdx.x;
  if (b < stat_blocks) {
    const int64_t row = b * (kThreads / 32) + (threadIdx.x >> 5);
    if (row < T) {
      if (wide) stats_row_wide(x, T, d, S, eps, ssq, rstd, row, threadIdx.x & 31);
      else stats_row(x, T, d, S, eps, ssq, rstd, row, threadIdx.x & 31);
    }
  } else {
    fold_part(gamma, A, Ap, nvec, row_vecs, b - stat_blocks, gridDim.x - stat_blocks);
  }
}

__global__ void __launch_bounds__(kThreads) swiglu_fwd_kernel(
    const uint4* __restrict__ g, const uint4* __restrict__ u, uint4* __restrict__ h, int64_t nvec) {
  pdl_enter();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    float fg[8], fu[8], fh[8];
    unpack8(g[i], fg);
    unpack8(u[i], fu);
#pragma unroll
    for (int e = 0; e < 8; ++e) fh[e] = silu_f(fg[e]) * fu[e];
    h[i] = pack8(fh);
  }
}

__global__ void __launch_bounds__(kThreads) swiglu_bwd_kernel(
    const uint4* __restrict__ g, const uint4* __restrict__ u, const uint4* __restrict__ dh,
    uint4* __restrict__ dg, uint4* __restrict__ du, int64_t nvec) {
  pdl_enter();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    float fg[8], fu[8], fd[8], og[8], ou[8];
    unpack8(g[i], fg);
    unpack8(u[i], fu);
    unpack8(dh[i], fd);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      og[e] = fd[e] * fu[e] * silu_grad_f(fg[e]);
      ou[e] = fd[e] * silu_f(fg[e]);
    }
    dg[i] = pack8(og);
    du[i] = pack8(ou);
  }
}

__global__ void __launch_bounds__(kThreads) add_kernel(const uint4* a, const uint4* b, uint4* out,
                                                       int64_t nvec) {
  pdl_enter();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    float fa[8], fb[8];
    unpack8(a[i], fa);
    unpack8(b[i], fb);
#pragma unroll
    for (int e = 0; e < 8; ++e) fa[e] += fb[e];
    out[i] = pack8(fa);
  }
}

// Most split-K splits the host plans (its planner stops at 8).
constexpr int kMaxSplits = 8;

// out = bf16(sum_s part[s]) over `count` elements, splits summed in index order. Every
// split's value is loaded before the sum, so a thread has all its loads in flight at once
// (MAXS: the most splits this instantiation takes, 4 or kMaxSplits).
template <int MAXS>
__global__ void __launch_bounds__(kThreads) splitk_sum_bf16_kernel(
    const float4* __restrict__ part, int splits, int64_t count4, uint2* __restrict__ out) {
  pdl_enter();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < count4;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    float4 v[MAXS];
#pragma unroll
    for (int s = 0; s < MAXS; ++s)
      if (s < splits) v[s] = __ldg(part + static_cast<int64_t>(s) * count4 + i);
    float4 acc = v[0];
#pragma unroll
    for (int s = 1; s < MAXS; ++s) {
      if (s >= splits) break;
      acc.x += v[s].x; acc.y += v[s].y; acc.z += v[s].z; acc.w += v[s].w;
    }
    out[i] = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
}

// One block per row j of G = sum_s part[s] ([d, kr], splits summed in order): dA =
// bf16(gamma_j * G[j, :]) and dgamma_j = bf16(sum_m A[j, m] * G[j, m]), the row sum
// reduced in a fixed order (per thread, then per warp, then over the warps). Without
// gamma: dA = bf16(G). Each thread takes 8 columns at a time (MAXS: the most splits this
// instantiation takes, 4 or kMaxSplits).
template <int MAXS>
__global__ void __launch_bounds__(kThreads) splitk_finalize_dA_kernel(
    const float* __restrict__ part, int splits, int64_t d, int64_t kr,
    const __nv_bfloat16* __restrict__ gamma, const __nv_bfloat16* __restrict__ A,
    __nv_bfloat16* __restrict__ dA, __nv_bfloat16* __restrict__ dgamma) {
  pdl_enter();
  __shared__ float wsum[kThreads / 32];
  const int64_t j = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float g = gamma != nullptr ? __bfloat162float(gamma[j]) : 1.0f;
  const int64_t nv = kr / 8;
  const int64_t plane = d * kr;
  float acc = 0.0f;
  for (int64_t i = threadIdx.x; i < nv; i += kThreads) {
    const int64_t off = j * kr + i * 8;
    // four splits' 8 values at a time in flight before they are added (splits summed in
    // index order)
    float G[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int s0 = 0; s0 < MAXS; s0 += 4) {
      if (s0 >= splits) break;
      float4 b[4][2];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (s0 + q < splits) {
          b[q][0] = __ldg(reinterpret_cast<const float4*>(part + (s0 + q) * plane + off));
          b[q][1] = __ldg(reinterpret_cast<const float4*>(part + (s0 + q) * plane + off + 4));
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (s0 + q >= splits) break;
        if (s0 + q == 0) {
          G[0] = b[0][0].x; G[1] = b[0][0].y; G[2] = b[0][0].z; G[3] = b[0][0].w;
          G[4] = b[0][1].x; G[5] = b[0][1].y; G[6] = b[0][1].z; G[7] = b[0][1].w;
        } else {
          G[0] += b[q][0].x; G[1] += b[q][0].y; G[2] += b[q][0].z; G[3] += b[q][0].w;
          G[4] += b[q][1].x; G[5] += b[q][1].y; G[6] += b[q][1].z; G[7] += b[q][1].w;
        }
      }
    }
    float o[8];
    if (gamma != nullptr) {
      float a[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(A + off)), a);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc = fmaf(a[e], G[e], acc);
        o[e] = g * G[e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = G[e];
    }
    *reinterpret_cast<uint4*>(dA + off) = pack8(o);
  }
  if (dgamma != nullptr) {
    acc = warp_sum(acc);
    if (lane == 0) wsum[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int w = 0; w < kThreads / 32; ++w) t += wsum[w];
      dgamma[j] = __float2bfloat16_rn(t);
    }
  }
}

// dgamma_j = bf16(sum_t dgpart[t][j]), tiles summed in index order.
__global__ void __launch_bounds__(kThreads) dgamma_reduce_kernel(
    const float* __restrict__ dgpart, int ntiles, int64_t d, __nv_bfloat16* __restrict__ dgamma) {
  pdl_enter();
  const int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (j >= d) return;
  float acc = 0.0f;
  for (int t = 0; t < ntiles; ++t) acc += dgpart[static_cast<int64_t>(t) * d + j];
  dgamma[j] = __float2bfloat16_rn(acc);
}

// Bounded-wait self-test: waits on an mbarrier that nothing arrives on. The wait
// gives up after limit_ns, records the timeout and the kernel returns normally.
__global__ void wait_timeout_probe_kernel(DeviceError* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    bool done = false;
    while (!done) {
      if (mbar_try_wait(&bar, 0)) break;
      if (globaltimer_ns() - t0 > limit_ns) {
        record_error(err, kErrTimeout, 100);
        done = true;
      }
    }
    // Complete the barrier's phase so nothing is left pending at exit.
    mbar_arrive(&bar);
  }
  __syncthreads();
}

int grid_for(int64_t work, int per_block) {
  int64_t g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > 148 * 32) g = 148 * 32;
  return static_cast<int>(g);
}

}  // namespace

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("BOOST_PDL");
    return e == nullptr || std::atoi(e) != 0;
  }();
  return on;
}

cudaError_t launch_rmsnorm_stats(const void* x, int64_t T, int64_t d, int S, float eps,
                                 float* ssq, float* rstd, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int rows_per_block = kThreads / 32;
  const int64_t grid = (T + rows_per_block - 1) / rows_per_block;
  const bool wide = (d / S) % 256 == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  return launch_k(wide ? rmsnorm_stats_wide_kernel : rmsnorm_stats_kernel, grid, stream,
                  static_cast<const __nv_bfloat16*>(x), T, d, S, eps, ssq, rstd);
}

cudaError_t launch_btp_reduce(const float* zpart, const float* ssq, int S, int64_t T,
                              int64_t kr, int64_t d, float eps, int act, void* a, float* rstd,
                              cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  return launch_k(btp_reduce_kernel, grid_for(T * (kr / 8), kThreads), stream,
      zpart, ssq, S, T, kr, d, eps, act, static_cast<uint4*>(a), rstd);
}

cudaError_t launch_stats_fold(const void* x, int64_t T, int64_t d, int S, float eps, float* ssq,
                              float* rstd, const void* gamma, const void* A, void* Ap, int64_t kr,
                              cudaStream_t stream) {
  if (T == 0) return launch_fold_gamma(gamma, A, Ap, d, kr, stream);
  if (d * kr == 0) return launch_rmsnorm_stats(x, T, d, S, eps, ssq, rstd, stream);
  const int rows_per_block = kThreads / 32;
  const int64_t stat_blocks = (T + rows_per_block - 1) / rows_per_block;
  const int64_t nvec = d * (kr / 8);
  const int64_t fold_blocks = grid_for(nvec, kThreads * kFoldUnroll);
  const int wide = ((d / S) % 256 == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0) ? 1 : 0;
  return launch_k(stats_fold_kernel, stat_blocks + fold_blocks, stream,
      static_cast<const __nv_bfloat16*>(x), T, d, S, eps, ssq, rstd, wide, stat_blocks,
      static_cast<const __nv_bfloat16*>(gamma), static_cast<const uint4*>(A),
      static_cast<uint4*>(Ap), nvec, kr / 8);
}

cudaError_t launch_fold_gamma(const void* gamma, const void* A, void* Ap, int64_t d, int64_t kr,
                              cudaStream_t stream) {
  if (d * kr == 0) return cudaSuccess;
  const int64_t nvec = d * (kr / 8);
  return launch_k(fold_gamma_kernel, grid_for(nvec, kThreads * kFoldUnroll), stream,
      static_cast<const __nv_bfloat16*>(gamma), static_cast<const uint4*>(A),
      static_cast<uint4*>(Ap), nvec, kr / 8);
}

cudaError_t launch_swiglu_fwd(const void* g, const void* u, void* h, int64_t count,
                              cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  return launch_k(swiglu_fwd_kernel, grid_for(count / 8, kThreads), stream,
      static_cast<const uint4*>(g), static_cast<const uint4*>(u), static_cast<uint4*>(h),
      count / 8);
}

cudaError_t launch_swiglu_bwd(const void* g, const void* u, const void* dh, void* dg, void* du,
                              int64_t count, cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  return launch_k(swiglu_bwd_kernel, grid_for(count / 8, kThreads), stream,
      static_cast<const uint4*>(g), static_cast<const uint4*>(u), static_cast<const uint4*>(dh),
      static_cast<uint4*>(dg), static_cast<uint4*>(du), count / 8);
}

cudaError_t launch_add(const void* a, const void* b, void* out, int64_t count,
                       cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  return launch_k(add_kernel, grid_for(count / 8, kThreads), stream,
      static_cast<const uint4*>(a), static_cast<const uint4*>(b), static_cast<uint4*>(out),
      count / 8);
}

cudaError_t launch_splitk_sum_bf16(const float* part, int splits, int64_t count, void* out,
                                   cudaStream_t stream) {
  if (splits < 1 || splits > kMaxSplits) return cudaErrorInvalidValue;
  if (count == 0) return cudaSuccess;
  const auto kern = splits <= 4 ? splitk_sum_bf16_kernel<4> : splitk_sum_bf16_kernel<kMaxSplits>;
  return launch_k(kern, grid_for(count / 4, kThreads), stream,
      reinterpret_cast<const float4*>(part), splits, count / 4, static_cast<uint2*>(out));
}

cudaError_t launch_splitk_finalize_dA(const float* part, int splits, int64_t d, int64_t kr,
                                      const void* gamma, const void* A, void* dA, void* dgamma,
                                      cudaStream_t stream) {
  if (splits < 1 || splits > kMaxSplits) return cudaErrorInvalidValue;
  if (d == 0) return cudaSuccess;
  const auto kern =
      splits <= 4 ? splitk_finalize_dA_kernel<4> : splitk_finalize_dA_kernel<kMaxSplits>;
  return launch_k(kern, d, stream,
      part, splits, d, kr, static_cast<const __nv_bfloat16*>(gamma),
      static_cast<const __nv_bfloat16*>(A), static_cast<__nv_bfloat16*>(dA),
      static_cast<__nv_bfloat16*>(dgamma));
}

cudaError_t launch_dgamma_reduce(const float* dgpart, int ntiles, int64_t d, void* dgamma,
                                 cudaStream_t stream) {
  if (d == 0) return cudaSuccess;
  return launch_k(dgamma_reduce_kernel, (d + kThreads - 1) / kThreads, stream,
      dgpart, ntiles, d, static_cast<__nv_bfloat16*>(dgamma));
}

cudaError_t launch_wait_timeout_probe(DeviceError* err, uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace boost_gb300
