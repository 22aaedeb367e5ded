// boost_block.cu -- C ABI of the bottleneck block: argument validation, workspace
// layout, launch plans, TMA tensor maps, and the forward/backward launch sequences.
//
// Operation: the CoLA-style low-rank bottleneck of "BOOST: BOttleneck-Optimized
// Scalable Training Framework for Low-Rank Large Language Models" (technical
// summary §2.1-§2.2): Online-RMSNorm statistics with deferred normalisation,
// grouped down-projection over concatenated weights, batched up-projection, and a
// backward that recomputes the bottleneck activation inside the block.
#include "boost_block.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <vector>

#include "internal.h"
#include "profile.h"

namespace boost_gb300 {
cudaError_t launch_gemm_fwd_modes(int bn, int mode, int cg, int mcm, int mcn,
                                  const GemmParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_gemm_bwd_modes(int bn, int mode, int cg, int mcm, int mcn,
                                  const GemmParams& p, int num_sms, cudaStream_t stream);
int gemm_resident_fwd(int bn, int mode, int cg, int mcm, int mcn, int num_sms);
int gemm_resident_bwd(int bn, int mode, int cg, int mcm, int mcn, int num_sms);

cudaError_t launch_gemm(int bn, int mode, int cg, int mcm, int mcn, const GemmParams& p,
                        int num_sms, cudaStream_t stream) {
  if (mode == EPI_ACT || mode == EPI_BF16 || mode == EPI_UPGLU || mode == EPI_BF16T)
    return launch_gemm_fwd_modes(bn, mode, cg, mcm, mcn, p, num_sms, stream);
  return launch_gemm_bwd_modes(bn, mode, cg, mcm, mcn, p, num_sms, stream);
}

int gemm_resident(int bn, int mode, int cg, int mcm, int mcn, int num_sms) {
  if (mode == EPI_ACT || mode == EPI_BF16 || mode == EPI_UPGLU || mode == EPI_BF16T)
    return gemm_resident_fwd(bn, mode, cg, mcm, mcn, num_sms);
  return gemm_resident_bwd(bn, mode, cg, mcm, mcn, num_sms);
}
}  // namespace boost_gb300

using namespace boost_gb300;

namespace {

constexpr size_t kAlign = 256;
constexpr int64_t kMaxDim = (1ll << 31) - 1;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Two buffers of `bytes` each that overlap without being the same buffer.
bool partial_overlap(const void* a, const void* b, uint64_t bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x != y && x < y + bytes && y < x + bytes;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// --------------------------------------------------------------- devices
int current_num_sms() {
  // per-device cache; host threads may fill it concurrently (same value)
  static std::atomic<int> cache[64];
  constexpr int kFallback = 152;   // GB300; only when the runtime cannot be asked
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return kFallback;
  }
  if (cache[dev].load(std::memory_order_relaxed) == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return kFallback;
    }
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return cache[dev].load(std::memory_order_relaxed);
}

uint64_t wait_limit_ns() {
  static uint64_t v = [] {
    const char* e = std::getenv("BOOST_WAIT_LIMIT_MS");
    double ms = e ? std::atof(e) : 2000.0;
    if (!(ms > 0.0)) ms = 2000.0;
    return static_cast<uint64_t>(ms * 1e6);
  }();
  return v;
}

// ----------------------------------------------------------- tensor maps
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
    cudaGetLastError();
  });
  return fn;
}

// 3-D bf16 view: dims (d0 contiguous, d1, d2), byte strides of d1 and d2, box b0 x b1 x b2,
// 128-byte swizzle (operand loads) or 64-byte swizzle (32-wide epilogue store boxes),
// zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2,
              bool sw64 = false) {
  EncodeFn enc = get_encode();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   sw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Maps for the epilogue's TMA stores (the SwiGLU epilogue modes store through TMA; the
// others use plain stores and need none): out (`batches` matrices of rows x cols,
// out_bstride apart) and out2 (`batches2` of them), leading dimension ldo, 32 x 32
// boxes. An output whose map cannot be made is written with plain stores.
void set_out_maps(GemmParams& g, int64_t rows, int64_t cols, int64_t batches,
                  int64_t batches2 = 1) {
  const uint64_t ld = static_cast<uint64_t>(g.ldo) * 2;
  if (g.out != nullptr &&
      make_map(&g.tmO[0], g.out, cols, rows, batches, ld,
               (batches > 1 ? static_cast<uint64_t>(g.out_bstride) : rows * g.ldo) * 2, 32, 32, 1,
               true))
    g.tma_out |= 1;
  if (g.out2 != nullptr &&
      make_map(&g.tmO[1], g.out2, cols, rows, batches2, ld, rows * g.ldo * 2, 32, 32, 1, true))
    g.tma_out |= 2;
}

// A row-major [rows, cols] bf16 matrix (rows < 2^31), viewed 3-D as (cols, rows, 1).
bool map_2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_cols,
            uint32_t box_rows) {
  return make_map(m, base, cols, rows, 1, cols * 2, rows * cols * 2, box_cols, box_rows, 1);
}

OperandView kmajor_2d() { return OperandView{1, 0, 2, 0}; }   // (k, mn, -)
OperandView mnmajor_2d() { return OperandView{0, 1, 2, 1}; }  // (mn, k, -)

// ------------------------------------------------------------------ plan
// Launch shape of one GEMM: tile width, CTA pair (cg = 2), and pairs per cluster along
// M (mcm, sharing B) and along N (mcn, sharing A) by multicast.
struct Shape {
  int bn, cg, mcm, mcn;
  int64_t super_m() const { return int64_t{kBM} * cg * mcm; }
  int64_t super_n() const { return int64_t{bn} * mcn; }
  int a_rows() const { return 64; }   // every TMA box is 64 rows (see load_operand)
  int b_rows() const { return 64; }
};

struct Plan {
  int64_t T, d, r, k, n, kr;
  Shape down, dual, up, dx, wB, wA;
  int tpg_down, tpg_dual;           // super-tiles per group of r columns (K2, K4)
  int n_cols_dual;                  // rows of K4's q partials (column tiles x halves)
  int n_cols_wA;                    // rows of K6's dgamma partials (column tiles x halves)
  int splits_B, kbps_B, splits_A, kbps_A;
  size_t off_rstd, off_ssq, off_Ap, off_a, off_dzs, off_q, off_dg, off_partB, off_partA, total;
};

// Split-K choice for a weight gradient: minimise the estimated time
//   waves(s) * k-blocks per split * t_kb  +  partial bytes / HBM bandwidth  +  t_fix,
// where a wave is one pass of `groups` CTA groups over the tile list, t_kb is the
// time of one 64-deep k-block of a 256x256 tile on a CTA pair (about 0.5 us at the
// measured ~1.2-1.3 PFLOP/s), the fp32 partials are written once and read once, and
// t_fix (10 us) is the finaliser's own launch and ramp beyond its bytes. (Without t_fix
// the 1B block's two weight gradients split 5 ways. Unsplit measured 1.2% faster on the
// step: 0.585 -> 0.578 ms. The other workloads' plans do not change.)
int env_int(const char* name, int dflt);

void choose_splits(int64_t tiles, int64_t nkb, int groups, int64_t out_elems, int& splits,
                   int& kbps) {
  constexpr double kTkb = 0.5e-6;          // seconds per k-block per tile
  constexpr double kHbm = 6.0e12;          // bytes per second
  constexpr double kFix = 10e-6;           // seconds: the finaliser beyond its bytes
  splits = 1;
  kbps = static_cast<int>(nkb);
  static const int forced = env_int("BOOST_SPLITK", 0);   // > 0: this many splits (tuning)
  if (forced > 0) {
    const int64_t per = cdiv(nkb, std::min<int64_t>(forced, 8));
    splits = static_cast<int>(cdiv(nkb, per));
    kbps = static_cast<int>(per);
    return;
  }
  double best = 1e300;
  for (int s = 1; s <= 8; ++s) {
    if (s > 1 && nkb / s < 4) break;
    const int64_t per = cdiv(nkb, s);
    const int64_t s_eff = cdiv(nkb, per);
    const int64_t waves = cdiv(tiles * s_eff, groups);
    double cost = static_cast<double>(waves * per) * kTkb;
    if (s_eff > 1) cost += 2.0 * 4.0 * static_cast<double>(s_eff) * out_elems / kHbm + kFix;
    if (cost < best * (1.0 - 1e-6)) {
      best = cost;
      splits = static_cast<int>(s_eff);
      kbps = static_cast<int>(per);
    }
  }
}

int env_int(const char* name, int dflt) {
  const char* e = std::getenv(name);
  return e ? std::atoi(e) : dflt;
}

// Tile width for an N extent.
int pick_bn(int64_t n) { return n >= 256 ? 256 : (n >= 128 ? 128 : 64); }

// Launch shape for an M x N output (N tiled per group of `group` columns when > 0).
// CTA pairs for M >= 256; two pairs stacked along M sharing B when M >= 512; a 2 x 2
// arrangement sharing A too when N allows whole 512-wide super-tiles.
Shape pick_shape(int64_t m, int64_t n, int64_t group, int bn_cap = 256) {
  static const int forced_cg = env_int("BOOST_CG", 0);   // 1 or 2 forces (tuning)
  static const int mc_limit = env_int("BOOST_MC", 4);    // 1: none, 2: along M, 4: 2 x 2
  Shape sh{std::min(pick_bn(group > 0 ? group : n), bn_cap), 1, 1, 1};
  if (sh.bn >= 128) sh.cg = (forced_cg == 1 || forced_cg == 2) ? forced_cg : (m >= 256 ? 2 : 1);
  if (sh.cg == 2 && sh.bn == 256 && m >= 512 && mc_limit >= 2) {
    sh.mcm = 2;
    const bool n_ok = group > 0 ? (group % 512 == 0) : (n >= 512);
    if (n_ok && mc_limit >= 4) sh.mcn = 2;
  }
  return sh;
}

Plan make_plan(const boost_block_desc& D, int sms) {
  Plan P{};
  P.T = D.T; P.d = D.d; P.r = D.r; P.k = D.k; P.n = D.n; P.kr = D.k * D.r;
  P.down = pick_shape(D.T, P.kr, D.r);
  P.tpg_down = static_cast<int>(cdiv(D.r, P.down.super_n()));
  static const int dual_bn = env_int("BOOST_DUAL_BN", 256);
  P.dual = pick_shape(D.T, P.kr, D.r, dual_bn == 256 ? 256 : (dual_bn == 64 ? 64 : 128));
  P.tpg_dual = static_cast<int>(cdiv(D.r, P.dual.super_n()));
  // q partial rows: one per BN-wide column tile per epilogue half
  P.n_cols_dual = static_cast<int>(P.k * P.tpg_dual * P.dual.mcn * kEpiHalves);
  P.up = pick_shape(D.T, D.n, 0);
  P.dx = pick_shape(D.T, D.d, 0);
  const int64_t nkb_T = cdiv(std::max<int64_t>(D.T, 1), kBK);
  P.wB = pick_shape(D.r, D.n, 0);
  const int64_t tiles_B = D.k * cdiv(D.r, P.wB.super_m()) * cdiv(D.n, P.wB.super_n());
  choose_splits(tiles_B, nkb_T,
                gemm_resident(P.wB.bn, EPI_F32, P.wB.cg, P.wB.mcm, P.wB.mcn, sms),
                D.k * D.r * D.n, P.splits_B, P.kbps_B);
  P.wA = pick_shape(D.d, P.kr, 0);
  P.n_cols_wA = static_cast<int>(cdiv(P.kr, P.wA.super_n()) * P.wA.mcn * kEpiHalves);
  const int64_t tiles_A = cdiv(D.d, P.wA.super_m()) * cdiv(P.kr, P.wA.super_n());
  choose_splits(tiles_A, nkb_T,
                gemm_resident(P.wA.bn, EPI_F32, P.wA.cg, P.wA.mcm, P.wA.mcn, sms),
                D.d * P.kr, P.splits_A, P.kbps_A);

  size_t off = align_up(sizeof(DeviceError));
  P.off_rstd = off; off = align_up(off + sizeof(float) * D.T);
  P.off_ssq = off;  off = align_up(off + sizeof(float) * D.T * std::max(D.S, 1));
  P.off_Ap = off;   off = align_up(off + 2ull * D.d * P.kr);
  P.off_a = off;    off = align_up(off + 2ull * D.T * P.kr);
  P.off_dzs = off;  off = align_up(off + 2ull * D.T * P.kr);
  P.off_q = off;    off = align_up(off + sizeof(float) * P.n_cols_dual * D.T);
  P.off_dg = off;   off = align_up(off + sizeof(float) * P.n_cols_wA * D.d);
  const size_t partB = P.splits_B > 1 ? sizeof(float) * P.splits_B * D.k * D.r * D.n : 0;
  const size_t partA = P.splits_A > 1 ? sizeof(float) * P.splits_A * D.d * P.kr : 0;
  // separate regions: dB and dA may run concurrently (on two streams)
  P.off_partB = off; off = align_up(off + partB);
  P.off_partA = off; off = align_up(off + partA);
  P.total = off;
  return P;
}

double stats_bytes(const Plan& P, int S) { return 2.0 * P.T * P.d + 4.0 * P.T * (S + 1); }
double fold_bytes(const Plan& P) { return 4.0 * P.d * P.kr + 2.0 * P.d; }

boost_status validate_desc(const boost_block_desc* D) {
  if (D == nullptr) return BOOST_ERR_INVALID_ARG;
  if (D->T < 0 || D->d < 1 || D->r < 1 || D->k < 1 || D->n < 1) return BOOST_ERR_INVALID_ARG;
  if (D->act != BOOST_ACT_IDENTITY && D->act != BOOST_ACT_SILU) return BOOST_ERR_INVALID_ARG;
  if (D->has_norm != 0 && D->has_norm != 1) return BOOST_ERR_INVALID_ARG;
  if (D->has_norm) {
    if (D->S < 1) return BOOST_ERR_INVALID_ARG;
    if (!(D->eps >= 0.0f) || !std::isfinite(D->eps)) return BOOST_ERR_INVALID_ARG;
    if (D->d % D->S != 0) return BOOST_ERR_UNSUPPORTED_SHAPE;
  }
  if (D->d % 8 || D->r % 8 || D->n % 8) return BOOST_ERR_UNSUPPORTED_SHAPE;
  const int64_t kr = D->k * D->r;
  if (D->T > kMaxDim || D->d > kMaxDim || kr > kMaxDim || D->n > kMaxDim || D->k > 65535)
    return BOOST_ERR_UNSUPPORTED_SHAPE;
  // every row of every tensor and the flattened [k*T] / [k*r] extents fit 32-bit coordinates
  if (D->k * D->T > kMaxDim || D->k * D->r > kMaxDim) return BOOST_ERR_UNSUPPORTED_SHAPE;
  return BOOST_OK;
}

boost_status check_ptrs(std::initializer_list<const void*> required,
                        std::initializer_list<const void*> optional) {
  for (const void* p : required) {
    if (p == nullptr) return BOOST_ERR_INVALID_ARG;
    if (!aligned16(p)) return BOOST_ERR_ALIGNMENT;
  }
  for (const void* p : optional)
    if (p != nullptr && !aligned16(p)) return BOOST_ERR_ALIGNMENT;
  return BOOST_OK;
}

boost_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return BOOST_ERR_WORKSPACE;
  if (ws_bytes < need) return BOOST_ERR_WORKSPACE;
  return BOOST_OK;
}

template <typename T>
T* ws_at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

boost_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return BOOST_OK;
  return BOOST_ERR_CUDA;
}

GemmParams base_params(const Plan& P, DeviceError* err) {
  GemmParams g;
  std::memset(&g, 0, sizeof(g));
  g.splits = 1;
  g.batch = 1;
  g.num_seg = 1;
  g.err = err;
  g.wait_limit_ns = wait_limit_ns();
  (void)P;
  return g;
}

// Tile order of a weight-gradient GEMM (K = T, both operands streamed from HBM): the
// faster-moving index is the dimension with fewer tiles, so that the slabs of the other
// operand are read by all their tiles within one wave (from L2) instead of once per
// column (or row) of tiles. Measured on the down block's dA (22 x 2 tiles): M fastest
// read h twice from DRAM.
int32_t inner_m(int64_t M, int64_t N, const Shape& sh) {
  return cdiv(M, sh.super_m()) <= cdiv(N, sh.super_n()) ? 1 : 0;
}

// Down-projection GEMM parameters shared by the forward (K2) and the recompute (K4):
// M = T, N = k*r tiled per group (tpg tiles per group), K = d; A operand x (K-major),
// B operand A' (MN-major).
bool down_segment(GemmParams& g, const Plan& P, const void* x, const void* Ap, const Shape& sh,
                  int tpg) {
  if (!map_2d(&g.tmA[0], x, P.T, P.d, 64, sh.a_rows())) return false;
  if (!map_2d(&g.tmB[0], Ap, P.d, P.kr, 64, 64)) return false;
  g.seg[0].a = kmajor_2d();
  g.seg[0].b = mnmajor_2d();
  g.seg[0].num_kb = static_cast<int32_t>(cdiv(P.d, kBK));
  g.M = static_cast<int32_t>(P.T);
  g.N = static_cast<int32_t>(P.kr);
  g.n_tiles = static_cast<int32_t>(P.k * tpg);
  g.group_n = static_cast<int32_t>(P.r);
  g.group_tiles = tpg;
  g.m_inner = 0;
  return true;
}

// ------------------------------------------------- write counting (debug)
// While a caller has handed in a count buffer (boost_debug_count_writes), every GEMM
// operation gets its own count plane, shaped like its output (split and batch planes
// included), and its epilogues add 1 per element written; a log records each plane's
// geometry so the caller can check that every output element is written exactly once.
struct WriteCounter {
  std::mutex mu;
  int32_t* base = nullptr;
  int64_t capacity = 0, cursor = 0;
  bool overflow = false;
  std::vector<int64_t> log;   // kLogFields values per operation
};
constexpr int kLogFields = 8;

WriteCounter& write_counter() {
  static WriteCounter w;
  return w;
}

void attach_counts(GemmParams& g, int mode) {
  WriteCounter& w = write_counter();
  std::lock_guard<std::mutex> lk(w.mu);
  if (w.base == nullptr) return;
  const int64_t splits = std::max<int64_t>(g.splits, 1);
  // the fused up-projection writes two batch planes (gate, up) from one tile list
  const int64_t planes = mode == EPI_UPGLU ? 2 : std::max<int64_t>(g.batch, 1);
  const int64_t extent = (splits - 1) * g.out_sstride + (planes - 1) * g.out_bstride +
                         static_cast<int64_t>(g.M - 1) * g.ldo + g.N;
  if (w.cursor + extent > w.capacity) {
    w.overflow = true;
    return;
  }
  g.visits = w.base + w.cursor;
  w.log.insert(w.log.end(), {w.cursor, static_cast<int64_t>(g.M), static_cast<int64_t>(g.N),
                             g.ldo, planes, splits, g.out_bstride, g.out_sstride});
  w.cursor += extent;
}

// ------------------------------------------------------ co-scheduling
// Launch shapes with clusters of eight CTAs leave SMs that no such cluster fits (152 SMs
// hold 15 clusters of 8). For GEMMs over the token rows, the last rows of the output
// can run concurrently as a plain CTA-pair launch on a second stream that those SMs
// pick up; the row split follows the two launches' measured per-SM rates.
struct CoStreams {
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool ok = false;
  std::mutex order;   // one fork / launch / join sequence at a time per device
};

CoStreams* co_streams() {
  static CoStreams cs[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  CoStreams& c = cs[dev];
  if (!c.ok) {
    if (cudaStreamCreateWithFlags(&c.side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    c.ok = true;
  }
  return &c;
}

// Launch one GEMM over its M rows; with co-scheduling enabled and a 2 x 2 cluster shape,
// split the rows between that launch and a CTA-pair launch on a side stream. By default
// the side launch takes 130 of every 1000 rows (rounded to whole super-tiles of the
// cluster launch), the best single setting measured over the LLaMA-2 shapes. A planned
// split replaces it where it is predicted to save at least 2%: the split minimising the
// larger of the two launches' wave counts, a pair's 256 x 256 tile costing `cost`
// cluster super-tile waves (the side SMs' pairs have no multicast partner and share L2
// with the cluster launch, which costs them most where the tiles' K is short: 1.25 at
// K >= 12288, 1.5 at K >= 1024, 2 below, fitted to per-GEMM timings of the 7B MLP, the 1B
// block and the 40B pair against fixed splits). On the 7B MLP this moves the gate/up
// dual kernel, the fused up-projection and the SwiGLU backward to 26-27 cluster rows
// (2-3% faster each); the 1B block keeps the fixed split everywhere. BOOST_COSCHED_ROWCOST sets one cost (percent) for every K;
// BOOST_COSCHED > 0 fixes the side launch's rows per 1000 (no planning), 0 turns the
// split off.
cudaError_t launch_gemm_rows(const Shape& sh, int mode, const GemmParams& g_in, int sms,
                             cudaStream_t s) {
  GemmParams g = g_in;
  attach_counts(g, mode);
  static const int permille = env_int("BOOST_COSCHED", -1);
  static const int row_cost_pct = env_int("BOOST_COSCHED_ROWCOST", 0);
  const int64_t M = g.M;
  const int64_t unit = sh.super_m();
  if (permille == 0 || sh.mcm * sh.mcn < 4 || M < 8 * unit)
    return launch_gemm(sh.bn, mode, sh.cg, sh.mcm, sh.mcn, g, sms, s);
  GemmParams a = g, b = g;
  // the side launch tiles N by single pairs (BN wide); group-aligned because a 2 x 2
  // grouped shape requires groups of a multiple of 512 columns
  if (g.group_tiles > 0) {
    b.group_tiles = static_cast<int32_t>(cdiv(g.group_n, sh.bn));
    b.n_tiles = g.n_tiles / g.group_tiles * b.group_tiles;
  } else {
    b.n_tiles = static_cast<int32_t>(cdiv(g.N, sh.bn));
  }
  auto fixed_split = [&](int64_t pm) {
    const int64_t side_rows = M * pm / 1000 / 256 * 256;
    return side_rows > 0 ? std::min(M, cdiv(M - side_rows, unit) * unit) : M;
  };
  int64_t main_rows = fixed_split(permille > 0 ? permille : 130);
  if (permille < 0) {
    const int64_t r_main = gemm_resident(sh.bn, mode, sh.cg, sh.mcm, sh.mcn, sms);
    const int64_t r_side = (sms - r_main * sh.cg * sh.mcm * sh.mcn) / 2;
    if (r_main > 0 && r_side > 0) {
      int64_t k_tile = 0;   // K of one tile, over its segments (one split's share)
      for (int sg = 0; sg < g.num_seg; ++sg)
        k_tile += static_cast<int64_t>(g.splits > 1 ? g.kb_per_split : g.seg[sg].num_kb) * kBK;
      const int pct = row_cost_pct > 0 ? row_cost_pct
                                       : (k_tile >= 12288 ? 125 : (k_tile >= 1024 ? 150 : 200));
      const double cost = pct / 100.0;
      const int64_t units = static_cast<int64_t>(g.batch) * std::max<int32_t>(g.splits, 1);
      // predicted time (cluster waves) of a split keeping `rows` rows in the cluster launch
      auto waves = [&](int64_t rows) {
        const int64_t side = M - rows;
        const double t_main =
            static_cast<double>(cdiv(units * cdiv(rows, unit) * a.n_tiles, r_main));
        const double t_side =
            side > 0 ? static_cast<double>(cdiv(units * cdiv(side, 256) * b.n_tiles, r_side)) * cost
                     : 0.0;
        return std::max(t_main, t_side);
      };
      double best = 1e300;
      int64_t best_rows = main_rows;
      for (int64_t i = cdiv(M, unit); i * unit * 2 >= M; --i) {
        const int64_t rows = std::min(i * unit, M);
        const double t = waves(rows);
        if (t < best * 0.999) {
          best = t;
          best_rows = rows;
        }
      }
      if (best < 0.98 * waves(main_rows)) main_rows = best_rows;
    }
  }
  if (main_rows >= M) return launch_gemm(sh.bn, mode, sh.cg, sh.mcm, sh.mcn, g, sms, s);
  CoStreams* cs = co_streams();
  if (cs == nullptr) return launch_gemm(sh.bn, mode, sh.cg, sh.mcm, sh.mcn, g, sms, s);
  a.m_base = 0;
  a.m_extent = static_cast<int32_t>(main_rows);
  b.m_base = static_cast<int32_t>(main_rows);
  b.m_extent = static_cast<int32_t>(M - main_rows);
  std::lock_guard<std::mutex> lk(cs->order);
  cudaError_t e = cudaEventRecord(cs->fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs->side, cs->fork, 0);
  if (e == cudaSuccess) e = launch_gemm(sh.bn, mode, sh.cg, sh.mcm, sh.mcn, a, sms, s);
  if (e == cudaSuccess) e = launch_gemm(sh.bn, mode, 2, 1, 1, b, sms, cs->side);
  if (e == cudaSuccess) prof_note_kernels(1);
  if (e == cudaSuccess) e = cudaEventRecord(cs->join, cs->side);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, cs->join, 0);
  return e;
}

// Launch a GEMM whose rows are too few to split (the weight gradients, M = r or d): with
// 2 x 2 clusters, the last output columns run as a CTA-pair launch on the SMs no
// cluster fits, on the side stream. The column split minimises the larger of the two
// launches' wave counts, a pair's 256 x 256 tile costing `cost` cluster super-tile waves
// (a lone pair has no multicast partner and shares L2 with the cluster launch; 1.25
// measured alone). BOOST_COSCHED_COLS sets the cost in percent, 0 turns this off.
cudaError_t launch_gemm_cols(const Shape& sh, int mode, const GemmParams& g_in, int sms,
                             cudaStream_t s) {
  GemmParams g = g_in;
  attach_counts(g, mode);
  static const int cost_pct = env_int("BOOST_COSCHED_COLS", 125);
  const double kPairTileCost = cost_pct / 100.0;
  if (cost_pct <= 0 || sh.mcm * sh.mcn < 4 || g.group_tiles > 0 || g.n_base != 0)
    return launch_gemm(sh.bn, mode, sh.cg, sh.mcm, sh.mcn, g, sms, s);
  const int64_t r_main = gemm_resident(sh.bn, mode, sh.cg, sh.mcm, sh.mcn, sms);
  const int64_t r_side = (sms - r_main * sh.cg * sh.mcm * sh.mcn) / 2;
  const int64_t super_n = sh.super_n();
  const int64_t n_super = cdiv(g.N, super_n);
  if (r_main <= 0 || r_side <= 0 || n_super < 2)
    return launch_gemm(sh.bn, mode, sh.cg, sh.mcm, sh.mcn, g, sms, s);
  const int64_t units = static_cast<int64_t>(g.batch) * g.splits;
  const int64_t m_super = cdiv(g.M, sh.super_m()), m_pair = cdiv(g.M, 256);
  double best = static_cast<double>(cdiv(units * m_super * n_super, r_main));
  int64_t best_nm = n_super;
  for (int64_t nm = 1; nm < n_super; ++nm) {
    const double t_main = static_cast<double>(cdiv(units * m_super * nm, r_main));
    const int64_t side_tiles = units * m_pair * cdiv(g.N - nm * super_n, sh.bn);
    const double t_side = static_cast<double>(cdiv(side_tiles, r_side)) * kPairTileCost;
    const double t = std::max(t_main, t_side);
    if (t < best * 0.999) {
      best = t;
      best_nm = nm;
    }
  }
  if (best_nm == n_super) return launch_gemm(sh.bn, mode, sh.cg, sh.mcm, sh.mcn, g, sms, s);
  CoStreams* cs = co_streams();
  if (cs == nullptr) return launch_gemm(sh.bn, mode, sh.cg, sh.mcm, sh.mcn, g, sms, s);
  GemmParams a = g, b = g;
  a.n_tiles = static_cast<int32_t>(best_nm);
  b.n_base = static_cast<int32_t>(best_nm * super_n);
  b.n_tiles = static_cast<int32_t>(cdiv(g.N - b.n_base, sh.bn));
  std::lock_guard<std::mutex> lk(cs->order);
  cudaError_t e = cudaEventRecord(cs->fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs->side, cs->fork, 0);
  if (e == cudaSuccess) e = launch_gemm(sh.bn, mode, sh.cg, sh.mcm, sh.mcn, a, sms, s);
  if (e == cudaSuccess) e = launch_gemm(sh.bn, mode, 2, 1, 1, b, sms, cs->side);
  if (e == cudaSuccess) prof_note_kernels(1);
  if (e == cudaSuccess) e = cudaEventRecord(cs->join, cs->side);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, cs->join, 0);
  return e;
}

// Independent steps of one call run on two more streams forked from the caller's stream
// and joined back to it (on every exit path) before the call returns: the three
// backward GEMMs after the dual kernel (dB and dA on the extra streams, dx on the
// caller's), and the statistics and the gamma fold before a normed block's GEMMs.
// Each persistent GEMM fills the GPU on its own; running them concurrently lets one's
// last, partly filled wave overlap the next one's start. Off by default
// (BOOST_FORK_STREAMS=1 turns it on): since every GEMM's cluster launch has a
// co-scheduled pair launch on the remaining SMs, concurrent GEMMs mostly contend for
// SMs and cluster placement, and the one-stream order measured faster (7B MLP
// 3.412-3.421 -> 3.384-3.402 ms, 1B block 0.591-0.594 -> 0.582 ms, 13B layer equal,
// 40B pair about 1% slower). Per-device streams and events, created on first use; one
// fork/join at a time.
struct ForkStreams {
  cudaStream_t aux[2] = {nullptr, nullptr};
  cudaEvent_t fork = nullptr, join[2] = {nullptr, nullptr};
  bool ok = false;
  std::mutex order;
};

ForkStreams* fork_streams() {
  static ForkStreams bs[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  ForkStreams& b = bs[dev];
  if (!b.ok) {
    for (int i = 0; i < 2; ++i)
      if (cudaStreamCreateWithFlags(&b.aux[i], cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&b.join[i], cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
      }
    if (cudaEventCreateWithFlags(&b.fork, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    b.ok = true;
  }
  return &b;
}

bool forks_enabled() {
  static const int on = env_int("BOOST_FORK_STREAMS", 0);
  return on != 0;
}

class StreamFork {
 public:
  explicit StreamFork(cudaStream_t s) : s_(s) {
    if (!forks_enabled() || (bs_ = fork_streams()) == nullptr) return;
    lk_ = std::unique_lock<std::mutex>(bs_->order);
    if (cudaEventRecord(bs_->fork, s_) != cudaSuccess ||
        cudaStreamWaitEvent(bs_->aux[0], bs_->fork, 0) != cudaSuccess ||
        cudaStreamWaitEvent(bs_->aux[1], bs_->fork, 0) != cudaSuccess) {
      cudaGetLastError();
      bs_ = nullptr;
      lk_.unlock();
    }
  }
  ~StreamFork() {   // join on every exit path, so the caller's stream orders all of it
    if (bs_ == nullptr) return;
    for (int i = 0; i < 2; ++i) {
      cudaEventRecord(bs_->join[i], bs_->aux[i]);
      cudaStreamWaitEvent(s_, bs_->join[i], 0);
    }
  }
  StreamFork(const StreamFork&) = delete;
  StreamFork& operator=(const StreamFork&) = delete;
  cudaStream_t stream(int i) const { return bs_ != nullptr ? bs_->aux[i] : s_; }

 private:
  cudaStream_t s_;
  ForkStreams* bs_ = nullptr;
  std::unique_lock<std::mutex> lk_;
};

}  // namespace

// =================================================================== C ABI
extern "C" {

const char* boost_status_string(boost_status s) {
  switch (s) {
    case BOOST_OK: return "ok";
    case BOOST_ERR_INVALID_ARG: return "invalid argument";
    case BOOST_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case BOOST_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case BOOST_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case BOOST_ERR_CUDA: return "CUDA runtime error";
    case BOOST_ERR_TIMEOUT: return "device wait timed out";
    case BOOST_ERR_DEVICE_CHECK: return "device consistency check failed";
  }
  return "unknown status";
}

size_t boost_block_workspace_bytes(const boost_block_desc* desc) {
  if (validate_desc(desc) != BOOST_OK) return 0;
  return make_plan(*desc, current_num_sms()).total;
}

boost_status boost_block_ws_init(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr || ws_bytes < sizeof(DeviceError) ||
      (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0)
    return BOOST_ERR_WORKSPACE;
  return cuda_status(
      cudaMemsetAsync(ws, 0, sizeof(DeviceError), static_cast<cudaStream_t>(stream)));
}

boost_status boost_block_layout(const boost_block_desc* desc, int64_t* shard_off,
                                int64_t* group_col_off, int64_t* exchange_elems) {
  boost_status st = validate_desc(desc);
  if (st != BOOST_OK) return st;
  const int32_t S = desc->has_norm ? desc->S : 1;
  if (desc->d % S != 0) return BOOST_ERR_UNSUPPORTED_SHAPE;
  if (shard_off)
    for (int32_t s = 0; s <= S; ++s) shard_off[s] = s * (desc->d / S);
  if (group_col_off)
    for (int64_t i = 0; i <= desc->k; ++i) group_col_off[i] = i * desc->r;
  if (exchange_elems) *exchange_elems = desc->T * (desc->k * desc->r + 1);
  return BOOST_OK;
}

boost_status boost_rmsnorm_stats(const boost_block_desc* desc, const void* x, float* ssq,
                                 float* rstd, void* stream) {
  boost_status st = validate_desc(desc);
  if (st != BOOST_OK) return st;
  if (!desc->has_norm) return BOOST_ERR_INVALID_ARG;
  if (desc->T == 0) return BOOST_OK;
  st = check_ptrs({x, rstd}, {ssq});
  if (st != BOOST_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Plan P = make_plan(*desc, current_num_sms());
  ProfScope ps(s, K_STATS, 0.0, stats_bytes(P, desc->S));
  return cuda_status(launch_rmsnorm_stats(x, desc->T, desc->d, desc->S, desc->eps, ssq, rstd, s));
}

}  // extern "C"

namespace {

// K3, the batched up-projection y[i] = a[:, group i] @ B[i]; with `glu` (k == 2) one
// kernel computes both groups of a tile and also writes h = silu(y[0]) * y[1]. With
// `res` (k == 1) the epilogue adds the residual: y = bf16(bf16(a @ B) + res).
cudaError_t launch_up(const Plan& P, const void* a, const void* B, void* y, void* h, bool glu,
                      DeviceError* err, int sms, cudaStream_t s, const void* res = nullptr) {
  cudaError_t e;
  GemmParams u = base_params(P, err);
  if (!make_map(&u.tmA[0], a, P.r, P.k, P.T, P.r * 2, P.kr * 2, 64, 1, P.up.a_rows()))
    return cudaErrorInvalidValue;   // a tensor map could not be encoded
  if (!make_map(&u.tmB[0], B, P.n, P.r, P.k, P.n * 2, P.r * P.n * 2, 64, 64, 1))
    return cudaErrorInvalidValue;
  u.seg[0].a = OperandView{2, 0, 1, 0};   // a as (r, k, T): K-major, batch = group
  u.seg[0].b = OperandView{0, 1, 2, 1};   // B as (n, r, k): MN-major
  u.seg[0].num_kb = static_cast<int32_t>(cdiv(P.r, kBK));
  u.M = static_cast<int32_t>(P.T);
  u.N = static_cast<int32_t>(P.n);
  u.batch = static_cast<int32_t>(P.k);
  u.n_tiles = static_cast<int32_t>(cdiv(P.n, P.up.super_n()));
  u.m_inner = 0;
  if (glu) {
    // Grouped raster order, 8 rows of super-tiles at a time: with n fastest the gate, up
    // and h tiles streaming through L2 evicted B between rows, and every row re-read all
    // of B from DRAM. Measured on the 7B MLP at 8192 tokens: 290 -> 141 MB of DRAM
    // reads, 260 -> 250 us; groups of 4 and 8 tie in the 16384-token step, 16 is slower.
    static const int up_m_group = env_int("BOOST_UP_MGROUP", 8);
    u.m_group = up_m_group;
  }
  u.out = y;
  u.ldo = P.n;
  u.out_bstride = P.T * P.n;
  if (glu) {
    // one tile list; segment 0 = the gate group into accumulator 0, segment 1 = the up
    // group (same maps, batch index + 1) into accumulator 1
    u.batch = 1;
    u.num_seg = 2;
    u.seg[1] = u.seg[0];
    u.seg[1].batch_add = 1;
    u.tmA[1] = u.tmA[0];
    u.tmB[1] = u.tmB[0];
    u.out2 = h;
    set_out_maps(u, P.T, P.n, 2, 1);
    // the fused epilogue stores gate, up and h only through these maps
    if (u.tma_out != 3) return cudaErrorInvalidValue;
    ProfScope ps(s, K_UP_GLU, 2.0 * P.T * P.kr * P.n,
                 2.0 * (P.T * P.kr + P.kr * P.n + P.k * P.T * P.n + P.T * P.n));
    e = launch_gemm_rows(P.up, EPI_UPGLU, u, sms, s);
  } else {
    // with a short K the epilogue's stores weigh most: store them through TMA
    // (the residual is read by the plain-store epilogue)
    static const int tma_up_max_r = env_int("BOOST_TMA_UP_MAX_R", 512);
    const bool tma = P.r <= tma_up_max_r && res == nullptr;
    if (tma) set_out_maps(u, P.T, P.n, P.k);
    u.res = static_cast<const __nv_bfloat16*>(res);
    u.ldr = P.n;
    ProfScope ps(s, K_UP, 2.0 * P.T * P.kr * P.n,
                 2.0 * (P.T * P.kr + P.kr * P.n + P.k * P.T * P.n * (res ? 2 : 1)));
    e = launch_gemm_rows(P.up, tma ? EPI_BF16T : EPI_BF16, u, sms, s);
  }
  return e;
}

// Forward of one block. With `glu` (k == 2: gate and up groups) the up-projection
// computes both groups of a tile in one kernel and its epilogue also writes
// h = silu(gate) * up. With `payload` non-NULL the down-projection runs as the explicit
// emulation of the bottleneck-aware TP exchange: per-shard partial products and sums
// of squares into the payload, then the reduction that stands in for the all-reduce.
boost_status block_fwd_impl(const boost_block_desc* desc, const void* x, const void* gamma,
                            const void* A, const void* B, void* y, void* h, bool glu,
                            float* rstd, float* payload, bool btp, void* ws, size_t ws_bytes,
                            void* stream, const void* res = nullptr, bool with_res = false) {
  boost_status st = validate_desc(desc);
  if (st != BOOST_OK) return st;
  const boost_block_desc& D = *desc;
  if (!D.has_norm && (gamma != nullptr || rstd != nullptr)) return BOOST_ERR_INVALID_ARG;
  if (glu && D.k != 2) return BOOST_ERR_INVALID_ARG;
  if (with_res) {
    // y = res + block(x): one output group, res shaped like it
    if (D.k != 1 || (D.T > 0 && res == nullptr)) return BOOST_ERR_INVALID_ARG;
    if (res != nullptr && !aligned16(res)) return BOOST_ERR_ALIGNMENT;
    // the epilogue reads each residual element before writing the same output element,
    // so res may be y itself, but not a shifted view of it
    if (res != nullptr && y != nullptr &&
        partial_overlap(res, y, 2ull * static_cast<uint64_t>(D.T) * static_cast<uint64_t>(D.n)))
      return BOOST_ERR_INVALID_ARG;
  }
  // With no tokens the [T, ...] tensors are empty and may be NULL.
  st = D.T == 0 ? check_ptrs({A, B}, {gamma, rstd, x, y, h})
                : check_ptrs({x, A, B, y}, {gamma, rstd, h});
  if (st != BOOST_OK) return st;
  if (glu && D.T > 0 && h == nullptr) return BOOST_ERR_INVALID_ARG;
  if (D.has_norm && gamma == nullptr) return BOOST_ERR_INVALID_ARG;
  if (btp) {
    // every shard is a whole number of the GEMM's 64-deep k-blocks
    if (D.d % D.S != 0 || (D.d / D.S) % kBK != 0) return BOOST_ERR_UNSUPPORTED_SHAPE;
    if (D.T > 0 && payload == nullptr) return BOOST_ERR_INVALID_ARG;
    if (payload != nullptr && !aligned16(payload)) return BOOST_ERR_ALIGNMENT;
  }
  const int sms = current_num_sms();
  const Plan P = make_plan(D, sms);
  st = check_ws(ws, ws_bytes, P.total);
  if (st != BOOST_OK) return st;
  if (D.T == 0) return BOOST_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceError* err = ws_at<DeviceError>(ws, 0);

  const void* Ap = A;
  float* rs = nullptr;
  float* zpart = payload;                                   // [S, T, kr]
  float* ssq_x = btp && D.has_norm ? payload + D.S * D.T * P.kr : nullptr;   // [S, T]
  if (D.has_norm && !forks_enabled()) {
    // the statistics and the fold in one launch (under the emulated exchange the shard
    // sums of squares go into the payload)
    rs = rstd ? rstd : ws_at<float>(ws, P.off_rstd);
    ProfScope ps(s, K_STATS_FOLD, 0.0, stats_bytes(P, D.S) + fold_bytes(P));
    if (launch_stats_fold(x, D.T, D.d, D.S, D.eps, btp ? ssq_x : ws_at<float>(ws, P.off_ssq),
                          btp ? ws_at<float>(ws, P.off_rstd) : rs, gamma, A,
                          ws_at<void>(ws, P.off_Ap), P.kr, s) != cudaSuccess)
      return BOOST_ERR_CUDA;
    Ap = ws_at<void>(ws, P.off_Ap);
  } else if (D.has_norm) {
    rs = rstd ? rstd : ws_at<float>(ws, P.off_rstd);
    cudaError_t e;
    StreamFork fork(s);   // the fold runs beside the statistics
    {
      // (under the emulated exchange the shard sums of squares go into the payload; the
      // row scale is formed again after the reduction, from the exchanged sums)
      ProfScope ps(s, K_STATS, 0.0, stats_bytes(P, D.S));
      e = launch_rmsnorm_stats(x, D.T, D.d, D.S, D.eps,
                               btp ? ssq_x : ws_at<float>(ws, P.off_ssq),
                               btp ? ws_at<float>(ws, P.off_rstd) : rs, s);
    }
    if (e != cudaSuccess) return BOOST_ERR_CUDA;
    {
      ProfScope ps(fork.stream(0), K_FOLD, 0.0, fold_bytes(P));
      e = launch_fold_gamma(gamma, A, ws_at<void>(ws, P.off_Ap), D.d, P.kr, fork.stream(0));
    }
    if (e != cudaSuccess) return BOOST_ERR_CUDA;
    Ap = ws_at<void>(ws, P.off_Ap);
  }   // joined: the down-projection needs both
  void* a = ws_at<void>(ws, P.off_a);

  GemmParams g = base_params(P, err);
  if (!down_segment(g, P, x, Ap, P.down, P.tpg_down)) return BOOST_ERR_CUDA;
  cudaError_t e;
  if (!btp) {
    // K2: a = act(s * (x @ A')) over all k groups in one GEMM.
    g.act = D.act;
    g.rstd = rs;
    g.out = a;
    g.ldo = P.kr;
    ProfScope ps(s, K_DOWN, 2.0 * P.T * P.d * P.kr,
                 2.0 * (P.T * P.d + P.d * P.kr + P.T * P.kr) + 4.0 * P.T);
    e = launch_gemm_rows(P.down, EPI_ACT, g, sms, s);
  } else {
    // Each shard's unscaled partial product x[:, shard] @ A'[shard, :] (a split-K GEMM
    // whose splits are the shards), then the reduction over the shards that stands in
    // for the all-reduce, with the deferred row scale and the activation after it.
    g.splits = D.S;
    g.kb_per_split = static_cast<int32_t>(D.d / D.S / kBK);
    g.out = zpart;
    g.ldo = P.kr;
    g.out_sstride = D.T * P.kr;
    {
      ProfScope ps(s, K_BTP_PARTIAL, 2.0 * P.T * P.d * P.kr,
                   2.0 * (P.T * P.d + P.d * P.kr) + 4.0 * D.S * P.T * P.kr);
      e = launch_gemm_rows(P.down, EPI_F32, g, sms, s);
    }
    if (e == cudaSuccess) {
      ProfScope ps(s, K_BTP_REDUCE, 0.0,
                   4.0 * D.S * P.T * (P.kr + (D.has_norm ? 1 : 0)) + 2.0 * P.T * P.kr +
                       (D.has_norm ? 4.0 * P.T : 0.0));
      e = launch_btp_reduce(zpart, ssq_x, static_cast<int>(D.S), D.T, P.kr, D.d, D.eps, D.act, a,
                            D.has_norm ? rs : nullptr, s);
    }
  }
  if (e != cudaSuccess) return BOOST_ERR_CUDA;

  // K3: y[i] = a[:, group i] @ B[i], batched over the k groups (plus the residual).
  e = launch_up(P, a, B, y, h, glu, err, sms, s, with_res ? res : nullptr);
  return cuda_status(e);
}

}  // namespace

extern "C" {

boost_status boost_block_fwd(const boost_block_desc* desc, const void* x, const void* gamma,
                             const void* A, const void* B, void* y, float* rstd, void* ws,
                             size_t ws_bytes, void* stream) {
  return block_fwd_impl(desc, x, gamma, A, B, y, nullptr, false, rstd, nullptr, false, ws,
                        ws_bytes, stream);
}

boost_status boost_block_up(const boost_block_desc* desc, const void* a, const void* B, void* y,
                            void* h, void* ws, size_t ws_bytes, void* stream) {
  boost_status st = validate_desc(desc);
  if (st != BOOST_OK) return st;
  const boost_block_desc& D = *desc;
  const bool glu = h != nullptr;
  if (glu && D.k != 2) return BOOST_ERR_INVALID_ARG;
  st = D.T == 0 ? check_ptrs({B}, {a, y, h}) : check_ptrs({a, B, y}, {h});
  if (st != BOOST_OK) return st;
  const int sms = current_num_sms();
  const Plan P = make_plan(D, sms);
  st = check_ws(ws, ws_bytes, P.total);
  if (st != BOOST_OK) return st;
  if (D.T == 0) return BOOST_OK;
  const cudaError_t e = launch_up(P, a, B, y, h, glu, ws_at<DeviceError>(ws, 0), sms,
                                  static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

boost_status boost_block_fwd_btp(const boost_block_desc* desc, const void* x, const void* gamma,
                                 const void* A, const void* B, void* y, float* rstd,
                                 float* payload, void* ws, size_t ws_bytes, void* stream) {
  return block_fwd_impl(desc, x, gamma, A, B, y, nullptr, false, rstd, payload, true, ws,
                        ws_bytes, stream);
}

boost_status boost_block_fwd_swiglu(const boost_block_desc* desc, const void* x,
                                    const void* gamma, const void* A, const void* B, void* y,
                                    void* h, float* rstd, void* ws, size_t ws_bytes,
                                    void* stream) {
  return block_fwd_impl(desc, x, gamma, A, B, y, h, true, rstd, nullptr, false, ws, ws_bytes,
                        stream);
}

boost_status boost_block_fwd_residual(const boost_block_desc* desc, const void* x,
                                      const void* gamma, const void* A, const void* B,
                                      const void* res, void* y, float* rstd, void* ws,
                                      size_t ws_bytes, void* stream) {
  return block_fwd_impl(desc, x, gamma, A, B, y, nullptr, false, rstd, nullptr, false, ws,
                        ws_bytes, stream, res, true);
}

}  // extern "C"

namespace {

// Backward of one block. With `gate` non-NULL the block's input is h = silu(gate) * up
// (no norm) and, instead of dx, its dgrad epilogue writes dgate and dup.
boost_status block_bwd_impl(const boost_block_desc* desc, const void* x, const void* gamma,
                            const void* A, const void* B, const float* rstd, const void* dy,
                            void* dx, void* dgamma, void* dA, void* dB, const void* gate,
                            const void* up, void* dgate, void* dup, void* ws, size_t ws_bytes,
                            void* stream, const void* dx_res = nullptr, bool with_res = false) {
  boost_status st = validate_desc(desc);
  if (st != BOOST_OK) return st;
  const boost_block_desc& D = *desc;
  if (with_res) {
    // dx = res + the block's input gradient (res shaped like dx)
    if (gate != nullptr || (D.T > 0 && dx_res == nullptr)) return BOOST_ERR_INVALID_ARG;
    if (dx_res != nullptr && !aligned16(dx_res)) return BOOST_ERR_ALIGNMENT;
    if (dx_res != nullptr && dx != nullptr &&
        partial_overlap(dx_res, dx, 2ull * static_cast<uint64_t>(D.T) * static_cast<uint64_t>(D.d)))
      return BOOST_ERR_INVALID_ARG;
  }
  const bool glu = gate != nullptr;
  if (!D.has_norm && (gamma != nullptr || rstd != nullptr || dgamma != nullptr))
    return BOOST_ERR_INVALID_ARG;
  if (glu) {
    if (D.has_norm) return BOOST_ERR_INVALID_ARG;
    st = D.T == 0 ? check_ptrs({A, B, dA, dB}, {x, dy, gate, up, dgate, dup})
                  : check_ptrs({x, A, B, dy, gate, up, dgate, dup, dA, dB}, {});
  } else {
    st = D.T == 0 ? check_ptrs({A, B, dA, dB}, {gamma, rstd, dgamma, x, dy, dx})
                  : check_ptrs({x, A, B, dy, dx, dA, dB}, {gamma, rstd, dgamma});
  }
  if (st != BOOST_OK) return st;
  if (D.has_norm && (gamma == nullptr || dgamma == nullptr)) return BOOST_ERR_INVALID_ARG;
  const int sms = current_num_sms();
  const Plan P = make_plan(D, sms);
  st = check_ws(ws, ws_bytes, P.total);
  if (st != BOOST_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D.T == 0) {  // no tokens: weight gradients are zero, dx is empty
    cudaError_t e = cudaMemsetAsync(dA, 0, 2ull * D.d * P.kr, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, 2ull * D.k * D.r * D.n, s);
    if (e == cudaSuccess && dgamma) e = cudaMemsetAsync(dgamma, 0, 2ull * D.d, s);
    return cuda_status(e);
  }
  DeviceError* err = ws_at<DeviceError>(ws, 0);

  const void* Ap = A;
  const float* rs = nullptr;
  if (D.has_norm && rstd == nullptr && !forks_enabled()) {
    // the row scale recomputed: the statistics and the fold in one launch
    float* r = ws_at<float>(ws, P.off_rstd);
    ProfScope ps(s, K_STATS_FOLD, 0.0, stats_bytes(P, D.S) + fold_bytes(P));
    if (launch_stats_fold(x, D.T, D.d, D.S, D.eps, ws_at<float>(ws, P.off_ssq), r, gamma, A,
                          ws_at<void>(ws, P.off_Ap), P.kr, s) != cudaSuccess)
      return BOOST_ERR_CUDA;
    rs = r;
    Ap = ws_at<void>(ws, P.off_Ap);
  } else if (D.has_norm) {
    std::unique_ptr<StreamFork> fork;   // the fold beside the statistics, when both run
    cudaStream_t sf = s;
    if (rstd == nullptr) {
      fork = std::make_unique<StreamFork>(s);
      sf = fork->stream(0);
      float* r = ws_at<float>(ws, P.off_rstd);
      ProfScope ps(s, K_STATS, 0.0, stats_bytes(P, D.S));
      if (launch_rmsnorm_stats(x, D.T, D.d, D.S, D.eps, ws_at<float>(ws, P.off_ssq), r, s) !=
          cudaSuccess)
        return BOOST_ERR_CUDA;
      rs = r;
    } else {
      rs = rstd;
    }
    {
      ProfScope ps(sf, K_FOLD, 0.0, fold_bytes(P));
      if (launch_fold_gamma(gamma, A, ws_at<void>(ws, P.off_Ap), D.d, P.kr, sf) != cudaSuccess)
        return BOOST_ERR_CUDA;
    }
    Ap = ws_at<void>(ws, P.off_Ap);
  }   // joined before the dual kernel
  void* a = ws_at<void>(ws, P.off_a);
  void* dzs = ws_at<void>(ws, P.off_dzs);
  float* qpart = ws_at<float>(ws, P.off_q);

  // K4: per tile two accumulators, z (recomputed, K = d) and dy_i @ B_i^T (K = n).
  GemmParams g = base_params(P, err);
  if (!down_segment(g, P, x, Ap, P.dual, P.tpg_dual)) return BOOST_ERR_CUDA;
  if (!make_map(&g.tmA[1], dy, P.n, P.T, P.k, P.n * 2, P.T * P.n * 2, 64, P.dual.a_rows(), 1))
    return BOOST_ERR_CUDA;
  if (!make_map(&g.tmB[1], B, P.n, P.r, P.k, P.n * 2, P.r * P.n * 2, 64, P.dual.b_rows(), 1))
    return BOOST_ERR_CUDA;
  g.num_seg = 2;
  g.seg[1].a = OperandView{1, 0, 2, 0};   // dy as (n, T, k): K-major, batch = group
  g.seg[1].b = OperandView{1, 0, 2, 0};   // B as (n, r, k): K-major rows of B_i
  g.seg[1].num_kb = static_cast<int32_t>(cdiv(P.n, kBK));
  g.seg[1].batch_from_n = 1;
  g.seg[1].b_n_local = 1;
  g.act = D.act;
  g.rstd = rs;
  g.out = a;
  g.out2 = dzs;
  g.ldo = P.kr;
  g.qpart = D.has_norm ? qpart : nullptr;
  // With a short K the epilogue weighs more: store a and dzs through TMA. Measured:
  // 1B block (K = 2048 + 2048) dual 1251 -> 1281 TFLOP/s; long K keeps plain stores.
  static const int tma_dual_max_k = env_int("BOOST_TMA_DUAL_MAX_K", 4096);
  const bool dual_tma = P.d + P.n <= tma_dual_max_k;
  if (dual_tma) set_out_maps(g, P.T, P.kr, 1, 1);
  // rows of super-tiles per group of a grouped raster order (m fastest within a group);
  // 0 or 1: n fastest
  static const int dual_m_group = env_int("BOOST_DUAL_MGROUP", 0);
  g.m_group = dual_m_group;
  cudaError_t e;
  {
    ProfScope ps(s, K_DUAL, 2.0 * P.T * P.kr * (P.d + P.n),
                 2.0 * (P.T * P.d + P.d * P.kr + P.k * P.T * P.n + P.kr * P.n + 2 * P.T * P.kr) +
                     4.0 * P.T * (P.n_cols_dual + 1));
    e = launch_gemm_rows(P.dual, dual_tma ? EPI_DUALT : EPI_DUAL, g, sms, s);
  }
  if (e != cudaSuccess) return BOOST_ERR_CUDA;

  StreamFork fork(s);
  const double wB_flops = 2.0 * P.T * P.kr * P.n;
  const double wB_bytes = 2.0 * (P.T * P.kr + P.k * P.T * P.n + P.kr * P.n);
  const double wA_flops = 2.0 * P.T * P.d * P.kr;
  const double wA_bytes = 2.0 * (P.T * P.d + P.T * P.kr + P.d * P.kr) +
                          (D.has_norm ? 2.0 * (P.d * P.kr + 2 * P.d) : 0.0);

  // K5: dB[i] = a[:, group i]^T @ dy[i]  (M = r, N = n, K = T).
  {
    const cudaStream_t sb = fork.stream(0);
    float* part = ws_at<float>(ws, P.off_partB);
    GemmParams w = base_params(P, err);
    if (!make_map(&w.tmA[0], a, P.r, P.k, P.T, P.r * 2, P.kr * 2, 64, 1, 64)) return BOOST_ERR_CUDA;
    if (!make_map(&w.tmB[0], dy, P.n, P.T, P.k, P.n * 2, P.T * P.n * 2, 64, 64, 1))
      return BOOST_ERR_CUDA;
    w.seg[0].a = OperandView{0, 2, 1, 1};  // a as (r, k, T): MN-major, K = T
    w.seg[0].b = OperandView{0, 1, 2, 1};  // dy as (n, T, k): MN-major, K = T
    w.seg[0].num_kb = static_cast<int32_t>(cdiv(P.T, kBK));
    w.M = static_cast<int32_t>(P.r);
    w.N = static_cast<int32_t>(P.n);
    w.batch = static_cast<int32_t>(P.k);
    w.n_tiles = static_cast<int32_t>(cdiv(P.n, P.wB.super_n()));
    w.m_inner = inner_m(P.r, P.n, P.wB);
    w.ldo = P.n;
    w.out_bstride = P.r * P.n;
    if (P.splits_B > 1) {
      w.splits = P.splits_B;
      w.kb_per_split = P.kbps_B;
      w.out = part;
      w.out_sstride = P.k * P.r * P.n;
      {
        ProfScope ps(sb, K_WGRAD_B, wB_flops, wB_bytes);
        e = launch_gemm_cols(P.wB, EPI_F32, w, sms, sb);
      }
      if (e == cudaSuccess) {
        ProfScope ps(sb, K_SPLITK_SUM, 0.0, (4.0 * P.splits_B + 2.0) * P.kr * P.n);
        e = launch_splitk_sum_bf16(part, P.splits_B, P.k * P.r * P.n, dB, sb);
      }
    } else {
      w.out = dB;
      ProfScope ps(sb, K_WGRAD_B, wB_flops, wB_bytes);
      e = launch_gemm_cols(P.wB, EPI_BF16, w, sms, sb);
    }
    if (e != cudaSuccess) return BOOST_ERR_CUDA;
  }

  // K6: G = x^T @ dzs (M = d, N = k*r, K = T); dA = gamma (.) G, dgamma = rowsum(A (.) G).
  {
    const cudaStream_t sa = fork.stream(1);
    float* part = ws_at<float>(ws, P.off_partA);
    GemmParams w = base_params(P, err);
    if (!map_2d(&w.tmA[0], x, P.T, P.d, 64, 64)) return BOOST_ERR_CUDA;
    if (!map_2d(&w.tmB[0], dzs, P.T, P.kr, 64, 64)) return BOOST_ERR_CUDA;
    w.seg[0].a = mnmajor_2d();
    w.seg[0].b = mnmajor_2d();
    w.seg[0].num_kb = static_cast<int32_t>(cdiv(P.T, kBK));
    w.M = static_cast<int32_t>(P.d);
    w.N = static_cast<int32_t>(P.kr);
    w.n_tiles = static_cast<int32_t>(cdiv(P.kr, P.wA.super_n()));
    w.m_inner = inner_m(P.d, P.kr, P.wA);
    w.ldo = P.kr;
    if (P.splits_A > 1) {
      w.splits = P.splits_A;
      w.kb_per_split = P.kbps_A;
      w.out = part;
      w.out_sstride = P.d * P.kr;
      {
        ProfScope ps(sa, K_WGRAD_A, wA_flops, wA_bytes);
        e = launch_gemm_cols(P.wA, EPI_F32, w, sms, sa);
      }
      if (e == cudaSuccess) {
        ProfScope ps(sa, K_FINALIZE_DA, 0.0, (4.0 * P.splits_A + 4.0) * P.d * P.kr + 4.0 * P.d);
        e = launch_splitk_finalize_dA(part, P.splits_A, P.d, P.kr, D.has_norm ? gamma : nullptr,
                                      A, dA, D.has_norm ? dgamma : nullptr, sa);
      }
    } else {
      w.out = dA;
      w.gamma = D.has_norm ? static_cast<const __nv_bfloat16*>(gamma) : nullptr;
      w.wA = D.has_norm ? static_cast<const __nv_bfloat16*>(A) : nullptr;
      w.dgpart = D.has_norm ? ws_at<float>(ws, P.off_dg) : nullptr;
      {
        ProfScope ps(sa, K_WGRAD_A, wA_flops, wA_bytes);
        e = launch_gemm_cols(P.wA, EPI_DA, w, sms, sa);
      }
      if (e == cudaSuccess && D.has_norm) {
        ProfScope ps(sa, K_DGAMMA, 0.0, 4.0 * P.n_cols_wA * P.d + 2.0 * P.d);
        e = launch_dgamma_reduce(ws_at<float>(ws, P.off_dg), P.n_cols_wA, P.d, dgamma, sa);
      }
    }
    if (e != cudaSuccess) return BOOST_ERR_CUDA;
  }

  // K7: dx = dzs @ A'^T - (s^2 q / d) x  (M = T, N = d, K = k*r).
  {
    GemmParams w = base_params(P, err);
    if (!map_2d(&w.tmA[0], dzs, P.T, P.kr, 64, P.dx.a_rows())) return BOOST_ERR_CUDA;
    if (!map_2d(&w.tmB[0], Ap, P.d, P.kr, 64, P.dx.b_rows())) return BOOST_ERR_CUDA;
    w.seg[0].a = kmajor_2d();
    w.seg[0].b = kmajor_2d();
    w.seg[0].num_kb = static_cast<int32_t>(cdiv(P.kr, kBK));
    w.M = static_cast<int32_t>(P.T);
    w.N = static_cast<int32_t>(P.d);
    w.n_tiles = static_cast<int32_t>(cdiv(P.d, P.dx.super_n()));
    w.m_inner = 0;
    w.out = dx;
    w.ldo = P.d;
    if (with_res) {
      w.res = static_cast<const __nv_bfloat16*>(dx_res);
      w.ldr = P.d;
    }
    if (glu) {
      w.out = dgate;
      w.out2 = dup;
      set_out_maps(w, P.T, P.d, 1, 1);
      // the SwiGLU backward stores dgate and dup only through these maps
      if (w.tma_out != 3) return BOOST_ERR_CUDA;
      // the epilogue streams gate and up through TMA (required by this mode)
      if (!make_map(&w.tmE[0], gate, P.d, P.T, 1, P.d * 2, P.T * P.d * 2, 32, 32, 1, true) ||
          !make_map(&w.tmE[1], up, P.d, P.T, 1, P.d * 2, P.T * P.d * 2, 32, 32, 1, true))
        return BOOST_ERR_CUDA;
      w.tma_in = 1;
    }
    if (D.has_norm) {
      w.rstd = rs;
      w.qpart = qpart;
      w.nq = P.n_cols_dual;
      w.d_norm = static_cast<int32_t>(P.d);
      // the RMSNorm term's x streams through TMA
      if (!make_map(&w.tmE[0], x, P.d, P.T, 1, P.d * 2, P.T * P.d * 2, 32, 32, 1, true))
        return BOOST_ERR_CUDA;
      w.tma_in = 1;
    }
    ProfScope ps(s, glu ? K_DX_GLU : K_DX, 2.0 * P.T * P.kr * P.d,
                 2.0 * (P.T * P.kr + P.d * P.kr +
                        P.T * P.d * (glu ? 4 : (D.has_norm ? 2 : 1) + (with_res ? 1 : 0))) +
                     4.0 * P.T * (P.n_cols_dual + 1));
    e = launch_gemm_rows(P.dx, glu ? EPI_GLU : EPI_DX, w, sms, s);
  }
  return cuda_status(e);
}

}  // namespace

extern "C" {

boost_status boost_block_bwd(const boost_block_desc* desc, const void* x, const void* gamma,
                             const void* A, const void* B, const float* rstd, const void* dy,
                             void* dx, void* dgamma, void* dA, void* dB, void* ws,
                             size_t ws_bytes, void* stream) {
  return block_bwd_impl(desc, x, gamma, A, B, rstd, dy, dx, dgamma, dA, dB, nullptr, nullptr,
                        nullptr, nullptr, ws, ws_bytes, stream);
}

boost_status boost_block_bwd_residual(const boost_block_desc* desc, const void* x,
                                      const void* gamma, const void* A, const void* B,
                                      const float* rstd, const void* dy, const void* res,
                                      void* dx, void* dgamma, void* dA, void* dB, void* ws,
                                      size_t ws_bytes, void* stream) {
  return block_bwd_impl(desc, x, gamma, A, B, rstd, dy, dx, dgamma, dA, dB, nullptr, nullptr,
                        nullptr, nullptr, ws, ws_bytes, stream, res, true);
}

boost_status boost_block_bwd_swiglu(const boost_block_desc* desc, const void* h, const void* A,
                                    const void* B, const void* dy, const void* gate,
                                    const void* up, void* dgate, void* dup, void* dA, void* dB,
                                    void* ws, size_t ws_bytes, void* stream) {
  if (gate == nullptr) return BOOST_ERR_INVALID_ARG;
  return block_bwd_impl(desc, h, nullptr, A, B, nullptr, dy, nullptr, nullptr, dA, dB, gate, up,
                        dgate, dup, ws, ws_bytes, stream);
}

boost_status boost_block_ws_layout(const boost_block_desc* desc, size_t* off_a, size_t* off_dzs,
                                   size_t* off_Ap, size_t* off_rstd) {
  boost_status st = validate_desc(desc);
  if (st != BOOST_OK) return st;
  const Plan P = make_plan(*desc, current_num_sms());
  if (off_a) *off_a = P.off_a;
  if (off_dzs) *off_dzs = P.off_dzs;
  if (off_Ap) *off_Ap = P.off_Ap;
  if (off_rstd) *off_rstd = P.off_rstd;
  return BOOST_OK;
}

boost_status boost_debug_count_writes(int32_t* counts, int64_t capacity) {
  if (counts != nullptr && (capacity <= 0 || !aligned16(counts))) return BOOST_ERR_INVALID_ARG;
  WriteCounter& w = write_counter();
  std::lock_guard<std::mutex> lk(w.mu);
  w.base = counts;
  w.capacity = counts != nullptr ? capacity : 0;
  if (counts != nullptr) {
    w.cursor = 0;
    w.overflow = false;
    w.log.clear();
  }
  return BOOST_OK;
}

int64_t boost_debug_count_log(int64_t* log, int64_t max_ops) {
  WriteCounter& w = write_counter();
  std::lock_guard<std::mutex> lk(w.mu);
  if (w.overflow) return -1;
  const int64_t ops = static_cast<int64_t>(w.log.size()) / kLogFields;
  if (log != nullptr)
    for (int64_t i = 0; i < std::min(ops, max_ops) * kLogFields; ++i) log[i] = w.log[i];
  return ops;
}

boost_status boost_block_check(void* ws, void* stream) {
  if (ws == nullptr) return BOOST_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return BOOST_ERR_CUDA;
  DeviceError h;
  e = cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return BOOST_ERR_CUDA;
  if (h.code != 0) {
    DeviceError z{};
    cudaMemcpy(ws, &z, sizeof(z), cudaMemcpyHostToDevice);
    if (h.code == kErrTimeout) return BOOST_ERR_TIMEOUT;
    return BOOST_ERR_DEVICE_CHECK;
  }
  return BOOST_OK;
}

boost_status boost_swiglu_fwd(int64_t T, int64_t n, const void* gate, const void* up, void* h,
                              void* stream) {
  if (T < 0 || n < 0) return BOOST_ERR_INVALID_ARG;
  if (n % 8) return BOOST_ERR_UNSUPPORTED_SHAPE;
  if (T * n == 0) return BOOST_OK;
  boost_status st = check_ptrs({gate, up, h}, {});
  if (st != BOOST_OK) return st;
  ProfScope ps(static_cast<cudaStream_t>(stream), K_SWIGLU_FWD, 0.0, 6.0 * T * n);
  return cuda_status(launch_swiglu_fwd(gate, up, h, T * n, static_cast<cudaStream_t>(stream)));
}

boost_status boost_swiglu_bwd(int64_t T, int64_t n, const void* gate, const void* up,
                              const void* dh, void* dgate, void* dup, void* stream) {
  if (T < 0 || n < 0) return BOOST_ERR_INVALID_ARG;
  if (n % 8) return BOOST_ERR_UNSUPPORTED_SHAPE;
  if (T * n == 0) return BOOST_OK;
  boost_status st = check_ptrs({gate, up, dh, dgate, dup}, {});
  if (st != BOOST_OK) return st;
  ProfScope ps(static_cast<cudaStream_t>(stream), K_SWIGLU_BWD, 0.0, 10.0 * T * n);
  return cuda_status(
      launch_swiglu_bwd(gate, up, dh, dgate, dup, T * n, static_cast<cudaStream_t>(stream)));
}

boost_status boost_add(int64_t count, const void* a, const void* b, void* out, void* stream) {
  if (count < 0) return BOOST_ERR_INVALID_ARG;
  if (count % 8) return BOOST_ERR_UNSUPPORTED_SHAPE;
  if (count == 0) return BOOST_OK;
  boost_status st = check_ptrs({a, b, out}, {});
  if (st != BOOST_OK) return st;
  ProfScope ps(static_cast<cudaStream_t>(stream), K_ADD, 0.0, 6.0 * count);
  return cuda_status(launch_add(a, b, out, count, static_cast<cudaStream_t>(stream)));
}

boost_status boost_debug_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us,
                                      void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return BOOST_ERR_INVALID_ARG;
  boost_status st = check_ws(ws, ws_bytes, sizeof(DeviceError));
  if (st != BOOST_OK) return st;
  return cuda_status(launch_wait_timeout_probe(ws_at<DeviceError>(ws, 0),
                                               static_cast<uint64_t>(limit_us) * 1000ull,
                                               static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
