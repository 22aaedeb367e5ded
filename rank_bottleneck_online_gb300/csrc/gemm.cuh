// gemm.cuh -- persistent, warp-specialised tcgen05 GEMM engine for sm_103a with the
// bottleneck block's fused epilogues.
//
// One CTA per SM walks a static list of output tiles (128*CG x BN). Roles:
//   warp 0, lane 0 : TMA producer; fills a ring of shared-memory stages
//                    (A tile 128x64, B tile (BN/CG)x64, bf16, 128-byte swizzle)
//   warp 1         : allocates TMEM; lane 0 (of the even CTA when CG = 2) issues
//                    tcgen05.mma (M=128*CG, N=BN, K=16) into a TMEM accumulator and
//                    commits the stage / accumulator barriers
//   warps 2..9     : epilogue; tcgen05.ld of the accumulator (two warps per TMEM lane
//                    quarter taking alternate 32-column chunks, one output row per
//                    thread), fused math, stores through per-warp shared-memory
//                    staging (coalesced plain stores, or TMA bulk stores in the SwiGLU
//                    modes), epilogue inputs (x, gate, up) streamed in by TMA
// CG = 2 runs each tile on a CTA pair (a cluster of two SMs, tcgen05 cta_group::2):
// each SM stages its own 128 rows of A and half of the BN rows of B, so the operand
// bytes each SM moves per MMA flop are 2/3 of the single-SM tile's. The even CTA
// issues the MMAs; both CTAs' loads complete on its stage barriers, and its commits
// are multicast to both CTAs.
// MCM x MCN pairs form one cluster (2, 4 or 8 CTAs) covering a (256*MCM) x (BN*MCN)
// super-tile. Pairs in the same column (along M) need the same B rows and pairs in the
// same row (along N) the same A rows, so each CTA loads one 64-row slice of its shared
// operand and multicasts it to the CTAs that share it: MCM = 2 saves a quarter and
// MCM = MCN = 2 half of the L2->SM bytes per MMA flop. A stage is refilled once every
// pair of the cluster has released it.
// Accumulators are double-buffered in TMEM so the epilogue of tile i overlaps the
// mainloop of tile i+1, except with two 256-column accumulators per tile (EPI_DUAL,
// EPI_DUALT, EPI_UPGLU), which fill TMEM; EPI_UPGLU then frees each accumulator as
// soon as it has been read into registers, before its stores. A launch may cover a
// row range (m_base, m_extent) or start at a column (n_base) of the output, so that
// two launches of different cluster shapes can share one GEMM. Every mbarrier wait is
// bounded (ptx.cuh).
//
// Operands are described by "views" of 3-D tensor maps: which map dimension
// carries the MN index, which the K index and which the batch index, and whether
// the operand is K-major (K contiguous) or MN-major (MN contiguous). This lets one
// kernel read x, a, dzs, dy and the weights in their natural row-major layouts,
// including transposed uses (x^T, a^T, dy^T) without any transpose pass.
#pragma once

#include <cuda.h>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace boost_gb300 {

constexpr int kBM = 128;           // rows per tile (TMEM lanes)
constexpr int kBK = 64;            // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kUmmaK = 16;         // K per tcgen05.mma (kind::f16)
// Epilogue warps: kEpiWarps (two per TMEM lane quarter, alternating 32-column chunks).
// The SwiGLU-backward mode takes kGluEpiWarps (CTA pairs only); 12 (three per quarter,
// 128 registers a thread) measured slower than 8 on the 7B MLP: the extra staging cost
// the mainloop an operand stage (5 -> 4). Modes that write per-row partial sums (one row
// per column tile and warp of a lane quarter) keep kEpiWarps, which the host sizes those
// partials with.
constexpr int kEpiWarps = 8;
constexpr int kEpiHalves = kEpiWarps / 4;
#ifndef BOOST_GLU_EPI_WARPS
#define BOOST_GLU_EPI_WARPS 8
#endif
// SwiGLU backward: outputs written over their own inputs in the loader's slots (two
// slots per warp, no separate store ring); 0 keeps one input slot and two store slots.
#ifndef BOOST_GLU_IN_PLACE
#define BOOST_GLU_IN_PLACE 1
#endif
// Dual recompute + dgrad: the bottleneck activation a = act(s z) is formed and stored as
// soon as the first segment's MMAs (z) complete, while the second segment's still run;
// only dzs and the row sums wait for the whole tile. 0: all of it after the whole tile.
#ifndef BOOST_DUAL_SPLIT_EPI
#define BOOST_DUAL_SPLIT_EPI 1
#endif
constexpr int kGluEpiWarps = BOOST_GLU_EPI_WARPS;

enum EpiMode : int {
  EPI_ACT = 0,     // out_bf16 = act(s_row * acc)               (down-projection fwd)
  EPI_BF16 = 1,    // out_bf16 = acc                            (up-projection, dB)
  EPI_F32 = 2,     // out_f32[split] = acc                      (split-K partials)
  EPI_DUAL = 3,    // two accumulators: a, dzs, per-row q partials (recompute + dgrad)
  EPI_DX = 4,      // out_bf16 = acc - (s^2 q / d) x            (dgrad x + RMSNorm bwd)
  EPI_DA = 5,      // out_bf16 = gamma_row * acc, dgamma partials (wgrad of A)
  EPI_GLU = 6,     // dh = bf16(acc); out = dh*up*silu'(gate), out2 = dh*silu(gate) (SwiGLU bwd)
  EPI_UPGLU = 7,   // two accumulators: gate, up = bf16(acc0), bf16(acc1) to out[0], out[1];
                   // out2 = h = bf16(silu(gate) * up)     (up-projection + SwiGLU fwd)
  EPI_BF16T = 8,   // EPI_BF16 through TMA stores (short-K up-projections, where the
                   // epilogue's stores weigh most)
  EPI_DUALT = 9,   // EPI_DUAL through TMA stores (short K: the epilogue weighs more)
};

// the two dual-accumulator recompute + dgrad modes
__host__ __device__ constexpr bool is_dual(int mode) {
  return mode == EPI_DUAL || mode == EPI_DUALT;
}

struct OperandView {
  int8_t mn_dim;    // tensor-map dimension carrying the M (or N) index
  int8_t k_dim;     // dimension carrying K
  int8_t b_dim;     // dimension carrying the batch / group index
  int8_t mn_major;  // 1: MN contiguous (boxes 64 MN x 64 K); 0: K contiguous (box 64 K x rows)
};

struct Segment {
  OperandView a, b;
  int32_t num_kb;        // k-blocks of 64 over the whole K of this segment
  int32_t batch_from_n;  // batch index = the tile's group instead of the tile's batch
  int32_t b_n_local;     // B operand's MN coordinate is the column within the group
  int32_t batch_add;     // added to the batch index of both operands of this segment
};

struct GemmParams {
  CUtensorMap tmA[2];
  CUtensorMap tmB[2];
  CUtensorMap tmO[2];         // bf16 outputs out / out2 as (cols, rows, batch), 32 x 32 boxes
  CUtensorMap tmE[2];         // bf16 epilogue inputs shaped like the output, 32 x 32 boxes
                              // (EPI_GLU: gate, up; EPI_DX: x)
  int32_t tma_out;            // bit i: tmO[i] is valid (else plain stores)
  int32_t tma_in;             // 1: the epilogue inputs stream through tmE (EPI_GLU: required)
  Segment seg[2];
  int32_t num_seg;
  int32_t M, N;               // output extent (per batch)
  int32_t batch;              // batches in the tile list
  int32_t m_tiles, n_tiles;
  int32_t m_base;             // first output row of this launch (rows [m_base, m_base+m_extent))
  int32_t m_extent;           // rows of this launch (0: all of M from m_base)
  int32_t n_base;             // first output column of this launch (ungrouped tiling;
                              // a multiple of the launch's tile width)
  int32_t splits, kb_per_split;
  int32_t m_inner;            // tile order: 1 = m fastest within (batch, split)
  int32_t m_group;            // m_inner == 0 and > 1: rows of super-tiles taken m fastest
                              // in groups of this many, n next (grouped raster order)
  int32_t group_n;            // columns per group (grouped tiling)
  int32_t group_tiles;        // >0: N tiled per group, this many tiles per group
  int32_t act;                // 0 identity, 1 SiLU
  int32_t d_norm;             // EPI_DX: full d of the RMSNorm mean
  int32_t nq;                 // EPI_DX: number of q partial rows to sum
  // epilogue tensors (elements, not bytes, for strides)
  void* out;                  // bf16 or fp32 output
  void* out2;                 // EPI_DUAL: dzs; EPI_GLU: dup; EPI_UPGLU: h
  int64_t ldo;                // leading dimension of out/out2
  int64_t out_bstride;        // batch stride of out
  int64_t out_sstride;        // split stride of out (EPI_F32)
  const float* rstd;          // [M] row scale or nullptr (s == 1)
  float* qpart;               // EPI_DUAL out / EPI_DX in: [n_tiles or nq][M]
  float* dgpart;              // EPI_DA out: [n_tiles][M]
  const __nv_bfloat16* gamma; // EPI_DA: gamma [M]
  const __nv_bfloat16* wA;    // EPI_DA: A [M, N]
  const __nv_bfloat16* res;   // EPI_BF16, EPI_DX (one batch): residual [M, N] added to the
                              // bf16 output, out = bf16(bf16(result) + res), or NULL
  int64_t ldr;                // leading dimension of res
  DeviceError* err;
  uint64_t wait_limit_ns;
  int32_t* visits;            // debug: per-element write counts, indexed like out (or NULL)
};

template <int BN, int MODE, int CG, int MCM = 1, int MCN = 1>
struct GemmCfg {
  // (single-CTA tiles stage twice the B rows: no room for the extra warps' staging)
  static constexpr int kEpiW = (MODE == EPI_GLU && CG == 2) ? kGluEpiWarps : kEpiWarps;
  static constexpr int kHalves = kEpiW / 4;                     // warps per lane quarter
  static constexpr int kThreads = 32 * (2 + kEpiW);             // producer, MMA, epilogue
  // two accumulators per tile, one per segment
  static constexpr bool kDual = (is_dual(MODE) || MODE == EPI_UPGLU);
  static constexpr int kBRows = BN / CG;                          // B rows staged per CTA
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = kBRows * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // Epilogue output path. TMA stores (a ring of 2 KB slots per warp, one bulk store per
  // 32 x 32 bf16 chunk) take the global write latency off the epilogue warps, which
  // pays where the epilogue is the bottleneck (the SwiGLU epilogues); elsewhere they
  // compete with the operand loads for the SM's TMA unit, and plain coalesced stores
  // through the warp's staging block measured faster.
  static constexpr bool kTmaStore =
      (MODE == EPI_GLU || MODE == EPI_UPGLU || MODE == EPI_BF16T || MODE == EPI_DUALT);
  // Epilogue inputs streamed by TMA (EpiLoader): gate and up for EPI_GLU, x for EPI_DX,
  // kEpiDepth chunks ahead of the consumer. One chunk ahead measured faster than two:
  // the shared memory a second slot takes costs the mainloop a pipeline stage, and these
  // short-K GEMMs with heavy epilogue traffic need the deeper operand pipeline more.
  static constexpr int kEpiStreams = (MODE == EPI_GLU) ? 2 : (MODE == EPI_DX ? 1 : 0);
  // EPI_GLU in place: each warp's gate/up slot also holds the chunk's dgate/dup for their
  // TMA stores, so the shared memory of the store ring buys a second input slot instead:
  // the loads run two chunks ahead of the consumer (each slot is reloaded as soon as the
  // stores from it have read it).
  static constexpr bool kInPlace = (MODE == EPI_GLU) && BOOST_GLU_IN_PLACE;
  static constexpr int kEpiDepth = kInPlace ? 2 : 1;
  // Staging per warp: load slots (the loader's kEpiDepth x kEpiStreams 2 KB slots, or one
  // 2 KB slot for EPI_DA's synchronous loads), then the store slots (2 KB each); fp32
  // partials use one 4 KB block.
  static constexpr int kStoreSlots = (MODE == EPI_F32 || kInPlace) ? 0 : (kTmaStore ? 2 : 1);
  static constexpr int kLoadBytes =
      kEpiStreams > 0 ? kEpiDepth * kEpiStreams * 2048 : (MODE == EPI_DA ? 2048 : 0);
  static constexpr int kWarpStg = (MODE == EPI_F32) ? 4096 : kLoadBytes + 2048 * kStoreSlots;
  static constexpr int kLdBars = kEpiStreams > 0 ? kEpiW * kEpiDepth : 0;
  static constexpr int kStgBytes = kEpiW * kWarpStg;
  static constexpr int kStagesRaw = (232448 - 2048 - kStgBytes) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static constexpr int kAccCols = kDual ? 2 * BN : BN;            // columns per accumulator set
  static constexpr int kAccStages = (2 * kAccCols <= 512) ? 2 : 1;
  // EPI_UPGLU with one accumulator set: the epilogue frees the first accumulator (gate)
  // before it reads the second, so the next tile's first segment overlaps the rest of
  // the epilogue. One "empty" barrier per accumulator then.
  static constexpr bool kSplitRelease = (MODE == EPI_UPGLU && kAccStages == 1);
  static constexpr int kTemptyBars = kSplitRelease ? 2 : kAccStages;
  static constexpr int kTmemColsRaw = kAccStages * kAccCols;
  static constexpr int kTmemCols = kTmemColsRaw <= 32 ? 32 : kTmemColsRaw <= 64 ? 64
                                   : kTmemColsRaw <= 128 ? 128 : kTmemColsRaw <= 256 ? 256 : 512;
  // dual modes: one "z complete" barrier per accumulator set (the first segment's MMAs)
  static constexpr int kZBars = (is_dual(MODE) && BOOST_DUAL_SPLIT_EPI) ? kAccStages : 0;
  static constexpr int kBarBytes =
      8 * (2 * kStages + kAccStages + kTemptyBars + 1 + kLdBars + kZBars) + 16;
  // staging slots 1024-byte aligned (the 64-byte swizzle pattern of a TMA box repeats
  // every 512 bytes)
  static constexpr int kStgOffset = (kStages * kStageBytes + kBarBytes + 1023) / 1024 * 1024;
  static constexpr int kSmemBytes = 1024 /*align slack*/ + kStgOffset + kStgBytes;
  static constexpr int kMmaM = kBM * CG;                    // M of one tcgen05.mma
  static constexpr int kPairs = MCM * MCN;                  // pairs per cluster
  static constexpr int kTileM = kBM * CG * MCM;            // super-tile rows
  static constexpr int kTileN = BN * MCN;                  // super-tile columns
  static constexpr int kCluster = CG * kPairs;
  static_assert(kTmemColsRaw <= 512, "TMEM overflow");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be 64, 128, 192 or 256");
  static_assert(CG == 1 || CG == 2, "CG is 1 or 2");
  static_assert(kPairs == 1 || (CG == 2 && BN == 256 && MCM <= 2 && MCN <= 2),
                "multicast needs 256-wide pair tiles");
  static_assert(kMmaM == 128 || kMmaM == 256, "tcgen05.mma kind::f16 M is 128 or 256 here");
  static_assert(kBRows % 64 == 0, "each CTA stages whole 64-row B boxes");
  static_assert(kStages >= 3, "pipeline too shallow");
  static_assert(kSmemBytes <= 232448, "over the 227 KB shared-memory limit per CTA");
  static_assert(kEpiW % 4 == 0 && kEpiW >= 4 && kEpiW <= 16, "whole lane quarters");
  static_assert((!is_dual(MODE) && MODE != EPI_DA) || kHalves == kEpiHalves,
                "per-row partial sums are sized for the default epilogue warps");
  static_assert(MODE != EPI_UPGLU || (BN / 32) % kHalves == 0, "whole chunks per warp");
};

struct TileCoord {
  int32_t batch, split, m0, n_blk;
  int32_t n0, n_end;      // output columns [n0, n_end) of this tile
  int32_t group, n_local; // grouped tiling: group index and column within the group
};

// Tiles are ordered (split, batch, outer, inner). With group_tiles > 0 the N
// extent is tiled per group of group_n columns, so no tile straddles two groups.
template <int BN, int TILE_M>
__device__ __forceinline__ TileCoord decode_tile(const GemmParams& p, int32_t tile) {
  const int32_t per = p.m_tiles * p.n_tiles;
  const int32_t bs = tile / per;
  const int32_t rem = tile - bs * per;
  int32_t mb, nb;
  if (p.m_inner) {
    mb = rem % p.m_tiles;
    nb = rem / p.m_tiles;
  } else if (p.m_group > 1) {
    // group g holds super-tile rows [g G, g G + gm) (gm < G in the last group), all n;
    // within it m is fastest, so a wave shares B columns and the group's rows of A
    const int32_t full = p.m_group * p.n_tiles;
    const int32_t g = rem / full;
    const int32_t gm = min(p.m_group, p.m_tiles - g * p.m_group);
    const int32_t idx = rem - g * full;
    mb = g * p.m_group + idx % gm;
    nb = idx / gm;
  } else {
    nb = rem % p.n_tiles;
    mb = rem / p.n_tiles;
  }
  TileCoord c;
  c.split = bs / p.batch;
  c.batch = bs - c.split * p.batch;
  c.m0 = p.m_base + mb * TILE_M;
  c.n_blk = nb + p.n_base / BN;   // column-tile index over the whole output
  if (p.group_tiles > 0) {
    c.group = nb / p.group_tiles;
    c.n_local = (nb - c.group * p.group_tiles) * BN;
    c.n0 = c.group * p.group_n + c.n_local;
    c.n_end = min(c.n0 + BN, (c.group + 1) * p.group_n);
  } else {
    c.n0 = p.n_base + nb * BN;
    c.n_end = min(c.n0 + BN, p.N);
    c.group = 0;
    c.n_local = c.n0;
  }
  return c;
}

__device__ __forceinline__ void kb_range(const GemmParams& p, int seg, int32_t split,
                                         int32_t& kb0, int32_t& kb1) {
  const int32_t nkb = p.seg[seg].num_kb;
  if (p.splits <= 1) {
    kb0 = 0;
    kb1 = nkb;
  } else {
    kb0 = split * p.kb_per_split;
    kb1 = min(nkb, kb0 + p.kb_per_split);
  }
}

// Issue the TMA boxes of one operand tile (`rows` MN rows x 64 K) into `dst`: every box
// covers 64 MN rows x 64 K (K-major: 64 rows of 128 B; MN-major: one 64-wide atom of
// 64 K rows), 8 KB, placed at dst + 8 KB * j. One set of tensor maps therefore serves
// every tile shape. CG = 1 completes on the local barrier `bar`; CG = 2 on the pair
// barrier at cluster address `bar_cluster` (the even CTA's stage barrier).
template <int CG>
__device__ __forceinline__ void load_operand(const CUtensorMap* tm, const OperandView& v,
                                             uint8_t* dst, uint64_t* bar, uint32_t bar_cluster,
                                             int32_t mn, int32_t k, int32_t b, int rows) {
  int32_t c[3] = {0, 0, 0};
  c[v.k_dim] = k;
  c[v.b_dim] = b;
  for (int j = 0; j < rows / 64; ++j) {
    c[v.mn_dim] = mn + 64 * j;
    if constexpr (CG == 2)
      tma_load_3d_pair(dst + j * 8192, tm, bar_cluster, c[0], c[1], c[2]);
    else
      tma_load_3d(dst + j * 8192, tm, bar, c[0], c[1], c[2]);
  }
}

// One 64-row slice (K-major: a 64 K x 64 row box; MN-major: one 64-wide atom) of an
// operand shared by two pairs, multicast to the CTAs in `mask`.
__device__ __forceinline__ void load_operand_mc(const CUtensorMap* tm, const OperandView& v,
                                                uint8_t* dst, uint32_t bar_cluster, uint16_t mask,
                                                int32_t mn, int32_t k, int32_t b) {
  int32_t c[3] = {0, 0, 0};
  c[v.k_dim] = k;
  c[v.b_dim] = b;
  c[v.mn_dim] = mn;
  tma_load_3d_pair_mc(dst, tm, bar_cluster, mask, c[0], c[1], c[2]);
}

__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int mn_major, int kk) {
  // K-major: rows of 128 B (64 K), 8-row groups 1024 B apart; a K step of 16 is +32 B.
  // MN-major: boxes of [64 K rows][64 MN], 8 KB apart along MN (LBO), 8-row K groups
  // 1024 B apart (SBO); a K step of 16 is two groups, +2048 B.
  return mn_major ? smem_desc_sw128(base + kk * 2048, 8192, 1024)
                  : smem_desc_sw128(base + kk * 32, 16, 1024);
}

// logistic(z) with the hardware exp2 and a fast reciprocal divide; the rounding of
// the bf16 results it feeds dominates its few-ulp fp32 error.
__device__ __forceinline__ float sigmoid_f(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// The activation of the down-projection epilogue. The forward and the backward's
// recompute both call this, so the recomputed activation is bitwise the forward one.
__device__ __forceinline__ float act_fwd(float z, int act) {
  return act == 1 ? z * sigmoid_f(z) : z;
}

// ------------------------------------------------------------ staging
// Each epilogue warp owns a 4 KB shared-memory block through which it turns its
// row-per-thread accumulator chunk (32 rows x 32 columns) into row-contiguous
// global accesses. 16-byte chunks are XOR-swizzled by row so that both the
// row-per-lane side and the contiguous side are free of bank conflicts.

// bf16: row r is 64 B; chunk c of row r sits at chunk slot c ^ ((r >> 1) & 3).
__device__ __forceinline__ void stage_store_bf16(uint8_t* stg, int lane, const uint32_t (&pk)[16],
                                                 __nv_bfloat16* g, int64_t ld, int rows_valid,
                                                 int cols_valid) {
  uint4* mine = reinterpret_cast<uint4*>(stg + lane * 64);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    mine[c ^ sw] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 8 * j + (lane >> 2), c = lane & 3;
    const uint4 v = reinterpret_cast<const uint4*>(stg + r * 64)[c ^ ((r >> 1) & 3)];
    if (r < rows_valid && c * 8 < cols_valid)
      *reinterpret_cast<uint4*>(g + static_cast<int64_t>(r) * ld + c * 8) = v;
  }
  __syncwarp();
}

// fp32: row r is 128 B; chunk c of row r sits at chunk slot c ^ (r & 7).
__device__ __forceinline__ void stage_store_f32(uint8_t* stg, int lane, const float (&v)[32],
                                                float* g, int64_t ld, int rows_valid,
                                                int cols_valid) {
  float4* mine = reinterpret_cast<float4*>(stg + lane * 128);
  const int sw = lane & 7;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    mine[c ^ sw] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = 4 * j + (lane >> 3), c = lane & 7;
    const float4 x = reinterpret_cast<const float4*>(stg + r * 128)[c ^ (r & 7)];
    if (r < rows_valid && c * 4 < cols_valid)
      *reinterpret_cast<float4*>(g + static_cast<int64_t>(r) * ld + c * 4) = x;
  }
  __syncwarp();
}

// Coalesced read of a 32 x 32 bf16 block (row r at g + r*ld), delivered as this lane's
// row in fp32; out-of-range rows or columns read as zero.
__device__ __forceinline__ void stage_load_bf16(uint8_t* stg, int lane, const __nv_bfloat16* g,
                                                int64_t ld, int rows_valid, int cols_valid,
                                                float (&out)[32]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 8 * j + (lane >> 2), c = lane & 3;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < rows_valid && c * 8 < cols_valid)
      v = *reinterpret_cast<const uint4*>(g + static_cast<int64_t>(r) * ld + c * 8);
    reinterpret_cast<uint4*>(stg + r * 64)[c ^ ((r >> 1) & 3)] = v;
  }
  __syncwarp();
  const uint4* mine = reinterpret_cast<const uint4*>(stg + lane * 64);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 u = mine[c ^ sw];
    out[8 * c + 0] = bf16_lo(u.x); out[8 * c + 1] = bf16_hi(u.x);
    out[8 * c + 2] = bf16_lo(u.y); out[8 * c + 3] = bf16_hi(u.y);
    out[8 * c + 4] = bf16_lo(u.z); out[8 * c + 5] = bf16_hi(u.z);
    out[8 * c + 6] = bf16_lo(u.w); out[8 * c + 7] = bf16_hi(u.w);
  }
  __syncwarp();
}

// A warp's ring of 2 KB shared-memory slots for TMA stores of bf16 32 x 32 chunks. Only
// lane 0 issues and tracks the stores (bulk groups are per thread).
template <int kSlots, bool kTma>
struct StoreRing {
  uint8_t* base;
  int next;
};

// Store this warp's 32 x 32 bf16 chunk (lane = row; pk = the row's 32 values, packed) at
// column col0, row row0, batch `batch` of output map `tm`. The chunk goes through the
// next slot of the ring (64-byte swizzled rows, the map's layout) and one TMA store,
// which clips rows and columns outside the map; the warp does not wait for the global
// write. With `tma` false (no map, or the chunk is cut by a group boundary inside the
// tensor, which the map cannot clip) it is written with coalesced plain stores instead.
template <int kSlots, bool kTma, bool kEvictFirst = false>
__device__ __forceinline__ void store_chunk_bf16(StoreRing<kSlots, kTma>& ring, int lane,
                                                 const uint32_t (&pk)[16], const CUtensorMap* tm,
                                                 bool tma, int32_t col0, int32_t row0,
                                                 int32_t batch, __nv_bfloat16* g, int64_t ld,
                                                 int rows_valid, int cols_valid) {
  if constexpr (!kTma) {
    (void)tm; (void)tma; (void)col0; (void)row0; (void)batch;
    stage_store_bf16(ring.base, lane, pk, g, ld, rows_valid, cols_valid);
    return;
  }
  uint8_t* slot = ring.base + ring.next * 2048;
  ring.next = ring.next + 1 == kSlots ? 0 : ring.next + 1;
  if (tma) {
    // the store that last used this slot was committed kSlots - 1 groups ago (or an
    // intervening plain store already drained every group)
    if (lane == 0) bulk_wait_group_read<kSlots - 1>();
    __syncwarp();
    uint4* mine = reinterpret_cast<uint4*>(slot + lane * 64);
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      mine[c ^ sw] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if constexpr (kEvictFirst) tma_store_3d_hint(tm, slot, col0, row0, batch, l2_evict_first());
      else tma_store_3d(tm, slot, col0, row0, batch);
      bulk_commit_group();
    }
  } else {
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
    stage_store_bf16(slot, lane, pk, g, ld, rows_valid, cols_valid);
  }
}

// Read this lane's row (32 bf16 values, 64-byte swizzled 32 x 32 block) as fp32.
__device__ __forceinline__ void slot_row_f32(const uint8_t* slot, int lane, float (&out)[32]) {
  const uint4* mine = reinterpret_cast<const uint4*>(slot + lane * 64);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 u = mine[c ^ sw];
    out[8 * c + 0] = bf16_lo(u.x); out[8 * c + 1] = bf16_hi(u.x);
    out[8 * c + 2] = bf16_lo(u.y); out[8 * c + 3] = bf16_hi(u.y);
    out[8 * c + 4] = bf16_lo(u.z); out[8 * c + 5] = bf16_hi(u.z);
    out[8 * c + 6] = bf16_lo(u.w); out[8 * c + 7] = bf16_hi(u.w);
  }
}

// Per-warp stream of the epilogue's bf16 inputs (kStreams tensors shaped like the
// output, e.g. gate and up): for every 32 x 32 chunk the warp will write, in the order
// it writes them and across tile boundaries, one TMA load per tensor into a ring of
// kDepth slots, kDepth chunks ahead of the consumer. The loads do not depend on the
// accumulator, so the next tile's first chunks are in flight before its MMAs finish.
// Lane 0 issues; every lane waits on the slot's mbarrier (bounded) before reading.
template <int BN, int TILE_N, int TILE_M, int kStreams, int kDepth, int kHalves,
          bool kInPlaceUse = false>
struct EpiLoader {
  static constexpr bool kInPlace = kInPlaceUse;
  static constexpr int kChunks = (BN / 32 + kHalves - 1) / kHalves;   // most chunks a warp takes
  // gate and up of the SwiGLU backward are read once: keep them from displacing operands
  static constexpr bool kEvictFirst = (kStreams == 2);
  static constexpr int kSlotBytes = kStreams * 2048;
  const GemmParams* p;
  uint8_t* slots;          // kDepth slots of kStreams 2 KB blocks
  uint64_t* bars;          // kDepth mbarriers of this warp
  int32_t tile, tile_stride, num_tiles;   // issue cursor: next tile ...
  int j;                                  // ... and chunk index within it
  int32_t row_off, col_off;               // this warp's rows / this pair's columns in a tile
  int half;
  uint32_t issued, consumed;
  // coordinates of tile `decoded` (decoding takes integer divisions: once per tile, not
  // once per chunk)
  int32_t decoded, pn0, pend, m0;

  // Issue the loads of the next chunk this warp will write (if any) into the next slot.
  __device__ __forceinline__ void issue_next(int lane) {
    while (tile < num_tiles) {
      if (tile != decoded) {
        const TileCoord tc = decode_tile<TILE_N, TILE_M>(*p, tile);
        decoded = tile;
        pn0 = tc.n0 + col_off;
        pend = min(pn0 + BN, tc.n_end);
        m0 = tc.m0;
      }
      const int32_t col0 = pn0 + (half + j * kHalves) * 32;
      if (j < kChunks && col0 < pend) {
        const uint32_t slot = issued % kDepth;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[slot], kSlotBytes);
#pragma unroll
          for (int t = 0; t < kStreams; ++t)
            if constexpr (kEvictFirst)
              tma_load_3d_hint(slots + slot * kSlotBytes + t * 2048, &p->tmE[t], &bars[slot],
                               col0, m0 + row_off, 0, l2_evict_first());
            else
              tma_load_3d(slots + slot * kSlotBytes + t * 2048, &p->tmE[t], &bars[slot], col0,
                          m0 + row_off, 0);
        }
        ++issued;
        ++j;
        return;
      }
      tile += tile_stride;   // the rest of this tile's chunks lie past its columns
      j = 0;
    }
  }

  __device__ __forceinline__ void start(int lane) {
    for (int d = 0; d < kDepth; ++d) issue_next(lane);
  }

  // The inputs of the warp's next chunk, one row per lane; then refill the slot.
  __device__ __forceinline__ void consume(int lane, float (&out)[kStreams][32]) {
    const uint32_t slot = consumed % kDepth;
    bounded_wait(&bars[slot], (consumed / kDepth) & 1u, p->err, 9, p->wait_limit_ns);
#pragma unroll
    for (int t = 0; t < kStreams; ++t)
      slot_row_f32(slots + slot * kSlotBytes + t * 2048, lane, out[t]);
    ++consumed;
    fence_proxy_async_smem();   // these reads precede the next TMA write into the slot
    __syncwarp();
    issue_next(lane);
  }

  // In-place use: wait for the warp's next chunk and return its slot (tensor t at
  // + t * 2 KB, 64-byte swizzled rows). The caller overwrites the slot with its outputs,
  // stores them from it and then calls refill().
  __device__ __forceinline__ uint8_t* wait_slot() {
    const uint32_t slot = consumed % kDepth;
    bounded_wait(&bars[slot], (consumed / kDepth) & 1u, p->err, 9, p->wait_limit_ns);
    ++consumed;
    return slots + slot * kSlotBytes;
  }

  // In-place use: once this warp's stores have read the slot just consumed (lane 0 issued
  // and committed them), load the chunk kDepth ahead into it.
  __device__ __forceinline__ void refill(int lane) {
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
    issue_next(lane);
  }

  // Wait for loads still in flight (only after an early exit from the tile loop).
  __device__ __forceinline__ void drain() {
    while (consumed < issued) {
      const uint32_t slot = consumed % kDepth;
      bounded_wait(&bars[slot], (consumed / kDepth) & 1u, p->err, 10, p->wait_limit_ns);
      ++consumed;
    }
  }
};

// Stand-in for modes without streamed inputs.
struct NoLoader {
  static constexpr bool kInPlace = false;
  __device__ __forceinline__ void start(int) {}
  __device__ __forceinline__ void drain() {}
};

// Debug write counting: this lane's row of a 32 x 32 chunk whose element (0, 0) is at
// index `base` of the output adds 1 to each element it writes.
__device__ __forceinline__ void count_writes(const GemmParams& p, int64_t base, int lane,
                                             int rows_valid, int cols_valid) {
  if (lane < rows_valid) {
    int32_t* v = p.visits + base + static_cast<int64_t>(lane) * p.ldo;
    for (int c = 0; c < 32 && c < cols_valid; ++c) atomicAdd(v + c, 1);
  }
}

// SwiGLU backward of two adjacent columns: the down-projection's input gradient dh (the
// accumulator pair a0, a1, rounded to bf16 as a separate pass would have stored it) and
// the bf16 gate and up pairs g2, u2 give dgate = dh * up * silu'(gate) and
// dup = dh * silu(gate), packed as bf16 pairs.
__device__ __forceinline__ void glu_pair(float a0, float a1, uint32_t g2, uint32_t u2,
                                         uint32_t& dgate, uint32_t& dup) {
  const uint32_t dh2 = pack_bf16x2(a0, a1);   // both rounded in one convert
  float dgo[2], duo[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float dh = h == 0 ? bf16_lo(dh2) : bf16_hi(dh2);
    const float z = h == 0 ? bf16_lo(g2) : bf16_hi(g2);
    const float u = h == 0 ? bf16_lo(u2) : bf16_hi(u2);
    const float sg = sigmoid_f(z);
    dgo[h] = dh * u * (sg * (1.0f + z * (1.0f - sg)));
    duo[h] = dh * (z * sg);
  }
  dgate = pack_bf16x2(dgo[0], dgo[1]);
  dup = pack_bf16x2(duo[0], duo[1]);
}

// One 32 x 32 chunk of the SwiGLU backward in place (rows [row0, row0 + 32), columns
// [col0, col0 + 32)): the accumulator (this lane's row) and the chunk's gate and up from
// the loader's slot give dgate and dup, which each lane writes over its own row of gate
// and up in the slot (same 64-byte swizzled layout as the output maps); lane 0 stores
// both with TMA (evict-first in L2: written once) and the loader reloads the slot.
template <class Loader>
__device__ __forceinline__ void glu_chunk_in_place(const GemmParams& p, Loader& ld, int lane,
                                                   uint32_t t_col, int32_t col0, int32_t row0,
                                                   int rows_valid, int cols_valid) {
  float v[32];
  tmem_ld_32x32b_x32(t_col, v);
  uint8_t* slot = ld.wait_slot();
  tmem_ld_wait();
  uint4* gr = reinterpret_cast<uint4*>(slot + lane * 64);
  uint4* ur = reinterpret_cast<uint4*>(slot + 2048 + lane * 64);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    const uint4 gq = gr[c4 ^ sw], uq = ur[c4 ^ sw];
    const float* a = v + 8 * c4;
    uint4 dg, du;
    glu_pair(a[0], a[1], gq.x, uq.x, dg.x, du.x);
    glu_pair(a[2], a[3], gq.y, uq.y, dg.y, du.y);
    glu_pair(a[4], a[5], gq.z, uq.z, dg.z, du.z);
    glu_pair(a[6], a[7], gq.w, uq.w, dg.w, du.w);
    gr[c4 ^ sw] = dg;
    ur[c4 ^ sw] = du;
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    const uint64_t pol = l2_evict_first();
    tma_store_3d_hint(&p.tmO[0], slot, col0, row0, 0, pol);
    tma_store_3d_hint(&p.tmO[1], slot + 2048, col0, row0, 0, pol);
    bulk_commit_group();
  }
  if (p.visits != nullptr)
    count_writes(p, static_cast<int64_t>(row0) * p.ldo + col0, lane, rows_valid, cols_valid);
  ld.refill(lane);
}

// First part of the dual modes' epilogue, run while the tile's second segment is still
// on the tensor cores: this warp's chunks of the bottleneck activation
// a = bf16(act(s * z)) from the complete z accumulator (TMEM columns [0, BN) at t_row),
// with the same expression as the forward's down-projection epilogue, so the
// recomputed a is bitwise the forward's.
template <int BN, int kHalves, int kSlots, bool kTma>
__device__ __forceinline__ void dual_act_chunks(const GemmParams& p, int32_t row0, int32_t n0,
                                                int32_t n_end, uint32_t t_row,
                                                StoreRing<kSlots, kTma>& ring, int lane,
                                                int half) {
  const int32_t row = row0 + lane;
  const int rows_valid = p.M - row0 < 32 ? p.M - row0 : 32;
  const float s_row = (p.rstd != nullptr && row < p.M) ? p.rstd[row] : 1.0f;
#pragma unroll 1
  for (int c = half; c < BN / 32; c += kHalves) {
    const int32_t col0 = n0 + c * 32;
    const int cols_valid = n_end - col0;
    if (cols_valid <= 0) break;            // warp-uniform
    const bool whole = cols_valid >= 32 || n_end == p.N;
    float v[32];
    tmem_ld_32x32b_x32(t_row + c * 32, v);
    tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[i] = pack_bf16x2(act_fwd(s_row * v[2 * i], p.act), act_fwd(s_row * v[2 * i + 1], p.act));
    const int64_t base = static_cast<int64_t>(row0) * p.ldo + col0;
    store_chunk_bf16(ring, lane, pk, &p.tmO[0], whole && (p.tma_out & 1), col0, row0, 0,
                     static_cast<__nv_bfloat16*>(p.out) + base, p.ldo, rows_valid, cols_valid);
    if (p.visits != nullptr) count_writes(p, base, lane, rows_valid, cols_valid);
  }
}

// out = bf16(bf16(result) + res) on this warp's packed 32 x 32 chunk, when the launch has a
// residual: the same two roundings as storing the result and adding res in a separate
// pass. The residual chunk comes in through the warp's 2 KB store block (coalesced rows),
// which the chunk's store reuses afterwards.
__device__ __forceinline__ void add_residual(const GemmParams& p, uint8_t* blk, int lane,
                                             int32_t row0, int32_t col0, int rows_valid,
                                             int cols_valid, uint32_t (&pk)[16]) {
  if (p.res == nullptr) return;
  float rv[32];
  stage_load_bf16(blk, lane, p.res + static_cast<int64_t>(row0) * p.ldr + col0, p.ldr,
                  rows_valid, cols_valid, rv);
#pragma unroll
  for (int i = 0; i < 16; ++i)
    pk[i] = pack_bf16x2(bf16_lo(pk[i]) + rv[2 * i], bf16_hi(pk[i]) + rv[2 * i + 1]);
}

// Epilogue of one tile for the calling warp: its 32 TMEM lanes of the accumulator set
// at column `t_row` hold output rows [row0, row0 + 32); this thread owns row0 + lane.
// Columns [n0, n_end) are written, 32 at a time, through the warp's staging block.
// `col_tile` indexes the per-row partial sums (q, dgamma) of this BN-wide column tile.
// `half` selects the 32-column chunks of this warp (half, half + kHalves, ...), kHalves
// being the warps per lane quarter; the per-row partial sums are written per warp of a
// quarter, at row col_tile * kHalves + half.
// `stg` is the warp's load slot (fp32 staging for EPI_F32), `ring` its store slots, `ld`
// its input stream (EPI_GLU, EPI_DX).
template <int BN, int MODE, int kHalves, int kSlots, bool kTma, class Loader>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const TileCoord& tc,
                                              int32_t row0, int32_t n0, int32_t n_end,
                                              uint32_t t_row, uint8_t* stg,
                                              StoreRing<kSlots, kTma>& ring, Loader& ld,
                                              int lane, int32_t col_tile, int half) {
  const int32_t row = row0 + lane;
  const bool row_ok = row < p.M;
  const int rows_valid = p.M - row0 < 32 ? p.M - row0 : 32;
  float s_row = 1.0f;
  if constexpr (MODE == EPI_ACT || is_dual(MODE) || MODE == EPI_DX) {
    if (p.rstd != nullptr && row_ok) s_row = p.rstd[row];
  }
  float rowsum = 0.0f;
  float coef = 0.0f;
  if constexpr (MODE == EPI_DX) {
    if (p.rstd != nullptr && row_ok) {
      float qs = 0.0f;
      for (int j = 0; j < p.nq; ++j) qs += p.qpart[static_cast<int64_t>(j) * p.M + row];
      coef = s_row * s_row * qs / static_cast<float>(p.d_norm);
    }
  }
  float g_row = 1.0f;
  if constexpr (MODE == EPI_DA) {
    if (p.gamma != nullptr && row_ok) g_row = __bfloat162float(p.gamma[row]);
  }
#pragma unroll 1
  for (int c = half; c < BN / 32; c += kHalves) {
    const int32_t col0 = n0 + c * 32;
    const int cols_valid = n_end - col0;
    if (cols_valid <= 0) break;            // warp-uniform: the rest of the tile is outside N
    if constexpr (MODE == EPI_GLU && Loader::kInPlace) {
      glu_chunk_in_place(p, ld, lane, t_row + c * 32, col0, row0, rows_valid, cols_valid);
    } else {
      const bool whole = cols_valid >= 32 || n_end == p.N;   // the maps clip at N only
      float v[32];
      tmem_ld_32x32b_x32(t_row + c * 32, v);
      float w[32];
      if constexpr (is_dual(MODE)) tmem_ld_32x32b_x32(t_row + BN + c * 32, w);
      tmem_ld_wait();
      if constexpr (MODE == EPI_F32) {
        const int64_t base = tc.split * p.out_sstride + tc.batch * p.out_bstride +
                             static_cast<int64_t>(row0) * p.ldo + col0;
        stage_store_f32(stg, lane, v, static_cast<float*>(p.out) + base, p.ldo, rows_valid,
                        cols_valid);
        if (p.visits != nullptr) count_writes(p, base, lane, rows_valid, cols_valid);
      } else {
        uint32_t pk[16];
        if constexpr (MODE == EPI_ACT) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(act_fwd(s_row * v[2 * i], p.act),
                                act_fwd(s_row * v[2 * i + 1], p.act));
        } else if constexpr (MODE == EPI_BF16 || MODE == EPI_BF16T) {
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
          if constexpr (MODE == EPI_BF16) add_residual(p, ring.base, lane, row0, col0, rows_valid,
                                                      cols_valid, pk);
        } else if constexpr (is_dual(MODE)) {
          // a = act(z) (recompute) and dzs = s * act'(z) * (dy B^T); row partial of dz * z.
          uint32_t pk2[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float a2[2], d2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float z = s_row * v[i + h];
              float dz;
              if (p.act == 1) {
                const float sg = sigmoid_f(z);
                a2[h] = z * sg;
                dz = w[i + h] * (sg * (1.0f + z * (1.0f - sg)));
              } else {
                a2[h] = z;
                dz = w[i + h];
              }
              if (i + h < cols_valid) rowsum += dz * z;
              d2[h] = s_row * dz;
            }
            if constexpr (!BOOST_DUAL_SPLIT_EPI) pk[i / 2] = pack_bf16x2(a2[0], a2[1]);
            pk2[i / 2] = pack_bf16x2(d2[0], d2[1]);
          }
          __nv_bfloat16* o2 = static_cast<__nv_bfloat16*>(p.out2) +
                              static_cast<int64_t>(row0) * p.ldo + col0;
          store_chunk_bf16(ring, lane, pk2, &p.tmO[1], whole && (p.tma_out & 2), col0, row0, 0, o2,
                           p.ldo, rows_valid, cols_valid);
        } else if constexpr (MODE == EPI_GLU) {
          // SwiGLU backward on the down-projection's input gradient dh (rounded to bf16,
          // the value a separate pass would have stored): dgate and dup of h = silu(g)*u.
          float gu[2][32];   // gate, up
          ld.consume(lane, gu);
          uint32_t pk2[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float dgo[2], duo[2];
            const uint32_t dh2 = pack_bf16x2(v[i], v[i + 1]);   // both rounded in one convert
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float dh = h == 0 ? bf16_lo(dh2) : bf16_hi(dh2);
              const float z = gu[0][i + h];
              const float sg = sigmoid_f(z);
              dgo[h] = dh * gu[1][i + h] * (sg * (1.0f + z * (1.0f - sg)));
              duo[h] = dh * (z * sg);
            }
            pk[i / 2] = pack_bf16x2(dgo[0], dgo[1]);
            pk2[i / 2] = pack_bf16x2(duo[0], duo[1]);
          }
          __nv_bfloat16* o2 = static_cast<__nv_bfloat16*>(p.out2) +
                              static_cast<int64_t>(row0) * p.ldo + col0;
          // (dgate and dup are written once here: evict-first in L2)
          store_chunk_bf16<kSlots, kTma, true>(ring, lane, pk2, &p.tmO[1],
                                               whole && (p.tma_out & 2), col0, row0, 0, o2,
                                               p.ldo, rows_valid, cols_valid);
        } else if constexpr (MODE == EPI_DX) {
          float xv[1][32];
          if (p.tma_in) {                          // RMSNorm term: x streamed by the loader
            ld.consume(lane, xv);
          } else {                                 // no norm: coef == 0
#pragma unroll
            for (int i = 0; i < 32; ++i) xv[0][i] = 0.0f;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(v[2 * i] - coef * xv[0][2 * i],
                                v[2 * i + 1] - coef * xv[0][2 * i + 1]);
          add_residual(p, ring.base, lane, row0, col0, rows_valid, cols_valid, pk);
        } else if constexpr (MODE == EPI_DA) {
          if (p.wA != nullptr) {
            float av[32];
            stage_load_bf16(stg, lane, p.wA + static_cast<int64_t>(row0) * p.ldo + col0, p.ldo,
                            rows_valid, cols_valid, av);
#pragma unroll
            for (int i = 0; i < 32; ++i) rowsum += av[i] * v[i];
          }
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(g_row * v[2 * i], g_row * v[2 * i + 1]);
        }
        // (dual modes with the split epilogue stored a before the tile was complete)
        if constexpr (!(is_dual(MODE) && BOOST_DUAL_SPLIT_EPI)) {
          const int64_t base =
              tc.batch * p.out_bstride + static_cast<int64_t>(row0) * p.ldo + col0;
          store_chunk_bf16<kSlots, kTma, MODE == EPI_GLU>(
              ring, lane, pk, &p.tmO[0], whole && (p.tma_out & 1), col0, row0, tc.batch,
              static_cast<__nv_bfloat16*>(p.out) + base, p.ldo, rows_valid, cols_valid);
          if (p.visits != nullptr) count_writes(p, base, lane, rows_valid, cols_valid);
        }
      }
    }
  }
  if constexpr (is_dual(MODE)) {
    if (row_ok && p.qpart != nullptr)
      p.qpart[static_cast<int64_t>(col_tile * kHalves + half) * p.M + row] = rowsum;
  }
  if constexpr (MODE == EPI_DA) {
    if (row_ok && p.dgpart != nullptr)
      p.dgpart[static_cast<int64_t>(col_tile * kHalves + half) * p.M + row] = rowsum;
  }
}

// silu(g) * u on bf16 gate and up values, the same expression (and the same sigmoid) as
// the stand-alone SwiGLU forward kernel, so that the fused and the separate paths give
// identical h.
__device__ __forceinline__ float swiglu_h(float g, float u) { return g * sigmoid_f(g) * u; }

// Epilogue of the fused up-projection + SwiGLU forward for the calling warp (rows
// [row0, row0 + 32), columns [n0, n_end), the 32-column chunks half, half + kHalves,
// ...). Accumulator 0 (gate, TMEM columns [0, BN)) is read first and kept in registers
// as bf16; then, if `release0` is set, this warp's arrival on it lets the MMA warp start
// the next tile's gate segment. Accumulator 1 (up, columns [BN, 2 BN)) is read next,
// also kept as bf16, and `release1` frees it (or the whole accumulator set) before any
// store: the next tile's MMAs then overlap all of this tile's gate, up and
// h = silu(gate) * up stores. Gate and up of the warp's columns take 128 registers a
// thread, so the TMEM loads are 16 columns wide to keep the transient small. The stores
// go through the output maps only (the launch requires both), evict-first in L2.
template <int BN, int CG, int kHalves, int kSlots, bool kTma>
__device__ __forceinline__ void epilogue_upglu(const GemmParams& p, int32_t row0, int32_t n0,
                                               int32_t n_end, uint32_t t_row,
                                               StoreRing<kSlots, kTma>& ring, int lane, int half,
                                               uint64_t* release0, uint64_t* release1,
                                               uint32_t leader_rank) {
  constexpr int kChunks = BN / 32 / kHalves;
  const int rows_valid = p.M - row0 < 32 ? p.M - row0 : 32;
  __nv_bfloat16* y0 = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(row0) * p.ldo;
  __nv_bfloat16* y1 = y0 + p.out_bstride;
  __nv_bfloat16* hh = static_cast<__nv_bfloat16*>(p.out2) + static_cast<int64_t>(row0) * p.ldo;
  auto release = [&](uint64_t* bar) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if constexpr (CG == 2) mbar_arrive_cluster(mapa_shared(smem_u32(bar), leader_rank));
      else mbar_arrive(bar);
    }
  };
  uint32_t gk[kChunks][16];
  uint32_t uk[kChunks][16];
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    const int c = half + j * kHalves;
    if (n0 + c * 32 < n_end) {              // warp-uniform
#pragma unroll
      for (int hh16 = 0; hh16 < 2; ++hh16) {
        float v[16];
        tmem_ld_32x32b_x16(t_row + c * 32 + hh16 * 16, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i) gk[j][hh16 * 8 + i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
      }
    }
  }
  if (release0 != nullptr) release(release0);
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    const int c = half + j * kHalves;
    if (n0 + c * 32 < n_end) {              // warp-uniform
#pragma unroll
      for (int hh16 = 0; hh16 < 2; ++hh16) {   // 16 columns per load: fewer live registers
        float w[16];
        tmem_ld_32x32b_x16(t_row + BN + c * 32 + hh16 * 16, w);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i) uk[j][hh16 * 8 + i] = pack_bf16x2(w[2 * i], w[2 * i + 1]);
      }
    }
  }
  release(release1);
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    const int32_t col0 = n0 + (half + j * kHalves) * 32;
    if (col0 < n_end) {                     // warp-uniform
      store_chunk_bf16<kSlots, kTma, true>(ring, lane, gk[j], &p.tmO[0], true, col0, row0, 0,
                                           y0 + col0, p.ldo, rows_valid, n_end - col0);
      store_chunk_bf16<kSlots, kTma, true>(ring, lane, uk[j], &p.tmO[0], true, col0, row0, 1,
                                           y1 + col0, p.ldo, rows_valid, n_end - col0);
      // h after gate and up have gone to shared memory, in place of this chunk's gate
      // registers (the live set stays at gate + up)
#pragma unroll
      for (int i = 0; i < 16; ++i)
        gk[j][i] = pack_bf16x2(swiglu_h(bf16_lo(gk[j][i]), bf16_lo(uk[j][i])),
                               swiglu_h(bf16_hi(gk[j][i]), bf16_hi(uk[j][i])));
      const uint32_t (&hk)[16] = gk[j];
      store_chunk_bf16<kSlots, kTma, true>(ring, lane, hk, &p.tmO[1], true, col0, row0, 0,
                                           hh + col0, p.ldo, rows_valid, n_end - col0);
    }
  }
  if (p.visits != nullptr) {                // debug write counting (gate and up)
#pragma unroll 1
    for (int j = 0; j < kChunks; ++j) {
      const int32_t col0 = n0 + (half + j * kHalves) * 32;
      if (col0 < n_end) {
        const int64_t base = static_cast<int64_t>(row0) * p.ldo + col0;
        count_writes(p, base, lane, rows_valid, n_end - col0);
        count_writes(p, base + p.out_bstride, lane, rows_valid, n_end - col0);
      }
    }
  }
}

template <int BN, int MODE, int CG, int MCM, int MCN>
__global__ void __launch_bounds__(GemmCfg<BN, MODE, CG, MCM, MCN>::kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmParams p) {
  using Cfg = GemmCfg<BN, MODE, CG, MCM, MCN>;
  constexpr int CL = Cfg::kCluster;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + Cfg::kStages * Cfg::kABytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + Cfg::kStages * Cfg::kStageBytes);
  uint64_t* empty_bar = full_bar + Cfg::kStages;
  uint64_t* tfull_bar = empty_bar + Cfg::kStages;
  uint64_t* tempty_bar = tfull_bar + Cfg::kAccStages;
  uint64_t* done_bar = tempty_bar + Cfg::kTemptyBars;
  uint64_t* ld_bar = done_bar + 1;                   // kLdBars: the epilogue loaders'
  uint64_t* zfull_bar = ld_bar + Cfg::kLdBars;       // kZBars: z of the dual modes complete
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(zfull_bar + Cfg::kZBars);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = (CL > 1) ? cluster_ctarank() : 0u;   // rank in the cluster
  const uint32_t rank = crank % CG;                  // position in the CTA pair
  const uint32_t pp = crank / CG;                    // pair index in the cluster
  const uint32_t pm = pp % MCM;                      // the pair's row in the super-tile
  const uint32_t pn = pp / MCM;                      // the pair's column in the super-tile
  const uint32_t leader_rank = pp * CG;              // cluster rank of this pair's even CTA
  const bool leader = (rank == 0);
  const int32_t num_tiles = p.batch * p.splits * p.m_tiles * p.n_tiles;
  const int32_t first_tile = static_cast<int32_t>(blockIdx.x) / CL;
  const int32_t tile_stride = static_cast<int32_t>(gridDim.x) / CL;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&full_bar[s], 1);           // the even CTA's expect_tx covers both CTAs
      mbar_init(&empty_bar[s], Cfg::kPairs);  // freed once every pair of the cluster is done
    }
    for (int s = 0; s < Cfg::kAccStages; ++s) mbar_init(&tfull_bar[s], 1);
    for (int s = 0; s < Cfg::kTemptyBars; ++s)
      mbar_init(&tempty_bar[s], Cfg::kEpiW * CG);   // one arrival per epilogue warp of the pair
    mbar_init(done_bar, 1);
    for (int s = 0; s < Cfg::kLdBars; ++s) mbar_init(&ld_bar[s], 1);
    for (int s = 0; s < Cfg::kZBars; ++s) mbar_init(&zfull_bar[s], 1);
    fence_barrier_init();
  }
  if (warp == 2 && lane == 0 && Cfg::kEpiStreams > 0 && p.tma_in) {
    for (int t = 0; t < Cfg::kEpiStreams; ++t) tma_prefetch_desc(&p.tmE[t]);
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA[0]);
    tma_prefetch_desc(&p.tmB[0]);
    if (p.num_seg > 1) {
      tma_prefetch_desc(&p.tmA[1]);
      tma_prefetch_desc(&p.tmB[1]);
    }
  }
  if (warp == 1) {
    if constexpr (CG == 2) {
      tmem_alloc_pair(tmem_holder, Cfg::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, Cfg::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (CL > 1) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // Everything above touches only shared memory, TMEM and the kernel parameters, so it
  // may overlap the previous kernel on the stream; global memory waits for it. The next
  // kernel may be scheduled from here: its CTAs fit on an SM only once this kernel's CTA
  // there has exited, and this CTA's TMEM is already held.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed_mask = 0, parity_mask = 0;   // per stage: armed, parity of last arm
      bool ok = true;
      for (int32_t tile = first_tile; tile < num_tiles && ok; tile += tile_stride) {
        const TileCoord tc = decode_tile<Cfg::kTileN, Cfg::kTileM>(p, tile);
        const int32_t m_own =
            tc.m0 + static_cast<int32_t>(pm) * (kBM * CG) + static_cast<int32_t>(rank) * kBM;
        const int32_t n_half =
            static_cast<int32_t>(pn) * BN + static_cast<int32_t>(rank) * Cfg::kBRows;
        for (int sg = 0; sg < p.num_seg && ok; ++sg) {
          const Segment& S = p.seg[sg];
          int32_t b = tc.batch;
          int32_t nb = tc.n0;
          if (S.batch_from_n) b = tc.group;
          b += S.batch_add;
          if (S.b_n_local) nb = tc.n_local;
          int32_t kb0, kb1;
          kb_range(p, sg, tc.split, kb0, kb1);
          for (int32_t kb = kb0; kb < kb1; ++kb) {
            if (!bounded_wait(&empty_bar[stage], phase ^ 1u, p.err, 1, p.wait_limit_ns)) {
              ok = false;
              break;
            }
            // CG = 2: only the even CTA arms its stage barrier, for both CTAs' bytes; the
            // odd CTA's copies complete on that barrier too (no cross-CTA arrive, so no
            // cluster-scope fence per stage).
            uint32_t bar_cluster = 0;
            if constexpr (CG == 2)
              bar_cluster = mapa_shared(smem_u32(&full_bar[stage]), leader_rank);
            if (leader) mbar_arrive_expect_tx(&full_bar[stage], CG * Cfg::kStageBytes);
            armed_mask |= 1u << stage;
            parity_mask = (parity_mask & ~(1u << stage)) | (phase << stage);
            if constexpr (MCN == 2) {
              // the pairs of this row need the same A rows: each issues one 64-row slice
              uint16_t mask = 0;
              for (uint32_t j = 0; j < MCN; ++j) mask |= 1u << ((j * MCM + pm) * CG + rank);
              load_operand_mc(&p.tmA[sg], S.a, sA + stage * Cfg::kABytes + pn * 8192, bar_cluster,
                              mask, m_own + static_cast<int32_t>(pn) * 64, kb * kBK, b);
            } else {
              load_operand<CG>(&p.tmA[sg], S.a, sA + stage * Cfg::kABytes, &full_bar[stage],
                               bar_cluster, m_own, kb * kBK, b, kBM);
            }
            if constexpr (MCM == 2) {
              // the pairs of this column need the same B rows: each issues one 64-row slice
              uint16_t mask = 0;
              for (uint32_t i = 0; i < MCM; ++i) mask |= 1u << ((pn * MCM + i) * CG + rank);
              load_operand_mc(&p.tmB[sg], S.b, sB + stage * Cfg::kBBytes + pm * 8192, bar_cluster,
                              mask, nb + n_half + static_cast<int32_t>(pm) * 64, kb * kBK, b);
            } else {
              load_operand<CG>(&p.tmB[sg], S.b, sB + stage * Cfg::kBBytes, &full_bar[stage],
                               bar_cluster, nb + n_half, kb * kBK, b, Cfg::kBRows);
            }
            if (++stage == Cfg::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Drain: the copies started here have landed before the CTA exits. Both CTAs'
      // copies complete on the even CTA's barriers, so the even CTA waits for them.
      if (leader) {
        for (int s = 0; s < Cfg::kStages; ++s) {
          if (armed_mask & (1u << s)) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&full_bar[s], (parity_mask >> s) & 1u)) {
              if (globaltimer_ns() - t0 > p.wait_limit_ns) {
                record_error(p.err, kErrTimeout, 7);
                break;
              }
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      // The MMA is 128 x CG rows (one pair); every pair of a cluster issues its own.
      const uint32_t idesc0 =
          idesc_bf16_f32(Cfg::kMmaM, BN, p.seg[0].a.mn_major, p.seg[0].b.mn_major);
      const uint32_t idesc1 =
          idesc_bf16_f32(Cfg::kMmaM, BN, p.seg[1].a.mn_major, p.seg[1].b.mn_major);
      // Shared-memory offsets below 256 KB: the 14-bit start-address field (16 B units)
      // holds every stage address plus three K steps without carrying into the next field.
      const uint32_t sA_u32 = smem_u32(sA);
      const uint32_t sB_u32 = smem_u32(sB);
      for (int32_t tile = first_tile; tile < num_tiles && ok; tile += tile_stride) {
        const TileCoord tc = decode_tile<Cfg::kTileN, Cfg::kTileM>(p, tile);
        if constexpr (!Cfg::kSplitRelease) {
          if (!bounded_wait(&tempty_bar[acc], acc_phase ^ 1u, p.err, 2, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        for (int sg = 0; sg < p.num_seg && ok; ++sg) {
          if constexpr (Cfg::kSplitRelease) {
            // segment sg accumulates into accumulator sg: wait until it has been read
            if (!bounded_wait(&tempty_bar[sg], acc_phase ^ 1u, p.err, 2, p.wait_limit_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const uint32_t d_tmem = tmem_base + acc * Cfg::kAccCols + sg * BN;
          const int a_mn = p.seg[sg].a.mn_major, b_mn = p.seg[sg].b.mn_major;
          const uint32_t idesc = sg == 0 ? idesc0 : idesc1;
          // Descriptor bits other than the start address are fixed per segment; a K step
          // of 16 advances the start address by 32 B (K-major) or 2048 B (MN-major).
          const uint64_t a_hi = desc_hi_sw128(a_mn ? 8192u : 16u, 1024u);
          const uint64_t b_hi = desc_hi_sw128(b_mn ? 8192u : 16u, 1024u);
          const uint64_t a_step = a_mn ? (2048u >> 4) : (32u >> 4);
          const uint64_t b_step = b_mn ? (2048u >> 4) : (32u >> 4);
          int32_t kb0, kb1;
          kb_range(p, sg, tc.split, kb0, kb1);
          for (int32_t kb = kb0; kb < kb1; ++kb) {
            if (!bounded_wait(&full_bar[stage], phase, p.err, 3, p.wait_limit_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = a_hi | (((sA_u32 + stage * Cfg::kABytes) >> 4) & 0x3FFFu);
            const uint64_t bd = b_hi | (((sB_u32 + stage * Cfg::kBBytes) >> 4) & 0x3FFFu);
#pragma unroll
            for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
              const uint32_t accum = (kk > 0 || kb > kb0) ? 1u : 0u;
              if constexpr (CG == 2)
                tc_mma_bf16_pair(d_tmem, ad + kk * a_step, bd + kk * b_step, idesc, accum);
              else
                tc_mma_bf16(d_tmem, ad + kk * a_step, bd + kk * b_step, idesc, accum);
            }
            if constexpr (CG == 2)
              tc_commit_pair_mc(&empty_bar[stage], static_cast<uint16_t>((1u << CL) - 1u));
            else
              tc_commit(&empty_bar[stage]);
            if (++stage == Cfg::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if constexpr (Cfg::kZBars > 0) {
            // dual modes: z (segment 0) is complete once these MMAs are; the epilogue
            // stores a = act(s z) while segment 1 runs
            if (sg == 0 && ok) {
              if constexpr (CG == 2)
                tc_commit_pair_mc(&zfull_bar[acc], static_cast<uint16_t>(0x3u << leader_rank));
              else
                tc_commit(&zfull_bar[acc]);
            }
          }
        }
        if constexpr (CG == 2)
          tc_commit_pair_mc(&tfull_bar[acc], static_cast<uint16_t>(0x3u << leader_rank));
        else
          tc_commit(&tfull_bar[acc]);
        if (++acc == Cfg::kAccStages) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs issued by this thread are complete before TMEM is released.
      if constexpr (CG == 2) tc_commit_pair(done_bar); else tc_commit(done_bar);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(done_bar, 0)) {
        if (globaltimer_ns() - t0 > p.wait_limit_ns) {
          record_error(p.err, kErrTimeout, 8);
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;                    // TMEM lane quarter of this warp
    const int half = (warp - 2) / 4;           // which alternate column chunks it takes
    uint8_t* stg = smem + Cfg::kStgOffset + (warp - 2) * Cfg::kWarpStg;
    StoreRing<Cfg::kStoreSlots, Cfg::kTmaStore> ring{stg + Cfg::kLoadBytes, 0};
    constexpr int kStreams = Cfg::kEpiStreams > 0 ? Cfg::kEpiStreams : 1;
    using Loader = typename std::conditional<
        (Cfg::kEpiStreams > 0),
        EpiLoader<BN, Cfg::kTileN, Cfg::kTileM, kStreams, Cfg::kEpiDepth, Cfg::kHalves,
                  Cfg::kInPlace>,
        NoLoader>::type;
    Loader ld{};
    if constexpr (Cfg::kEpiStreams > 0) {
      ld.p = &p;
      ld.slots = stg;
      ld.bars = ld_bar + (warp - 2) * Cfg::kEpiDepth;
      ld.tile = first_tile;
      ld.tile_stride = tile_stride;
      ld.num_tiles = p.tma_in ? num_tiles : 0;
      ld.j = 0;
      ld.row_off =
          static_cast<int32_t>(pm) * (kBM * CG) + static_cast<int32_t>(rank) * kBM + q * 32;
      ld.col_off = static_cast<int32_t>(pn) * BN;
      ld.half = half;
      ld.issued = 0;
      ld.consumed = 0;
      ld.decoded = -1;
    }
    ld.start(lane);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int32_t tile = first_tile; tile < num_tiles; tile += tile_stride) {
      const TileCoord tc = decode_tile<Cfg::kTileN, Cfg::kTileM>(p, tile);
      const int32_t row0 = tc.m0 + static_cast<int32_t>(pm) * (kBM * CG) +
                           static_cast<int32_t>(rank) * kBM + q * 32;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * Cfg::kAccCols);
      // this pair's columns of the super-tile (may be empty past the group or N end)
      const int32_t pn0 = tc.n0 + static_cast<int32_t>(pn) * BN;
      const int32_t pend = min(pn0 + BN, tc.n_end);
      if constexpr (Cfg::kZBars > 0) {
        if (!bounded_wait(&zfull_bar[acc], acc_phase, p.err, 11, p.wait_limit_ns)) break;
        tc_fence_after();
        dual_act_chunks<BN, Cfg::kHalves, Cfg::kStoreSlots, Cfg::kTmaStore>(
            p, row0, pn0, pend, t_row, ring, lane, half);
      }
      if (!bounded_wait(&tfull_bar[acc], acc_phase, p.err, 4, p.wait_limit_ns)) break;
      tc_fence_after();
      if constexpr (MODE == EPI_UPGLU) {
        epilogue_upglu<BN, CG, Cfg::kHalves, Cfg::kStoreSlots, Cfg::kTmaStore>(
            p, row0, pn0, pend, t_row, ring, lane, half,
            Cfg::kSplitRelease ? &tempty_bar[0] : nullptr,
            &tempty_bar[Cfg::kSplitRelease ? 1 : acc], leader_rank);
      } else {
        epilogue_tile<BN, MODE, Cfg::kHalves, Cfg::kStoreSlots, Cfg::kTmaStore>(
            p, tc, row0, pn0, pend, t_row, stg, ring, ld, lane,
            tc.n_blk * MCN + static_cast<int32_t>(pn), half);
      }
      if constexpr (MODE != EPI_UPGLU) {   // (the SwiGLU epilogue released its own)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          uint64_t* bar = &tempty_bar[acc];
          if constexpr (CG == 2) mbar_arrive_cluster(mapa_shared(smem_u32(bar), leader_rank));
          else mbar_arrive(bar);
        }
      }
      if (++acc == Cfg::kAccStages) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    ld.drain();
    // this warp's TMA stores have read their slots and written global memory
    if constexpr (Cfg::kTmaStore) {
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
  }

  tc_fence_before();
  if constexpr (CL > 1) cluster_sync(); else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CG == 2) tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    else tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace boost_gb300
