// LM head of the tree-verify step: z = h W^T for every tree node, with the
// softmax statistics (row max, log-sum-exp of z/temperature), argmax (lowest
// index on ties) and the top-2 gap, fused into the GEMM epilogue so that in
// greedy mode no [T, V] tensor is ever written.
// [EAGLE] workflow paragraph (page title in include/eagle.h): the frozen LM
// head gives the next-token distribution of every node.
//
// Kernels:
//   lmhead_tc_kernel       bf16: persistent tcgen05 GEMM, one 128-row tile of
//                          tree rows per CTA.  Each CTA (or cluster of up to
//                          eight CTAs, one row tile each, in pairs that issue
//                          256-row MMAs together and share every W stage by
//                          TMA multicast) owns a contiguous slice of the
//                          vocabulary and streams its rows of W once through a
//                          TMA ring; tree rows sit on TMEM lanes, so every
//                          thread owns one row and its softmax statistics are
//                          thread-local.  One partial per (row, slice).
//   lmhead_tile_kernel     CUDA-core kernel for fp32 inputs (tensor cores
//                          would round them to tf32): per-(row, 64-vocab
//                          tile) partials.
//   lmhead_finalize_kernel per (row, vocab chunk): combines the partials of
//                          the row; in PROB mode rewrites z as softmax(z/T)
//                          (LOGITS mode leaves z).
#include <math.h>

#include <algorithm>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc.cuh"

using namespace eagle;

namespace {

constexpr int kVT = 64;     // vocab rows per tile
constexpr int kRT = 64;     // tree rows per tile
constexpr int kKC = 32;     // hidden-dim chunk
constexpr int kTileThreads = 256;
constexpr int kFinThreads = 256;
constexpr int kFinChunk = 16384;  // vocab entries normalised per finalize CTA

// partial statistics of one (row, vocab tile)
struct Partial {
  float m;       // max logit in the tile
  float s;       // sum exp((z - m) / temperature) over the tile
  float second;  // second-largest logit in the tile (duplicates count)
  int idx;       // vocab index of the max (lowest on ties)
};

template <typename TIn>
__global__ void __launch_bounds__(kTileThreads)
lmhead_tile_kernel(int T, int H, int V, float temperature, const TIn* __restrict__ h,
                   const TIn* __restrict__ w, float* __restrict__ z_out,
                   Partial* __restrict__ part, int n_vtiles, int* status) {
  pdl_begin();
  __shared__ float Ws[kKC][kVT + 1];
  __shared__ float Hs[kKC][kRT + 1];
  __shared__ float Zs[kRT][kVT + 1];
  const int vt = blockIdx.x, rt = blockIdx.y;
  const int v0 = vt * kVT, r0 = rt * kRT;
  const int tid = threadIdx.x;
  const int tv = tid % 16, tr = tid / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += kKC) {
    for (int e = tid; e < kVT * kKC; e += kTileThreads) {
      const int vv = e / kKC, kk = e % kKC;
      const int v = v0 + vv, kx = k0 + kk;
      Ws[kk][vv] = (v < V && kx < H) ? to_f32(w[(size_t)v * H + kx]) : 0.f;
    }
    for (int e = tid; e < kRT * kKC; e += kTileThreads) {
      const int rr = e / kKC, kk = e % kKC;
      const int r = r0 + rr, kx = k0 + kk;
      Hs[kk][rr] = (r < T && kx < H) ? to_f32(h[(size_t)r * H + kx]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKC; ++kk) {
      float a[4], c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = Ws[kk][tv + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) c[j] = Hs[kk][tr + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], c[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) Zs[tr + 16 * j][tv + 16 * i] = acc[i][j];
  __syncthreads();
  if (z_out) {
    for (int e = tid; e < kRT * kVT; e += kTileThreads) {
      const int rr = e / kVT, vv = e % kVT;
      const int r = r0 + rr, v = v0 + vv;
      if (r < T && v < V) z_out[(size_t)r * V + v] = Zs[rr][vv];
    }
  }
  if (tid < kRT) {
    const int r = r0 + tid;
    if (r < T) {
      const int nv = min(kVT, V - v0);
      float m = -INFINITY, second = -INFINITY;
      int idx = v0;
      bool bad = false;
      for (int vv = 0; vv < nv; ++vv) {
        const float x = Zs[tid][vv];
        bad |= !isfinite(x);
        if (x > m) {
          second = m;
          m = x;
          idx = v0 + vv;
        } else if (x > second) {
          second = x;
        }
      }
      float s = 0.f;
      for (int vv = 0; vv < nv; ++vv) s += expf(__fdiv_rn(Zs[tid][vv] - m, temperature));
      if (bad) fail(status, EAGLE_ERR_NUMERIC);
      Partial p;
      p.m = m;
      p.s = s;
      p.second = second;
      p.idx = idx;
      part[(size_t)r * n_vtiles + vt] = p;
    }
  }
}

__global__ void __launch_bounds__(kFinThreads)
lmhead_finalize_kernel(int T, int V, float temperature, const Partial* __restrict__ part,
                       int n_vtiles, int32_t* argmax, float* row_max, float* row_lse,
                       float* top2_gap, float* q) {
  pdl_begin();
  __shared__ float s_f[32];
  __shared__ int s_i[32];
  __shared__ float s_m, s_lse;
  __shared__ int s_idx;
  const int r = blockIdx.x;
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  const Partial* pr = part + (size_t)r * n_vtiles;
  // global max and its lowest index
  float m = -INFINITY;
  int idx = 0x7fffffff;
  for (int t = tid; t < n_vtiles; t += blockDim.x) {
    const Partial p = pr[t];
    if (p.m > m || (p.m == m && p.idx < idx)) {
      m = p.m;
      idx = p.idx;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    if (m2 > m || (m2 == m && i2 < idx)) {
      m = m2;
      idx = i2;
    }
  }
  if (l == 0) {
    s_f[w] = m;
    s_i[w] = idx;
  }
  __syncthreads();
  if (tid == 0) {
    for (int j = 1; j < (int)(blockDim.x >> 5); ++j)
      if (s_f[j] > m || (s_f[j] == m && s_i[j] < idx)) {
        m = s_f[j];
        idx = s_i[j];
      }
    s_m = m;
    s_idx = idx;
  }
  __syncthreads();
  m = s_m;
  idx = s_idx;
  // second largest and the rescaled sum of exponentials
  float second = -INFINITY, s = 0.f;
  for (int t = tid; t < n_vtiles; t += blockDim.x) {
    const Partial p = pr[t];
    second = fmaxf(second, (p.idx == idx) ? p.second : p.m);
    s += p.s * expf(__fdiv_rn(p.m - m, temperature));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    second = fmaxf(second, __shfl_xor_sync(0xffffffffu, second, o));
    s += __shfl_xor_sync(0xffffffffu, s, o);
  }
  __syncthreads();
  if (l == 0) {
    s_f[w] = second;
    s_i[w] = __float_as_int(s);
  }
  __syncthreads();
  if (tid == 0) {
    float sec = -INFINITY, tot = 0.f;
    for (int j = 0; j < (int)(blockDim.x >> 5); ++j) {
      sec = fmaxf(sec, s_f[j]);
      tot += __int_as_float(s_i[j]);
    }
    const float lse = __fdiv_rn(m, temperature) + logf(tot);
    s_lse = lse;
    if (blockIdx.y == 0) {
      argmax[r] = idx;
      row_max[r] = m;
      row_lse[r] = lse;
      top2_gap[r] = (V >= 2) ? m - sec : INFINITY;
    }
  }
  __syncthreads();
  if (q) {
    const ProbScales sc = prob_scales(temperature, s_lse);
    const int c0 = blockIdx.y * kFinChunk, c1 = min(V, c0 + kFinChunk);
    float* row = q + (size_t)r * V;
    for (int v = c0 + tid; v < c1; v += blockDim.x) row[v] = prob_from_logit(row[v], sc);
  }
}


// ---------------------------------------------------------------------------
// tcgen05 path
//
// MMA D[t, v] = sum_k h[t, k] W[v, k]: M = 128 tree rows (TMEM lanes; rows at
// or past T are don't-care), N = one vocabulary block of up to `blk` rows
// (256), K in 64-element chunks (128-byte-swizzled K-major tiles).  The
// vocabulary is cut into balanced slices in units of 32 rows, each slice into
// blocks.  Two TMEM accumulators alternate between blocks, so the softmax
// epilogue of one block overlaps the MMAs of the next.  A W stage is one
// chunk of one block (<= blk x 128 bytes, TMA boxes of 32 rows); an h stage is
// one chunk of the CTA's tree rows.
//
// More than 128 tree rows: a cluster of C CTAs shares one vocabulary slice,
// each CTA holding its own 128-row tile of h and its own accumulators.  Every
// W stage is loaded once for the whole cluster by TMA multicast, and a stage
// is refilled only after every MMA issuer of the cluster has released it
// (the MMA commit arrives on the stage's barrier in every CTA).  W then
// streams from memory once per 128*C tree rows.  The CTAs form pairs
// (cta_group::2; an odd tile count gets one CTA of rows past T): the even
// CTA of a pair issues MMAs of M = 256 (its rows, then its peer's) x N = 256,
// each CTA holding its own h tile and one 128-row half of every W stage
// (even CTAs the first half, odd CTAs the second, each half multicast to the
// CTAs of its parity).  So each SM receives and reads half of every W stage
// instead of all of it, per MMA of its own 128 rows.  The odd CTA reports
// each of its stages to the even one as it lands (a remote mbarrier arrive),
// and its epilogue releases the accumulators into the even CTA's barrier.
// W and h are requested by two threads of their own, so the W ring (from
// memory) runs as far ahead as its stages allow while the h ring (from L2)
// keeps fewer.  W never depends on an earlier kernel, so the first W stages
// are requested before the kernel waits for its predecessor.
// ---------------------------------------------------------------------------
// warp 0 W copies, warp 1 MMA (or, in the odd CTA of a pair, stage reports),
// warps 2-9 epilogue, warp 10 h copies
constexpr int kTcThreads = 352;
constexpr int kHWarp = 10;
constexpr int kEpiWarps = 8;      // two per TMEM lane quarter, one per column half
constexpr int kBK = 64;           // bf16 per 128-byte swizzled row (one chunk)
constexpr int kUnit = 32;         // vocabulary rows per TMA box
constexpr int kBlkMax = 256;      // vocabulary rows per MMA (its N), at most
constexpr int kTileRows = 128;    // tree rows per CTA (the MMA's M)
// Row tiles sharing one W stream: at most a portable cluster of 8 (a
// build-time option, so that other cluster caps can be measured).
#ifndef EAGLE_LMHEAD_MAX_CLUSTER
#define EAGLE_LMHEAD_MAX_CLUSTER 8
#endif
constexpr int kMaxCluster = EAGLE_LMHEAD_MAX_CLUSTER;
constexpr int kMaxHStages = 6;       // h ring barriers held (stages used: 4 or kBigHStages)
// h stages of a CTA that takes the whole shared memory (a build-time option,
// so that the split between the h and W rings can be measured)
#ifndef EAGLE_LMHEAD_BIG_HSTAGES
#define EAGLE_LMHEAD_BIG_HSTAGES 4
#endif
constexpr int kBigHStages = EAGLE_LMHEAD_BIG_HSTAGES;
static_assert(kBigHStages >= 1 && kBigHStages <= kMaxHStages, "h stages beyond the barriers held");
// Cluster launches (row tiles sharing W) pair their CTAs: cta_group::2 MMAs
// of M = 256 over two SMs, each SM holding its own 128 tree rows and half of
// every W stage, so each SM writes and reads half the W bytes per MMA of
// its own rows (a build-time option, so that unpaired clusters can be
// measured).
#ifndef EAGLE_LMHEAD_PAIR
#define EAGLE_LMHEAD_PAIR 1
#endif
constexpr bool kPairCluster = EAGLE_LMHEAD_PAIR != 0;
constexpr int kPairRows = 2 * kTileRows;   // tree rows of one pair MMA (its M)
// Unpaired cluster launches use 512-row blocks over both TMEM accumulators
// (each h chunk then serves two W halves); paired ones 256-row blocks in
// alternating accumulators, so that the epilogue of one block overlaps the
// MMAs of the next (a build-time option, so that both can be measured).
#ifndef EAGLE_LMHEAD_DUAL
#define EAGLE_LMHEAD_DUAL (EAGLE_LMHEAD_PAIR ? 0 : 1)
#endif
constexpr bool kDualCluster = EAGLE_LMHEAD_DUAL != 0;
constexpr int kMaxWStages = 12;
constexpr size_t kSmemLimit = 227 * 1024;
// A W ring within this budget (when it still holds four stages) leaves room
// on the SM for one CTA of the tree expand (up to ~55 KB), which the step
// runs concurrently with the LM head.
constexpr size_t kSmemShared = 171 * 1024;
constexpr int kSmsForOthers = 16;
constexpr size_t kTcSharedBytes = 1024 + 2 * 128 * 16;
// LOGITS / PROB mode: every epilogue warp stages its 32 rows x 8 logits in one
// of two 1 KB shared-memory boxes (32-byte swizzle) and writes them with a
// bulk tensor store, so each global write covers whole 32-byte row segments
// instead of one 16-byte piece of 32 rows per store instruction.
constexpr int kZBoxCols = 8;
constexpr int kZBoxBytes = 32 * kZBoxCols * 4;
constexpr size_t kZStageBytes = (size_t)8 * 2 * kZBoxBytes;   // 8 warps x 2 boxes

struct TcShared {
  uint64_t h_full[kMaxHStages], h_empty[kMaxHStages];
  uint64_t w_full[kMaxWStages], w_empty[kMaxWStages];
  uint64_t tmem_full[2], tmem_empty[2], xbar, drain;
  uint32_t tmem_base;
  int abort_flag;
  Partial xchg[128];   // column half 1's partial of every row
};

static_assert(sizeof(TcShared) <= kTcSharedBytes, "TcShared must fit its shared-memory slot");

struct TcLayout {
  int h_rows, h_stage_bytes, h_stages, blk, w_stage_bytes, w_stages;
  bool z_tma;   // logits staged for bulk tensor stores
  size_t smem;
};

// `h_rows`: tree rows of one h stage (one CTA's tile, rounded up to 8);
// `z_tma`: logits are written and the staging boxes should be held when
// they fit beside the rings (a smaller CTA writes logits directly).
// `pair`: a CTA of a pair holds half of every W stage.
TcLayout tc_layout(int h_rows, bool z_tma, bool pair = false) {
  TcLayout L;
  L.h_rows = h_rows;
  L.h_stage_bytes = h_rows * 128;
  // 256-row blocks: narrower MMAs cost more shared-memory reads per W byte
  // than the overlap of a short slice's epilogue gains
  L.blk = kBlkMax;
  L.h_stages = 4;
  L.w_stage_bytes = (pair ? L.blk / 2 : L.blk) * 128;
  size_t fixed = 1024 + (size_t)L.h_stages * L.h_stage_bytes + kTcSharedBytes;
  // a pair takes the whole shared memory: its W ring (16 KB stages) covers
  // the memory latency only with about eight stages
  size_t limit = pair ? kSmemLimit : kSmemShared;
  if (!pair && fixed + 4 * (size_t)L.w_stage_bytes > kSmemShared) {
    // the whole shared memory, split between the h ring (re-read from L2
    // for every block) and the W ring (measured at 128 rows x 4096 x 128256
    // in clusters of six: 3 h + 5 W stages 881 us, 4 + 4 781 us, 2 + 6
    // 1199 us)
    limit = kSmemLimit;
    L.h_stages = kBigHStages;
    fixed = 1024 + (size_t)L.h_stages * L.h_stage_bytes + kTcSharedBytes;
  }
  // the staging boxes only where four W stages still fit beside them
  L.z_tma = z_tma && fixed + kZStageBytes + 4 * (size_t)L.w_stage_bytes <= limit;
  if (L.z_tma) fixed += kZStageBytes;
  L.w_stages = (int)std::min<size_t>(kMaxWStages, (limit - fixed) / L.w_stage_bytes);
  L.smem = fixed + (size_t)L.w_stages * L.w_stage_bytes;
  return L;
}

// 2^x by the SFU's approximate exponential (relative error about 2^-22;
// subnormal results flush to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Merge partial b into a (same row, disjoint vocabulary): the max with the
// lowest index on ties; the loser's max competes for second place.
__device__ __forceinline__ void merge_partial(Partial& a, const Partial& b, float k2) {
  if (b.m == -INFINITY) return;
  if (a.m == -INFINITY) {
    a = b;
    return;
  }
  const bool b_wins = (b.m > a.m) || (b.m == a.m && b.idx < a.idx);
  const Partial& w = b_wins ? b : a;
  const Partial& o = b_wins ? a : b;
  Partial r;
  r.m = w.m;
  r.idx = w.idx;
  r.second = fmaxf(w.second, o.m);
  r.s = w.s + o.s * ex2_approx((o.m - w.m) * k2);
  a = r;
}

// T: tree rows of this launch (at most 128 * C); C: CTAs per cluster, 1
// exactly when MULTI is false.  Partials go to part[t * slices + slice].
// DUAL: a block is blk_max = 512 vocabulary rows, its two 256-row halves
// accumulated in the two TMEM accumulators by turns for every h chunk, so
// each h chunk serves twice the MMA work (half the h traffic and twice the
// time to refill an h stage); the epilogue of a block then no longer
// overlaps the next block's MMAs.  Otherwise a block is one accumulator and
// consecutive blocks alternate.
template <bool MULTI, bool DUAL, bool PAIR>
__global__ void __launch_bounds__(kTcThreads, 1)
lmhead_tc_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_w,
                 const __grid_constant__ CUtensorMap map_z, int T, int H, int V,
                 float temperature, float* __restrict__ z_out, int z_tma,
                 Partial* __restrict__ part, int n_units, int h_stage_bytes, int h_stages,
                 int blk_max, int w_stages, int C, int* status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* h_smem = base;
  unsigned char* w_smem = base + h_stages * h_stage_bytes;
  static_assert(!PAIR || MULTI, "pairs are cluster launches");
  const int w_rows_max = DUAL ? blk_max / 2 : blk_max;   // W rows of one stage
  // PAIR: a CTA holds rows 0-127 (even rank) or 128-255 (odd) of every stage
  const int w_stage_bytes = (PAIR ? w_rows_max / 2 : w_rows_max) * 128;
  TcShared* sh = reinterpret_cast<TcShared*>(w_smem + (size_t)w_stages * w_stage_bytes);
  // logit staging boxes (1024-byte aligned: every ring stage is a multiple of 1 KB)
  unsigned char* z_smem = w_smem + (size_t)w_stages * w_stage_bytes + kTcSharedBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!MULTI) C = 1;
  const int rank = MULTI ? (int)tc::cluster_ctarank() : 0;   // this CTA's row tile
  const uint16_t all_ctas = (uint16_t)((1u << C) - 1u);
  // PAIR: par 0 is the pair's leader (it issues the pair's MMAs); a W box
  // goes to the CTAs of one parity (`group`), requested by each of them in
  // turn
  const int par = PAIR ? (rank & 1) : 0;
  const int leader = rank & ~1;
  const int groups = PAIR ? C / 2 : C;
  const int gi = PAIR ? rank >> 1 : rank;
  const uint16_t group_mask = PAIR ? (uint16_t)((par ? 0xAAAAu : 0x5555u) & all_ctas) : all_ctas;
  const uint16_t pair_mask = (uint16_t)(3u << leader);
  const int slices = gridDim.x / C;
  const int slice = blockIdx.x / C;
  // the cluster's slice of the vocabulary: rows [r_begin, r_end), 32-row units
  const int u0 = (int)((long long)n_units * slice / slices);
  const int u1 = (int)((long long)n_units * (slice + 1) / slices);
  const int r_begin = u0 * kUnit, r_end = u1 * kUnit;
  const int n_blocks = (r_end - r_begin + blk_max - 1) / blk_max;
  const int KB = (H + kBK - 1) / kBK;
  auto blk_rows = [&](int blk) { return min(blk_max, r_end - (r_begin + blk * blk_max)); };
  // W stages of a block's chunk (halves with rows), their rows and first row
  auto n_halves = [&](int blk) { return (DUAL && blk_rows(blk) > w_rows_max) ? 2 : 1; };
  auto half_rows = [&](int blk, int hf) { return min(w_rows_max, blk_rows(blk) - hf * w_rows_max); };
  auto half_y0 = [&](int blk, int hf) { return r_begin + blk * blk_max + hf * w_rows_max; };
  // W stages in all, (block, chunk, half) block-major
  const int total = n_blocks == 0 ? 0 : ((n_blocks - 1) * n_halves(0) + n_halves(n_blocks - 1)) * KB;
  // this CTA's share of a W stage (chunk kb of the block at row y0):
  // boxes rank, rank + C, ... (multicast to all)
  auto load_w_box = [&](int stage, int rows, int kb, int y0, uint64_t pol) {
    if (PAIR) {
      // this CTA's half; rows past the block are never read by the epilogue
      rows = min(w_rows_max / 2, max(0, rows - par * (w_rows_max / 2)));
      y0 += par * (w_rows_max / 2);
    }
    tc::mbar_arrive_expect_tx(&sh->w_full[stage], (uint32_t)(rows * 128));
    unsigned char* dst = w_smem + (size_t)stage * w_stage_bytes;
    for (int u = gi * kUnit; u < rows; u += groups * kUnit) {
      if (MULTI)
        tc::tma_load_2d_mc_hint(dst + u * 128, &map_w, &sh->w_full[stage], kb * kBK, y0 + u,
                                group_mask, pol);
      else
        tc::tma_load_2d_hint(dst + u * 128, &map_w, &sh->w_full[stage], kb * kBK, y0 + u, pol);
    }
  };
  // W stages requested before waiting for the previous kernel
  const int w_early = min(w_stages, total);

  if (threadIdx.x == 0) {
    // a leader's stages are full once its own copies landed and its peer
    // reported its own; its accumulators are free once both CTAs' epilogues
    // have read them
    const uint32_t full_count = (PAIR && par == 0) ? 2 : 1;
    for (int i = 0; i < h_stages; ++i) {
      tc::mbar_init(&sh->h_full[i], full_count);
      tc::mbar_init(&sh->h_empty[i], 1);
    }
    for (int i = 0; i < w_stages; ++i) {
      tc::mbar_init(&sh->w_full[i], full_count);
      tc::mbar_init(&sh->w_empty[i], PAIR ? C / 2 : C);   // every MMA issuer releases the stage
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sh->tmem_full[i], 1);
      tc::mbar_init(&sh->tmem_empty[i], (PAIR && par == 0) ? 2 * kEpiWarps : kEpiWarps);
    }
    tc::mbar_init(&sh->xbar, 32 * kEpiWarps);
    tc::mbar_init(&sh->drain, 1);
    sh->abort_flag = 0;
    tc::fence_barrier_init();
  }
  // the peers' barriers exist before any multicast reaches them
  if (MULTI) tc::cluster_sync_all();
  if (threadIdx.x == 0) {
    tc::prefetch_tensormap(&map_h);
    tc::prefetch_tensormap(&map_w);
    const uint64_t pol_w = tc::policy_evict_first();
    int i = 0;
    for (int blk = 0; blk < n_blocks && i < w_early; ++blk)
      for (int kb = 0; kb < KB && i < w_early; ++kb)
        for (int hf = 0; hf < n_halves(blk) && i < w_early; ++hf, ++i)
          load_w_box(i, half_rows(blk, hf), kb, half_y0(blk, hf), pol_w);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tc::tmem_alloc_pair(&sh->tmem_base, 512);
      tc::tmem_relinquish_pair();
    } else {
      tc::tmem_alloc(&sh->tmem_base, 512);
      tc::tmem_relinquish();
    }
  }
  pdl_begin();   // h (and the outputs) follow the previous kernel
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int* abort_flag = &sh->abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ W copies
    if (lane == 0) {
      const uint64_t pol_w = tc::policy_evict_first();
      // W stage i (past the ones requested early) as soon as its slot is
      // free; nested loops keep divisions off the refill path
      int ws = 0, issued_w = w_early;
      uint32_t wph = 0;
      bool ok = true;
      int i = 0;
      for (int blk = 0; blk < n_blocks && ok; ++blk) {
        const int nh = n_halves(blk);
        for (int kb = 0; kb < KB && ok; ++kb) {
          for (int hf = 0; hf < nh && ok; ++hf, ++i) {
            if (i >= w_early) {
              if (!(ok = tc::mbar_wait(&sh->w_empty[ws], wph ^ 1, abort_flag, status))) break;
              load_w_box(ws, half_rows(blk, hf), kb, half_y0(blk, hf), pol_w);
              ++issued_w;
            }
            if (++ws == w_stages) { ws = 0; wph ^= 1; }
          }
        }
      }
      if (ok && MULTI) {
        // the last release of every stage, the peers' included, has arrived:
        // nothing more reaches this CTA's shared memory
        for (int i = max(0, total - w_stages); i < total && ok; ++i)
          ok = tc::mbar_wait(&sh->w_empty[i % w_stages], (i / w_stages) & 1, abort_flag, status);
      }
      if (!ok) {
        // let every copy still in flight land before the CTA exits
        // (the last copy issued into each slot: waiting for its phase
        // returns at once if it has landed, whether consumed or not)
        int never = 0;
        for (int i = max(0, issued_w - w_stages); i < issued_w; ++i)
          tc::mbar_wait(&sh->w_full[i % w_stages], (i / w_stages) & 1, &never, nullptr,
                        200000000ll);
      }
    }
  } else if (warp == kHWarp) {
    // ------------------------------------------------------------ h copies
    // (a ring of its own, so that the W ring runs as far ahead as its
    // stages allow: h comes from L2, W from memory)
    if (lane == 0) {
      const uint64_t pol_h = tc::policy_evict_last();
      int hs = 0, issued_h = 0;
      uint32_t hph = 0;
      bool ok = true;
      for (int blk = 0; blk < n_blocks && ok; ++blk) {
        for (int kb = 0; kb < KB && ok; ++kb) {
          if (!(ok = tc::mbar_wait(&sh->h_empty[hs], hph ^ 1, abort_flag, status))) break;
          tc::mbar_arrive_expect_tx(&sh->h_full[hs], (uint32_t)h_stage_bytes);
          tc::tma_load_2d_hint(h_smem + hs * h_stage_bytes, &map_h, &sh->h_full[hs], kb * kBK,
                               rank * kTileRows, pol_h);
          ++issued_h;
          if (++hs == h_stages) { hs = 0; hph ^= 1; }
        }
      }
      if (!ok) {
        int never = 0;
        for (int i = max(0, issued_h - h_stages); i < issued_h; ++i)
          tc::mbar_wait(&sh->h_full[i % h_stages], (i / h_stages) & 1, &never, nullptr,
                        200000000ll);
      }
    }
  } else if (warp == 1 && PAIR && par == 1) {
    // ------------------------------------------------------------ pair peer
    // The leader issues the pair's MMAs: report every h and W stage of this
    // CTA to it as soon as the stage has landed here.
    if (lane == 0) {
      int hs = 0, ws = 0;
      uint32_t hph = 0, wph = 0;
      bool ok = true;
      for (int blk = 0; blk < n_blocks && ok; ++blk) {
        const int nh = n_halves(blk);
        for (int kb = 0; kb < KB && ok; ++kb) {
          if (!(ok = tc::mbar_wait(&sh->h_full[hs], hph, abort_flag, status))) break;
          tc::mbar_arrive_remote<true>(&sh->h_full[hs], (uint32_t)leader);
          if (++hs == h_stages) { hs = 0; hph ^= 1; }
          for (int hf = 0; hf < nh && ok; ++hf) {
            if (!(ok = tc::mbar_wait(&sh->w_full[ws], wph, abort_flag, status))) break;
            tc::mbar_arrive_remote<true>(&sh->w_full[ws], (uint32_t)leader);
            if (++ws == w_stages) { ws = 0; wph ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Each W stage is released (its MMAs committed) as soon as its MMAs are
    // issued: with clusters, a stage is refilled only once every CTA has
    // released it, so an early release keeps the shared ring full.
    if (lane == 0) {
      int hs = 0, ws = 0;
      uint32_t hph = 0, wph = 0, tph = 0;   // tph bit b: phase of accumulator b
      bool ok = true;
      for (int blk = 0; blk < n_blocks && ok; ++blk) {
        const int ab = DUAL ? 0 : (blk & 1);
        if (!(ok = tc::mbar_wait(&sh->tmem_empty[ab], ((tph >> ab) & 1u) ^ 1u, abort_flag,
                                       status)))
          break;
        tph ^= 1u << ab;
        tc::fence_after_thread_sync();
        const int nh = n_halves(blk);
        for (int kb = 0; kb < KB && ok; ++kb) {
          if (!(ok = tc::mbar_wait(&sh->h_full[hs], hph, abort_flag, status))) break;
          const uint64_t da = tc::desc_kmajor_sw128(tc::smem_u32(h_smem + hs * h_stage_bytes));
          const uint32_t acc = kb > 0 ? 1u : 0u;
          for (int hf = 0; hf < nh && ok; ++hf) {
            if (!(ok = tc::mbar_wait(&sh->w_full[ws], wph, abort_flag, status))) break;
            tc::fence_after_thread_sync();
            // DUAL: half hf accumulates at TMEM column 256 * hf
            const uint32_t d = tmem + (uint32_t)((ab + hf) * kBlkMax);
            const uint64_t db =
                tc::desc_kmajor_sw128(tc::smem_u32(w_smem + (size_t)ws * w_stage_bytes));
            // K steps of 16 advance the descriptors' start address by 32 bytes
            if constexpr (PAIR) {
              // always all 256 columns: those past the block are never read
              const uint32_t idesc = tc::idesc_bf16_f32(kPairRows, kBlkMax);
              tc::mma_f16_pair(d, da, db, idesc, acc);
              tc::mma_f16_pair(d, da + 2, db + 2, idesc, 1u);
              tc::mma_f16_pair(d, da + 4, db + 4, idesc, 1u);
              tc::mma_f16_pair(d, da + 6, db + 6, idesc, 1u);
              tc::mma_commit_pair_mc(&sh->w_empty[ws], all_ctas);
            } else {
              const uint32_t idesc = tc::idesc_bf16_f32(128, half_rows(blk, hf));
              tc::mma_f16(d, da, db, idesc, acc);
              tc::mma_f16(d, da + 2, db + 2, idesc, 1u);
              tc::mma_f16(d, da + 4, db + 4, idesc, 1u);
              tc::mma_f16(d, da + 6, db + 6, idesc, 1u);
              if (MULTI)
                tc::mma_commit_mc(&sh->w_empty[ws], all_ctas);
              else
                tc::mma_commit(&sh->w_empty[ws]);
            }
            if (++ws == w_stages) { ws = 0; wph ^= 1; }
          }
          if (!ok) break;
          if constexpr (PAIR)
            tc::mma_commit_pair_mc(&sh->h_empty[hs], pair_mask);
          else
            tc::mma_commit(&sh->h_empty[hs]);
          if (++hs == h_stages) { hs = 0; hph ^= 1; }
        }
        if (ok) {
          if constexpr (PAIR)
            tc::mma_commit_pair_mc(&sh->tmem_full[ab], pair_mask);
          else
            tc::mma_commit(&sh->tmem_full[ab]);
        }
      }
      // every MMA issued by this thread has finished before TMEM is freed
      if constexpr (PAIR)
        tc::mma_commit_pair_mc(&sh->drain, (uint16_t)(1u << rank));
      else
        tc::mma_commit(&sh->drain);
      int never = 0;
      tc::mbar_wait(&sh->drain, 0, &never, nullptr, 200000000ll);
    }
  } else if (warp >= 2 && warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int chalf = (warp - 2) >> 2;   // second or first half of every block's columns
    const int t = rank * kTileRows + quad * 32 + lane;   // tree row held by this thread
    const bool row_ok = t < T;
    const bool quad_live = rank * kTileRows + quad * 32 < T;   // warp-uniform
    const float k2 = 1.4426950408889634f / temperature;   // log2(e) / temperature
    const bool vec = ((V & 3) == 0);
    Partial p;
    p.m = -INFINITY;
    p.s = 0.f;
    p.second = -INFINITY;
    p.idx = 0x7fffffff;
    bool bad = false;
    uint32_t tph = 0;
    // this warp's two staging boxes: row `lane` at lane * 32 bytes, its two
    // 16-byte halves swapped on rows 4-7 of every 8 (the 32-byte swizzle)
    unsigned char* zbox = z_smem + (size_t)(warp - 2) * 2 * kZBoxBytes;
    const int zsw = (lane >> 2) & 1;
    int zb = 0;
    for (int blk = 0; blk < n_blocks; ++blk) {
      const int ab = DUAL ? 0 : (blk & 1);
      const int rows = blk_rows(blk);
      // every lane waits; the warp proceeds only if all of them saw the phase
      const bool got =
          tc::mbar_wait(&sh->tmem_full[ab], (tph >> ab) & 1u, abort_flag, status);
      if (!__all_sync(0xffffffffu, got)) break;
      tph ^= 1u << ab;
      tc::fence_after_thread_sync();
      const int half_cols = blk_max / 2;
      for (int c = chalf * half_cols; c < (chalf + 1) * half_cols && c < rows && quad_live;
           c += 32) {
        float v[32];
        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(quad * 32) << 16) +
                                   (uint32_t)(ab * kBlkMax + c), v);
        const int vb = r_begin + blk * blk_max + c;
        const int nvalid = min(min(32, rows - c), V - vb);
        if (z_tma && nvalid > 0) {
          // boxes of 8 columns x the warp's 32 rows; columns past V and rows
          // past T fall outside the tensor and are not written
#pragma unroll
          for (int j = 0; j < 32; j += kZBoxCols) {
            if (vb + j < V) {   // warp-uniform
              unsigned char* box = zbox + zb * kZBoxBytes;
              if (lane == 0) tc::bulk_wait_read<1>();   // the box's previous store has read it
              __syncwarp();
              float4* row = reinterpret_cast<float4*>(box + lane * 32);
              row[zsw] = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
              row[zsw ^ 1] = make_float4(v[j + 4], v[j + 5], v[j + 6], v[j + 7]);
              tc::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tc::tma_store_2d(&map_z, box, vb + j, rank * kTileRows + quad * 32);
                tc::bulk_commit();
              }
              zb ^= 1;
            }
          }
        }
        if (!row_ok || nvalid <= 0) continue;
        bool fin = true;
        if (nvalid == 32) {
#pragma unroll
          for (int i = 0; i < 32; ++i) fin &= fabsf(v[i]) < INFINITY;
        } else {
          // ragged end of the vocabulary: only real entries count
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i < nvalid) fin &= fabsf(v[i]) < INFINITY;
            else v[i] = -INFINITY;
          }
        }
        bad |= !fin;
        if (z_out && !z_tma) {
          float* dst = z_out + (size_t)t * V + vb;
          if (vec && nvalid == 32) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < nvalid) dst[i] = v[i];
          }
        }
        float cm = -INFINITY, cs = -INFINITY;
        int ci = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float x = v[i];
          if (x > cm) {
            cs = cm;
            cm = x;
            ci = i;
          } else if (x > cs) {
            cs = x;
          }
        }
        if (cm > p.m) {
          p.second = fmaxf(p.m, cs);
          p.s = (p.m == -INFINITY) ? 0.f : p.s * ex2_approx((p.m - cm) * k2);
          p.m = cm;
          p.idx = vb + ci;
        } else {
          p.second = fmaxf(p.second, cm);
        }
        const float mk = p.m * k2;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          a0 += ex2_approx(fmaf(v[i], k2, -mk));
          a1 += ex2_approx(fmaf(v[i + 1], k2, -mk));
        }
        p.s += a0 + a1;
      }
      tc::fence_before_thread_sync();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && par == 1)
          tc::mbar_arrive_remote(&sh->tmem_empty[ab], (uint32_t)leader);
        else
          tc::mbar_arrive(&sh->tmem_empty[ab]);
      }
    }
    // the logits are written before the kernel ends
    if (z_tma && lane == 0) tc::bulk_wait_all();
    if (bad) fail(status, EAGLE_ERR_NUMERIC);
    // the two column halves of every row: half 1 hands its partial to half 0
    const int tl = quad * 32 + lane;
    if (chalf == 1) sh->xchg[tl] = p;
    tc::mbar_arrive(&sh->xbar);
    const bool gx = tc::mbar_wait(&sh->xbar, 0, abort_flag, status);
    if (chalf == 0 && row_ok && gx) {
      merge_partial(p, sh->xchg[tl], k2);
      part[(size_t)t * slices + slice] = p;
    }
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  if constexpr (PAIR) {
    // both CTAs' epilogues are past their last TMEM read and the leader's
    // MMAs have finished before the pair frees its columns; no CTA leaves
    // while a peer may still deliver into its shared memory
    tc::cluster_sync_all();
    if (warp == 1) {
      tc::fence_after_thread_sync();
      tc::tmem_dealloc_pair(tmem, 512);
    }
  } else {
    if (warp == 1) {
      tc::fence_after_thread_sync();
      tc::tmem_dealloc(tmem, 512);
    }
    // no CTA leaves while a peer may still deliver into its shared memory
    if (MULTI) tc::cluster_sync_all();
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), 128-byte swizzled boxes of
// 64 columns x box_rows rows; out-of-range elements read as zero.
bool make_map_bf16(CUtensorMap* map, const void* ptr, int rows, int cols, int box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp32 logits [rows, cols] (cols contiguous, cols % 4 == 0) written in
// boxes of kZBoxCols columns x 32 rows from 32-byte-swizzled shared memory.
bool make_map_z(CUtensorMap* map, float* ptr, int rows, int cols) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {(cuuint32_t)kZBoxCols, 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int n[kMaxDevices] = {};
  const int dev = current_device_slot();
  if (!n[dev]) {
    int c = 0;
    int d = 0;
    cudaGetDevice(&d);
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || c <= 0)
      c = 148;
    n[dev] = c;
  }
  return n[dev];
}

// Clusters of C tensor-core CTAs that fit on the current GPU at once (0:
// none), per device and shared-memory size.
int max_clusters(int C, size_t smem) {
  static std::mutex mu;
  static int cached_all[kMaxDevices][kMaxCluster + 1] = {};
  static size_t cached_smem[kMaxDevices][kMaxCluster + 1] = {};
  std::lock_guard<std::mutex> lock(mu);
  const int dev = current_device_slot();
  int* cached = cached_all[dev];
  if (cached_smem[dev][C] != smem) {
    cached[C] = 0;
    cached_smem[dev][C] = smem;
  }
  if (!cached[C]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(C * 64));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(
            &n, (const void*)lmhead_tc_kernel<true, kDualCluster, kPairCluster>,
            &cfg) !=
        cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cached[C] = n > 0 ? n : -1;
  }
  return std::max(cached[C], 0);
}

// The tensor-core kernel with programmatic dependent launch, in clusters of
// C CTAs when C > 1.
template <typename... Args>
cudaError_t launch_tc(int C, dim3 grid, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (C > 1) ? 2 : 1;
  return (C > 1) ? cudaLaunchKernelEx(
                       &cfg, lmhead_tc_kernel<true, kDualCluster, kPairCluster>,
                       std::forward<Args>(args)...)
                 : cudaLaunchKernelEx(&cfg, lmhead_tc_kernel<false, false, false>,
                                      std::forward<Args>(args)...);
}

}  // namespace

// One partial per (row, vocab tile of 64) on the CUDA-core path and per
// (row, CTA) on the tensor-core path, whose CTAs each own at least 16 rows.
extern "C" size_t eagle_lmhead_workspace_bytes(int T, int V) {
  if (T < 0 || V < 1) return 0;
  return (size_t)T * ((V + 15) / 16) * sizeof(Partial);
}

extern "C" eagle_status eagle_lmhead_softmax(eagle_dtype dtype, int T, int H, int V,
                                             float temperature, int mode, const void* d_h,
                                             const void* d_w, int32_t* d_argmax,
                                             float* d_row_max, float* d_row_lse,
                                             float* d_top2_gap, float* d_q, void* d_ws,
                                             size_t ws_bytes, int* d_status,
                                             eagle_stream_t stream) {
  EAGLE_HOST_CHECK(T >= 0 && H >= 1 && V >= 1, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(temperature > 0.f && isfinite(temperature), EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(mode == EAGLE_LMHEAD_GREEDY || mode == EAGLE_LMHEAD_PROB ||
                       mode == EAGLE_LMHEAD_LOGITS,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(dtype == EAGLE_F32 || dtype == EAGLE_BF16, EAGLE_ERR_UNSUPPORTED);
  if (T == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_h && d_w && d_argmax && d_row_max && d_row_lse && d_top2_gap && d_status,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(mode == EAGLE_LMHEAD_GREEDY || d_q, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(ws_bytes >= eagle_lmhead_workspace_bytes(T, V) && d_ws, EAGLE_ERR_WORKSPACE);
  cudaStream_t s = (cudaStream_t)stream;
  Partial* part = static_cast<Partial*>(d_ws);
  float* z = (mode == EAGLE_LMHEAD_GREEDY) ? nullptr : d_q;
  // PROB mode normalises the logits in place afterwards; LOGITS keeps them
  float* q_norm = (mode == EAGLE_LMHEAD_PROB) ? d_q : nullptr;
  const bool tc_ok = dtype == EAGLE_BF16 && (H % 8) == 0 &&
                     (((uintptr_t)d_h | (uintptr_t)d_w) & 15) == 0 &&
                     (!z || ((uintptr_t)z & 15) == 0);
  if (tc_ok) {
    CUtensorMap map_w;
    if (!make_map_bf16(&map_w, d_w, V, H, kUnit)) return EAGLE_ERR_CUDA;
    static PerDeviceOnce attr_once;
    // the whole unified L1 as shared memory, so that a CTA of the
    // concurrently running tree expand fits beside this one
    if (attr_once.run([] {
          cudaError_t e = cudaFuncSetAttribute(lmhead_tc_kernel<false, false, false>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kSmemLimit);
          if (e == cudaSuccess)
            e = cudaFuncSetAttribute(
                lmhead_tc_kernel<true, kDualCluster, kPairCluster>,
                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
          if (e == cudaSuccess)
            e = cudaFuncSetAttribute(lmhead_tc_kernel<false, false, false>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
          return e;
        }) != cudaSuccess)
      return EAGLE_ERR_CUDA;
    const int n_units = (V + kUnit - 1) / kUnit;
    // Row tiles of 128, one CTA each; the tiles of one launch form clusters
    // that share the W stream.  As few launches as the largest resident
    // cluster allows, with the tiles spread evenly over them (every CTA of
    // a launch holds real rows), so W is streamed once per launch.
    const int tiles = (T + kTileRows - 1) / kTileRows;
    // logits through bulk tensor stores need 16-byte row strides
    const bool z_want = z && (V % 4) == 0;
    const size_t tile_smem = tc_layout(kTileRows, z_want, kPairCluster).smem;
    // CTAs of a cluster of c row tiles: paired clusters take an even count
    // (a last CTA past the rows computes zero rows and writes nothing)
    auto ctas = [](int c) { return (kPairCluster && c > 1) ? (c + 1) & ~1 : c; };
    int passes = 1, C = tiles;
    while (C > 1 && (ctas(C) > kMaxCluster || max_clusters(ctas(C), tile_smem) < 1)) {
      ++passes;
      C = (tiles + passes - 1) / passes;
    }
    // one slice per resident cluster of C CTAs; one tile: leave a few SMs to
    // the attention, which the step runs while the LM head is still
    // streaming W (it does not fit beside an LM head CTA)
    const int slices =
        (C > 1) ? std::min(max_clusters(ctas(C), tile_smem), n_units)
                : std::min(std::max(1, sm_count() - kSmsForOthers), n_units);
    for (int p = 0, tile0 = 0; p < passes; ++p) {
      const int nt = std::min(C, tiles - tile0);    // tiles of this launch
      const int r0 = tile0 * kTileRows;
      const int Ts = std::min(nt * kTileRows, T - r0);
      tile0 += nt;
      const int Cp = (C > 1) ? ctas(nt) : 1;
      const TcLayout TL =
          tc_layout((Cp > 1 || Ts > kTileRows) ? kTileRows : ((Ts + 7) / 8) * 8, z_want,
                    Cp > 1 && kPairCluster);
      const __nv_bfloat16* hs = static_cast<const __nv_bfloat16*>(d_h) + (size_t)r0 * H;
      float* zs = z ? z + (size_t)r0 * V : nullptr;
      CUtensorMap map_h, map_z = map_w;   // without staging map_z is never read
      if (!make_map_bf16(&map_h, hs, Ts, H, TL.h_rows)) return EAGLE_ERR_CUDA;
      if (TL.z_tma && !make_map_z(&map_z, zs, Ts, V)) return EAGLE_ERR_CUDA;
      // a last launch with fewer tiles keeps the slice count of the others
      // (its clusters are smaller, so they are resident too)
      if (launch_tc(Cp, dim3(slices * Cp), TL.smem, s, map_h, map_w, map_z, Ts, H, V,
                    temperature, zs, (int)TL.z_tma, part + (size_t)r0 * slices, n_units,
                    TL.h_stage_bytes, TL.h_stages,
                    (Cp > 1 && kDualCluster) ? 2 * TL.blk : TL.blk, TL.w_stages,
                    Cp,
                    d_status) !=
          cudaSuccess)
        return EAGLE_ERR_CUDA;
    }
    dim3 fgrid(T, q_norm ? (V + kFinChunk - 1) / kFinChunk : 1);
    return launch_status(launch_pdl(lmhead_finalize_kernel, fgrid, dim3(kFinThreads), 0, s, T, V,
                                    temperature, (const Partial*)part, slices, d_argmax, d_row_max,
                                    d_row_lse, d_top2_gap, q_norm));
  }
  const int n_vtiles = (V + kVT - 1) / kVT;
  dim3 grid(n_vtiles, (T + kRT - 1) / kRT);
  cudaError_t e;
  if (dtype == EAGLE_BF16)
    e = launch_pdl(lmhead_tile_kernel<__nv_bfloat16>, grid, dim3(kTileThreads), 0, s, T, H, V,
                   temperature, static_cast<const __nv_bfloat16*>(d_h),
                   static_cast<const __nv_bfloat16*>(d_w), z, part, n_vtiles, d_status);
  else
    e = launch_pdl(lmhead_tile_kernel<float>, grid, dim3(kTileThreads), 0, s, T, H, V,
                   temperature, static_cast<const float*>(d_h), static_cast<const float*>(d_w), z,
                   part, n_vtiles, d_status);
  if (e != cudaSuccess) return EAGLE_ERR_CUDA;
  dim3 fgrid(T, q_norm ? (V + kFinChunk - 1) / kFinChunk : 1);
  return launch_status(launch_pdl(lmhead_finalize_kernel, fgrid, dim3(kFinThreads), 0, s, T, V,
                                  temperature, (const Partial*)part, n_vtiles, d_argmax,
                                  d_row_max, d_row_lse, d_top2_gap, q_norm));
}

// ---------------------------------------------------------------------------
// Allocation-free variant of eagle_lmhead_softmax.
//
// The per-row partial statistics live in a fixed array in the library's own
// device memory instead of a caller-provided workspace.  Every GPU that
// loads the library holds this array until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_lmhead_scratch[kNoAllocScratchBytes];

// Device address of g_lmhead_scratch, resolved once per device with that
// device current (the host-side symbol is only a stand-in, not an address).
void* noalloc_scratch(int* err) {
  static std::mutex mu;
  static void* ptr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = EAGLE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_lmhead_scratch) != cudaSuccess || !p) {
      *err = EAGLE_ERR_CUDA;
      return nullptr;
    }
    ptr[dev] = p;
  }
  return ptr[dev];
}

}  // namespace

extern "C" size_t eagle_lmhead_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" eagle_status eagle_lmhead_softmax_noalloc(eagle_dtype dtype, int T, int H, int V,
                                                     float temperature, int mode,
                                                     const void* d_h, const void* d_w,
                                                     int32_t* d_argmax, float* d_row_max,
                                                     float* d_row_lse, float* d_top2_gap,
                                                     float* d_q, int* d_status,
                                                     eagle_stream_t stream) {
  EAGLE_HOST_CHECK(T >= 0 && V >= 1, EAGLE_ERR_INVALID_ARG);
  // the partials of this call must fit the fixed scratch array
  const size_t need = eagle_lmhead_workspace_bytes(T, V);
  EAGLE_HOST_CHECK(need <= kNoAllocScratchBytes, EAGLE_ERR_WORKSPACE);
  int err = EAGLE_OK;
  void* scratch = noalloc_scratch(&err);
  if (!scratch) return (eagle_status)err;
  // nothing in the scratch needs clearing: every partial the finalize pass
  // reads is written earlier in the same call
  return eagle_lmhead_softmax(dtype, T, H, V, temperature, mode, d_h, d_w, d_argmax, d_row_max,
                              d_row_lse, d_top2_gap, d_q, scratch, kNoAllocScratchBytes, d_status,
                              stream);
}
