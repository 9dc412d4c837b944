// One decoder layer of the target model over the draft tree.
// [EAGLE] workflow paragraph and [S4000] "EAGLE的创新点" item 2 (page titles
// in include/eagle.h): the verify pass is one forward pass of the target
// model over every tree token; the tree attention (tree_attn.cu) is one of
// its steps.  The layer around it (LLaMA-shaped: RMSNorm, Q/K/V with rotary
// positions, output projection + residual, RMSNorm, SwiGLU MLP + residual)
// is built from the kernels here:
//
//   rmsnorm_kernel         y = bf16(x / sqrt(mean(x^2) + eps) * g), one CTA
//                          per row.
//   rope_table_kernel      position of every node (cache length + depth) and
//                          its rotation cos / sin per frequency, one CTA per
//                          sequence.
//   cast_bf16_kernel       fp32 -> bf16 (the attention output feeding the
//                          output projection).
//   gemm_tc_kernel         Y = A W^T on tcgen05 for A [T, K] (tree rows on
//                          TMEM lanes) and W [N, K] streamed once through a
//                          TMA ring; T > 128 runs clusters of row tiles that
//                          share each W stage by TMA multicast.  Epilogues
//                          (fp32 accumulators read from TMEM, 32 columns at a
//                          time per row):
//                            STORE     bf16 Y;
//                            ACCUM     out += Y in fp32 (the residual stream);
//                            SWIGLU    W rows are gate / up in alternating
//                                      16-row groups: bf16 silu(g) * u;
//                            QKV_ROPE  W rows are [Wq; Wk; Wv] with the rotary
//                                      pairs (j, j + D/2) of every q / k head
//                                      on adjacent rows: q, k rotated by the
//                                      node's position and stored [T, H, D],
//                                      v stored as is.
#include <math.h>

#include <algorithm>

#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc.cuh"

using namespace eagle;

namespace {

// ---------------------------------------------------------------------------
// small kernels
// ---------------------------------------------------------------------------
constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
rmsnorm_kernel(int T, int H, float eps, const float* __restrict__ x,
               const __nv_bfloat16* __restrict__ g, __nv_bfloat16* __restrict__ y, int* status) {
  pdl_begin();
  __shared__ float s_part[kNormThreads / 32];
  const int t = blockIdx.x;
  const float* xr = x + (size_t)t * H;
  float ss = 0.f;
  bool bad = false;
  for (int i = threadIdx.x; i < H; i += kNormThreads) {
    const float v = xr[i];
    bad |= !isfinite(v);
    ss = fmaf(v, v, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
  if (__syncthreads_or(bad) && threadIdx.x == 0) fail(status, EAGLE_ERR_NUMERIC);
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += s_part[w];
  const float inv = 1.f / sqrtf(tot / (float)H + eps);
  __nv_bfloat16* yr = y + (size_t)t * H;
  for (int i = threadIdx.x; i < H; i += kNormThreads)
    yr[i] = __float2bfloat16_rn(xr[i] * inv * __bfloat162float(g[i]));
}

__global__ void __launch_bounds__(256)
cast_bf16_kernel(size_t n, const float* __restrict__ x, __nv_bfloat16* __restrict__ y) {
  pdl_begin();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t k = i; k < n; k += stride) y[k] = __float2bfloat16_rn(x[k]);
}

// Positions (cache length + depth) and the rotation of every (node, pair j)
// by pos * theta^(-2j/D).  One thread per (node, pair) over the whole grid:
// the node's sequence by binary search of tree_off, its depth by walking
// parent[] (a parent precedes its child, so the walk ends; a parent that
// does not is reported), the angle formed in fp64 and reduced modulo 2 pi in
// fp64 (2 pi as a head and tail pair), then sine and cosine in fp32 on the
// reduced angle (|r| <= pi).
constexpr int kRopeThreads = 256;
__global__ void __launch_bounds__(kRopeThreads)
rope_table_kernel(int B, int T, int D, double log2_theta, const int* __restrict__ tree_off,
                  const int* __restrict__ parent, const int* __restrict__ kv_off,
                  const int* __restrict__ kv_len, int* __restrict__ pos,
                  float2* __restrict__ cs, int* status) {
  pdl_begin();
  const int half = D / 2;
  const long long e = (long long)blockIdx.x * kRopeThreads + threadIdx.x;
  if (e >= (long long)T * half) return;
  const int t = (int)(e / half), j = (int)(e % half);
  int lo = 0, hi = B;   // tree_off[lo] <= t < tree_off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tree_off[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int b = lo, t0 = tree_off[b], n = tree_off[b + 1] - t0;
  const int L = kv_off ? kv_off[b + 1] - kv_off[b] : kv_len[b];
  int d = 0;
  bool bad = (L < 0 || n < 1);
  for (int a = t - t0; a > 0 && !bad; ++d) {
    const int p = parent[t0 + a];
    bad = (p < 0 || p >= a);
    a = p;
  }
  if (t - t0 == 0 && parent[t0] != -1) bad = true;
  if (bad) {
    if (j == 0) fail(status, EAGLE_ERR_INVALID_TREE);
    return;
  }
  const int ps = L + d;
  if (j == 0) pos[t] = ps;
  const double ang = (double)ps * exp2(-2.0 * (double)j / (double)D * log2_theta);
  const double two_pi_hi = 6.283185307179586;              // 2 pi rounded to fp64
  const double two_pi_lo = 2.4492935982947064e-16;         // 2 pi - two_pi_hi
  const double k = rint(ang / two_pi_hi);
  const double r = fma(-k, two_pi_lo, fma(-k, two_pi_hi, ang));
  float sn, cn;
  sincosf((float)r, &sn, &cn);
  cs[(size_t)t * half + j] = make_float2(cn, sn);
}

// ---------------------------------------------------------------------------
// tcgen05 GEMM with layer epilogues
// ---------------------------------------------------------------------------
constexpr int kGThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr int kGEpiWarps = 8;    // two per TMEM lane quarter, one per column half
constexpr int kGBK = 64;         // bf16 per 128-byte swizzled row (one K chunk)
constexpr int kGUnit = 32;       // W rows per TMA box (and per epilogue chunk)
constexpr int kGBlk = 256;       // W rows per MMA (its N), at most; TMEM accumulator stride
constexpr int kGTile = 128;      // tree rows per CTA (the MMA's M)
constexpr int kGMaxCluster = 8;
// The A (tree rows) and W rings advance together, one K chunk per stage, so
// the bytes in flight are (A chunk + W chunk) x the stages of the shorter
// ring.  A narrow W slice (few W rows per CTA) makes its A chunk the larger
// one: the stages are then many and small.
constexpr int kGMaxHStages = 24;
constexpr int kGMaxWStages = 48;
// A GEMM with few W rows for the GPU (one row tile, fewer 256-row blocks
// than half the SMs) splits K over a cluster of up to this many CTAs per
// block; their fp32 partial blocks are summed in rank order through
// distributed shared memory before the epilogue.
constexpr int kGMaxSplit = 8;
// ... with every CTA keeping at least this many K chunks, and all clusters
// resident at once (a second wave of clusters cost more than the split
// gains: 65 rows x K = 4096 in 16 clusters of 8 with 15 resident took 56 us
// against 37 us unsplit, 29 us in 16 clusters of 4); a build-time option
#ifndef EAGLE_GEMM_MIN_SPLIT_CHUNKS
#define EAGLE_GEMM_MIN_SPLIT_CHUNKS 8
#endif
constexpr int kGMinSplitChunks = EAGLE_GEMM_MIN_SPLIT_CHUNKS;
constexpr int kPartStride = kGBlk + 4;   // floats per partial row (bank spread)
enum { CL_NONE = 0, CL_ROWS = 1, CL_SPLITK = 2 };
constexpr size_t kGSmemLimit = 227 * 1024;
constexpr size_t kGShared = 2048;

enum Epi { EPI_STORE = 0, EPI_ACCUM = 1, EPI_SWIGLU = 2, EPI_QKV_ROPE = 3 };

struct GemmShared {
  uint64_t h_full[kGMaxHStages], h_empty[kGMaxHStages];
  uint64_t w_full[kGMaxWStages], w_empty[kGMaxWStages];
  uint64_t tmem_full[2], tmem_empty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(GemmShared) <= kGShared, "GemmShared must fit its slot");

struct GemmArgs {
  int T, N, K, C;           // rows, W rows, reduction length, CTAs per cluster
  int n_units, w_stages, h_stages, h_stage_bytes;
  int blk_max;              // W rows per block (and per W stage), a multiple of 32, <= 256
  int ks;                   // split-K: CTAs of a cluster sharing one block (else 1)
  int epi;
  // outputs of the epilogues
  __nv_bfloat16* y;         // STORE [T, N]; SWIGLU [T, N/2]
  float* acc_out;           // ACCUM [T, N]: acc_out = (resid or acc_out) + Y
  const float* resid;
  __nv_bfloat16* q;         // QKV_ROPE: q [T, Hq, D], k [T, Hkv, D], v [T, Hkv, D]
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  const float2* cs;         // [T, D/2] rotation cos / sin per node
  int Hq, Hkv, D;
  int* status;
};

__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 16 bf16 values (two 16-byte stores) from fp32 v[0..15] to dst (16-byte
// aligned).
__device__ __forceinline__ void store16_bf16(__nv_bfloat16* dst, const float* v) {
  uint4 a, b;
  a.x = pack2_bf16(v[0], v[1]);
  a.y = pack2_bf16(v[2], v[3]);
  a.z = pack2_bf16(v[4], v[5]);
  a.w = pack2_bf16(v[6], v[7]);
  b.x = pack2_bf16(v[8], v[9]);
  b.y = pack2_bf16(v[10], v[11]);
  b.z = pack2_bf16(v[12], v[13]);
  b.w = pack2_bf16(v[14], v[15]);
  reinterpret_cast<uint4*>(dst)[0] = a;
  reinterpret_cast<uint4*>(dst)[1] = b;
}

// Epilogue of one 32-column chunk (W rows n0 .. n0+31) of row t.
__device__ __forceinline__ void gemm_epilogue(const GemmArgs& A, int t, int n0, float (&v)[32]) {
  switch (A.epi) {
    case EPI_STORE: {
      __nv_bfloat16* dst = A.y + (size_t)t * A.N + n0;
      store16_bf16(dst, v);
      store16_bf16(dst + 16, v + 16);
      break;
    }
    case EPI_ACCUM: {
      float4* dst = reinterpret_cast<float4*>(A.acc_out + (size_t)t * A.N + n0);
      const float4* src =
          A.resid ? reinterpret_cast<const float4*>(A.resid + (size_t)t * A.N + n0) : dst;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float4 r = src[i];
        r.x += v[4 * i];
        r.y += v[4 * i + 1];
        r.z += v[4 * i + 2];
        r.w += v[4 * i + 3];
        dst[i] = r;
      }
      break;
    }
    case EPI_SWIGLU: {
      // rows n0 .. n0+15 are gate rows of outputs n0/2 .. n0/2+15, rows
      // n0+16 .. n0+31 the matching up rows
      float m[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float gt = v[i];
        m[i] = gt / (1.f + expf(-gt)) * v[16 + i];
      }
      store16_bf16(A.y + (size_t)t * (A.N / 2) + n0 / 2, m);
      break;
    }
    default: {   // EPI_QKV_ROPE
      const int D = A.D, half = D / 2;
      const int qcols = A.Hq * D, kcols = A.Hkv * D;
      if (n0 >= qcols + kcols) {
        __nv_bfloat16* dst = A.v + (size_t)t * kcols + (n0 - qcols - kcols);
        store16_bf16(dst, v);
        store16_bf16(dst + 16, v + 16);
        break;
      }
      const bool is_q = n0 < qcols;
      const int c = is_q ? n0 : n0 - qcols;
      const int head = c / D, j0 = (c % D) / 2;   // pairs j0 .. j0+15 of the head
      const float2* cst = A.cs + (size_t)t * half + j0;
      float lo[16], hi[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float2 r = cst[m];
        const float x1 = v[2 * m], x2 = v[2 * m + 1];
        lo[m] = fmaf(x1, r.x, -x2 * r.y);
        hi[m] = fmaf(x1, r.y, x2 * r.x);
      }
      __nv_bfloat16* dst =
          (is_q ? A.q + ((size_t)t * A.Hq + head) * D : A.k + ((size_t)t * A.Hkv + head) * D);
      store16_bf16(dst + j0, lo);
      store16_bf16(dst + half + j0, hi);
      break;
    }
  }
}

// CL_ROWS: the row tiles of a cluster share every W stage by multicast.
// CL_SPLITK: the CTAs of a cluster take consecutive K ranges of one block.
template <int CL>
__global__ void __launch_bounds__(kGThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w,
               const GemmArgs A) {
  constexpr bool MULTI = (CL == CL_ROWS);
  constexpr bool SPLITK = (CL == CL_SPLITK);
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* h_smem = base;
  const int h_stages = A.h_stages;
  unsigned char* w_smem = base + h_stages * A.h_stage_bytes;
  const int blk_max = A.blk_max;
  const int w_stage_bytes = blk_max * 128;
  const int w_stages = A.w_stages;
  GemmShared* sh = reinterpret_cast<GemmShared*>(w_smem + (size_t)w_stages * w_stage_bytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = MULTI ? A.C : 1;
  const int KS = SPLITK ? A.ks : 1;
  const int rank = MULTI ? (int)tc::cluster_ctarank() : 0;    // this CTA's row tile
  const int krank = SPLITK ? (int)tc::cluster_ctarank() : 0;  // this CTA's K range
  const uint16_t all_ctas = (uint16_t)((1u << C) - 1u);
  const int slices = gridDim.x / (C * KS);
  const int slice = blockIdx.x / (C * KS);
  const int u0 = (int)((long long)A.n_units * slice / slices);
  const int u1 = (int)((long long)A.n_units * (slice + 1) / slices);
  const int r_begin = u0 * kGUnit, r_end = u1 * kGUnit;
  const int n_blocks = (r_end - r_begin + blk_max - 1) / blk_max;
  // K chunks kb0 .. kb0 + KB - 1 (split-K: this CTA's share)
  const int KB_all = (A.K + kGBK - 1) / kGBK;
  const int kb0 = (int)((long long)KB_all * krank / KS);
  const int KB = (int)((long long)KB_all * (krank + 1) / KS) - kb0;
  const int total = n_blocks * KB;
  int* status = A.status;
  auto blk_rows = [&](int blk) { return min(blk_max, r_end - (r_begin + blk * blk_max)); };
  auto load_w = [&](int stage, int rows, int kb, int y0, uint64_t pol) {
    tc::mbar_arrive_expect_tx(&sh->w_full[stage], (uint32_t)(rows * 128));
    unsigned char* dst = w_smem + (size_t)stage * w_stage_bytes;
    for (int u = rank * kGUnit; u < rows; u += C * kGUnit) {
      if (MULTI)
        tc::tma_load_2d_mc_hint(dst + u * 128, &map_w, &sh->w_full[stage], (kb0 + kb) * kGBK,
                                y0 + u, all_ctas, pol);
      else
        tc::tma_load_2d_hint(dst + u * 128, &map_w, &sh->w_full[stage], (kb0 + kb) * kGBK,
                             y0 + u, pol);
    }
  };
  const int w_early = min(w_stages, total);

  if (threadIdx.x == 0) {
    for (int i = 0; i < h_stages; ++i) {
      tc::mbar_init(&sh->h_full[i], 1);
      tc::mbar_init(&sh->h_empty[i], 1);
    }
    for (int i = 0; i < w_stages; ++i) {
      tc::mbar_init(&sh->w_full[i], 1);
      tc::mbar_init(&sh->w_empty[i], C);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sh->tmem_full[i], 1);
      tc::mbar_init(&sh->tmem_empty[i], kGEpiWarps);
    }
    tc::mbar_init(&sh->drain, 1);
    sh->abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (MULTI) tc::cluster_sync_all();
  if (threadIdx.x == 0) {
    tc::prefetch_tensormap(&map_a);
    tc::prefetch_tensormap(&map_w);
    // weights never depend on an earlier kernel: the first stages go out
    // before the dependency wait
    const uint64_t pol_w = tc::policy_evict_first();
    for (int i = 0; i < w_early; ++i) {
      const int blk = i / KB;
      load_w(i, blk_rows(blk), i - blk * KB, r_begin + blk * blk_max, pol_w);
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(&sh->tmem_base, 512);
    tc::tmem_relinquish();
  }
  pdl_begin();   // A and the outputs follow the previous kernel
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int* abort_flag = &sh->abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = tc::policy_evict_first();
      const uint64_t pol_h = tc::policy_evict_last();
      int hs = 0, ws = 0, issued_h = 0, issued_w = w_early;
      uint32_t hph = 0, wph = 0;
      bool ok = true;
      int i = 0;
      for (int blk = 0; blk < n_blocks && ok; ++blk) {
        const int rows = blk_rows(blk);
        const int y0 = r_begin + blk * blk_max;
        for (int kb = 0; kb < KB && ok; ++kb, ++i) {
          if (!(ok = tc::mbar_wait(&sh->h_empty[hs], hph ^ 1, abort_flag, status))) break;
          tc::mbar_arrive_expect_tx(&sh->h_full[hs], (uint32_t)A.h_stage_bytes);
          tc::tma_load_2d_hint(h_smem + hs * A.h_stage_bytes, &map_a, &sh->h_full[hs],
                               (kb0 + kb) * kGBK, rank * kGTile, pol_h);
          ++issued_h;
          if (++hs == h_stages) { hs = 0; hph ^= 1; }
          if (i >= w_early) {
            if (!(ok = tc::mbar_wait(&sh->w_empty[ws], wph ^ 1, abort_flag, status))) break;
            load_w(ws, rows, kb, y0, pol_w);
            ++issued_w;
          }
          if (++ws == w_stages) { ws = 0; wph ^= 1; }
        }
      }
      if (ok && MULTI) {
        for (int j = max(0, total - w_stages); j < total && ok; ++j)
          ok = tc::mbar_wait(&sh->w_empty[j % w_stages], (j / w_stages) & 1, abort_flag, status);
      }
      if (!ok) {
        int never = 0;
        // (the last copy issued into each slot: waiting for its phase
        // returns at once if it has landed, whether consumed or not)
        for (int j = max(0, issued_w - w_stages); j < issued_w; ++j)
          tc::mbar_wait(&sh->w_full[j % w_stages], (j / w_stages) & 1, &never, nullptr,
                        200000000ll);
        for (int j = max(0, issued_h - h_stages); j < issued_h; ++j)
          tc::mbar_wait(&sh->h_full[j % h_stages], (j / h_stages) & 1, &never, nullptr,
                        200000000ll);
      }
    }
  } else if (warp == 1) {
    // A K chunk's stages are released (its MMAs committed) right after its
    // MMAs are issued; the next chunk's waits follow.
    if (lane == 0) {
      int hs = 0, ws = 0;
      uint32_t hph = 0, wph = 0, tph = 0;
      bool ok = true;
      auto wait_chunk = [&](int& h_at, int& w_at) -> bool {
        h_at = hs;
        w_at = ws;
        if (!tc::mbar_wait(&sh->h_full[hs], hph, abort_flag, status)) return false;
        if (!tc::mbar_wait(&sh->w_full[ws], wph, abort_flag, status)) return false;
        if (++hs == h_stages) { hs = 0; hph ^= 1; }
        if (++ws == w_stages) { ws = 0; wph ^= 1; }
        return true;
      };
      for (int blk = 0; blk < n_blocks && ok; ++blk) {
        const int ab = blk & 1;
        if (!(ok = tc::mbar_wait(&sh->tmem_empty[ab], ((tph >> ab) & 1u) ^ 1u, abort_flag,
                                 status)))
          break;
        tph ^= 1u << ab;
        const uint32_t idesc = tc::idesc_bf16_f32(128, blk_rows(blk));
        const uint32_t d = tmem + (uint32_t)(ab * kGBlk);
        int h_at, w_at;
        if (!(ok = wait_chunk(h_at, w_at))) break;
        for (int kb = 0; kb < KB; ++kb) {
          tc::fence_after_thread_sync();
          const uint64_t da = tc::desc_kmajor_sw128(tc::smem_u32(h_smem + h_at * A.h_stage_bytes));
          const uint64_t db = tc::desc_kmajor_sw128(tc::smem_u32(w_smem + (size_t)w_at * w_stage_bytes));
          // K steps of 16 advance the descriptors' start address by 32 bytes
          tc::mma_f16(d, da, db, idesc, kb > 0 ? 1u : 0u);
          tc::mma_f16(d, da + 2, db + 2, idesc, 1u);
          tc::mma_f16(d, da + 4, db + 4, idesc, 1u);
          tc::mma_f16(d, da + 6, db + 6, idesc, 1u);
          if (MULTI)
            tc::mma_commit_mc(&sh->w_empty[w_at], all_ctas);
          else
            tc::mma_commit(&sh->w_empty[w_at]);
          tc::mma_commit(&sh->h_empty[h_at]);
          if (kb + 1 < KB && !(ok = wait_chunk(h_at, w_at))) break;
        }
        if (ok) tc::mma_commit(&sh->tmem_full[ab]);
      }
      tc::mma_commit(&sh->drain);
      int never = 0;
      tc::mbar_wait(&sh->drain, 0, &never, nullptr, 200000000ll);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int chalf = (warp - 2) >> 2;
    const int t = rank * kGTile + quad * 32 + lane;   // tree row of this thread
    const bool row_ok = t < A.T;
    const bool quad_live = rank * kGTile + quad * 32 < A.T;
    uint32_t tph = 0;
    for (int blk = 0; blk < n_blocks; ++blk) {
      const int ab = blk & 1;
      const int rows = blk_rows(blk);
      const bool got = tc::mbar_wait(&sh->tmem_full[ab], (tph >> ab) & 1u, abort_flag, status);
      if (!__all_sync(0xffffffffu, got)) break;
      tph ^= 1u << ab;
      tc::fence_after_thread_sync();
      // two warps per lane quarter split a block's columns at a multiple of 32
      const int half_cols = ((blk_max / 2 + kGUnit - 1) / kGUnit) * kGUnit;
      for (int c = chalf * half_cols; c < (chalf + 1) * half_cols && c < rows && quad_live;
           c += kGUnit) {
        float v[32];
        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(quad * 32) << 16) +
                                   (uint32_t)(ab * kGBlk + c), v);
        if (SPLITK) {
          // this K range's partial of (row, c .. c+31) into the (idle) rings
          if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) +
                                                    (size_t)t * kPartStride + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        } else if (row_ok) {
          gemm_epilogue(A, t, r_begin + blk * blk_max + c, v);
        }
      }
      tc::fence_before_thread_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->tmem_empty[ab]);
    }
  }
  if (SPLITK) {
    // every CTA's partial is in its shared memory: sum the K ranges in rank
    // order, CTA krank taking every KS-th (row, 32-column) piece, then the
    // epilogue on the sum
    tc::cluster_sync_all();
    cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
    const int rows = blk_rows(0);
    const int ppr = rows / kGUnit;                 // pieces per row
    const int pieces = A.T * ppr;
    const int mine_n = (pieces > krank) ? (pieces - krank + KS - 1) / KS : 0;   // this CTA's
    auto piece_at = [&](int m) {                   // m-th piece of this CTA: its partial here
      const int j = krank + KS * m;
      return reinterpret_cast<float*>(base) + (size_t)(j / ppr) * kPartStride + (j % ppr) * kGUnit;
    };
    // every thread sums 4-column slices of this CTA's pieces over the K
    // ranges (the ranks' loads in flight together, added in rank order) into
    // this CTA's own partial, which no other CTA reads ...
    for (int it = threadIdx.x; it < mine_n * (kGUnit / 4); it += blockDim.x) {
      float* slot = piece_at(it / (kGUnit / 4)) + (it % (kGUnit / 4)) * 4;
      float4 x[kGMaxSplit];
#pragma unroll
      for (int r = 0; r < kGMaxSplit; ++r)
        if (r < KS) x[r] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(slot, r));
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < kGMaxSplit; ++r)
        if (r < KS) {
          sum.x += x[r].x;
          sum.y += x[r].y;
          sum.z += x[r].z;
          sum.w += x[r].w;
        }
      *reinterpret_cast<float4*>(slot) = sum;
    }
    __syncthreads();
    // ... then one thread per piece runs the epilogue from it
    for (int m = threadIdx.x; m < mine_n; m += blockDim.x) {
      const int j = krank + KS * m;
      const float4* src = reinterpret_cast<const float4*>(piece_at(m));
      float v[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 x = src[i];
        v[4 * i] = x.x;
        v[4 * i + 1] = x.y;
        v[4 * i + 2] = x.z;
        v[4 * i + 3] = x.w;
      }
      gemm_epilogue(A, j / ppr, r_begin + (j % ppr) * kGUnit, v);
    }
    // no CTA leaves while a peer may still read its shared memory
    tc::cluster_sync_all();
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, 512);
  }
  if (MULTI) tc::cluster_sync_all();
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode() {
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

// 2-D bf16 [rows, cols] -> 128-byte swizzled boxes of 64 columns x box_rows.
bool g_map(CUtensorMap* map, const void* ptr, int rows, int cols, int box_rows) {
  auto enc = g_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kGBK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_sm_count() {
  static int n[kMaxDevices] = {};
  const int dev = current_device_slot();
  if (!n[dev]) {
    int c = 0, d = 0;
    cudaGetDevice(&d);
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || c <= 0)
      c = 148;
    n[dev] = c;
  }
  return n[dev];
}

struct GLayout {
  int h_stage_bytes, h_stages, w_stages, blk;
  size_t smem;
};

// `blk`: W rows per block (a multiple of 32).  Both rings get as many
// stages as fit side by side (each K chunk needs its A and its W stage);
// bytes left over go to extra W stages, which are requested before the
// kernel waits for its predecessor.
GLayout g_layout(int h_rows, int blk) {
  GLayout L;
  L.h_stage_bytes = h_rows * 128;
  L.blk = blk;
  const size_t wb = (size_t)blk * 128;
  const size_t room = kGSmemLimit - 1024 - kGShared;
  L.h_stages = (int)std::min<size_t>(kGMaxHStages, room / (L.h_stage_bytes + wb));
  const size_t left = room - (size_t)L.h_stages * L.h_stage_bytes;
  L.w_stages = (int)std::min<size_t>(kGMaxWStages, left / wb);
  L.smem = 1024 + kGShared + (size_t)L.h_stages * L.h_stage_bytes + (size_t)L.w_stages * wb;
  return L;
}

// Clusters of C CTAs of the given kind resident at once (0: none), per
// device, cluster size and shared-memory size.
template <int CL>
int g_max_clusters(int C, size_t smem) {
  static std::mutex mu;
  static int cached[kMaxDevices][kGMaxCluster + 1] = {};
  static size_t cached_smem[kMaxDevices][kGMaxCluster + 1] = {};
  std::lock_guard<std::mutex> lock(mu);
  const int dev = current_device_slot();
  if (cached_smem[dev][C] != smem) {
    cached[dev][C] = 0;
    cached_smem[dev][C] = smem;
  }
  if (!cached[dev][C]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(C * 64));
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)gemm_tc_kernel<CL>, &cfg) !=
        cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cached[dev][C] = n > 0 ? n : -1;
  }
  return std::max(cached[dev][C], 0);
}

eagle_status gemm_launch(int T, int N, int K, const void* d_a, const void* d_w, GemmArgs A,
                         cudaStream_t s) {
  static PerDeviceOnce attr_once;
  if (attr_once.run([] {
        cudaError_t e = cudaSuccess;
        for (auto k : {gemm_tc_kernel<CL_NONE>, gemm_tc_kernel<CL_ROWS>, gemm_tc_kernel<CL_SPLITK>})
          if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kGSmemLimit);
        return e;
      }) != cudaSuccess)
    return EAGLE_ERR_CUDA;
  CUtensorMap map_w;
  if (!g_map(&map_w, d_w, N, K, kGUnit)) return EAGLE_ERR_CUDA;
  const int n_units = N / kGUnit;
  const int tiles = (T + kGTile - 1) / kGTile;
  const int KB_all = (K + kGBK - 1) / kGBK;
  // one row tile and few 256-row blocks: split K over clusters instead
  const int n_blk = (N + kGBlk - 1) / kGBlk;
  int ks = (tiles == 1 && 2 * n_blk <= g_sm_count())
               ? std::min({kGMaxSplit, g_sm_count() / n_blk, KB_all / kGMinSplitChunks})
               : 1;
  const GLayout LS = g_layout(((T + 7) / 8) * 8, kGBlk);
  while (ks >= 2 && g_max_clusters<CL_SPLITK>(ks, LS.smem) < n_blk) --ks;
  if (ks >= 2) {
    const GLayout& L = LS;
    CUtensorMap map_a;
    if (!g_map(&map_a, d_a, T, K, L.h_stage_bytes / 128)) return EAGLE_ERR_CUDA;
    GemmArgs P = A;
    P.T = T;
    P.N = N;
    P.K = K;
    P.C = 1;
    P.ks = ks;
    P.n_units = n_units;
    P.w_stages = L.w_stages;
    P.h_stages = L.h_stages;
    P.h_stage_bytes = L.h_stage_bytes;
    P.blk_max = L.blk;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_blk * ks));
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)ks;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<CL_SPLITK>, map_a, map_w, P) == cudaSuccess
               ? EAGLE_OK
               : EAGLE_ERR_CUDA;
  }
  const GLayout TL = g_layout(kGTile, kGBlk);
  int passes = 1, C = tiles;
  while (C > 1 && (C > kGMaxCluster || g_max_clusters<CL_ROWS>(C, TL.smem) < 1)) {
    ++passes;
    C = (tiles + passes - 1) / passes;
  }
  const int slices = (C > 1) ? std::min(g_max_clusters<CL_ROWS>(C, TL.smem), n_units)
                             : std::min(g_sm_count(), n_units);
  for (int p = 0, tile0 = 0; p < passes; ++p) {
    const int nt = std::min(C, tiles - tile0);
    const int r0 = tile0 * kGTile;
    const int Ts = std::min(nt * kGTile, T - r0);
    tile0 += nt;
    const int Cp = (C > 1) ? nt : 1;
    const int slice_units = (n_units + slices - 1) / slices;
    const GLayout L = g_layout((Cp > 1 || Ts > kGTile) ? kGTile : ((Ts + 7) / 8) * 8,
                               std::min(kGBlk, slice_units * kGUnit));
    CUtensorMap map_a;
    const __nv_bfloat16* ap = static_cast<const __nv_bfloat16*>(d_a) + (size_t)r0 * K;
    if (!g_map(&map_a, ap, Ts, K, L.h_stage_bytes / 128)) return EAGLE_ERR_CUDA;
    GemmArgs P = A;
    P.T = Ts;
    P.N = N;
    P.K = K;
    P.C = Cp;
    P.ks = 1;
    P.n_units = n_units;
    P.w_stages = L.w_stages;
    P.h_stages = L.h_stages;
    P.h_stage_bytes = L.h_stage_bytes;
    P.blk_max = L.blk;
    // the pass's rows: shift every row-indexed output
    if (P.y) P.y += (size_t)r0 * (A.epi == EPI_SWIGLU ? N / 2 : N);
    if (P.acc_out) P.acc_out += (size_t)r0 * N;
    if (P.resid) P.resid += (size_t)r0 * N;
    if (P.q) P.q += (size_t)r0 * A.Hq * A.D;
    if (P.k) P.k += (size_t)r0 * A.Hkv * A.D;
    if (P.v) P.v += (size_t)r0 * A.Hkv * A.D;
    if (P.cs) P.cs += (size_t)r0 * (A.D / 2);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(slices * Cp));
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)Cp;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (Cp > 1) ? 2 : 1;
    const cudaError_t e =
        (Cp > 1) ? cudaLaunchKernelEx(&cfg, gemm_tc_kernel<CL_ROWS>, map_a, map_w, P)
                 : cudaLaunchKernelEx(&cfg, gemm_tc_kernel<CL_NONE>, map_a, map_w, P);
    if (e != cudaSuccess) return EAGLE_ERR_CUDA;
  }
  return EAGLE_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace

extern "C" eagle_status eagle_rmsnorm(int T, int H, float eps, const float* d_x,
                                      const void* d_gain, void* d_y, int* d_status,
                                      eagle_stream_t stream) {
  EAGLE_HOST_CHECK(T >= 0 && H >= 1 && eps >= 0.f && isfinite(eps), EAGLE_ERR_INVALID_ARG);
  if (T == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_x && d_gain && d_y && d_status, EAGLE_ERR_INVALID_ARG);
  return launch_status(launch_pdl(rmsnorm_kernel, dim3(T), dim3(kNormThreads), 0,
                                  (cudaStream_t)stream, T, H, eps, d_x,
                                  static_cast<const __nv_bfloat16*>(d_gain),
                                  static_cast<__nv_bfloat16*>(d_y), d_status));
}

extern "C" eagle_status eagle_cast_bf16(size_t n, const float* d_x, void* d_y,
                                        eagle_stream_t stream) {
  if (n == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_x && d_y, EAGLE_ERR_INVALID_ARG);
  const int grid = (int)std::min<size_t>((n + 255) / 256, 4096);
  return launch_status(launch_pdl(cast_bf16_kernel, dim3(grid), dim3(256), 0,
                                  (cudaStream_t)stream, n, d_x,
                                  static_cast<__nv_bfloat16*>(d_y)));
}

extern "C" eagle_status eagle_tree_rope_table(int B, int T, int D, float theta,
                                              const int32_t* d_tree_off,
                                              const int32_t* d_parent, const int32_t* d_kv_off,
                                              const int32_t* d_kv_len, int32_t* d_pos,
                                              float* d_cos_sin, int* d_status,
                                              eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 0 && D >= 2 && D % 2 == 0 && theta > 1.f && isfinite(theta),
                   EAGLE_ERR_INVALID_ARG);
  if (B == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_tree_off && d_parent && d_pos && d_cos_sin && d_status,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK((d_kv_off != nullptr) != (d_kv_len != nullptr), EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(T >= 0, EAGLE_ERR_INVALID_ARG);
  if (T == 0) return EAGLE_OK;
  const long long work = (long long)T * (D / 2);
  return launch_status(launch_pdl(rope_table_kernel,
                                  dim3((unsigned)((work + kRopeThreads - 1) / kRopeThreads)),
                                  dim3(kRopeThreads), 0, (cudaStream_t)stream, B, T, D,
                                  log2((double)theta), d_tree_off, d_parent, d_kv_off, d_kv_len,
                                  d_pos, reinterpret_cast<float2*>(d_cos_sin), d_status));
}

extern "C" eagle_status eagle_gemm(int epilogue, int T, int N, int K, const void* d_a,
                                   const void* d_w, void* d_y, float* d_accum,
                                   const float* d_resid, void* d_q,
                                   void* d_k, void* d_v, const float* d_cos_sin, int Hq, int Hkv,
                                   int D, int* d_status, eagle_stream_t stream) {
  EAGLE_HOST_CHECK(T >= 0 && N >= 1 && K >= 1, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(epilogue >= EAGLE_EPI_STORE && epilogue <= EAGLE_EPI_QKV_ROPE,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(N % kGUnit == 0 && K % 8 == 0, EAGLE_ERR_UNSUPPORTED);
  if (T == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_a && d_w && d_status && aligned16(d_a) && aligned16(d_w),
                   EAGLE_ERR_INVALID_ARG);
  GemmArgs A = {};
  A.epi = epilogue;
  A.status = d_status;
  switch (epilogue) {
    case EAGLE_EPI_STORE:
    case EAGLE_EPI_SWIGLU:
      EAGLE_HOST_CHECK(d_y && aligned16(d_y), EAGLE_ERR_INVALID_ARG);
      A.y = static_cast<__nv_bfloat16*>(d_y);
      break;
    case EAGLE_EPI_ACCUM:
      EAGLE_HOST_CHECK(d_accum && aligned16(d_accum) && (!d_resid || aligned16(d_resid)),
                       EAGLE_ERR_INVALID_ARG);
      A.acc_out = d_accum;
      A.resid = d_resid;
      break;
    default:
      EAGLE_HOST_CHECK(Hq >= 1 && Hkv >= 1 && D >= 32 && D % 32 == 0, EAGLE_ERR_UNSUPPORTED);
      EAGLE_HOST_CHECK(N == (Hq + 2 * Hkv) * D, EAGLE_ERR_INVALID_ARG);
      EAGLE_HOST_CHECK(d_q && d_k && d_v && d_cos_sin && aligned16(d_q) && aligned16(d_k) &&
                           aligned16(d_v),
                       EAGLE_ERR_INVALID_ARG);
      A.q = static_cast<__nv_bfloat16*>(d_q);
      A.k = static_cast<__nv_bfloat16*>(d_k);
      A.v = static_cast<__nv_bfloat16*>(d_v);
      A.cs = reinterpret_cast<const float2*>(d_cos_sin);
      A.Hq = Hq;
      A.Hkv = Hkv;
      A.D = D;
      break;
  }
  return gemm_launch(T, N, K, d_a, d_w, A, (cudaStream_t)stream);
}
