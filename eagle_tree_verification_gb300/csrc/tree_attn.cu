// Tree attention of the tree-verify step.
// [S4000] "EAGLE的创新点" item 2 and [EAGLE] workflow paragraph (page titles
// in include/eagle.h): one forward pass verifies every path of the draft
// tree, because node i attends to the cached context and to exactly its own
// ancestors and itself.
//
// Two kernels:
//   tree_attn_tc_kernel    bf16, head dim 128: one CTA per (sequence, kv head,
//                          128-row tile of (node, query head) rows, cache
//                          chunk).  TMA brings Q (once) and 128-key K/V blocks
//                          (two-stage ring) into 128-byte-swizzled shared
//                          memory; tcgen05.mma computes S = Q K^T into TMEM;
//                          two threads per query row (one per key half)
//                          apply the mask (cache bound, or the row's
//                          ancestor bitset built on chip from parent[]) and
//                          the online softmax, write P (bf16 hi + lo) into
//                          TMEM, and tcgen05.mma adds P V into the half's
//                          fp32 accumulator in TMEM (rescaled only when the
//                          running max grows by more than a set margin).
//                          The cache chunks of one (sequence, head, tile)
//                          form a thread-block cluster and merge their
//                          partial rows through distributed shared memory.
//   tree_attn_warp_kernel  CUDA-core kernel for fp32 inputs and other shapes:
//                          one warp per (node, query head).
// The ancestor mask is never stored: it is derived from parent[] on the fly.
#include <math.h>

#include <algorithm>

#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc.cuh"

using namespace eagle;
namespace cg = cooperative_groups;

namespace {

constexpr int kWarpsPerBlock = 4;

// Where the cache keys of a sequence live: contiguous rows kv_off[b] ..
// kv_off[b+1]-1, or (page_size > 0) pages of a pool named by a block table,
// with the sequence's length in kv_len[b].
struct CacheIndex {
  const int* kv_off;
  const int* kv_len;
  const int* block_table;
  int page_size, max_pages, n_pages;
};

template <typename TIn, int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
tree_attn_warp_kernel(int B, int T, int Hq, int Hkv, float scale, int max_nodes, int max_kv,
                      const TIn* __restrict__ q, const TIn* __restrict__ k_tree,
                      const TIn* __restrict__ v_tree, const TIn* __restrict__ k_cache,
                      const TIn* __restrict__ v_cache, const CacheIndex ci,
                      const int* __restrict__ tree_off, const int* __restrict__ parent,
                      float* __restrict__ out, int* status) {
  pdl_begin();
  constexpr int PER = D / 32;
  const int warp = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= T * Hq) return;
  const int t = warp / Hq, h = warp % Hq;
  const int g = h / (Hq / Hkv);
  // sequence of node t: last b with tree_off[b] <= t
  int lo = 0, hi = B;  // tree_off[lo] <= t < tree_off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tree_off[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int b = lo;
  const int t0 = tree_off[b], n = tree_off[b + 1] - t0;
  const bool paged = ci.page_size > 0;
  const int c0 = paged ? 0 : ci.kv_off[b];
  const int L = paged ? ci.kv_len[b] : ci.kv_off[b + 1] - c0;
  if (n > max_nodes || L > max_kv || L < 0) {
    if (lane == 0) fail(status, EAGLE_ERR_INVALID_TREE);
    return;
  }
  float qv[PER], acc[PER];
  const TIn* qp = q + ((size_t)t * Hq + h) * D;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    qv[e] = to_f32(qp[lane + 32 * e]) * scale;
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  auto visit = [&](const TIn* kp, const TIn* vp) {
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) s = fmaf(qv[e], to_f32(kp[lane + 32 * e]), s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mn = fmaxf(m, s);
    const float corr = expf(m - mn);
    const float p = expf(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = fmaf(p, to_f32(vp[lane + 32 * e]), acc[e] * corr);
    m = mn;
  };
  for (int j = 0; j < L; ++j) {
    int row = c0 + j;
    if (paged) {
      int page = ci.block_table[(size_t)b * ci.max_pages + j / ci.page_size];
      if (page < 0 || page >= ci.n_pages) {
        if (lane == 0) fail(status, EAGLE_ERR_INVALID_ARG);
        page = 0;
      }
      row = page * ci.page_size + j % ci.page_size;
    }
    const size_t off = ((size_t)row * Hkv + g) * D;
    visit(k_cache + off, v_cache + off);
  }
  // ancestors and the node itself, following parent[] (order is irrelevant)
  int i = t - t0;
  int steps = 0;
  while (i >= 0) {
    const size_t off = ((size_t)(t0 + i) * Hkv + g) * D;
    visit(k_tree + off, v_tree + off);
    const int p = parent[t0 + i];
    if ((i == 0 && p != -1) || (i > 0 && (p < 0 || p >= i)) || ++steps > n) {
      if (lane == 0) fail(status, EAGLE_ERR_INVALID_TREE);
      break;
    }
    i = p;
  }
  float* op = out + ((size_t)t * Hq + h) * D;
  const float inv = 1.f / l;
#pragma unroll
  for (int e = 0; e < PER; ++e) op[lane + 32 * e] = acc[e] * inv;
}

template <typename TIn>
eagle_status launch_warp(int D, int B, int T, int Hq, int Hkv, float scale, int max_nodes,
                         int max_kv, const void* q, const void* kt, const void* vt,
                         const void* kc, const void* vc, const CacheIndex& ci,
                         const int* tree_off, const int* parent, float* out, int* status,
                         cudaStream_t s) {
  const int warps = T * Hq;
  const int grid = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const TIn* Q = static_cast<const TIn*>(q);
  const TIn* KT = static_cast<const TIn*>(kt);
  const TIn* VT = static_cast<const TIn*>(vt);
  const TIn* KC = static_cast<const TIn*>(kc);
  const TIn* VC = static_cast<const TIn*>(vc);
  auto kern = (D == 64) ? tree_attn_warp_kernel<TIn, 64> : tree_attn_warp_kernel<TIn, 128>;
  return launch_status(launch_pdl(kern, dim3(grid), dim3(kWarpsPerBlock * 32), 0, s, B, T, Hq,
                                  Hkv, scale, max_nodes, max_kv, Q, KT, VT, KC, VC, ci,
                                  tree_off, parent, out, status));
}

// ---------------------------------------------------------------------------
// tcgen05 path (bf16, D = 128)
// ---------------------------------------------------------------------------
constexpr int kAttThreads = 320;        // warp 0 TMA, warp 1 MMA, warps 2-9 rows
constexpr float kRescaleLog2 = 8.f;     // rescale O only when the max grows by > 2^8
constexpr int kKeyBlk = 128;            // keys per block (the S MMA's N)
constexpr int kHalfBytes = 128 * 128;   // 128 rows x 64 bf16 (one swizzle atom wide)
constexpr int kTileBytes = 2 * kHalfBytes;  // 128 rows x 128 bf16
constexpr int kTargetCtas = 152;        // SMs of a GB300
constexpr int kMaxSplit = 8;            // cache chunks of one tile: one portable cluster
constexpr int kMaxOrder = 256;          // sequences ordered by cache length (more: as given)
constexpr size_t kAttSharedBytes = 5120;
// cluster merge inside the K/V stage memory: O rows [NC][rows per owner][32]
// float4 (at most 136 x 512 B), then (max, sum) pairs
constexpr int kMergeMlOffset = 73728;
static_assert(kMergeMlOffset >= (128 + kMaxSplit) * 512, "merge rows overlap the (max, sum) pairs");
static_assert(kMergeMlOffset + (128 + kMaxSplit) * 8 <= 4 * kTileBytes, "merge exceeds the K/V stages");
// Q, two K stages, two V stages; the merge reuses the K stages for O rows
constexpr size_t kAttSmem = 1024 + 5 * (size_t)kTileBytes + kAttSharedBytes;

struct AttShared {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full, s_empty;        // S ready / read by every row warp
  uint64_t p_full;                 // P written by every row warp
  uint64_t pv_done, o_done, drain;
  uint64_t fbar;                   // row-half exchange after the key loop
  uint32_t tmem_base;
  int abort_flag;
  float xchg[2][2][128];           // [m | l][half][row]
  float2 ml[128];                  // (m, l) of every row, read by the cluster
  int par[EAGLE_MAX_TREE_NODES];   // parent[] of the sequence
};

static_assert(sizeof(AttShared) <= kAttSharedBytes, "AttShared must fit its shared-memory slot");

struct AttPlan {
  int G, MT, NC, CK;  // heads per kv head, row tiles, cache chunks, keys per chunk
};

// `split_cap`: the largest number of cache chunks per row tile whose
// clusters all fit on the GPU at once.  (Measured at 16 ragged sequences of
// 512..16384 keys, 256 tiles: splitting the longest caches into clusters of
// four chunks took 461 us against 224 us unsplit -- clusters of 170 KB CTAs
// wait for four free SMs of one GPC -- so launches of more tiles than SMs
// stay unsplit.)
#ifndef EAGLE_ATTN_MIN_SPLIT
#define EAGLE_ATTN_MIN_SPLIT 1
#endif
AttPlan att_plan(int B, int Hq, int Hkv, int max_nodes, int max_kv, int split_cap) {
  AttPlan P;
  P.G = Hq / Hkv;
  P.MT = (max_nodes * P.G + 127) / 128;
  const int tiles = std::max(1, B * Hkv * P.MT);
  const int nc = std::max(EAGLE_ATTN_MIN_SPLIT,
                          std::min(split_cap, std::max(1, kTargetCtas / tiles)));
  int ck = (max_kv + nc - 1) / nc;
  ck = std::max(256, ((ck + kKeyBlk - 1) / kKeyBlk) * kKeyBlk);
  P.CK = ck;
  P.NC = std::max(1, (max_kv + ck - 1) / ck);
  return P;
}

struct AttParams {
  int B, Hq, Hkv, G, MT, NC, CK, max_nodes, max_kv;
  float scale_log2;
  const int* kv_off;       // contiguous cache: rows kv_off[b] .. kv_off[b+1]-1
  // paged cache (page_size > 0): sequence b's key pos lives in row
  // block_table[b * max_pages + pos / page_size] * page_size + pos % page_size
  // of the page pool; its length is kv_len[b]
  int page_size, max_pages, n_pages;
  const int* block_table;
  const int* kv_len;
  const int* tree_off;
  const int* parent;
  float* out;
  int* status;
};

// 2^x by the SFU's approximate exponential (relative error about 2^-22;
// subnormal results flush to zero, 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// MN-major (rows of 64 N-elements, one row per K index) 128-byte-swizzled
// operand: `lbo` = bytes between the two 64-wide halves along N, 8-row
// groups along K are 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t smem_addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// D[tmem] (+)= A[tmem] * B[smem]: A (M x K, K-major, two 16-bit elements per
// 32-bit column) is read from tensor memory.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// One CTA per (sequence, kv head, 128-row tile, cache chunk); the chunks of
// a tile form a thread-block cluster and merge their partial softmax rows
// through distributed shared memory.  Two threads per query row, one per
// half of every key block; each half keeps its own running max, sum and
// output accumulator, so the halves never wait for each other inside the
// key loop and are merged once at the end.  TMEM columns: S at 0 (refilled
// with the next block as soon as every row has read it), P at 128 (per key
// half: bf16 hi at +0, lo at +32), O of key half 0 at 256, of half 1 at 384.
__global__ void __launch_bounds__(kAttThreads, 1)
tree_attn_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_kc,
                    const __grid_constant__ CUtensorMap map_vc,
                    const __grid_constant__ CUtensorMap map_kt,
                    const __grid_constant__ CUtensorMap map_vt, const AttParams A) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* q_sm = base;                       // [2 halves][128 rows][128 B]
  unsigned char* k_sm = base + kTileBytes;          // 2 stages
  unsigned char* v_sm = base + 3 * kTileBytes;      // 2 stages
  AttShared* sh = reinterpret_cast<AttShared*>(base + 5 * kTileBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A contiguous KV cache and its offsets are resident state that the
  // kernel queued just before this one does not write: the first cache
  // blocks are requested before waiting for it (the tree and the queries
  // come after the wait).  A paged cache is read only after the wait (a
  // commit of accepted tokens may have just written its pages).
  const bool paged = A.page_size > 0;
  if (paged) pdl_begin();
  // work item: tile * NC + c, the cache chunks of a tile adjacent (one
  // cluster); tiles go to the sequences longest cache first (ties: lower
  // index), so the longest work starts in the first wave
  auto seq_len = [&](int u) { return paged ? A.kv_len[u] : A.kv_off[u + 1] - A.kv_off[u]; };
  __shared__ int s_seq[kMaxOrder];
  const int c = blockIdx.x % A.NC;
  const int tile = blockIdx.x / A.NC;
  const int mt = tile % A.MT;
  const int g = (tile / A.MT) % A.Hkv;
  int b = tile / (A.MT * A.Hkv);
  if (A.B <= kMaxOrder) {
    for (int t = threadIdx.x; t < A.B; t += blockDim.x) {
      const int Lt = seq_len(t);
      int rank = 0;
      for (int u = 0; u < A.B; ++u) {
        const int Lu = seq_len(u);
        rank += (Lu > Lt) || (Lu == Lt && u < t);
      }
      s_seq[rank] = t;
    }
    __syncthreads();
    b = s_seq[b];
  }
  const int kv0 = paged ? 0 : A.kv_off[b];
  const int L = paged ? A.kv_len[b] : A.kv_off[b + 1] - kv0;
  const bool bad_kv = (L < 0 || L > A.max_kv);
  // chunks that carry cache keys of this sequence; the last one also takes
  // the tree keys
  const int n_chunks = bad_kv ? 1 : max(1, (L + A.CK - 1) / A.CK);
  const int key_begin = c * A.CK;
  const int key_end = bad_kv ? key_begin : min(L, key_begin + A.CK);
  const int n_cache_blk = (key_end > key_begin) ? (key_end - key_begin + kKeyBlk - 1) / kKeyBlk : 0;
  const int early = paged ? 0 : min(2, n_cache_blk);
  int t0 = 0;   // set after the dependency wait
  // row of cache key pos in the cache tensor (128 keys from a multiple of
  // 128 never straddle a page: page sizes are multiples of 128)
  auto cache_row = [&](int pos) -> int {
    if (!paged) return kv0 + pos;
    int page = A.block_table[(size_t)b * A.max_pages + pos / A.page_size];
    if (page < 0 || page >= A.n_pages) {
      fail(A.status, EAGLE_ERR_INVALID_ARG);
      page = 0;
    }
    return page * A.page_size + pos % A.page_size;
  };
  auto block_row = [&](int j) {   // first key row of block j in its tensor
    return (j < n_cache_blk) ? cache_row(key_begin + j * kKeyBlk) : t0 + (j - n_cache_blk) * kKeyBlk;
  };
  auto load_k = [&](int j) {
    const int st = j & 1;
    unsigned char* kd = k_sm + st * kTileBytes;
    const CUtensorMap* mk = (j < n_cache_blk) ? &map_kc : &map_kt;
    tc::mbar_arrive_expect_tx(&sh->k_full[st], kTileBytes);
    tc::tma_load_3d(kd, mk, &sh->k_full[st], 0, g, block_row(j));
    tc::tma_load_3d(kd + kHalfBytes, mk, &sh->k_full[st], 64, g, block_row(j));
  };
  auto load_v = [&](int j) {
    const int st = j & 1;
    unsigned char* vd = v_sm + st * kTileBytes;
    const CUtensorMap* mv = (j < n_cache_blk) ? &map_vc : &map_vt;
    tc::mbar_arrive_expect_tx(&sh->v_full[st], kTileBytes);
    tc::tma_load_3d(vd, mv, &sh->v_full[st], 0, g, block_row(j));
    tc::tma_load_3d(vd + kHalfBytes, mv, &sh->v_full[st], 64, g, block_row(j));
  };
  if (threadIdx.x == 0) {
    tc::mbar_init(&sh->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sh->k_full[i], 1);
      tc::mbar_init(&sh->k_empty[i], 1);
      tc::mbar_init(&sh->v_full[i], 1);
      tc::mbar_init(&sh->v_empty[i], 1);
    }
    tc::fence_barrier_init();
    for (int j = 0; j < early; ++j) {
      load_k(j);
      load_v(j);
    }
  }
  if (!paged) pdl_begin();

  t0 = A.tree_off[b];
  const int n = A.tree_off[b + 1] - t0;
  const bool bad_seq = bad_kv || n < 1 || n > A.max_nodes;
  const int nodes_per_tile = 128 / A.G;
  // the whole cluster (same tile) leaves together
  if (bad_seq || mt * nodes_per_tile >= n) {
    if (bad_seq && c == 0 && mt == 0 && threadIdx.x == 0) fail(A.status, EAGLE_ERR_INVALID_TREE);
    if (threadIdx.x == 0) {
      // the cache blocks requested above land before the CTA leaves
      int never = 0;
      for (int j = 0; j < early; ++j) {
        tc::mbar_wait(&sh->k_full[j], 0, &never, nullptr, 200000000ll);
        tc::mbar_wait(&sh->v_full[j], 0, &never, nullptr, 200000000ll);
      }
    }
    return;
  }
  const bool with_tree = (c == n_chunks - 1);
  const int n_tree_blk = with_tree ? (n + kKeyBlk - 1) / kKeyBlk : 0;
  const int nblk = n_cache_blk + n_tree_blk;
  // row quads (32 rows) holding at least one node of the tile
  int active_quads = 0;
  for (int q = 0; q < 4; ++q) active_quads += ((mt * 128 + q * 32) / A.G < n);
  const int active_warps = 2 * active_quads;
  volatile int* abort_flag = &sh->abort_flag;
  int* status = A.status;

  if (threadIdx.x == 0) {
    tc::mbar_init(&sh->s_full, 1);
    tc::mbar_init(&sh->s_empty, active_warps);
    tc::mbar_init(&sh->p_full, active_warps);
    tc::mbar_init(&sh->pv_done, 1);
    tc::mbar_init(&sh->o_done, 1);
    tc::mbar_init(&sh->drain, 1);
    tc::mbar_init(&sh->fbar, 32 * active_warps);
    sh->abort_flag = 0;
    tc::fence_barrier_init();
    // the queries and the first blocks not requested before the wait
    if (nblk > 0) {
      tc::mbar_arrive_expect_tx(&sh->q_full, kTileBytes);
      const int node0 = t0 + mt * nodes_per_tile;
      tc::tma_load_3d(q_sm, &map_q, &sh->q_full, 0, g * A.G, node0);
      tc::tma_load_3d(q_sm + kHalfBytes, &map_q, &sh->q_full, 64, g * A.G, node0);
      for (int j = early; j < min(2, nblk); ++j) {
        load_k(j);
        load_v(j);
      }
    }
  }
  for (int i = threadIdx.x; i < n; i += kAttThreads) sh->par[i] = A.parent[t0 + i];
  if (warp == 1) {
    tc::tmem_alloc(&sh->tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const uint32_t tmem = sh->tmem_base;

  // row-thread state carried into the merge
  const int quad = warp & 3;
  const int half = (warp - 2) >> 2;                 // key half of every block
  const int r = quad * 32 + lane;                   // row in the tile
  const bool row_warp = warp >= 2 && quad < active_quads;
  float o0[32], o1[32];                             // output columns half*64 .. +63
  float m_row = -INFINITY, l_row = 0.f;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA
    if (lane == 0 && nblk > 2) {
      // K slots free after S, V slots only after PV: K(j+1) goes out before
      // V(j), the order in which the two kinds of slot are released
      bool tok = true;
      uint32_t kph = 0, vph = 0;   // bit st: phase parity of the empty barriers
      int nk = 2, nv = 2;          // blocks issued
      auto next_k = [&]() -> bool {
        const int st = nk & 1;
        if (!tc::mbar_wait(&sh->k_empty[st], (kph >> st) & 1u, abort_flag, status)) return false;
        kph ^= 1u << st;
        load_k(nk++);
        return true;
      };
      tok = next_k();
      while (tok && nv < nblk) {
        if (nk < nblk && !(tok = next_k())) break;
        const int st = nv & 1;
        if (!(tok = tc::mbar_wait(&sh->v_empty[st], (vph >> st) & 1u, abort_flag, status))) break;
        vph ^= 1u << st;
        load_v(nv++);
      }
      if (!tok) {
        // let the copies in flight (at most the last two of each kind) land
        int never = 0;
        tc::mbar_wait(&sh->q_full, 0, &never, nullptr, 200000000ll);
        for (int j = max(0, nk - 2); j < nk; ++j)
          tc::mbar_wait(&sh->k_full[j & 1], (j >> 1) & 1, &never, nullptr, 200000000ll);
        for (int j = max(0, nv - 2); j < nv; ++j)
          tc::mbar_wait(&sh->v_full[j & 1], (j >> 1) & 1, &never, nullptr, 200000000ll);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      if (nblk > 0) {
        const uint32_t idesc_s = tc::idesc_bf16_f32(128, kKeyBlk);
        const uint32_t idesc_o = tc::idesc_bf16_f32(128, 128) | (1u << 16);  // B is MN-major
        const uint32_t q_addr = tc::smem_u32(q_sm);
        bool mok = tc::mbar_wait(&sh->q_full, 0, abort_flag, status);
        uint32_t kph = 0, vph = 0;   // bit st: phase parity per stage
        auto issue_s = [&](int j) -> bool {
          const int st = j & 1;
          if (!tc::mbar_wait(&sh->k_full[st], (kph >> st) & 1u, abort_flag, status)) return false;
          kph ^= 1u << st;
          tc::fence_after_thread_sync();
          const uint32_t k_addr = tc::smem_u32(k_sm + st * kTileBytes);
#pragma unroll
          for (int k16 = 0; k16 < 8; ++k16) {
            const uint32_t off = (uint32_t)((k16 >> 2) * kHalfBytes + (k16 & 3) * 32);
            tc::mma_f16(tmem, tc::desc_kmajor_sw128(q_addr + off),
                        tc::desc_kmajor_sw128(k_addr + off), idesc_s, k16 > 0 ? 1u : 0u);
          }
          tc::mma_commit(&sh->s_full);
          tc::mma_commit(&sh->k_empty[st]);
          return true;
        };
        if (mok) mok = issue_s(0);
        for (int j = 0; j < nblk && mok; ++j) {
          const int st = j & 1;
          if (j + 1 < nblk) {
            // the next S goes into the slot as soon as every row has read this one
            if (!(mok = tc::mbar_wait(&sh->s_empty, (uint32_t)(j & 1), abort_flag, status))) break;
            if (!(mok = issue_s(j + 1))) break;
          }
          if (!(mok = tc::mbar_wait(&sh->p_full, (uint32_t)(j & 1), abort_flag, status))) break;
          if (!(mok = tc::mbar_wait(&sh->v_full[st], (vph >> st) & 1u, abort_flag, status))) break;
          vph ^= 1u << st;
          tc::fence_after_thread_sync();
          const uint32_t v_addr = tc::smem_u32(v_sm + st * kTileBytes);
          // O_h += P_hi V_h + P_lo V_h for key half h: A = P from the half's
          // TMEM columns, B = V rows of that half (MN-major, 128-byte rows).
          // The two halves' accumulator chains are interleaved (each in its
          // own order), so the tensor pipe always has an independent MMA.
          // (One bf16 P alone would round every weight by up to 2^-8 of
          // itself -- up to 2^-8 of sum_j p_j |v_j| in the output when few
          // keys dominate, above the 2e-3 bound; hi + lo keep 2^-16.)
#pragma unroll
          for (int part = 0; part < 2; ++part) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint32_t a_tm = tmem + (uint32_t)(128 + h * 64 + part * 32 + kk * 8);
                const uint32_t key = (uint32_t)(h * 64 + kk * 16);
                mma_f16_tmem_a(tmem + 256u + (uint32_t)(h * 128), a_tm,
                               desc_mnmajor_sw128(v_addr + key * 128u, kHalfBytes), idesc_o,
                               (j > 0 || part > 0 || kk > 0) ? 1u : 0u);
              }
            }
          }
          tc::mma_commit(&sh->pv_done);
          tc::mma_commit(&sh->v_empty[st]);
        }
        if (mok) tc::mma_commit(&sh->o_done);
      }
      tc::mma_commit(&sh->drain);
      int never = 0;
      tc::mbar_wait(&sh->drain, 0, &never, nullptr, 200000000ll);
    }
  } else if (row_warp) {
    // ------------------------------------------------------------ rows
    const int qrow = mt * 128 + r;                    // (node, head) row of (b, g)
    const int node = qrow / A.G;
    const bool row_ok = node < n;
    // ancestor-or-self bits of this row's node: word w covers tree nodes
    // 32*w .. 32*w+31
    uint32_t anc[EAGLE_MAX_TREE_NODES / 32];
#pragma unroll
    for (int w = 0; w < EAGLE_MAX_TREE_NODES / 32; ++w) anc[w] = 0u;
    if (row_ok && with_tree) {
      int j = node, steps = 0;
      while (j >= 0) {
#pragma unroll
        for (int w = 0; w < EAGLE_MAX_TREE_NODES / 32; ++w)
          if ((j >> 5) == w) anc[w] |= 1u << (j & 31);
        const int p = sh->par[j];
        if ((j == 0) ? (p != -1) : (p < 0 || p >= j) || ++steps > n) {
          if (half == 0) fail(status, EAGLE_ERR_INVALID_TREE);
          break;
        }
        j = p;
      }
    }
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t o_own = trow + 256u + (uint32_t)(half * 128);   // this key half's O
    float m = -INFINITY, l = 0.f;   // this key half's running max (log2 units) and sum
    for (int j = 0; j < nblk && ok; ++j) {
      const bool got = tc::mbar_wait(&sh->s_full, (uint32_t)(j & 1), abort_flag, status);
      if (!(ok = __all_sync(0xffffffffu, got))) break;
      tc::fence_after_thread_sync();
      const bool tree_blk = j >= n_cache_blk;
      const int tb = tree_blk ? j - n_cache_blk : 0;          // tree block 0 or 1
      const int key0 = (tree_blk ? tb * kKeyBlk : key_begin + j * kKeyBlk) + half * 64;
      const int key_lim = tree_blk ? n : key_end;
      const uint32_t s_addr = trow + (uint32_t)(half * 64);
      float v0[32], v1[32];
      tc::tmem_ld_32x32b_x32(s_addr, v0);
      tc::tmem_ld_32x32b_x32(s_addr + 32u, v1);
      // the S slot may take the next block
      tc::fence_before_thread_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->s_empty);
      // bitset words for key columns half*64 .. +63 of tree block tb (static indices)
      const uint32_t w0 = !tree_blk ? 0xffffffffu
                          : tb ? (half ? anc[6] : anc[4]) : (half ? anc[2] : anc[0]);
      const uint32_t w1 = !tree_blk ? 0xffffffffu
                          : tb ? (half ? anc[7] : anc[5]) : (half ? anc[3] : anc[1]);
      const int nv0 = min(32, max(0, key_lim - key0));
      const int nv1 = min(32, max(0, key_lim - key0 - 32));
      if (tree_blk || nv1 < 32) {
        // masked or ragged block (warp-uniform): hidden scores become -inf
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (!(i < nv0 && ((w0 >> i) & 1u))) v0[i] = -INFINITY;
          if (!(i < nv1 && ((w1 >> i) & 1u))) v1[i] = -INFINITY;
        }
      }
      float bm0 = v0[0], bm1 = v1[0];
#pragma unroll
      for (int i = 1; i < 32; ++i) {
        bm0 = fmaxf(bm0, v0[i]);
        bm1 = fmaxf(bm1, v1[i]);
      }
      const float bm = fmaxf(bm0, bm1) * A.scale_log2;
      const float mn = fmaxf(m, bm);
      const bool first = (m == -INFINITY);
      const bool rescale = !first && (mn > m + kRescaleLog2);
      const float mu = (first || rescale) ? mn : m;     // reference max for this block's P
      // P = exp2(s - mu) = hi + lo, both bf16: hi keeps the top 16 bits of
      // the fp32 value, lo = P - hi (exact in fp32) truncated the same way;
      // |P - hi - lo| < 2^-14 P.  Computed before waiting for the previous
      // PV, which still reads the P columns.
      float psum = 0.f;
      // a half-row with nothing visible yet keeps mu = -inf: its scores are
      // all -inf, and any finite offset gives P = 0
      const float neg_mu = (mu == -INFINITY) ? 0.f : -mu;
      uint32_t hi0[16], lo0[16], hi1[16], lo1[16];
      auto split = [&](const float (&v)[32], uint32_t (&hi)[16], uint32_t (&lo)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2_approx(fmaf(v[2 * i], A.scale_log2, neg_mu));
          const float p1 = ex2_approx(fmaf(v[2 * i + 1], A.scale_log2, neg_mu));
          const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
          hi[i] = __byte_perm(b0, b1, 0x7632);
          const float r0 = p0 - __uint_as_float(b0 & 0xffff0000u);
          const float r1 = p1 - __uint_as_float(b1 & 0xffff0000u);
          lo[i] = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
          psum += p0 + p1;
        }
      };
      split(v0, hi0, lo0);
      split(v1, hi1, lo1);
      if (j >= 1) {
        // the previous PV has read P and finished O (every earlier PV was
        // waited for one block before)
        const bool g4 = tc::mbar_wait(&sh->pv_done, (uint32_t)((j - 1) & 1), abort_flag, status);
        if (!(ok = __all_sync(0xffffffffu, g4))) break;
        tc::fence_after_thread_sync();
      }
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? ex2_approx(m - mu) : 1.f;
        float o[32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          tc::tmem_ld_32x32b_x32(o_own + (uint32_t)(cc * 32), o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tmem_st_32x32b_x32(o_own + (uint32_t)(cc * 32), o);
        }
        l *= f;
      }
      // hi to the half's P columns +0 .., lo to +32 ..
      const uint32_t pcol = trow + (uint32_t)(128 + half * 64);
      tmem_st_32x32b_x16(pcol, hi0);
      tmem_st_32x32b_x16(pcol + 16u, hi1);
      tmem_st_32x32b_x16(pcol + 32u, lo0);
      tmem_st_32x32b_x16(pcol + 48u, lo1);
      tmem_wait_st();
      l += psum;
      m = mu;
      tc::fence_before_thread_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->p_full);
    }
    if (!ok) {
      m = -INFINITY;
      l = 0.f;
    }
    // ---- merge the two key halves: (m, l) exchange, then this thread's
    // output columns half*64 .. +63 from both accumulators
    sh->xchg[0][half][r] = m;
    sh->xchg[1][half][r] = l;
    tc::mbar_arrive(&sh->fbar);
    const bool gf = tc::mbar_wait(&sh->fbar, 0, abort_flag, status);
    ok = __all_sync(0xffffffffu, gf) && ok;
    const float mo = sh->xchg[0][half ^ 1][r], lo_ = sh->xchg[1][half ^ 1][r];
    const float M = fmaxf(m, mo);
    const float ws = (m == -INFINITY) ? 0.f : ex2_approx(m - M);
    const float wo = (mo == -INFINITY) ? 0.f : ex2_approx(mo - M);
    m_row = M;
    l_row = ws * l + wo * lo_;
    bool have_o = false;
    if (ok && nblk > 0) {
      const bool got = tc::mbar_wait(&sh->o_done, 0, abort_flag, status);
      if ((ok = __all_sync(0xffffffffu, got))) {
        have_o = true;
        tc::fence_after_thread_sync();
        const uint32_t o_oth = trow + 256u + (uint32_t)((half ^ 1) * 128);
        float t[32];
        tc::tmem_ld_32x32b_x32(o_own + (uint32_t)(half * 64), o0);
        tc::tmem_ld_32x32b_x32(o_oth + (uint32_t)(half * 64), t);
#pragma unroll
        for (int i = 0; i < 32; ++i) o0[i] = ws * o0[i] + wo * t[i];
        tc::tmem_ld_32x32b_x32(o_own + (uint32_t)(half * 64 + 32), o1);
        tc::tmem_ld_32x32b_x32(o_oth + (uint32_t)(half * 64 + 32), t);
#pragma unroll
        for (int i = 0; i < 32; ++i) o1[i] = ws * o1[i] + wo * t[i];
      }
    }
    if (!have_o) {
#pragma unroll
      for (int i = 0; i < 32; ++i) o0[i] = o1[i] = 0.f;
    }
    if (!ok) {
      m_row = -INFINITY;
      l_row = 0.f;
    }
  }

  // ---------------------------------------------------------------- output
  if (A.NC == 1) {
    if (row_warp) {
      const int qrow = mt * 128 + r;
      const int node = qrow / A.G, hh = qrow % A.G;
      if (node < n && ok) {
        float* orow = A.out + ((size_t)(t0 + node) * A.Hq + g * A.G + hh) * 128 + half * 64;
        const float inv = 1.f / l_row;
#pragma unroll
        for (int d = 0; d < 32; d += 4) {
          *reinterpret_cast<float4*>(orow + d) =
              make_float4(o0[d] * inv, o0[d + 1] * inv, o0[d + 2] * inv, o0[d + 3] * inv);
          *reinterpret_cast<float4*>(orow + 32 + d) =
              make_float4(o1[d] * inv, o1[d + 1] * inv, o1[d + 2] * inv, o1[d + 3] * inv);
        }
      }
    }
  } else {
    // merge the cluster's chunks: out = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
    // Rows [R0(c), R0(c+1)) belong to CTA c; every CTA pushes its partial
    // rows into the owner's K/V stage memory (free once the whole cluster
    // is past its key loop), and owners combine from local shared memory.
    cg::cluster_group cluster = cg::this_cluster();
    const int NC = A.NC;
    const int RPO = (128 + NC - 1) / NC;            // rows per owner, at most
    float4* mbuf = reinterpret_cast<float4*>(k_sm);                   // [NC][RPO][32]
    float2* mlbuf = reinterpret_cast<float2*>(k_sm + kMergeMlOffset); // [NC][RPO]
    auto row0 = [&](int cc) { return (128 * cc) / NC; };
    cluster.sync();
    if (row_warp) {
      int owner = 0;
      while (owner + 1 < NC && row0(owner + 1) <= r) ++owner;
      const int lrow = r - row0(owner);
      float4* dst = cluster.map_shared_rank(mbuf, owner) + (size_t)(c * RPO + lrow) * 32;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c4 = half * 16 + i;
        dst[c4 ^ (lrow & 31)] = make_float4(o0[4 * i], o0[4 * i + 1], o0[4 * i + 2], o0[4 * i + 3]);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c4 = half * 16 + 8 + i;
        dst[c4 ^ (lrow & 31)] = make_float4(o1[4 * i], o1[4 * i + 1], o1[4 * i + 2], o1[4 * i + 3]);
      }
      if (half == 0) cluster.map_shared_rank(mlbuf, owner)[c * RPO + lrow] = make_float2(m_row, l_row);
    }
    cluster.sync();
    const int R0 = row0(c), R1 = row0(c + 1);
    for (int idx = threadIdx.x; idx < (R1 - R0) * 32; idx += kAttThreads) {
      const int lrow = idx / 32, c4 = idx % 32;
      const int qrow = mt * 128 + R0 + lrow;
      const int node = qrow / A.G, hh = qrow % A.G;
      if (node >= n) continue;
      float M = -INFINITY;
      for (int cc = 0; cc < NC; ++cc) M = fmaxf(M, mlbuf[cc * RPO + lrow].x);
      float Ls = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int cc = 0; cc < NC; ++cc) {
        const float2 ml = mlbuf[cc * RPO + lrow];
        if (ml.x == -INFINITY) continue;
        const float w = ex2_approx(ml.x - M);
        const float4 x = mbuf[(cc * RPO + lrow) * 32 + (c4 ^ (lrow & 31))];
        Ls += w * ml.y;
        acc.x += w * x.x;
        acc.y += w * x.y;
        acc.z += w * x.z;
        acc.w += w * x.w;
      }
      const float inv = 1.f / Ls;
      *reinterpret_cast<float4*>(A.out + ((size_t)(t0 + node) * A.Hq + g * A.G + hh) * 128 +
                                 c4 * 4) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_thread_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 att_encode() {
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

// 3-D bf16 tensor [rows, heads, 128] -> boxes of 64 x box_heads x box_rows,
// 128-byte swizzle; out-of-range elements read as zero.
bool make_map_3d(CUtensorMap* map, const void* ptr, int rows, int heads, int box_heads,
                 int box_rows) {
  auto enc = att_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)std::max(rows, 1)};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Largest cluster size <= kMaxSplit such that `tiles` clusters of the
// attention kernel are resident at once (one wave), per device.
int split_cap_for(int tiles) {
  static std::mutex mu;
  static int cache[kMaxDevices][kMaxSplit + 1];
  static bool filled[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (!filled[dev]) {
    for (int nc = 1; nc <= kMaxSplit; ++nc) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)nc);
      cfg.blockDim = dim3(kAttThreads);
      cfg.dynamicSmemBytes = kAttSmem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = (unsigned)nc;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int q = 0;
      if (cudaOccupancyMaxActiveClusters(&q, tree_attn_tc_kernel, &cfg) != cudaSuccess) q = 0;
      cache[dev][nc] = q;
    }
    (void)cudaGetLastError();
    filled[dev] = true;
  }
  int nc = kMaxSplit;
  while (nc > 1 && cache[dev][nc] < tiles) --nc;
  return nc;
}

bool tc_shape_ok(eagle_dtype dtype, int Hq, int Hkv, int D) {
  if (dtype != EAGLE_BF16 || D != 128) return false;
  const int G = Hq / Hkv;
  return G >= 1 && G <= 128 && (128 % G) == 0;
}

}  // namespace

// Neither path needs global scratch: the tensor-core path merges its cache
// chunks inside a thread-block cluster.
extern "C" size_t eagle_tree_attn_workspace_bytes(int B, int T, int Hq, int Hkv, int D,
                                                  int max_nodes, int max_kv) {
  (void)B;
  (void)T;
  (void)Hq;
  (void)Hkv;
  (void)D;
  (void)max_nodes;
  (void)max_kv;
  return 0;
}

namespace {

// Both entry points: the cache is `cache_rows` rows of [Hkv, D] in kc / vc,
// indexed by `ci`.
eagle_status attn_impl(eagle_dtype dtype, int B, int T, int Hq, int Hkv, int D, float scale,
                       int max_nodes, int max_kv, int cache_rows, const void* d_q,
                       const void* d_k_tree, const void* d_v_tree, const void* d_k_cache,
                       const void* d_v_cache, const CacheIndex& ci, const int32_t* d_tree_off,
                       const int32_t* d_parent, float* d_out, int* d_status, cudaStream_t s) {
  const uintptr_t align = (uintptr_t)d_q | (uintptr_t)d_k_tree | (uintptr_t)d_v_tree |
                          (uintptr_t)d_k_cache | (uintptr_t)d_v_cache | (uintptr_t)d_out;
  const bool pages_ok = ci.page_size == 0 || ci.page_size % kKeyBlk == 0;
  if (tc_shape_ok(dtype, Hq, Hkv, D) && (align & 15) == 0 && pages_ok) {
    static PerDeviceOnce attr_once;
    if (attr_once.run([] {
          return cudaFuncSetAttribute(tree_attn_tc_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttSmem);
        }) != cudaSuccess)
      return EAGLE_ERR_CUDA;
    const int G = Hq / Hkv;
    const int tiles = B * Hkv * ((max_nodes * G + 127) / 128);
    const AttPlan P = att_plan(B, Hq, Hkv, max_nodes, max_kv, split_cap_for(tiles));
    CUtensorMap mq, mkc, mvc, mkt, mvt;
    const void* kc = (cache_rows > 0) ? d_k_cache : d_k_tree;   // never read when empty
    const void* vc = (cache_rows > 0) ? d_v_cache : d_v_tree;
    const int rows_c = (cache_rows > 0) ? cache_rows : T;
    if (!make_map_3d(&mq, d_q, T, Hq, P.G, 128 / P.G) ||
        !make_map_3d(&mkc, kc, rows_c, Hkv, 1, kKeyBlk) ||
        !make_map_3d(&mvc, vc, rows_c, Hkv, 1, kKeyBlk) ||
        !make_map_3d(&mkt, d_k_tree, T, Hkv, 1, kKeyBlk) ||
        !make_map_3d(&mvt, d_v_tree, T, Hkv, 1, kKeyBlk))
      return EAGLE_ERR_CUDA;
    AttParams A;
    A.B = B;
    A.Hq = Hq;
    A.Hkv = Hkv;
    A.G = P.G;
    A.MT = P.MT;
    A.NC = P.NC;
    A.CK = P.CK;
    A.max_nodes = max_nodes;
    A.max_kv = max_kv;
    A.scale_log2 = scale * 1.4426950408889634f;
    A.kv_off = ci.kv_off;
    A.page_size = ci.page_size;
    A.max_pages = ci.max_pages;
    A.n_pages = ci.n_pages;
    A.block_table = ci.block_table;
    A.kv_len = ci.kv_len;
    A.tree_off = d_tree_off;
    A.parent = d_parent;
    A.out = d_out;
    A.status = d_status;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * Hkv * P.MT * P.NC));
    cfg.blockDim = dim3(kAttThreads);
    cfg.dynamicSmemBytes = kAttSmem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = (unsigned)P.NC;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = (P.NC > 1) ? 2 : 1;
    return launch_status(cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel, mq, mkc, mvc, mkt, mvt, A));
  }
  if (dtype == EAGLE_BF16)
    return launch_warp<__nv_bfloat16>(D, B, T, Hq, Hkv, scale, max_nodes, max_kv, d_q, d_k_tree,
                                      d_v_tree, d_k_cache, d_v_cache, ci, d_tree_off, d_parent,
                                      d_out, d_status, s);
  return launch_warp<float>(D, B, T, Hq, Hkv, scale, max_nodes, max_kv, d_q, d_k_tree, d_v_tree,
                            d_k_cache, d_v_cache, ci, d_tree_off, d_parent, d_out, d_status, s);
}

}  // namespace

extern "C" eagle_status eagle_tree_attn(eagle_dtype dtype, int B, int T, int Hq, int Hkv, int D,
                                        float scale, int max_nodes, int max_kv, int kv_rows,
                                        const void* d_q,
                                        const void* d_k_tree, const void* d_v_tree,
                                        const void* d_k_cache, const void* d_v_cache,
                                        const int32_t* d_kv_off, const int32_t* d_tree_off,
                                        const int32_t* d_parent, float* d_out, void* d_ws,
                                        size_t ws_bytes, int* d_status, eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 1 && T >= 0 && Hq >= 1 && Hkv >= 1 && max_kv >= 0, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(Hq % Hkv == 0, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(D == 64 || D == 128, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(dtype == EAGLE_F32 || dtype == EAGLE_BF16, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(max_nodes >= 1 && max_nodes <= EAGLE_MAX_TREE_NODES, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(isfinite(scale), EAGLE_ERR_INVALID_ARG);
  if (T == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_q && d_k_tree && d_v_tree && d_kv_off && d_tree_off && d_parent && d_out &&
                       d_status,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(max_kv == 0 || (d_k_cache && d_v_cache), EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(ws_bytes >= eagle_tree_attn_workspace_bytes(B, T, Hq, Hkv, D, max_nodes, max_kv),
                   EAGLE_ERR_WORKSPACE);
  EAGLE_HOST_CHECK(kv_rows >= 0, EAGLE_ERR_INVALID_ARG);
  (void)d_ws;
  CacheIndex ci = {d_kv_off, nullptr, nullptr, 0, 0, 0};
  return attn_impl(dtype, B, T, Hq, Hkv, D, scale, max_nodes, max_kv, kv_rows, d_q, d_k_tree,
                   d_v_tree, d_k_cache, d_v_cache, ci, d_tree_off, d_parent, d_out, d_status,
                   (cudaStream_t)stream);
}

extern "C" eagle_status eagle_tree_attn_paged(
    eagle_dtype dtype, int B, int T, int Hq, int Hkv, int D, float scale, int max_nodes,
    int max_kv, int page_size, int n_pages, int max_pages, const void* d_q,
    const void* d_k_tree, const void* d_v_tree, const void* d_k_pages, const void* d_v_pages,
    const int32_t* d_block_table, const int32_t* d_kv_len, const int32_t* d_tree_off,
    const int32_t* d_parent, float* d_out, int* d_status, eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 1 && T >= 0 && Hq >= 1 && Hkv >= 1 && max_kv >= 0, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(Hq % Hkv == 0, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(D == 64 || D == 128, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(dtype == EAGLE_F32 || dtype == EAGLE_BF16, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(max_nodes >= 1 && max_nodes <= EAGLE_MAX_TREE_NODES, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(isfinite(scale), EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(page_size >= 1 && n_pages >= 0 && max_pages >= 0, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK((long long)max_pages * page_size >= max_kv, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK((long long)n_pages * page_size <= 0x7fffffffll, EAGLE_ERR_UNSUPPORTED);
  if (T == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_q && d_k_tree && d_v_tree && d_kv_len && d_tree_off && d_parent && d_out &&
                       d_status,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(max_kv == 0 || (d_k_pages && d_v_pages && d_block_table && n_pages >= 1),
                   EAGLE_ERR_INVALID_ARG);
  CacheIndex ci = {nullptr, d_kv_len, d_block_table, page_size, max_pages, n_pages};
  return attn_impl(dtype, B, T, Hq, Hkv, D, scale, max_nodes, max_kv,
                   max_kv > 0 ? n_pages * page_size : 0, d_q, d_k_tree, d_v_tree, d_k_pages,
                   d_v_pages, ci, d_tree_off, d_parent, d_out, d_status, (cudaStream_t)stream);
}
