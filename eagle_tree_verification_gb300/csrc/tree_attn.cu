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
//                          one thread per query row applies the mask (cache
//                          bound, or the row's ancestor bitset built on chip
//                          from parent[]) and the online softmax, writes P
//                          (bf16) back to shared memory, and tcgen05.mma
//                          forms P V into TMEM, which the same thread folds
//                          into its fp32 output row.  Chunks of one
//                          (sequence, head, tile) are merged by the last CTA
//                          to finish (atomic ticket, no waiting).
//   tree_attn_warp_kernel  CUDA-core kernel for fp32 inputs and other shapes:
//                          one warp per (node, query head).
// The ancestor mask is never stored: it is derived from parent[] on the fly.
#include <math.h>

#include <algorithm>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc.cuh"

using namespace eagle;

namespace {

constexpr int kWarpsPerBlock = 4;

template <typename TIn, int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
tree_attn_warp_kernel(int B, int T, int Hq, int Hkv, float scale, int max_nodes, int max_kv,
                      const TIn* __restrict__ q, const TIn* __restrict__ k_tree,
                      const TIn* __restrict__ v_tree, const TIn* __restrict__ k_cache,
                      const TIn* __restrict__ v_cache, const int* __restrict__ kv_off,
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
  const int c0 = kv_off[b], L = kv_off[b + 1] - c0;
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
    const size_t off = ((size_t)(c0 + j) * Hkv + g) * D;
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
                         const void* kc, const void* vc, const int* kv_off, const int* tree_off,
                         const int* parent, float* out, int* status, cudaStream_t s) {
  const int warps = T * Hq;
  const int grid = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const TIn* Q = static_cast<const TIn*>(q);
  const TIn* KT = static_cast<const TIn*>(kt);
  const TIn* VT = static_cast<const TIn*>(vt);
  const TIn* KC = static_cast<const TIn*>(kc);
  const TIn* VC = static_cast<const TIn*>(vc);
  auto kern = (D == 64) ? tree_attn_warp_kernel<TIn, 64> : tree_attn_warp_kernel<TIn, 128>;
  return launch_status(launch_pdl(kern, dim3(grid), dim3(kWarpsPerBlock * 32), 0, s, B, T, Hq,
                                  Hkv, scale, max_nodes, max_kv, Q, KT, VT, KC, VC, kv_off,
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
constexpr size_t kAttSmem = 1024 + 7 * (size_t)kTileBytes + 1280;

struct AttShared {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full, p_free, o_done, drain;
  uint64_t xbar, fbar, tbar0, tbar1;   // row-thread exchanges and the merge ticket
  uint32_t tmem_base;
  int abort_flag;
  int is_last;
  float xchg[2][128];   // per-row values exchanged between the two column halves
};

static_assert(sizeof(AttShared) <= 1280, "AttShared must fit its shared-memory slot");

struct AttPlan {
  int G, MT, NC, CK;  // heads per kv head, row tiles, cache chunks, keys per chunk
  size_t off_ml, off_o, total;
};

AttPlan att_plan(int B, int Hq, int Hkv, int max_nodes, int max_kv) {
  AttPlan P;
  P.G = Hq / Hkv;
  P.MT = (max_nodes * P.G + 127) / 128;
  const int per_chunk_items = std::max(1, B * Hkv * P.MT);
  int nc = std::max(1, kTargetCtas / per_chunk_items);
  int ck = (max_kv + nc - 1) / nc;
  ck = std::max(256, ((ck + kKeyBlk - 1) / kKeyBlk) * kKeyBlk);
  P.CK = ck;
  P.NC = std::max(1, (max_kv + ck - 1) / ck);
  const size_t tiles = (size_t)B * Hkv * P.MT;
  const size_t items = tiles * P.NC;
  P.off_ml = ((tiles * 4) + 255) & ~(size_t)255;
  P.off_o = P.off_ml + ((items * 128 * 8 + 255) & ~(size_t)255);
  P.total = P.off_o + items * 128 * 128 * 4;
  return P;
}

struct AttParams {
  int B, Hq, Hkv, G, MT, NC, CK, max_nodes, max_kv;
  float scale_log2;
  const int* kv_off;
  const int* tree_off;
  const int* parent;
  float* out;
  int* counters;       // [B*Hkv*MT]
  float2* part_ml;     // [items][128] (m, l)
  float* part_o;       // [items][128][128]
  int* status;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
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
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kAttThreads, 1)
tree_attn_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_kc,
                    const __grid_constant__ CUtensorMap map_vc,
                    const __grid_constant__ CUtensorMap map_kt,
                    const __grid_constant__ CUtensorMap map_vt, const AttParams A) {
  pdl_begin();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* q_sm = base;                       // [2 halves][128 rows][128 B]
  unsigned char* k_sm = base + kTileBytes;          // 2 stages
  unsigned char* v_sm = base + 3 * kTileBytes;      // 2 stages
  unsigned char* p_sm = base + 5 * kTileBytes;      // P, high bf16 part
  unsigned char* pl_sm = base + 6 * kTileBytes;     // P, low bf16 part
  AttShared* sh = reinterpret_cast<AttShared*>(base + 7 * kTileBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work item: ((b * Hkv + g) * NC + c) * MT + mt  (row tiles of one chunk adjacent)
  int item = blockIdx.x;
  const int mt = item % A.MT;
  item /= A.MT;
  const int c = item % A.NC;
  item /= A.NC;
  const int g = item % A.Hkv;
  const int b = item / A.Hkv;
  const int tile_id = (b * A.Hkv + g) * A.MT + mt;
  const int item_id = tile_id * A.NC + c;

  const int t0 = A.tree_off[b];
  const int n = A.tree_off[b + 1] - t0;
  const int kv0 = A.kv_off[b];
  const int L = A.kv_off[b + 1] - kv0;
  const bool bad_seq = (n < 1 || n > A.max_nodes || L < 0 || L > A.max_kv);
  // chunks that carry cache keys of this sequence; the last one also takes
  // the tree keys
  const int n_chunks = bad_seq ? 1 : max(1, (L + A.CK - 1) / A.CK);
  const int nodes_per_tile = 128 / A.G;
  const bool tile_used = !bad_seq && mt * nodes_per_tile < n;
  if (c >= n_chunks || !tile_used) {
    if (bad_seq && c == 0 && mt == 0 && threadIdx.x == 0) fail(A.status, EAGLE_ERR_INVALID_TREE);
    return;
  }
  const int key_begin = c * A.CK;
  const int key_end = min(L, key_begin + A.CK);
  const int n_cache_blk = (key_end - key_begin + kKeyBlk - 1) / kKeyBlk;
  const bool with_tree = (c == n_chunks - 1);
  const int n_tree_blk = with_tree ? (n + kKeyBlk - 1) / kKeyBlk : 0;
  const int nblk = n_cache_blk + n_tree_blk;

  if (threadIdx.x == 0) {
    tc::mbar_init(&sh->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sh->k_full[i], 1);
      tc::mbar_init(&sh->k_empty[i], 1);
      tc::mbar_init(&sh->v_full[i], 1);
      tc::mbar_init(&sh->v_empty[i], 1);
      tc::mbar_init(&sh->s_full[i], 1);
      tc::mbar_init(&sh->s_empty[i], 8);
    }
    tc::mbar_init(&sh->p_full, 8);
    tc::mbar_init(&sh->p_free, 1);
    tc::mbar_init(&sh->o_done, 1);
    tc::mbar_init(&sh->drain, 1);
    tc::mbar_init(&sh->xbar, 256);
    tc::mbar_init(&sh->fbar, 256);
    tc::mbar_init(&sh->tbar0, 256);
    tc::mbar_init(&sh->tbar1, 1);
    sh->abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&sh->tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_thread_sync();
  __syncthreads();
  tc::fence_after_thread_sync();
  const uint32_t tmem = sh->tmem_base;     // S[0] at +0, S[1] at +128, O at +256
  volatile int* abort_flag = &sh->abort_flag;
  int* status = A.status;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA
    if (lane == 0) {
      bool ok = true;
      tc::mbar_arrive_expect_tx(&sh->q_full, kTileBytes);
      const int node0 = t0 + mt * nodes_per_tile;
      tc::tma_load_3d(q_sm, &map_q, &sh->q_full, 0, g * A.G, node0);
      tc::tma_load_3d(q_sm + kHalfBytes, &map_q, &sh->q_full, 64, g * A.G, node0);
      uint32_t eph = 0;   // bit st: phase parity of stage st's empty barriers
      int issued = 0;
      for (int j = 0; j < nblk && ok; ++j) {
        const int st = j & 1;
        if (j >= 2) {
          if (!(ok = tc::mbar_wait(&sh->k_empty[st], (eph >> st) & 1u, abort_flag, status))) break;
          if (!(ok = tc::mbar_wait(&sh->v_empty[st], (eph >> st) & 1u, abort_flag, status))) break;
          eph ^= 1u << st;
        }
        const CUtensorMap* mk = (j < n_cache_blk) ? &map_kc : &map_kt;
        const CUtensorMap* mv = (j < n_cache_blk) ? &map_vc : &map_vt;
        const int row = (j < n_cache_blk) ? kv0 + key_begin + j * kKeyBlk
                                          : t0 + (j - n_cache_blk) * kKeyBlk;
        unsigned char* kd = k_sm + st * kTileBytes;
        unsigned char* vd = v_sm + st * kTileBytes;
        tc::mbar_arrive_expect_tx(&sh->k_full[st], kTileBytes);
        tc::tma_load_3d(kd, mk, &sh->k_full[st], 0, g, row);
        tc::tma_load_3d(kd + kHalfBytes, mk, &sh->k_full[st], 64, g, row);
        tc::mbar_arrive_expect_tx(&sh->v_full[st], kTileBytes);
        tc::tma_load_3d(vd, mv, &sh->v_full[st], 0, g, row);
        tc::tma_load_3d(vd + kHalfBytes, mv, &sh->v_full[st], 64, g, row);
        ++issued;
      }
      if (!ok) {
        // let the copies in flight (at most the last two blocks) land
        int never = 0;
        tc::mbar_wait(&sh->q_full, 0, &never, nullptr, 200000000ll);
        for (int j = max(0, issued - 2); j < issued; ++j) {
          tc::mbar_wait(&sh->k_full[j & 1], (j >> 1) & 1, &never, nullptr, 200000000ll);
          tc::mbar_wait(&sh->v_full[j & 1], (j >> 1) & 1, &never, nullptr, 200000000ll);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      const uint32_t idesc_s = tc::idesc_bf16_f32(128, kKeyBlk);
      const uint32_t idesc_o = tc::idesc_bf16_f32(128, 128) | (1u << 16);  // B is MN-major
      const uint32_t q_addr = tc::smem_u32(q_sm);
      const uint32_t p_addr = tc::smem_u32(p_sm);
      const uint32_t pl_addr = tc::smem_u32(pl_sm);
      bool ok = tc::mbar_wait(&sh->q_full, 0, abort_flag, status);
      uint32_t kph = 0, vph = 0, seph = 0;   // bit st: phase parity per stage
      uint32_t pph = 0;
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (j >= 2) {
          if (!tc::mbar_wait(&sh->s_empty[st], (seph >> st) & 1u, abort_flag, status)) return false;
          seph ^= 1u << st;
        }
        if (!tc::mbar_wait(&sh->k_full[st], (kph >> st) & 1u, abort_flag, status)) return false;
        kph ^= 1u << st;
        tc::fence_after_thread_sync();
        const uint32_t k_addr = tc::smem_u32(k_sm + st * kTileBytes);
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16) {
          const uint32_t off = (uint32_t)((k16 >> 2) * kHalfBytes + (k16 & 3) * 32);
          tc::mma_f16(tmem + (uint32_t)(st * 128), tc::desc_kmajor_sw128(q_addr + off),
                      tc::desc_kmajor_sw128(k_addr + off), idesc_s, k16 > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sh->s_full[st]);
        tc::mma_commit(&sh->k_empty[st]);
        return true;
      };
      if (ok && nblk > 0) ok = issue_s(0);
      for (int j = 0; j < nblk && ok; ++j) {
        if (j + 1 < nblk && !(ok = issue_s(j + 1))) break;
        const int st = j & 1;
        if (!(ok = tc::mbar_wait(&sh->p_full, pph, abort_flag, status))) break;
        pph ^= 1;
        if (!(ok = tc::mbar_wait(&sh->v_full[st], (vph >> st) & 1u, abort_flag, status))) break;
        vph ^= 1u << st;
        tc::fence_after_thread_sync();
        const uint32_t v_addr = tc::smem_u32(v_sm + st * kTileBytes);
        // O += P_hi V + P_lo V: A = P parts (K-major, keys contiguous),
        // B = V (MN-major: one 128-byte row per key and d-half)
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t pa = part ? pl_addr : p_addr;
#pragma unroll
          for (int k16 = 0; k16 < 8; ++k16) {
            const uint32_t a_off = (uint32_t)((k16 >> 2) * kHalfBytes + (k16 & 3) * 32);
            tc::mma_f16(tmem + 256u, tc::desc_kmajor_sw128(pa + a_off),
                        desc_mnmajor_sw128(v_addr + (uint32_t)(k16 * 16 * 128), kHalfBytes),
                        idesc_o, (j > 0 || part > 0 || k16 > 0) ? 1u : 0u);
          }
        }
        tc::mma_commit(&sh->p_free);
        tc::mma_commit(&sh->v_empty[st]);
      }
      if (ok) tc::mma_commit(&sh->o_done);
      tc::mma_commit(&sh->drain);
      int never = 0;
      tc::mbar_wait(&sh->drain, 0, &never, nullptr, 200000000ll);
    }
  } else {
    // ------------------------------------------------------------ rows
    // two threads per query row: half 0 owns key columns / d columns 0-63,
    // half 1 owns 64-127
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;                   // row in the tile
    const int qrow = mt * 128 + r;                    // (node, head) row of (b, g)
    const int node = qrow / A.G, hh = qrow % A.G;
    const bool row_ok = node < n;
    // ancestor-or-self bits of this row's node for the key columns this
    // thread owns: word w covers tree nodes 32*w .. 32*w+31
    uint32_t anc[EAGLE_MAX_TREE_NODES / 32];
#pragma unroll
    for (int w = 0; w < EAGLE_MAX_TREE_NODES / 32; ++w) anc[w] = 0u;
    if (row_ok && with_tree) {
      int j = node, steps = 0;
      while (j >= 0) {
#pragma unroll
        for (int w = 0; w < EAGLE_MAX_TREE_NODES / 32; ++w)
          if ((j >> 5) == w) anc[w] |= 1u << (j & 31);
        const int p = __ldg(A.parent + t0 + j);
        if ((j == 0) ? (p != -1) : (p < 0 || p >= j) || ++steps > n) {
          if (half == 0) fail(status, EAGLE_ERR_INVALID_TREE);
          break;
        }
        j = p;
      }
    }
    const uint32_t p_row = tc::smem_u32(p_sm) + (uint32_t)(half * kHalfBytes + r * 128);
    const uint32_t pl_row = tc::smem_u32(pl_sm) + (uint32_t)(half * kHalfBytes + r * 128);
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t o_addr = trow + 256u + (uint32_t)(half * 64);
    float m = -INFINITY, l = 0.f;   // l: this half's share of the normaliser
    uint32_t sph = 0, pfph = 0;   // sph bit st: phase parity of s_full[st]
    bool ok = true;
    for (int j = 0; j < nblk && ok; ++j) {
      const int st = j & 1;
      const bool got = tc::mbar_wait(&sh->s_full[st], (sph >> st) & 1u, abort_flag, status);
      if (!(ok = __all_sync(0xffffffffu, got))) break;
      sph ^= 1u << st;
      tc::fence_after_thread_sync();
      const bool tree_blk = j >= n_cache_blk;
      const int tb = tree_blk ? j - n_cache_blk : 0;          // tree block 0 or 1
      const int key0 = (tree_blk ? tb * kKeyBlk : key_begin + j * kKeyBlk) + half * 64;
      const int key_lim = tree_blk ? n : key_end;
      const uint32_t s_addr = trow + (uint32_t)(st * 128 + half * 64);
      float v0[32], v1[32];
      tc::tmem_ld_32x32b_x32(s_addr, v0);
      tc::tmem_ld_32x32b_x32(s_addr + 32u, v1);
      // bitset words for key columns half*64 .. +63 of tree block tb (static indices)
      const uint32_t w0 = !tree_blk ? 0xffffffffu
                          : tb ? (half ? anc[6] : anc[4]) : (half ? anc[2] : anc[0]);
      const uint32_t w1 = !tree_blk ? 0xffffffffu
                          : tb ? (half ? anc[7] : anc[5]) : (half ? anc[3] : anc[1]);
      const int nv0 = min(32, max(0, key_lim - key0));
      const int nv1 = min(32, max(0, key_lim - key0 - 32));
      float bm = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (i < nv0 && ((w0 >> i) & 1u)) bm = fmaxf(bm, v0[i]);
        if (i < nv1 && ((w1 >> i) & 1u)) bm = fmaxf(bm, v1[i]);
      }
      bm *= A.scale_log2;
      // the previous PV product must be complete before P, O or the exchange
      // slot (read by the other half before it released that product) is reused
      if (j >= 1) {
        const bool g2 = tc::mbar_wait(&sh->p_free, pfph, abort_flag, status);
        if (!(ok = __all_sync(0xffffffffu, g2))) break;
        pfph ^= 1;
        tc::fence_after_thread_sync();
      }
      // the row's block max: combine with the other half
      sh->xchg[half][r] = bm;
      tc::mbar_arrive(&sh->xbar);
      const bool g3 = tc::mbar_wait(&sh->xbar, (uint32_t)(j & 1), abort_flag, status);
      if (!(ok = __all_sync(0xffffffffu, g3))) break;
      bm = fmaxf(bm, sh->xchg[half ^ 1][r]);
      const float mn = fmaxf(m, bm);
      const bool first = (m == -INFINITY);
      const bool rescale = !first && (mn > m + kRescaleLog2);
      const float mu = (first || rescale) ? mn : m;     // reference max for this block's P
      if (rescale) {
        const float f = exp2f(m - mu);
        float o[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          tc::tmem_ld_32x32b_x32(o_addr + (uint32_t)(cc * 32), o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tmem_st_32x32b_x32(o_addr + (uint32_t)(cc * 32), o);
        }
        l *= f;
      }
      // P = exp2(s - mu) split into bf16 hi + lo, into the swizzled P tiles
      float psum = 0.f;
      auto emit = [&](float (&v)[32], int nvc, uint32_t wc, int cc) {
        float lo[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const bool vis = (i < nvc) && ((wc >> i) & 1u);
          const float pv = vis ? exp2f(fmaf(v[i], A.scale_log2, -mu)) : 0.f;
          const float hi = __bfloat162float(__float2bfloat16_rn(pv));
          lo[i] = pv - hi;
          v[i] = hi;
          psum += pv;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = cc * 4 + u;   // 16-byte unit of this half's 128-byte row
          const uint32_t off = (uint32_t)(((unit ^ (r & 7)) & 7) * 16);
          st_shared_v4(p_row + off, pack_bf16(v[u * 8 + 0], v[u * 8 + 1]),
                       pack_bf16(v[u * 8 + 2], v[u * 8 + 3]), pack_bf16(v[u * 8 + 4], v[u * 8 + 5]),
                       pack_bf16(v[u * 8 + 6], v[u * 8 + 7]));
          st_shared_v4(pl_row + off, pack_bf16(lo[u * 8 + 0], lo[u * 8 + 1]),
                       pack_bf16(lo[u * 8 + 2], lo[u * 8 + 3]),
                       pack_bf16(lo[u * 8 + 4], lo[u * 8 + 5]),
                       pack_bf16(lo[u * 8 + 6], lo[u * 8 + 7]));
        }
      };
      emit(v0, nv0, w0, 0);
      emit(v1, nv1, w1, 1);
      l += psum;
      m = mu;
      fence_proxy_async_smem();
      tc::fence_before_thread_sync();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&sh->s_empty[st]);
        tc::mbar_arrive(&sh->p_full);
      }
    }
    // ---- the output rows: O (in TMEM) / l
    float o0[32], o1[32];
    if (ok && nblk > 0) {
      const bool got = tc::mbar_wait(&sh->o_done, 0, abort_flag, status);
      if ((ok = __all_sync(0xffffffffu, got))) {
        tc::fence_after_thread_sync();
        tc::tmem_ld_32x32b_x32(o_addr, o0);
        tc::tmem_ld_32x32b_x32(o_addr + 32u, o1);
      }
    }
    if (!ok) {
#pragma unroll
      for (int i = 0; i < 32; ++i) o0[i] = o1[i] = 0.f;
    }
    // full normaliser = this half's share + the other half's (the slot is
    // free: the other half read it before releasing the last PV product)
    sh->xchg[half][r] = l;
    tc::mbar_arrive(&sh->fbar);
    {
      const bool got = tc::mbar_wait(&sh->fbar, 0, abort_flag, status);
      ok = __all_sync(0xffffffffu, got) && ok;
    }
    const float l_row = l + sh->xchg[half ^ 1][r];
    const int h = g * A.G + hh;
    float* orow = A.out + ((size_t)(t0 + node) * A.Hq + h) * 128 + half * 64;
    if (n_chunks == 1) {
      if (row_ok && ok) {
        const float inv = 1.f / l_row;
#pragma unroll
        for (int d = 0; d < 32; d += 4) {
          *reinterpret_cast<float4*>(orow + d) =
              make_float4(o0[d] * inv, o0[d + 1] * inv, o0[d + 2] * inv, o0[d + 3] * inv);
          *reinterpret_cast<float4*>(orow + 32 + d) =
              make_float4(o1[d] * inv, o1[d + 1] * inv, o1[d + 2] * inv, o1[d + 3] * inv);
        }
      }
    } else {
      float* po = A.part_o + ((size_t)item_id * 128 + r) * 128 + half * 64;
      if (half == 0) A.part_ml[(size_t)item_id * 128 + r] = make_float2(m, l_row);
#pragma unroll
      for (int d = 0; d < 32; d += 4) {
        *reinterpret_cast<float4*>(po + d) = make_float4(o0[d], o0[d + 1], o0[d + 2], o0[d + 3]);
        *reinterpret_cast<float4*>(po + 32 + d) =
            make_float4(o1[d], o1[d + 1], o1[d + 2], o1[d + 3]);
      }
      __threadfence();
      tc::mbar_arrive(&sh->tbar0);
      if (threadIdx.x == 64) {
        // every row thread's partial is written: take the ticket
        int never = 0;
        sh->is_last = 0;
        if (tc::mbar_wait(&sh->tbar0, 0, abort_flag, status)) {
          const int prev = atomicAdd(&A.counters[tile_id], 1);
          sh->is_last = (prev == n_chunks - 1);
          if (sh->is_last) A.counters[tile_id] = 0;
        }
        (void)never;
        tc::mbar_arrive(&sh->tbar1);
      }
      const bool got_t = tc::mbar_wait(&sh->tbar1, 0, abort_flag, status);
      if (got_t && sh->is_last && row_ok) {
        __threadfence();
        float M = -INFINITY;
        for (int cc = 0; cc < n_chunks; ++cc)
          M = fmaxf(M, __ldcg(&A.part_ml[((size_t)(tile_id * A.NC + cc)) * 128 + r]).x);
        float Lsum = 0.f;
#pragma unroll
        for (int d = 0; d < 32; ++d) o0[d] = o1[d] = 0.f;
        for (int cc = 0; cc < n_chunks; ++cc) {
          const size_t it = (size_t)(tile_id * A.NC + cc);
          const float2 ml = __ldcg(&A.part_ml[it * 128 + r]);
          const float wgt = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
          Lsum += ml.y * wgt;
          const float4* src =
              reinterpret_cast<const float4*>(A.part_o + (it * 128 + r) * 128 + half * 64);
#pragma unroll
          for (int d = 0; d < 8; ++d) {
            const float4 x = __ldcg(src + d);
            o0[4 * d] = fmaf(x.x, wgt, o0[4 * d]);
            o0[4 * d + 1] = fmaf(x.y, wgt, o0[4 * d + 1]);
            o0[4 * d + 2] = fmaf(x.z, wgt, o0[4 * d + 2]);
            o0[4 * d + 3] = fmaf(x.w, wgt, o0[4 * d + 3]);
            const float4 y = __ldcg(src + 8 + d);
            o1[4 * d] = fmaf(y.x, wgt, o1[4 * d]);
            o1[4 * d + 1] = fmaf(y.y, wgt, o1[4 * d + 1]);
            o1[4 * d + 2] = fmaf(y.z, wgt, o1[4 * d + 2]);
            o1[4 * d + 3] = fmaf(y.w, wgt, o1[4 * d + 3]);
          }
        }
        const float inv = 1.f / Lsum;
#pragma unroll
        for (int d = 0; d < 32; d += 4) {
          *reinterpret_cast<float4*>(orow + d) =
              make_float4(o0[d] * inv, o0[d + 1] * inv, o0[d + 2] * inv, o0[d + 3] * inv);
          *reinterpret_cast<float4*>(orow + 32 + d) =
              make_float4(o1[d] * inv, o1[d + 1] * inv, o1[d + 2] * inv, o1[d + 3] * inv);
        }
      }
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

bool tc_shape_ok(eagle_dtype dtype, int Hq, int Hkv, int D) {
  if (dtype != EAGLE_BF16 || D != 128) return false;
  const int G = Hq / Hkv;
  return G >= 1 && G <= 128 && (128 % G) == 0;
}

}  // namespace

// Scratch of the tensor-core path (split-K partials and merge tickets); the
// CUDA-core path needs none.  Depends on shapes only, not on the device.
extern "C" size_t eagle_tree_attn_workspace_bytes(int B, int T, int Hq, int Hkv, int D,
                                                  int max_nodes, int max_kv) {
  (void)T;
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || max_nodes < 1 || max_kv < 0) return 0;
  if (!tc_shape_ok(EAGLE_BF16, Hq, Hkv, D)) return 0;
  return att_plan(B, Hq, Hkv, max_nodes, max_kv).total;
}

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
  cudaStream_t s = (cudaStream_t)stream;
  const uintptr_t align = (uintptr_t)d_q | (uintptr_t)d_k_tree | (uintptr_t)d_v_tree |
                          (uintptr_t)d_k_cache | (uintptr_t)d_v_cache | (uintptr_t)d_out;
  if (tc_shape_ok(dtype, Hq, Hkv, D) && (align & 15) == 0) {
    const AttPlan P = att_plan(B, Hq, Hkv, max_nodes, max_kv);
    EAGLE_HOST_CHECK(d_ws && ws_bytes >= P.total, EAGLE_ERR_WORKSPACE);
    EAGLE_HOST_CHECK(((uintptr_t)d_ws & 255) == 0, EAGLE_ERR_INVALID_ARG);
    CUtensorMap mq, mkc, mvc, mkt, mvt;
    const void* kc = (kv_rows > 0) ? d_k_cache : d_k_tree;   // never read when empty
    const void* vc = (kv_rows > 0) ? d_v_cache : d_v_tree;
    const int rows_c = (kv_rows > 0) ? kv_rows : T;
    if (!make_map_3d(&mq, d_q, T, Hq, P.G, 128 / P.G) ||
        !make_map_3d(&mkc, kc, rows_c, Hkv, 1, kKeyBlk) ||
        !make_map_3d(&mvc, vc, rows_c, Hkv, 1, kKeyBlk) ||
        !make_map_3d(&mkt, d_k_tree, T, Hkv, 1, kKeyBlk) ||
        !make_map_3d(&mvt, d_v_tree, T, Hkv, 1, kKeyBlk))
      return EAGLE_ERR_CUDA;
    static bool attr = false;
    if (!attr) {
      if (cudaFuncSetAttribute(tree_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kAttSmem) != cudaSuccess)
        return EAGLE_ERR_CUDA;
      attr = true;
    }
    char* ws = static_cast<char*>(d_ws);
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
    A.kv_off = d_kv_off;
    A.tree_off = d_tree_off;
    A.parent = d_parent;
    A.out = d_out;
    A.counters = reinterpret_cast<int*>(ws);
    A.part_ml = reinterpret_cast<float2*>(ws + P.off_ml);
    A.part_o = reinterpret_cast<float*>(ws + P.off_o);
    A.status = d_status;
    if (cudaMemsetAsync(ws, 0, (size_t)B * Hkv * P.MT * sizeof(int), s) != cudaSuccess)
      return EAGLE_ERR_CUDA;
    const int grid = B * Hkv * P.NC * P.MT;
    return launch_status(launch_pdl(tree_attn_tc_kernel, dim3(grid), dim3(kAttThreads), kAttSmem,
                                    s, mq, mkc, mvc, mkt, mvt, A));
  }
  if (dtype == EAGLE_BF16)
    return launch_warp<__nv_bfloat16>(D, B, T, Hq, Hkv, scale, max_nodes, max_kv, d_q, d_k_tree,
                                      d_v_tree, d_k_cache, d_v_cache, d_kv_off, d_tree_off,
                                      d_parent, d_out, d_status, s);
  return launch_warp<float>(D, B, T, Hq, Hkv, scale, max_nodes, max_kv, d_q, d_k_tree, d_v_tree,
                            d_k_cache, d_v_cache, d_kv_off, d_tree_off, d_parent, d_out, d_status,
                            s);
}
