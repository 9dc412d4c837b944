// EAGLE-2 dynamic draft tree: expand (per-node top-k, cumulative scores,
// beam frontier) and finalize (global top-budget rerank).
// [EAGLE-2] §2 "EAGLE-2 的核心創新：動態草稿樹" items 1-3 (page title in
// include/eagle.h): confidence per draft node, adaptive expansion, greedy
// selection under a fixed draft-token budget.  A node's value is its
// cumulative draft log-prob.
//
// Two launches per level.  The level's draft rows (the only large data:
// F x V fp32) are cut into chunks spread over the whole GPU; each CTA stages
// its chunk in shared memory and writes the chunk's top-k list.  Then one
// CTA per sequence merges every row's chunk lists (one warp per row, many
// loads in flight) and builds the children and the next frontier.  The
// finalize is one CTA per sequence working in shared memory.  Selection keys
// are 64-bit integers (ordered value bits | inverted index), so every tie
// rule is a plain max, and a warp keeps its running top-k as a sorted list
// across its lanes.
#include <algorithm>

#include "common.cuh"

using namespace eagle;

namespace {

constexpr int kExpandThreads = 256;
constexpr int kChunkMax = 8192;     // floats staged per CTA
constexpr int kFinalThreads = 1024;
constexpr int kMaxChunks = 64;      // chunks per row (V <= 64 * 8192)

struct PoolLayout {
  int P;         // candidate capacity per sequence
  int rows_max;  // B * k
  int S0, S1;    // chunks per row at level 0 / later levels
  size_t off_count, off_frontier, off_token, off_parent, off_depth, off_prow, off_score,
      off_partial, total;
};

int chunks_for(int rows, int V) {
  int s = (304 + rows - 1) / rows;                   // ~2 CTAs per SM in total
  s = std::min(s, kMaxChunks);                       // row merge fits in smem
  s = std::min(s, std::max(1, V / 512));             // chunks of >= 512 tokens
  s = std::max(s, (V + kChunkMax - 1) / kChunkMax);  // chunk fits in smem
  return std::max(s, 1);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

PoolLayout pool_layout(int B, int k, int depth, int V) {
  PoolLayout L;
  L.P = k + (depth - 1) * k * k;
  L.rows_max = B * k;
  L.S0 = chunks_for(B, V);
  L.S1 = chunks_for(B * k, V);
  const size_t parts = std::max((size_t)B * L.S0, (size_t)B * k * L.S1) * k;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.off_count = take((size_t)B * 4);
  L.off_frontier = take((size_t)B * k * 4);
  L.off_token = take((size_t)B * L.P * 4);
  L.off_parent = take((size_t)B * L.P * 4);
  L.off_depth = take((size_t)B * L.P * 4);
  L.off_prow = take((size_t)B * L.P * 4);
  L.off_score = take((size_t)B * L.P * 4);
  L.off_partial = take(parts * 8);
  L.total = o;
  return L;
}

struct PoolPtrs {
  int* count;
  int* frontier;
  int* token;
  int* parent;
  int* depth;
  int* prow;
  float* score;
  unsigned long long* partial;
};

PoolPtrs pool_ptrs(void* base, const PoolLayout& L) {
  char* c = static_cast<char*>(base);
  PoolPtrs p;
  p.count = reinterpret_cast<int*>(c + L.off_count);
  p.frontier = reinterpret_cast<int*>(c + L.off_frontier);
  p.token = reinterpret_cast<int*>(c + L.off_token);
  p.parent = reinterpret_cast<int*>(c + L.off_parent);
  p.depth = reinterpret_cast<int*>(c + L.off_depth);
  p.prow = reinterpret_cast<int*>(c + L.off_prow);
  p.score = reinterpret_cast<float*>(c + L.off_score);
  p.partial = reinterpret_cast<unsigned long long*>(c + L.off_partial);
  return p;
}

struct LevelParams {
  int B, V, k, F, R, S, level, P;
  const float* logp;
  PoolPtrs pool;
  int* status;
};

__device__ __forceinline__ unsigned long long shfl_u64(unsigned long long v, int src) {
  return __shfl_sync(0xffffffffu, v, src);
}
__device__ __forceinline__ unsigned long long shfl_up_u64(unsigned long long v, int d) {
  return __shfl_up_sync(0xffffffffu, v, d);
}

// Warp-wide running top-k: lane j holds the j-th largest key seen (0 =
// empty), `thr` the k-th (0 while fewer than k).  Feeds 32 keys (one per
// lane) at a time.
struct WarpTopk {
  unsigned long long mine = 0ull, thr = 0ull;
  __device__ __forceinline__ void feed(unsigned long long key, int k) {
    const int lane = threadIdx.x & 31;
    unsigned bal = __ballot_sync(0xffffffffu, key > thr);
    while (bal) {
      const int src = __ffs(bal) - 1;
      bal &= bal - 1;
      const unsigned long long cand = shfl_u64(key, src);
      if (cand <= thr) continue;  // uniform: the threshold may have risen
      const int pos = __popc(__ballot_sync(0xffffffffu, lane < k && mine > cand));
      const unsigned long long up = shfl_up_u64(mine, 1);
      if (lane < k) {
        if (lane > pos) mine = up;
        else if (lane == pos) mine = cand;
      }
      thr = shfl_u64(mine, k - 1);
    }
  }
};

// Level kernel 1: top-k of one chunk of one draft row per CTA.
__global__ void __launch_bounds__(kExpandThreads) expand_chunk_kernel(const LevelParams A) {
  __shared__ __align__(16) float s_val[kChunkMax];
  __shared__ unsigned long long s_wtop[(kExpandThreads / 32) * EAGLE_MAX_TOPK];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int row = blockIdx.x / A.S;       // global frontier row: b * F + f
  const int chunk = blockIdx.x % A.S;
  const int b = row / A.F;
  const int f = row % A.F;
  const int local_row = (A.level == 0) ? 0 : 1 + (A.level - 1) * A.k + f;
  const float* src = A.logp + ((size_t)b * A.R + local_row) * A.V;
  const int csize = (A.V + A.S - 1) / A.S;
  const int c0 = min(A.V, chunk * csize), c1 = min(A.V, c0 + csize);
  const int n = c1 - c0;
  const int k = A.k;
  // stage the chunk (vectorised when the row and the chunk are 16-byte aligned)
  int bad = 0;
  if (((A.V | csize) & 3) == 0) {
    const float4* s4 = reinterpret_cast<const float4*>(src + c0);
    for (int i = tid; i < (n >> 2); i += blockDim.x) {
      const float4 x = __ldg(s4 + i);
      reinterpret_cast<float4*>(s_val)[i] = x;
      bad |= !(isfinite(x.x) && isfinite(x.y) && isfinite(x.z) && isfinite(x.w));
    }
  } else {
    for (int i = tid; i < n; i += blockDim.x) {
      const float x = __ldg(src + c0 + i);
      s_val[i] = x;
      bad |= !isfinite(x);
    }
  }
  if (__syncthreads_or(bad) && tid == 0) fail(A.status, EAGLE_ERR_NUMERIC);
  // each warp a contiguous slice, then warp 0 merges the warps' lists
  const int per = (n + nw - 1) / nw;
  const int lo = min(n, warp * per), cnt = min(n, lo + per) - lo;
  WarpTopk wt;
  for (int base = 0; base < cnt; base += 32) {
    const int i = base + lane;
    wt.feed(i < cnt ? desc_key(s_val[lo + i], (uint32_t)(c0 + lo + i)) : 0ull, k);
  }
  if (lane < k) s_wtop[warp * k + lane] = wt.mine;
  __syncthreads();
  if (warp == 0) {
    WarpTopk m;
    for (int base = 0; base < nw * k; base += 32) {
      const int i = base + lane;
      m.feed(i < nw * k ? s_wtop[i] : 0ull, k);
    }
    if (lane < k) A.pool.partial[((size_t)row * A.S + chunk) * k + lane] = m.mine;
  }
}

// Level kernel 2 (one CTA per sequence): merge every row's chunk lists
// (one warp per row) and build the children and the next frontier.
constexpr int kMergeThreads = 512;
constexpr int kMergeBatch = 8;          // 32-key batches loaded before use

__global__ void __launch_bounds__(kMergeThreads) expand_merge_kernel(const LevelParams A) {
  __shared__ unsigned long long s_row[EAGLE_MAX_TOPK][EAGLE_MAX_TOPK];
  __shared__ unsigned long long s_cand[EAGLE_MAX_TOPK * EAGLE_MAX_TOPK];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int b = blockIdx.x;
  const int k = A.k, F = A.F;
  const int n = A.S * k;                  // candidates per row
  for (int f = warp; f < F; f += nw) {
    const unsigned long long* src = A.pool.partial + (size_t)(b * F + f) * n;
    WarpTopk wt;
    for (int base0 = 0; base0 < n; base0 += 32 * kMergeBatch) {
      unsigned long long buf[kMergeBatch];
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        const int i = base0 + j * 32 + lane;
        buf[j] = (i < n) ? __ldcg(src + i) : 0ull;
      }
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) wt.feed(buf[j], k);
    }
    if (lane < k) s_row[f][lane] = wt.mine;
  }
  __syncthreads();
  const int nc = F * k;  // children in creation order (f-major, rank-minor)
  const int base = A.pool.count[b];
  int* tok = A.pool.token + (size_t)b * A.P;
  int* par = A.pool.parent + (size_t)b * A.P;
  int* dep = A.pool.depth + (size_t)b * A.P;
  int* prw = A.pool.prow + (size_t)b * A.P;
  float* sco = A.pool.score + (size_t)b * A.P;
  int* front = A.pool.frontier + (size_t)b * k;
  for (int c = tid; c < nc; c += blockDim.x) {
    const int ff = c / k, rr = c % k;
    const unsigned long long key = s_row[ff][rr];
    const int pidx = (A.level == 0) ? -1 : front[ff];
    const float pscore = (A.level == 0) ? 0.f : sco[pidx];
    const float sc = __fadd_rn(pscore, key_value(key));
    const int at = base + c;
    tok[at] = (int)key_index(key);
    par[at] = pidx;
    dep[at] = A.level + 1;
    prw[at] = (A.level == 0) ? 0 : 1 + (A.level - 1) * k + ff;
    sco[at] = sc;
    s_cand[c] = desc_key(sc, (uint32_t)c);
  }
  __syncthreads();
  // next frontier: rank of every child by (score desc, creation order)
  for (int c = tid; c < nc; c += blockDim.x) {
    const unsigned long long me = s_cand[c];
    int rank = 0;
#pragma unroll 8
    for (int j = 0; j < nc; ++j) rank += (s_cand[j] > me);
    if (rank < k) front[rank] = base + c;
  }
  if (tid == 0) A.pool.count[b] = base + nc;
}

struct FinalParams {
  int B, k, R, P;
  const int* budget;
  const int* root_token;
  PoolPtrs pool;
  int* tree_off;
  int* parent;
  int* tokens;
  int* node_depth;
  float* score;
  int* p_row_of_node;
  int* status;
};

// Finalize, one CTA per sequence: rank every pool entry by (score desc,
// creation order), keep the top `budget`, number the kept nodes by (depth,
// score desc, creation order) and write the tree.
__global__ void __launch_bounds__(kFinalThreads) expand_finalize_kernel(const FinalParams A) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned long long* s_key = reinterpret_cast<unsigned long long*>(smem_raw);  // [P]
  int* s_list = reinterpret_cast<int*>(s_key + A.P);                            // [P]
  int* s_num = s_list + A.P;                                                    // [P]
  int* s_node = s_num + A.P;                                                    // [P]
  __shared__ int s_nsel;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int n = A.pool.count[b];
  const int bud = A.budget[b];
  const int keep = min(max(bud, 0), n);
  const float* sco = A.pool.score + (size_t)b * A.P;
  if (tid == 0) {
    s_nsel = 0;
    if (bud < 0) fail(A.status, EAGLE_ERR_INVALID_ARG);
  }
  for (int i = tid; i < n; i += blockDim.x) {
    s_key[i] = desc_key(sco[i], (uint32_t)i);
    s_node[i] = -1;
  }
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) {
    const unsigned long long me = s_key[i];
    int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
    int j = 0;
    for (; j + 4 <= n; j += 4) {
      r0 += (s_key[j] > me);
      r1 += (s_key[j + 1] > me);
      r2 += (s_key[j + 2] > me);
      r3 += (s_key[j + 3] > me);
    }
    for (; j < n; ++j) r0 += (s_key[j] > me);
    if (r0 + r1 + r2 + r3 < keep) s_list[atomicAdd(&s_nsel, 1)] = i;
  }
  __syncthreads();
  const int ns = s_nsel;
  const int* tok = A.pool.token + (size_t)b * A.P;
  const int* par = A.pool.parent + (size_t)b * A.P;
  const int* dep = A.pool.depth + (size_t)b * A.P;
  const int* prw = A.pool.prow + (size_t)b * A.P;
  int off = 0;
  for (int j = 0; j < b; ++j) off += min(max(A.budget[j], 0), A.pool.count[j]) + 1;
  // node number of every kept entry: 1 + rank by (depth, score desc, creation)
  for (int a = tid; a < ns; a += blockDim.x) {
    const int ia = s_list[a];
    const int da = dep[ia];
    const unsigned long long ka = s_key[ia];
    int rank = 0;
    for (int c = 0; c < ns; ++c) {
      const int ic = s_list[c];
      rank += (dep[ic] < da) || (dep[ic] == da && s_key[ic] > ka);
    }
    s_num[a] = 1 + rank;
    s_node[ia] = 1 + rank;
  }
  __syncthreads();
  for (int a = tid; a < ns; a += blockDim.x) {
    const int ia = s_list[a];
    const int pp = par[ia];
    const int pnode = (pp < 0) ? 0 : s_node[pp];
    if (pnode < 0) fail(A.status, EAGLE_ERR_INVALID_TREE);  // not parent-closed
    const int at = off + s_num[a];
    A.parent[at] = pnode;
    A.tokens[at] = tok[ia];
    A.node_depth[at] = dep[ia];
    A.score[at] = sco[ia];
    A.p_row_of_node[at] = b * A.R + prw[ia];
  }
  if (tid == 0) {
    A.tree_off[b] = off;
    if (b == A.B - 1) A.tree_off[A.B] = off + ns + 1;
    A.parent[off] = -1;
    A.tokens[off] = A.root_token ? A.root_token[b] : -1;
    A.node_depth[off] = 0;
    A.score[off] = 0.f;
    A.p_row_of_node[off] = -1;
  }
}

}  // namespace

extern "C" size_t eagle_draft_pool_bytes(int B, int k, int depth, int V) {
  if (B < 1 || k < 1 || k > EAGLE_MAX_TOPK || depth < 1 || depth > EAGLE_MAX_DEPTH || V < k ||
      V > kMaxChunks * kChunkMax)
    return 0;
  return pool_layout(B, k, depth, V).total;
}

extern "C" eagle_status eagle_draft_expand(int B, int V, int k, int depth, int level,
                                           int finalize, const float* d_draft_logp,
                                           const int32_t* d_budget, const int32_t* d_root_token,
                                           void* d_pool, size_t pool_bytes, int32_t* d_tree_off,
                                           int32_t* d_parent, int32_t* d_tokens,
                                           int32_t* d_node_depth, float* d_score,
                                           int32_t* d_p_row_of_node, int* d_status,
                                           eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 1 && V >= 1, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(k >= 1 && k <= EAGLE_MAX_TOPK && k <= V, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(depth >= 1 && depth <= EAGLE_MAX_DEPTH, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(V <= kMaxChunks * kChunkMax, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(d_pool && d_status, EAGLE_ERR_INVALID_ARG);
  const PoolLayout L = pool_layout(B, k, depth, V);
  EAGLE_HOST_CHECK(pool_bytes >= L.total, EAGLE_ERR_WORKSPACE);
  EAGLE_HOST_CHECK(((uintptr_t)d_pool & 255) == 0, EAGLE_ERR_INVALID_ARG);
  const PoolPtrs pp = pool_ptrs(d_pool, L);
  cudaStream_t s = (cudaStream_t)stream;
  const int R = 1 + (depth - 1) * k;
  if (!finalize) {
    EAGLE_HOST_CHECK(level >= 0 && level < depth, EAGLE_ERR_INVALID_ARG);
    EAGLE_HOST_CHECK(d_draft_logp, EAGLE_ERR_INVALID_ARG);
    if (level == 0) {
      // fresh tree: zero the pool fill counts
      cudaError_t e = cudaMemsetAsync(static_cast<char*>(d_pool), 0, L.off_frontier, s);
      if (e != cudaSuccess) return EAGLE_ERR_CUDA;
    }
    LevelParams A;
    A.B = B;
    A.V = V;
    A.k = k;
    A.F = (level == 0) ? 1 : k;
    A.R = R;
    A.S = (level == 0) ? L.S0 : L.S1;
    A.level = level;
    A.P = L.P;
    A.logp = d_draft_logp;
    A.pool = pp;
    A.status = d_status;
    expand_chunk_kernel<<<B * A.F * A.S, kExpandThreads, 0, s>>>(A);
    if (cudaGetLastError() != cudaSuccess) return EAGLE_ERR_CUDA;
    expand_merge_kernel<<<B, kMergeThreads, 0, s>>>(A);
    return launch_status(cudaGetLastError());
  }
  EAGLE_HOST_CHECK(d_budget && d_tree_off && d_parent && d_tokens && d_node_depth && d_score &&
                       d_p_row_of_node,
                   EAGLE_ERR_INVALID_ARG);
  FinalParams F;
  F.B = B;
  F.k = k;
  F.R = R;
  F.P = L.P;
  F.budget = d_budget;
  F.root_token = d_root_token;
  F.pool = pp;
  F.tree_off = d_tree_off;
  F.parent = d_parent;
  F.tokens = d_tokens;
  F.node_depth = d_node_depth;
  F.score = d_score;
  F.p_row_of_node = d_p_row_of_node;
  F.status = d_status;
  const size_t smem = (size_t)L.P * (8 + 4 + 4 + 4);
  EAGLE_HOST_CHECK(smem <= 200 * 1024, EAGLE_ERR_UNSUPPORTED);
  if (smem > 40 * 1024) {
    cudaFuncSetAttribute(expand_finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
  }
  expand_finalize_kernel<<<B, kFinalThreads, smem, s>>>(F);
  return launch_status(cudaGetLastError());
}
