// EAGLE-1 static draft tree.
// [EAGLE-2] §2 "EAGLE-2 的核心創新：動態草稿樹" (EAGLE-1's fixed top-k tree, the
// structure the dynamic tree replaces) and [S4000] "EAGLE的创新点" item 1 (the
// draft keeps the top tokens at every step); page titles in include/eagle.h.
//
// The tree's shape is a template fixed ahead of time: template node i is the
// tmpl_rank[i]-th most probable token (log-prob descending, token ascending)
// of the draft row its parent was expanded with.  Two kernels:
//   static_rank_kernel    one CTA per (template node, sequence); a node with
//                         children selects the top max-rank tokens of its
//                         draft row exactly (64-bit keys: ordered value bits,
//                         inverted index, so every tie rule is an integer
//                         comparison) and writes its children's tokens and
//                         own log-probs.
//   static_finish_kernel  one CTA per sequence: depths, cumulative scores in
//                         root-to-leaf order (the dynamic tree's definition,
//                         fp32(parent score + logp)), parents and offsets.
#include <math.h>

#include "common.cuh"

using namespace eagle;

namespace {

constexpr int kStThreads = 512;
constexpr int kFinThreads = EAGLE_MAX_TREE_NODES;

struct StaticParams {
  int B, V, N, R, K;               // K: ranks 0 .. K-1 may appear
  const int* tmpl_parent;
  const int* tmpl_rank;
  const int* tmpl_row;
  const float* logp;               // [B, R, V]
  const int* root_token;
  int* tree_off;
  int* parent;
  int* tokens;
  int* depth;
  float* score;
  int* p_row;
  int* status;
};

// Candidate buffer of one CTA: at most K threads own an element at or above
// the bound (their maxima are the K largest), each at most ceil(V / threads)
// elements.
inline size_t rank_smem_bytes(int V, int K) {
  return (size_t)K * ((V + kStThreads - 1) / kStThreads) * sizeof(unsigned long long);
}

__global__ void __launch_bounds__(kStThreads)
static_rank_kernel(const StaticParams P) {
  pdl_begin();
  extern __shared__ unsigned long long s_cand[];
  __shared__ unsigned long long s_max[kStThreads];
  __shared__ unsigned long long s_top[EAGLE_MAX_TOPK];
  __shared__ unsigned long long s_bound;
  __shared__ int s_k, s_n, s_bad;
  const int j = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_k = 0;
    s_n = 0;
    s_bad = 0;
  }
  __syncthreads();
  // the template must be topological (checked by every CTA, so none reads
  // a bad parent); children of j: the largest rank among them
  for (int i = tid; i < P.N; i += kStThreads) {
    const int p = P.tmpl_parent[i];
    if ((i == 0) ? (p != -1) : (p < 0 || p >= i)) atomicOr(&s_bad, 2);
    if (i > 0 && p == j) {
      const int r = P.tmpl_rank[i];
      if (r < 0 || r >= P.K) atomicOr(&s_bad, 1);
      else atomicMax(&s_k, r + 1);
    }
  }
  __syncthreads();
  if (s_bad) {
    // a template error is seen by every CTA and reported once; a bad rank
    // by the CTA of the parent that has it
    if (tid == 0 && b == 0 && (!(s_bad & 2) || j == 0))
      fail(P.status, (s_bad & 2) ? EAGLE_ERR_INVALID_TREE : EAGLE_ERR_INVALID_ARG);
    return;
  }
  const int K = s_k;
  if (K == 0) return;                                  // a leaf
  const int row = P.tmpl_row[j];
  if (row < 0 || row >= P.R) {
    if (tid == 0 && b == 0) fail(P.status, EAGLE_ERR_INVALID_ARG);
    return;
  }
  const float* x = P.logp + ((size_t)b * P.R + row) * P.V;
  // pass 1: every thread's largest key
  unsigned long long best = 0ull;
  bool bad = false;
  for (int i = tid; i < P.V; i += kStThreads) {
    const float v = __ldg(x + i);
    bad |= !isfinite(v);
    const unsigned long long key = desc_key(v, (uint32_t)i);
    best = key > best ? key : best;
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) fail(P.status, EAGLE_ERR_NUMERIC);
    return;
  }
  s_max[tid] = best;
  __syncthreads();
  // the K-th largest thread maximum bounds the K-th largest key from below
  // (the K threads with the largest maxima each hold one key at or above
  // it); keys are distinct, so exactly one thread has rank K-1.  Threads
  // without elements hold 0, below every real key (K <= V).
  int above = 0;
  for (int u = 0; u < kStThreads; ++u) above += (s_max[u] > best);
  if (above == K - 1) s_bound = best;
  __syncthreads();
  const unsigned long long bound = s_bound;
  // pass 2: every key at or above the bound
  if (best >= bound) {
    for (int i = tid; i < P.V; i += kStThreads) {
      const unsigned long long key = desc_key(__ldg(x + i), (uint32_t)i);
      if (key >= bound) s_cand[atomicAdd(&s_n, 1)] = key;
    }
  }
  __syncthreads();
  // rank the candidates: position = number of larger candidates
  const int n = s_n;
  for (int c = tid; c < n; c += kStThreads) {
    const unsigned long long key = s_cand[c];
    int r = 0;
    for (int u = 0; u < n; ++u) r += (s_cand[u] > key);
    if (r < K) s_top[r] = key;
  }
  __syncthreads();
  // the children: token of their rank, own log-prob (made cumulative by
  // the finish kernel), the row they were drafted from
  for (int i = tid; i < P.N; i += kStThreads) {
    if (i > 0 && P.tmpl_parent[i] == j) {
      const int tok = (int)key_index(s_top[P.tmpl_rank[i]]);
      const size_t o = (size_t)b * P.N + i;
      P.tokens[o] = tok;
      P.score[o] = __ldg(x + tok);
      P.p_row[o] = b * P.R + row;
    }
  }
}

__global__ void __launch_bounds__(kFinThreads)
static_finish_kernel(const StaticParams P) {
  pdl_begin();
  __shared__ int s_par[EAGLE_MAX_TREE_NODES];
  __shared__ float s_sc[EAGLE_MAX_TREE_NODES];
  __shared__ int s_bad, s_maxdep;
  const int b = blockIdx.x, i = threadIdx.x;
  const bool live = i < P.N;
  const size_t o = (size_t)b * P.N + i;
  if (i == 0) {
    s_bad = 0;
    s_maxdep = 0;
  }
  int p = -1;
  float own = 0.f;
  if (live) {
    p = P.tmpl_parent[i];
    s_par[i] = p;
    own = (i > 0) ? P.score[o] : 0.f;
  }
  if (live && ((i == 0) ? (p != -1) : (p < 0 || p >= i))) atomicOr(&s_bad, 1);
  __syncthreads();
  if (s_bad) {
    if (i == 0) fail(P.status, EAGLE_ERR_INVALID_TREE);
    return;
  }
  // depth by walking up: every parent precedes its child, so the walk ends
  int d = 0;
  if (live)
    for (int a = i; a > 0; a = s_par[a]) ++d;
  if (live) {
    atomicMax(&s_maxdep, d);
    if (i == 0) s_sc[0] = 0.f;
  }
  __syncthreads();
  // cumulative scores level by level, each the fp32 sum of the parent's
  // final score and the node's own log-prob
  for (int lev = 1; lev <= s_maxdep; ++lev) {
    if (live && d == lev) s_sc[i] = __fadd_rn(s_sc[p], own);
    __syncthreads();
  }
  if (live) {
    P.parent[o] = p;
    P.depth[o] = d;
    P.score[o] = s_sc[i];
    if (i == 0) {
      P.tokens[o] = P.root_token[b];
      P.p_row[o] = -1;
    }
  }
  if (i == 0) {
    P.tree_off[b] = b * P.N;
    if (b == P.B - 1) P.tree_off[P.B] = P.B * P.N;
  }
}

}  // namespace

extern "C" eagle_status eagle_draft_static(int B, int V, int N, int R, int max_rank,
                                           const int32_t* d_tmpl_parent,
                                           const int32_t* d_tmpl_rank,
                                           const int32_t* d_tmpl_row, const float* d_draft_logp,
                                           const int32_t* d_root_token, int32_t* d_tree_off,
                                           int32_t* d_parent, int32_t* d_tokens,
                                           int32_t* d_node_depth, float* d_score,
                                           int32_t* d_p_row_of_node, int* d_status,
                                           eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 0 && V >= 1 && R >= 0, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(N >= 1 && N <= EAGLE_MAX_TREE_NODES, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(max_rank >= 1 && max_rank <= EAGLE_MAX_TOPK && max_rank <= V,
                   EAGLE_ERR_UNSUPPORTED);
  if (B == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_tmpl_parent && d_tmpl_rank && d_tmpl_row && d_root_token && d_tree_off &&
                       d_parent && d_tokens && d_node_depth && d_score && d_p_row_of_node &&
                       d_status,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(N == 1 || (R >= 1 && d_draft_logp), EAGLE_ERR_INVALID_ARG);
  const size_t smem = rank_smem_bytes(V, max_rank);
  EAGLE_HOST_CHECK(smem <= 200 * 1024, EAGLE_ERR_UNSUPPORTED);
  cudaStream_t s = (cudaStream_t)stream;
  StaticParams P;
  P.B = B;
  P.V = V;
  P.N = N;
  P.R = R;
  P.K = max_rank;
  P.tmpl_parent = d_tmpl_parent;
  P.tmpl_rank = d_tmpl_rank;
  P.tmpl_row = d_tmpl_row;
  P.logp = d_draft_logp;
  P.root_token = d_root_token;
  P.tree_off = d_tree_off;
  P.parent = d_parent;
  P.tokens = d_tokens;
  P.depth = d_node_depth;
  P.score = d_score;
  P.p_row = d_p_row_of_node;
  P.status = d_status;
  if (N > 1) {
    static PerDeviceOnce attr_once;
    if (attr_once.run([] {
          return cudaFuncSetAttribute(static_rank_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        }) != cudaSuccess)
      return EAGLE_ERR_CUDA;
    const eagle_status st = launch_status(
        launch_pdl(static_rank_kernel, dim3(N, B), dim3(kStThreads), smem, s, P));
    if (st != EAGLE_OK) return st;
  }
  return launch_status(launch_pdl(static_finish_kernel, dim3(B), dim3(kFinThreads), 0, s, P));
}
