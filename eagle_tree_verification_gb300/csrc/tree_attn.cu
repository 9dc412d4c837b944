// Tree attention of the tree-verify step.
// [S4000] "EAGLE的创新点" item 2 and [EAGLE] workflow paragraph (page titles
// in include/eagle.h): one forward pass verifies every path of the draft
// tree, because node i attends to the cached context and to exactly its own
// ancestors and itself.
//
// This file holds the reference-grade CUDA-core kernel: one warp per (node,
// query head), an online softmax over [cache | root..node path].  The
// ancestor set is read from parent[] on the fly, never stored as a mask.
#include <math.h>

#include "common.cuh"

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
  if (D == 64)
    tree_attn_warp_kernel<TIn, 64><<<grid, kWarpsPerBlock * 32, 0, s>>>(
        B, T, Hq, Hkv, scale, max_nodes, max_kv, Q, KT, VT, KC, VC, kv_off, tree_off, parent, out,
        status);
  else
    tree_attn_warp_kernel<TIn, 128><<<grid, kWarpsPerBlock * 32, 0, s>>>(
        B, T, Hq, Hkv, scale, max_nodes, max_kv, Q, KT, VT, KC, VC, kv_off, tree_off, parent, out,
        status);
  return launch_status(cudaGetLastError());
}

}  // namespace

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

extern "C" eagle_status eagle_tree_attn(eagle_dtype dtype, int B, int T, int Hq, int Hkv, int D,
                                        float scale, int max_nodes, int max_kv, const void* d_q,
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
  (void)d_ws;
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype == EAGLE_BF16)
    return launch_warp<__nv_bfloat16>(D, B, T, Hq, Hkv, scale, max_nodes, max_kv, d_q, d_k_tree,
                                      d_v_tree, d_k_cache, d_v_cache, d_kv_off, d_tree_off,
                                      d_parent, d_out, d_status, s);
  return launch_warp<float>(D, B, T, Hq, Hkv, scale, max_nodes, max_kv, d_q, d_k_tree, d_v_tree,
                            d_k_cache, d_v_cache, d_kv_off, d_tree_off, d_parent, d_out, d_status,
                            s);
}
