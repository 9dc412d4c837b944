// Glue kernels of the draft -> verify -> accept -> commit loop.
// [EAGLE] workflow paragraph (page title in include/eagle.h): the draft head
// reads the target's features and the embedding of the sampled token, the
// frozen LM head turns its output into the next-token distribution of every
// draft node, the target verifies the tree in one pass, and the accepted
// tokens join the context.  These kernels move data between those steps:
//   draft_rows_kernel  LM-head logits of the draft nodes -> the expand's
//                      log-prob rows and the walk's probability rows;
//   embed_kernel       tree tokens -> the target's input rows (fp32);
//   advance_kernel     after the walk: the next step's root token (the
//                      bonus token) and context feature (the target's
//                      output at the last accepted node).
#include <algorithm>

#include "common.cuh"

using namespace eagle;

namespace {

// Row r of z (sequence b = r / F, frontier rank f = r % F) goes to local
// row 0 (level 0) or 1 + (level-1) k + f of the sequence's R rows.
__global__ void __launch_bounds__(256)
draft_rows_kernel(int V, int F, int level, int k, int R, const float* __restrict__ z,
                  const float* __restrict__ lse, float* __restrict__ logp,
                  float* __restrict__ prob) {
  pdl_begin();
  const int r = blockIdx.y, b = r / F, f = r % F;
  const int local = (level == 0) ? 0 : 1 + (level - 1) * k + f;
  const float l = lse[r];
  const ProbScales sc = prob_scales(1.f, l);
  const float* zr = z + (size_t)r * V;
  const size_t dst = ((size_t)b * R + local) * V;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < V; j += gridDim.x * blockDim.x) {
    const float x = zr[j];
    logp[dst + j] = __fsub_rn(x, l);
    if (prob) prob[dst + j] = prob_from_logit(x, sc);
  }
}

__global__ void __launch_bounds__(256)
embed_kernel(int H, int V, const int* __restrict__ tokens, const __nv_bfloat16* __restrict__ emb,
             float* __restrict__ x, int* status) {
  pdl_begin();
  const int t = blockIdx.x;
  int tok = tokens[t];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) fail(status, EAGLE_ERR_INVALID_ARG);
    tok = 0;
  }
  const __nv_bfloat16* e = emb + (size_t)tok * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x) x[(size_t)t * H + i] = __bfloat162float(e[i]);
}

__global__ void __launch_bounds__(256)
advance_kernel(int H, int max_depth, const int* __restrict__ tree_off,
               const int* __restrict__ accept_len, const int* __restrict__ accepted_nodes,
               const int* __restrict__ out_tokens, const float* __restrict__ resid,
               __nv_bfloat16* __restrict__ f_ctx, int* __restrict__ root_token, int* status) {
  pdl_begin();
  const int b = blockIdx.x;
  const int W = max_depth + 1;
  const int a = accept_len[b];
  const int t0 = tree_off[b], n = tree_off[b + 1] - t0;
  const int last = (a >= 0 && a <= max_depth) ? accepted_nodes[(size_t)b * W + a] : -1;
  if (last < 0 || last >= n) {
    if (threadIdx.x == 0) fail(status, EAGLE_ERR_INVALID_ARG);
    return;
  }
  const float* src = resid + (size_t)(t0 + last) * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    f_ctx[(size_t)b * H + i] = __float2bfloat16_rn(src[i]);
  if (threadIdx.x == 0) root_token[b] = out_tokens[(size_t)b * W + a];
}

}  // namespace

extern "C" eagle_status eagle_draft_rows(int B, int V, int k, int depth, int level,
                                         const float* d_z, const float* d_lse, float* d_logp,
                                         float* d_prob, eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 1 && V >= 1 && k >= 1 && depth >= 1 && level >= 0 && level < depth,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(d_z && d_lse && d_logp, EAGLE_ERR_INVALID_ARG);
  const int F = (level == 0) ? 1 : k;
  const int R = 1 + (depth - 1) * k;
  const int gx = std::min(64, (V + 255) / 256);
  return launch_status(launch_pdl(draft_rows_kernel, dim3(gx, B * F), dim3(256), 0,
                                  (cudaStream_t)stream, V, F, level, k, R, d_z, d_lse, d_logp,
                                  d_prob));
}

extern "C" eagle_status eagle_embed_rows(int T, int H, int V, const int32_t* d_tokens,
                                         const void* d_emb, float* d_x, int* d_status,
                                         eagle_stream_t stream) {
  EAGLE_HOST_CHECK(T >= 0 && H >= 1 && V >= 1, EAGLE_ERR_INVALID_ARG);
  if (T == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_tokens && d_emb && d_x && d_status, EAGLE_ERR_INVALID_ARG);
  return launch_status(launch_pdl(embed_kernel, dim3(T), dim3(256), 0, (cudaStream_t)stream, H,
                                  V, d_tokens, static_cast<const __nv_bfloat16*>(d_emb), d_x,
                                  d_status));
}

extern "C" eagle_status eagle_loop_advance(int B, int H, int max_depth, const int32_t* d_tree_off,
                                           const int32_t* d_accept_len,
                                           const int32_t* d_accepted_nodes,
                                           const int32_t* d_out_tokens, const float* d_resid,
                                           void* d_f_ctx, int32_t* d_root_token, int* d_status,
                                           eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 0 && H >= 1 && max_depth >= 0, EAGLE_ERR_INVALID_ARG);
  if (B == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_tree_off && d_accept_len && d_accepted_nodes && d_out_tokens && d_resid &&
                       d_f_ctx && d_root_token && d_status,
                   EAGLE_ERR_INVALID_ARG);
  return launch_status(launch_pdl(advance_kernel, dim3(B), dim3(256), 0, (cudaStream_t)stream, H,
                                  max_depth, d_tree_off, d_accept_len, d_accepted_nodes,
                                  d_out_tokens, d_resid, static_cast<__nv_bfloat16*>(d_f_ctx),
                                  d_root_token, d_status));
}
