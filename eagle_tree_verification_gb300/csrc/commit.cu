// Commit of a verify step's accepted tokens to a paged KV cache.
// [EAGLE] speculative-sampling paragraph (page title in include/eagle.h):
// alpha accepted drafts turn into alpha + 1 tokens; the tree's root (the
// last token of the previous step) and the alpha accepted nodes join the
// context, so their keys and values -- computed by the verify pass, already
// rotated to their positions -- are appended to the sequence's cache.
//
// One CTA per sequence: it reads the sequence's length once, copies the
// root-to-last-accepted path's K and V rows into the pages at positions
// kv_len .. kv_len + alpha (16-byte vectors), and only then, after a CTA
// barrier, advances kv_len, so no other reader of the length is involved.
#include "common.cuh"

using namespace eagle;

namespace {

constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads)
kv_commit_kernel(int row_bytes, int page_size, int n_pages, int max_pages, int max_depth,
                 const int* __restrict__ tree_off, const int* __restrict__ accept_len,
                 const int* __restrict__ accepted_nodes, const unsigned char* __restrict__ k_tree,
                 const unsigned char* __restrict__ v_tree, unsigned char* __restrict__ k_pages,
                 unsigned char* __restrict__ v_pages, const int* __restrict__ block_table,
                 int* __restrict__ kv_len, int* status) {
  pdl_begin();
  __shared__ int s_ok;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int t0 = tree_off[b], n = tree_off[b + 1] - t0;
  const int L = kv_len[b];
  const int alpha = accept_len[b];
  const int W = max_depth + 1;
  if (tid == 0) {
    bool ok = alpha >= 0 && alpha <= max_depth && L >= 0 &&
              (long long)L + alpha + 1 <= (long long)max_pages * page_size;
    for (int i = 0; ok && i <= alpha; ++i) {
      const int node = accepted_nodes[(size_t)b * W + i];
      const int pos = L + i;
      const int page = block_table[(size_t)b * max_pages + pos / page_size];
      ok = node >= 0 && node < n && page >= 0 && page < n_pages;
    }
    s_ok = ok;
    if (!ok) fail(status, EAGLE_ERR_INVALID_ARG);
  }
  __syncthreads();
  if (!s_ok) return;
  const int vec_per_row = row_bytes / 16;
  const int total = (alpha + 1) * vec_per_row;
  for (int e = tid; e < total; e += kCommitThreads) {
    const int i = e / vec_per_row, c = e % vec_per_row;
    const int node = accepted_nodes[(size_t)b * W + i];
    const int pos = L + i;
    const int page = block_table[(size_t)b * max_pages + pos / page_size];
    const size_t dst = ((size_t)page * page_size + pos % page_size) * row_bytes + (size_t)c * 16;
    const size_t src = (size_t)(t0 + node) * row_bytes + (size_t)c * 16;
    *reinterpret_cast<uint4*>(k_pages + dst) = *reinterpret_cast<const uint4*>(k_tree + src);
    *reinterpret_cast<uint4*>(v_pages + dst) = *reinterpret_cast<const uint4*>(v_tree + src);
  }
  __syncthreads();
  if (tid == 0) kv_len[b] = L + alpha + 1;
}

}  // namespace

extern "C" eagle_status eagle_kv_commit_paged(eagle_dtype dtype, int B, int Hkv, int D,
                                              int page_size, int n_pages, int max_pages,
                                              int max_depth, const int32_t* d_tree_off,
                                              const int32_t* d_accept_len,
                                              const int32_t* d_accepted_nodes,
                                              const void* d_k_tree, const void* d_v_tree,
                                              void* d_k_pages, void* d_v_pages,
                                              const int32_t* d_block_table, int32_t* d_kv_len,
                                              int* d_status, eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 0 && Hkv >= 1 && D >= 1 && max_depth >= 0, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(dtype == EAGLE_F32 || dtype == EAGLE_BF16, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(page_size >= 1 && n_pages >= 1 && max_pages >= 1, EAGLE_ERR_INVALID_ARG);
  const int row_bytes = Hkv * D * (dtype == EAGLE_BF16 ? 2 : 4);
  EAGLE_HOST_CHECK(row_bytes % 16 == 0, EAGLE_ERR_UNSUPPORTED);
  if (B == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_tree_off && d_accept_len && d_accepted_nodes && d_k_tree && d_v_tree &&
                       d_k_pages && d_v_pages && d_block_table && d_kv_len && d_status,
                   EAGLE_ERR_INVALID_ARG);
  const uintptr_t al = (uintptr_t)d_k_tree | (uintptr_t)d_v_tree | (uintptr_t)d_k_pages |
                       (uintptr_t)d_v_pages;
  EAGLE_HOST_CHECK((al & 15) == 0, EAGLE_ERR_INVALID_ARG);
  return launch_status(launch_pdl(
      kv_commit_kernel, dim3(B), dim3(kCommitThreads), 0, (cudaStream_t)stream, row_bytes,
      page_size, n_pages, max_pages, max_depth, d_tree_off, d_accept_len, d_accepted_nodes,
      static_cast<const unsigned char*>(d_k_tree), static_cast<const unsigned char*>(d_v_tree),
      static_cast<unsigned char*>(d_k_pages), static_cast<unsigned char*>(d_v_pages),
      d_block_table, d_kv_len, d_status));
}
