// LM head of the tree-verify step: z = h W^T for every tree node, with the
// softmax statistics (row max, log-sum-exp of z/temperature), argmax (lowest
// index on ties) and the top-2 gap, fused into the GEMM epilogue so that in
// greedy mode no [T, V] tensor is ever written.
// [EAGLE] workflow paragraph (page title in include/eagle.h): the frozen LM
// head gives the next-token distribution of every node.
//
// Two kernels:
//   lmhead_tile_kernel     one CTA per (vocab tile, row tile): fp32-accumulated
//                          GEMM over H, then per-(row, vocab tile) partial
//                          statistics; in PROB mode it also writes z.
//   lmhead_finalize_kernel per (row, vocab chunk): combines the partials of
//                          the row; in PROB mode rewrites z as softmax(z/T).
#include <math.h>

#include "common.cuh"

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
  const int arg_tile = idx / kVT;
  for (int t = tid; t < n_vtiles; t += blockDim.x) {
    const Partial p = pr[t];
    second = fmaxf(second, (t == arg_tile) ? p.second : p.m);
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
    const float lse = s_lse;
    const int c0 = blockIdx.y * kFinChunk, c1 = min(V, c0 + kFinChunk);
    float* row = q + (size_t)r * V;
    for (int v = c0 + tid; v < c1; v += blockDim.x)
      row[v] = expf(__fdiv_rn(row[v], temperature) - lse);
  }
}

}  // namespace

extern "C" size_t eagle_lmhead_workspace_bytes(int T, int V) {
  if (T < 0 || V < 1) return 0;
  return (size_t)T * ((V + kVT - 1) / kVT) * sizeof(Partial);
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
  EAGLE_HOST_CHECK(mode == EAGLE_LMHEAD_GREEDY || mode == EAGLE_LMHEAD_PROB,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(dtype == EAGLE_F32 || dtype == EAGLE_BF16, EAGLE_ERR_UNSUPPORTED);
  if (T == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_h && d_w && d_argmax && d_row_max && d_row_lse && d_top2_gap && d_status,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(mode == EAGLE_LMHEAD_GREEDY || d_q, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(ws_bytes >= eagle_lmhead_workspace_bytes(T, V) && d_ws, EAGLE_ERR_WORKSPACE);
  cudaStream_t s = (cudaStream_t)stream;
  const int n_vtiles = (V + kVT - 1) / kVT;
  Partial* part = static_cast<Partial*>(d_ws);
  float* z = (mode == EAGLE_LMHEAD_PROB) ? d_q : nullptr;
  dim3 grid(n_vtiles, (T + kRT - 1) / kRT);
  if (dtype == EAGLE_BF16)
    lmhead_tile_kernel<__nv_bfloat16><<<grid, kTileThreads, 0, s>>>(
        T, H, V, temperature, static_cast<const __nv_bfloat16*>(d_h),
        static_cast<const __nv_bfloat16*>(d_w), z, part, n_vtiles, d_status);
  else
    lmhead_tile_kernel<float><<<grid, kTileThreads, 0, s>>>(
        T, H, V, temperature, static_cast<const float*>(d_h), static_cast<const float*>(d_w), z,
        part, n_vtiles, d_status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return EAGLE_ERR_CUDA;
  dim3 fgrid(T, z ? (V + kFinChunk - 1) / kFinChunk : 1);
  lmhead_finalize_kernel<<<fgrid, kFinThreads, 0, s>>>(T, V, temperature, part, n_vtiles,
                                                       d_argmax, d_row_max, d_row_lse,
                                                       d_top2_gap, z);
  return launch_status(cudaGetLastError());
}
