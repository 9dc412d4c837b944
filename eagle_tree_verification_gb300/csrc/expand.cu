// EAGLE-2 dynamic draft tree: expand (per-node top-k, cumulative scores,
// beam frontier) and finalize (global top-budget rerank).
// [EAGLE-2] §2 "EAGLE-2 的核心創新：動態草稿樹" items 1-3 (page title in
// include/eagle.h): confidence per draft node, adaptive expansion, greedy
// selection under a fixed draft-token budget.  A node's value is its
// cumulative draft log-prob.
//
// One launch per level, or (eagle_draft_expand_all, every draft row ready
// before the call) every level's chunk lists in one launch and the merges
// and finalize in one more.  The level's draft rows (the only large data:
// F x V fp32) are cut into chunks spread over the whole GPU; each CTA keeps
// its chunk in registers and finds the chunk's exact top-k with a threshold:
// the k-th largest of 32 group maxima is a lower bound of the chunk's k-th
// largest key, so only the few keys above it take part in the exact rank
// count.  The last CTA of a sequence to finish (an atomic ticket) merges the
// rows' chunk lists the same way (one warp per row), then builds the
// children and the next frontier.  A level's rows do not depend on the
// level before it, so past level 0 only that merging CTA waits for the
// previous level: the chunk work overlaps the previous merge.  The finalize
// is one CTA per sequence: a radix select of the budget-th largest score
// key, then the numbering.
// Selection keys are 64-bit integers (ordered value bits | inverted index),
// so every tie rule is a plain integer comparison and all keys are distinct.
#include <algorithm>

#include "common.cuh"
#include "tc.cuh"

using namespace eagle;

namespace {

constexpr int kLvThreads = 512;
constexpr int kLvWarps = kLvThreads / 32;
constexpr int kGroups = 32;            // half-warp groups per CTA (>= any k)
constexpr int kCandCap = kLvThreads;   // chunk candidates held at once
constexpr int kMaxVec = 4;             // float4 loads per thread
constexpr int kOneWave = 304;          // two resident CTAs on each of 152 SMs
constexpr int kRowCap = 128;           // row-merge candidates held at once
constexpr int kMergeRegs = 8;          // chunk-list keys per lane kept in registers
constexpr int kFinalThreads = 1024;
constexpr int kMaxV = 1 << 19;
constexpr size_t kFusedSmemMax = 64 * 1024;  // finalize memory fused into a level
constexpr size_t kFinishSmemMax = 160 * 1024;  // finalize memory beside the merges of all levels
// Bound-raising rounds never exceed (keys / (cap - k)); past these limits a
// selection stops with EAGLE_ERR_TIMEOUT instead of looping.
constexpr int kChunkRounds = 32;   // keys per chunk <= 8192, cap - k >= 480
constexpr int kRowRounds = 128;    // keys per row <= 8192, cap - k >= 96

struct ChunkPlan {
  int vec;  // float4 loads per thread
  int S;    // chunks per row
};

// Smallest chunks that still fit the level in one wave of CTAs (more chunks
// mean more lists to merge); the largest chunks when nothing fits.
ChunkPlan chunk_plan(int rows, int V) {
  ChunkPlan p{1, 1};
  for (p.vec = 1;; p.vec *= 2) {
    p.S = ceil_div(V, (long long)kLvThreads * 4 * p.vec);
    if (p.vec == kMaxVec || (long long)rows * p.S <= kOneWave) break;
  }
  return p;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Tickets come twice, for even and odd levels: a level ranks its chunks
// while the previous one still merges.  Chunk lists likewise, or (all
// levels ranked in one launch) once per level.
struct PoolLayout {
  int P;             // candidate capacity per sequence
  ChunkPlan c0, c1;  // level 0 / later levels
  size_t parts;      // chunk-list keys of one level
  size_t off_count, off_ticket, off_frontier, off_fscore, off_token, off_parent, off_depth,
      off_prow, off_score, off_partial, total;
};

PoolLayout pool_layout(int B, int k, int depth, int V) {
  PoolLayout L;
  L.P = k + (depth - 1) * k * k;
  L.c0 = chunk_plan(B, V);
  L.c1 = chunk_plan(B * k, V);
  L.parts = std::max((size_t)B * L.c0.S, (size_t)B * k * L.c1.S) * k;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.off_count = take((size_t)B * 4);
  L.off_ticket = take((size_t)2 * B * 4);
  L.off_frontier = take((size_t)B * k * 4);
  L.off_fscore = take((size_t)B * k * 4);
  L.off_token = take((size_t)B * L.P * 4);
  L.off_parent = take((size_t)B * L.P * 4);
  L.off_depth = take((size_t)B * L.P * 4);
  L.off_prow = take((size_t)B * L.P * 4);
  L.off_score = take((size_t)B * L.P * 4);
  // chunk lists: by level parity for level-by-level builds, one slice per
  // level when every level is ranked in one launch
  L.off_partial = take((size_t)std::max(2, depth) * L.parts * 8);
  L.total = o;
  return L;
}

struct PoolPtrs {
  int* count;     // [B] pool fill
  int* ticket;    // [2, B] CTAs of a level that have finished, by level parity
  int* frontier;  // [B, k] pool index of the frontier, by rank
  float* fscore;  // [B, k] its score
  int* token;
  int* parent;
  int* depth;
  int* prow;
  float* score;
  unsigned long long* partial;  // chunk top-k lists, [2, parts] by level parity
};

PoolPtrs pool_ptrs(void* base, const PoolLayout& L) {
  char* c = static_cast<char*>(base);
  PoolPtrs p;
  p.count = reinterpret_cast<int*>(c + L.off_count);
  p.ticket = reinterpret_cast<int*>(c + L.off_ticket);
  p.frontier = reinterpret_cast<int*>(c + L.off_frontier);
  p.fscore = reinterpret_cast<float*>(c + L.off_fscore);
  p.token = reinterpret_cast<int*>(c + L.off_token);
  p.parent = reinterpret_cast<int*>(c + L.off_parent);
  p.depth = reinterpret_cast<int*>(c + L.off_depth);
  p.prow = reinterpret_cast<int*>(c + L.off_prow);
  p.score = reinterpret_cast<float*>(c + L.off_score);
  p.partial = reinterpret_cast<unsigned long long*>(c + L.off_partial);
  return p;
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

struct LevelParams {
  int B, V, k, F, R, S, level, P;
  bool vec_ok;     // rows 16-byte aligned: float4 loads
  bool fused;      // the last level: also finalize every sequence (fin)
  bool rows_wait;  // the rows come from the kernel just before: read them after the wait
  const float* logp;
  PoolPtrs pool;
  FinalParams fin;
  int* status;
};

__device__ void finalize_sequence(const FinalParams& A, int b, unsigned char* smem_raw);

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}
__device__ __forceinline__ unsigned lanemask_lt() {
  return (1u << (threadIdx.x & 31)) - 1u;
}

// The key of the first lane named in `bal` (warp-uniform), or `fallback`
// when `bal` is empty or that key is the empty key 0.  Callers pass 1 as the
// fallback bound: every real key (never 0) is at least 1.
__device__ __forceinline__ unsigned long long pick_lane(unsigned bal, unsigned long long v,
                                                        unsigned long long fallback) {
  const int src = bal ? __ffs(bal) - 1 : 0;
  const unsigned long long got = __shfl_sync(0xffffffffu, v, src);
  return (bal && got) ? got : fallback;
}

// Number of lanes whose key is larger than this lane's (keys distinct or
// 0): 32 register shuffles, no shared memory.
__device__ __forceinline__ int warp_rank_desc(unsigned long long key) {
  int r = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) r += (__shfl_sync(0xffffffffu, key, j) > key);
  return r;
}

// Largest key of the warp (every lane gets it): the high and low words by
// two warp reductions.
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long key) {
  const uint32_t hi = (uint32_t)(key >> 32);
  const uint32_t mh = __reduce_max_sync(0xffffffffu, hi);
  const uint32_t ml = __reduce_max_sync(0xffffffffu, hi == mh ? (uint32_t)key : 0u);
  return ((unsigned long long)mh << 32) | ml;
}

struct MergeShared {
  unsigned long long cand[kLvWarps][kRowCap];
  unsigned long long row[EAGLE_MAX_TOPK][EAGLE_MAX_TOPK];
  int fidx[EAGLE_MAX_TOPK];
  float fsc[EAGLE_MAX_TOPK];
  int base;
};

// Exact top-k (descending) of n keys at `src` (written by other CTAs: read
// through L2) by one warp; out[0..k) in order, 0 where fewer than k keys.
__device__ void warp_row_topk(const unsigned long long* src, int n, int k,
                              unsigned long long* cand, unsigned long long* out, int* status) {
  const int lane = threadIdx.x & 31;
  // keys in tiles of 32 x kMergeRegs, loads of a tile in flight together;
  // a single tile stays in registers for the second pass
  const int ntiles = (n + 32 * kMergeRegs - 1) / (32 * kMergeRegs);
  unsigned long long reg[kMergeRegs];
  auto load_tile = [&](int tile) {
#pragma unroll
    for (int r = 0; r < kMergeRegs; ++r) {
      const int i = (tile * kMergeRegs + r) * 32 + lane;
      reg[r] = (i < n) ? __ldcg(src + i) : 0ull;
    }
  };
  unsigned long long lmax = 0;
  for (int tile = 0; tile < ntiles; ++tile) {
    load_tile(tile);
#pragma unroll
    for (int r = 0; r < kMergeRegs; ++r) lmax = umax64(lmax, reg[r]);
  }
  // lower bound of the k-th largest: the k-th largest lane maximum
  const int lrank = warp_rank_desc(lmax);
  unsigned long long tau = pick_lane(__ballot_sync(0xffffffffu, lrank == k - 1), lmax, 1ull);
  int cnt;
  for (int round = 0;; ++round) {
    cnt = 0;
    auto offer = [&](unsigned long long key) {
      const bool pred = key >= tau;
      const unsigned bal = __ballot_sync(0xffffffffu, pred);
      const int pos = cnt + __popc(bal & lanemask_lt());
      if (pred && pos < kRowCap) cand[pos] = key;
      cnt += __popc(bal);
    };
    for (int tile = 0; tile < ntiles; ++tile) {
      if (ntiles > 1) load_tile(tile);
#pragma unroll
      for (int r = 0; r < kMergeRegs; ++r) offer(reg[r]);
    }
    __syncwarp();
    if (cnt <= kRowCap) break;
    if (round == kRowRounds) {
      if (lane == 0) fail(status, EAGLE_ERR_TIMEOUT);
      cnt = kRowCap;
      break;
    }
    // too many: the k-th largest of the held ones is a higher lower bound
    // (each round drops at least kRowCap - k keys)
    unsigned long long m[kRowCap / 32];
    int rk[kRowCap / 32];
#pragma unroll
    for (int t = 0; t < kRowCap / 32; ++t) {
      m[t] = cand[t * 32 + lane];
      rk[t] = 0;
    }
    for (int j = 0; j < kRowCap; ++j) {
      const unsigned long long c = cand[j];
#pragma unroll
      for (int t = 0; t < kRowCap / 32; ++t) rk[t] += (c > m[t]);
    }
    __syncwarp();
    unsigned long long nt = 0;
#pragma unroll
    for (int t = 0; t < kRowCap / 32; ++t)
      nt = umax64(nt, pick_lane(__ballot_sync(0xffffffffu, rk[t] == k - 1), m[t], 0ull));
    tau = nt;
  }
  if (cnt <= 32) {
    // one candidate per lane: exact ranks by shuffles
    const unsigned long long me = (lane < cnt) ? cand[lane] : 0ull;
    const int r = warp_rank_desc(me);
    if (lane < cnt && r < k) out[r] = me;
  } else {
    for (int t = lane; t < cnt; t += 32) {
      const unsigned long long me = cand[t];
      int r = 0;
#pragma unroll 8
      for (int j = 0; j < cnt; ++j) r += (cand[j] > me);
      if (r < k) out[r] = me;
    }
  }
  for (int t = cnt + lane; t < k; t += 32) out[t] = 0ull;
  __syncwarp();
}

struct ChunkShared {
  float grpv[kGroups];
  unsigned long long cand[kCandCap];
  unsigned long long top[EAGLE_MAX_TOPK];
  unsigned long long tau;
  unsigned long long kth;   // the chunk's k-th largest key (0: fewer than k found)
  int kth_row;              // ... and its row
  int cnt, last;
};

// Exact top-k of one chunk (row, chunk) held in registers -- element
// c0 + (j * threads + tid) * 4 + e in v[j][e] -- published to the pool's
// partial lists by thread 0.  With take_ticket, thread 0 also counts the
// chunk on the sequence's ticket; returns true in the CTA that drew the
// last one.
struct NoRefill {
  __device__ void operator()() const {}
};

// `refill` runs on thread 32 once the candidates are counted (warp 1 is
// idle while warp 0 ranks them): the streaming kernel requests its next
// stage there, off the other phases' barriers.
// `bound` (optional, the same in every thread): a key that at least k keys
// of the row reach, e.g. the k-th largest key of another chunk of the row;
// 0 when none is known.  Then only keys above it are kept (a key below it
// is below the row's k-th, and keys are unique), the bound search over the
// group maxima is skipped, and the chunk may publish fewer than k keys.  On
// return it is raised to this chunk's k-th largest key when that is larger.
// PIPE (a streaming CTA with two ChunkShared buffers used by turns, `other`
// the previous chunk's): no barrier before the candidates and none after the
// ranking, so warp 0 ranks this chunk while the other warps load and offer
// the next one; they all meet at the next chunk's candidate barrier (no warp
// gets two chunks ahead).  There, thread 0 resets the other buffer's count
// and every thread folds the previous chunk's k-th key into the bound (the
// bound lags one chunk).  A timed-out wait shows in `abort` after that
// barrier; the call then returns true at once (else false).
template <int VEC, bool PIPE = false, typename Refill = NoRefill>
__device__ bool chunk_topk(const LevelParams& A, int row, int chunk, const float (&v)[VEC][4],
                           ChunkShared& C, bool take_ticket = true, const Refill& refill = Refill(),
                           unsigned long long* bound = nullptr, ChunkShared* other = nullptr,
                           volatile int* abort = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned long long b_in = bound ? *bound : 0ull;
  const int b = row / A.F;
  const int k = A.k;
  const int c0 = chunk * (kLvThreads * 4 * VEC);
  // Values (past the row's end: -inf).  Only the few candidates get 64-bit
  // keys; the per-token work is a max, a finiteness FMA and a compare.
  const bool ragged = c0 + kLvThreads * 4 * VEC > A.V;   // block-uniform
  float x[VEC][4];
  float fin = 0.f;   // sum of v * 0: NaN iff some value is not finite
  if (!ragged) {
#pragma unroll
    for (int j = 0; j < VEC; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[j][e] = v[j][e];
        fin = fmaf(v[j][e], 0.f, fin);
      }
  } else {
#pragma unroll
    for (int j = 0; j < VEC; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool real = c0 + (j * kLvThreads + tid) * 4 + e < A.V;
        x[j][e] = real ? v[j][e] : -INFINITY;
        if (real) fin = fmaf(v[j][e], 0.f, fin);
      }
  }
  float own_max = -INFINITY;   // this thread's largest value
#pragma unroll
  for (int j = 0; j < VEC; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) own_max = fmaxf(own_max, x[j][e]);
  if (b_in == 0) {
    float tmax = own_max;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    if ((lane & 15) == 0) C.grpv[warp * 2 + (lane >> 4)] = tmax;
  }
  // With a bound no barrier comes before the candidates: the count was
  // reset at the end of the previous call (of the same row), and the
  // finiteness check joins the candidates' barrier.  A stale C.kth there is
  // the previous chunk's, already folded into the bound.
  if (b_in == 0) {
    if (tid == 0) {
      C.cnt = 0;
      C.kth = 0ull;
    }
    if (__syncthreads_or(!(fin == 0.f)) && tid == 0) fail(A.status, EAGLE_ERR_NUMERIC);
    if constexpr (PIPE) {
      if (*abort) return true;
    }
  }
  // every warp: the largest group maximum that at least k group maxima
  // reach -- at least k tokens of the chunk are >= it (ties included): the
  // k-th largest of the 32 group maxima counted with multiplicity, found by
  // taking the largest remaining value (and its copies) until k are taken.
  // (Measured: warp 0 alone plus a CTA barrier cost ~9x this.)
  float tau_val;
  unsigned long long tau_key = b_in;   // later rounds (or a given bound): the bound as a key
  if (b_in != 0) {
    tau_val = key_value(b_in);
  } else {
    uint32_t ob = ordered_bits(C.grpv[lane]);
    uint32_t top = 0u;
    for (int need = k; need > 0;) {   // at most k rounds (k <= 32 lanes)
      top = __reduce_max_sync(0xffffffffu, ob);
      need -= __popc(__ballot_sync(0xffffffffu, ob == top));
      if (ob == top) ob = 0u;   // below every ordered value of a non-NaN float
    }
    // fewer than k real tokens: every real (finite) token qualifies
    tau_val = fmaxf(from_ordered_bits(top), -3.402823466e38f);
  }
  int cnt;
  for (int round = 0;; ++round) {
    // round 0 compares values only (with a key bound this also keeps the
    // few tokens whose value equals the bound's but whose key is below it:
    // they rank below the chunk's true list and never displace it); later
    // rounds compare keys.  A warp none of whose threads holds a value at
    // the bound offers nothing (most warps: a chunk has few candidates).
    if (__any_sync(0xffffffffu, own_max >= tau_val))
#pragma unroll
    for (int j = 0; j < VEC; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float val = x[j][e];
        const uint32_t idx = (uint32_t)(c0 + (j * kLvThreads + tid) * 4 + e);
        const bool pred = (val >= tau_val) && (round == 0 || desc_key(val, idx) >= tau_key);
        const unsigned bal = __ballot_sync(0xffffffffu, pred);
        if (bal) {
          const int leader = __ffs(bal) - 1;
          int base = 0;
          if (lane == leader) base = atomicAdd(&C.cnt, __popc(bal));
          base = __shfl_sync(0xffffffffu, base, leader);
          const int pos = base + __popc(bal & lanemask_lt());
          if (pred && pos < kCandCap) C.cand[pos] = desc_key(val, idx);
        }
      }
    if (round == 0 && b_in != 0) {
      if (__syncthreads_or(!(fin == 0.f)) && tid == 0) fail(A.status, EAGLE_ERR_NUMERIC);
    } else {
      __syncthreads();
    }
    if constexpr (PIPE) {
      if (round == 0) {
        if (*abort) return true;
        if (tid == 0) other->cnt = 0;
        if (other->kth_row == row && other->kth > *bound) *bound = other->kth;
      }
    }
    if (round == 0 && tid == 32) refill();
    cnt = C.cnt;
    if (cnt <= kCandCap) break;
    if (round == kChunkRounds) {
      if (tid == 0) fail(A.status, EAGLE_ERR_TIMEOUT);
      cnt = kCandCap;
      break;
    }
    // too many: raise the bound to the k-th largest of the held keys
    // (each round drops at least kCandCap - k of them)
    const unsigned long long me = C.cand[tid];
    int rank = 0;
#pragma unroll 8
    for (int i = 0; i < kCandCap; ++i) rank += (C.cand[i] > me);
    __syncthreads();
    if (rank == k - 1) C.tau = me;
    if (tid == 0) C.cnt = 0;
    __syncthreads();
    tau_key = C.tau;
  }
  // ---- exact ranks, and the chunk list published; the sequence's last CTA
  // merges.  The list's writers meet at a warp barrier, then one thread takes
  // the ticket with an acquire-release atomic: the stores are visible to the
  // CTA that draws the last ticket, and that CTA's reads follow the atomic
  // (then a CTA barrier).
  unsigned long long* part = A.pool.partial + ((size_t)row * A.S + chunk) * k;
  if (cnt <= 32) {
    // one candidate per lane of warp 0: ranks by shuffles, written at once
    if (warp == 0) {
      const unsigned long long me = (lane < cnt) ? C.cand[lane] : 0ull;
      const int rank = warp_rank_desc(me);
      if (lane < cnt && rank < k) part[rank] = me;
      if (lane >= cnt && lane < k) part[lane] = 0ull;   // fewer than k tokens (or above the bound)
      const unsigned kb = __ballot_sync(0xffffffffu, lane < cnt && rank == k - 1);
      const unsigned long long kv = __shfl_sync(0xffffffffu, me, kb ? __ffs(kb) - 1 : 0);
      if (lane == 0) {
        if (kb) C.kth = kv;
        else if (PIPE) C.kth = 0ull;
        C.kth_row = row;
      }
    }
  } else {
    if (tid < cnt) {
      const unsigned long long me = C.cand[tid];
      int rank = 0;
#pragma unroll 8
      for (int i = 0; i < cnt; ++i) rank += (C.cand[i] > me);
      if (rank < k) C.top[rank] = me;
    }
    __syncthreads();
    if (warp == 0 && lane < k) part[lane] = C.top[lane];
    if (tid == 0) {
      C.kth = C.top[k - 1];
      C.kth_row = row;
    }
  }
  if (warp == 0) {
    __syncwarp();
    if (lane == 0) {
      C.last = 0;
      if (take_ticket) {
        int t;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                     : "=r"(t)
                     : "l"(A.pool.ticket + b)
                     : "memory");
        C.last = (t == A.F * A.S - 1);
      }
    }
  }
  if constexpr (PIPE) return false;
  __syncthreads();
  if (bound && C.kth > *bound) *bound = C.kth;
  // nothing reads the count past the barrier above; the next call's
  // candidates follow a barrier of the caller's
  if (tid == 0) C.cnt = 0;
  return C.last != 0;
}

// The sequence's last CTA: per-row top-k over the chunk lists, children,
// next frontier.
__device__ void merge_sequence(const LevelParams& A, int b, MergeShared& M) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = A.k;
  const int F = A.F;
  int* front = A.pool.frontier + (size_t)b * k;
  float* fsc = A.pool.fscore + (size_t)b * k;
  // frontier scores and the pool fill, by the last warp (which has no row
  // when F < warps), so the row warps start at once
  {
    const int lt = tid - (kLvThreads - 32);
    if (lt >= 0 && lt < F) {
      M.fidx[lt] = (A.level == 0) ? -1 : __ldcg(front + lt);
      M.fsc[lt] = (A.level == 0) ? 0.f : __ldcg(fsc + lt);
    }
    if (lt == 31) {
      M.base = __ldcg(A.pool.count + b);
      A.pool.ticket[b] = 0;  // ready for the next level
    }
  }
  const int n = A.S * k;
  for (int ff = warp; ff < F; ff += kLvWarps)
    warp_row_topk(A.pool.partial + (size_t)(b * F + ff) * n, n, k, M.cand[warp], M.row[ff],
                  A.status);
  __syncthreads();
  const int nc = F * k;  // children in creation order (f-major, rank-minor)
  const int base = M.base;
  if (base < 0 || base + nc > A.P) {  // more levels than the pool was sized for
    if (tid == 0) fail(A.status, EAGLE_ERR_INVALID_ARG);
    return;
  }
  int* tok = A.pool.token + (size_t)b * A.P;
  int* par = A.pool.parent + (size_t)b * A.P;
  int* dep = A.pool.depth + (size_t)b * A.P;
  int* prw = A.pool.prow + (size_t)b * A.P;
  float* sco = A.pool.score + (size_t)b * A.P;
  if (warp == 0) {
    // next frontier: the k largest children by (score desc, creation
    // order).  Row f's children come out of its top-k in descending key
    // order (fp32 addition of the row's score is monotone, ties fall to the
    // earlier child), so this is a k-way merge of the rows' lists: lane f
    // holds row f's next child, one warp maximum per frontier entry.
    int p = 0;
    for (int i = 0; i < k; ++i) {
      unsigned long long key = 0ull;
      if (lane < F && p < k)
        key = desc_key(__fadd_rn(M.fsc[lane], key_value(M.row[lane][p])), (uint32_t)(lane * k + p));
      const unsigned long long mx = warp_max_key(key);
      if (key == mx && mx != 0ull) {
        front[i] = base + lane * k + p;
        fsc[i] = key_value(mx);
        ++p;
      }
    }
  } else {
    // the children, in creation order (f-major, rank-minor)
    for (int c = tid - 32; c < nc; c += kLvThreads - 32) {
      const int ff = c / k, rr = c % k;
      const unsigned long long key = M.row[ff][rr];
      const int at = base + c;
      tok[at] = (int)key_index(key);
      par[at] = M.fidx[ff];
      dep[at] = A.level + 1;
      prw[at] = (A.level == 0) ? 0 : 1 + (A.level - 1) * k + ff;
      sco[at] = __fadd_rn(M.fsc[ff], key_value(key));
    }
  }
  if (tid == 0) A.pool.count[b] = base + nc;
}

// One level.  CTA (row, chunk): exact top-k of the chunk -> partial list.
// The sequence's last CTA: per-row top-k, children, next frontier.
template <int VEC>
__global__ void __launch_bounds__(kLvThreads, 2) expand_level_kernel(const LevelParams A) {
  // A level's draft rows and its chunk lists do not depend on the level
  // before it (whose lists are the other parity's), so past level 0 only
  // the merging CTA waits for it.  Level 0 follows the pool reset.  Rows
  // written by the kernel just before this one are read after the wait.
  if (A.level == 0 || A.rows_wait) pdl_begin();
  __shared__ ChunkShared C;
  __shared__ MergeShared M;
  const int tid = threadIdx.x;
  const int row = blockIdx.x / A.S, chunk = blockIdx.x % A.S;
  const int b = row / A.F, f = row % A.F;
  const int k = A.k;
  const int local_row = (A.level == 0) ? 0 : 1 + (A.level - 1) * k + f;
  const float* src = A.logp + ((size_t)b * A.R + local_row) * A.V;
  const int c0 = chunk * (kLvThreads * 4 * VEC);
  // ---- chunk in registers: element c0 + (j * threads + tid) * 4 + e
  float v[VEC][4];
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    const int i0 = c0 + (j * kLvThreads + tid) * 4;
    if (A.vec_ok && i0 + 4 <= A.V) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(src + i0));
      v[j][0] = x.x;
      v[j][1] = x.y;
      v[j][2] = x.z;
      v[j][3] = x.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[j][e] = (i0 + e < A.V) ? __ldg(src + i0 + e) : 0.f;
    }
  }
  if (!chunk_topk<VEC>(A, row, chunk, v, C)) return;
  if (A.level > 0 && !A.rows_wait) pdl_begin();   // the level before: frontier, pool fill
  merge_sequence(A, b, M);
  if (A.fused) {
    // the last level: this CTA holds the sequence's complete pool
    __threadfence_block();
    __syncthreads();
    extern __shared__ __align__(16) unsigned char dyn_smem[];
    finalize_sequence(A.fin, b, dyn_smem);
  }
}

// Streaming variant for levels larger than one wave of CTAs: persistent CTAs
// walk a contiguous range of chunks (8192 tokens each) through a two-stage
// ring of bulk copies into shared memory, so the next chunk arrives while
// the current one is ranked.  A CTA counts its chunks of a sequence on the
// sequence's ticket once, when it leaves that sequence; the CTA that
// completes a sequence merges it before moving on.
constexpr int kStreamVec = kMaxVec;
constexpr int kStreamChunk = kLvThreads * 4 * kStreamVec;   // tokens per chunk
#ifndef EAGLE_EXPAND_STAGES
#define EAGLE_EXPAND_STAGES 2
#endif
constexpr int kStreamStages = EAGLE_EXPAND_STAGES;   // chunk stages in flight per streaming CTA
constexpr size_t kStreamSmem = (size_t)kStreamStages * kStreamChunk * 4;

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(tc::smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(kLvThreads, 2)
expand_level_stream_kernel(const LevelParams A, int total_chunks) {
  // as expand_level_kernel: past level 0 a CTA waits for the level before
  // only when it is about to merge
  bool waited = (A.level == 0 || A.rows_wait);
  if (waited) pdl_begin();
  __shared__ ChunkShared C;
  __shared__ MergeShared M;
  __shared__ uint64_t full[kStreamStages];
  __shared__ int abort_flag, s_last;
  extern __shared__ __align__(128) unsigned char stage_mem[];   // kStreamSmem bytes
  const int tid = threadIdx.x;
  const int k = A.k;
  const int per_seq = A.F * A.S;
  const int id0 = (int)((long long)total_chunks * blockIdx.x / gridDim.x);
  const int id1 = (int)((long long)total_chunks * (blockIdx.x + 1) / gridDim.x);
  auto issue = [&](int id, int st) {
    const int row = id / A.S, chunk = id % A.S;
    const int b = row / A.F, f = row % A.F;
    const int local_row = (A.level == 0) ? 0 : 1 + (A.level - 1) * k + f;
    const int c0 = chunk * kStreamChunk;
    const uint32_t bytes = (uint32_t)min(kStreamChunk, A.V - c0) * 4u;   // V % 4 == 0
    tc::mbar_arrive_expect_tx(&full[st], bytes);
    bulk_load(stage_mem + (size_t)st * kStreamChunk * 4,
              A.logp + ((size_t)b * A.R + local_row) * A.V + c0, bytes, &full[st]);
  };
  if (tid == 0) {
    for (int st = 0; st < kStreamStages; ++st) tc::mbar_init(&full[st], 1);
    abort_flag = 0;
    tc::fence_barrier_init();
    for (int st = 0; st < kStreamStages; ++st)
      if (id0 + st < id1) issue(id0 + st, st);
  }
  __syncthreads();
  // count `n` finished chunks of sequence b; merge it if they were the last
  auto leave_sequence = [&](int b, int n) {
    if (tid == 0) {
      int t;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
                   : "=r"(t)
                   : "l"(A.pool.ticket + b), "r"(n)
                   : "memory");
      s_last = (t + n == per_seq);
    }
    __syncthreads();
    if (s_last) {
      if (!waited) {
        pdl_begin();
        waited = true;
      }
      merge_sequence(A, b, M);
    }
    __syncthreads();
  };
  int i = 0, cur_b = -1, cur_n = 0;
  bool aborted = false;
  // the k-th largest key of this CTA's earlier chunks of the current row
  int bound_row = -1;
  unsigned long long bound = 0ull;
  for (int id = id0; id < id1; ++id, ++i) {
    const int st = i % kStreamStages;
    const bool got =
        tc::mbar_wait(&full[st], (uint32_t)((i / kStreamStages) & 1), &abort_flag, A.status);
    float v[kStreamVec][4];
    const float4* sm4 = reinterpret_cast<const float4*>(stage_mem + (size_t)st * kStreamChunk * 4);
#pragma unroll
    for (int j = 0; j < kStreamVec; ++j) {
      const float4 x = got ? sm4[j * kLvThreads + tid] : make_float4(0.f, 0.f, 0.f, 0.f);
      v[j][0] = x.x;
      v[j][1] = x.y;
      v[j][2] = x.z;
      v[j][3] = x.w;
    }
    // every thread has the stage in registers (it is refilled during the
    // ranking below)
    if (!__syncthreads_and(got)) {
      aborted = true;
      break;
    }
    auto refill = [&]() {
      if (id + kStreamStages < id1) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(id + kStreamStages, st);
      }
    };
    const int row = id / A.S, chunk = id % A.S;
    const int b = row / A.F;
    if (b != cur_b) {
      if (cur_b >= 0) leave_sequence(cur_b, cur_n);
      cur_b = b;
      cur_n = 0;
    }
    if (row != bound_row) {
      bound_row = row;
      bound = 0ull;
    }
    chunk_topk<kStreamVec>(A, row, chunk, v, C, false, refill, &bound);
    ++cur_n;
  }
  if (!aborted && cur_b >= 0) leave_sequence(cur_b, cur_n);
  if (aborted && tid == 0) {
    // let the copies still in flight land before the CTA leaves
    int never = 0;
    for (int j = i; j < i + kStreamStages; ++j)
      if (id0 + j < id1)
        tc::mbar_wait(&full[j % kStreamStages], (uint32_t)((j / kStreamStages) & 1), &never,
                      nullptr, 200000000ll);
  }
}

// Every level's chunk lists in one launch, when all draft rows are ready
// before it: chunk ids run level by level (level 0's B rows, then B k rows
// per later level, S chunks each); each persistent CTA walks a contiguous
// range through the same two-stage ring as the streaming level kernel, with
// the row bound carried along a row, and writes its lists to the level's
// slice of the pool (`level_keys` keys apart).  The levels are merged
// afterwards: every level of a sequence and its finalize by one CTA
// (expand_finish_kernel), or, when the finalize's shared memory does not fit
// beside the merge's, one launch per level (expand_merge_kernel) and the
// finalize launch.
__global__ void __launch_bounds__(kLvThreads, 2)
expand_all_stream_kernel(const LevelParams A, long long level_keys, int total_chunks) {
  pdl_begin();   // the pool reset comes just before
  __shared__ ChunkShared C2[2];   // by chunk parity (chunk_topk's PIPE mode)
  __shared__ uint64_t full[kStreamStages];
  __shared__ int abort_flag;
  extern __shared__ __align__(128) unsigned char stage_mem[];   // kStreamSmem bytes
  const int tid = threadIdx.x;
  const int k = A.k, S = A.S;
  const int n0 = A.B * S, n1 = A.B * k * S;   // chunks of level 0, of a later level
  auto decode = [&](int id, int& level, int& row, int& chunk) {
    int x = id;
    level = 0;
    if (id >= n0) {
      level = 1 + (id - n0) / n1;
      x = (id - n0) % n1;
    }
    row = x / S;
    chunk = x % S;
  };
  const int id0 = (int)((long long)total_chunks * blockIdx.x / gridDim.x);
  const int id1 = (int)((long long)total_chunks * (blockIdx.x + 1) / gridDim.x);
  auto issue = [&](int id, int st) {
    int level, row, chunk;
    decode(id, level, row, chunk);
    const int F = level ? k : 1;
    const int b = row / F, f = row % F;
    const int local_row = (level == 0) ? 0 : 1 + (level - 1) * k + f;
    const int c0 = chunk * kStreamChunk;
    const uint32_t bytes = (uint32_t)min(kStreamChunk, A.V - c0) * 4u;   // V % 4 == 0
    tc::mbar_arrive_expect_tx(&full[st], bytes);
    bulk_load(stage_mem + (size_t)st * kStreamChunk * 4,
              A.logp + ((size_t)b * A.R + local_row) * A.V + c0, bytes, &full[st]);
  };
  if (tid == 0) {
    for (int st = 0; st < kStreamStages; ++st) tc::mbar_init(&full[st], 1);
    abort_flag = 0;
    for (int c = 0; c < 2; ++c) {
      C2[c].cnt = 0;
      C2[c].kth = 0ull;
      C2[c].kth_row = -1;
    }
    tc::fence_barrier_init();
    for (int st = 0; st < kStreamStages; ++st)
      if (id0 + st < id1) issue(id0 + st, st);
  }
  __syncthreads();
  LevelParams Al = A;   // the current level's view: F, level, its pool slice
  int cur_level = -1, bound_row = -1;
  unsigned long long bound = 0ull;
  int i = 0;
  bool aborted = false;
  for (int id = id0; id < id1; ++id, ++i) {
    const int st = i % kStreamStages;
    const bool got =
        tc::mbar_wait(&full[st], (uint32_t)((i / kStreamStages) & 1), &abort_flag, A.status);
    float v[kStreamVec][4];
    const float4* sm4 = reinterpret_cast<const float4*>(stage_mem + (size_t)st * kStreamChunk * 4);
#pragma unroll
    for (int j = 0; j < kStreamVec; ++j) {
      const float4 x = got ? sm4[j * kLvThreads + tid] : make_float4(0.f, 0.f, 0.f, 0.f);
      v[j][0] = x.x;
      v[j][1] = x.y;
      v[j][2] = x.z;
      v[j][3] = x.w;
    }
    // no barrier here: the stage is refilled only after the candidates'
    // barrier, by which every thread has read it
    auto refill = [&]() {
      if (id + kStreamStages < id1) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(id + kStreamStages, st);
      }
    };
    int level, row, chunk;
    decode(id, level, row, chunk);
    if (level != cur_level) {
      cur_level = level;
      Al.level = level;
      Al.F = level ? k : 1;
      Al.pool.partial = A.pool.partial + (size_t)level * level_keys;
      bound_row = -1;
    }
    if (row != bound_row) {
      bound_row = row;
      bound = 0ull;
    }
    if (chunk_topk<kStreamVec, true>(Al, row, chunk, v, C2[i & 1], false, refill, &bound,
                                     &C2[(i & 1) ^ 1], &abort_flag)) {
      aborted = true;
      break;
    }
  }
  if (aborted && tid == 0) {
    // let the copies still in flight land before the CTA leaves
    int never = 0;
    for (int j = i; j < i + kStreamStages; ++j)
      if (id0 + j < id1)
        tc::mbar_wait(&full[j % kStreamStages], (uint32_t)((j / kStreamStages) & 1), &never,
                      nullptr, 200000000ll);
  }
}

// One level's merge for every sequence (one CTA each), after its chunk
// lists and the level before are complete.
__global__ void __launch_bounds__(kLvThreads, 1) expand_merge_kernel(const LevelParams A) {
  pdl_begin();
  __shared__ MergeShared M;
  merge_sequence(A, blockIdx.x, M);
}

// Every level's merge of one sequence in turn, then its finalize: a
// sequence's levels depend only on its own earlier levels, so one CTA per
// sequence runs them all (`smem_raw`: the finalize's P * 44 bytes).
__global__ void __launch_bounds__(kLvThreads, 1)
expand_finish_kernel(const LevelParams A, int depth, long long level_keys) {
  pdl_begin();
  __shared__ MergeShared M;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int b = blockIdx.x;
  LevelParams Al = A;
  for (int level = 0; level < depth; ++level) {
    Al.level = level;
    Al.F = level ? A.k : 1;
    Al.pool.partial = A.pool.partial + (size_t)level * level_keys;
    merge_sequence(Al, b, M);
    // the frontier, its scores and the pool fill went to global memory:
    // the next level (this CTA) reads them back
    __threadfence_block();
    __syncthreads();
  }
  finalize_sequence(A.fin, b, smem_raw);
}

// Finalize one sequence with the calling CTA (any block size that is a
// multiple of 64): keep the `budget` pool entries of largest key (score
// desc, creation order) -- a radix select of the budget-th key -- number the
// kept nodes by (depth, score desc, creation order) and write the tree.
// `smem_raw`: 44 * P bytes of shared memory.  Every sequence's pool holds
// P = k + (depth-1) k^2 entries after the last level, which fixes the node
// offset of each sequence without waiting for the others.
__device__ void finalize_sequence(const FinalParams& A, int b, unsigned char* smem_raw) {
  // every pool array of the sequence in shared memory, loaded in one round
  // trip (the pool holds P slots whatever its fill)
  const int P = A.P;
  unsigned long long* s_key = reinterpret_cast<unsigned long long*>(smem_raw);  // [P]
  unsigned long long* c_key = s_key + P;     // kept keys, compacted           [P]
  int* s_dep = reinterpret_cast<int*>(c_key + P);                              // [P]
  int* s_par = s_dep + P;
  int* s_tok = s_par + P;
  int* s_prw = s_tok + P;
  int* s_node = s_prw + P;
  int* s_list = s_node + P;                  // pool index of each kept entry
  int* c_dep = s_list + P;                   // its depth, compacted
  // three histograms in rotation: the one scanned in pass p-1 is cleared in
  // pass p and filled in pass p+2, so a pass needs a single barrier
  __shared__ int s_hist[3][256];
  __shared__ int s_nsel, s_off, s_n;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x;
  const int bud = A.budget[b];
  if (tid == 0) {
    s_nsel = 0;
    s_n = max(0, min(__ldcg(A.pool.count + b), P));
    if (bud < 0) fail(A.status, EAGLE_ERR_INVALID_ARG);
  }
  if (warp == 1) {
    // node offset of this sequence: sum over earlier sequences of kept + root
    int off = 0;
    for (int j = lane; j < b; j += 32) off += min(max(A.budget[j], 0), P) + 1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) off += __shfl_xor_sync(0xffffffffu, off, o);
    if (lane == 0) s_off = off;
  }
  for (int i = tid; i < 2 * 256; i += nthreads) s_hist[i >> 8][i & 255] = 0;
  {
    const size_t o = (size_t)b * P;
    for (int i = tid; i < P; i += nthreads) {
      s_key[i] = desc_key(__ldcg(A.pool.score + o + i), (uint32_t)i);
      s_dep[i] = __ldcg(A.pool.depth + o + i);
      s_par[i] = __ldcg(A.pool.parent + o + i);
      s_tok[i] = __ldcg(A.pool.token + o + i);
      s_prw[i] = __ldcg(A.pool.prow + o + i);
      s_node[i] = -1;
    }
  }
  __syncthreads();
  const int n = s_n;
  const int keep = min(max(bud, 0), n);
  // radix select (8 bits at a time, high to low) of the keep-th largest key
  unsigned long long prefix = 0, mask = 0;
  int rem = keep;
  if (keep > 0 && keep < n) {
    for (int shift = 56, p = 0; shift >= 0; shift -= 8, ++p) {
      int* hist = s_hist[p % 3];
      for (int i0 = 0; i0 < n; i0 += nthreads) {   // uniform trip count
        const int i = i0 + tid;
        const unsigned long long key = (i < n) ? s_key[i] : 0ull;
        const int bin = (i < n && (key & mask) == prefix) ? (int)(key >> shift) & 255 : 256;
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (bin < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
      }
      __syncthreads();
      // every warp finds the digit holding the rem-th largest key (the same
      // answer in each), scanning bins from the top
      int h[8], tot = 0;
#pragma unroll
      for (int d = 0; d < 8; ++d) {
        h[d] = hist[lane * 8 + d];
        tot += h[d];
      }
      int incl = tot;  // sum over this lane and the lanes above it
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += t;
      }
      int above = incl - tot, digit = -1, nrem = 0, eq = 0;
#pragma unroll
      for (int d = 7; d >= 0; --d) {
        if (above < rem && rem <= above + h[d]) {
          digit = lane * 8 + d;
          nrem = rem - above;
          eq = h[d];
        }
        above += h[d];
      }
      const unsigned owner = __ballot_sync(0xffffffffu, digit >= 0);
      const int src = owner ? __ffs(owner) - 1 : 0;
      digit = __shfl_sync(0xffffffffu, digit, src);
      nrem = __shfl_sync(0xffffffffu, nrem, src);
      eq = __shfl_sync(0xffffffffu, eq, src);
      // the histogram scanned in the pass before is free again
      for (int i = tid; i < 256; i += nthreads) s_hist[(p + 2) % 3][i] = 0;
      prefix |= (unsigned long long)digit << shift;
      mask |= 255ull << shift;
      rem = nrem;
      if (eq == rem) break;  // every key under this prefix is kept
    }
  }
  // kept: keys >= the threshold (prefix, low bits zero), exactly `keep` of
  // them; compacted with their depths
  const unsigned long long tau = (keep == 0) ? ~0ull : (keep == n ? 1ull : prefix);
  for (int i = tid; i < n; i += nthreads) {
    const unsigned long long key = s_key[i];
    if (keep > 0 && key >= tau) {
      const int at = atomicAdd(&s_nsel, 1);
      s_list[at] = i;
      c_key[at] = key;
      c_dep[at] = s_dep[i];
    }
  }
  __syncthreads();
  const int ns = s_nsel;
  const int off = s_off;
  // node number of every kept entry: 1 + rank by (depth, score desc,
  // creation); gs lanes share one entry's count
  int gs = 1;
  while (gs < 32 && 2 * gs * ns <= nthreads) gs *= 2;
  const int sub = lane & (gs - 1);
  for (int a0 = 0; a0 < ns; a0 += nthreads / gs) {
    const int a = a0 + tid / gs;
    const int da = (a < ns) ? c_dep[a] : 0;
    const unsigned long long ka = (a < ns) ? c_key[a] : 0ull;
    int rank = 0;
#pragma unroll 4
    for (int c = sub; c < ns; c += gs) {
      const int dc = c_dep[c];
      rank += (dc < da) || (dc == da && c_key[c] > ka);
    }
    for (int o = gs >> 1; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (a < ns && sub == 0) s_node[s_list[a]] = 1 + rank;
  }
  __syncthreads();
  for (int a = tid; a < ns; a += nthreads) {
    const int ia = s_list[a];
    const int pp = s_par[ia];
    const int pnode = (pp < 0) ? 0 : (pp < n ? s_node[pp] : -1);
    if (pnode < 0) fail(A.status, EAGLE_ERR_INVALID_TREE);  // not parent-closed
    const int at = off + s_node[ia];
    A.parent[at] = pnode;
    A.tokens[at] = s_tok[ia];
    A.node_depth[at] = s_dep[ia];
    A.score[at] = key_value(s_key[ia]);
    A.p_row_of_node[at] = b * A.R + s_prw[ia];
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

__global__ void __launch_bounds__(kFinalThreads) expand_finalize_kernel(const FinalParams A) {
  pdl_begin();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  finalize_sequence(A, blockIdx.x, smem_raw);
}

}  // namespace

extern "C" size_t eagle_draft_pool_bytes(int B, int k, int depth, int V) {
  if (B < 1 || k < 1 || k > EAGLE_MAX_TOPK || depth < 1 || depth > EAGLE_MAX_DEPTH || V < k ||
      V > kMaxV)
    return 0;
  return pool_layout(B, k, depth, V).total;
}

namespace {

eagle_status expand_impl(bool rows_wait, int B, int V, int k, int depth, int level, int finalize,
                         const float* d_draft_logp, const int32_t* d_budget,
                         const int32_t* d_root_token, void* d_pool, size_t pool_bytes,
                         int32_t* d_tree_off, int32_t* d_parent, int32_t* d_tokens,
                         int32_t* d_node_depth, float* d_score, int32_t* d_p_row_of_node,
                         int* d_status, eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 1 && V >= 1, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(k >= 1 && k <= EAGLE_MAX_TOPK && k <= V, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(depth >= 1 && depth <= EAGLE_MAX_DEPTH, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(V <= kMaxV, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(d_pool && d_status, EAGLE_ERR_INVALID_ARG);
  const PoolLayout L = pool_layout(B, k, depth, V);
  EAGLE_HOST_CHECK(pool_bytes >= L.total, EAGLE_ERR_WORKSPACE);
  EAGLE_HOST_CHECK(((uintptr_t)d_pool & 255) == 0, EAGLE_ERR_INVALID_ARG);
  const PoolPtrs pp = pool_ptrs(d_pool, L);
  cudaStream_t s = (cudaStream_t)stream;
  const int R = 1 + (depth - 1) * k;
  EAGLE_HOST_CHECK(finalize >= 0 && finalize <= 2, EAGLE_ERR_INVALID_ARG);
  FinalParams F;
  const size_t fin_smem = (size_t)L.P * (2 * 8 + 7 * 4);
  if (finalize) {
    EAGLE_HOST_CHECK(d_budget && d_tree_off && d_parent && d_tokens && d_node_depth && d_score &&
                         d_p_row_of_node,
                     EAGLE_ERR_INVALID_ARG);
    EAGLE_HOST_CHECK(fin_smem <= 200 * 1024, EAGLE_ERR_UNSUPPORTED);
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
  }
  auto launch_finalize = [&]() -> eagle_status {
    if (fin_smem > 40 * 1024 &&
        cudaFuncSetAttribute(expand_finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)fin_smem) != cudaSuccess)
      return EAGLE_ERR_CUDA;
    return launch_status(launch_pdl(expand_finalize_kernel, dim3(B), dim3(kFinalThreads), fin_smem,
                                    s, F));
  };
  if (finalize == 1) return launch_finalize();
  // one level (finalize == 2: the last level, with the finalize fused in)
  EAGLE_HOST_CHECK(level >= 0 && level < depth, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(finalize == 0 || level == depth - 1, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(d_draft_logp, EAGLE_ERR_INVALID_ARG);
  if (level == 0) {
    // fresh tree: zero the pool fill counts and the level tickets
    cudaError_t e = cudaMemsetAsync(static_cast<char*>(d_pool), 0, L.off_frontier, s);
    if (e != cudaSuccess) return EAGLE_ERR_CUDA;
  }
  const ChunkPlan cp = (level == 0) ? L.c0 : L.c1;
  LevelParams A;
  A.B = B;
  A.V = V;
  A.k = k;
  A.F = (level == 0) ? 1 : k;
  A.R = R;
  A.S = cp.S;
  A.level = level;
  A.P = L.P;
  A.vec_ok = (V % 4 == 0) && ((uintptr_t)d_draft_logp % 16 == 0);
  A.rows_wait = rows_wait;
  A.logp = d_draft_logp;
  A.pool = pp;
  A.pool.ticket = pp.ticket + (size_t)(level & 1) * B;
  A.pool.partial = pp.partial + (size_t)(level & 1) * L.parts;
  A.status = d_status;
  void (*kern)(const LevelParams) = (cp.vec == 1)   ? expand_level_kernel<1>
                                    : (cp.vec == 2) ? expand_level_kernel<2>
                                                    : expand_level_kernel<4>;
  static PerDeviceOnce carveout_once;
  // the whole unified L1 as shared memory wherever an expand CTA lands
  // first, so that the LM head running beside the expand still fits
  if (carveout_once.run([] {
        for (auto k : {expand_level_kernel<1>, expand_level_kernel<2>, expand_level_kernel<4>}) {
          const cudaError_t e = cudaFuncSetAttribute(
              k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
          if (e != cudaSuccess) return e;
        }
        return cudaFuncSetAttribute(expand_level_stream_kernel,
                                    cudaFuncAttributePreferredSharedMemoryCarveout,
                                    cudaSharedmemCarveoutMaxShared);
      }) != cudaSuccess)
    return EAGLE_ERR_CUDA;
  // levels beyond one wave even at the largest chunks stream through
  // persistent CTAs (no finalize fusion there)
  const long long total_chunks = (long long)B * A.F * A.S;
  const bool stream_it = A.vec_ok && cp.vec == kMaxVec && total_chunks > kOneWave;
  if (stream_it) {
    A.fused = false;
    A.fin = F;
    static PerDeviceOnce attr_once;
    if (attr_once.run([] {
          return cudaFuncSetAttribute(expand_level_stream_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kStreamSmem);
        }) != cudaSuccess)
      return EAGLE_ERR_CUDA;
    const int grid = (int)std::min<long long>(total_chunks, kOneWave);
    const eagle_status st =
        launch_status(launch_pdl(expand_level_stream_kernel, dim3(grid), dim3(kLvThreads),
                                 kStreamSmem, s, A, (int)total_chunks));
    if (st != EAGLE_OK || finalize != 2) return st;
    return launch_finalize();
  }
  // fuse the finalize when its shared memory fits beside the level's
  A.fused = (finalize == 2) && fin_smem <= kFusedSmemMax;
  A.fin = F;
  const size_t dyn = A.fused ? fin_smem : 0;
  if (dyn > 0 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn) !=
          cudaSuccess)
    return EAGLE_ERR_CUDA;
  const eagle_status st =
      launch_status(launch_pdl(kern, dim3(B * A.F * A.S), dim3(kLvThreads), dyn, s, A));
  if (st != EAGLE_OK || finalize != 2 || A.fused) return st;
  return launch_finalize();
}

}  // namespace

extern "C" eagle_status eagle_draft_expand(int B, int V, int k, int depth, int level,
                                           int finalize, const float* d_draft_logp,
                                           const int32_t* d_budget, const int32_t* d_root_token,
                                           void* d_pool, size_t pool_bytes, int32_t* d_tree_off,
                                           int32_t* d_parent, int32_t* d_tokens,
                                           int32_t* d_node_depth, float* d_score,
                                           int32_t* d_p_row_of_node, int* d_status,
                                           eagle_stream_t stream) {
  return expand_impl(false, B, V, k, depth, level, finalize, d_draft_logp, d_budget, d_root_token,
                     d_pool, pool_bytes, d_tree_off, d_parent, d_tokens, d_node_depth, d_score,
                     d_p_row_of_node, d_status, stream);
}

// Every level and the finalize in one call (all draft rows ready): one
// launch ranks every level's chunks, then one merge launch per level and
// the finalize.  Rows that are not 16-byte aligned rows of a multiple of 4
// entries take the level-by-level path instead.
extern "C" eagle_status eagle_draft_expand_all(int B, int V, int k, int depth,
                                               const float* d_draft_logp,
                                               const int32_t* d_budget,
                                               const int32_t* d_root_token, void* d_pool,
                                               size_t pool_bytes, int32_t* d_tree_off,
                                               int32_t* d_parent, int32_t* d_tokens,
                                               int32_t* d_node_depth, float* d_score,
                                               int32_t* d_p_row_of_node, int* d_status,
                                               eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 1 && V >= 1, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(k >= 1 && k <= EAGLE_MAX_TOPK && k <= V, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(depth >= 1 && depth <= EAGLE_MAX_DEPTH, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(V <= kMaxV, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(d_pool && d_status && d_draft_logp && d_budget && d_tree_off && d_parent &&
                       d_tokens && d_node_depth && d_score && d_p_row_of_node,
                   EAGLE_ERR_INVALID_ARG);
  const PoolLayout L = pool_layout(B, k, depth, V);
  EAGLE_HOST_CHECK(pool_bytes >= L.total, EAGLE_ERR_WORKSPACE);
  EAGLE_HOST_CHECK(((uintptr_t)d_pool & 255) == 0, EAGLE_ERR_INVALID_ARG);
  auto level_call = [&](int level, int finalize) {
    return expand_impl(false, B, V, k, depth, level, finalize, d_draft_logp, d_budget,
                       d_root_token, d_pool, pool_bytes, d_tree_off, d_parent, d_tokens,
                       d_node_depth, d_score, d_p_row_of_node, d_status, stream);
  };
  if (V % 4 != 0 || ((uintptr_t)d_draft_logp & 15) != 0) {
    for (int level = 0; level < depth; ++level) {
      const eagle_status st = level_call(level, level == depth - 1 ? 2 : 0);
      if (st != EAGLE_OK) return st;
    }
    return EAGLE_OK;
  }
  const PoolPtrs pp = pool_ptrs(d_pool, L);
  cudaStream_t s = (cudaStream_t)stream;
  const int R = 1 + (depth - 1) * k;
  const int S = (int)ceil_div(V, (long long)kStreamChunk);
  // fresh tree: zero the pool fill counts and the level tickets
  if (cudaMemsetAsync(static_cast<char*>(d_pool), 0, L.off_frontier, s) != cudaSuccess)
    return EAGLE_ERR_CUDA;
  LevelParams A = {};
  A.B = B;
  A.V = V;
  A.k = k;
  A.F = 1;
  A.R = R;
  A.S = S;
  A.level = 0;
  A.P = L.P;
  A.vec_ok = true;
  A.fused = false;
  A.rows_wait = false;
  A.logp = d_draft_logp;
  A.pool = pp;
  A.status = d_status;
  static PerDeviceOnce attr_once;
  if (attr_once.run([] {
        cudaError_t e = cudaFuncSetAttribute(expand_all_stream_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kStreamSmem);
        if (e == cudaSuccess)
          e = cudaFuncSetAttribute(expand_all_stream_kernel,
                                   cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxShared);
        return e;
      }) != cudaSuccess)
    return EAGLE_ERR_CUDA;
  const long long total = (long long)B * S + (long long)(depth - 1) * B * k * S;
  EAGLE_HOST_CHECK(total < (1ll << 31), EAGLE_ERR_UNSUPPORTED);
  const int grid = (int)std::min<long long>(total, kOneWave);
  eagle_status st = launch_status(launch_pdl(expand_all_stream_kernel, dim3(grid),
                                             dim3(kLvThreads), kStreamSmem, s, A,
                                             (long long)L.parts, (int)total));
  if (st != EAGLE_OK) return st;
  // every level's merge and the finalize in one launch (one CTA per
  // sequence), when the finalize's shared memory fits beside the merge's
  const size_t fin_smem = (size_t)L.P * (2 * 8 + 7 * 4);
  if (fin_smem <= kFinishSmemMax) {
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
    A.fin = F;
    // (its static shared memory plus the finalize's may pass 48 KB)
    static PerDeviceOnce finish_once;
    if (finish_once.run([] {
          return cudaFuncSetAttribute(expand_finish_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kFinishSmemMax);
        }) != cudaSuccess)
      return EAGLE_ERR_CUDA;
    return launch_status(launch_pdl(expand_finish_kernel, dim3(B), dim3(kLvThreads), fin_smem, s,
                                    A, depth, (long long)L.parts));
  }
  for (int level = 0; level < depth && st == EAGLE_OK; ++level) {
    LevelParams M = A;
    M.level = level;
    M.F = level ? k : 1;
    M.pool.partial = pp.partial + (size_t)level * L.parts;
    st = launch_status(launch_pdl(expand_merge_kernel, dim3(B), dim3(kLvThreads), 0, s, M));
  }
  if (st != EAGLE_OK) return st;
  return level_call(depth - 1, 1);
}

extern "C" eagle_status eagle_draft_expand_dep(int B, int V, int k, int depth, int level,
                                               int finalize, const float* d_draft_logp,
                                               const int32_t* d_budget,
                                               const int32_t* d_root_token, void* d_pool,
                                               size_t pool_bytes, int32_t* d_tree_off,
                                               int32_t* d_parent, int32_t* d_tokens,
                                               int32_t* d_node_depth, float* d_score,
                                               int32_t* d_p_row_of_node, int* d_status,
                                               eagle_stream_t stream) {
  return expand_impl(true, B, V, k, depth, level, finalize, d_draft_logp, d_budget, d_root_token,
                     d_pool, pool_bytes, d_tree_off, d_parent, d_tokens, d_node_depth, d_score,
                     d_p_row_of_node, d_status, stream);
}

// ---------------------------------------------------------------------------
// Input rows of the draft head for one level (the draft-tree loop).
// Level 0: row b = [f_ctx[b] ; emb[root_token[b]]] (the root).  Level d >= 1:
// the frontier left by level d-1, by rank: row b*k + f = [feature of the
// node's parent ; emb[node's token]], the parent's feature found among the
// previous level's rows (feat_prev / node_prev, F_prev per sequence, node
// -1 = the root).  node_cur receives the rows' pool indices.
// ---------------------------------------------------------------------------
namespace {

__global__ void __launch_bounds__(256)
head_input_kernel(PoolPtrs pool, int k, int P, int H, int level, int F_prev,
                  const int* __restrict__ node_prev, int* __restrict__ node_cur,
                  const __nv_bfloat16* __restrict__ feat_prev,
                  const __nv_bfloat16* __restrict__ f_ctx, const int* __restrict__ root_token,
                  const __nv_bfloat16* __restrict__ emb, int V,
                  __nv_bfloat16* __restrict__ a_out, int* status) {
  pdl_begin();
  const int F = (level == 0) ? 1 : k;
  const int r = blockIdx.x, b = r / F, f = r % F;
  __shared__ int s_src, s_tok;
  if (threadIdx.x == 0) {
    int tok, src;
    if (level == 0) {
      tok = root_token[b];
      src = -1;
      node_cur[r] = -1;
    } else {
      const int q = __ldcg(pool.frontier + (size_t)b * k + f);
      tok = __ldcg(pool.token + (size_t)b * P + q);
      const int p = __ldcg(pool.parent + (size_t)b * P + q);
      src = -2;
      for (int j = 0; j < F_prev; ++j)
        if (node_prev[b * F_prev + j] == p) {
          src = b * F_prev + j;
          break;
        }
      node_cur[r] = q;
    }
    if (tok < 0 || tok >= V || src == -2) {
      fail(status, EAGLE_ERR_INVALID_ARG);
      tok = 0;
      src = (level == 0) ? -1 : b * F_prev;
    }
    s_src = src;
    s_tok = tok;
  }
  __syncthreads();
  const __nv_bfloat16* fs = (s_src < 0) ? f_ctx + (size_t)b * H : feat_prev + (size_t)s_src * H;
  const __nv_bfloat16* es = emb + (size_t)s_tok * H;
  __nv_bfloat16* dst = a_out + (size_t)r * 2 * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    dst[i] = fs[i];
    dst[H + i] = es[i];
  }
}

}  // namespace

extern "C" eagle_status eagle_draft_head_input(int B, int V, int k, int depth, int level, int H,
                                               const void* d_pool, size_t pool_bytes,
                                               const int32_t* d_node_prev, int32_t* d_node_cur,
                                               const void* d_feat_prev, const void* d_f_ctx,
                                               const int32_t* d_root_token, const void* d_emb,
                                               void* d_a, int* d_status, eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 1 && V >= 1 && H >= 1, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(k >= 1 && k <= EAGLE_MAX_TOPK && k <= V, EAGLE_ERR_UNSUPPORTED);
  EAGLE_HOST_CHECK(depth >= 1 && depth <= EAGLE_MAX_DEPTH && level >= 0 && level < depth,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(d_pool && d_node_cur && d_f_ctx && d_root_token && d_emb && d_a && d_status,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(level == 0 || (d_node_prev && d_feat_prev), EAGLE_ERR_INVALID_ARG);
  const PoolLayout L = pool_layout(B, k, depth, V);
  EAGLE_HOST_CHECK(pool_bytes >= L.total, EAGLE_ERR_WORKSPACE);
  const PoolPtrs pp = pool_ptrs(const_cast<void*>(d_pool), L);
  const int F = (level == 0) ? 1 : k;
  const int F_prev = (level <= 1) ? 1 : k;
  return launch_status(launch_pdl(
      head_input_kernel, dim3(B * F), dim3(256), 0, (cudaStream_t)stream, pp, k, L.P, H, level,
      F_prev, d_node_prev, d_node_cur, static_cast<const __nv_bfloat16*>(d_feat_prev),
      static_cast<const __nv_bfloat16*>(d_f_ctx), d_root_token,
      static_cast<const __nv_bfloat16*>(d_emb), V, static_cast<__nv_bfloat16*>(d_a), d_status));
}
