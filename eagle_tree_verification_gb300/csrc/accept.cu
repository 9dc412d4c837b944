// Acceptance walks of the tree-verify step.
//
// eagle_accept_greedy      [S4000] greedy-decoding paragraph; [EAGLE]
//                          speculative-sampling paragraph (alpha -> alpha+1).
// eagle_accept_stochastic  [S4000] random-decoding paragraph; [EAGLE]
//                          "多轮投机采样"; [EAGLE-2] §2 basic principle.
// (page titles are listed in include/eagle.h)
//
// The stochastic walk is sequential in the tree but every rejection needs a
// full-vocabulary pass (residual max(0, q - p) and its normaliser).  One
// thread-block cluster serves one sequence: the vocabulary row is split into
// `slice`-sized pieces, one per CTA, held in registers for the whole node,
// so each visited node's q and p rows are read from HBM exactly once and
// every rejection round runs out of registers.  Each round publishes its
// integer sums (and the tested token's values) through distributed shared
// memory: each CTA pushes its values into every CTA's shared memory, then
// one cluster barrier; every CTA then takes the identical
// decision (the data it decides on is bit-identical), so control flow stays
// uniform across the cluster without any spin-wait.
#include <math.h>

#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;
using namespace eagle;

namespace {

// Stochastic walk launch shapes.  Wide: 1024-thread CTAs, one per SM, at
// most 8 vocabulary entries per thread before the cluster doubles (the
// fastest per sequence).  Narrow: 512-thread CTAs, two per SM, at most 16
// entries per thread -- twice the sequences resident at once, each slower.
// Narrow in smaller clusters, for when the narrow clusters do not all fit:
// among the sizes down to half the narrow one whose clusters are all
// resident, the fewest entries per thread (a rejection round's cost follows
// them), then the fewest CTAs; if none fits, the most clusters resident.
// The wide shape is taken when every sequence's cluster is resident at once.
// (Measured at 16 sequences of V = 128256, one visited node and 8 rejection
// rounds each: wide 206.7 us in three waves of clusters of 16, narrow
// 195.0 us with 14 of 16 resident; clusters of 8 with 16 or 32 entries per
// thread 237.8 / 274.6 us; clusters of 12, all 16 resident, 24 entries per
// thread (21 used), 127.3 us with the later per-entry changes; clusters of
// 13 with 20 entries per thread (19.3 used), 114.1 us.)
constexpr int kWideThreads = 1024, kWidePrefer = 8;
constexpr int kNarrowThreads = 512, kNarrowPrefer = 16;
constexpr int kWalkMaxCluster = 16;
constexpr float kTwo40 = 1099511627776.0f;  // 2^40
constexpr float kTwo24 = 16777216.0f;       // 2^24

// ---------------------------------------------------------------------------
// greedy
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32)
accept_greedy_kernel(int max_nodes, const int* __restrict__ tree_off,
                     const int* __restrict__ parent, const int* __restrict__ tokens,
                     const int* __restrict__ argmax, int max_depth,
                     int* __restrict__ accept_len, int* __restrict__ accepted_nodes,
                     int* __restrict__ out_tokens, int* status) {
  pdl_begin();
  extern __shared__ int sm[];
  int* s_par = sm;
  int* s_tok = sm + max_nodes;
  const int b = blockIdx.x;
  const int lane = threadIdx.x;
  const int W = max_depth + 1;
  int* o_nodes = accepted_nodes + (size_t)b * W;
  int* o_tok = out_tokens + (size_t)b * W;
  for (int i = lane; i < W; i += 32) {
    o_nodes[i] = -1;
    o_tok[i] = -1;
  }
  const int t0 = tree_off[b];
  const int n = tree_off[b + 1] - t0;
  if (n < 1 || n > max_nodes) {
    if (lane == 0) {
      fail(status, EAGLE_ERR_INVALID_TREE);
      accept_len[b] = -1;
    }
    return;
  }
  bool bad = false;
  for (int i = lane; i < n; i += 32) {
    const int p = parent[t0 + i];
    s_par[i] = p;
    s_tok[i] = tokens[t0 + i];
    bad |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) {
      fail(status, EAGLE_ERR_INVALID_TREE);
      accept_len[b] = -1;
    }
    return;
  }
  __syncwarp();
  int cur = 0, alpha = 0;
  if (lane == 0) o_nodes[0] = 0;
  while (true) {
    const int want = argmax[t0 + cur];
    int found = -1;
    // children have larger indices than their parent (topological order)
    for (int base = cur + 1; base < n; base += 32) {
      const int i = base + lane;
      const bool m = (i < n) && s_par[i] == cur && s_tok[i] == want;
      const unsigned bal = __ballot_sync(0xffffffffu, m);
      if (bal) {
        found = base + __ffs(bal) - 1;
        break;
      }
    }
    if (found < 0) break;
    if (alpha + 1 > max_depth) {
      if (lane == 0) fail(status, EAGLE_ERR_INVALID_ARG);
      break;
    }
    if (lane == 0) {
      o_tok[alpha] = s_tok[found];
      o_nodes[alpha + 1] = found;
    }
    ++alpha;
    cur = found;
  }
  if (lane == 0) {
    o_tok[alpha] = argmax[t0 + cur];
    accept_len[b] = alpha;
  }
}

// ---------------------------------------------------------------------------
// stochastic
// ---------------------------------------------------------------------------
struct StochParams {
  int max_nodes, V, R, mode, max_depth, slice;
  const int* tree_off;
  const int* parent;
  const int* tokens;
  const float* q;          // probabilities, or logits when the walk normalises
  const float* row_lse;    // logits only: log-sum-exp of every row
  float temperature;       // logits only
  const float* p_rows;
  const int* p_row_of_node;
  const float* u_accept;
  const float* u_sample;
  int* accept_len;
  int* accepted_nodes;
  int* out_tokens;
  int* status;
};

__device__ __forceinline__ bool is_prob(float x) { return x >= 0.f && x <= 1.f; }



// Fixed-point weights.  For r in [0, 1], x = r * 2^40 is exact in fp32.
// W = trunc(x) as an integer, and fp32(W) rounded to nearest, computed with
// 32-bit operations only: below 2^23 x fits a 32-bit truncation; from 2^23
// on every fp32 value is an integer, so W = x and fp32(W) = x.
__device__ __forceinline__ unsigned long long fixed40_int(float r) {
  const float x = r * kTwo40;
  if (x < 8388608.f) return (unsigned long long)__float2uint_rz(x);
  const uint32_t bits = __float_as_uint(x);
  const int e = (int)(bits >> 23) - 127;                       // 23 .. 40
  const unsigned long long m = (bits & 0x7fffffu) | 0x800000u;
  return m << (e - 23);
}
// fp32(W) = trunc(x) itself: below 2^23 the truncation is exact in fp32,
// above it x is already an integer.
__device__ __forceinline__ float fixed40_f(float r) { return truncf(r * kTwo40); }

// Divisor of one rejection round: z, an estimate of 1/z and z/2.
struct RoundDiv {
  float z, rz, hz;
};
__device__ __forceinline__ RoundDiv round_div(float z) {
  return RoundDiv{z, (z > 0.f) ? __frcp_rn(z) : 0.f, 0.5f * z};
}

// x / z rounded to nearest, for finite x >= 0 and z > 0 with the quotient
// in [2^-64, 2^64] (here x, z < 2^41 are integers).  Markstein's correction
// of the reciprocal estimate (P. Markstein, IBM J. Res. Dev. 34(1), 1990):
// q0 = x * rz, then q1 = q0 + (x - q0 z) rz with fused multiply-adds.  q1 is
// kept only when the exact remainder r = x - q1 z (one fused multiply-add;
// exact because q1 is within an ulp of x/z) proves it is the nearest float:
// |r| < z ulp(q1) / 2, or z ulp(q1) / 4 when q1 is a power of two (the
// floats below it are half as far apart).  Anything else -- a tie, or an
// estimate that is not provably nearest -- goes to the IEEE division.
__device__ __forceinline__ float div_rn_by(float x, const RoundDiv& d) {
  if (x == 0.f) return 0.f;
  const float q0 = x * d.rz;
  const float q1 = fmaf(fmaf(-q0, d.z, x), d.rz, q0);
  const float r = fmaf(-q1, d.z, x);
  const uint32_t b = __float_as_uint(q1);
  const float ulp = __uint_as_float((b & 0x7f800000u) - (23u << 23));   // 2^(exponent - 23)
  const float lim = ((b & 0x7fffffu) == 0u) ? 0.5f * ulp * d.hz : ulp * d.hz;
  return (fabsf(r) < lim) ? q1 : __fdiv_rn(x, d.z);
}

// Two sums over the block at once; every thread gets both totals.  One
// barrier: the warps' partial sums go to s_tmp[par] (alternate the parity
// from one call to the next, so a call never overwrites partials another
// warp may still be reading), and every warp adds them up itself.
__device__ void block_sum2_u64(unsigned long long& a, unsigned long long& b,
                               unsigned long long (*s_tmp)[2][32], int par) {
  a = warp_sum_u64(a);
  b = warp_sum_u64(b);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    s_tmp[par][0][w] = a;
    s_tmp[par][1][w] = b;
  }
  __syncthreads();
  const int nw = blockDim.x >> 5;
  a = warp_sum_u64((l < nw) ? s_tmp[par][0][l] : 0ull);
  b = warp_sum_u64((l < nw) ? s_tmp[par][1][l] : 0ull);
}

// Exclusive scan over the block of one value per thread; returns the
// exclusive prefix, *total receives the block sum.  s_tmp: 33 entries.
__device__ unsigned long long block_excl_scan_u64(unsigned long long v, unsigned long long* s_tmp,
                                                  unsigned long long* total) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (l >= o) inc += y;
  }
  __syncthreads();
  if (l == 31) s_tmp[w] = inc;
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    unsigned long long t = (l < nw) ? s_tmp[l] : 0ull;
    unsigned long long ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, ti, o);
      if (l >= o) ti += y;
    }
    if (l < nw) s_tmp[l] = ti - t;  // exclusive prefix of warp totals
    if (l == 31) s_tmp[32] = ti;
  }
  __syncthreads();
  *total = s_tmp[32];
  return s_tmp[w] + inc - v;
}

// The tested token's target and draft values of one rejection round, kept
// by the CTA that owns the token (its sums go straight to every CTA).
struct RoundSlot {
  float qt, pt;           // q_k[t], p_k[t]
};

// One pass over this thread's slice entries.  UPD: the rejection update of
// token t_rej -- q <- fp32(W(max(0, q - p))) / zf (when the residual sum is
// positive), and in NO_REPLACE mode p <- fp32(W(p)) / spf with t_rej's entry
// zeroed; zf and spf are the weight sums rounded to fp32, and each quotient
// is one IEEE division (round to nearest).  SUMS (on the updated values): the residual weight sum, the draft
// weight sum without t_next, and q, p at t_next into `slot`.  One pass per
// rejection round, the same operations as an update followed by the sums.
// This thread's entries of the draft row: in registers, or (SMEM) in shared
// memory at sm[e * THREADS] (element e of the thread), which keeps a narrow
// CTA's 16 entries per thread within the registers of two CTAs per SM.
template <int E, int THREADS, bool SMEM>
struct DraftSlice {
  float reg[SMEM ? 1 : E];
  float* sm;
  __device__ __forceinline__ float get(int e) const {
    if constexpr (SMEM) return sm[e * THREADS];
    else return reg[e];
  }
  __device__ __forceinline__ void set(int e, float v) {
    if constexpr (SMEM) sm[e * THREADS] = v;
    else reg[e] = v;
  }
};

__host__ __device__ constexpr bool draft_in_smem(int e, int threads) {
  return threads == kNarrowThreads || e == 16;
}

// Entries per thread the walk kernel is built for: the smallest that holds e.
__host__ __device__ constexpr int walk_elems(int e) {
  return e <= 4 ? 4 : e <= 8 ? 8 : e <= 16 ? 16 : e <= 20 ? 20 : e <= 24 ? 24 : 32;
}
constexpr int kWalkElemKinds = 6;
__host__ __device__ constexpr int walk_elems_index(int E) {
  return E == 4 ? 0 : E == 8 ? 1 : E == 16 ? 2 : E == 20 ? 3 : E == 24 ? 4 : 5;
}

template <int E, int THREADS, bool UPD, bool SUMS, bool SMEM>
__device__ __forceinline__ void walk_pass(float (&q)[E], DraftSlice<E, THREADS, SMEM>& p, int v0, int nv,
                                          bool no_replace, int t_rej, const RoundDiv& zf,
                                          const RoundDiv& spf,
                                          bool z_pos, int t_next, unsigned long long& sw,
                                          unsigned long long& sp, RoundSlot& slot) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = tid + e * THREADS;
    float pe = p.get(e);
    if (UPD) {
      const float qa = q[e], pa = pe;
      if (z_pos) q[e] = div_rn_by(fixed40_f(fmaxf(0.f, __fsub_rn(qa, pa))), zf);
      if (no_replace) {
        pe = (v0 + i == t_rej) ? 0.f : (spf.z > 0.f ? div_rn_by(fixed40_f(pa), spf) : 0.f);
        p.set(e, pe);
      }
    }
    if (SUMS) {
      sw += fixed40_int(fmaxf(0.f, __fsub_rn(q[e], pe)));
      if (no_replace && v0 + i != t_next) sp += fixed40_int(pe);
      if (i < nv && v0 + i == t_next) {
        slot.qt = q[e];
        slot.pt = pe;
      }
    }
  }
}

// Element e of thread `tid` is vocabulary entry v0 + tid + THREADS*e.
// LOGITS: P.q holds logits; each visited row is normalised as it is loaded,
// by the LM head's probability-mode expression.
template <int E, bool LOGITS, int THREADS>
__global__ void __launch_bounds__(THREADS, THREADS == kWideThreads ? 1 : 2)
accept_stochastic_kernel(const StochParams P) {
  pdl_begin();
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  const unsigned CS = cluster.num_blocks();
  const int b = blockIdx.x / CS;
  const int tid = threadIdx.x, lane = tid & 31;

  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* s_q = reinterpret_cast<float*>(smem_raw);            // slice, for sampling
  int* s_par = reinterpret_cast<int*>(s_q + P.slice);
  int* s_tok = s_par + P.max_nodes;
  int* s_kids = s_tok + P.max_nodes;
  float* s_ua = reinterpret_cast<float*>(s_kids + P.max_nodes);   // u_accept of each child
  // narrow CTAs and 16 entries per thread: the draft row's entries in
  // shared memory, E per thread (16-byte aligned)
  constexpr bool kPSmem = draft_in_smem(E, THREADS);
  float* s_p = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(s_ua + P.max_nodes) + 15) & ~(uintptr_t)15);
  __shared__ unsigned long long s_red[66];
  __shared__ unsigned long long s_sum2[2][2][32];   // block_sum2_u64 partials, by round parity
  __shared__ RoundSlot s_slot[2];            // double-buffered by round parity
  // What every CTA of the cluster pushed here, by round parity: its sums,
  // the tested token's q and p (from the CTA that owns the token), and for
  // the bonus token its total weight.  Pushing before the cluster barrier
  // leaves only local reads after it.
  __shared__ unsigned long long s_all[2][16][2];
  __shared__ float s_test[2][2];
  __shared__ unsigned long long s_tots[16];
  __shared__ int s_flag, s_nk;

  const int v0 = (int)rank * P.slice;
  const int nv = max(0, min(P.V, v0 + P.slice) - v0);
  const int W = P.max_depth + 1;
  const bool writer = (rank == 0);
  int* o_nodes = P.accepted_nodes + (size_t)b * W;
  int* o_tok = P.out_tokens + (size_t)b * W;
  if (writer) {
    for (int i = tid; i < W; i += blockDim.x) {
      o_nodes[i] = -1;
      o_tok[i] = -1;
    }
  }
  const int t0 = P.tree_off[b];
  const int n = P.tree_off[b + 1] - t0;
  // All checks below read the same global data in every CTA, so the early
  // exits are taken by the whole cluster together.
  if (n < 1 || n > P.max_nodes) {
    if (writer && tid == 0) {
      fail(P.status, EAGLE_ERR_INVALID_TREE);
      P.accept_len[b] = -1;
    }
    return;
  }
  if (tid == 0) s_flag = 0;
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) {
    const int pp = P.parent[t0 + i];
    const int tk = P.tokens[t0 + i];
    s_par[i] = pp;
    s_tok[i] = tk;
    if ((i == 0) ? (pp != -1) : (pp < 0 || pp >= i)) atomicOr(&s_flag, 1);
    if (i > 0 && (tk < 0 || tk >= P.V)) atomicOr(&s_flag, 2);
  }
  __syncthreads();
  if (s_flag) {
    if (writer && tid == 0) {
      fail(P.status, (s_flag & 1) ? EAGLE_ERR_INVALID_TREE : EAGLE_ERR_INVALID_ARG);
      P.accept_len[b] = -1;
    }
    return;
  }

  const bool no_replace = (P.mode == EAGLE_SAMPLE_NO_REPLACE);
  float q[E];
  DraftSlice<E, THREADS, kPSmem> p;
  p.sm = s_p + tid;
  int cur = 0, alpha = 0, par = 0;
  bool stop = false;
  if (writer && tid == 0) o_nodes[0] = 0;

  while (true) {
    // every warp has read the previous node's child list before it is
    // rewritten
    __syncthreads();
    // children of cur in index order, by warp 0 (children follow their
    // parent: only indices past cur are looked at)
    if (tid < 32) {
      int c = 0;
      for (int base = cur + 1; base < n; base += 32) {
        const int i = base + tid;
        const bool kid = (i < n) && s_par[i] == cur;
        const unsigned bal = __ballot_sync(0xffffffffu, kid);
        if (kid) {
          // the child's acceptance uniform comes along: no global load in a round
          const int pos = c + __popc(bal & ((1u << tid) - 1u));
          s_kids[pos] = i;
          s_ua[pos] = P.u_accept[t0 + i];
        }
        c += __popc(bal);
      }
      if (tid == 0) s_nk = c;
    }
    __syncthreads();
    const int nk = s_nk;
    int prow = 0;
    if (nk > 0) {
      prow = P.p_row_of_node[t0 + s_kids[0]];
      if (prow < 0 || prow >= P.R) {  // uniform
        if (writer && tid == 0) fail(P.status, EAGLE_ERR_INVALID_ARG);
        stop = true;
        break;
      }
    }
    // this CTA's slice of q[cur] (and of the draft row) into registers
    {
      const float* qrow = P.q + (size_t)(t0 + cur) * P.V + v0;
      const float* prw = P.p_rows + (size_t)prow * P.V + v0;
      const ProbScales sc = prob_scales(P.temperature, LOGITS ? __ldg(P.row_lse + t0 + cur) : 0.f);
      int bad = 0;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int i = tid + e * THREADS;
        q[e] = 0.f;
        p.set(e, 0.f);
        if (i < nv) {
          q[e] = __ldg(qrow + i);
          if (LOGITS) q[e] = prob_from_logit(q[e], sc);
          bad |= !is_prob(q[e]);
          if (nk > 0) {
            const float pv = __ldg(prw + i);
            p.set(e, pv);
            bad |= !is_prob(pv);
          }
        }
      }
      if (__syncthreads_or(bad) && tid == 0) fail(P.status, EAGLE_ERR_NUMERIC);
    }

    // the cluster's totals for one round: residual and draft weight sums,
    // and q, p at the tested token (from the CTA that owns it)
    unsigned long long Z = 0, SP = 0;
    float qt = 0.f, pt = 0.f;
    auto reduce_round = [&](unsigned long long sw, unsigned long long sp, int t) {
      block_sum2_u64(sw, sp, s_sum2, par);
      const unsigned owner = (unsigned)(t / P.slice);
      if (tid < (int)CS) {
        unsigned long long* d = cluster.map_shared_rank(&s_all[par][rank][0], (unsigned)tid);
        d[0] = sw;
        d[1] = sp;
        if (owner == rank) {
          float* dt = cluster.map_shared_rank(&s_test[par][0], (unsigned)tid);
          dt[0] = s_slot[par].qt;
          dt[1] = s_slot[par].pt;
        }
      }
      cluster.sync();
      // every warp adds the CTAs' sums itself: no barrier after the reads
      unsigned long long a = 0, bb = 0;
      if (lane < (int)CS) {
        a = s_all[par][lane][0];
        bb = s_all[par][lane][1];
      }
      Z = warp_sum_u64(a);
      SP = warp_sum_u64(bb);
      qt = s_test[par][0];
      pt = s_test[par][1];
      par ^= 1;
    };
    if (nk > 0) {
      // sums as if the first child were rejected, and its tested values
      unsigned long long sw = 0, sp = 0;
      const int t = s_tok[s_kids[0]];
      const RoundDiv none{0.f, 0.f, 0.f};
      walk_pass<E, THREADS, false, true, kPSmem>(q, p, v0, nv, no_replace, -1, none, none, false, t,
                                                 sw, sp, s_slot[par]);
      reduce_round(sw, sp, t);
    }
    bool moved = false;
    for (int j = 0; j < nk; ++j) {
      const int c = s_kids[j];
      const int t = s_tok[c];
      const float ua = s_ua[j];
      if (!(ua >= 0.f && ua < 1.f) && writer && tid == 0) fail(P.status, EAGLE_ERR_INVALID_ARG);
      // exact: a product of two fp32 values is exact in fp64.  (fp64 and
      // 64-bit integer conversions run on a narrow pipe: one lane of each
      // warp evaluates them and the warp shares the result.)
      const bool accept =
          __shfl_sync(0xffffffffu, lane == 0 ? (double)ua * (double)pt < (double)qt : false, 0);
      if (accept) {
        if (alpha + 1 > P.max_depth) {
          if (writer && tid == 0) fail(P.status, EAGLE_ERR_INVALID_ARG);
          stop = true;
          break;
        }
        if (writer && tid == 0) {
          o_tok[alpha] = t;
          o_nodes[alpha + 1] = c;
        }
        ++alpha;
        cur = c;
        moved = true;
        break;
      }
      // rejected: q_{k+1} = fp32(W) / fp32(Z), p_{k+1} likewise
      // (NO_REPLACE); every operation rounds to nearest once
      float zf = 0.f, spf = 0.f;
      if (lane == 0) {
        zf = (Z > 0ull) ? __ull2float_rn(Z) : 0.f;
        spf = (SP > 0ull) ? __ull2float_rn(SP) : 0.f;
      }
      zf = __shfl_sync(0xffffffffu, zf, 0);
      spf = __shfl_sync(0xffffffffu, spf, 0);
      const RoundDiv zd = round_div(zf), spd = round_div(spf);
      if (j + 1 < nk) {
        // update, and the next child's sums, in one pass
        unsigned long long sw = 0, sp = 0;
        const int tn = s_tok[s_kids[j + 1]];
        walk_pass<E, THREADS, true, true, kPSmem>(q, p, v0, nv, no_replace, t, zd, spd, Z > 0ull, tn,
                                                  sw, sp, s_slot[par]);
        reduce_round(sw, sp, tn);
      } else {
        unsigned long long sw = 0, sp = 0;
        walk_pass<E, THREADS, true, false, kPSmem>(q, p, v0, nv, no_replace, t, zd, spd, Z > 0ull, -1,
                                                   sw, sp, s_slot[par]);
      }
    }
    if (moved) continue;
    if (stop) break;

    // Bonus token: inverse CDF of the current q over integer weights.
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = tid + e * THREADS;
      if (i < nv) s_q[i] = q[e];
    }
    __syncthreads();
    {
      const int per = (nv + (int)blockDim.x - 1) / (int)blockDim.x;
      const int c0 = min(nv, tid * per), c1 = min(nv, c0 + per);
      unsigned long long mine = 0;
      // a rotated start keeps the lanes of a warp on different banks
      const int len = c1 - c0;
      for (int j = 0; j < len; ++j) mine += fixed40_int(s_q[c0 + (j + tid) % len]);
      unsigned long long cta_total;
      const unsigned long long excl = block_excl_scan_u64(mine, s_red, &cta_total);
      if (tid < (int)CS) *cluster.map_shared_rank(&s_tots[rank], (unsigned)tid) = cta_total;
      cluster.sync();
      unsigned long long all = 0, bef = 0;
      if (lane < (int)CS) {
        all = s_tots[lane];
        bef = (lane < (int)rank) ? all : 0ull;
      }
      const unsigned long long Z = warp_sum_u64(all);
      const unsigned long long before = warp_sum_u64(bef);
      const float us = P.u_sample[t0 + cur];
      if (!(us >= 0.f && us < 1.f)) {
        if (writer && tid == 0) fail(P.status, EAGLE_ERR_INVALID_ARG);
      } else if (Z == 0ull) {
        if (writer && tid == 0) fail(P.status, EAGLE_ERR_NUMERIC);
      } else {
        const unsigned long long U = (unsigned long long)__float2uint_rz(us * kTwo24);
        const unsigned long long lo = U * Z;
        const unsigned long long hi = __umul64hi(U, Z);
        const unsigned long long target = (hi << 40) | (lo >> 24);
        if (target >= before && target < before + cta_total) {
          const unsigned long long local = target - before;
          if (local >= excl && local < excl + mine) {
            unsigned long long acc = excl;
            for (int i = c0; i < c1; ++i) {
              acc += fixed40_int(s_q[i]);
              if (acc > local) {
                o_tok[alpha] = v0 + i;
                break;
              }
            }
          }
        }
      }
    }
    break;
  }
  if (writer && tid == 0) P.accept_len[b] = alpha;
  // Keep this CTA's shared memory alive until every DSMEM read has finished.
  cluster.sync();
}

// Cluster size and per-thread element count for a vocabulary: the smallest
// cluster (up to 16 CTAs) whose slices need at most `prefer` entries per
// thread, at most 32.
int pick_cluster(int V, int threads, int prefer, int* slice_out, int* elems_out) {
  for (int cs = 1; cs <= kWalkMaxCluster; cs <<= 1) {
    int slice = (V + cs - 1) / cs;
    slice = (slice + 3) & ~3;
    const int e = (slice + threads - 1) / threads;
    if (e > prefer && cs < kWalkMaxCluster) continue;
    if (e > 32) return -1;
    *slice_out = slice;
    *elems_out = walk_elems(e);
    return cs;
  }
  return -1;
}

// The same with a given cluster size (0 if a slice needs more than 32
// entries per thread).
int fixed_cluster(int V, int threads, int cs, int* slice_out, int* elems_out) {
  int slice = (V + cs - 1) / cs;
  slice = (slice + 3) & ~3;
  const int e = (slice + threads - 1) / threads;
  if (e > 32) return 0;
  *slice_out = slice;
  *elems_out = walk_elems(e);
  return cs;
}


}  // namespace

extern "C" eagle_status eagle_accept_greedy(int B, int max_nodes, const int32_t* d_tree_off,
                                            const int32_t* d_parent, const int32_t* d_tokens,
                                            const int32_t* d_argmax, int max_depth,
                                            int32_t* d_accept_len, int32_t* d_accepted_nodes,
                                            int32_t* d_out_tokens, int* d_status,
                                            eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 0 && max_depth >= 0, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(max_nodes >= 1 && max_nodes <= EAGLE_MAX_TREE_NODES, EAGLE_ERR_UNSUPPORTED);
  if (B == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_tree_off && d_parent && d_tokens && d_argmax && d_accept_len &&
                       d_accepted_nodes && d_out_tokens && d_status,
                   EAGLE_ERR_INVALID_ARG);
  const size_t smem = (size_t)max_nodes * 2 * sizeof(int);
  return launch_status(launch_pdl(accept_greedy_kernel, dim3(B), dim3(32), smem,
                                  (cudaStream_t)stream, max_nodes, d_tree_off, d_parent,
                                  d_tokens, d_argmax, max_depth, d_accept_len, d_accepted_nodes,
                                  d_out_tokens, d_status));
}

namespace {

// Clusters of `cs` CTAs of `kern` resident on the current GPU at once (0 if
// the query fails), cached per device and configuration.
int resident_clusters(const void* kern, int threads, int cs, size_t smem) {
  struct Entry {
    const void* kern;
    int dev, cs;
    size_t smem;
    int n;
  };
  static std::mutex mu;
  // (up to ten shapes are looked at per vocabulary size, tree size and mode)
  constexpr int kCache = 128;
  static Entry cache[kCache];
  static int used = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].kern == kern && cache[i].dev == dev && cache[i].cs == cs && cache[i].smem == smem)
      return cache[i].n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cs, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (used < kCache) cache[used++] = Entry{kern, dev, cs, smem, n};
  return n;
}

#ifdef EAGLE_WALK_DIV_TEST
// Test build only: out[i] = div_rn_by(x[i], z[i]), to compare with the
// IEEE division on many operand pairs.
__global__ void walk_div_test_kernel(const float* x, const float* z, float* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = div_rn_by(x[i], round_div(z[i]));
}
#endif

// Both stochastic entry points: d_q holds probabilities, or logits with
// row_lse and temperature (LOGITS).
eagle_status launch_stochastic(bool logits, int B, int max_nodes, int V, int R, int mode,
                               const int32_t* d_tree_off, const int32_t* d_parent,
                               const int32_t* d_tokens, const float* d_q, const float* d_row_lse,
                               float temperature, const float* d_p_rows,
                               const int32_t* d_p_row_of_node, const float* d_u_accept,
                               const float* d_u_sample, int max_depth, int32_t* d_accept_len,
                               int32_t* d_accepted_nodes, int32_t* d_out_tokens, int* d_status,
                               eagle_stream_t stream) {
  EAGLE_HOST_CHECK(B >= 0 && V >= 1 && R >= 0 && max_depth >= 0, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(mode == EAGLE_SAMPLE_REPLACE || mode == EAGLE_SAMPLE_NO_REPLACE,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(!logits || (temperature > 0.f && isfinite(temperature)),
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(max_nodes >= 1 && max_nodes <= EAGLE_MAX_TREE_NODES, EAGLE_ERR_UNSUPPORTED);
  if (B == 0) return EAGLE_OK;
  EAGLE_HOST_CHECK(d_tree_off && d_parent && d_tokens && d_q && d_u_accept && d_u_sample &&
                       d_p_row_of_node && d_accept_len && d_accepted_nodes && d_out_tokens &&
                       d_status,
                   EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(!logits || d_row_lse, EAGLE_ERR_INVALID_ARG);
  EAGLE_HOST_CHECK(R == 0 || d_p_rows, EAGLE_ERR_INVALID_ARG);
  using Kern = void (*)(const StochParams);
  // shapes: 0 wide; 1 narrow; 2 narrow in smaller clusters (more entries
  // per thread, more clusters resident)
#define EAGLE_WALK_KERNS(L, T)                                                              \
  {accept_stochastic_kernel<4, L, T>,  accept_stochastic_kernel<8, L, T>,                  \
   accept_stochastic_kernel<16, L, T>, accept_stochastic_kernel<20, L, T>,                 \
   accept_stochastic_kernel<24, L, T>, accept_stochastic_kernel<32, L, T>}
  static const Kern kerns[2][2][kWalkElemKinds] = {
      {EAGLE_WALK_KERNS(false, kWideThreads), EAGLE_WALK_KERNS(true, kWideThreads)},
      {EAGLE_WALK_KERNS(false, kNarrowThreads), EAGLE_WALK_KERNS(true, kNarrowThreads)}};
#undef EAGLE_WALK_KERNS
  static PerDeviceOnce attr_once[2][2][kWalkElemKinds];
  // a shape's cluster size, slice, kernel and shared memory, attributes set
  struct Shape {
    int cs, slice, threads, elems;
    Kern kern;
    size_t smem;
  };
  // kind 2: the narrow shape with `cs2` CTAs per cluster
  auto shape = [&](int kind, Shape* sh, int cs2 = 0) -> eagle_status {
    int elems = 0;
    const int narrow = kind > 0 ? 1 : 0;
    sh->threads = narrow ? kNarrowThreads : kWideThreads;
    if (kind == 2)
      sh->cs = fixed_cluster(V, sh->threads, cs2, &sh->slice, &elems);
    else
      sh->cs = pick_cluster(V, sh->threads, narrow ? kNarrowPrefer : kWidePrefer, &sh->slice,
                            &elems);
    if (sh->cs <= 0) return EAGLE_ERR_UNSUPPORTED;
    sh->elems = elems;
    sh->smem = (size_t)sh->slice * sizeof(float) + (size_t)max_nodes * 4 * sizeof(int) +
               (draft_in_smem(elems, sh->threads) ? (size_t)elems * sh->threads * sizeof(float) + 16
                                                  : 0);
    const int ai = walk_elems_index(elems);
    sh->kern = kerns[narrow][logits ? 1 : 0][ai];
    const Kern kern = sh->kern;
    if (attr_once[narrow][logits ? 1 : 0][ai].run([&] {
          cudaError_t e =
              cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
          if (e != cudaSuccess) return e;
          // room for two CTAs' slices side by side
          if (narrow)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
          if (e != cudaSuccess) return e;
          return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      160 * 1024);
        }) != cudaSuccess)
      return EAGLE_ERR_CUDA;
    return EAGLE_OK;
  };
  // the first shape whose clusters are all resident at once, else the one
  // with the most resident
  Shape sh;
  eagle_status st = shape(0, &sh);
  if (st != EAGLE_OK) return st;
  if (B > 1 && sh.cs > 1) {
    int best_n = resident_clusters((const void*)sh.kern, sh.threads, sh.cs, sh.smem);
    Shape c;
    if (B > best_n && shape(1, &c) == EAGLE_OK) {
      const int n = resident_clusters((const void*)c.kern, c.threads, c.cs, c.smem);
      if (n > best_n) {
        best_n = n;
        sh = c;
      }
      // smaller narrow clusters: the fewest entries per thread (a rejection
      // round's cost follows them) among the sizes whose clusters are all
      // resident; if none is, the most resident
      if (B > best_n && c.cs >= 4) {
        int found = 0;
        for (int cs2 = c.cs - 1; cs2 >= (c.cs + 1) / 2; --cs2) {
          Shape d;
          if (shape(2, &d, cs2) != EAGLE_OK) continue;
          const int nd = resident_clusters((const void*)d.kern, d.threads, d.cs, d.smem);
          if (nd >= B) {
            if (!found || d.elems < sh.elems || (d.elems == sh.elems && d.cs < sh.cs)) sh = d;
            found = 1;
          } else if (!found && nd > best_n) {
            best_n = nd;
            sh = d;
          }
        }
      }
    }
  }
  StochParams P;
  P.max_nodes = max_nodes;
  P.V = V;
  P.R = R;
  P.mode = mode;
  P.max_depth = max_depth;
  P.slice = sh.slice;
  P.tree_off = d_tree_off;
  P.parent = d_parent;
  P.tokens = d_tokens;
  P.q = d_q;
  P.row_lse = d_row_lse;
  P.temperature = temperature;
  P.p_rows = d_p_rows;
  P.p_row_of_node = d_p_row_of_node;
  P.u_accept = d_u_accept;
  P.u_sample = d_u_sample;
  P.accept_len = d_accept_len;
  P.accepted_nodes = d_accepted_nodes;
  P.out_tokens = d_out_tokens;
  P.status = d_status;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * sh.cs), 1, 1);
  cfg.blockDim = dim3((unsigned)sh.threads, 1, 1);
  cfg.dynamicSmemBytes = sh.smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)sh.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return launch_status(cudaLaunchKernelEx(&cfg, sh.kern, P));
}

}  // namespace

extern "C" eagle_status eagle_accept_stochastic(
    int B, int max_nodes, int V, int R, int mode, const int32_t* d_tree_off,
    const int32_t* d_parent, const int32_t* d_tokens, const float* d_q, const float* d_p_rows,
    const int32_t* d_p_row_of_node, const float* d_u_accept, const float* d_u_sample,
    int max_depth, int32_t* d_accept_len, int32_t* d_accepted_nodes, int32_t* d_out_tokens,
    int* d_status, eagle_stream_t stream) {
  return launch_stochastic(false, B, max_nodes, V, R, mode, d_tree_off, d_parent, d_tokens, d_q,
                           nullptr, 1.f, d_p_rows, d_p_row_of_node, d_u_accept, d_u_sample,
                           max_depth, d_accept_len, d_accepted_nodes, d_out_tokens, d_status,
                           stream);
}

extern "C" eagle_status eagle_accept_stochastic_logits(
    int B, int max_nodes, int V, int R, int mode, const int32_t* d_tree_off,
    const int32_t* d_parent, const int32_t* d_tokens, const float* d_z, const float* d_row_lse,
    float temperature, const float* d_p_rows, const int32_t* d_p_row_of_node,
    const float* d_u_accept, const float* d_u_sample, int max_depth, int32_t* d_accept_len,
    int32_t* d_accepted_nodes, int32_t* d_out_tokens, int* d_status, eagle_stream_t stream) {
  return launch_stochastic(true, B, max_nodes, V, R, mode, d_tree_off, d_parent, d_tokens, d_z,
                           d_row_lse, temperature, d_p_rows, d_p_row_of_node, d_u_accept,
                           d_u_sample, max_depth, d_accept_len, d_accepted_nodes, d_out_tokens,
                           d_status, stream);
}

#ifdef EAGLE_WALK_DIV_TEST
extern "C" EAGLE_API int eagle_test_walk_div(const float* d_x, const float* d_z, float* d_out, int n,
                                             eagle_stream_t stream) {
  if (n <= 0) return 0;
  walk_div_test_kernel<<<(n + 255) / 256, 256, 0, (cudaStream_t)stream>>>(d_x, d_z, d_out, n);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}
#endif
