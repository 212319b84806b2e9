// Online calibration of the sparse candidate tree on the GPU.
//
// Paper review ("Medusa: Simple LLM Inference Acceleration Framework with
// Multiple Decoding Heads"), section "方法细节": the sparse tree is built from
// the per-head top-i accuracies measured on calibration data, adding nodes
// greedily by their contribution to the expected acceptance length.  Here the
// accuracies are measured on the verify steps themselves and the tree is
// rebuilt on the device:
//   medusa_accept_stats            counts, per (head, rank), the candidates
//                                  tested (parent accepted) and accepted (kept
//                                  on the accepted path);
//   medusa_acc_update              folds the counts into the accuracy table
//                                  (the old table weighs as pseudo-counts);
//   medusa_topology_greedy_device  greedy sparse tree from the table, written
//                                  in the device layout the other calls read.
#include <math.h>

#include "common.cuh"
#include "host_util.h"

namespace medusa {

constexpr int kStatThreads = 256;  // >= MEDUSA_MAX_NODES
constexpr int kGreedyThreads = 256;

// ------------------------------------------------------------------ statistics

// Grid B.  Thread n >= 1 tests node n against row b's accepted path.
__global__ void __launch_bounds__(kStatThreads)
accept_stats_kernel(const int32_t* __restrict__ path_nodes, const int32_t* __restrict__ accept_len,
                    const int32_t* __restrict__ parent, const int32_t* __restrict__ depth,
                    const int32_t* __restrict__ rank, int N, int Dmax, int R,
                    unsigned long long* __restrict__ tested, unsigned long long* __restrict__ accepted,
                    int32_t* d_status) {
  __shared__ int path[MEDUSA_MAX_DEPTH + 1];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, n = threadIdx.x;
  const int A = accept_len[b];
  const bool ok = A >= 1 && A <= Dmax + 1;
  if (!ok) {
    if (n == 0) set_status(d_status, MEDUSA_DEV_BAD_INDEX);
    return;
  }
  if (n <= Dmax) path[n] = n < A ? path_nodes[(size_t)b * (Dmax + 1) + n] : -1;
  __syncthreads();
  if (n < 1 || n >= N) return;
  const int d = depth[n], r = rank[n];
  if (d < 1 || d > Dmax || r < 0 || r >= R) {
    set_status(d_status, MEDUSA_DEV_BAD_TOPOLOGY);
    return;
  }
  if (d - 1 < A && parent[n] == path[d - 1]) {
    atomicAdd(&tested[(size_t)(d - 1) * R + r], 1ull);
    if (d < A && path[d] == n) atomicAdd(&accepted[(size_t)(d - 1) * R + r], 1ull);
  }
}

// acc = (accepted + w acc) / (tested + w) per entry, each operation rounded on
// its own (no contraction); entries with tested + w == 0 keep their value.
__global__ void acc_update_kernel(double* __restrict__ acc, const unsigned long long* __restrict__ tested,
                                  const unsigned long long* __restrict__ accepted, int n, double w) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const double den = __dadd_rn((double)tested[i], w);
  if (den > 0.0) acc[i] = __ddiv_rn(__dadd_rn((double)accepted[i], __dmul_rn(w, acc[i])), den);
}

// ------------------------------------------------------------------ greedy tree

typedef unsigned __int128 u128;

// Canonical key of a tree path: (length << 80) | ranks, 5 bits per level with
// the first level most significant (R <= 32, depth <= 16).  Keys order like
// the canonical order: shorter paths first, then lexicographic.
__device__ __forceinline__ u128 child_key(u128 parent_key, int parent_len, int r) {
  return parent_key + ((u128)1 << 80) + ((u128)(unsigned)r << (5 * (MEDUSA_MAX_DEPTH - 1 - parent_len)));
}
__device__ __forceinline__ int key_rank(u128 key, int level) {
  return (int)((key >> (5 * (MEDUSA_MAX_DEPTH - 1 - level))) & 31u);
}

struct GreedyState {
  u128 key[MEDUSA_MAX_NODES];       // canonical key of chosen node i
  double score[MEDUSA_MAX_NODES];
  double best_sc[MEDUSA_MAX_NODES]; // best not-yet-chosen child of chosen node i: score
  int len[MEDUSA_MAX_NODES];
  uint32_t kids[MEDUSA_MAX_NODES];  // bit r: child with rank r already chosen
  int pchosen[MEDUSA_MAX_NODES];    // chosen index of the parent
  int canon[MEDUSA_MAX_NODES];      // canonical index of chosen node i
  int best_r[MEDUSA_MAX_NODES];     // and its rank (-1: none left)
  double acc[MEDUSA_MAX_DEPTH * MEDUSA_MAX_TOPK];
};

// A frontier candidate: child of chosen node a with rank r (a < 0: none).
struct Cand {
  double sc;
  u128 key;
  int a, r;
};

// Greedy preference of candidate x over y: scores within a relative 1e-12 are
// ties, broken by canonical order (the key).
//
// Scores are products of table entries in [0, 1], so non-negative: their bit
// patterns order like their values, and the integer distance d of the patterns
// counts units in the last place.  Two normal doubles d ulps apart differ by at
// most d 2^-52 and (within a factor of two of each other) at least d 2^-54 of
// the larger, so d <= 4000 is always inside the 1e-12 window and d >= 20000
// always outside; only the band between, zeros and subnormals take the double
// test (double arithmetic is slow on this GPU; the outcome is the same).
__device__ __forceinline__ bool beats(const Cand& x, const Cand& y) {
  if (y.a < 0) return x.a >= 0;
  if (x.a < 0) return false;
  const long long ia = __double_as_longlong(x.sc), ib = __double_as_longlong(y.sc);
  const long long d = ia > ib ? ia - ib : ib - ia;
  bool tie;
  if ((ia >> 52) == 0 || (ib >> 52) == 0 || (d > 4000 && d < 20000))
    tie = fabs(x.sc - y.sc) <= 1e-12 * fmax(fabs(x.sc), fabs(y.sc));
  else
    tie = d <= 4000;
  if (tie) return x.key < y.key;
  return ia > ib;
}

__device__ __forceinline__ u128 shfl_xor_u128(u128 v, int o) {
  const unsigned long long lo = (unsigned long long)v, hi = (unsigned long long)(v >> 64);
  return ((u128)__shfl_xor_sync(0xffffffffu, hi, o) << 64) | __shfl_xor_sync(0xffffffffu, lo, o);
}
__device__ __forceinline__ u128 shfl_u128(u128 v, int src) {
  const unsigned long long lo = (unsigned long long)v, hi = (unsigned long long)(v >> 64);
  return ((u128)__shfl_sync(0xffffffffu, hi, src) << 64) | __shfl_sync(0xffffffffu, lo, src);
}

// Warp argmax under `beats`; lane 0's winner is the result, broadcast.
__device__ __forceinline__ void warp_best(Cand& c) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    Cand y;
    y.sc = __shfl_xor_sync(0xffffffffu, c.sc, o);
    y.key = shfl_xor_u128(c.key, o);
    y.a = __shfl_xor_sync(0xffffffffu, c.a, o);
    y.r = __shfl_xor_sync(0xffffffffu, c.r, o);
    if (beats(y, c)) c = y;
  }
  c.sc = __shfl_sync(0xffffffffu, c.sc, 0);
  c.key = shfl_u128(c.key, 0);
  c.a = __shfl_sync(0xffffffffu, c.a, 0);
  c.r = __shfl_sync(0xffffffffu, c.r, 0);
}

// One warp: the best child of chosen node a that is not chosen yet (lane = rank).
__device__ __forceinline__ void refresh_best_child(GreedyState& s, int a, int K, int R, int lane) {
  Cand c;
  c.sc = 0.0;
  c.key = 0;
  c.a = -1;
  c.r = -1;
  const int la = s.len[a];
  if (lane < R && la < K && !((s.kids[a] >> lane) & 1u)) {
    c.sc = s.score[a] * s.acc[la * R + lane];
    c.key = child_key(s.key[a], la, lane);
    c.a = a;
    c.r = lane;
  }
  warp_best(c);
  if (lane == 0) {
    s.best_sc[a] = c.sc;
    s.best_r[a] = c.r;
  }
}

// One CTA.  Device buffer: parent[n], depth[n], rank[n], retrieve[n][K + 1].
// meta = {n_nodes, max_depth, n_leaves, max_rank}.
__global__ void __launch_bounds__(kGreedyThreads)
greedy_tree_kernel(const double* __restrict__ acc_in, int K, int R, int n_nodes, int32_t* __restrict__ out,
                   int32_t* __restrict__ meta, int32_t* d_status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GreedyState& s = *reinterpret_cast<GreedyState*>(smem_raw);
  __shared__ int s_bad;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int i = tid; i < K * R; i += kGreedyThreads) {
    double v = acc_in[i];
    if (!(v >= 0.0 && v <= 1.0)) {  // NaN or out of [0, 1]: clamped and reported
      s_bad = 1;
      v = v > 1.0 ? 1.0 : 0.0;
    }
    s.acc[i] = v;
  }
  if (tid == 0) {
    s.key[0] = 0;
    s.len[0] = 0;
    s.score[0] = 1.0;
    s.kids[0] = 0u;
    s.pchosen[0] = -1;
  }
  __syncthreads();
  if (tid == 0 && s_bad) set_status(d_status, MEDUSA_DEV_BAD_INDEX);

  // Greedy growth, one warp.  Every chosen node keeps its best child not chosen
  // yet; a round takes the best of those (the frontier's best under `beats`),
  // adds it, and refreshes the best child of the new node and of its parent.
  if (warp == 0) {
    refresh_best_child(s, 0, K, R, lane);
    __syncwarp();
    for (int c = 1; c < n_nodes; ++c) {
      Cand best;
      best.sc = 0.0;
      best.key = 0;
      best.a = -1;
      best.r = -1;
      for (int a = lane; a < c; a += 32) {
        Cand x;
        x.r = s.best_r[a];
        if (x.r < 0) continue;
        x.sc = s.best_sc[a];
        x.key = child_key(s.key[a], s.len[a], x.r);
        x.a = a;
        if (beats(x, best)) best = x;
      }
      warp_best(best);
      // The host checks that n_nodes nodes exist, so a candidate is always found.
      const int a = best.a < 0 ? 0 : best.a, r = best.r < 0 ? 0 : best.r;
      if (lane == 0) {
        s.key[c] = best.key;
        s.len[c] = s.len[a] + 1;
        s.score[c] = best.sc;
        s.kids[c] = 0u;
        s.kids[a] |= 1u << r;
        s.pchosen[c] = a;
      }
      __syncwarp();
      refresh_best_child(s, c, K, R, lane);
      refresh_best_child(s, a, K, R, lane);
      __syncwarp();
    }
  }
  __syncthreads();

  // Canonical order, then the device topology arrays.
  for (int t = tid; t < n_nodes; t += kGreedyThreads) {
    int k = 0;
    const u128 kt = s.key[t];
    for (int u = 0; u < n_nodes; ++u) k += s.key[u] < kt ? 1 : 0;
    s.canon[t] = k;
  }
  __syncthreads();
  int32_t* parent = out;
  int32_t* depth = out + n_nodes;
  int32_t* rankv = out + 2 * n_nodes;
  int32_t* retrieve = out + 3 * n_nodes;
  const int W = K + 1;
  for (int t = tid; t < n_nodes; t += kGreedyThreads) {
    const int ci = s.canon[t];
    parent[ci] = t == 0 ? -1 : s.canon[s.pchosen[t]];
    depth[ci] = s.len[t];
    rankv[ci] = s.len[t] ? key_rank(s.key[t], s.len[t] - 1) : -1;
  }
  // Leaves (no chosen child) in canonical order: row = canonical leaves before it.
  for (int t = tid; t < n_nodes; t += kGreedyThreads) {
    for (int j = 0; j < W; ++j) retrieve[(size_t)t * W + j] = -1;
  }
  __syncthreads();
  for (int t = tid; t < n_nodes; t += kGreedyThreads) {
    if (s.kids[t]) continue;
    int row = 0;
    for (int u = 0; u < n_nodes; ++u) row += (!s.kids[u] && s.canon[u] < s.canon[t]) ? 1 : 0;
    for (int a = t; a >= 0; a = s.pchosen[a]) retrieve[(size_t)row * W + s.len[a]] = s.canon[a];
  }
  if (tid == 0) {
    int md = 0, leaves = 0, mr = 0;
    for (int t = 0; t < n_nodes; ++t) {
      md = max(md, s.len[t]);
      leaves += s.kids[t] ? 0 : 1;
      if (s.len[t]) mr = max(mr, key_rank(s.key[t], s.len[t] - 1) + 1);
    }
    meta[0] = n_nodes;
    meta[1] = md;
    meta[2] = leaves;
    meta[3] = mr;
  }
}

}  // namespace medusa

using namespace medusa;

extern "C" medusa_status medusa_accept_stats(const int32_t* path_nodes, const int32_t* accept_len,
                                             const medusa_dev_topology* t, int B, int Dmax, int R,
                                             uint64_t* tested, uint64_t* accepted, int32_t* d_status,
                                             medusa_stream_t stream) {
  if (!path_nodes || !accept_len || !t || !t->parent || !t->depth || !t->rank || !tested || !accepted)
    return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || t->n_nodes < 1 || t->n_nodes > MEDUSA_MAX_NODES || Dmax < t->max_depth || Dmax > MEDUSA_MAX_DEPTH ||
      R < t->max_rank || R < 1 || R > MEDUSA_MAX_TOPK)
    return MEDUSA_ERR_INVALID_ARG;
  launch_pdl(accept_stats_kernel, dim3(B), dim3(kStatThreads), 0, reinterpret_cast<cudaStream_t>(stream), path_nodes,
             accept_len, t->parent, t->depth, t->rank, t->n_nodes, Dmax, R,
             reinterpret_cast<unsigned long long*>(tested), reinterpret_cast<unsigned long long*>(accepted),
             d_status);
  return launch_status();
}

extern "C" medusa_status medusa_acc_update(double* acc, const uint64_t* tested, const uint64_t* accepted, int K,
                                           int R, double weight, medusa_stream_t stream) {
  if (!acc || !tested || !accepted || K < 1 || K > MEDUSA_MAX_DEPTH || R < 1 || R > MEDUSA_MAX_TOPK ||
      !(weight >= 0.0))
    return MEDUSA_ERR_INVALID_ARG;
  const int n = K * R;
  launch_pdl(acc_update_kernel, dim3((n + 255) / 256), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream), acc,
             reinterpret_cast<const unsigned long long*>(tested),
             reinterpret_cast<const unsigned long long*>(accepted), n, weight);
  return launch_status();
}

extern "C" size_t medusa_topology_greedy_device_elems(int K, int n_nodes) {
  if (K < 1 || n_nodes < 1) return 0;
  return (size_t)3 * n_nodes + (size_t)n_nodes * (K + 1);
}

extern "C" medusa_status medusa_topology_greedy_device(const double* acc, int K, int R, int n_nodes, int32_t* d_buf,
                                                       size_t buf_elems, int32_t* d_meta, medusa_dev_topology* out,
                                                       int32_t* d_status, medusa_stream_t stream) {
  if (!acc || !d_buf || !d_meta || !out) return MEDUSA_ERR_INVALID_ARG;
  if (K < 1 || K > MEDUSA_MAX_DEPTH || R < 1 || R > MEDUSA_MAX_TOPK || n_nodes < 1 || n_nodes > MEDUSA_MAX_NODES)
    return MEDUSA_ERR_INVALID_ARG;
  // Enough candidate paths must exist: 1 + R + R^2 + ... + R^K >= n_nodes.
  long long avail = 1, level = 1;
  for (int d = 1; d <= K && avail < n_nodes; ++d) {
    level *= R;
    avail += level;
  }
  if (avail < n_nodes) return MEDUSA_ERR_INVALID_ARG;
  if (buf_elems < medusa_topology_greedy_device_elems(K, n_nodes)) return MEDUSA_ERR_INVALID_ARG;
  const size_t smem = sizeof(GreedyState);
  if (cudaFuncSetAttribute(greedy_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MEDUSA_ERR_CUDA;
  launch_pdl(greedy_tree_kernel, dim3(1), dim3(kGreedyThreads), smem, reinterpret_cast<cudaStream_t>(stream), acc, K,
             R, n_nodes, d_buf, d_meta, d_status);
  out->n_nodes = n_nodes;
  out->max_depth = K;  // bounds: the exact values land in d_meta
  out->n_leaves = n_nodes;
  out->max_rank = R;
  out->parent = d_buf;
  out->depth = d_buf + n_nodes;
  out->rank = d_buf + 2 * n_nodes;
  out->retrieve = d_buf + 3 * n_nodes;
  return launch_status();
}
