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

struct GreedyState {
  int8_t path[MEDUSA_MAX_NODES][MEDUSA_MAX_DEPTH];
  int len[MEDUSA_MAX_NODES];
  double score[MEDUSA_MAX_NODES];
  uint32_t kids[MEDUSA_MAX_NODES];  // bit r: child with rank r already chosen
  int pchosen[MEDUSA_MAX_NODES];    // chosen index of the parent
  int canon[MEDUSA_MAX_NODES];      // canonical index of chosen node i
  double acc[MEDUSA_MAX_DEPTH * MEDUSA_MAX_TOPK];
};

// Canonical order of chosen node a's child with rank ra vs chosen node b's
// child with rank rb: shorter path first, then lexicographic.
__device__ __forceinline__ bool child_less(const GreedyState& s, int a, int ra, int b, int rb) {
  const int la = s.len[a] + 1, lb = s.len[b] + 1;
  if (la != lb) return la < lb;
  for (int j = 0; j < la; ++j) {
    const int x = j < la - 1 ? s.path[a][j] : ra;
    const int y = j < lb - 1 ? s.path[b][j] : rb;
    if (x != y) return x < y;
  }
  return false;
}

// Canonical order of two chosen nodes.
__device__ __forceinline__ bool node_less(const GreedyState& s, int a, int b) {
  if (s.len[a] != s.len[b]) return s.len[a] < s.len[b];
  for (int j = 0; j < s.len[a]; ++j)
    if (s.path[a][j] != s.path[b][j]) return s.path[a][j] < s.path[b][j];
  return false;
}

// Greedy preference of candidate (sa; child of a with rank ra) over (sb; b, rb):
// scores within a relative 1e-12 are ties, broken by canonical order.
__device__ __forceinline__ bool beats(const GreedyState& s, double sa, int a, int ra, double sb, int b, int rb) {
  if (b < 0) return a >= 0;
  if (a < 0) return false;
  if (fabs(sa - sb) <= 1e-12 * fmax(fabs(sa), fabs(sb))) return child_less(s, a, ra, b, rb);
  return sa > sb;
}

// One CTA.  Device buffer: parent[n], depth[n], rank[n], retrieve[n][K + 1].
// meta = {n_nodes, max_depth, n_leaves, max_rank}.
__global__ void __launch_bounds__(kGreedyThreads)
greedy_tree_kernel(const double* __restrict__ acc_in, int K, int R, int n_nodes, int32_t* __restrict__ out,
                   int32_t* __restrict__ meta, int32_t* d_status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GreedyState& s = *reinterpret_cast<GreedyState*>(smem_raw);
  __shared__ double w_sc[kGreedyThreads / 32];
  __shared__ int w_a[kGreedyThreads / 32], w_r[kGreedyThreads / 32];
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
    s.len[0] = 0;
    s.score[0] = 1.0;
    s.kids[0] = 0u;
    s.pchosen[0] = -1;
  }
  __syncthreads();
  if (tid == 0 && s_bad) set_status(d_status, MEDUSA_DEV_BAD_INDEX);

  for (int c = 1; c < n_nodes; ++c) {
    // Best frontier candidate: (chosen node a, rank r) not yet chosen.
    double best_s = 0.0;
    int best_a = -1, best_r = -1;
    for (int idx = tid; idx < c * R; idx += kGreedyThreads) {
      const int a = idx / R, r = idx - a * R;
      if (s.len[a] >= K || ((s.kids[a] >> r) & 1u)) continue;
      const double sc = s.score[a] * s.acc[s.len[a] * R + r];
      if (beats(s, sc, a, r, best_s, best_a, best_r)) {
        best_s = sc;
        best_a = a;
        best_r = r;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const double s2 = __shfl_xor_sync(0xffffffffu, best_s, o);
      const int a2 = __shfl_xor_sync(0xffffffffu, best_a, o);
      const int r2 = __shfl_xor_sync(0xffffffffu, best_r, o);
      if (beats(s, s2, a2, r2, best_s, best_a, best_r)) {
        best_s = s2;
        best_a = a2;
        best_r = r2;
      }
    }
    if (lane == 0) {
      w_sc[warp] = best_s;
      w_a[warp] = best_a;
      w_r[warp] = best_r;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kGreedyThreads / 32; ++w)
        if (beats(s, w_sc[w], w_a[w], w_r[w], best_s, best_a, best_r)) {
          best_s = w_sc[w];
          best_a = w_a[w];
          best_r = w_r[w];
        }
      // The host checks that n_nodes nodes exist, so a candidate is always found.
      const int a = best_a < 0 ? 0 : best_a, r = best_r < 0 ? 0 : best_r;
      for (int j = 0; j < s.len[a]; ++j) s.path[c][j] = s.path[a][j];
      s.path[c][s.len[a]] = (int8_t)r;
      s.len[c] = s.len[a] + 1;
      s.score[c] = best_s;
      s.kids[c] = 0u;
      s.kids[a] |= 1u << r;
      s.pchosen[c] = a;
    }
    __syncthreads();
  }

  // Canonical order, then the device topology arrays.
  for (int t = tid; t < n_nodes; t += kGreedyThreads) {
    int k = 0;
    for (int u = 0; u < n_nodes; ++u) k += node_less(s, u, t) ? 1 : 0;
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
    rankv[ci] = s.len[t] ? s.path[t][s.len[t] - 1] : -1;
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
      if (s.len[t]) mr = max(mr, s.path[t][s.len[t] - 1] + 1);
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
