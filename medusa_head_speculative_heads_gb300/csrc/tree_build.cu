// medusa_tree_build: packs every batch row's candidate tree into token ids,
// tree position ids and the ancestor-only attention mask.
//
// Skill-pack guide ("Medusa 多解码头推理加速全解析"), sections "树形注意力" (root,
// then one level per Medusa head, each node branching into that head's top
// candidates) and "候选生成" (candidates built from per-head top-k lists).
// Paper review, FAQ "树注意力为什么能一次验证多条候选": each token attends only
// to its own branch's predecessors, and positions follow the tree.
//
// One CTA per batch row, one thread per node; the topology is staged in
// shared memory first.  CTA 0 also writes the mask (batch-independent): each
// thread walks its own ancestor chain (at most MEDUSA_MAX_DEPTH steps) and
// writes its mask row of ceil(N/32) words.
#include "common.cuh"
#include "host_util.h"

namespace medusa {

constexpr int kMaskWords = MEDUSA_MAX_NODES / 32;

__global__ void __launch_bounds__(MEDUSA_MAX_NODES)
tree_build_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ depth,
                  const int32_t* __restrict__ rank, int N, const int32_t* __restrict__ root_tok,
                  const int32_t* __restrict__ topk_idx, int K, int topk,
                  const int32_t* __restrict__ prefix_len, int32_t* __restrict__ tokens,
                  int32_t* __restrict__ pos, uint32_t* __restrict__ mask, int32_t* d_status) {
  __shared__ int s_parent[MEDUSA_MAX_NODES], s_depth[MEDUSA_MAX_NODES];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, n = threadIdx.x;
  // Every independent load first (one round trip), then the top-k gather.
  int rk = 0, L = 0, tok0 = 0;
  if (n < N) {
    s_parent[n] = parent[n];
    s_depth[n] = depth[n];
    rk = rank[n];
    L = prefix_len[b];
    if (n == 0) tok0 = root_tok[b];
  }
  __syncthreads();
  if (n >= N) return;
  const int dn = s_depth[n];
  int tok;
  if (n == 0) {
    tok = tok0;
  } else {
    if (dn < 1 || dn > K || rk < 0 || rk >= topk) {
      set_status(d_status, MEDUSA_DEV_BAD_INDEX);
      tok = -1;
    } else {
      tok = topk_idx[((size_t)b * K + (dn - 1)) * topk + rk];
    }
  }
  tokens[(size_t)b * N + n] = tok;
  pos[(size_t)b * N + n] = L + dn;

  if (b == 0) {
    const int W = (N + 31) / 32;
    uint32_t row[kMaskWords];
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w) row[w] = 0u;
    int a = n, steps = 0;
    bool ok = true;
    while (a >= 0) {
      if (a >= N || steps > MEDUSA_MAX_DEPTH) { ok = false; break; }
#pragma unroll
      for (int w = 0; w < kMaskWords; ++w)
        if (w == (a >> 5)) row[w] |= 1u << (a & 31);
      const int p = s_parent[a];
      if (a > 0 && (p >= a || p < 0 || s_depth[p] != s_depth[a] - 1)) { ok = false; break; }
      a = a == 0 ? -1 : p;
      ++steps;
    }
    if (!ok) {
      set_status(d_status, MEDUSA_DEV_BAD_TOPOLOGY);
#pragma unroll
      for (int w = 0; w < kMaskWords; ++w) row[w] = 0u;
    }
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w)
      if (w < W && mask) mask[(size_t)n * W + w] = row[w];
  }
}

}  // namespace medusa

using namespace medusa;

extern "C" medusa_status medusa_tree_build(const medusa_dev_topology* t, const int32_t* root_tok,
                                           const int32_t* topk_idx, int B, int K, int topk,
                                           const int32_t* prefix_len, int32_t* tokens, int32_t* pos,
                                           uint32_t* mask, int32_t* d_status,
                                           medusa_stream_t stream) {
  if (!t || !root_tok || !topk_idx || !prefix_len || !tokens || !pos) return MEDUSA_ERR_INVALID_ARG;
  if (!t->parent || !t->depth || !t->rank) return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || K < 1 || K > MEDUSA_MAX_DEPTH || topk < 1 || topk > MEDUSA_MAX_TOPK) return MEDUSA_ERR_INVALID_ARG;
  if (t->n_nodes < 1 || t->n_nodes > MEDUSA_MAX_NODES) return MEDUSA_ERR_INVALID_ARG;
  if (t->max_depth > K || t->max_rank > topk) return MEDUSA_ERR_INVALID_ARG;
  const int threads = (t->n_nodes + 31) / 32 * 32;
  launch_pdl(tree_build_kernel, dim3(B), dim3(threads), 0, reinterpret_cast<cudaStream_t>(stream), 
      t->parent, t->depth, t->rank, t->n_nodes, root_tok, topk_idx, K, topk, prefix_len, tokens, pos,
      mask, d_status);
  return launch_status();
}
