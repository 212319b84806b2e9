// medusa_typical_accept: typical acceptance over every batch row's tree.
//
// Paper review ("Medusa: Simple LLM Inference Acceleration Framework with
// Multiple Decoding Heads"), section "Medusa 的三个核心组件": a candidate is
// accepted when its probability under the base model exceeds
// min(eps, delta * exp(-H(p))); the first token is accepted greedily and
// unconditionally and the longest valid prefix is kept.  Section "方法细节":
// at temperature 0 this is greedy decoding.  Skill-pack guide, "树形验证":
// the longest valid candidate is accepted.
//
// Two kernels.  node_stats: one CTA per (node, row) reads the node's fp32
// logit row once for the argmax and once more (from L2) for the tempered
// partition function S and E = sum e^((z-m)/T) (z-m)/T, giving
// H = ln S - E/S; it then tests every child of the node.  select_path: one
// CTA per row propagates acceptance level by level (a node is accepted iff its
// parent is and it passed), picks the deepest accepted node (lowest index on
// ties) and writes the path, its length and the next root token.
#include <limits.h>

#include "common.cuh"
#include "host_util.h"

namespace medusa {

constexpr int kStatThreads = 256;

__device__ __forceinline__ void block_argmax(float& v, int& i, float* sv, int* si) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    if (ranks_ahead(v2, i2, v, i)) { v = v2; i = i2; }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { sv[warp] = v; si[warp] = i; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (ranks_ahead(sv[w], si[w], v, i)) { v = sv[w]; i = si[w]; }
    sv[0] = v; si[0] = i;
  }
  __syncthreads();
  v = sv[0]; i = si[0];
  __syncthreads();
}

__device__ __forceinline__ float block_sum(float v, float* s) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) s[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += s[w];
    s[0] = t;
  }
  __syncthreads();
  float r = s[0];
  __syncthreads();
  return r;
}

// Grid (N, B).  Writes, for every child c of node n: pass[b][c], and the
// optional p_tok / thr; for node n itself: amax[b][n].
__global__ void __launch_bounds__(kStatThreads)
node_stats_kernel(const float* __restrict__ logits, const int32_t* __restrict__ tokens,
                  const int32_t* __restrict__ parent, int N, int V, float T, float eps, float delta,
                  int32_t* __restrict__ pass, int32_t* __restrict__ amax, float* __restrict__ p_tok,
                  float* __restrict__ thr_out, int32_t* d_status) {
  __shared__ float sv[kStatThreads / 32];
  __shared__ int si[kStatThreads / 32];
  const int n = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const float* z = logits + ((size_t)b * N + n) * V;
  const bool vec = (V & 3) == 0 && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0);

  float mv = -INFINITY;
  int mi = INT_MAX;
  if (vec) {
    const float4* z4 = reinterpret_cast<const float4*>(z);
    for (int q = tid; q < V / 4; q += kStatThreads) {
      float4 t = z4[q];
      float e[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (ranks_ahead(e[j], 4 * q + j, mv, mi)) { mv = e[j]; mi = 4 * q + j; }
    }
  } else {
    for (int v = tid; v < V; v += kStatThreads)
      if (ranks_ahead(z[v], v, mv, mi)) { mv = z[v]; mi = v; }
  }
  block_argmax(mv, mi, sv, si);

  float S = 1.f, thr;
  if (T > 0.f) {
    const float inv_t = 1.f / T;
    float s = 0.f, e = 0.f;
    if (vec) {
      const float4* z4 = reinterpret_cast<const float4*>(z);
      for (int q = tid; q < V / 4; q += kStatThreads) {
        float4 t = z4[q];
        float x[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float a = (x[j] - mv) * inv_t;
          float w = expf(a);
          s += w;
          e = fmaf(w, a, e);
        }
      }
    } else {
      for (int v = tid; v < V; v += kStatThreads) {
        float a = (z[v] - mv) * inv_t;
        float w = expf(a);
        s += w;
        e = fmaf(w, a, e);
      }
    }
    S = block_sum(s, sv);
    float E = block_sum(e, sv);
    float H = logf(S) - E / S;
    thr = fminf(eps, delta * expf(-H));
  } else {
    thr = fminf(eps, delta);
  }

  if (tid == 0) amax[(size_t)b * N + n] = mi;
  if (n == 0 && tid == 0) {
    pass[(size_t)b * N] = 1;
    if (p_tok) p_tok[(size_t)b * N] = 1.f;
    if (thr_out) thr_out[(size_t)b * N] = 0.f;
  }
  for (int c = 1 + tid; c < N; c += kStatThreads) {
    if (parent[c] != n) continue;
    const int x = tokens[(size_t)b * N + c];
    int ok;
    float p;
    if (x < 0 || x >= V) {
      set_status(d_status, MEDUSA_DEV_BAD_INDEX);
      ok = 0;
      p = 0.f;
    } else if (T > 0.f) {
      p = expf((z[x] - mv) / T) / S;
      ok = p > thr;
    } else {
      ok = x == mi;
      p = ok ? 1.f : 0.f;
    }
    pass[(size_t)b * N + c] = ok;
    if (p_tok) p_tok[(size_t)b * N + c] = p;
    if (thr_out) thr_out[(size_t)b * N + c] = thr;
  }
}

// Grid B; block = N rounded up to a warp multiple (<= 256).
__global__ void __launch_bounds__(MEDUSA_MAX_NODES)
select_path_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ depth, int N,
                   int max_depth, const int32_t* __restrict__ pass, const int32_t* __restrict__ amax,
                   int32_t* __restrict__ accept_len, int32_t* __restrict__ path_nodes,
                   int32_t* __restrict__ next_tok, int32_t* d_status) {
  __shared__ int acc[MEDUSA_MAX_NODES];
  __shared__ int s_key[MEDUSA_MAX_NODES / 32];
  __shared__ int s_bad;
  const int b = blockIdx.x, c = threadIdx.x;
  if (c == 0) s_bad = 0;
  __syncthreads();
  int dc = -1, pc = -1;
  if (c < N) {
    dc = depth[c];
    pc = parent[c];
    if (c > 0 && (pc < 0 || pc >= c || dc < 1 || dc > max_depth)) s_bad = 1;
    acc[c] = c == 0 ? 1 : 0;
  }
  __syncthreads();
  if (s_bad) {
    if (c == 0) {
      set_status(d_status, MEDUSA_DEV_BAD_TOPOLOGY);
      accept_len[b] = 1;
      next_tok[b] = amax[(size_t)b * N];
      for (int j = 0; j <= max_depth; ++j) path_nodes[(size_t)b * (max_depth + 1) + j] = j ? -1 : 0;
    }
    return;
  }
  for (int d = 1; d <= max_depth; ++d) {
    if (c < N && dc == d) acc[c] = acc[pc] && pass[(size_t)b * N + c];
    __syncthreads();
  }
  // Deepest accepted node, lowest index: maximise key = depth * 512 + (511 - c).
  int key = (c < N && acc[c]) ? dc * 512 + (511 - c) : -1;
#pragma unroll
  for (int o = 16; o; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
  if ((c & 31) == 0) s_key[c >> 5] = key;
  __syncthreads();
  if (c == 0) {
    int best_key = s_key[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) best_key = max(best_key, s_key[w]);
    const int best = 511 - (best_key & 511);
    const int db = best_key >> 9;
    int32_t* pn = path_nodes + (size_t)b * (max_depth + 1);
    for (int j = db + 1; j <= max_depth; ++j) pn[j] = -1;
    int a = best;
    for (int j = db; j >= 0; --j) {
      pn[j] = a;
      a = j ? parent[a] : -1;
    }
    accept_len[b] = db + 1;
    next_tok[b] = amax[(size_t)b * N + best];
  }
}

}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_typical_accept_workspace_size(int B, int N) {
  if (B <= 0 || N <= 0) return 0;
  WsCarver w(nullptr);
  w.take<int32_t>((size_t)B * N);
  w.take<int32_t>((size_t)B * N);
  return w.used;
}

extern "C" medusa_status medusa_typical_accept(const float* logits, const int32_t* tokens,
                                               const medusa_dev_topology* t, int B, int V,
                                               float temperature, float eps, float delta,
                                               int32_t* accept_len, int32_t* path_nodes,
                                               int32_t* next_tok, float* p_tok_or_null,
                                               float* thr_or_null, void* ws, size_t ws_bytes,
                                               int32_t* d_status, medusa_stream_t stream) {
  if (!logits || !tokens || !t || !t->parent || !t->depth || !accept_len || !path_nodes || !next_tok)
    return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || V < 1 || t->n_nodes < 1 || t->n_nodes > MEDUSA_MAX_NODES) return MEDUSA_ERR_INVALID_ARG;
  if (t->max_depth < 0 || t->max_depth > MEDUSA_MAX_DEPTH) return MEDUSA_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || !(eps >= 0.f) || !(delta >= 0.f)) return MEDUSA_ERR_INVALID_ARG;
  const int N = t->n_nodes;
  if (!ws || ws_bytes < medusa_typical_accept_workspace_size(B, N)) return MEDUSA_ERR_WORKSPACE;
  WsCarver wc(ws);
  int32_t* pass = wc.take<int32_t>((size_t)B * N);
  int32_t* amax = wc.take<int32_t>((size_t)B * N);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  node_stats_kernel<<<dim3(N, B), kStatThreads, 0, s>>>(logits, tokens, t->parent, N, V, temperature,
                                                        eps, delta, pass, amax, p_tok_or_null,
                                                        thr_or_null, d_status);
  const int threads = (N + 31) / 32 * 32;
  select_path_kernel<<<B, threads, 0, s>>>(t->parent, t->depth, N, t->max_depth, pass, amax,
                                           accept_len, path_nodes, next_tok, d_status);
  return launch_status();
}
