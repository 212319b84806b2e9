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
// Two kernels.  node_partial: one CTA per (vocabulary chunk, node, row) reads
// its slice of the node's fp32 logits once for the max/argmax and once more
// (from L1/L2) for the tempered sums S_c = sum e^((z-m_c)/T) and
// E_c = sum e^((z-m_c)/T) (z-m_c)/T.  select_path: one CTA per row combines the
// chunk partials exactly (a few threads per node and a shuffle reduction) (S = sum_c S_c e^((m_c-m)/T), E likewise), giving
// H = ln S - E/S and the threshold per node, tests every child against its
// parent's distribution, propagates acceptance level by level (a node is
// accepted iff its parent is and it passed), picks the deepest accepted node
// (lowest index on ties) and writes the path, its length and the next root
// token.
#include <limits.h>

#include "common.cuh"
#include "host_util.h"

namespace medusa {

constexpr int kPartThreads = 128;
constexpr int kChunkValues = 2048;
constexpr int kMaxChunks = 32;

int accept_chunks(int V) {
  int c = (V + kChunkValues - 1) / kChunkValues;
  return c < 1 ? 1 : c > kMaxChunks ? kMaxChunks : c;
}

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

// Grid (C, N, B).  part[(b*N + n)*C + c] = {max, argmax (bits), S_c, E_c}.
__global__ void __launch_bounds__(kPartThreads)
node_partial_kernel(const float* __restrict__ logits, int N, int V, int C, float T, float4* __restrict__ part) {
  __shared__ float sv[kPartThreads / 32];
  __shared__ int si[kPartThreads / 32];
  const int c = blockIdx.x, n = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const float* z = logits + ((size_t)b * N + n) * V;
  const int cs = ((V + C - 1) / C + 3) & ~3;  // chunk size, a multiple of 4
  const int lo = c * cs, hi = min(V, lo + cs);
  // While an earlier kernel on the stream finishes, bring this chunk into L2
  // (a hint: L2 is where every write lands, so nothing stale can be read).
  for (int v = lo + tid * 32; v < hi; v += kPartThreads * 32) prefetch_l2(z + v);
  pdl_wait();
  pdl_trigger();
  const bool vec = (V & 3) == 0 && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0);

  // Chunks of at most kPartThreads x 16 values (V up to 65536): the chunk
  // stays in registers between the max and the sums (16-byte loads all in
  // flight, one memory pass) and the warps meet twice in shared memory.
  constexpr int kRegQ = 4;  // float4 per thread
  if (vec && hi - lo <= kPartThreads * 4 * kRegQ) {
    __shared__ float4 wsum[kPartThreads / 32];
    const float4* z4 = reinterpret_cast<const float4*>(z);
    float4 q[kRegQ];
#pragma unroll
    for (int k = 0; k < kRegQ; ++k) {
      const int qi = (lo >> 2) + tid + k * kPartThreads;
      q[k] = qi < (hi >> 2) ? z4[qi] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    float mv = -INFINITY;
    int mi = INT_MAX;
#pragma unroll
    for (int k = 0; k < kRegQ; ++k) {
      const int qi = (lo >> 2) + tid + k * kPartThreads;
      const float e[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (qi < (hi >> 2) && ranks_ahead(e[j], 4 * qi + j, mv, mi)) { mv = e[j]; mi = 4 * qi + j; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, mv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, mi, o);
      if (ranks_ahead(v2, i2, mv, mi)) { mv = v2; mi = i2; }
    }
    const int lane = tid & 31, warp = tid >> 5;
    if (lane == 0) { sv[warp] = mv; si[warp] = mi; }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kPartThreads / 32; ++w)
      if (ranks_ahead(sv[w], si[w], mv, mi)) { mv = sv[w]; mi = si[w]; }
    float S = 0.f, E = 0.f;
    if (T > 0.f && lo < hi) {
      const float inv_t = 1.f / T;
      float s2 = 0.f, e2 = 0.f;
#pragma unroll
      for (int k = 0; k < kRegQ; ++k) {
        const int qi = (lo >> 2) + tid + k * kPartThreads;
        if (qi >= (hi >> 2)) continue;
        const float x[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float a = (x[j] - mv) * inv_t;
          const float w = expf(a);
          s2 += w;
          e2 = fmaf(w, a, e2);
        }
      }
      s2 = warp_sum(s2);
      e2 = warp_sum(e2);
      if (lane == 0) wsum[warp] = make_float4(s2, e2, 0.f, 0.f);
      __syncthreads();
      if (tid == 0)
        for (int w = 0; w < kPartThreads / 32; ++w) {
          S += wsum[w].x;
          E += wsum[w].y;
        }
    }
    if (tid == 0) part[((size_t)b * N + n) * C + c] = make_float4(mv, __int_as_float(mi), S, E);
    return;
  }

  float mv = -INFINITY;
  int mi = INT_MAX;
  if (vec) {
    const float4* z4 = reinterpret_cast<const float4*>(z);
    for (int q = (lo >> 2) + tid; q < (hi >> 2); q += kPartThreads) {
      const float4 t = z4[q];
      const float e[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (ranks_ahead(e[j], 4 * q + j, mv, mi)) { mv = e[j]; mi = 4 * q + j; }
    }
  } else {
    for (int v = lo + tid; v < hi; v += kPartThreads)
      if (ranks_ahead(z[v], v, mv, mi)) { mv = z[v]; mi = v; }
  }
  block_argmax(mv, mi, sv, si);

  float S = 0.f, E = 0.f;
  if (T > 0.f && lo < hi) {
    const float inv_t = 1.f / T;
    float s = 0.f, e = 0.f;
    if (vec) {
      const float4* z4 = reinterpret_cast<const float4*>(z);
      for (int q = (lo >> 2) + tid; q < (hi >> 2); q += kPartThreads) {
        const float4 t = z4[q];
        const float x[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float a = (x[j] - mv) * inv_t;
          const float w = expf(a);
          s += w;
          e = fmaf(w, a, e);
        }
      }
    } else {
      for (int v = lo + tid; v < hi; v += kPartThreads) {
        const float a = (z[v] - mv) * inv_t;
        const float w = expf(a);
        s += w;
        e = fmaf(w, a, e);
      }
    }
    S = block_sum(s, sv);
    E = block_sum(e, sv);
  }
  if (tid == 0) part[((size_t)b * N + n) * C + c] = make_float4(mv, __int_as_float(mi), S, E);
}

// Combines two partial statistics (max, argmax, S, E) of one logit row.
__device__ __forceinline__ void combine_stats(float& m, int& a, float& S, float& E, float m2, int a2, float S2,
                                              float E2, float inv_t) {
  float mn = m;
  int an = a;
  if (ranks_ahead(m2, a2, m, a)) { mn = m2; an = a2; }
  float Sn = 0.f, En = 0.f;
  if (S > 0.f) {
    const float d = (m - mn) * inv_t, w = expf(d);
    Sn = S * w;
    En = w * fmaf(S, d, E);
  }
  if (S2 > 0.f) {
    const float d = (m2 - mn) * inv_t, w = expf(d);
    Sn = fmaf(S2, w, Sn);
    En = fmaf(w, fmaf(S2, d, E2), En);
  }
  m = mn;
  a = an;
  S = Sn;
  E = En;
}

constexpr int kSelectThreads = 256;

// Grid B; block 256.  `grp` threads (a power of two <= 8 with grp * N <= 256)
// combine the chunk partials of one node, then one thread per node tests it
// against its parent and the tree is resolved level by level.
__global__ void __launch_bounds__(kSelectThreads)
select_path_kernel(const float* __restrict__ logits, const int32_t* __restrict__ tokens,
                   const int32_t* __restrict__ parent, const int32_t* __restrict__ depth, int N, int V,
                   int max_depth, int C, int grp, float T, float eps, float delta, const float4* __restrict__ part,
                   int32_t* __restrict__ accept_len, int32_t* __restrict__ path_nodes,
                   int32_t* __restrict__ next_tok, float* __restrict__ p_tok, float* __restrict__ thr_out,
                   int32_t* d_status) {
  __shared__ int acc[MEDUSA_MAX_NODES], pass[MEDUSA_MAX_NODES], amax[MEDUSA_MAX_NODES], par[MEDUSA_MAX_NODES],
      dep[MEDUSA_MAX_NODES];
  __shared__ float zmax[MEDUSA_MAX_NODES], ssum[MEDUSA_MAX_NODES], thr[MEDUSA_MAX_NODES];
  __shared__ int s_key[kSelectThreads / 32];
  __shared__ int s_bad;
  const int b = blockIdx.x, tid = threadIdx.x, c = tid;
  pdl_wait();
  pdl_trigger();
  if (tid == 0) s_bad = 0;
  // the topology and token of node c, loaded with the partials below (one
  // round trip), then the logit of that token under its parent's distribution
  // (the second round trip overlaps the combination of the partials)
  const int dc_ld = c < N ? depth[c] : -1, pc_ld = c < N ? parent[c] : -1;
  const int x_ld = (c > 0 && c < N) ? tokens[(size_t)b * N + c] : -1;
  const bool z_ok = c > 0 && c < N && pc_ld >= 0 && pc_ld < N && x_ld >= 0 && x_ld < V;
  const float z_px = z_ok ? logits[((size_t)b * N + pc_ld) * V + x_ld] : 0.f;
  // 1. statistics of every node: grp threads per node, strided over the chunks
  {
    const int node = tid / grp, sub = tid % grp;
    const float inv_t = T > 0.f ? 1.f / T : 0.f;
    float m = -INFINITY, S = 0.f, E = 0.f;
    int a = INT_MAX;
    if (node < N) {
      const float4* pp = part + ((size_t)b * N + node) * C;
#pragma unroll 4
      for (int k = sub; k < C; k += grp) {
        const float4 q = pp[k];
        combine_stats(m, a, S, E, q.x, __float_as_int(q.y), q.z, q.w, inv_t);
      }
    }
    for (int o = 1; o < grp; o <<= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const int a2 = __shfl_xor_sync(0xffffffffu, a, o);
      const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
      const float E2 = __shfl_xor_sync(0xffffffffu, E, o);
      combine_stats(m, a, S, E, m2, a2, S2, E2, inv_t);
    }
    if (node < N && sub == 0) {
      float th;
      if (T > 0.f) {
        const float H = logf(S) - E / S;
        th = fminf(eps, delta * expf(-H));
      } else {
        th = fminf(eps, delta);
        S = 1.f;
      }
      zmax[node] = m;
      ssum[node] = S;
      thr[node] = th;
      amax[node] = a;
    }
  }
  __syncthreads();
  int dc = -1, pc = -1;
  if (c < N) {
    dc = dc_ld;
    pc = pc_ld;
    acc[c] = c == 0 ? 1 : 0;
    par[c] = pc;
    dep[c] = dc;
  }
  __syncthreads();
  // The level loop and the path walk below index shared memory with par[] and
  // stop on depths: the root must be (parent -1, depth 0) and every other node
  // must sit one level below an earlier node.
  if (c < N) {
    const bool bad = c == 0 ? (pc != -1 || dc != 0)
                            : (pc < 0 || pc >= c || dc < 1 || dc > max_depth || dep[pc] != dc - 1);
    if (bad) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (c == 0) {
      set_status(d_status, MEDUSA_DEV_BAD_TOPOLOGY);
      accept_len[b] = 1;
      next_tok[b] = amax[0];
      for (int j = 0; j <= max_depth; ++j) path_nodes[(size_t)b * (max_depth + 1) + j] = j ? -1 : 0;
    }
    return;
  }
  // Child tests against the parent's distribution.
  if (c < N) {
    int ok = 1;
    float p = 1.f, t = 0.f;
    if (c > 0) {
      const int x = x_ld;
      t = thr[pc];
      if (x < 0 || x >= V) {
        set_status(d_status, MEDUSA_DEV_BAD_INDEX);
        ok = 0;
        p = 0.f;
      } else if (T > 0.f) {
        p = expf((z_px - zmax[pc]) / T) / ssum[pc];
        ok = p > t;
      } else {
        ok = x == amax[pc];
        p = ok ? 1.f : 0.f;
      }
    }
    pass[c] = ok;
    if (p_tok) p_tok[(size_t)b * N + c] = p;
    if (thr_out) thr_out[(size_t)b * N + c] = t;
  }
  __syncthreads();
  for (int d = 1; d <= max_depth; ++d) {
    if (c < N && dc == d) acc[c] = acc[pc] && pass[c];
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
      a = j ? par[a] : -1;  // the walk stays in shared memory
    }
    accept_len[b] = db + 1;
    next_tok[b] = amax[best];
  }
}

// Argument checks shared by the entry points of this file.
medusa_status typical_accept_check(const float* logits, const int32_t* tokens, const medusa_dev_topology* t, int B,
                                   int V, float temperature, float eps, float delta, const int32_t* accept_len,
                                   const int32_t* path_nodes, const int32_t* next_tok) {
  if (!logits || !tokens || !t || !t->parent || !t->depth || !accept_len || !path_nodes || !next_tok)
    return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || V < 1 || t->n_nodes < 1 || t->n_nodes > MEDUSA_MAX_NODES) return MEDUSA_ERR_INVALID_ARG;
  if (t->max_depth < 0 || t->max_depth > MEDUSA_MAX_DEPTH) return MEDUSA_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || !(eps >= 0.f) || !(delta >= 0.f)) return MEDUSA_ERR_INVALID_ARG;
  return MEDUSA_OK;
}

// Enqueues both kernels with `part` (B * N * accept_chunks(V) float4) as scratch.
medusa_status typical_accept_launch(const float* logits, const int32_t* tokens, const medusa_dev_topology* t,
                                    int B, int V, float temperature, float eps, float delta, int32_t* accept_len,
                                    int32_t* path_nodes, int32_t* next_tok, float* p_tok_or_null,
                                    float* thr_or_null, float4* part, int32_t* d_status, cudaStream_t s) {
  const int N = t->n_nodes;
  const int C = accept_chunks(V);
  launch_pdl(node_partial_kernel, dim3(C, N, B), dim3(kPartThreads), 0, s, logits, N, V, C, temperature, part);
  int grp = 1;
  while (grp < 8 && grp * 2 * N <= kSelectThreads) grp *= 2;
  launch_pdl(select_path_kernel, dim3(B), dim3(kSelectThreads), 0, s, logits, tokens, t->parent, t->depth, N, V, t->max_depth, C, grp,
                                                  temperature, eps, delta, part, accept_len, path_nodes, next_tok,
                                                  p_tok_or_null, thr_or_null, d_status);
  return launch_status();
}

}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_typical_accept_workspace_size(int B, int N, int V) {
  if (B <= 0 || N <= 0 || V <= 0) return 0;
  return (size_t)B * N * accept_chunks(V) * sizeof(float4);
}

extern "C" medusa_status medusa_typical_accept(const float* logits, const int32_t* tokens,
                                               const medusa_dev_topology* t, int B, int V,
                                               float temperature, float eps, float delta,
                                               int32_t* accept_len, int32_t* path_nodes,
                                               int32_t* next_tok, float* p_tok_or_null,
                                               float* thr_or_null, void* ws, size_t ws_bytes,
                                               int32_t* d_status, medusa_stream_t stream) {
  medusa_status st = typical_accept_check(logits, tokens, t, B, V, temperature, eps, delta, accept_len, path_nodes,
                                          next_tok);
  if (st != MEDUSA_OK) return st;
  if (!ws || ws_bytes < medusa_typical_accept_workspace_size(B, t->n_nodes, V)) return MEDUSA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 15u) return MEDUSA_ERR_INVALID_ARG;
  return typical_accept_launch(logits, tokens, t, B, V, temperature, eps, delta, accept_len, path_nodes, next_tok,
                               p_tok_or_null, thr_or_null, static_cast<float4*>(ws), d_status,
                               reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ allocation-free variant
//
// For callers that may not allocate device memory at the point where they run
// the acceptance step: code inside a region whose memory budget was fixed at
// start-up (the KV cache took the rest of the GPU), plugins that run under a
// host framework which owns every allocation, or loops that must never call
// into the CUDA allocator because it can synchronise the device.  The
// per-chunk statistics live in one static device array instead of a caller
// workspace.  The array exists once per GPU that loads this library and stays
// allocated until the process exits.

namespace medusa {

// 1 MiB of float4 partials: B * N * accept_chunks(V) <= 65536.
constexpr size_t kNoallocScratchBytes = MEDUSA_ACCEPT_NOALLOC_MAX_BYTES;
static __device__ __align__(256) float4 g_accept_scratch[kNoallocScratchBytes / sizeof(float4)];

// Device address of g_accept_scratch in the current context.  Host code sees
// only a host-side stand-in for the symbol, which must never reach a kernel.
// The address is looked up on every call (a runtime query that allocates
// nothing once this library's device code is loaded in the context), so a
// context created after cudaDeviceReset gets its own array's address rather
// than a stale one.  The first lookup in a context may load that device code,
// which is when the array itself is allocated.
static medusa_status accept_scratch(float4** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return MEDUSA_ERR_CUDA;
  }
  *out = static_cast<float4*>(p);
  return MEDUSA_OK;
}

}  // namespace medusa

extern "C" medusa_status medusa_typical_accept_noalloc(const float* logits, const int32_t* tokens,
                                                       const medusa_dev_topology* t, int B, int V,
                                                       float temperature, float eps, float delta,
                                                       int32_t* accept_len, int32_t* path_nodes,
                                                       int32_t* next_tok, float* p_tok_or_null,
                                                       float* thr_or_null, int32_t* d_status,
                                                       medusa_stream_t stream) {
  medusa_status st = typical_accept_check(logits, tokens, t, B, V, temperature, eps, delta, accept_len, path_nodes,
                                          next_tok);
  if (st != MEDUSA_OK) return st;
  if (medusa_typical_accept_workspace_size(B, t->n_nodes, V) > kNoallocScratchBytes) return MEDUSA_ERR_UNSUPPORTED;
  float4* scratch = nullptr;
  st = accept_scratch(&scratch);
  if (st != MEDUSA_OK) return st;
  // node_partial writes every entry the select kernel reads, so nothing in the
  // array has to start at zero.
  return typical_accept_launch(logits, tokens, t, B, V, temperature, eps, delta, accept_len, path_nodes, next_tok,
                               p_tok_or_null, thr_or_null, scratch, d_status, reinterpret_cast<cudaStream_t>(stream));
}
