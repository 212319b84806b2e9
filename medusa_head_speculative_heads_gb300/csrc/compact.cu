// medusa_kv_compact: appends the accepted path's tree keys/values to the
// contiguous KV cache.
//
// Skill-pack guide ("Medusa 多解码头推理加速全解析"), section "树形验证": the tree
// is verified against past_key_values with use_cache, so the accepted tokens'
// keys and values join the cache for the next step.  The accepted rows are
// gathered from the tree K/V buffers to rows prefix_len .. prefix_len +
// accept_len - 1 of every layer.
//
// Kernel 1 moves 16-byte (or 4-byte) words: one CTA per (layer, row, path
// slot, K or V) row of Hkv x d elements at a time (decode and checks once per
// CTA, two words in flight per thread); slots past accept_len do nothing.
// Kernel 2 writes new_len after kernel 1 has read prefix_len, so new_len may
// alias prefix_len; when it does not, kernel 1's first B threads write it
// and kernel 2 is not launched.
#include <limits.h>

#include "common.cuh"
#include "host_util.h"

namespace medusa {

// new_len of row b: prefix_len + accept_len when the row is valid (accept
// length in range, fits the cache, every path node in range), else unchanged.
__device__ __forceinline__ int kv_new_len(const int32_t* prefix_len, const int32_t* accept_len,
                                          const int32_t* path_nodes, int b, int Lmax, int Dmax, int N) {
  const int L = prefix_len[b], A = accept_len[b];
  bool ok = A >= 1 && A <= Dmax + 1 && L >= 0 && L + A <= Lmax;
  for (int j = 0; ok && j < A; ++j) {
    const int nj = path_nodes[(size_t)b * (Dmax + 1) + j];
    ok = nj >= 0 && nj < N;
  }
  return ok ? L + A : L;
}

template <typename WORD>
__global__ void kv_gather_kernel(WORD* __restrict__ kc, WORD* __restrict__ vc, const WORD* __restrict__ kt,
                                 const WORD* __restrict__ vt, const int32_t* __restrict__ path_nodes,
                                 const int32_t* __restrict__ accept_len, const int32_t* __restrict__ prefix_len,
                                 int nl, int B, int N, int Lmax, int Dmax, int words_per_row,
                                 int rows_total, int32_t* d_status, int32_t* __restrict__ new_len_separate) {
  pdl_wait();
  pdl_trigger();
  if (new_len_separate) {  // does not alias prefix_len: written here, no second kernel
    const long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (b < B) new_len_separate[b] = kv_new_len(prefix_len, accept_len, path_nodes, (int)b, Lmax, Dmax, N);
  }
  // One CTA per (layer, row, path slot, K or V) row of words at a time: the
  // decode, the checks and the source slot are per CTA, the threads move
  // the row's words.  row = ((l * B + b) * (Dmax + 1) + i) * 2 + kv.
  for (int row = blockIdx.x; row < rows_total; row += gridDim.x) {
    int r = row;
    const int kv = r & 1;
    r >>= 1;
    const int i = r % (Dmax + 1);
    r /= Dmax + 1;
    const int b = r % B;
    const int l = r / B;
    const int A = accept_len[b], L = prefix_len[b];
    const bool first = l == 0 && i == 0 && kv == 0 && threadIdx.x == 0;
    if (A < 1 || A > Dmax + 1 || L < 0) {
      if (first) set_status(d_status, MEDUSA_DEV_BAD_INDEX);
      continue;
    }
    if (L + A > Lmax) {
      if (first) set_status(d_status, MEDUSA_DEV_CACHE_OVERFLOW);
      continue;
    }
    if (i >= A) continue;
    // A malformed path makes the whole row skip: check every slot.
    bool ok = true;
    for (int j = 0; j < A; ++j) {
      const int nj = path_nodes[(size_t)b * (Dmax + 1) + j];
      ok = ok && nj >= 0 && nj < N;
    }
    if (!ok) {
      if (first) set_status(d_status, MEDUSA_DEV_BAD_INDEX);
      continue;
    }
    const int src = path_nodes[(size_t)b * (Dmax + 1) + i];
    const WORD* from = (kv ? vt : kt) + (((size_t)l * B + b) * N + src) * words_per_row;
    WORD* to = (kv ? vc : kc) + (((size_t)l * B + b) * Lmax + L + i) * words_per_row;
    int w = threadIdx.x;
    for (; w + blockDim.x < words_per_row; w += 2 * blockDim.x) {  // two words in flight per thread
      const WORD a = from[w], c = from[w + blockDim.x];
      to[w] = a;
      to[w + blockDim.x] = c;
    }
    if (w < words_per_row) to[w] = from[w];
  }
}

__global__ void kv_len_kernel(const int32_t* prefix_len, const int32_t* accept_len, int32_t* new_len,
                              int B, int Lmax, int Dmax, const int32_t* __restrict__ path_nodes, int N) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  new_len[b] = kv_new_len(prefix_len, accept_len, path_nodes, b, Lmax, Dmax, N);
}

}  // namespace medusa

using namespace medusa;

extern "C" medusa_status medusa_kv_compact(void* kc, void* vc, const void* kt, const void* vt,
                                           const int32_t* path_nodes, const int32_t* accept_len,
                                           const int32_t* prefix_len, int32_t* new_len,
                                           int n_layers, int B, int N, int Hkv, int d, int Lmax,
                                           int Dmax, medusa_dtype dt, int32_t* d_status,
                                           medusa_stream_t stream) {
  if (!kc || !vc || !kt || !vt || !path_nodes || !accept_len || !prefix_len || !new_len)
    return MEDUSA_ERR_INVALID_ARG;
  if (n_layers < 1 || B < 1 || N < 1 || N > MEDUSA_MAX_NODES || Hkv < 1 || d < 1 || Lmax < 1)
    return MEDUSA_ERR_INVALID_ARG;
  if (Dmax < 0 || Dmax > MEDUSA_MAX_DEPTH || !dtype_ok(dt)) return MEDUSA_ERR_INVALID_ARG;
  const size_t row_bytes = (size_t)Hkv * d * dtype_bytes(dt);
  const size_t cache_bytes = (size_t)n_layers * B * Lmax * row_bytes;
  const size_t tree_bytes = (size_t)n_layers * B * N * row_bytes;
  if (overlaps(kc, cache_bytes, kt, tree_bytes) || overlaps(kc, cache_bytes, vt, tree_bytes) ||
      overlaps(vc, cache_bytes, kt, tree_bytes) || overlaps(vc, cache_bytes, vt, tree_bytes) ||
      overlaps(kc, cache_bytes, vc, cache_bytes))
    return MEDUSA_ERR_ALIAS;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool v16 = row_bytes % 16 == 0 && aligned16(kc) && aligned16(vc) && aligned16(kt) && aligned16(vt);
  if (!v16 && (row_bytes % 4 || ((uintptr_t)kc | (uintptr_t)vc | (uintptr_t)kt | (uintptr_t)vt) & 3u))
    return MEDUSA_ERR_INVALID_ARG;
  const int wpr = (int)(row_bytes / (v16 ? 16 : 4));
  const long long rows_ll = (long long)n_layers * B * (Dmax + 1) * 2;
  if (rows_ll > INT_MAX) return MEDUSA_ERR_INVALID_ARG;
  const int rows_total = (int)rows_ll;
  const int threads = wpr >= 256 ? 256 : (wpr + 31) / 32 * 32;
  long long blocks = rows_total;
  const long long cap = (long long)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks * threads < B) blocks = (B + threads - 1) / threads;  // the first B threads write new_len
  // One kernel when new_len is a separate buffer the grid's first B threads can write.
  const bool fused = !overlaps(new_len, (size_t)B * 4, prefix_len, (size_t)B * 4) && blocks * threads >= B;
  int32_t* nl_sep = fused ? new_len : nullptr;
  if (v16)
    launch_pdl(kv_gather_kernel<uint4>, dim3((int)blocks), dim3(threads), 0, s, (uint4*)kc, (uint4*)vc, (const uint4*)kt,
                                                           (const uint4*)vt, path_nodes, accept_len,
                                                           prefix_len, n_layers, B, N, Lmax, Dmax,
                                                           wpr, rows_total, d_status, nl_sep);
  else
    launch_pdl(kv_gather_kernel<uint32_t>, dim3((int)blocks), dim3(threads), 0, s, (uint32_t*)kc, (uint32_t*)vc,
                                                               (const uint32_t*)kt, (const uint32_t*)vt,
                                                               path_nodes, accept_len, prefix_len,
                                                               n_layers, B, N, Lmax, Dmax, wpr, rows_total,
                                                               d_status, nl_sep);
  if (!fused)
    launch_pdl(kv_len_kernel, dim3((B + 127) / 128), dim3(128), 0, s, prefix_len, accept_len, new_len, B, Lmax,
               Dmax, path_nodes, N);
  return launch_status();
}
