// medusa_heads: K Medusa ResBlock heads over the last hidden state, then the
// per-head top-k.
//
// Paper review ("Medusa: Simple LLM Inference Acceleration Framework with
// Multiple Decoding Heads", section "Medusa 的三个核心组件"): head k computes
// p^(k) = softmax(W2^(k) (SiLU(W1^(k) h) + h)).  Skill-pack guide
// ("Medusa 多解码头推理加速全解析", section "候选生成"): top-k per head.
//
// At decode batch sizes the heads are a weight stream: every weight byte is
// used B times.  Two GEMV kernels stream W1 (then fuse SiLU + residual) and W2
// with 16-byte non-allocating loads, several rows per warp so that each lane
// keeps 8 independent 16-byte loads in flight, and the vector operand staged in
// shared memory as fp32.  The top-k runs in two passes: per-chunk candidate
// lists, then one merge per (row, head).
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "host_util.h"

namespace medusa {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kRowsPerWarp = 4;
constexpr int kMaxBatchPerPass = 8;

template <typename TW>
struct Vec16 {
  static constexpr int n = 16 / (int)sizeof(TW);
};

// acc[i][bb] += <W row (r+i) chunk at column c, x[bb] chunk at column c>
template <typename TW, int BB, int NR>
__device__ __forceinline__ void fma_chunk(const uint4 (&w)[NR], const float* __restrict__ xs, int C,
                                          int c, float (&acc)[NR][BB]) {
  constexpr int VEC = Vec16<TW>::n;
#pragma unroll
  for (int bb = 0; bb < BB; ++bb) {
    float x[VEC];
    const float4* xp = reinterpret_cast<const float4*>(xs + (size_t)bb * C + c);
#pragma unroll
    for (int q = 0; q < VEC / 4; ++q) {
      float4 t = xp[q];
      x[4 * q] = t.x; x[4 * q + 1] = t.y; x[4 * q + 2] = t.z; x[4 * q + 3] = t.w;
    }
#pragma unroll
    for (int i = 0; i < NR; ++i) {
      float f[VEC];
      if constexpr (sizeof(TW) == 2) unpack_bf16x8(w[i], f); else unpack_f32x4(w[i], f);
      float a = acc[i][bb];
#pragma unroll
      for (int e = 0; e < VEC; ++e) a = fmaf(f[e], x[e], a);
      acc[i][bb] = a;
    }
  }
}

// One warp: dot products of NR consecutive rows (starting at `row`) with the
// BB staged vectors.  Lane l reads 16-byte chunks l, l+32, ... of each row,
// two chunks per row per iteration (2*NR loads in flight per lane).
template <typename TW, int BB, int NR>
__device__ __forceinline__ void warp_rows(const TW* __restrict__ W, int C, const float* __restrict__ xs,
                                          int lane, float (&acc)[NR][BB]) {
  constexpr int VEC = Vec16<TW>::n;
  constexpr int STEP = 32 * VEC;
#pragma unroll
  for (int i = 0; i < NR; ++i)
#pragma unroll
    for (int bb = 0; bb < BB; ++bb) acc[i][bb] = 0.f;
  int c = lane * VEC;
  for (; c + STEP < C; c += 2 * STEP) {
    uint4 wa[NR], wb[NR];
#pragma unroll
    for (int i = 0; i < NR; ++i) wa[i] = ldg_stream(W + (size_t)i * C + c);
#pragma unroll
    for (int i = 0; i < NR; ++i) wb[i] = ldg_stream(W + (size_t)i * C + c + STEP);
    fma_chunk<TW, BB, NR>(wa, xs, C, c, acc);
    fma_chunk<TW, BB, NR>(wb, xs, C, c + STEP, acc);
  }
  if (c < C) {
    uint4 wa[NR];
#pragma unroll
    for (int i = 0; i < NR; ++i) wa[i] = ldg_stream(W + (size_t)i * C + c);
    fma_chunk<TW, BB, NR>(wa, xs, C, c, acc);
  }
#pragma unroll
  for (int i = 0; i < NR; ++i)
#pragma unroll
    for (int bb = 0; bb < BB; ++bb) acc[i][bb] = warp_sum(acc[i][bb]);
}

// kFirst = true : rows are W1 rows; x = h (batch rows b0..b0+BB-1);
//                 out[b][k][j] = SiLU(acc) + h[b][j]          (u, fp32)
// kFirst = false: rows are W2 rows; x = u[b][k];
//                 out[b][k][v] = acc                          (z, fp32)
// Grid (ctas_per_head, K); block 256; dynamic smem BB * C floats.
template <typename TW, int BB, bool kFirst>
__global__ void __launch_bounds__(kGemvThreads)
heads_gemv_kernel(const TW* __restrict__ W, const TW* __restrict__ h, const float* __restrict__ u,
                  int B, int b0, int K, int rows_per_head, int C, float* __restrict__ out) {
  extern __shared__ float xs[];  // [BB][C]
  const int k = blockIdx.y;
  for (int idx = threadIdx.x; idx < BB * C; idx += kGemvThreads) {
    int bb = idx / C, c = idx - bb * C, b = b0 + bb;
    float v = 0.f;
    if (b < B) v = kFirst ? load_elem<TW>(h, (size_t)b * C + c) : u[((size_t)b * K + k) * C + c];
    xs[idx] = v;
  }
  __syncthreads();

  // Balanced contiguous row ranges: CTA, then warp.
  const int ctas = gridDim.x;
  const int r_lo = (int)((long long)rows_per_head * blockIdx.x / ctas);
  const int r_hi = (int)((long long)rows_per_head * (blockIdx.x + 1) / ctas);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = r_hi - r_lo;
  const int w_lo = r_lo + n * warp / kGemvWarps;
  const int w_hi = r_lo + n * (warp + 1) / kGemvWarps;
  const TW* Wk = W + (size_t)k * rows_per_head * C;

  auto emit = [&](int row, int bb, float acc) {
    int b = b0 + bb;
    if (b >= B) return;
    size_t o = ((size_t)b * K + k) * rows_per_head + row;
    if constexpr (kFirst) {
      float hv = load_elem<TW>(h, (size_t)b * C + row);
      out[o] = acc / (1.f + expf(-acc)) + hv;
    } else {
      out[o] = acc;
    }
  };

  int r = w_lo;
  for (; r + kRowsPerWarp <= w_hi; r += kRowsPerWarp) {
    float acc[kRowsPerWarp][BB];
    warp_rows<TW, BB, kRowsPerWarp>(Wk + (size_t)r * C, C, xs, lane, acc);
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
      for (int bb = 0; bb < BB; ++bb)
        if (lane == ((i * BB + bb) & 31)) emit(r + i, bb, acc[i][bb]);
  }
  for (; r < w_hi; ++r) {
    float acc[1][BB];
    warp_rows<TW, BB, 1>(Wk + (size_t)r * C, C, xs, lane, acc);
#pragma unroll
    for (int bb = 0; bb < BB; ++bb)
      if (lane == (bb & 31)) emit(r, bb, acc[0][bb]);
  }
}

// ------------------------------------------------------------------- top-k

constexpr int kTopkChunk = 2048;  // values per partial CTA
constexpr int kTopkMaxChunks = 64;

inline int topk_chunks(int V) {
  int c = ceil_div(V, kTopkChunk);
  return c < 1 ? 1 : (c > kTopkMaxChunks ? kTopkMaxChunks : c);
}

// Inserts (v, i) into the thread's sorted list (column `tid` of s_val/s_idx,
// KC slots, best first) if it ranks ahead of the last kept entry.
template <int KC, int NT>
__device__ __forceinline__ void list_insert(float* s_val, int* s_idx, int tid, float v, int i,
                                            float& worst_v, int& worst_i) {
  if (!ranks_ahead(v, i, worst_v, worst_i)) return;
  int pos = KC - 1;
  while (pos > 0) {
    float pv = s_val[(pos - 1) * NT + tid];
    int pi = s_idx[(pos - 1) * NT + tid];
    if (!ranks_ahead(v, i, pv, pi)) break;
    s_val[pos * NT + tid] = pv;
    s_idx[pos * NT + tid] = pi;
    --pos;
  }
  s_val[pos * NT + tid] = v;
  s_idx[pos * NT + tid] = i;
  worst_v = s_val[(KC - 1) * NT + tid];
  worst_i = s_idx[(KC - 1) * NT + tid];
}

// One CTA ranks either a slice of a dense row (index = column) or a list of
// (value, index) candidates (x_idx != NULL).  Grid (chunks, rows); writes
// topk entries per (row, chunk), best first.  Every thread keeps its own
// sorted list of KC entries in shared memory; the lists are then merged by
// topk rounds of a block-wide argmax over the list heads.
template <int KC, int NT>
__global__ void __launch_bounds__(NT)
topk_kernel(const float* __restrict__ x, const int* __restrict__ x_idx, int n_per_row, int chunks,
            int topk, float* __restrict__ out_val, int* __restrict__ out_idx) {
  __shared__ float s_val[KC * NT];
  __shared__ int s_idx[KC * NT];
  __shared__ float w_val[NT / 32];
  __shared__ int w_idx[NT / 32], w_own[NT / 32];
  __shared__ int win_own;

  const int tid = threadIdx.x, row = blockIdx.y, chunk = blockIdx.x;
  const int lo = (int)((long long)n_per_row * chunk / chunks);
  const int hi = (int)((long long)n_per_row * (chunk + 1) / chunks);
#pragma unroll
  for (int j = 0; j < KC; ++j) {
    s_val[j * NT + tid] = -INFINITY;
    s_idx[j * NT + tid] = INT_MAX;
  }
  float worst_v = -INFINITY;
  int worst_i = INT_MAX;
  const float* xr = x + (size_t)row * n_per_row;
  const int* xi = x_idx ? x_idx + (size_t)row * n_per_row : nullptr;
  for (int p = lo + tid; p < hi; p += NT) {
    float v = xr[p];
    int i = xi ? xi[p] : p;
    list_insert<KC, NT>(s_val, s_idx, tid, v, i, worst_v, worst_i);
  }

  int head = 0;
  const int lane = tid & 31, warp = tid >> 5;
  float* ov = out_val + ((size_t)row * chunks + chunk) * topk;
  int* oi = out_idx + ((size_t)row * chunks + chunk) * topk;
  for (int r = 0; r < topk; ++r) {
    float v = head < KC ? s_val[head * NT + tid] : -INFINITY;
    int i = head < KC ? s_idx[head * NT + tid] : INT_MAX;
    int own = tid;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      float v2 = __shfl_xor_sync(0xffffffffu, v, o);
      int i2 = __shfl_xor_sync(0xffffffffu, i, o);
      int own2 = __shfl_xor_sync(0xffffffffu, own, o);
      if (ranks_ahead(v2, i2, v, i) || (v2 == v && i2 == i && own2 < own)) { v = v2; i = i2; own = own2; }
    }
    if (lane == 0) { w_val[warp] = v; w_idx[warp] = i; w_own[warp] = own; }
    __syncthreads();
    if (tid == 0) {
      float bv = w_val[0]; int bi = w_idx[0], bo = w_own[0];
      for (int w = 1; w < NT / 32; ++w)
        if (ranks_ahead(w_val[w], w_idx[w], bv, bi)) { bv = w_val[w]; bi = w_idx[w]; bo = w_own[w]; }
      ov[r] = bv;
      oi[r] = bi;
      win_own = bo;
    }
    __syncthreads();
    if (tid == win_own) ++head;
    __syncthreads();
  }
}

static medusa_status launch_topk(const float* x, int rows, int V, int topk, float* cand_val, int* cand_idx,
                                 float* out_val, int* out_idx, cudaStream_t s) {
  const int chunks = topk_chunks(V);
  auto run = [&](const float* src, const int* src_idx, int n, int nch, float* dv, int* di) {
    dim3 grid(nch, rows);
    if (topk <= 4) topk_kernel<4, 256><<<grid, 256, 0, s>>>(src, src_idx, n, nch, topk, dv, di);
    else if (topk <= 8) topk_kernel<8, 256><<<grid, 256, 0, s>>>(src, src_idx, n, nch, topk, dv, di);
    else if (topk <= 16) topk_kernel<16, 256><<<grid, 256, 0, s>>>(src, src_idx, n, nch, topk, dv, di);
    else topk_kernel<32, 128><<<grid, 128, 0, s>>>(src, src_idx, n, nch, topk, dv, di);
  };
  if (chunks == 1) {
    run(x, nullptr, V, 1, out_val, out_idx);
  } else {
    run(x, nullptr, V, chunks, cand_val, cand_idx);
    run(cand_val, cand_idx, chunks * topk, 1, out_val, out_idx);
  }
  return launch_status();
}

static size_t topk_ws_bytes(int rows, int V, int topk) {
  WsCarver w(nullptr);
  w.take<float>((size_t)rows * topk_chunks(V) * topk);
  w.take<int>((size_t)rows * topk_chunks(V) * topk);
  return w.used;
}

// ------------------------------------------------------------------- GEMV launch

template <typename TW, bool kFirst>
static void launch_gemv_bb(int BB, const TW* W, const TW* h, const float* u, int B, int b0, int K,
                           int rows_per_head, int C, float* out, cudaStream_t s) {
  const size_t smem = (size_t)BB * C * sizeof(float);
  auto go = [&](auto kern) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGemvThreads, smem);
    if (per_sm < 1) per_sm = 1;
    int total = per_sm * device_sm_count();
    int per_head = total / K;
    if (per_head < 1) per_head = 1;
    int max_useful = ceil_div(rows_per_head, kRowsPerWarp);
    if (per_head > max_useful) per_head = max_useful;
    kern<<<dim3(per_head, K), kGemvThreads, smem, s>>>(W, h, u, B, b0, K, rows_per_head, C, out);
  };
  switch (BB) {
    case 1: go(heads_gemv_kernel<TW, 1, kFirst>); break;
    case 2: go(heads_gemv_kernel<TW, 2, kFirst>); break;
    case 4: go(heads_gemv_kernel<TW, 4, kFirst>); break;
    default: go(heads_gemv_kernel<TW, 8, kFirst>); break;
  }
}

template <typename TW>
static void launch_heads_gemv(const TW* h, const TW* w1, const TW* w2, int B, int H, int V, int K,
                              float* u, float* z, cudaStream_t s) {
  for (int b0 = 0; b0 < B; b0 += kMaxBatchPerPass) {
    int nb = B - b0 < kMaxBatchPerPass ? B - b0 : kMaxBatchPerPass;
    int BB = nb <= 1 ? 1 : nb <= 2 ? 2 : nb <= 4 ? 4 : 8;
    launch_gemv_bb<TW, true>(BB, w1, h, nullptr, B, b0, K, H, H, u, s);
  }
  for (int b0 = 0; b0 < B; b0 += kMaxBatchPerPass) {
    int nb = B - b0 < kMaxBatchPerPass ? B - b0 : kMaxBatchPerPass;
    int BB = nb <= 1 ? 1 : nb <= 2 ? 2 : nb <= 4 ? 4 : 8;
    launch_gemv_bb<TW, false>(BB, w2, nullptr, u, B, b0, K, V, H, z, s);
  }
}

static size_t heads_ws_bytes(int B, int H, int V, int K, int topk, bool need_z) {
  WsCarver w(nullptr);
  w.take<float>((size_t)B * K * H);
  if (need_z) w.take<float>((size_t)B * K * V);
  w.take<float>((size_t)B * K * topk_chunks(V) * topk);
  w.take<int>((size_t)B * K * topk_chunks(V) * topk);
  return w.used;
}

}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_heads_workspace_size(int B, int H, int V, int K, int topk) {
  if (B <= 0 || H <= 0 || V <= 0 || K <= 0 || topk <= 0) return 0;
  return heads_ws_bytes(B, H, V, K, topk, true);
}

extern "C" medusa_status medusa_heads(const void* h, const void* w1, const void* w2, int B, int H,
                                      int V, int K, int topk, medusa_dtype dt, int32_t* topk_idx,
                                      float* topk_logit, float* logits_or_null, void* ws,
                                      size_t ws_bytes, int32_t* d_status, medusa_stream_t stream) {
  (void)d_status;
  if (!h || !w1 || !w2 || !topk_idx || !topk_logit) return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > 64 || H < 8 || H % 8 || V < 1 || K < 1 || K > MEDUSA_MAX_DEPTH) return MEDUSA_ERR_INVALID_ARG;
  if (topk < 1 || topk > MEDUSA_MAX_TOPK || topk > V || !dtype_ok(dt)) return MEDUSA_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w1) || !aligned16(w2)) return MEDUSA_ERR_INVALID_ARG;
  if (logits_or_null && !aligned16(logits_or_null)) return MEDUSA_ERR_INVALID_ARG;
  const int bb_max = B > 4 ? 8 : B > 2 ? 4 : B > 1 ? 2 : 1;
  if ((size_t)bb_max * H * sizeof(float) > 220 * 1024) return MEDUSA_ERR_UNSUPPORTED;
  const bool need_z = logits_or_null == nullptr;
  if (!ws || ws_bytes < heads_ws_bytes(B, H, V, K, topk, need_z)) return MEDUSA_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  WsCarver wc(ws);
  float* u = wc.take<float>((size_t)B * K * H);
  float* z = need_z ? wc.take<float>((size_t)B * K * V) : logits_or_null;
  float* cv = wc.take<float>((size_t)B * K * topk_chunks(V) * topk);
  int* ci = wc.take<int>((size_t)B * K * topk_chunks(V) * topk);
  if (dt == MEDUSA_BF16)
    launch_heads_gemv<uint16_t>((const uint16_t*)h, (const uint16_t*)w1, (const uint16_t*)w2, B, H, V, K, u, z, s);
  else
    launch_heads_gemv<float>((const float*)h, (const float*)w1, (const float*)w2, B, H, V, K, u, z, s);
  medusa_status st = launch_status();
  if (st != MEDUSA_OK) return st;
  return launch_topk(z, B * K, V, topk, cv, ci, topk_logit, topk_idx, s);
}

extern "C" size_t medusa_head_topk_workspace_size(int rows, int V, int topk) {
  if (rows <= 0 || V <= 0 || topk <= 0) return 0;
  return topk_ws_bytes(rows, V, topk);
}

extern "C" medusa_status medusa_head_topk(const float* logits, int rows, int V, int topk,
                                          int32_t* topk_idx, float* topk_logit, void* ws,
                                          size_t ws_bytes, medusa_stream_t stream) {
  if (!logits || !topk_idx || !topk_logit || rows < 1 || V < 1) return MEDUSA_ERR_INVALID_ARG;
  if (topk < 1 || topk > MEDUSA_MAX_TOPK || topk > V) return MEDUSA_ERR_INVALID_ARG;
  if (topk_chunks(V) > 1 && (!ws || ws_bytes < topk_ws_bytes(rows, V, topk))) return MEDUSA_ERR_WORKSPACE;
  WsCarver wc(ws);
  float* cv = wc.take<float>((size_t)rows * topk_chunks(V) * topk);
  int* ci = wc.take<int>((size_t)rows * topk_chunks(V) * topk);
  return launch_topk(logits, rows, V, topk, cv, ci, topk_logit, topk_idx,
                     reinterpret_cast<cudaStream_t>(stream));
}
