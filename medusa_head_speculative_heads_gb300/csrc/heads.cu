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
// shared memory as fp32.  The top-k is fused: every W2 CTA ranks its own slice
// of the vocabulary (one warp per batch row) and the last CTA of each head
// merges the per-CTA candidate lists (a separate merge kernel only when they
// do not fit its shared memory).
#include <float.h>
#include <limits.h>

#include <type_traits>

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
// BB staged vectors.  Lane l reads 16-byte chunks l, l+32, ... of each row, U
// chunks per row per iteration with U * NR ~ 8 loads in flight per lane
// whatever the row count (a warp left with one or two rows would otherwise
// walk its rows one latency at a time).  Chunks are accumulated in ascending
// order in every case.
template <typename TW, int BB, int NR>
__device__ __forceinline__ void warp_rows(const TW* __restrict__ W, int C, const float* __restrict__ xs,
                                          int lane, float (&acc)[NR][BB]) {
  constexpr int VEC = Vec16<TW>::n;
  constexpr int STEP = 32 * VEC;
  constexpr int U = NR >= 4 ? 2 : (8 + NR - 1) / NR;
#pragma unroll
  for (int i = 0; i < NR; ++i)
#pragma unroll
    for (int bb = 0; bb < BB; ++bb) acc[i][bb] = 0.f;
  int c = lane * VEC;
  for (; c + (U - 1) * STEP < C; c += U * STEP) {
    uint4 w[U][NR];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < NR; ++i) w[u][i] = ldg_stream(W + (size_t)i * C + c + u * STEP);
#pragma unroll
    for (int u = 0; u < U; ++u) fma_chunk<TW, BB, NR>(w[u], xs, C, c + u * STEP, acc);
  }
  for (; c < C; c += STEP) {
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

// Warp-level top-k: ranks the n values v[0..n) (index idx[i], or base + i when
// idx is null) by (value desc, index asc) and writes the best `topk` to
// out_v/out_i (lane 0 writes).  Each round every lane scans its strided values
// for the best one ranked strictly behind the previous round's winner, then a
// shuffle argmax picks the round's winner: no shared state, no block barrier.
// v/idx should live in shared memory (every round re-reads them).
__device__ __forceinline__ void warp_topk(const float* v, const int* idx, int n, int base, int topk,
                                          float* out_v, int* out_i) {
  const int lane = threadIdx.x & 31;
  float pv = INFINITY;
  int pi = -1;
  for (int r = 0; r < topk; ++r) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int i = lane; i < n; i += 32) {
      const float val = v[i];
      const int id = idx ? idx[i] : base + i;
      if (ranks_ahead(pv, pi, val, id) && ranks_ahead(val, id, bv, bi)) { bv = val; bi = id; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ranks_ahead(v2, i2, bv, bi)) { bv = v2; bi = i2; }
    }
    if (lane == 0) { out_v[r] = bv; out_i[r] = bi; }
    pv = bv;
    pi = bi;
  }
}

// Bitonic sort of one (value, index) pair per lane across the warp, best
// first (value descending, index ascending): afterwards lane r holds the
// pair of rank r.  Every lane must take part.
__device__ __forceinline__ void warp_sort32(float& v, int& id) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, j);
      const int oi = __shfl_xor_sync(0xffffffffu, id, j);
      // in a block of k lanes sorted best-first (bit k clear) the lower lane
      // of each pair keeps the better element; in the others, the worse
      const bool keep_better = ((lane & j) == 0) == ((lane & k) == 0);
      if (keep_better == ranks_ahead(ov, oi, v, id)) { v = ov; id = oi; }
    }
  }
}

// warp_topk with the values held in registers: lane l keeps v[l + 32 j],
// j < RV (n <= 32 RV), read from shared memory once.  Same ranking and output
// as warp_topk (idx null: index base + i).  First a threshold: the lanes'
// best pairs are distinct elements, so the topk-th best of them, (T, Ti),
// ranks at or behind the row's topk-th best, and every top-k pair ranks at or
// ahead of it; when at most 32 pairs do (the usual case), they go through
// s_v / s_i (32 entries of shared memory) into one warp sort.  Otherwise topk
// rounds of register compares and the shuffle argmax.  Both keep the
// dependent shuffle steps few: at the end of a streaming pass, with other
// CTAs still loading, each one waits behind their memory traffic.
template <int RV>
__device__ __forceinline__ void warp_topk_regs(const float* v, int n, int base, int topk, float* out_v, int* out_i,
                                               float* s_v, int* s_i) {
  const int lane = threadIdx.x & 31;
  float x[RV];
#pragma unroll
  for (int j = 0; j < RV; ++j) x[j] = lane + 32 * j < n ? v[lane + 32 * j] : -INFINITY;
  float lv = -INFINITY;
  int li = INT_MAX;
#pragma unroll
  for (int j = 0; j < RV; ++j)
    if (lane + 32 * j < n && ranks_ahead(x[j], base + lane + 32 * j, lv, li)) {
      lv = x[j];
      li = base + lane + 32 * j;
    }
  warp_sort32(lv, li);
  const float T = __shfl_sync(0xffffffffu, lv, topk - 1);
  const int Ti = __shfl_sync(0xffffffffu, li, topk - 1);
  auto cand = [&](int j) {
    const int id = base + lane + 32 * j;
    return lane + 32 * j < n && (ranks_ahead(x[j], id, T, Ti) || (x[j] == T && id == Ti));
  };
  int c = 0;
#pragma unroll
  for (int j = 0; j < RV; ++j) c += cand(j) ? 1 : 0;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (total <= 32) {
    int pos = incl - c;
#pragma unroll
    for (int j = 0; j < RV; ++j)
      if (cand(j)) {
        s_v[pos] = x[j];
        s_i[pos] = base + lane + 32 * j;
        ++pos;
      }
    __syncwarp();
    float cv = lane < total ? s_v[lane] : -INFINITY;
    int ci = lane < total ? s_i[lane] : INT_MAX;
    __syncwarp();
    warp_sort32(cv, ci);
    if (lane < topk) { out_v[lane] = cv; out_i[lane] = ci; }
    return;
  }
  float pv = INFINITY;
  int pi = -1;
  for (int r = 0; r < topk; ++r) {
    float bv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int j = 0; j < RV; ++j) {
      const int id = base + lane + 32 * j;
      if (lane + 32 * j < n && ranks_ahead(pv, pi, x[j], id) && ranks_ahead(x[j], id, bv, bi)) {
        bv = x[j];
        bi = id;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ranks_ahead(v2, i2, bv, bi)) { bv = v2; bi = i2; }
    }
    if (lane == 0) { out_v[r] = bv; out_i[r] = bi; }
    pv = bv;
    pi = bi;
  }
}

// warp_merge_sorted with each lane owning lists lane + 32 j (j < LPL, so
// nlists <= 32 LPL): their head positions and head pairs live in registers;
// a round compares them, takes the shuffle argmax (with the owning lane), and
// only the winning lane reads its list's next pair.
template <int LPL>
__device__ __forceinline__ void warp_merge_sorted_regs(const float* v, const int* idx, int nlists, int len, int topk,
                                                       float* out_v, int* out_i) {
  const int lane = threadIdx.x & 31;
  int hpos[LPL];
  float hv[LPL];
  int hi[LPL];
#pragma unroll
  for (int j = 0; j < LPL; ++j) {
    const int L = lane + 32 * j;
    hpos[j] = 0;
    const bool ok = L < nlists && len > 0;
    hv[j] = ok ? v[L * len] : -INFINITY;
    hi[j] = ok ? idx[L * len] : INT_MAX;
  }
  for (int r = 0; r < topk; ++r) {
    float bv = -INFINITY;
    int bi = INT_MAX, bl = -1;
#pragma unroll
    for (int j = 0; j < LPL; ++j)
      if (lane + 32 * j < nlists && hpos[j] < len && ranks_ahead(hv[j], hi[j], bv, bi)) {
        bv = hv[j];
        bi = hi[j];
        bl = lane + 32 * j;
      }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      const int l2 = __shfl_xor_sync(0xffffffffu, bl, o);
      if (ranks_ahead(v2, i2, bv, bi)) { bv = v2; bi = i2; bl = l2; }
    }
    if (lane == 0) { out_v[r] = bv; out_i[r] = bi; }
    // the owner of the winning list moves to its next pair
    if (bl >= 0 && (bl & 31) == lane) {
#pragma unroll
      for (int j = 0; j < LPL; ++j)
        if (bl == lane + 32 * j) {
          const int p = ++hpos[j];
          hv[j] = p < len ? v[bl * len + p] : -INFINITY;
          hi[j] = p < len ? idx[bl * len + p] : INT_MAX;
        }
    }
  }
}

// Warp-level merge of `nlists` lists, each sorted best first and `len` long
// (v/idx[list * len + j]), into the best `topk` (lane 0 writes out_v/out_i).
// Each round compares only the lists' current heads; hp[] (shared memory,
// nlists ints) holds the head positions.
__device__ __forceinline__ void warp_merge_sorted(const float* v, const int* idx, int nlists, int len, int topk,
                                                  int* hp, float* out_v, int* out_i) {
  const int lane = threadIdx.x & 31;
  for (int L = lane; L < nlists; L += 32) hp[L] = 0;
  __syncwarp();
  for (int r = 0; r < topk; ++r) {
    float bv = -INFINITY;
    int bi = INT_MAX, bl = -1;
    for (int L = lane; L < nlists; L += 32) {
      const int hpos = hp[L];
      if (hpos < len) {
        const float val = v[L * len + hpos];
        const int id = idx[L * len + hpos];
        if (ranks_ahead(val, id, bv, bi)) { bv = val; bi = id; bl = L; }
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      const int l2 = __shfl_xor_sync(0xffffffffu, bl, o);
      if (ranks_ahead(v2, i2, bv, bi)) { bv = v2; bi = i2; bl = l2; }
    }
    if (lane == 0) {
      out_v[r] = bv;
      out_i[r] = bi;
      if (bl >= 0) hp[bl] += 1;
    }
    __syncwarp();
  }
}

// kFirst = true : rows are W1 rows; x = h (batch rows b0..b0+BB-1);
//                 u[b][k][j] = SiLU(acc) + h[b][j]                  (fp32)
// kFirst = false: rows are W2 rows; x = u[b][k]; z = acc goes to `out` when
//                 requested, and the CTA ranks its own rows: the top-k of its
//                 slice of every (b, k) vocabulary row is written to
//                 cand_{v,i}[(b*K + k) * gridDim.x + blockIdx.x][topk].
// Grid (ctas_per_head, K); block 256; dynamic smem BB * C floats (+ BB * cap
// floats holding the CTA's logits for the ranking).
// One vector (the decode case), measured per step: the W1 pass runs four CTAs
// per SM (64 registers, no spills; five CTAs at 48 registers spilled and the
// step was ~0.7 % slower) and the W2 pass is left to the compiler (80
// registers, no spills, three CTAs per SM).  Both at five: W2 spilled and the
// step was 7.5 us slower; both at six: far slower.
template <typename TW, int BB, bool kFirst>
__global__ void __launch_bounds__(kGemvThreads, BB == 1 && kFirst ? 4 : 1)
heads_gemv_kernel(const TW* __restrict__ W, const TW* __restrict__ h, const float* __restrict__ u,
                  int B, int b0, int K, int rows_per_head, int C, float* __restrict__ out, int topk,
                  float* __restrict__ cand_v, int* __restrict__ cand_i, int* __restrict__ counters,
                  int n_counters, float* __restrict__ top_v, int* __restrict__ top_i) {
  extern __shared__ float xs[];  // [BB][C], then [BB][cap]
  __shared__ int s_last;
  __shared__ float s_tv[kFirst ? 1 : kGemvWarps][32];  // a ranking warp's threshold candidates
  __shared__ int s_ti[kFirst ? 1 : kGemvWarps][32];
  // Balanced contiguous row ranges: CTA, then warp (launch parameters only).
  const int ctas = gridDim.x;
  const int cap = (rows_per_head + ctas - 1) / ctas;
  const int r_lo = (int)((long long)rows_per_head * blockIdx.x / ctas);
  const int r_hi = (int)((long long)rows_per_head * (blockIdx.x + 1) / ctas);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = r_hi - r_lo;
  const int w_lo = r_lo + n * warp / kGemvWarps;
  const int w_hi = r_lo + n * (warp + 1) / kGemvWarps;
  const TW* Wk = W + (size_t)blockIdx.y * rows_per_head * C;
  // The weights are never written during a step: while an earlier kernel on
  // the stream finishes, warm L2 with this warp's first row.
  if (w_hi > w_lo) {
    const char* row0 = reinterpret_cast<const char*>(Wk + (size_t)w_lo * C);
    for (int off = lane * 128; off < C * (int)sizeof(TW); off += 32 * 128) prefetch_l2(row0 + off);
  }
  pdl_wait();
  pdl_trigger();
  const int k = blockIdx.y;
  if constexpr (kFirst) {
    // The W2 passes that follow count their finished CTAs here.
    if (b0 == 0 && blockIdx.x == 0 && blockIdx.y == 0)
      for (int i = threadIdx.x; i < n_counters; i += kGemvThreads) counters[i] = 0;
  }
  // Stage the vector(s) in shared memory: 16-byte loads, four per thread issued
  // before the first store (one round trip, not one per element), rows past B
  // as zeros; element by element when the rows are not 16-byte aligned.
  constexpr int XV = kFirst ? Vec16<TW>::n : 4;  // elements per 16-byte chunk
  const void* x_base = kFirst ? static_cast<const void*>(h) : static_cast<const void*>(u);
  if (C % XV == 0 && (reinterpret_cast<uintptr_t>(x_base) & 15u) == 0) {
    constexpr int XU = 4;
    const int per_row = C / XV, nch = BB * per_row;
    for (int i0 = threadIdx.x; i0 < nch; i0 += kGemvThreads * XU) {
      uint4 raw[XU];
#pragma unroll
      for (int j = 0; j < XU; ++j) {
        const int i = i0 + j * kGemvThreads, bb = i / per_row, cc = i - bb * per_row, b = b0 + bb;
        raw[j] = make_uint4(0u, 0u, 0u, 0u);
        if (i < nch && b < B)
          raw[j] = kFirst ? *reinterpret_cast<const uint4*>(h + (size_t)b * C + (size_t)cc * XV)
                          : *reinterpret_cast<const uint4*>(u + ((size_t)b * K + k) * C + (size_t)cc * XV);
      }
#pragma unroll
      for (int j = 0; j < XU; ++j) {
        const int i = i0 + j * kGemvThreads;
        if (i >= nch) break;
        float f[XV];
        if constexpr (XV == 8) unpack_bf16x8(raw[j], f);
        else unpack_f32x4(raw[j], f);
        float4* dst = reinterpret_cast<float4*>(xs + (size_t)i * XV);
#pragma unroll
        for (int e = 0; e < XV / 4; ++e) dst[e] = make_float4(f[4 * e], f[4 * e + 1], f[4 * e + 2], f[4 * e + 3]);
      }
    }
  } else {
    for (int idx = threadIdx.x; idx < BB * C; idx += kGemvThreads) {
      int bb = idx / C, c = idx - bb * C, b = b0 + bb;
      float v = 0.f;
      if (b < B) v = kFirst ? load_elem<TW>(h, (size_t)b * C + c) : u[((size_t)b * K + k) * C + c];
      xs[idx] = v;
    }
  }
  __syncthreads();

  float* zs = xs + BB * C;

  auto emit = [&](int row, int bb, float acc) {
    int b = b0 + bb;
    if (b >= B) return;
    size_t o = ((size_t)b * K + k) * rows_per_head + row;
    if constexpr (kFirst) {
      float hv = load_elem<TW>(h, (size_t)b * C + row);
      out[o] = acc / (1.f + expf(-acc)) + hv;
    } else {
      if (out) out[o] = acc;
      zs[bb * cap + (row - r_lo)] = acc;
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
  // The remaining 1-3 rows in one pass (their loads in flight together).
  auto tail = [&](auto nr) {
    constexpr int NR = decltype(nr)::value;
    float acc[NR][BB];
    warp_rows<TW, BB, NR>(Wk + (size_t)r * C, C, xs, lane, acc);
#pragma unroll
    for (int i = 0; i < NR; ++i)
#pragma unroll
      for (int bb = 0; bb < BB; ++bb)
        if (lane == ((i * BB + bb) & 31)) emit(r + i, bb, acc[i][bb]);
  };
  switch (w_hi - r) {
    case 3: tail(std::integral_constant<int, 3>{}); break;
    case 2: tail(std::integral_constant<int, 2>{}); break;
    case 1: tail(std::integral_constant<int, 1>{}); break;
    default: break;
  }
  if constexpr (!kFirst) {
    __syncthreads();
    for (int bb = warp; bb < BB; bb += kGemvWarps) {
      const int b = b0 + bb;
      if (b >= B) continue;
      const size_t row = ((size_t)b * K + k) * ctas + blockIdx.x;
      if (n <= 32 * 12)
        warp_topk_regs<12>(zs + bb * cap, n, r_lo, topk, cand_v + row * topk, cand_i + row * topk, s_tv[warp],
                           s_ti[warp]);
      else
        warp_topk(zs + bb * cap, nullptr, n, r_lo, topk, cand_v + row * topk, cand_i + row * topk);
    }
    if (top_v) {
      // The last CTA of this head (in this batch pass) merges every CTA's
      // sorted candidate list: candidates are published with a fence before
      // the counter increment, and read back through L2.
      __threadfence();
      __syncthreads();
      int* cnt = counters + (b0 / kMaxBatchPerPass) * K + k;
      if (threadIdx.x == 0) s_last = atomicAdd(cnt, 1) == ctas - 1;
      __syncthreads();
      if (s_last) {
        __threadfence();
        float* mv = xs;  // the staged x is no longer needed: [BB][ctas * topk] values
        int* mi = reinterpret_cast<int*>(xs + BB * ctas * topk);
        int* hp = mi + BB * ctas * topk;
        for (int bb = 0; bb < BB; ++bb) {
          const int b = b0 + bb;
          if (b >= B) continue;
          const size_t base = ((size_t)b * K + k) * ctas * topk;
          // every load of a thread in flight before its first store (one round trip)
          constexpr int MU = 8;
          const int n = ctas * topk;
          for (int i0 = threadIdx.x; i0 < n; i0 += kGemvThreads * MU) {
            float cv[MU];
            int ci[MU];
#pragma unroll
            for (int j = 0; j < MU; ++j) {
              const int i = i0 + j * kGemvThreads;
              if (i < n) {
                cv[j] = __ldcg(cand_v + base + i);
                ci[j] = __ldcg(cand_i + base + i);
              }
            }
#pragma unroll
            for (int j = 0; j < MU; ++j) {
              const int i = i0 + j * kGemvThreads;
              if (i < n) {
                mv[bb * n + i] = cv[j];
                mi[bb * n + i] = ci[j];
              }
            }
          }
        }
        __syncthreads();
        for (int bb = warp; bb < BB; bb += kGemvWarps) {
          const int b = b0 + bb;
          if (b >= B) continue;
          const size_t o = ((size_t)b * K + k) * topk;
          if (ctas <= 32 * 4)
            warp_merge_sorted_regs<4>(mv + bb * ctas * topk, mi + bb * ctas * topk, ctas, topk, topk, top_v + o,
                                      top_i + o);
          else
            warp_merge_sorted(mv + bb * ctas * topk, mi + bb * ctas * topk, ctas, topk, topk, hp + warp * ctas,
                            top_v + o, top_i + o);
        }
        if (threadIdx.x == 0) *cnt = 0;
      }
    }
  }
}

// ------------------------------------------------------------------- top-k

constexpr int kTopkThreads = 256;
constexpr int kTopkChunk = 4096;  // (value, index) pairs one CTA stages and ranks

inline int chunks_for(long long n) {
  long long c = (n + kTopkChunk - 1) / kTopkChunk;
  return c < 1 ? 1 : (int)c;
}

// One CTA ranks a slice (<= kTopkChunk pairs) of one row: (value, index)
// pairs, index = column when x_idx is null.  The slice is staged in shared
// memory once; every warp ranks a sub-slice with warp_topk, then warp 0 ranks
// the 8 x topk survivors.  Grid (chunks, rows); out[row][chunk][topk].
__global__ void __launch_bounds__(kTopkThreads)
topk_block_kernel(const float* __restrict__ x, const int* __restrict__ x_idx, int n_per_row, int chunks,
                  int topk, float* __restrict__ out_v, int* __restrict__ out_i) {
  __shared__ float cv[kTopkChunk];
  __shared__ int ci[kTopkChunk];
  __shared__ float sv[kTopkThreads / 32 * MEDUSA_MAX_TOPK];
  __shared__ int si[kTopkThreads / 32 * MEDUSA_MAX_TOPK];
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y, chunk = blockIdx.x, warp = threadIdx.x >> 5;
  const int lo = (int)((long long)n_per_row * chunk / chunks);
  const int hi = (int)((long long)n_per_row * (chunk + 1) / chunks);
  const int n = hi - lo;  // <= kTopkChunk by construction of `chunks`
  const float* xr = x + (size_t)row * n_per_row + lo;
  const int* xi = x_idx ? x_idx + (size_t)row * n_per_row + lo : nullptr;
  for (int i = threadIdx.x; i < n; i += kTopkThreads) {
    cv[i] = xr[i];
    ci[i] = xi ? xi[i] : lo + i;
  }
  __syncthreads();
  const int w_lo = (int)((long long)n * warp / (kTopkThreads / 32));
  const int w_hi = (int)((long long)n * (warp + 1) / (kTopkThreads / 32));
  warp_topk(cv + w_lo, ci + w_lo, w_hi - w_lo, 0, topk, sv + warp * topk, si + warp * topk);
  __syncthreads();
  if (warp == 0) {
    const size_t o = ((size_t)row * chunks + chunk) * topk;
    warp_topk(sv, si, (kTopkThreads / 32) * topk, 0, topk, out_v + o, out_i + o);
  }
}

// One CTA per row: the best `topk` (<= kRowTopkMax) of n logits, ranked
// (value desc, index asc), in two passes over the row with few divergent
// branches.
//  1. Every thread takes the best of its values; the topk-th best of these
//     thread maxima (found by one warp), T, is a lower bound for the row's topk-th best (at least
//     topk distinct values, the maxima ranked at or ahead of T, rank at or
//     ahead of T), so every one of the row's best topk ranks at or ahead of T.
//  2. The row is read again (from L1/L2) and the values ranked at or ahead of
//     T, typically a few dozen, are appended to shared memory.
//  3. topk rounds of a warp argmax over those candidates, each taking the
//     best one ranked behind the previous round's winner, give the result in
//     order.  Should more candidates than fit rank at or ahead of T, the
//     rounds scan the whole row with the whole block instead (exact, slower).
// Grid rows; out[row][topk].
constexpr int kRowThreads = 256;
constexpr int kRowCap = 2048;  // candidates kept in shared memory

// Warp-wide best (value, index) of the lanes' arguments; every lane gets it.
__device__ __forceinline__ void warp_best(float& v, int& id) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, id, o);
    if (ranks_ahead(v2, i2, v, id)) { v = v2; id = i2; }
  }
}

// Block-wide best (value, index) of the threads' arguments; every thread gets it.
__device__ __forceinline__ void block_best(float& v, int& id, float* sv, int* si) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_best(v, id);
  if (lane == 0) { sv[warp] = v; si[warp] = id; }
  __syncthreads();
  v = sv[0];
  id = si[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
    if (ranks_ahead(sv[w], si[w], v, id)) { v = sv[w]; id = si[w]; }
  __syncthreads();
}


__global__ void __launch_bounds__(kRowThreads)
topk_rows_kernel(const float* __restrict__ x, int n, int topk, float* __restrict__ out_v, int* __restrict__ out_i) {
  __shared__ float cv[kRowCap];
  __shared__ int ci[kRowCap];
  __shared__ float sv[kRowThreads / 32];
  __shared__ int si[kRowThreads / 32];
  __shared__ int s_count;
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, tid = threadIdx.x;
  const float* xr = x + (size_t)row * n;
  const bool vec = (n & 3) == 0 && (reinterpret_cast<uintptr_t>(xr) & 15u) == 0;
  const int n4 = n >> 2;
  // Visits every (value, index) of this thread's share of the row.
  auto scan = [&](auto&& f) {
    if (vec) {
      const float4* x4 = reinterpret_cast<const float4*>(xr);
      constexpr int U = 4;
      for (int q0 = tid; q0 < n4; q0 += kRowThreads * U) {
        float4 t[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int q = q0 + u * kRowThreads;
          if (q < n4) t[u] = x4[q];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int q = q0 + u * kRowThreads;
          if (q < n4) {
            f(t[u].x, 4 * q);
            f(t[u].y, 4 * q + 1);
            f(t[u].z, 4 * q + 2);
            f(t[u].w, 4 * q + 3);
          }
        }
      }
    } else {
      for (int i = tid; i < n; i += kRowThreads) f(xr[i], i);
    }
  };
  // 1. thread maxima, then the topk-th best of them (warp 0 alone)
  float mv = -INFINITY;
  int mi = INT_MAX;
  scan([&](float v, int i) {
    if (ranks_ahead(v, i, mv, mi)) { mv = v; mi = i; }
  });
  cv[tid] = mv;
  ci[tid] = mi;
  __syncthreads();
  if (tid < 32) {
    float pv = INFINITY;
    int pi = -1;
    for (int r = 0; r < topk; ++r) {
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int j = tid; j < kRowThreads; j += 32)
        if (ranks_ahead(pv, pi, cv[j], ci[j]) && ranks_ahead(cv[j], ci[j], bv, bi)) { bv = cv[j]; bi = ci[j]; }
      warp_best(bv, bi);
      pv = bv;
      pi = bi;
    }
    if (tid == 0) { sv[0] = pv; si[0] = pi; s_count = 0; }
  }
  __syncthreads();
  const float tv = sv[0];
  const int ti = si[0];
  // 2. candidates ranked at or ahead of (tv, ti)
  scan([&](float v, int i) {
    if (!ranks_ahead(tv, ti, v, i)) {
      const int slot = atomicAdd(&s_count, 1);
      if (slot < kRowCap) { cv[slot] = v; ci[slot] = i; }
    }
  });
  __syncthreads();
  const int c = s_count;
  // 3. topk rounds, each the best candidate ranked behind the previous winner
  // (warp 0 over the shared-memory candidates; the whole block over the row
  // when they did not fit)
  float pv = INFINITY;
  int pi = -1;
  if (c <= kRowCap) {
    if (tid < 32) {
      for (int r = 0; r < topk; ++r) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int j = tid; j < c; j += 32)
          if (ranks_ahead(pv, pi, cv[j], ci[j]) && ranks_ahead(cv[j], ci[j], bv, bi)) { bv = cv[j]; bi = ci[j]; }
        warp_best(bv, bi);
        if (tid == 0) {
          out_v[(size_t)row * topk + r] = bv;
          out_i[(size_t)row * topk + r] = bi;
        }
        pv = bv;
        pi = bi;
      }
    }
    return;
  }
  for (int r = 0; r < topk; ++r) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    scan([&](float v, int i) {
      if (ranks_ahead(pv, pi, v, i) && ranks_ahead(v, i, bv, bi)) { bv = v; bi = i; }
    });
    block_best(bv, bi, sv, si);
    if (tid == 0) {
      out_v[(size_t)row * topk + r] = bv;
      out_i[(size_t)row * topk + r] = bi;
    }
    pv = bv;
    pi = bi;
  }
}

constexpr int kRowTopkMax = 32;  // topk the row kernels rank

// Top-k of rows whose 32-element group maxima are known (written by the
// tensor-core W2 epilogue): one warp per row, no block barrier.
//  1. Each lane loads the maxima of its groups (16-byte loads, all in flight
//     for up to kGroupRegs x 4 groups per lane) and takes their best (value,
//     group).  The lanes' group sets are disjoint, so the topk-th best of the
//     32 lane bests (a warp bitonic sort), T, is at most the row's topk-th
//     best value: topk distinct groups, hence topk distinct elements, reach it.
//  2. Only groups whose maximum reaches T can hold a value >= T; each lane
//     reads its own such groups (eight 16-byte loads each, usually none or
//     one per lane) and appends their values >= T (every top-k element among
//     them) to the warp's list in shared memory.
//  3. Up to 32 candidates (about topk + a few for smooth logits) are ranked
//     by one warp sort, up to kGroupCand by topk warp-argmax rounds over the
//     list; more (many equal values) by topk rounds over the qualifying
//     groups themselves.
// topk <= 32.  gmax[row][groups], groups a multiple of 4 (16-byte rows), group
// g = elements [32 g, 32 g + 32) of x[row][n].
constexpr int kGroupWarps = 8;  // rows per CTA
constexpr int kGroupCand = 64;  // candidates a warp keeps
constexpr int kGroupRegs = 8;   // 16-byte group-maxima loads a lane keeps in registers

__device__ __forceinline__ float f4_at(const float4& q, int u) {
  return u == 0 ? q.x : u == 1 ? q.y : u == 2 ? q.z : q.w;
}

// The 32 elements of group g of row xr (n elements), eight 16-byte loads in flight when aligned.
__device__ __forceinline__ void load_group(const float* __restrict__ xr, int n, bool vec, int g, float (&v)[32]) {
  const int e0 = 32 * g;
  if (vec && e0 + 32 <= n) {
    float4 q[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) q[k] = reinterpret_cast<const float4*>(xr + e0)[k];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[4 * k] = q[k].x;
      v[4 * k + 1] = q[k].y;
      v[4 * k + 2] = q[k].z;
      v[4 * k + 3] = q[k].w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = e0 + k < n ? xr[e0 + k] : -INFINITY;
  }
}

__global__ void __launch_bounds__(32 * kGroupWarps)
topk_groups_kernel(const float* __restrict__ x, const float* __restrict__ gmax, int n, int groups, int topk,
                   int rows, float* __restrict__ out_v, int* __restrict__ out_i) {
  __shared__ float cv[kGroupWarps][kGroupCand];
  __shared__ int ci[kGroupWarps][kGroupCand];
  __shared__ int cnt[kGroupWarps];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kGroupWarps + warp;
  if (row >= rows) return;  // the warps are independent: no block barrier follows
  const float* xr = x + (size_t)row * n;
  const float4* g4 = reinterpret_cast<const float4*>(gmax + (size_t)row * groups);
  const int chunks = groups >> 2;  // 4 groups per 16-byte chunk; lane takes chunks lane + 32 j
  const bool in_regs = chunks <= 32 * kGroupRegs;
  const bool vec = (n & 3) == 0 && (reinterpret_cast<uintptr_t>(xr) & 15u) == 0;
  float4 gm[kGroupRegs];
  // 1. lane best over its groups
  float lv = -INFINITY;
  int lg = INT_MAX;
#pragma unroll 1
  for (int c0 = lane; c0 < chunks; c0 += 32 * kGroupRegs) {
#pragma unroll
    for (int r = 0; r < kGroupRegs; ++r) {
      const int c = c0 + 32 * r;
      gm[r] = c < chunks ? g4[c] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int r = 0; r < kGroupRegs; ++r)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int g = 4 * (c0 + 32 * r) + u;
        if (c0 + 32 * r < chunks && ranks_ahead(f4_at(gm[r], u), g, lv, lg)) { lv = f4_at(gm[r], u); lg = g; }
      }
  }
  // 2. T = the topk-th best lane best
  float tv = lv;
  int ti = lg;
  warp_sort32(tv, ti);
  const float T = __shfl_sync(0xffffffffu, tv, topk - 1);
  // 3. this lane's groups whose maximum reaches T: their elements >= T go to the warp's list
  if (lane == 0) cnt[warp] = 0;
  __syncwarp();
  // the j-th (0-based) group of this lane reaching T, or -1
  auto qualifying = [&](int j) -> int {
    int seen = 0;
    if (in_regs) {
#pragma unroll
      for (int r = 0; r < kGroupRegs; ++r)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = lane + 32 * r;
          if (c < chunks && f4_at(gm[r], u) >= T && seen++ == j) return 4 * c + u;
        }
      return -1;
    }
    for (int c = lane; c < chunks; c += 32) {
      const float4 q = g4[c];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (f4_at(q, u) >= T && seen++ == j) return 4 * c + u;
    }
    return -1;
  };
#pragma unroll 1
  for (int j = 0;; ++j) {
    const int g = qualifying(j);
    if (g < 0) break;
    float v[32];
    load_group(xr, n, vec, g, v);
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (v[k] >= T) {
        const int slot = atomicAdd(&cnt[warp], 1);
        if (slot < kGroupCand) { cv[warp][slot] = v[k]; ci[warp][slot] = 32 * g + k; }
      }
  }
  __syncwarp();
  const int c = cnt[warp];
  float* wv = out_v + (size_t)row * topk;
  int* wi = out_i + (size_t)row * topk;
  if (c <= 32) {
    float v = lane < c ? cv[warp][lane] : -INFINITY;
    int id = lane < c ? ci[warp][lane] : INT_MAX;
    warp_sort32(v, id);
    if (lane < topk) { wv[lane] = v; wi[lane] = id; }
    return;
  }
  float pv = INFINITY;
  int pi = -1;
#pragma unroll 1
  for (int r = 0; r < topk; ++r) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    if (c <= kGroupCand) {
      for (int k = lane; k < c; k += 32)
        if (ranks_ahead(pv, pi, cv[warp][k], ci[warp][k]) && ranks_ahead(cv[warp][k], ci[warp][k], bv, bi)) {
          bv = cv[warp][k];
          bi = ci[warp][k];
        }
    } else {
      // many values reach T (ties): rank the qualifying groups' elements directly
#pragma unroll 1
      for (int j = 0;; ++j) {
        const int g = qualifying(j);
        if (g < 0) break;
        float v[32];
        load_group(xr, n, vec, g, v);
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (ranks_ahead(pv, pi, v[k], 32 * g + k) && ranks_ahead(v[k], 32 * g + k, bv, bi)) {
            bv = v[k];
            bi = 32 * g + k;
          }
      }
    }
    warp_best(bv, bi);
    if (lane == 0) { wv[r] = bv; wi[r] = bi; }
    pv = bv;
    pi = bi;
  }
}

// Ranks `rows` rows of n pairs.  More than one chunk per row goes through the
// candidate buffers (rows x chunks x topk) and one more pass, which the
// callers size so that it fits a single chunk.
static medusa_status launch_topk(const float* x, const int* x_idx, int rows, int n, int topk, float* cand_val,
                                 int* cand_idx, float* out_val, int* out_idx, cudaStream_t s) {
  if (!x_idx && topk <= kRowTopkMax) {
    launch_pdl(topk_rows_kernel, dim3(rows), dim3(kRowThreads), 0, s, x, n, topk, out_val, out_idx);
    return launch_status();
  }
  const int chunks = chunks_for(n);
  if (chunks == 1) {
    launch_pdl(topk_block_kernel, dim3(1, rows), dim3(kTopkThreads), 0, s, x, x_idx, n, 1, topk, out_val, out_idx);
  } else {
    launch_pdl(topk_block_kernel, dim3(chunks, rows), dim3(kTopkThreads), 0, s, x, x_idx, n, chunks, topk, cand_val, cand_idx);
    launch_pdl(topk_block_kernel, dim3(1, rows), dim3(kTopkThreads), 0, s, cand_val, cand_idx, chunks * topk, 1, topk, out_val,
                                                              out_idx);
  }
  return launch_status();
}

static size_t topk_ws_bytes(int rows, int V, int topk) {
  WsCarver w(nullptr);
  w.take<float>((size_t)rows * chunks_for(V) * topk);
  w.take<int>((size_t)rows * chunks_for(V) * topk);
  return w.used;
}

// ------------------------------------------------------------------- GEMV launch

// CTAs per head of the W2 pass never exceed this (bounds the candidate lists:
// max_ctas_per_head * topk / kTopkChunk <= 32 chunks, whose 32 * topk survivors
// fit one merge chunk).
inline int max_ctas_per_head(int V) {
  int c = ceil_div(V, kRowsPerWarp);
  return c < 4096 ? c : 4096;
}

// The merge fits the W2 CTA's shared memory (staged x region) when every
// batch row's ctas * topk (value, index) pairs plus one head position per list
// fit in C floats.
inline bool merge_fits(int ctas, int topk, int C) { return (size_t)ctas * topk * 2 + ctas <= (size_t)C; }

template <typename TW, bool kFirst>
static int launch_gemv_bb(int BB, const TW* W, const TW* h, const float* u, int B, int b0, int K,
                          int rows_per_head, int C, float* out, int topk, float* cand_v, int* cand_i,
                          int* counters, int n_counters, float* top_v, int* top_i, cudaStream_t s) {
  int launched = 0;
  auto go = [&](auto kern) {
    const size_t xs_bytes = (size_t)BB * C * sizeof(float);
    const size_t est = xs_bytes + (kFirst ? 0 : 2048);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)est);
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGemvThreads, est);
    if (per_sm < 1) per_sm = 1;
    int per_head = per_sm * device_sm_count() / K;
    if (per_head < 1) per_head = 1;
    const int max_useful = kFirst ? ceil_div(rows_per_head, kRowsPerWarp) : max_ctas_per_head(rows_per_head);
    if (per_head > max_useful) per_head = max_useful;
    const int cap = ceil_div(rows_per_head, per_head);
    const size_t smem = xs_bytes + (kFirst ? 0 : (size_t)BB * cap * sizeof(float));
    if (smem > est) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const bool fuse = !kFirst && top_v && merge_fits(per_head, topk, C);
    launch_pdl(kern, dim3(per_head, K), dim3(kGemvThreads), smem, s, W, h, u, B, b0, K, rows_per_head, C, out, topk, cand_v,
                                                       cand_i, counters, n_counters, fuse ? top_v : nullptr,
                                                       fuse ? top_i : nullptr);
    launched = per_head;
  };
  switch (BB) {
    case 1: go(heads_gemv_kernel<TW, 1, kFirst>); break;
    case 2: go(heads_gemv_kernel<TW, 2, kFirst>); break;
    case 4: go(heads_gemv_kernel<TW, 4, kFirst>); break;
    default: go(heads_gemv_kernel<TW, 8, kFirst>); break;
  }
  return launched;
}

// Returns the CTAs per head of the W2 pass (candidates per (row, head) / topk).
template <typename TW>
static int launch_heads_gemv(const TW* h, const TW* w1, const TW* w2, int B, int H, int V, int K, int topk,
                             float* u, float* z_or_null, float* cand_v, int* cand_i, int* counters,
                             float* top_v, int* top_i, cudaStream_t s) {
  const int n_counters = ceil_div(B, kMaxBatchPerPass) * K;
  for (int b0 = 0; b0 < B; b0 += kMaxBatchPerPass) {
    int nb = B - b0 < kMaxBatchPerPass ? B - b0 : kMaxBatchPerPass;
    int BB = nb <= 1 ? 1 : nb <= 2 ? 2 : nb <= 4 ? 4 : 8;
    launch_gemv_bb<TW, true>(BB, w1, h, nullptr, B, b0, K, H, H, u, 0, nullptr, nullptr, counters, n_counters,
                             nullptr, nullptr, s);
  }
  int cph = 0;
  for (int b0 = 0; b0 < B; b0 += kMaxBatchPerPass) {
    int nb = B - b0 < kMaxBatchPerPass ? B - b0 : kMaxBatchPerPass;
    int BB = nb <= 1 ? 1 : nb <= 2 ? 2 : nb <= 4 ? 4 : 8;
    int c = launch_gemv_bb<TW, false>(BB, w2, nullptr, u, B, b0, K, V, H, z_or_null, topk, cand_v, cand_i,
                                      counters, n_counters, top_v, top_i, s);
    if (b0 == 0) cph = c;
    else if (c != cph) return -1;  // the candidate layout must match across passes
  }
  return cph;
}

static size_t heads_cand(int B, int V, int K, int topk) { return (size_t)B * K * max_ctas_per_head(V) * topk; }
static size_t heads_cand2(int B, int V, int K, int topk) {
  return (size_t)B * K * chunks_for((long long)max_ctas_per_head(V) * topk) * topk;
}

// tensor-core path (heads_tc.cu)
int heads_tc_bp(int B);
bool heads_tc_supported(int B, int H, const void* h, const void* w1, const void* w2);
medusa_status heads_tc_run(const uint16_t* h, const uint16_t* w1, const uint16_t* w2, int B, int H, int V, int K,
                           uint16_t* u2, float* z, float* gmax, int32_t* d_status, cudaStream_t s);
inline int heads_tc_groups(int V) { return 4 * ceil_div(V, 128); }

// Scratch of the tensor-core path: u split into hi/lo bf16 rows, z, the
// maxima of z's 32-row groups.
static size_t heads_tc_ws_bytes(int B, int H, int V, int K) {
  WsCarver w(nullptr);
  w.take<uint16_t>((size_t)K * 2 * heads_tc_bp(B) * H);
  w.take<float>((size_t)B * K * V);
  w.take<float>((size_t)B * K * heads_tc_groups(V));
  return w.used;
}

static size_t heads_ws_bytes(int B, int H, int V, int K, int topk) {
  if (B >= 4 && B <= 64 && H % 64 == 0) {
    // either path may run (the tensor-core one for bf16): size for both
    const size_t a = heads_tc_ws_bytes(B, H, V, K);
    WsCarver w(nullptr);
    w.take<float>((size_t)B * K * H);
    w.take<float>(heads_cand(B, V, K, topk));
    w.take<int>(heads_cand(B, V, K, topk));
    w.take<float>(heads_cand2(B, V, K, topk));
    w.take<int>(heads_cand2(B, V, K, topk));
    w.take<int>((size_t)ceil_div(B, kMaxBatchPerPass) * K);
    return a > w.used ? a : w.used;
  }
  WsCarver w(nullptr);
  w.take<float>((size_t)B * K * H);
  w.take<float>(heads_cand(B, V, K, topk));
  w.take<int>(heads_cand(B, V, K, topk));
  w.take<float>(heads_cand2(B, V, K, topk));
  w.take<int>(heads_cand2(B, V, K, topk));
  w.take<int>((size_t)ceil_div(B, kMaxBatchPerPass) * K);
  return w.used;
}

}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_heads_workspace_size(int B, int H, int V, int K, int topk) {
  if (B <= 0 || H <= 0 || V <= 0 || K <= 0 || topk <= 0) return 0;
  return heads_ws_bytes(B, H, V, K, topk);
}

extern "C" medusa_status medusa_heads(const void* h, const void* w1, const void* w2, int B, int H,
                                      int V, int K, int topk, medusa_dtype dt, int32_t* topk_idx,
                                      float* topk_logit, float* logits_or_null, void* ws,
                                      size_t ws_bytes, int32_t* d_status, medusa_stream_t stream) {
  if (!h || !w1 || !w2 || !topk_idx || !topk_logit) return MEDUSA_ERR_INVALID_ARG;
  if (B < 1 || B > 64 || H < 8 || H % 8 || V < 1 || K < 1 || K > MEDUSA_MAX_DEPTH) return MEDUSA_ERR_INVALID_ARG;
  if (topk < 1 || topk > MEDUSA_MAX_TOPK || topk > V || !dtype_ok(dt)) return MEDUSA_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w1) || !aligned16(w2)) return MEDUSA_ERR_INVALID_ARG;
  if (logits_or_null && !aligned16(logits_or_null)) return MEDUSA_ERR_INVALID_ARG;
  const int bb_max = B > 4 ? 8 : B > 2 ? 4 : B > 1 ? 2 : 1;
  if ((size_t)bb_max * H * sizeof(float) > 200 * 1024) return MEDUSA_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < heads_ws_bytes(B, H, V, K, topk)) return MEDUSA_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == MEDUSA_BF16 && heads_tc_supported(B, H, h, w1, w2)) {
    // Batches of 4 and more: both passes on tensor cores, then the top-k of z.
    WsCarver wt(ws);
    uint16_t* u2 = wt.take<uint16_t>((size_t)K * 2 * heads_tc_bp(B) * H);
    float* zt = wt.take<float>((size_t)B * K * V);
    float* gm = wt.take<float>((size_t)B * K * heads_tc_groups(V));
    float* z = logits_or_null ? logits_or_null : zt;
    medusa_status st = heads_tc_run((const uint16_t*)h, (const uint16_t*)w1, (const uint16_t*)w2, B, H, V, K, u2, z,
                                    gm, d_status, s);
    if (st != MEDUSA_OK) return st;
    // one ranking kernel, reading only the groups that can hold a top-k logit
    launch_pdl(topk_groups_kernel, dim3(ceil_div(B * K, kGroupWarps)), dim3(32 * kGroupWarps), 0, s, (const float*)z,
               (const float*)gm, V, heads_tc_groups(V), topk, B * K, topk_logit, topk_idx);
    return launch_status();
  }
  WsCarver wc(ws);
  float* u = wc.take<float>((size_t)B * K * H);
  float* cv = wc.take<float>(heads_cand(B, V, K, topk));
  int* ci = wc.take<int>(heads_cand(B, V, K, topk));
  float* cv2 = wc.take<float>(heads_cand2(B, V, K, topk));
  int* ci2 = wc.take<int>(heads_cand2(B, V, K, topk));
  int* counters = wc.take<int>((size_t)ceil_div(B, kMaxBatchPerPass) * K);
  int cph;
  if (dt == MEDUSA_BF16)
    cph = launch_heads_gemv<uint16_t>((const uint16_t*)h, (const uint16_t*)w1, (const uint16_t*)w2, B, H, V, K,
                                      topk, u, logits_or_null, cv, ci, counters, topk_logit, topk_idx, s);
  else
    cph = launch_heads_gemv<float>((const float*)h, (const float*)w1, (const float*)w2, B, H, V, K, topk, u,
                                   logits_or_null, cv, ci, counters, topk_logit, topk_idx, s);
  if (cph <= 0) return MEDUSA_ERR_CUDA;
  medusa_status st = launch_status();
  if (st != MEDUSA_OK) return st;
  if (merge_fits(cph, topk, H)) return MEDUSA_OK;  // the W2 pass merged the candidates itself
  // Otherwise merge the per-CTA candidate lists of every (row, head) here.
  return launch_topk(cv, ci, B * K, cph * topk, topk, cv2, ci2, topk_logit, topk_idx, s);
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
  if ((long long)chunks_for(V) * topk > kTopkChunk) return MEDUSA_ERR_UNSUPPORTED;  // V > 2^17 * 32 / topk
  if (chunks_for(V) > 1 && (!ws || ws_bytes < topk_ws_bytes(rows, V, topk))) return MEDUSA_ERR_WORKSPACE;
  WsCarver wc(ws);
  float* cv = wc.take<float>((size_t)rows * chunks_for(V) * topk);
  int* ci = wc.take<int>((size_t)rows * chunks_for(V) * topk);
  return launch_topk(logits, nullptr, rows, V, topk, cv, ci, topk_logit, topk_idx,
                     reinterpret_cast<cudaStream_t>(stream));
}
