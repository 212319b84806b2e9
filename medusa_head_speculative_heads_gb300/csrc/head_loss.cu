// medusa_head_loss: the Medusa-1 loss of the K heads and its gradient with
// respect to the head logits.
//
// Paper review ("Medusa: Simple LLM Inference Acceleration Framework with
// Multiple Decoding Heads"), "方法细节": Medusa-1 freezes the backbone and
// trains the heads on L1 = -sum_k lambda_k log p_t^(k)(y_{t+k+1}),
// lambda_k = 0.8^k.  Per head the loss is the mean, over the counted positions
// (padding targets, marked negative, are skipped), of lse(z) - z[target]; its
// gradient is lambda_k / n_k * (softmax(z) - onehot(target)).
//
// Three launches:
//  1. head_loss_count_kernel: n_k (one CTA per head) and the target range check.
//  2. head_loss_row_kernel: one CTA per (head, sequence, position) row.  Pass 1
//     streams the row from HBM (16-byte loads, several per thread in flight)
//     and keeps a per-thread running max and sum of exponentials, rescaled
//     once per group of loaded values; the CTA merges them into lse.  Pass 2
//     reads the row again (from L2, where pass 1 left it; a streaming hint,
//     since the line is dead afterwards) and writes the gradient with streaming
//     stores.  Reading each element before writing it in the same thread makes
//     the in-place form (gradient over the logits) safe.
//  3. head_loss_finalize_kernel: one CTA adds the per-row terms of each head in
//     a fixed order and forms the means and L1 (deterministic).
#include <math.h>

#include "common.cuh"
#include "host_util.h"

namespace medusa {

namespace hl {

// CTA shape of the row kernel.  Rows between their two passes stay in L2 for
// the second read: resident CTAs x row bytes ~ 152 x 3 x 128 KB (fp32,
// V = 32000) or 152 x 6 x 64 KB (bf16), about 58 MB of the 126 MB L2.  More
// CTAs per SM overlap more of one row's reduction with other rows' loads, but
// past this footprint the second reads start to miss (measured).
template <typename T>
struct RowShape;
template <>
struct RowShape<float> {
  static constexpr int threads = 512, blocks = 3;
};
template <>
struct RowShape<uint16_t> {
  static constexpr int threads = 256, blocks = 6;
};
constexpr int kU = 4;  // 16-byte loads in flight per thread
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
  const void* logits;
  void* dlogits;
  const int32_t* tokens;
  float* rows;      // [K][B][S] per-row terms
  int32_t* counts;  // [K]: n_k
  float* scale;     // [K]: c_k = lambda_k / n_k and log2(c_k), written by the count kernel
  float* lscale;
  float* loss;      // [K + 1]
  int32_t* d_status;
  int K, B, S, V, vec;
  double lambda[MEDUSA_MAX_HEAD_LOSS_HEADS];
};

// 2^x with the hardware approximation (PTX ex2.approx.ftz.f32: relative error
// about 2^-22; results below the normal range flush to zero).
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// (m, s) summarises exponentials as s * e^m; merging keeps the larger m.
__device__ __forceinline__ void merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;  // both empty
  s = s * ex2((m - M) * kLog2e) + s2 * ex2((m2 - M) * kLog2e);
  m = M;
}

template <typename T>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int n = 4;
  static constexpr uint32_t neg_inf = 0xff800000u;
  static __device__ __forceinline__ void unpack(const uint4& r, float* f) { unpack_f32x4(r, f); }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
  template <int U>
  static __device__ __forceinline__ float max_of(const uint4* r) {
    float m = __uint_as_float(r[0].x);
#pragma unroll
    for (int u = 0; u < U; ++u)
      m = fmaxf(fmaxf(m, fmaxf(__uint_as_float(r[u].x), __uint_as_float(r[u].y))),
                fmaxf(__uint_as_float(r[u].z), __uint_as_float(r[u].w)));
    return m;
  }
};
template <>
struct Vec<uint16_t> {
  static constexpr int n = 8;
  static constexpr uint32_t neg_inf = 0xff80ff80u;
  static __device__ __forceinline__ void unpack(const uint4& r, float* f) { unpack_bf16x8(r, f); }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    return make_uint4(bf16x2_rn(f[0], f[1]), bf16x2_rn(f[2], f[3]), bf16x2_rn(f[4], f[5]), bf16x2_rn(f[6], f[7]));
  }
  // Maximum of U x 8 bf16 values on packed pairs (exact: max selects one input).
  static __device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  }
  template <int U>
  static __device__ __forceinline__ float max_of(const uint4* r) {
    uint32_t m = max2(max2(r[0].x, r[0].y), max2(r[0].z, r[0].w));
#pragma unroll
    for (int u = 1; u < U; ++u) m = max2(m, max2(max2(r[u].x, r[u].y), max2(r[u].z, r[u].w)));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
  }
};

}  // namespace hl

__global__ void __launch_bounds__(256) head_loss_count_kernel(const hl::Params p) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_n[8];
  const int k = blockIdx.x + 1;
  const int per = p.S - k - 1;  // positions t = 0 .. per - 1 have a target
  int n = 0;
  bool bad = false;
  if (per > 0)
    for (long long i = threadIdx.x; i < (long long)p.B * per; i += blockDim.x) {
      const int b = (int)(i / per), t = (int)(i - (long long)b * per);
      const int y = p.tokens[(size_t)b * p.S + t + k + 1];
      if (y >= p.V) bad = true;
      else if (y >= 0) ++n;
    }
#pragma unroll
  for (int o = 16; o; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if ((threadIdx.x & 31) == 0) s_n[threadIdx.x >> 5] = n;
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    int tot = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_n[w];
    p.counts[k - 1] = tot;
    const double c = tot > 0 ? p.lambda[k - 1] / tot : 0.0;
    p.scale[k - 1] = (float)c;
    p.lscale[k - 1] = tot > 0 ? (float)log2(c) : 0.f;
    if (bad) set_status(p.d_status, MEDUSA_DEV_BAD_INDEX);
  }
}

template <typename T>
__global__ void __launch_bounds__(hl::RowShape<T>::threads, hl::RowShape<T>::blocks)
    head_loss_row_kernel(const hl::Params p) {
  using namespace hl;
  using Vt = Vec<T>;
  constexpr int E = Vt::n;
  constexpr int kThreads = RowShape<T>::threads;
  pdl_wait();
  pdl_trigger();
  __shared__ float s_m[kThreads / 32], s_s[kThreads / 32];
  __shared__ float s_lse;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int BS = p.B * p.S;
  const int r = blockIdx.x;
  const int k = r / BS + 1;
  const int rem = r - (k - 1) * BS;
  const int b = rem / p.S, t = rem - b * p.S;
  int y = t + k + 1 < p.S ? p.tokens[(size_t)b * p.S + t + k + 1] : -1;
  if (y >= p.V) y = -1;
  const int n = p.counts[k - 1];
  const T* z = static_cast<const T*>(p.logits) + (size_t)r * p.V;
  T* g = p.dlogits ? static_cast<T*>(p.dlogits) + (size_t)r * p.V : nullptr;

  if (y < 0 || n <= 0) {  // not counted: zero gradient row, zero term
    if (tid == 0) p.rows[r] = 0.f;
    if (g) {
      if (p.vec) {
        uint4* g4 = reinterpret_cast<uint4*>(g);
        for (int i = tid; i < p.V / E; i += kThreads) __stcs(g4 + i, make_uint4(0, 0, 0, 0));
      } else {
        for (int i = tid; i < p.V; i += kThreads) store_elem(g, i, 0.f);
      }
    }
    return;
  }

  // ---- pass 1: running max and sum of exp per thread
  float m = -INFINITY, s = 0.f;
  const int nv = p.vec ? p.V / E : 0;
  if (p.vec) {
    const uint4* z4 = reinterpret_cast<const uint4*>(z);
    for (int i0 = tid; i0 < nv; i0 += kThreads * kU) {
      uint4 raw[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * kThreads;
        raw[u] = i < nv ? z4[i] : make_uint4(Vt::neg_inf, Vt::neg_inf, Vt::neg_inf, Vt::neg_inf);
      }
      const float cm = Vt::template max_of<kU>(raw);
      if (cm > m) {
        s *= ex2((m - cm) * kLog2e);
        m = cm;
      }
      if (m > -INFINITY) {
        const float nm = -m * kLog2e;  // e^(v - m) = 2^(v log2 e - m log2 e), one FMA
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          float v[E];
          Vt::unpack(raw[u], v);
#pragma unroll
          for (int j = 0; j < E; ++j) s += ex2(fmaf(v[j], kLog2e, nm));
        }
      }
    }
  } else {
    for (int i = tid; i < p.V; i += kThreads) {
      const float x = load_elem(z, i);
      if (x > m) {
        s = s * ex2((m - x) * kLog2e) + 1.f;
        m = x;
      } else if (m > -INFINITY) {
        s += ex2((x - m) * kLog2e);
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    merge(m, s, m2, s2);
  }
  if (lane == 0) {
    s_m[warp] = m;
    s_s[warp] = s;
  }
  __syncthreads();
  if (tid == 0) {
    float M = s_m[0], sum = s_s[0];
    for (int w = 1; w < kThreads / 32; ++w) merge(M, sum, s_m[w], s_s[w]);
    const float lse = M + logf(sum);
    s_lse = lse;
    p.rows[r] = lse - load_elem(z, (size_t)y);
  }
  __syncthreads();
  if (!g) return;

  // ---- pass 2: gradient c * (softmax - onehot)
  const float lse = s_lse;
  const float c = p.scale[k - 1];
  // c * e^(z - lse) = 2^(z log2 e + (log2 c - lse log2 e)): one FMA and one ex2
  const float off = p.lscale[k - 1] - lse * kLog2e;
  if (p.vec) {
    const uint4* z4 = reinterpret_cast<const uint4*>(z);
    uint4* g4 = reinterpret_cast<uint4*>(g);
    for (int i0 = tid; i0 < nv; i0 += kThreads * kU) {
      uint4 raw[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * kThreads;
        if (i < nv) raw[u] = __ldcs(z4 + i);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * kThreads;
        if (i < nv) {
          float v[E], o[E];
          Vt::unpack(raw[u], v);
#pragma unroll
          for (int j = 0; j < E; ++j) o[j] = ex2(fmaf(v[j], kLog2e, off));
          if (i == y / E) {  // the target's vector: subtract c from its element
#pragma unroll
            for (int j = 0; j < E; ++j)
              if (j == y - i * E) o[j] -= c;
          }
          __stcs(g4 + i, Vt::pack(o));
        }
      }
    }
  } else {
    for (int i = tid; i < p.V; i += kThreads) {
      const float x = load_elem(z, i);
      store_elem(g, i, ex2(fmaf(x, kLog2e, off)) - (i == y ? c : 0.f));
    }
  }
}

// One CTA: per head, the sum of the row terms in a fixed order (each thread a
// fixed strided subset, then a fixed shuffle tree and the warps in order), the
// mean and L1.  fp32 throughout: the pairwise tree keeps the relative error
// near (rows per thread + 15) ulps, and double arithmetic runs at a small
// fraction of the fp32 rate on this GPU.
__global__ void __launch_bounds__(1024) head_loss_finalize_kernel(const hl::Params p) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_part[32];
  const int BS = p.B * p.S;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float total = 0.f;
  for (int k = 1; k <= p.K; ++k) {
    const float* rows = p.rows + (size_t)(k - 1) * BS;
    float a = 0.f;
#pragma unroll 8
    for (int i = threadIdx.x; i < BS; i += blockDim.x) a += rows[i];
#pragma unroll
    for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) s_part[warp] = a;
    __syncthreads();
    if (warp == 0) {
      float w = lane < nw ? s_part[lane] : 0.f;
#pragma unroll
      for (int o = 16; o; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
      if (lane == 0) {
        const int n = p.counts[k - 1];
        const float mean = n > 0 ? w / (float)n : 0.f;
        p.loss[k - 1] = mean;
        total += (float)p.lambda[k - 1] * mean;
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) p.loss[p.K] = total;
}

}  // namespace medusa

using namespace medusa;

// counts, scale, log2(scale): K 4-byte words each
static size_t head_loss_counts_bytes(int K) { return align_up((size_t)3 * K * 4, 16); }

extern "C" size_t medusa_head_loss_workspace_size(int K, int B, int S) {
  if (K < 1 || B < 1 || S < 1 || K > MEDUSA_MAX_HEAD_LOSS_HEADS) return 0;
  return head_loss_counts_bytes(K) + (size_t)K * B * S * sizeof(float);
}

extern "C" medusa_status medusa_head_loss(const void* logits, const int32_t* tokens, int K, int B, int S, int V,
                                          float decay, medusa_dtype dt, void* dlogits, float* loss,
                                          float* row_loss, void* ws, size_t ws_bytes, int32_t* d_status,
                                          medusa_stream_t stream) {
  if (!logits || !tokens || !loss) return MEDUSA_ERR_INVALID_ARG;
  if (K < 1 || K > MEDUSA_MAX_HEAD_LOSS_HEADS || B < 1 || S < 1 || V < 1) return MEDUSA_ERR_INVALID_ARG;
  if ((long long)K * B * S >= (1ll << 31) || !isfinite(decay)) return MEDUSA_ERR_INVALID_ARG;
  if (!dtype_ok(dt)) return MEDUSA_ERR_UNSUPPORTED;
  const size_t es = dtype_bytes(dt);
  if (reinterpret_cast<uintptr_t>(logits) % es || (dlogits && reinterpret_cast<uintptr_t>(dlogits) % es) ||
      reinterpret_cast<uintptr_t>(tokens) % 4 || reinterpret_cast<uintptr_t>(loss) % 4 ||
      (row_loss && reinterpret_cast<uintptr_t>(row_loss) % 4))
    return MEDUSA_ERR_INVALID_ARG;
  const size_t rows = (size_t)K * B * S;
  const size_t zb = rows * V * es, tb = (size_t)B * S * 4, lb = (size_t)(K + 1) * 4, rb = rows * 4;
  if (dlogits && dlogits != logits && overlaps(dlogits, zb, logits, zb)) return MEDUSA_ERR_ALIAS;
  if (dlogits && (overlaps(dlogits, zb, tokens, tb) || overlaps(dlogits, zb, loss, lb))) return MEDUSA_ERR_ALIAS;
  if (overlaps(loss, lb, logits, zb) || overlaps(loss, lb, tokens, tb)) return MEDUSA_ERR_ALIAS;
  if (row_loss && (overlaps(row_loss, rb, logits, zb) || overlaps(row_loss, rb, tokens, tb) ||
                   overlaps(row_loss, rb, loss, lb) || (dlogits && overlaps(row_loss, rb, dlogits, zb))))
    return MEDUSA_ERR_ALIAS;
  const size_t need = medusa_head_loss_workspace_size(K, B, S);
  if (!ws || ws_bytes < need || !aligned16(ws)) return MEDUSA_ERR_WORKSPACE;
  if (overlaps(ws, need, logits, zb) || overlaps(ws, need, tokens, tb) || overlaps(ws, need, loss, lb) ||
      (dlogits && overlaps(ws, need, dlogits, zb)) || (row_loss && overlaps(ws, need, row_loss, rb)))
    return MEDUSA_ERR_ALIAS;

  hl::Params p{};
  p.logits = logits;
  p.dlogits = dlogits;
  p.tokens = tokens;
  p.counts = static_cast<int32_t*>(ws);
  p.scale = reinterpret_cast<float*>(p.counts + K);
  p.lscale = p.scale + K;
  p.rows = row_loss ? row_loss
                    : reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + head_loss_counts_bytes(K));
  p.loss = loss;
  p.d_status = d_status;
  p.K = K;
  p.B = B;
  p.S = S;
  p.V = V;
  const size_t vec_elems = 16 / es;
  p.vec = (V % vec_elems == 0) && aligned16(logits) && (!dlogits || aligned16(dlogits));
  for (int k = 1; k <= K; ++k) p.lambda[k - 1] = pow((double)decay, (double)k);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  launch_pdl(head_loss_count_kernel, dim3(K), dim3(256), 0, s, p);
  if (dt == MEDUSA_BF16)
    launch_pdl(head_loss_row_kernel<uint16_t>, dim3((unsigned)rows), dim3(hl::RowShape<uint16_t>::threads), 0, s,
               p);
  else
    launch_pdl(head_loss_row_kernel<float>, dim3((unsigned)rows), dim3(hl::RowShape<float>::threads), 0, s, p);
  launch_pdl(head_loss_finalize_kernel, dim3(1), dim3(1024), 0, s, p);
  return launch_status();
}
