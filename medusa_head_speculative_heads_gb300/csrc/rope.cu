// medusa_tree_rope: rotary position embedding of the verify pass's tree tokens
// at their tree positions, in place on q and on the tree K buffer.
//
// Paper review ("Medusa: Simple LLM Inference Acceleration Framework with
// Multiple Decoding Heads"), FAQ "树注意力为什么能一次验证多条候选": the position
// encoding follows the tree, so node n of row b is encoded at
// pos[b][n] = prefix_len[b] + depth(n) (the positions medusa_tree_build
// writes).  The pages give no formula; the rotation is the rotate-half rotary
// embedding of the LLaMA family: for i < d/2 the pair (x[i], x[i + d/2]) turns
// by pos * base^(-2i/d).
//
// One CTA per (layer, row, node) token.  The CTA forms its d/2 angles once:
// pos * theta_i in double (theta_i computed on the host in double), reduced
// modulo 2 pi in double (multiply by 1 / (2 pi), round, fused multiply-add),
// then cos/sin in single precision of the reduced angle; every q and k head of
// the token is then rotated from 16-byte chunks (8 bf16 or 4 fp32 pairs per
// chunk and thread, a fixed chunk per thread, two heads' loads in flight; the
// first of them are issued before the angles are formed).
// HBM-bound: each element is read and written once.
#include <cmath>

#include "common.cuh"
#include "host_util.h"

namespace medusa {

constexpr int kRopeThreads = 256;
constexpr int kRopeMaxHalf = 128;  // d <= 256

struct RopeParams {
  double theta[kRopeMaxHalf];  // base^(-2i/d)
  int nl, B, N, Hq, Hkv, d;
};

template <typename T>
struct RopeVec;  // 16 bytes of T
template <>
struct RopeVec<float> {
  static constexpr int n = 4;
};
template <>
struct RopeVec<uint16_t> {
  static constexpr int n = 8;
};

__device__ __forceinline__ float rope_ld(const float* p) { return *p; }
__device__ __forceinline__ float rope_ld(const uint16_t* p) { return bf16_bits_to_f32(*p); }
__device__ __forceinline__ void rope_st(float* p, float v) { *p = v; }
__device__ __forceinline__ void rope_st(uint16_t* p, float v) { *p = (uint16_t)f32_to_bf16_bits(v); }

__device__ __forceinline__ void unpack16(const uint4& w, float* f, float) {
  f[0] = __uint_as_float(w.x);
  f[1] = __uint_as_float(w.y);
  f[2] = __uint_as_float(w.z);
  f[3] = __uint_as_float(w.w);
}
__device__ __forceinline__ void unpack16(const uint4& w, float* f, uint16_t) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint4 pack16(const float* f, float) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}
__device__ __forceinline__ uint4 pack16(const float* f, uint16_t) {
  uint32_t u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) u[i] = f32_to_bf16_bits(f[2 * i]) | (f32_to_bf16_bits(f[2 * i + 1]) << 16);
  return make_uint4(u[0], u[1], u[2], u[3]);
}

// Angles of this CTA's token: cs[i] = (cos, sin)(pos * theta_i), the product
// formed and reduced modulo 2 pi in double.
__device__ __forceinline__ void rope_angles(float2* cs, double ps, const RopeParams& p) {
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  constexpr double kInvTwoPi = 0.15915494309189533576888376337251;
  for (int i = threadIdx.x; i < p.d / 2; i += blockDim.x) {
    const double a = ps * p.theta[i];
    const double r = fma(-rint(a * kInvTwoPi), kTwoPi, a);  // |r| <= pi (+ rounding)
    float sn, cn;
    sincosf((float)r, &sn, &cn);
    cs[i] = make_float2(cn, sn);
  }
}

// 16-byte path: thread t owns chunk t % chunks (W pairs) of heads t / chunks,
// t / chunks + rows, ...; blockDim.x = chunks * rows.  All loads are issued
// before any rotation.
template <typename T>
__global__ void __launch_bounds__(kRopeThreads)
tree_rope_vec_kernel(T* __restrict__ q, T* __restrict__ k, const int32_t* __restrict__ pos,
                     const __grid_constant__ RopeParams p) {
  constexpr int W = RopeVec<T>::n;
  constexpr int U = 2;  // heads per thread and round (loads in flight)
  __shared__ float2 cs[kRopeMaxHalf];
  pdl_wait();
  pdl_trigger();
  const int bn = blockIdx.x, l = blockIdx.y;
  const int half = p.d / 2, chunks = half / W, rows = blockDim.x / chunks;
  const int c = threadIdx.x % chunks, h0 = threadIdx.x / chunks;
  const size_t tok = (size_t)l * p.B * p.N + bn;
  T* qt = q + tok * p.Hq * p.d;
  T* kt = k ? k + tok * p.Hkv * p.d : nullptr;
  const int heads = p.Hq + (k ? p.Hkv : 0);
  uint4 lo[U], hi[U];
  T* x[U];
  auto load = [&](int hb) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int h = hb + u * rows;
      x[u] = h < heads ? (h < p.Hq ? qt + (size_t)h * p.d : kt + (size_t)(h - p.Hq) * p.d) + c * W : nullptr;
      if (x[u]) {
        lo[u] = *reinterpret_cast<const uint4*>(x[u]);
        hi[u] = *reinterpret_cast<const uint4*>(x[u] + half);
      }
    }
  };
  // The first heads' loads are in flight while the angles are formed.
  load(h0);
  rope_angles(cs, (double)pos[bn], p);
  __syncthreads();
  const float2* t = cs + c * W;
  for (int hb = h0; hb < heads; hb += rows * U) {
    if (hb != h0) load(hb);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!x[u]) continue;
      float a[W], b[W];
      unpack16(lo[u], a, T());
      unpack16(hi[u], b, T());
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const float x0 = a[j], x1 = b[j];
        a[j] = x0 * t[j].x - x1 * t[j].y;
        b[j] = x1 * t[j].x + x0 * t[j].y;
      }
      if constexpr (sizeof(T) == 2) {
        *reinterpret_cast<uint4*>(x[u]) =
            make_uint4(bf16x2_rn(a[0], a[1]), bf16x2_rn(a[2], a[3]), bf16x2_rn(a[4], a[5]), bf16x2_rn(a[6], a[7]));
        *reinterpret_cast<uint4*>(x[u] + half) =
            make_uint4(bf16x2_rn(b[0], b[1]), bf16x2_rn(b[2], b[3]), bf16x2_rn(b[4], b[5]), bf16x2_rn(b[6], b[7]));
      } else {
        *reinterpret_cast<uint4*>(x[u]) = pack16(a, T());
        *reinterpret_cast<uint4*>(x[u] + half) = pack16(b, T());
      }
    }
  }
}

// Element-wise path (other head sizes or alignments): one pair per thread and step.
template <typename T>
__global__ void __launch_bounds__(kRopeThreads)
tree_rope_scalar_kernel(T* __restrict__ q, T* __restrict__ k, const int32_t* __restrict__ pos,
                        const __grid_constant__ RopeParams p) {
  __shared__ float2 cs[kRopeMaxHalf];
  pdl_wait();
  pdl_trigger();
  const int bn = blockIdx.x, l = blockIdx.y;
  rope_angles(cs, (double)pos[bn], p);
  __syncthreads();
  const int half = p.d / 2;
  const size_t tok = (size_t)l * p.B * p.N + bn;
  const int heads = p.Hq + (k ? p.Hkv : 0);
  for (int task = threadIdx.x; task < heads * half; task += blockDim.x) {
    const int h = task / half, i = task - h * half;
    T* x = h < p.Hq ? q + (tok * p.Hq + h) * p.d : k + (tok * p.Hkv + (h - p.Hq)) * p.d;
    const float2 t = cs[i];
    const float x0 = rope_ld(x + i), x1 = rope_ld(x + i + half);
    rope_st(x + i, x0 * t.x - x1 * t.y);
    rope_st(x + i + half, x1 * t.x + x0 * t.y);
  }
}

}  // namespace medusa

using namespace medusa;

extern "C" medusa_status medusa_tree_rope(void* q, void* k, const int32_t* pos, int n_layers, int B, int N, int Hq,
                                          int Hkv, int d, float base, medusa_dtype dt, medusa_stream_t stream) {
  if (!q || !pos) return MEDUSA_ERR_INVALID_ARG;
  if (n_layers < 1 || B < 1 || N < 1 || N > MEDUSA_MAX_NODES || Hq < 1 || (k && Hkv < 1)) return MEDUSA_ERR_INVALID_ARG;
  if (d < 2 || d % 2 || d > 2 * kRopeMaxHalf || !(base > 0.f) || !dtype_ok(dt)) return MEDUSA_ERR_INVALID_ARG;
  const size_t es = dtype_bytes(dt);
  const size_t tokens = (size_t)n_layers * B * N;
  if (k && overlaps(q, tokens * Hq * d * es, k, tokens * Hkv * d * es)) return MEDUSA_ERR_ALIAS;
  if ((size_t)B * N > 0x7fffffffu || n_layers > 65535) return MEDUSA_ERR_UNSUPPORTED;
  RopeParams p{};
  for (int i = 0; i < d / 2; ++i) p.theta[i] = std::pow((double)base, -2.0 * i / d);
  p.nl = n_layers;
  p.B = B;
  p.N = N;
  p.Hq = Hq;
  p.Hkv = k ? Hkv : 0;
  p.d = d;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int vw = dt == MEDUSA_BF16 ? 8 : 4;  // pairs per 16-byte chunk
  const bool vec = (d / 2) % vw == 0 && aligned16(q) && (!k || aligned16(k));
  const dim3 grid((unsigned)(B * N), (unsigned)n_layers);
  // 16-byte path: a block of whole rows of (d/2)/W chunk-threads.
  const int chunks = vec ? (d / 2) / vw : 1;
  const dim3 vblock(vec ? (unsigned)(kRopeThreads / chunks * chunks) : 1u), sblock(kRopeThreads);
  if (dt == MEDUSA_BF16) {
    auto* qq = static_cast<uint16_t*>(q);
    auto* kk = static_cast<uint16_t*>(k);
    if (vec) launch_pdl(tree_rope_vec_kernel<uint16_t>, grid, vblock, 0, s, qq, kk, pos, p);
    else launch_pdl(tree_rope_scalar_kernel<uint16_t>, grid, sblock, 0, s, qq, kk, pos, p);
  } else {
    auto* qq = static_cast<float*>(q);
    auto* kk = static_cast<float*>(k);
    if (vec) launch_pdl(tree_rope_vec_kernel<float>, grid, vblock, 0, s, qq, kk, pos, p);
    else launch_pdl(tree_rope_scalar_kernel<float>, grid, sblock, 0, s, qq, kk, pos, p);
  }
  return launch_status();
}
