// medusa_tree_attention: every tree node attends to the prefix KV cache and to
// its own tree ancestors (itself included), all layers in one call.
//
// Paper review ("Medusa: Simple LLM Inference Acceleration Framework with
// Multiple Decoding Heads"), section "Medusa 的三个核心组件": the tree mask lets
// a token look back only at its own branch's predecessors, so one forward pass
// verifies every candidate; FAQ "树注意力为什么能一次验证多条候选": the common
// prefix is computed once and shared.  Skill-pack guide, "树形验证":
// verification runs against past_key_values.
//
// Dispatch: bf16 with head_dim 128 (and 128 % G == 0) runs the tcgen05
// tensor-core kernel (attention_tc.cu); everything else runs the CUDA-core
// kernel below, fp32 arithmetic throughout (fp32 inputs never touch TF32).
//
// CUDA-core kernel: grid (query tiles of 64 rows, kv head, layer x row).  The
// query rows of one kv head are (node, q head of the group) pairs.  Key tiles
// of 32 rows (prefix rows first, then tree rows) are staged in shared memory as
// fp32; each warp owns 8 query rows, each lane one key of the tile and d/32
// output columns; online softmax in the log2 domain.
#include "common.cuh"
#include "host_util.h"

namespace medusa {

// tcgen05 path (attention_tc.cu)
bool tree_attention_tc_supported(int N, int Hq, int Hkv, int d, int Lmax, const void* q,
                                 const void* kc, const void* vc, const void* kt, const void* vt,
                                 const void* out);
size_t tree_attention_tc_ws_bytes(int n_layers, int B, int N, int Hq, int Hkv, int d, int Lmax);
medusa_status tree_attention_tc(const void* q, const void* kc, const void* vc, const void* kt,
                                const void* vt, const uint32_t* mask, const int32_t* prefix_len,
                                int n_layers, int B, int N, int Hq, int Hkv, int d, int Lmax,
                                float scale, void* out, void* ws, size_t ws_bytes,
                                int32_t* d_status, cudaStream_t s);

constexpr int kSimtThreads = 256;
constexpr int kSimtRows = 64;    // query rows per CTA
constexpr int kSimtKeys = 32;    // keys per tile
constexpr int kRowsPerWarpA = 8;

template <typename T, int DQ>
__global__ void __launch_bounds__(kSimtThreads)
tree_attn_simt_kernel(const T* __restrict__ q, const T* __restrict__ kc, const T* __restrict__ vc,
                      const T* __restrict__ kt, const T* __restrict__ vt,
                      const uint32_t* __restrict__ mask, const int32_t* __restrict__ prefix_len,
                      int B, int N, int Hq, int Hkv, int Lmax, float scale_log2, T* __restrict__ out,
                      int32_t* d_status) {
  pdl_wait();
  pdl_trigger();
  constexpr int D = 32 * DQ;
  constexpr int KP = D + 4;  // padded key row (16-byte aligned, conflict-free 128-bit reads)
  extern __shared__ __align__(16) float smem[];
  float* Qs = smem;                       // [64][D]
  float* Ks = Qs + kSimtRows * D;         // [32][KP]
  float* Vs = Ks + kSimtKeys * KP;        // [32][D]

  const int tile = blockIdx.x, g = blockIdx.y, lb = blockIdx.z;
  const int b = lb % B;
  const int G = Hq / Hkv, M = N * G, W = (N + 31) / 32;
  const int L = prefix_len[b];
  if (L < 0 || L > Lmax) {
    if (threadIdx.x == 0) set_status(d_status, MEDUSA_DEV_BAD_LENGTH);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int idx = tid; idx < kSimtRows * D; idx += kSimtThreads) {
    const int r = idx / D, c = idx - r * D, m = tile * kSimtRows + r;
    float v = 0.f;
    if (m < M) {
      const int i = m / G, h = g * G + m % G;
      v = load_elem<T>(q, (((size_t)lb * N + i) * Hq + h) * D + c) * scale_log2;
    }
    Qs[idx] = v;
  }

  float o[kRowsPerWarpA][DQ], mrow[kRowsPerWarpA], lrow[kRowsPerWarpA];
  int node[kRowsPerWarpA];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarpA; ++rr) {
    mrow[rr] = -INFINITY;
    lrow[rr] = 0.f;
    const int m = tile * kSimtRows + warp * kRowsPerWarpA + rr;
    node[rr] = m < M ? m / G : -1;
#pragma unroll
    for (int qd = 0; qd < DQ; ++qd) o[rr][qd] = 0.f;
  }

  const int n_pre = (L + kSimtKeys - 1) / kSimtKeys;
  const int n_tree = (N + kSimtKeys - 1) / kSimtKeys;
  for (int t = 0; t < n_pre + n_tree; ++t) {
    const bool tree = t >= n_pre;
    const int base = tree ? (t - n_pre) * kSimtKeys : t * kSimtKeys;
    const int count = min(kSimtKeys, (tree ? N : L) - base);
    const T* ksrc = tree ? kt : kc;
    const T* vsrc = tree ? vt : vc;
    const size_t rows_per_lb = tree ? (size_t)N : (size_t)Lmax;
    __syncthreads();
    for (int idx = tid; idx < kSimtKeys * D; idx += kSimtThreads) {
      const int j = idx / D, c = idx - j * D;
      float kv = 0.f, vv = 0.f;
      if (j < count) {
        const size_t off = (((size_t)lb * rows_per_lb + base + j) * Hkv + g) * D + c;
        kv = load_elem<T>(ksrc, off);
        vv = load_elem<T>(vsrc, off);
      }
      Ks[j * KP + c] = kv;
      Vs[j * D + c] = vv;
    }
    __syncthreads();

    float s[kRowsPerWarpA];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarpA; ++rr) s[rr] = 0.f;
    const float* kr = Ks + lane * KP;
    for (int c = 0; c < D; c += 4) {
      const float4 kk = *reinterpret_cast<const float4*>(kr + c);
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarpA; ++rr) {
        const float4 qq = *reinterpret_cast<const float4*>(Qs + (warp * kRowsPerWarpA + rr) * D + c);
        s[rr] = fmaf(qq.x, kk.x, s[rr]);
        s[rr] = fmaf(qq.y, kk.y, s[rr]);
        s[rr] = fmaf(qq.z, kk.z, s[rr]);
        s[rr] = fmaf(qq.w, kk.w, s[rr]);
      }
    }
    float p[kRowsPerWarpA];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarpA; ++rr) {
      bool valid = lane < count && node[rr] >= 0;
      if (valid && tree) {
        const int j = base + lane;
        valid = (mask[(size_t)node[rr] * W + (j >> 5)] >> (j & 31)) & 1u;
      }
      const float sv = valid ? s[rr] : -INFINITY;
      const float mnew = fmaxf(mrow[rr], warp_max(sv));
      if (mnew == -INFINITY) {  // nothing visible yet in this row
        p[rr] = 0.f;
        continue;
      }
      const float alpha = exp2f(mrow[rr] - mnew);
      p[rr] = valid ? exp2f(sv - mnew) : 0.f;
      lrow[rr] = lrow[rr] * alpha + warp_sum(p[rr]);
      mrow[rr] = mnew;
#pragma unroll
      for (int qd = 0; qd < DQ; ++qd) o[rr][qd] *= alpha;
    }
    for (int j = 0; j < count; ++j) {
      float vj[DQ];
#pragma unroll
      for (int qd = 0; qd < DQ; ++qd) vj[qd] = Vs[j * D + lane + 32 * qd];
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarpA; ++rr) {
        const float pj = __shfl_sync(0xffffffffu, p[rr], j);
#pragma unroll
        for (int qd = 0; qd < DQ; ++qd) o[rr][qd] = fmaf(pj, vj[qd], o[rr][qd]);
      }
    }
  }

#pragma unroll
  for (int rr = 0; rr < kRowsPerWarpA; ++rr) {
    const int m = tile * kSimtRows + warp * kRowsPerWarpA + rr;
    if (m >= M) continue;
    const int i = m / G, h = g * G + m % G;
    const float inv = 1.f / lrow[rr];
#pragma unroll
    for (int qd = 0; qd < DQ; ++qd)
      store_elem<T>(out, (((size_t)lb * N + i) * Hq + h) * D + lane + 32 * qd, o[rr][qd] * inv);
  }
}

template <typename T>
static medusa_status launch_simt(const void* q, const void* kc, const void* vc, const void* kt,
                                 const void* vt, const uint32_t* mask, const int32_t* prefix_len,
                                 int nl, int B, int N, int Hq, int Hkv, int d, int Lmax, float scale,
                                 void* out, int32_t* d_status, cudaStream_t s) {
  const int DQ = d / 32;
  const int M = N * (Hq / Hkv);
  dim3 grid((M + kSimtRows - 1) / kSimtRows, Hkv, nl * B);
  const size_t smem = (size_t)(kSimtRows * d + kSimtKeys * (d + 4) + kSimtKeys * d) * sizeof(float);
  const float sl2 = scale * 1.4426950408889634f;
  auto go = [&](auto kern) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_pdl(kern, dim3(grid), dim3(kSimtThreads), smem, s, (const T*)q, (const T*)kc, (const T*)vc, (const T*)kt,
                                          (const T*)vt, mask, prefix_len, B, N, Hq, Hkv, Lmax, sl2,
                                          (T*)out, d_status);
  };
  switch (DQ) {
    case 1: go(tree_attn_simt_kernel<T, 1>); break;
    case 2: go(tree_attn_simt_kernel<T, 2>); break;
    case 3: go(tree_attn_simt_kernel<T, 3>); break;
    case 4: go(tree_attn_simt_kernel<T, 4>); break;
    case 5: go(tree_attn_simt_kernel<T, 5>); break;
    case 6: go(tree_attn_simt_kernel<T, 6>); break;
    case 7: go(tree_attn_simt_kernel<T, 7>); break;
    default: go(tree_attn_simt_kernel<T, 8>); break;
  }
  return launch_status();
}

static bool use_tc(int N, int Hq, int Hkv, int d, int Lmax, medusa_dtype dt, const void* q,
                   const void* kc, const void* vc, const void* kt, const void* vt, const void* out) {
  return dt == MEDUSA_BF16 && tree_attention_tc_supported(N, Hq, Hkv, d, Lmax, q, kc, vc, kt, vt, out);
}

}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_tree_attention_workspace_size(int n_layers, int B, int N, int Hq, int Hkv,
                                                       int d, int Lmax, medusa_dtype dt) {
  if (n_layers < 1 || B < 1 || N < 1 || Hq < 1 || Hkv < 1 || d < 1 || Lmax < 0) return 0;
  if (dt == MEDUSA_BF16 && d == 128 && Hq % Hkv == 0 && 128 % (Hq / Hkv) == 0)
    return tree_attention_tc_ws_bytes(n_layers, B, N, Hq, Hkv, d, Lmax);
  return 0;
}

extern "C" medusa_status medusa_tree_attention(const void* q, const void* kc, const void* vc,
                                               const void* kt, const void* vt, const uint32_t* mask,
                                               const int32_t* prefix_len, int n_layers, int B, int N,
                                               int Hq, int Hkv, int d, int Lmax, float scale,
                                               medusa_dtype dt, void* out, void* ws, size_t ws_bytes,
                                               int32_t* d_status, medusa_stream_t stream) {
  if (!q || !kc || !vc || !kt || !vt || !mask || !prefix_len || !out) return MEDUSA_ERR_INVALID_ARG;
  if (n_layers < 1 || B < 1 || N < 1 || N > MEDUSA_MAX_NODES || Hq < 1 || Hkv < 1 || Hq % Hkv)
    return MEDUSA_ERR_INVALID_ARG;
  if (d < 32 || d > 256 || d % 32 || Lmax < 0 || !dtype_ok(dt) || !(scale > 0.f))
    return MEDUSA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (use_tc(N, Hq, Hkv, d, Lmax, dt, q, kc, vc, kt, vt, out)) {
    const size_t need = tree_attention_tc_ws_bytes(n_layers, B, N, Hq, Hkv, d, Lmax);
    if (need && (!ws || ws_bytes < need)) return MEDUSA_ERR_WORKSPACE;
    return tree_attention_tc(q, kc, vc, kt, vt, mask, prefix_len, n_layers, B, N, Hq, Hkv, d, Lmax,
                             scale, out, ws, ws_bytes, d_status, s);
  }
  if (dt == MEDUSA_BF16)
    return launch_simt<uint16_t>(q, kc, vc, kt, vt, mask, prefix_len, n_layers, B, N, Hq, Hkv, d,
                                 Lmax, scale, out, d_status, s);
  return launch_simt<float>(q, kc, vc, kt, vt, mask, prefix_len, n_layers, B, N, Hq, Hkv, d, Lmax,
                            scale, out, d_status, s);
}
