// medusa_linear: y = x W^T for the verify pass's tree tokens on tcgen05 tensor
// cores (bf16 operands, fp32 accumulation in tensor memory, bf16 out).
//
// Paper review ("Medusa: Simple LLM Inference Acceleration Framework with
// Multiple Decoding Heads"), roofline analysis in "实验设计与结果" and
// "局限性": verifying a tree of N candidates runs every linear layer of the
// backbone over B * N tokens instead of B, which lifts the operational
// intensity of decoding; past a batch of about 32 the linear layers become
// compute-bound.  This is that layer: x [T][K] (T = B * N tokens), W [Nout][K]
// (row-major, the usual (out, in) layout), y [T][Nout].
//
// Tiles of 128 output features (the weight rows, MMA M = 128) by up to 256
// tokens (MMA N = TN).  Few tiles (small T, narrow layers) would leave SMs idle
// while the weights stream from HBM, so each tile's K range is split S ways
// into fp32 partials, which a second kernel adds in a fixed order (four
// output features per thread; deterministic).  Roles (256 threads, persistent
// over the units): warp 0 lane 0 issues TMA loads of the W and x boxes
// (128-byte swizzle) into a 4- to 12-stage ring (216 KB); warp 1 owns TMEM and lane 0 issues the MMAs into one of
// two 256-column accumulators; warps 4-7 read the accumulator 32 columns at a
// time (one feature row per thread) and write y or the partial.  Every wait is
// bounded; a timeout sets MEDUSA_DEV_TIMEOUT, drains and frees TMEM.
#include <cuda.h>
#include <math.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "host_util.h"
#include "sm100.cuh"

namespace medusa {
using namespace sm100;

namespace lin {

constexpr int kThreads = 256;
constexpr int kMaxStages = 14;
constexpr int kMaxSplit = 16;
constexpr uint32_t kATile = 16384;        // 128 W rows x 128 bytes
constexpr uint32_t kRingBytes = 221184;   // 216 KB of stages
constexpr uint32_t kBarBytes = 512;
constexpr uint32_t kSmemBytes = kRingBytes + kBarBytes + 1024;  // + alignment slack of the base
constexpr uint32_t kTmemCols = 512;       // two accumulators of up to 256 columns
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint64_t kDrainNs = 100000000ull;

struct Params {
  int T, K, Nout, TN, mtiles, ntiles, S, kblocks, units, stages;
  int withhold_first;  // test hook: the first stage's loads are never issued
  uint32_t stage_bytes;
  uint16_t* y;
  float* part;       // [tiles][S][TN][128] when S > 1 (feature fastest: coalesced)
  int32_t* d_status;
};

struct Bars {
  uint64_t full[kMaxStages], empty[kMaxStages], acc_full[2], acc_empty[2], drain;
};
static_assert(sizeof(Bars) <= kBarBytes, "barriers overflow their slot");

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort, kWaitNs);
  return __all_sync(0xffffffffu, ok);
}

struct Unit {
  int tile, mt, nt, s, kb0, kb1;
};

__device__ __forceinline__ Unit decode(const Params& p, int u) {
  Unit x;
  x.tile = u / p.S;
  x.s = u - x.tile * p.S;
  x.mt = x.tile % p.mtiles;
  x.nt = x.tile / p.mtiles;
  x.kb0 = (int)((long long)p.kblocks * x.s / p.S);
  x.kb1 = (int)((long long)p.kblocks * (x.s + 1) / p.S);
  return x;
}

}  // namespace lin

__global__ void __launch_bounds__(lin::kThreads, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const lin::Params p) {
  using namespace lin;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kRingBytes);
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->acc_full[s], 1);
      mbar_init(&bars->acc_empty[s], 128);
    }
    mbar_init(&bars->drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tm_w);
    tma_prefetch(&tm_x);
    // The weights are not written while the layers of a pass run: while an
    // earlier kernel on the stream finishes, bring this CTA's first ring's
    // worth of weight boxes into L2 (x, an earlier layer's output, waits).
    if ((int)blockIdx.x < p.units) {
      const Unit x = decode(p, blockIdx.x);
      const int kend = x.kb1 < x.kb0 + p.stages ? x.kb1 : x.kb0 + p.stages;
      for (int kb = x.kb0; kb < kend; ++kb) tma_prefetch_l2_2d(&tm_w, kb * 64, x.mt * 128);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  pdl_trigger();
  const uint32_t tmem = s_tmem;
  const uint32_t b_bytes = (uint32_t)p.TN * 128;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int g = 0;
      bool alive = true;
      for (int u = blockIdx.x; u < p.units && alive; u += gridDim.x) {
        const Unit x = decode(p, u);
        for (int kb = x.kb0; kb < x.kb1; ++kb, ++g) {
          const int s = g % p.stages;
          if (g >= p.stages &&
              !(alive = mbar_wait_bounded(&bars->empty[s], ((g / p.stages) - 1) & 1, &s_abort, kWaitNs)))
            break;
          uint8_t* st = smem + s * p.stage_bytes;
          mbar_expect_tx(&bars->full[s], kATile + b_bytes);
          if (p.withhold_first && g == 0) continue;  // that stage never fills: the bounded waits expire
          tma_load_2d(st, &tm_w, &bars->full[s], kb * 64, x.mt * 128);
          tma_load_2d(st + kATile, &tm_x, &bars->full[s], kb * 64, x.nt * p.TN);
        }
      }
      if (!alive)
        for (int c = g - 1; c >= 0 && c >= g - p.stages; --c)
          mbar_wait_bounded(&bars->full[c % p.stages], (c / p.stages) & 1, nullptr, kDrainNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, p.TN, false, false);
    int g = 0, tc = 0;
    bool alive = true;
    for (int u = blockIdx.x; u < p.units && alive; u += gridDim.x, ++tc) {
      const Unit x = decode(p, u);
      const int ab = tc & 1;
      if (tc >= 2 && !(alive = warp_wait(&bars->acc_empty[ab], ((tc >> 1) - 1) & 1, &s_abort))) break;
      tc_fence_after();
      for (int kb = x.kb0; kb < x.kb1; ++kb, ++g) {
        const int s = g % p.stages;
        if (!(alive = warp_wait(&bars->full[s], (g / p.stages) & 1, &s_abort))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a = smem_u32(smem + s * p.stage_bytes);
          const uint32_t b = a + kATile;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mma_bf16(tmem + ab * 256, smem_desc_sw128(a + j * 32, 16, 1024), smem_desc_sw128(b + j * 32, 16, 1024),
                     idesc, (kb > x.kb0 || j > 0) ? 1u : 0u);
          mma_commit(&bars->empty[s]);
        }
        __syncwarp();
      }
      if (!alive) break;
      if (lane == 0) mma_commit(&bars->acc_full[ab]);
      __syncwarp();
    }
    if (!alive && lane == 0) {
      mma_commit(&bars->drain);
      mbar_wait_bounded(&bars->drain, 0, nullptr, kDrainNs);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int m = threadIdx.x - 128;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp - 4)) << 16);
    int tc = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++tc) {
      const Unit x = decode(p, u);
      const int ab = tc & 1;
      if (!warp_wait(&bars->acc_full[ab], (tc >> 1) & 1, &s_abort)) break;
      tc_fence_after();
      const int n = x.mt * 128 + m;      // output feature of this thread
      const int t0 = x.nt * p.TN;        // first token of the tile
      const bool direct = p.S == 1;
      float* pbase = direct ? nullptr : p.part + ((size_t)x.tile * p.S + x.s) * p.TN * 128 + m;
      for (int c = 0; c < p.TN; c += 32) {
        float v[32];
        tmem_ld32(lane_addr + ab * 256 + c, v);
        tmem_wait_ld();
        if (direct) {
          if (n < p.Nout) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int t = t0 + c + j;
              if (t < p.T) p.y[(size_t)t * p.Nout + n] = (uint16_t)f32_to_bf16_bits(v[j]);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)  // TN is a multiple of 16: the last chunk may be half used
            if (c + j < p.TN) pbase[(size_t)(c + j) * 128] = v[j];
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->acc_empty[ab]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // After the barrier: any role's timeout (even one raised after another role
  // finished) is visible here.
  if (threadIdx.x == 0 && s_abort) set_status(p.d_status, MEDUSA_DEV_TIMEOUT);
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Split K: y[t][n] = bf16(sum over s of the partials), s in order.  One thread
// per 4 consecutive output features of a token: the partials are feature
// fastest, so each split is one 16-byte load (all S issued before the first
// add) and the result one 8-byte store (element stores at a ragged feature
// tail or when Nout is not a multiple of 4).
__global__ void __launch_bounds__(256)
linear_reduce_kernel(const float* __restrict__ part, uint16_t* __restrict__ y, int T, int Nout, int TN,
                     int mtiles, int S) {
  pdl_wait();
  pdl_trigger();
  const int nq = (Nout + 3) >> 2;  // feature quads per token
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)T * nq) return;
  const int t = (int)(i / nq), n = (int)(i - (size_t)t * nq) * 4;
  const int tile = (t / TN) * mtiles + n / 128, col = t % TN, row = n % 128;
  const float4* src = reinterpret_cast<const float4*>(part + (((size_t)tile * S) * TN + col) * 128 + row);
  const size_t step = (size_t)TN * 128 / 4;  // one split, in float4
  float4 v[lin::kMaxSplit];
#pragma unroll
  for (int s = 0; s < lin::kMaxSplit; ++s)
    if (s < S) v[s] = __ldcg(src + s * step);
  float a0 = v[0].x, a1 = v[0].y, a2 = v[0].z, a3 = v[0].w;
#pragma unroll
  for (int s = 1; s < lin::kMaxSplit; ++s)
    if (s < S) {
      a0 += v[s].x;
      a1 += v[s].y;
      a2 += v[s].z;
      a3 += v[s].w;
    }
  uint16_t* out = y + (size_t)t * Nout + n;
  if ((Nout & 3) == 0) {
    *reinterpret_cast<uint2*>(out) = make_uint2(bf16x2_rn(a0, a1), bf16x2_rn(a2, a3));
  } else {
    const float a[4] = {a0, a1, a2, a3};
    for (int j = 0; j < 4 && n + j < Nout; ++j) out[j] = (uint16_t)f32_to_bf16_bits(a[j]);
  }
}

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 linear_encode_fn() {
  // Looked up once, thread-safely (function-local static initialisation).
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    cudaGetLastError();
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// bf16 rows of `cols` elements: box 64 columns x box_rows rows, 128-byte swizzle.
static bool linear_map(CUtensorMap* m, const void* base, int cols, long long rows, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return linear_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch geometry shared by the workspace query and the call.
struct LinearPlan {
  int TN, mtiles, ntiles, S, kblocks, units, grid, stages;
  uint32_t stage_bytes;
  size_t part_bytes;
};

static LinearPlan linear_plan(int T, int K, int Nout) {
  LinearPlan L{};
  L.TN = T <= 256 ? (T + 15) / 16 * 16 : 256;
  L.ntiles = (T + L.TN - 1) / L.TN;
  L.mtiles = (Nout + 127) / 128;
  L.kblocks = (K + 63) / 64;
  const int tiles = L.mtiles * L.ntiles;
  const int sms = device_sm_count();
  // Split K from a time model of this GPU (about 6.8 TB/s of HBM and 1.9
  // PFLOP/s of dense bf16, shared by the SMs): a tile costs the larger of its
  // MMA time and its weight-stream time on one SM; S splits run tiles * S
  // units in ceil(tiles * S / SMs) rounds and add the fp32 partials (written
  // and read back once) to the HBM traffic.
  const double sm_flops = 1.9e15 / sms, sm_bw = 6.8e12 / sms, hbm = 6.8e12;
  const double t_tile = fmax(2.0 * 128 * L.TN * (double)K / sm_flops, 128.0 * 2 * (double)K / sm_bw);
  L.S = 1;
  int max_s = L.kblocks / 4 > 1 ? L.kblocks / 4 : 1;  // at least 4 K blocks per unit
  if (max_s > lin::kMaxSplit) max_s = lin::kMaxSplit;
  double best = 1e30;
  for (int S = 1; S <= max_s; ++S) {
    const double rounds = (double)((tiles * S + sms - 1) / sms);
    const double cost = rounds * t_tile / S + (S > 1 ? (double)S * tiles * 128.0 * L.TN * 8.0 / hbm : 0.0);
    if (cost < best * (1.0 - 1e-9)) {
      best = cost;
      L.S = S;
    }
  }
  L.units = tiles * L.S;
  const int rounds = (L.units + sms - 1) / sms;
  L.grid = (L.units + rounds - 1) / rounds;
  L.stage_bytes = lin::kATile + (uint32_t)L.TN * 128;
  L.stages = (int)(lin::kRingBytes / L.stage_bytes);
  if (L.stages > lin::kMaxStages) L.stages = lin::kMaxStages;
  L.part_bytes = L.S > 1 ? (size_t)tiles * L.S * 128 * L.TN * sizeof(float) : 0;

  return L;
}

}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_linear_workspace_size(int T, int K, int Nout) {
  if (T < 1 || K < 1 || Nout < 1) return 0;
  const LinearPlan L = linear_plan(T, K, Nout);
  return L.part_bytes;
}

static medusa_status linear_call(const void* x, const void* w, void* y, int T, int K, int Nout, medusa_dtype dt,
                                 void* ws, size_t ws_bytes, int32_t* d_status, medusa_stream_t stream,
                                 int withhold_first) {
  if (!x || !w || !y || T < 1 || K < 8 || Nout < 1) return MEDUSA_ERR_INVALID_ARG;
  if (dt != MEDUSA_BF16) return MEDUSA_ERR_UNSUPPORTED;
  if (K % 8 || !aligned16(x) || !aligned16(w) || !aligned16(y)) return MEDUSA_ERR_INVALID_ARG;
  const size_t xb = (size_t)T * K * 2, wb = (size_t)Nout * K * 2, yb = (size_t)T * Nout * 2;
  if (overlaps(y, yb, x, xb) || overlaps(y, yb, w, wb)) return MEDUSA_ERR_ALIAS;
  const LinearPlan L = linear_plan(T, K, Nout);
  const size_t need = medusa_linear_workspace_size(T, K, Nout);
  if (need && (!ws || ws_bytes < need || !aligned16(ws))) return MEDUSA_ERR_WORKSPACE;
  if (linear_encode_fn() == nullptr) return MEDUSA_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap mw, mx;
  if (!linear_map(&mw, w, K, Nout, 128) || !linear_map(&mx, x, K, T, L.TN)) return MEDUSA_ERR_CUDA;
  lin::Params p{};
  p.T = T;
  p.K = K;
  p.Nout = Nout;
  p.TN = L.TN;
  p.mtiles = L.mtiles;
  p.ntiles = L.ntiles;
  p.S = L.S;
  p.kblocks = L.kblocks;
  p.units = L.units;
  p.stages = L.stages;
  p.stage_bytes = L.stage_bytes;
  p.y = static_cast<uint16_t*>(y);
  p.part = L.S > 1 ? static_cast<float*>(ws) : nullptr;
  p.d_status = d_status;
  p.withhold_first = withhold_first;
  if (cudaFuncSetAttribute(linear_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lin::kSmemBytes) !=
      cudaSuccess)
    return MEDUSA_ERR_CUDA;
  launch_pdl(linear_tc_kernel, dim3(L.grid), dim3(lin::kThreads), lin::kSmemBytes, s, mw, mx, p);
  if (L.S > 1) {
    const size_t quads = (size_t)T * ((Nout + 3) / 4);
    launch_pdl(linear_reduce_kernel, dim3((unsigned)((quads + 255) / 256)), dim3(256), 0, s,
               static_cast<const float*>(ws), p.y, T, Nout, L.TN, L.mtiles, L.S);
  }
  return launch_status();
}

extern "C" medusa_status medusa_linear(const void* x, const void* w, void* y, int T, int K, int Nout, medusa_dtype dt,
                                       void* ws, size_t ws_bytes, int32_t* d_status, medusa_stream_t stream) {
  return linear_call(x, w, y, T, K, Nout, dt, ws, ws_bytes, d_status, stream, 0);
}

extern "C" medusa_status medusa_linear_test_stall(const void* x, const void* w, void* y, int T, int K, int Nout,
                                                  void* ws, size_t ws_bytes, int32_t* d_status,
                                                  medusa_stream_t stream) {
  return linear_call(x, w, y, T, K, Nout, MEDUSA_BF16, ws, ws_bytes, d_status, stream, 1);
}

