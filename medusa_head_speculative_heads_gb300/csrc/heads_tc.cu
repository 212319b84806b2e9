// Medusa heads at decode batches of 4 and more, on tcgen05 tensor cores.
//
// Paper review ("Medusa: Simple LLM Inference Acceleration Framework with
// Multiple Decoding Heads"), section "Medusa 的三个核心组件":
// p^(k) = softmax(W2^(k) (SiLU(W1^(k) h) + h)).  At B >= 4 the weight stream is
// a real (skinny) matrix product, so both passes run as
//   D[128 weight rows, N] = W_tile[128, H] x X^T[H, N]
// with bf16 operands and an fp32 accumulator in tensor memory.  X holds the
// batch rows twice: rows 0..Bp-1 are the bf16 "hi" part of the fp32 vector and
// rows Bp..2Bp-1 the "lo" remainder (v = hi + lo to ~2^-16), so the epilogue
// sums D[:, b] + D[:, Bp + b] and the product keeps the fp32 vector's
// precision.  For W1, X = h (exact in bf16: no lo part, so the product has Bp
// columns); the W1 epilogue applies SiLU and the residual and writes u
// split into hi/lo for W2.  The W2 epilogue writes the fp32 logits z and, for
// every batch row, the maximum of each 32-row group (one warp's rows, by a
// shuffle transpose-reduction), which the group ranking kernel uses to read
// only the few groups that can hold a top-k logit.
//
// Roles (256 threads, one CTA per SM, persistent over 128-row tiles): warp 0
// lane 0 issues TMA loads of the A (weights) and B (vector) tiles into a ring
// sized per pass (the smaller the B tile, the more weight bytes in flight: W2
// 7 to 11 stages, W1, whose B tile has no lo rows, 9 to 12); warp 1 allocates
// TMEM and lane 0 issues the
// MMAs (four K=16 steps per 64-column stage) into one of two accumulators;
// warps 4-7 read the accumulator (one row per thread) and write the outputs,
// so the epilogue of one tile overlaps the main loop of the next.  The W1
// epilogue's residual h values are loaded before the accumulator wait.  Every wait is
// bounded; a timeout sets MEDUSA_DEV_TIMEOUT and the kernel drains its
// copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "host_util.h"
#include "sm100.cuh"

namespace medusa {
using namespace sm100;

namespace htc {

constexpr int kThreads = 256;
constexpr int kMaxStages = 12;
constexpr uint32_t kATile = 16384;  // 128 rows x 128 bytes
constexpr uint32_t kTmemCols = 256;  // two accumulators of up to 128 columns

// Ring geometry for a padded batch BP and a pass: the B tile holds BP rows of
// 128 bytes in the W1 pass (h) and 2 BP rows in the W2 pass (u, hi and lo).
template <int BP, bool W1>
struct Ring {
  static constexpr uint32_t kStageBytes = kATile + 128u * (W1 ? BP : 2 * BP);
  static constexpr int kStages = (int)(224u * 1024u / kStageBytes) < kMaxStages ? (int)(224u * 1024u / kStageBytes)
                                                                                 : kMaxStages;
  static constexpr uint32_t kOffBar = kStages * kStageBytes;
  static constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
  static_assert(kStageBytes % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};
constexpr int kNextBoxes = 24;  // W2 boxes per CTA the W1 pass brings into L2
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint64_t kDrainNs = 100000000ull;

struct Params {
  int K, R, H, B, Bp, N;  // R rows per head, N = 2 * Bp (rows of u2 per head)
  int mma_n;              // columns of the product: N (W2: hi and lo rows), Bp (W1: h is exact in bf16)
  int tiles_per_head, tiles;
  int next_R, next_tiles_per_head, next_tiles;  // W1 pass: the W2 pass's geometry (its first boxes go to L2)
  const uint16_t* h;      // [B][H] bf16 (W1 residual)
  uint16_t* u2;           // [K][N][H] bf16, W1 output (hi rows, then lo rows)
  float* z;               // [B][K][R] fp32, W2 output
  float* gmax;            // [B][K][4 tiles_per_head] fp32, W2: maximum of each 32-row group of z
  int32_t* d_status;
};

struct Bars {
  uint64_t full[kMaxStages], empty[kMaxStages], acc_full[2], acc_empty[2], drain;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort, kWaitNs);
  return __all_sync(0xffffffffu, ok);
}

// Column maxima of a warp: on entry a[0..N) holds this lane's values of N
// columns (N a power of two, 16 to 64).  Each step with lane offset O halves
// the columns a lane keeps (the lane with bit O set keeps the upper half) and
// takes the maximum with the partner's copy of them; once a lane keeps one
// column the remaining steps only combine partners.  On return lane L holds
// the warp maximum of columns 2L and 2L + 1 in a[0], a[1] (N = 64), of column
// L (N = 32), or of column L / 2 (N = 16).
template <int CUR, int O, int N>
__device__ __forceinline__ void warp_colmax_step(float (&a)[N], int lane) {
  if constexpr (O > 0) {
    if constexpr (CUR > 1) {
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < CUR / 2; ++i) {
        const float send = up ? a[i] : a[i + CUR / 2];
        const float keep = up ? a[i + CUR / 2] : a[i];
        a[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, O));
      }
      warp_colmax_step<CUR / 2, O / 2, N>(a, lane);
    } else {
      a[0] = fmaxf(a[0], __shfl_xor_sync(0xffffffffu, a[0], O));
      warp_colmax_step<1, O / 2, N>(a, lane);
    }
  }
}

template <int N, int O>
__device__ __forceinline__ void warp_colmax(float (&a)[N], int lane) {
  static_assert(N == 16 || N == 32 || N == 64, "columns");
  warp_colmax_step<N, O, N>(a, lane);
}

}  // namespace htc

template <int BP, bool W1>
__global__ void __launch_bounds__(htc::kThreads, 1)
heads_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_next, const htc::Params p) {
  constexpr int NC = 2 * BP;  // accumulator columns
  using namespace htc;
  constexpr int kStages = Ring<BP, W1>::kStages;
  constexpr uint32_t kStageBytes = Ring<BP, W1>::kStageBytes;
  constexpr uint32_t kOffBar = Ring<BP, W1>::kOffBar;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
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
  const int ksteps = p.H / 64;
  // Each CTA walks the K blocks of its tiles starting at its own offset, so
  // CTAs working in step do not all read the same vector box from L2 at once.
  const int k_rot = (int)((blockIdx.x * 5u) % (unsigned)ksteps);
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tm_a);
    tma_prefetch(&tm_b);
    // The weights are never written during a call, so before the dependency
    // wait: bring this CTA's first ring fill into L2 (in the order the loads
    // will want it) while an earlier kernel finishes, and in the W1 pass also
    // the next kStages .. kStages + kNextBoxes boxes of the first tile that
    // the W2 CTA of the same index will stream (its first kStages it fetches
    // itself).  The W1 weight loads are marked evict-first, so these lines
    // stay in L2 while the W1 pass streams through it.
    const int n = kStages < ksteps ? kStages : ksteps;
    if ((int)blockIdx.x < p.tiles) {
      const int tile = blockIdx.x;
      const int k = tile / p.tiles_per_head, m0 = (tile % p.tiles_per_head) * 128;
      for (int i = 0; i < n; ++i) {
        const int kk = i + k_rot < ksteps ? i + k_rot : i + k_rot - ksteps;
        tma_prefetch_l2_2d(&tm_a, kk * 64, k * p.R + m0);
      }
    }
    if (W1 && (int)blockIdx.x < p.next_tiles) {
      const int tile = blockIdx.x;
      const int k = tile / p.next_tiles_per_head, m0 = (tile % p.next_tiles_per_head) * 128;
      constexpr int kNextStages = Ring<BP, false>::kStages;
      const int lo = kNextStages < ksteps ? kNextStages : ksteps;
      const int hi = lo + kNextBoxes < ksteps ? lo + kNextBoxes : ksteps;
      for (int i = lo; i < hi; ++i) {
        const int kk = i + k_rot < ksteps ? i + k_rot : i + k_rot - ksteps;
        tma_prefetch_l2_2d(&tm_next, kk * 64, k * p.next_R + m0);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  pdl_trigger();
  const uint32_t tmem = s_tmem;
  const uint32_t b_bytes = (uint32_t)p.mma_n * 128;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int g = 0;
      bool alive = true;
      const uint64_t once = l2_policy_evict_first();  // every weight byte is read once per call
      for (int tile = blockIdx.x; tile < p.tiles && alive; tile += gridDim.x) {
        const int k = tile / p.tiles_per_head, m0 = (tile % p.tiles_per_head) * 128;
        for (int i = 0; i < ksteps; ++i, ++g) {
          const int kk = i + k_rot < ksteps ? i + k_rot : i + k_rot - ksteps;
          const int s = g % kStages;
          if (g >= kStages &&
              !(alive = mbar_wait_bounded(&bars->empty[s], ((g / kStages) - 1) & 1, &s_abort, kWaitNs)))
            break;
          uint8_t* st = smem + s * kStageBytes;
          mbar_expect_tx(&bars->full[s], kATile + b_bytes);
          tma_load_2d_hint(st, &tm_a, &bars->full[s], kk * 64, k * p.R + m0, once);
          tma_load_2d(st + kATile, &tm_b, &bars->full[s], kk * 64, W1 ? 0 : k * p.N);
        }
      }
      if (!alive)
        for (int c = g - 1; c >= 0 && c >= g - kStages; --c)
          mbar_wait_bounded(&bars->full[c % kStages], (c / kStages) & 1, nullptr, kDrainNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, p.mma_n, false, false);
    int g = 0, tc = 0;
    bool alive = true;
    for (int tile = blockIdx.x; tile < p.tiles && alive; tile += gridDim.x, ++tc) {
      const int ab = tc & 1;
      if (tc >= 2 && !(alive = warp_wait(&bars->acc_empty[ab], ((tc >> 1) - 1) & 1, &s_abort))) break;
      tc_fence_after();
      for (int i = 0; i < ksteps; ++i, ++g) {
        const int s = g % kStages;
        if (!(alive = warp_wait(&bars->full[s], (g / kStages) & 1, &s_abort))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a = smem_u32(smem + s * kStageBytes);
          const uint32_t b = a + kATile;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mma_bf16(tmem + ab * 128, smem_desc_sw128(a + j * 32, 16, 1024), smem_desc_sw128(b + j * 32, 16, 1024),
                     idesc, (i > 0 || j > 0) ? 1u : 0u);
          mma_commit(&bars->empty[s]);
        }
        __syncwarp();
      }
      if (!alive) break;
      if (lane == 0) mma_commit(&bars->acc_full[ab]);
      __syncwarp();
    }
    if (lane == 0) {
      // Wait (bounded) for every MMA and arrive this warp issued before TMEM
      // is released and the CTA's shared memory goes away.
      mma_commit(&bars->drain);
      mbar_wait_bounded(&bars->drain, 0, nullptr, kDrainNs);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int m = threadIdx.x - 128;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp - 4)) << 16);
    int tc = 0;
    for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++tc) {
      const int ab = tc & 1;
      // W1: this row's residual h[b][row] (bf16 pairs), loaded while the MMAs run.
      uint32_t hres[BP / 2];
      if (W1) {
        const int row = (tile % p.tiles_per_head) * 128 + m;
#pragma unroll
        for (int b2 = 0; b2 < BP / 2; ++b2) {
          const uint32_t lo = (2 * b2 < p.B && row < p.R) ? __ldg(p.h + (size_t)(2 * b2) * p.H + row) : 0u;
          const uint32_t hi = (2 * b2 + 1 < p.B && row < p.R) ? __ldg(p.h + (size_t)(2 * b2 + 1) * p.H + row) : 0u;
          hres[b2] = lo | (hi << 16);
        }
      }
      if (!warp_wait(&bars->acc_full[ab], (tc >> 1) & 1, &s_abort)) break;
      tc_fence_after();
      // W1 products have BP columns (no lo part), W2 products 2 BP.
      float v[NC];
      if (W1) {
#pragma unroll
        for (int c = 0; c < BP / 8; ++c) tmem_ld8(lane_addr + ab * 128 + c * 8, v + c * 8);
      } else {
#pragma unroll
        for (int c = 0; c < NC / 32; ++c) tmem_ld32(lane_addr + ab * 128 + c * 32, v + c * 32);
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->acc_empty[ab]);
      const int k = tile / p.tiles_per_head, row = (tile % p.tiles_per_head) * 128 + m;
      if (W1) {
        if (row >= p.R) continue;
#pragma unroll
        for (int b = 0; b < BP; ++b) {
          float val = 0.f;
          if (b < p.B) val = v[b] / (1.f + expf(-v[b])) + bf16_bits_to_f32((hres[b >> 1] >> (16 * (b & 1))) & 0xffffu);
          const uint32_t hi = f32_to_bf16_bits(val);
          const uint32_t lo = f32_to_bf16_bits(val - bf16_bits_to_f32(hi));
          p.u2[((size_t)k * p.N + b) * p.H + row] = (uint16_t)hi;
          p.u2[((size_t)k * p.N + BP + b) * p.H + row] = (uint16_t)lo;
        }
      } else {
        // z = hi and lo products summed; rows past the vocabulary and padded
        // batch columns enter the group maxima as -inf.
        constexpr int RB = BP > 32 ? 64 : BP;  // columns of the warp reduction (a power of two)
        float a[RB];
#pragma unroll
        for (int b = 0; b < BP; ++b) a[b] = (b < p.B && row < p.R) ? v[b] + v[BP + b] : -INFINITY;
#pragma unroll
        for (int b = BP; b < RB; ++b) a[b] = -INFINITY;
        if (row < p.R) {
#pragma unroll
          for (int b = 0; b < BP; ++b)
            if (b < p.B) p.z[((size_t)b * p.K + k) * p.R + row] = a[b];
        }
        // Maximum of this warp's 32 rows for every batch column, for the
        // ranking kernel: it skips every 32-row group whose maximum is below
        // its threshold.
        warp_colmax<RB, 16>(a, lane);
        const int groups = 4 * p.tiles_per_head, gi = (tile % p.tiles_per_head) * 4 + (warp - 4);
        if constexpr (RB == 64) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int b = 2 * lane + i;
            if (b < p.B) p.gmax[((size_t)b * p.K + k) * groups + gi] = a[i];
          }
        } else if constexpr (RB == 32) {
          if (lane < p.B) p.gmax[((size_t)lane * p.K + k) * groups + gi] = a[0];
        } else {
          if (!(lane & 1) && (lane >> 1) < p.B) p.gmax[((size_t)(lane >> 1) * p.K + k) * groups + gi] = a[0];
        }
      }
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

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 heads_encode_fn() {
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

// 2D bf16 map over rows of H elements: box 64 columns x box_rows rows, 128-byte swizzle.
static bool map_rows(CUtensorMap* m, const void* base, int H, long long rows, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)H * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return heads_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Padded batch of the tensor-core heads path (N = 2 * Bp columns, a multiple of 32).
int heads_tc_bp(int B) { return (B + 15) / 16 * 16; }

bool heads_tc_supported(int B, int H, const void* h, const void* w1, const void* w2) {
  return B >= 4 && B <= 64 && H % 64 == 0 && H >= 64 && aligned16(h) && aligned16(w1) && aligned16(w2) &&
         heads_encode_fn() != nullptr;
}

// The instantiation of one pass for a padded batch, with its shared memory.
struct heads_tc_pass {
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, htc::Params);
  uint32_t smem;
};
template <bool W1>
static heads_tc_pass heads_tc_pick(int Bp) {
  if (Bp == 16) return {heads_tc_kernel<16, W1>, htc::Ring<16, W1>::kSmemBytes};
  if (Bp == 32) return {heads_tc_kernel<32, W1>, htc::Ring<32, W1>::kSmemBytes};
  if (Bp == 48) return {heads_tc_kernel<48, W1>, htc::Ring<48, W1>::kSmemBytes};
  return {heads_tc_kernel<64, W1>, htc::Ring<64, W1>::kSmemBytes};
}

// Both passes: u2 = split(SiLU(W1 h) + h) ([K][2Bp][H] bf16, caller scratch),
// then z = W2 u ([B][K][V] fp32) and the maximum of every 32-row group of z
// ([B][K][4 ceil(V / 128)] fp32, groups past V hold -inf).
medusa_status heads_tc_run(const uint16_t* h, const uint16_t* w1, const uint16_t* w2, int B, int H, int V, int K,
                           uint16_t* u2, float* z, float* gmax, int32_t* d_status, cudaStream_t s) {
  const int Bp = heads_tc_bp(B), N = 2 * Bp;
  CUtensorMap ma1, mb1, ma2, mb2;
  if (!map_rows(&ma1, w1, H, (long long)K * H, 128) || !map_rows(&mb1, h, H, B, Bp) ||
      !map_rows(&ma2, w2, H, (long long)K * V, 128) || !map_rows(&mb2, u2, H, (long long)K * N, N))
    return MEDUSA_ERR_CUDA;
  const heads_tc_pass k1 = heads_tc_pick<true>(Bp), k2 = heads_tc_pick<false>(Bp);
  if (cudaFuncSetAttribute(k1.kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k1.smem) != cudaSuccess ||
      cudaFuncSetAttribute(k2.kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k2.smem) != cudaSuccess)
    return MEDUSA_ERR_CUDA;
  const int sms = device_sm_count();
  // Equal-cost tiles: as many rounds as the SM count forces, spread evenly.
  auto grid_for = [&](int tiles) {
    const int rounds = (tiles + sms - 1) / sms;
    return (tiles + rounds - 1) / rounds;
  };
  htc::Params p{};
  p.K = K;
  p.H = H;
  p.B = B;
  p.Bp = Bp;
  p.N = N;
  p.h = h;
  p.u2 = u2;
  p.z = z;
  p.gmax = gmax;
  p.d_status = d_status;
  // W1: rows per head = H
  p.R = H;
  p.mma_n = Bp;
  p.tiles_per_head = ceil_div(H, 128);
  p.tiles = K * p.tiles_per_head;
  p.next_R = V;
  p.next_tiles_per_head = ceil_div(V, 128);
  p.next_tiles = grid_for(K * p.next_tiles_per_head);  // the W2 CTAs' first tiles
  launch_pdl(k1.kern, dim3(grid_for(p.tiles)), dim3(htc::kThreads), k1.smem, s, ma1, mb1, ma2, p);
  // W2: rows per head = V
  p.R = V;
  p.mma_n = N;
  p.tiles_per_head = ceil_div(V, 128);
  p.tiles = K * p.tiles_per_head;
  launch_pdl(k2.kern, dim3(grid_for(p.tiles)), dim3(htc::kThreads), k2.smem, s, ma2, mb2, ma2, p);
  return launch_status();
}

}  // namespace medusa
