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
// tokens (MMA N = TN).  The K blocks of all tiles, laid end to end tile after
// tile, are divided evenly over the grid (one CTA per SM): CTA c takes the
// contiguous range [c W / G, (c + 1) W / G) of the W = tiles x K-block
// sequence, so no SM idles when the tile count is not a multiple of the SM
// count (a small T or narrow layer has fewer tiles than SMs; 172 tiles of a
// 22016-wide layer would otherwise take two rounds on 152 SMs).  A tile whose
// K range a CTA covers whole is written to y by that CTA; a tile shared by
// several CTAs (at most the first and the last of each CTA's range) leaves an
// fp32 partial per CTA, which a second kernel adds in CTA order (a fixed
// order: deterministic).  Roles (256 threads): warp 0 lane 0 issues TMA loads
// of the W and x boxes (128-byte swizzle) into a 4- to 14-stage ring (216 KB);
// warp 1 owns TMEM and lane 0 issues the MMAs into one of two 256-column
// accumulators; warps 4-7 read the accumulator 32 columns at a time (one
// feature row per thread) and write y or the partial.  Every wait is bounded;
// a timeout sets MEDUSA_DEV_TIMEOUT, drains and frees TMEM.
#include <cuda.h>
#include <math.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "medusa_test_hooks.h"
#include "host_util.h"
#include "sm100.cuh"

namespace medusa {
using namespace sm100;

namespace lin {

constexpr int kThreads = 256;
constexpr int kMaxStages = 14;
constexpr int kMinBlocksPerCta = 4;       // K blocks: fewer CTAs when the whole product is smaller
constexpr int kReduceCols = 16;           // token columns per block of the partial reduction
constexpr uint32_t kATile = 16384;        // 128 W rows x 128 bytes
constexpr uint32_t kRingBytes = 221184;   // 216 KB of stages
constexpr uint32_t kBarBytes = 512;
constexpr uint32_t kSmemBytes = kRingBytes + kBarBytes + 1024;  // + alignment slack of the base
constexpr uint32_t kTmemCols = 512;       // two accumulators of up to 256 columns
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint64_t kDrainNs = 100000000ull;

struct Params {
  int T, K, Nout, TN, mtiles, ntiles, kblocks, grid, stages;
  long long work;      // tiles x kblocks, divided evenly over the grid
  int withhold_first;  // test hook: the first stage's loads are never issued
  uint32_t stage_bytes;
  uint16_t* y;
  float* part;       // [grid][2][TN][128] when some tile is shared (feature fastest: coalesced)
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

// First flattened K block of CTA c (tile-major: block w is K block w % kblocks
// of tile w / kblocks); CTA c owns [work_begin(c), work_begin(c + 1)).
__host__ __device__ __forceinline__ long long work_begin(long long work, int grid, int c) {
  return work * c / grid;
}

// The CTA whose range holds flattened block w: the largest c with
// work_begin(c) <= w.
__device__ __forceinline__ int work_owner(long long work, int grid, long long w) {
  return (int)(((w + 1) * grid - 1) / work);
}

// One tile's part of a CTA's range: K blocks [kb0, kb1) of the tile; slot -1
// when that is the whole tile (y written directly), else the CTA's partial
// slot (0 for the first tile of its range, 1 for the last).
struct Seg {
  int mt, nt, kb0, kb1, slot;
};

__device__ __forceinline__ Seg segment(const Params& p, int tile, long long w0, long long w1, int first_tile) {
  Seg x;
  x.mt = tile % p.mtiles;
  x.nt = tile / p.mtiles;
  const long long base = (long long)tile * p.kblocks, end = base + p.kblocks;
  x.kb0 = (int)((w0 > base ? w0 : base) - base);
  x.kb1 = (int)((w1 < end ? w1 : end) - base);
  x.slot = (x.kb0 == 0 && x.kb1 == p.kblocks) ? -1 : (tile == first_tile ? 0 : 1);
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
  // This CTA's K blocks (non-empty: the grid is at most the block count).
  const long long w0 = work_begin(p.work, p.grid, blockIdx.x), w1 = work_begin(p.work, p.grid, blockIdx.x + 1);
  const int t_first = (int)(w0 / p.kblocks), t_last = (int)((w1 - 1) / p.kblocks);
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tm_w);
    tma_prefetch(&tm_x);
    // The weights are not written while the layers of a pass run: while an
    // earlier kernel on the stream finishes, bring this CTA's first ring's
    // worth of weight boxes into L2 (x, an earlier layer's output, waits).
    const Seg x = segment(p, t_first, w0, w1, t_first);
    const int kend = x.kb1 < x.kb0 + p.stages ? x.kb1 : x.kb0 + p.stages;
    for (int kb = x.kb0; kb < kend; ++kb) tma_prefetch_l2_2d(&tm_w, kb * 64, x.mt * 128);
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
      for (int t = t_first; t <= t_last && alive; ++t) {
        const Seg x = segment(p, t, w0, w1, t_first);
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
    for (int t = t_first; t <= t_last && alive; ++t, ++tc) {
      const Seg x = segment(p, t, w0, w1, t_first);
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
    for (int t = t_first; t <= t_last; ++t, ++tc) {
      const Seg x = segment(p, t, w0, w1, t_first);
      const int ab = tc & 1;
      if (!warp_wait(&bars->acc_full[ab], (tc >> 1) & 1, &s_abort)) break;
      tc_fence_after();
      const int n = x.mt * 128 + m;      // output feature of this thread
      const int t0 = x.nt * p.TN;        // first token of the tile
      const bool direct = x.slot < 0;
      float* pbase = direct ? nullptr : p.part + ((size_t)blockIdx.x * 2 + x.slot) * p.TN * 128 + m;
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

// Shared tiles: y = bf16(sum of the tile's partials, in CTA order).  Block x
// looks at the boundary between CTAs x and x + 1; when it falls inside a tile
// and no earlier boundary falls inside the same tile, the block adds that
// tile's partials for kReduceCols of its token columns (blockIdx.y): lane l
// takes output features 4l..4l+3 (one 16-byte load per contributing CTA and
// column), warp w columns 2w and 2w + 1.  The loads of four CTAs for both
// columns are issued before their adds (the sum stays in CTA order), and each
// result is one 8-byte store (element stores at a ragged feature tail or when
// Nout is not a multiple of 4).
__global__ void __launch_bounds__(256)
linear_reduce_kernel(const float* __restrict__ part, uint16_t* __restrict__ y, int T, int Nout, int TN,
                     int mtiles, int kblocks, long long work, int grid) {
  using namespace lin;
  pdl_wait();
  pdl_trigger();
  const int c = blockIdx.x + 1;  // first CTA after the boundary
  const long long wc = work_begin(work, grid, c);
  if (wc % kblocks == 0) return;  // on a tile edge: no tile shared here
  const int tile = (int)(wc / kblocks);
  const long long base = (long long)tile * kblocks;
  const long long wp = work_begin(work, grid, c - 1);
  if (wp > base) return;  // the boundary before this one is inside the same tile and takes it
  const int mt = tile % mtiles, nt = tile / mtiles;
  const int row = (threadIdx.x & 31) * 4, n = mt * 128 + row;
  if (n >= Nout) return;
  const int c_hi = work_owner(work, grid, base + kblocks - 1);
  const size_t slot_elems = (size_t)TN * 128;
  // CTA c - 1 holds the tile's first part: in its slot 0 when the tile is the
  // first of its range (it starts at the tile's first block), else slot 1; the
  // later CTAs start inside the tile, so it is their first (slot 0).
  const float* first = part + ((size_t)(c - 1) * 2 + (wp == base ? 0 : 1)) * slot_elems;
  const int col0 = blockIdx.y * kReduceCols + (threadIdx.x >> 5) * 2;
  bool ok[2];
  size_t off[2];
  float4 acc[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int col = col0 + i;
    ok[i] = col < TN && nt * TN + col < T;
    off[i] = (size_t)col * 128 + row;
    if (ok[i]) acc[i] = __ldcg(reinterpret_cast<const float4*>(first + off[i]));
  }
  for (int cc = c; cc <= c_hi; cc += 4) {
    float4 v[2][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 2; ++i)
        if (cc + j <= c_hi && ok[i])
          v[i][j] = __ldcg(reinterpret_cast<const float4*>(part + (size_t)(cc + j) * 2 * slot_elems + off[i]));
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 2; ++i)
        if (cc + j <= c_hi && ok[i]) {
          acc[i].x += v[i][j].x;
          acc[i].y += v[i][j].y;
          acc[i].z += v[i][j].z;
          acc[i].w += v[i][j].w;
        }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (!ok[i]) continue;
    uint16_t* out = y + (size_t)(nt * TN + col0 + i) * Nout + n;
    if ((Nout & 3) == 0) {
      *reinterpret_cast<uint2*>(out) = make_uint2(bf16x2_rn(acc[i].x, acc[i].y), bf16x2_rn(acc[i].z, acc[i].w));
    } else {
      const float a[4] = {acc[i].x, acc[i].y, acc[i].z, acc[i].w};
      for (int j = 0; j < 4 && n + j < Nout; ++j) out[j] = (uint16_t)f32_to_bf16_bits(a[j]);
    }
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
  int TN, mtiles, ntiles, kblocks, grid, stages;
  long long work;
  bool shared;  // some tile's K range spans two CTAs: partials and the reduce kernel
  uint32_t stage_bytes;
  size_t part_bytes;
};

static LinearPlan linear_plan(int T, int K, int Nout) {
  LinearPlan L{};
  L.TN = T <= 256 ? (T + 15) / 16 * 16 : 256;
  L.ntiles = (T + L.TN - 1) / L.TN;
  L.mtiles = (Nout + 127) / 128;
  L.kblocks = (K + 63) / 64;
  L.work = (long long)L.mtiles * L.ntiles * L.kblocks;
  // One CTA per SM, each with an equal share of the K blocks (at least
  // kMinBlocksPerCta of them).
  long long g = L.work / lin::kMinBlocksPerCta;
  if (g > device_sm_count()) g = device_sm_count();
  L.grid = g < 1 ? 1 : (int)g;
  L.shared = false;
  for (int c = 1; c < L.grid && !L.shared; ++c) L.shared = lin::work_begin(L.work, L.grid, c) % L.kblocks != 0;
  L.stage_bytes = lin::kATile + (uint32_t)L.TN * 128;
  L.stages = (int)(lin::kRingBytes / L.stage_bytes);
  if (L.stages > lin::kMaxStages) L.stages = lin::kMaxStages;
  L.part_bytes = L.shared ? (size_t)L.grid * 2 * L.TN * 128 * sizeof(float) : 0;
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
  p.kblocks = L.kblocks;
  p.grid = L.grid;
  p.work = L.work;
  p.stages = L.stages;
  p.stage_bytes = L.stage_bytes;
  p.y = static_cast<uint16_t*>(y);
  p.part = L.shared ? static_cast<float*>(ws) : nullptr;
  p.d_status = d_status;
  p.withhold_first = withhold_first;
  if (cudaFuncSetAttribute(linear_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lin::kSmemBytes) !=
      cudaSuccess)
    return MEDUSA_ERR_CUDA;
  launch_pdl(linear_tc_kernel, dim3(L.grid), dim3(lin::kThreads), lin::kSmemBytes, s, mw, mx, p);
  if (L.shared)
    launch_pdl(linear_reduce_kernel, dim3((unsigned)(L.grid - 1), (unsigned)((L.TN + lin::kReduceCols - 1) / lin::kReduceCols)),
               dim3(256), 0, s,
               static_cast<const float*>(ws), p.y, T, Nout, L.TN, L.mtiles, L.kblocks, L.work, L.grid);
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

