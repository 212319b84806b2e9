// Tree attention on tcgen05 tensor cores: bf16 q/k/v, head_dim 128, fp32
// scores/accumulators in tensor memory.
//
// Paper review ("Medusa: Simple LLM Inference Acceleration Framework with
// Multiple Decoding Heads"), section "Medusa 的三个核心组件" and FAQ
// "树注意力为什么能一次验证多条候选": every tree node attends to the shared prefix
// and to its own ancestors only, all candidates in one pass.
//
// Work item: (layer x row, head group, row tile).  The 128 MMA rows of a tile
// are query rows (node, q head of the GQA group).  When one kv head has at most
// 64 query rows (the 64-node trees with G = 1), two kv heads share a tile:
// rows 0-63 belong to head A and 64-127 to head B, the key tile holds 64 keys
// of A (columns 0-63) and the same 64 key positions of B (columns 64-127), and
// the off-diagonal score blocks are masked, so P is block-diagonal and PV
// keeps the heads apart.  This keeps all four TMEM lane quarters (and the four
// SM sub-partitions' exp units) busy.  Otherwise a tile holds 128 rows of one
// kv head and 128 keys.
//
// Roles (128 + 128 x SPLIT threads): warp 0 lane 0 issues TMA (Q once per
// item; K and V of every key tile into a six-slot ring of 32 KB half-tiles, a
// K slot freed as soon as its S = Q K^T is done, a V slot when its P V is
// done); warp 1 allocates TMEM and lane 0 issues S = Q K^T into one of two S
// buffers; warp 2 lane 0 issues O += P V with P read from tensor memory; the
// softmax warps from warp 4 on read S from TMEM, apply the prefix-length /
// ancestor mask, keep the online softmax in the log2 domain (O is rescaled in
// TMEM only when the row maximum grows by more than 2^8), write P (bf16 pairs)
// into one of two TMEM P buffers and finally normalise O and store the
// output.  With SPLIT = 2 each tile row has two softmax threads (warps 4-7 and
// 8-11 read the same TMEM lane quarters), each with half of the row's scores,
// half of P and half of O's columns: per tile they exchange their partial row
// maxima through shared memory (an mbarrier per lane quarter and tile parity,
// waited on with the same bound as every other wait) so both scale P by the
// same maximum, and they add their partial row sums once per item.  With P double
// buffered, the probabilities of tile t+1 wait only for the P V of tile t-1
// (and for that of tile t only when O has to be rescaled), and with the two
// MMA streams issued by different warps a score product never waits behind a
// PV.  Every wait is bounded: a timeout sets
// MEDUSA_DEV_TIMEOUT, all roles stop, outstanding copies and MMAs are waited
// for and TMEM is freed before the kernel returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "host_util.h"
#include "sm100.cuh"

// Softmax threads per row of a two-head (packed) tile: 1 or 2.
#ifndef MEDUSA_ATTN_PACKED_SPLIT
#define MEDUSA_ATTN_PACKED_SPLIT 1
#endif

namespace medusa {
using namespace sm100;

namespace tc {

// Threads of a CTA: warps 0-3 (TMA, two MMA issuers, one idle) and SPLIT
// groups of four softmax warps.
__host__ __device__ constexpr int threads_for(int split) { return 128 + 128 * split; }
constexpr int kMaxSlots = 6;                            // ring of K or V half-tiles
constexpr uint32_t kHalf = 16384;                       // 128 rows x 128 bytes
constexpr uint32_t kBox = 8192;                         // 64 rows x 128 bytes
constexpr uint32_t kOffQ = 0;                           // 2 d-halves
constexpr uint32_t kOffRing = 2 * kHalf;                // slot = K or V of one tile (2 d-halves)
constexpr uint32_t kSlotBytes = 2 * kHalf;
// Ring slots: six with one softmax thread per row; five with two, whose
// exchange buffers take static shared memory a sixth slot would need.
__host__ __device__ constexpr int slots_for(int split) { return split == 2 ? 5 : kMaxSlots; }
__host__ __device__ constexpr uint32_t off_bar(int split) { return kOffRing + slots_for(split) * kSlotBytes; }
__host__ __device__ constexpr uint32_t smem_bytes(int split) {
  return off_bar(split) + 512 + 1024;  // barriers + alignment slack
}
constexpr uint32_t kTmemCols = 512;                     // S0, S1, O (128 each), P0, P1 (64 each)
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;                         // P buffer b at kColP + 64 b (bf16 pairs)
constexpr uint64_t kWaitNs = 1000000000ull;             // 1 s per wait
constexpr uint64_t kDrainNs = 100000000ull;             // 100 ms per drain wait
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);

struct Params {
  const uint32_t* mask;
  const int32_t* prefix_len;
  uint16_t* out;
  int32_t* d_status;
  int nl, B, N, Hq, Hkv, G, Lmax, W;
  int packed;    // two kv heads per tile
  int mtiles;    // row tiles per head group
  int groups;    // head groups per (layer, row)
  int items;
  int units;       // work units: the first full_items items whole, then each remaining item in `pieces` parts
  int full_items;
  int pieces;      // key-range pieces per remaining item (1: nothing is split)
  float* part_o;   // [piece][128 rows][128] fp32 unnormalised O of each piece
  float* part_ml;  // [piece][128 rows][2] fp32 row maximum (log2 domain) and row sum of each piece
  int KT;        // key positions per tile: 64 packed, 128 otherwise
  int out32;     // output base 32-byte aligned (32-byte stores)
  float scale_log2;
};

struct Bars {
  uint64_t full[kMaxSlots], empty[kMaxSlots];
  uint64_t q_full, q_empty, s_full[2], s_free[2], p_full[2], pv_done[2], o_free, drain, drain_pv;
  uint64_t mx[2][4];  // SPLIT = 2: partial row maxima of a tile exchanged (tile parity, lane quarter)
  uint64_t lx[4];     // SPLIT = 2: partial row sums of an item exchanged (lane quarter)
};

// Load sequence of one item of T key tiles: for j = 0 .. T + kLag - 1, K(j)
// (j < T) and then V(j - kLag) (j >= kLag).  The score products run ahead of
// the PVs, which wait for their tile's softmax, so each V tile is loaded about
// kLag tiles after its K and lands when its PV is due instead of holding a
// ring slot.  Both MMA issuers walk this sequence; half-tile c of the whole
// sequence (items back to back, 2T each) uses ring slot c % NS (NS slots).
constexpr int kLag = 2;
template <int NS>
__device__ __forceinline__ int slot_of(int c) { return c % NS; }
template <int NS>
__device__ __forceinline__ uint32_t use_parity(int c) { return (uint32_t)(c / NS) & 1u; }

struct Item {
  int lb, b, h0, mt, L, T, n_pre;
  bool ok;
};

// Every lane of the warp waits; the warp continues only if all lanes saw the
// phase complete (keeps warp-collective tcgen05 operations convergent).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort, kWaitNs);
  return __all_sync(0xffffffffu, ok);
}

// 2^x on the SFU (PTX ex2.approx, flush-to-zero): relative error ~2^-22,
// far below the bf16 rounding P receives next.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32-byte global store (8 x 32-bit), ptr 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(ptr), "r"(v[0]), "r"(v[1]), "r"(v[2]),
               "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ Item decode(const Params& p, int it) {
  Item x;
  x.mt = it % p.mtiles;
  int r = it / p.mtiles;
  const int grp = r % p.groups;
  x.lb = r / p.groups;
  x.b = x.lb % p.B;
  x.h0 = p.packed ? 2 * grp : grp;
  x.L = p.prefix_len[x.b];
  x.ok = x.L >= 0 && x.L <= p.Lmax;
  x.n_pre = x.ok ? (x.L + p.KT - 1) / p.KT : 0;
  x.T = x.n_pre + (p.N + p.KT - 1) / p.KT;
  return x;
}

// A work unit: a whole item (piece -1), or key tiles [t0, t1) of one of the
// items after the first full_items, whose partial result goes to slot `piece`.
struct Unit {
  Item x;
  int t0, t1, piece;
};

__device__ __forceinline__ Unit decode_unit(const Params& p, int u) {
  Unit w;
  if (u < p.full_items) {
    w.x = decode(p, u);
    w.t0 = 0;
    w.t1 = w.x.T;
    w.piece = -1;
  } else {
    const int v = u - p.full_items, s = v % p.pieces;
    w.x = decode(p, p.full_items + v / p.pieces);
    w.t0 = s * w.x.T / p.pieces;
    w.t1 = (s + 1) * w.x.T / p.pieces;
    w.piece = v;
  }
  return w;
}

// Output row of tile row m of an item: (node, query head) and whether it exists.
struct RowTarget {
  int node, h, gq;
  bool ok;
};
__device__ __forceinline__ RowTarget row_target(const Params& p, const Item& x, int m) {
  RowTarget r;
  int rr;
  if (p.packed) { rr = m & 63; r.h = x.h0 + (m >> 6); }
  else { rr = x.mt * 128 + m; r.h = x.h0; }
  r.node = rr / p.G;
  r.gq = rr % p.G;
  r.ok = r.node < p.N && r.h < p.Hkv;
  return r;
}

}  // namespace tc

template <bool PACKED, int SPLIT>
__global__ void __launch_bounds__(tc::threads_for(SPLIT), 1)
tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                    const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kt,
                    const __grid_constant__ CUtensorMap tm_vt, const tc::Params p) {
  using namespace tc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kSlots = slots_for(SPLIT);
  static_assert(sizeof(Bars) <= 512, "barrier area");
  Bars* bars = reinterpret_cast<Bars*>(smem + off_bar(SPLIT));
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  // SPLIT = 2: the two halves' partial row maxima (tile parity, half, row) and sums
  __shared__ float s_mx[SPLIT == 2 ? 2 : 1][SPLIT][SPLIT == 2 ? 128 : 1];
  __shared__ float s_l[SPLIT][SPLIT == 2 ? 128 : 1];
  constexpr int kSoft = 128 * SPLIT;  // softmax threads

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], kSoft);
      mbar_init(&bars->p_full[s], kSoft);
      mbar_init(&bars->pv_done[s], 1);
      for (int q = 0; q < 4; ++q) mbar_init(&bars->mx[s][q], 32 * SPLIT);
    }
    for (int q = 0; q < 4; ++q) mbar_init(&bars->lx[q], 32 * SPLIT);
    mbar_init(&bars->o_free, kSoft);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->drain_pv, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tm_q);
    tma_prefetch(&tm_kc);
    tma_prefetch(&tm_vc);
    tma_prefetch(&tm_kt);
    tma_prefetch(&tm_vt);
    // The prefix cache is not written during a step: while an earlier kernel
    // on the stream finishes, warm L2 with the first two K and V tiles of this
    // CTA's first item (rows 0 .. 2 KT of its cache, whatever its length; the
    // item's row and heads come from the launch alone).
    if ((int)blockIdx.x < p.units) {
      const int first_item = (int)blockIdx.x < p.full_items
                                 ? (int)blockIdx.x
                                 : p.full_items + ((int)blockIdx.x - p.full_items) / p.pieces;
      const int r = first_item / p.mtiles;
      const int lb = r / p.groups, h0 = p.packed ? 2 * (r % p.groups) : r % p.groups;
      for (int t = 0; t < 2; ++t)
        for (int kv = 0; kv < 2; ++kv)
          for (int dh = 0; dh < 2; ++dh)
            for (int cb = 0; cb < 2; ++cb)
              tma_prefetch_l2_4d(kv ? &tm_vc : &tm_kc, 64 * dh, PACKED ? h0 + cb : h0,
                                 PACKED ? t * p.KT : t * p.KT + 64 * cb, lb);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Nothing above reads memory an earlier kernel may write.
  pdl_wait();
  pdl_trigger();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int g = 0, n = 0, issued = 0;
      bool alive = true;
      for (int u = blockIdx.x; u < p.units && alive; u += gridDim.x) {
        const Unit w = decode_unit(p, u);
        const Item& x = w.x;
        if (!x.ok || w.t1 <= w.t0) continue;
        if (n > 0 && !(alive = mbar_wait_bounded(&bars->q_empty, (n - 1) & 1, &s_abort, kWaitNs))) break;
        ++n;  // Q loads of item n-1 (0-based) issued below
        mbar_expect_tx(&bars->q_full, 2 * kHalf);
        for (int dh = 0; dh < 2; ++dh) {
          if (PACKED) {
            for (int s = 0; s < 2; ++s)
              tma_load_5d(smem + kOffQ + dh * kHalf + s * kBox, &tm_q, &bars->q_full, 64 * dh, 0, x.h0 + s, 0, x.lb);
          } else {
            tma_load_5d(smem + kOffQ + dh * kHalf, &tm_q, &bars->q_full, 64 * dh, 0, x.h0, x.mt * (128 / p.G), x.lb);
          }
        }
        int c = 2 * g;  // half-tiles of earlier units: two per tile
        const int cnt = w.t1 - w.t0;
        for (int j = 0; j < cnt + kLag && alive; ++j) {
          for (int kv = 0; kv < 2 && alive; ++kv) {
            const int tt = kv ? j - kLag : j;  // K(j), then V(j - kLag), relative to t0
            if (tt < 0 || tt >= cnt) continue;
            const int t = w.t0 + tt;
            const bool tree = t >= x.n_pre;
            const int j0 = (tree ? t - x.n_pre : t) * p.KT;
            const int sl = slot_of<kSlots>(c);
            if (c >= kSlots &&
                !(alive = mbar_wait_bounded(&bars->empty[sl], use_parity<kSlots>(c - kSlots), &s_abort, kWaitNs)))
              break;
            const CUtensorMap* mp = kv ? (tree ? &tm_vt : &tm_vc) : (tree ? &tm_kt : &tm_kc);
            uint8_t* dst = smem + kOffRing + sl * kSlotBytes;
            mbar_expect_tx(&bars->full[sl], kSlotBytes);
            for (int dh = 0; dh < 2; ++dh)
              for (int cb = 0; cb < 2; ++cb)
                tma_load_4d(dst + dh * kHalf + cb * kBox, mp, &bars->full[sl], 64 * dh,
                            PACKED ? x.h0 + cb : x.h0, PACKED ? j0 : j0 + 64 * cb, x.lb);
            issued = ++c;
          }
        }
        g += cnt;
      }
      if (!alive) {
        // Drain: wait (bounded, regardless of the abort flag) for the last
        // phase issued on every load barrier, so no copy lands after exit.
        if (n > 0) mbar_wait_bounded(&bars->q_full, (n - 1) & 1, nullptr, kDrainNs);
        for (int c = issued - 1; c >= 0 && c >= issued - kSlots; --c)
          mbar_wait_bounded(&bars->full[slot_of<kSlots>(c)], use_parity<kSlots>(c), nullptr, kDrainNs);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues S = Q K^T for every key tile, warp 2 issues O += P V.  Each
    // lane 0 commits only its own MMAs, so the score products never queue
    // behind a PV that is waiting for its softmax, and the tensor pipe takes
    // both streams.  Both warps walk the same load sequence to find their slots.
    const bool s_role = warp == 1;
    int g = 0, n = 0;
    bool alive = true;
    for (int u = blockIdx.x; u < p.units && alive; u += gridDim.x) {
      const Unit w = decode_unit(p, u);
      const Item& x = w.x;
      if (!x.ok) {
        if (s_role && lane == 0 && x.mt == 0 && w.t0 == 0) set_status(p.d_status, MEDUSA_DEV_BAD_LENGTH);
        continue;
      }
      if (w.t1 <= w.t0) continue;
      const int cnt = w.t1 - w.t0;
      if (s_role) {
        if (!(alive = warp_wait(&bars->q_full, n & 1, &s_abort))) break;
        tc_fence_after();
      }
      const int g0 = g;
      int c = 2 * g0;  // next half-tile of the load sequence
      for (int j = 0; j < cnt + kLag && alive; ++j) {
        if (j < cnt) {
          const int gj = g0 + j, ck = c++, sb = gj & 1;
          if (s_role) {
            if (!(alive = warp_wait(&bars->full[slot_of<kSlots>(ck)], use_parity<kSlots>(ck), &s_abort))) break;
            if (gj >= 2 && !(alive = warp_wait(&bars->s_free[sb], ((gj >> 1) - 1) & 1, &s_abort))) break;
            tc_fence_after();
            if (lane == 0) {
              const uint32_t qa = smem_u32(smem + kOffQ);
              const uint32_t ka = smem_u32(smem + kOffRing + slot_of<kSlots>(ck) * kSlotBytes);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                mma_bf16(tmem + sb * 128, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024),
                         kIdescQK, kk > 0);
              }
              // Releases first: the arrive a consumer waits for comes last.
              mma_commit(&bars->empty[slot_of<kSlots>(ck)]);
              if (j == cnt - 1) mma_commit(&bars->q_empty);
              mma_commit(&bars->s_full[sb]);
            }
            __syncwarp();
          }
        }
        if (j >= kLag) {
          const int tt = j - kLag, t = w.t0 + tt, gt = g0 + tt, cv = c++;
          if (!s_role) {
            if (tt == 0 && n > 0 && !(alive = warp_wait(&bars->o_free, (n - 1) & 1, &s_abort))) break;
            if (!(alive = warp_wait(&bars->p_full[gt & 1], (gt >> 1) & 1, &s_abort))) break;
            if (!(alive = warp_wait(&bars->full[slot_of<kSlots>(cv)], use_parity<kSlots>(cv), &s_abort))) break;
            uint8_t* vb = smem + kOffRing + slot_of<kSlots>(cv) * kSlotBytes;
            // The last prefix tile may run past prefix_len: zero those V rows
            // (stale cache rows may hold anything, and 0 * NaN is NaN).
            const int j0 = t * p.KT;
            if (t < x.n_pre && j0 + p.KT > x.L) {
              const int first = x.L - j0;  // first invalid key offset within a column block / tile
              for (int idx = lane; idx < 2 * 128 * 8; idx += 32) {
                const int dh = idx >> 10, r = (idx >> 3) & 127, cc = idx & 7;
                const int off = PACKED ? (r & 63) : r;
                if (off >= first)
                  *reinterpret_cast<uint4*>(vb + dh * kHalf + r * 128 + cc * 16) = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
              const uint32_t pa = tmem + kColP + 64 * (gt & 1);
              const uint32_t va = smem_u32(vb);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                mma_bf16_ts(tmem + kColO, pa + 8 * kk, smem_desc_sw128(va + kk * 2048, kHalf, 1024), kIdescPV,
                            (kk > 0 || tt > 0) ? 1u : 0u);
              }
              mma_commit(&bars->empty[slot_of<kSlots>(cv)]);
              mma_commit(&bars->pv_done[gt & 1]);
            }
            __syncwarp();
          }
        }
      }
      g = g0 + cnt;
      ++n;
    }
    if (lane == 0) {
      // Wait (bounded) for this warp's own MMAs and the arrives they signal
      // before TMEM is released and the CTA's shared memory goes away.
      uint64_t* d = s_role ? &bars->drain : &bars->drain_pv;
      mma_commit(d);
      mbar_wait_bounded(d, 0, nullptr, kDrainNs);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / epilogue
    // Softmax warp sw: lane quarter q4 (rows 32 q4 .. 32 q4 + 31 of the tile)
    // and half `half` of each row's scores, P columns and O columns.
    const int sw = warp - 4, q4 = sw & 3, half = sw >> 2;
    const int m = 32 * q4 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * q4) << 16);
    const int slot = PACKED ? (m >> 6) : 0;             // warp-uniform
    constexpr int NC = (PACKED ? 64 : 128) / SPLIT;     // score columns per thread
    constexpr int OC = 128 / SPLIT;                     // O / output columns per thread
    const int koff = NC * half;                         // first key of this thread within the tile's keys
    const int scol = (PACKED ? 64 * slot : 0) + koff;   // its first S column (and 2 x its first P column)
    // Packed tiles: each row's P columns outside its own head block stay zero.
    if (PACKED && half == 0) {
      uint32_t z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0u;
      for (int b = 0; b < 2; ++b) tmem_st32u(lane_addr + kColP + 64 * b + 32 * (1 - slot), z);
      tmem_wait_st();
    }
    int g = 0, nf = 0;
    bool alive = true;
    // The epilogue of an item (O / l -> bf16 output row, after the item's last
    // PV) runs, for two-head tiles, inside the next item's first tile after
    // that tile's P is published, so the wait for the last PV overlaps the
    // next item's first score product and softmax (the next item's first PV
    // waits for o_free).
    bool pend = false, pend_ok = false;
    uint16_t* pend_row = nullptr;
    float pend_l = 0.f, pend_m = 0.f;
    int pend_g = 0, pend_piece = -1;
    auto finish = [&]() -> bool {
      float l = pend_l;
      if constexpr (SPLIT == 2) {
        // the row sum is the two halves' partial sums (same maximum, same scale)
        s_l[half][m] = pend_l;
        mbar_arrive(&bars->lx[q4]);
        if (!warp_wait(&bars->lx[q4], nf & 1, &s_abort)) return false;
        l = s_l[0][m] + s_l[1][m];
      }
      ++nf;
      if (!warp_wait(&bars->pv_done[pend_g & 1], (pend_g >> 1) & 1, &s_abort)) return false;
      tc_fence_after();
      // A piece of an item leaves its unnormalised O, row maximum and row sum
      // for the merge kernel; a whole item writes O / l.
      float* part = pend_piece >= 0 ? p.part_o + ((size_t)pend_piece * 128 + m) * 128 : nullptr;
      if (pend_piece >= 0 && half == 0)
        *reinterpret_cast<float2*>(p.part_ml + ((size_t)pend_piece * 128 + m) * 2) = make_float2(pend_m, l);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // O in chunks of EC columns (one TMEM wait per chunk; 128-row tiles use
      // narrower chunks, their softmax already holds most registers).
      constexpr int EC = (PACKED ? 64 : 32) < OC ? (PACKED ? 64 : 32) : OC;
#pragma unroll
      for (int h2 = 0; h2 < OC / EC; ++h2) {
        float o[EC];
#pragma unroll
        for (int q = 0; q < EC / 32; ++q) tmem_ld32(lane_addr + kColO + OC * half + EC * h2 + 32 * q, o + 32 * q);
        tmem_wait_ld();
        if (part) {
          float4* dst = reinterpret_cast<float4*>(part + OC * half + EC * h2);
#pragma unroll
          for (int q = 0; q < EC / 4; ++q) dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        } else if (pend_ok) {
          uint32_t w[EC / 2];
#pragma unroll
          for (int e = 0; e < EC / 2; ++e) w[e] = pack_bf16x2(o[2 * e] * inv, o[2 * e + 1] * inv);
          uint16_t* dst = pend_row + OC * half + EC * h2;
          if (p.out32) {
#pragma unroll
            for (int q = 0; q < EC / 16; ++q) st_global_v8(dst + 16 * q, w + 8 * q);
          } else {
#pragma unroll
            for (int q = 0; q < EC / 8; ++q)
              *reinterpret_cast<uint4*>(dst + 8 * q) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free);
      pend = false;
      return true;
    };
    for (int u = blockIdx.x; u < p.units && alive; u += gridDim.x) {
      const Unit w = decode_unit(p, u);
      const Item& x = w.x;
      if (!x.ok) continue;
      if (w.t1 <= w.t0) {
        // an empty piece (an item with fewer key tiles than pieces): no keys
        if (half == 0)
          *reinterpret_cast<float2*>(p.part_ml + ((size_t)w.piece * 128 + m) * 2) = make_float2(-INFINITY, 0.f);
        continue;
      }
      // This thread's query row.
      int r, h;
      if (PACKED) { r = m & 63; h = x.h0 + slot; }
      else { r = x.mt * 128 + m; h = x.h0; }
      const int node = r / p.G, gq = r % p.G;
      const bool row_ok = node < p.N && h < p.Hkv;
      // The ancestor-mask words of this thread's keys in the tree key tiles
      // (one tile for two-head tiles: N <= 64 keys of 64; two otherwise:
      // N <= 256 keys of 128), loaded when the unit starts.  Loaded at the
      // tree tile itself, they waited an L2 round trip under the cache stream
      // (a tree tile's mask step measured ~5700 cycles against ~100 for a
      // prefix tile).  Keys at or past N are cleared here.
      constexpr int kTT = PACKED ? 1 : 2;
      constexpr int MW = NC / 32;
      uint32_t tmw[kTT][MW];
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt) {
#pragma unroll
        for (int wv = 0; wv < MW; ++wv) {
          const int j = tt * p.KT + koff + 32 * wv;  // first key of the word (a multiple of 32)
          uint32_t mk = (row_ok && j < p.N) ? __ldg(p.mask + (size_t)node * p.W + (j >> 5)) : 0u;
          const int lim = p.N - j;
          if (lim < 32) mk &= lim <= 0 ? 0u : ((1u << lim) - 1u);
          tmw[tt][wv] = mk;
        }
      }
      float m_used = -INFINITY, l = 0.f;
      for (int t = w.t0; t < w.t1; ++t, ++g) {
        const int sb = g & 1;
        if (!(alive = warp_wait(&bars->s_full[sb], (g >> 1) & 1, &s_abort))) break;
        tc_fence_after();
        float s[NC];
#pragma unroll
        for (int q = 0; q < NC / 32; ++q) tmem_ld32(lane_addr + sb * 128 + scol + 32 * q, s + 32 * q);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_free[sb]);

        const bool tree = t >= x.n_pre;
        const int j0 = (tree ? t - x.n_pre : t) * p.KT + koff;  // key of s[0]
        const float sc = p.scale_log2;
        // Raw-score maximum over the visible keys (scale > 0 keeps the order),
        // in four independent chains.
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (!tree && j0 + NC <= x.L && row_ok) {
          // keys entirely inside the prefix: every one is visible
#pragma unroll
          for (int c = 0; c < NC; ++c) m4[c & 3] = fmaxf(m4[c & 3], s[c]);
        } else if (tree) {
          // ancestors only (the words above; tree tile t - n_pre < kTT)
          const bool second = kTT > 1 && t - x.n_pre > 0;
          uint32_t mw[MW];
#pragma unroll
          for (int wv = 0; wv < MW; ++wv) mw[wv] = second ? tmw[kTT - 1][wv] : tmw[0][wv];
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            s[c] = ((mw[c >> 5] >> (c & 31)) & 1u) ? s[c] : -INFINITY;
            m4[c & 3] = fmaxf(m4[c & 3], s[c]);
          }
        } else {
          // the last prefix tile, partly past prefix_len (or a row that does not exist)
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            s[c] = (row_ok && j0 + c < x.L) ? s[c] : -INFINITY;
            m4[c & 3] = fmaxf(m4[c & 3], s[c]);
          }
        }
        float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        if constexpr (SPLIT == 2) {
          // both halves of the row continue with the maximum over all its keys
          s_mx[sb][half][m] = mx;
          mbar_arrive(&bars->mx[sb][q4]);
          if (!(alive = warp_wait(&bars->mx[sb][q4], (g >> 1) & 1, &s_abort))) break;
          mx = fmaxf(s_mx[sb][0][m], s_mx[sb][1][m]);
        }
        const float m_new = fmaxf(m_used, mx * sc);  // log2 domain
        const bool need = m_new > m_used + 8.f;
        const float f = need ? fast_exp2(m_used - m_new) : 1.f;  // 0 when m_used = -inf
        if (need) m_used = m_new;
        // Probabilities first (overlaps the previous tile's PV), packed to bf16.
        // exp2(-inf) = 0 covers the masked keys.  m_used is -inf only when
        // every score so far (this tile's included) is masked: the offset is
        // then 0, so each exp2 sees -inf and gives 0.
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[NC / 2];
        const float neg = m_used == -INFINITY ? 0.f : -m_used;
#pragma unroll
        for (int c = 0; c < NC; c += 2) {
          const float a = fast_exp2(fmaf(s[c], sc, neg));
          const float b2 = fast_exp2(fmaf(s[c + 1], sc, neg));
          rs4[(c >> 1) & 3] += a + b2;
          pk[c >> 1] = pack_bf16x2(a, b2);
        }
        const float rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        l = l * f + rs;
        if (t > w.t0 && __any_sync(0xffffffffu, need)) {
          // O is rescaled only after the previous tile's PV has landed in it.
          const int gp = g - 1;
          if (!(alive = warp_wait(&bars->pv_done[gp & 1], (gp >> 1) & 1, &s_abort))) break;
          tc_fence_after();
          float o[32];
#pragma unroll
          for (int c4 = 0; c4 < OC / 32; ++c4) {
            tmem_ld32(lane_addr + kColO + OC * half + 32 * c4, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= f;
            tmem_st32(lane_addr + kColO + OC * half + 32 * c4, o);
          }
        }
        // P buffer g & 1 is free once the PV of tile g - 2 has read it.
        const int pb = g & 1;
        if (g >= 2) {
          if (!(alive = warp_wait(&bars->pv_done[pb], ((g - 2) >> 1) & 1, &s_abort))) break;
          tc_fence_after();
        }
        const uint32_t pa = lane_addr + kColP + 64 * pb + (scol >> 1);
        if constexpr (NC / 2 == 16) {
          tmem_st16u(pa, pk);
        } else {
#pragma unroll
          for (int q = 0; q < NC / 64; ++q) tmem_st32u(pa + 32 * q, pk + 32 * q);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[pb]);
        // The previous item's epilogue (its PV(0) waits for O to be read out).
        if constexpr (PACKED) {
          if (t == w.t0 && pend && !(alive = finish())) break;
        }
      }
      if (!alive) break;
      pend = true;
      pend_ok = row_ok;
      pend_row = p.out + ((((size_t)x.lb * p.N + (row_ok ? node : 0)) * p.Hq) + (size_t)h * p.G + gq) * 128;
      pend_l = l;
      pend_m = m_used;
      pend_piece = w.piece;
      pend_g = g - 1;
      // 128-row tiles keep every score register live inside the tile loop:
      // their epilogue runs here, right after the item.
      if constexpr (!PACKED) {
        if (!(alive = finish())) break;
      }
    }
    if (alive && pend) alive = finish();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // After the barrier: any role's timeout (even one raised after another role
  // finished) is visible here.
  if (threadIdx.x == 0 && s_abort) set_status(p.d_status, MEDUSA_DEV_TIMEOUT);
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Merges the pieces of every split item: for each of its rows, the pieces'
// (O, m, l) combine as in the online softmax, O = sum_s 2^(m_s - M) O_s and
// l = sum_s 2^(m_s - M) l_s with M = max_s m_s, and the row is written as
// O / l.  One warp per (split item, row): the lanes share the pieces for M and
// l, then every lane adds its 4 columns of each piece's O (loads independent
// of one another, several in flight).  Grid: split items x 16, 8 warps each.
__global__ void __launch_bounds__(256) tree_attn_merge_kernel(const tc::Params p) {
  using namespace tc;
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + warp;
  const int v = gw >> 7, m = gw & 127;  // split item (0-based after the whole ones), tile row
  if (v >= p.items - p.full_items) return;
  const Item x = decode(p, p.full_items + v);
  if (!x.ok) return;
  const RowTarget rt = row_target(p, x, m);
  if (!rt.ok) return;
  const size_t base = (size_t)v * p.pieces;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  float M = -INFINITY;
  for (int s = lane; s < p.pieces; s += 32) {
    const float2 q = ml[(base + s) * 128 + m];
    if (q.y > 0.f) M = fmaxf(M, q.x);
  }
  M = warp_max(M);
  float l = 0.f;
  for (int s = lane; s < p.pieces; s += 32) {
    const float2 q = ml[(base + s) * 128 + m];
    if (q.y > 0.f) l = fmaf(fast_exp2(q.x - M), q.y, l);
  }
  l = warp_sum(l);
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = 0; s < p.pieces; ++s) {
    const size_t slot = (base + s) * 128 + m;
    const float2 q = ml[slot];
    const float4 po = reinterpret_cast<const float4*>(p.part_o + slot * 128)[lane];
    const float wgt = q.y > 0.f ? fast_exp2(q.x - M) : 0.f;  // a piece with no visible key adds nothing
    o.x = fmaf(wgt, po.x, o.x);
    o.y = fmaf(wgt, po.y, o.y);
    o.z = fmaf(wgt, po.z, o.z);
    o.w = fmaf(wgt, po.w, o.w);
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  uint16_t* dst = p.out + ((((size_t)x.lb * p.N + rt.node) * p.Hq) + (size_t)rt.h * p.G + rt.gq) * 128 + 4 * lane;
  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(o.x * inv, o.y * inv), pack_bf16x2(o.z * inv, o.w * inv));
}

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

static bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                     const cuuint32_t* box) {
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// How the items are divided.  When there are fewer than half as many items as
// SMs (few layers x rows x heads with long prefixes), each item is split into
// `pieces` key ranges so that (nearly) every SM streams part of the cache; a
// split needs at least two pieces per item and two key tiles per piece at the
// cache capacity.  Otherwise every item runs whole: with a round or more of
// items the cache stream already keeps HBM near its peak, and splitting the
// last round only adds partial traffic and a merge (measured slower on the
// Vicuna-7B step: 121 us instead of 101 us for the call).  The general form
// below (whole items in full rounds, then the last round's items split) is
// kept, with full rounds absent whenever a split happens.
struct AttnPlan {
  int items, full_items, pieces, units, grid;
  bool packed;
  size_t ws_bytes;
};
static AttnPlan attn_plan(int n_layers, int B, int N, int Hq, int Hkv, int Lmax, int sms) {
  AttnPlan a{};
  const int G = Hq / Hkv;
  a.packed = N * G <= 64;
  const int KT = a.packed ? 64 : 128;
  const int mtiles = a.packed ? 1 : (N * G + 127) / 128;
  const int groups = a.packed ? (Hkv + 1) / 2 : Hkv;
  a.items = n_layers * B * groups * mtiles;
  const int rem = 2 * a.items <= sms ? a.items : 0;
  const int max_tiles = (Lmax + KT - 1) / KT + (N + KT - 1) / KT;
  int pieces = rem > 0 ? sms / rem : 1;
  if (pieces > max_tiles / 2) pieces = max_tiles / 2;
  if (pieces >= 2) {
    a.pieces = pieces;
    a.full_items = a.items - rem;
    a.units = a.full_items + rem * pieces;
    a.grid = a.units < sms ? a.units : sms;
    a.ws_bytes = (size_t)rem * pieces * 128 * (128 + 2) * sizeof(float);
  } else {
    // Equal-cost items: as many rounds as the SM count forces, then spread
    // the items evenly over just enough CTAs (no ragged last round).
    a.pieces = 1;
    a.full_items = a.items;
    a.units = a.items;
    const int rounds = (a.items + sms - 1) / sms;
    a.grid = (a.items + rounds - 1) / rounds;
    a.ws_bytes = 0;
  }
  return a;
}

bool tree_attention_tc_supported(int N, int Hq, int Hkv, int d, int Lmax, const void* q, const void* kc,
                                 const void* vc, const void* kt, const void* vt, const void* out) {
  if (d != 128 || Hkv < 1 || Hq % Hkv || N < 1 || N > MEDUSA_MAX_NODES || Lmax < 1) return false;
  const int G = Hq / Hkv;
  if (G > 128 || 128 % G) return false;
  if (!aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(kt) || !aligned16(vt) || !aligned16(out))
    return false;
  return encode_fn() != nullptr;
}

size_t tree_attention_tc_ws_bytes(int n_layers, int B, int N, int Hq, int Hkv, int, int Lmax) {
  return attn_plan(n_layers, B, N, Hq, Hkv, Lmax, device_sm_count()).ws_bytes;
}

medusa_status tree_attention_tc(const void* q, const void* kc, const void* vc, const void* kt, const void* vt,
                                const uint32_t* mask, const int32_t* prefix_len, int n_layers, int B, int N,
                                int Hq, int Hkv, int d, int Lmax, float scale, void* out, void* ws, size_t ws_bytes,
                                int32_t* d_status, cudaStream_t s) {
  (void)d;
  const int G = Hq / Hkv;
  const AttnPlan plan = attn_plan(n_layers, B, N, Hq, Hkv, Lmax, device_sm_count());
  if (plan.ws_bytes && (!ws || ws_bytes < plan.ws_bytes || !aligned16(ws))) return MEDUSA_ERR_WORKSPACE;
  tc::Params p;
  p.mask = mask;
  p.prefix_len = prefix_len;
  p.out = static_cast<uint16_t*>(out);
  p.d_status = d_status;
  p.nl = n_layers;
  p.B = B;
  p.N = N;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.Lmax = Lmax;
  p.W = (N + 31) / 32;
  p.packed = N * G <= 64 ? 1 : 0;
  p.out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
  p.KT = p.packed ? 64 : 128;
  p.mtiles = p.packed ? 1 : (N * G + 127) / 128;
  p.groups = p.packed ? (Hkv + 1) / 2 : Hkv;
  p.items = n_layers * B * p.groups * p.mtiles;
  p.units = plan.units;
  p.full_items = plan.full_items;
  p.pieces = plan.pieces;
  p.part_o = plan.ws_bytes ? static_cast<float*>(ws) : nullptr;
  p.part_ml = plan.ws_bytes ? p.part_o + (size_t)(plan.items - plan.full_items) * plan.pieces * 128 * 128 : nullptr;
  p.scale_log2 = scale * 1.4426950408889634f;
  const cuuint64_t LB = (cuuint64_t)n_layers * B;
  const cuuint64_t es = 2;
  CUtensorMap mq, mkc, mvc, mkt, mvt;
  {
    const int rows = p.packed ? 64 : 128;
    cuuint64_t dims[5] = {128, (cuuint64_t)G, (cuuint64_t)Hkv, (cuuint64_t)N, LB};
    cuuint64_t str[4] = {128 * es, (cuuint64_t)G * 128 * es, (cuuint64_t)Hq * 128 * es,
                         (cuuint64_t)N * Hq * 128 * es};
    cuuint32_t box[5] = {64, (cuuint32_t)G, 1, (cuuint32_t)(rows / G), 1};
    if (!make_map(&mq, q, 5, dims, str, box)) return MEDUSA_ERR_CUDA;
  }
  {
    cuuint64_t dims[4] = {128, (cuuint64_t)Hkv, (cuuint64_t)Lmax, LB};
    cuuint64_t str[3] = {128 * es, (cuuint64_t)Hkv * 128 * es, (cuuint64_t)Lmax * Hkv * 128 * es};
    cuuint32_t box[4] = {64, 1, 64, 1};
    if (!make_map(&mkc, kc, 4, dims, str, box) || !make_map(&mvc, vc, 4, dims, str, box)) return MEDUSA_ERR_CUDA;
  }
  {
    cuuint64_t dims[4] = {128, (cuuint64_t)Hkv, (cuuint64_t)N, LB};
    cuuint64_t str[3] = {128 * es, (cuuint64_t)Hkv * 128 * es, (cuuint64_t)N * Hkv * 128 * es};
    cuuint32_t box[4] = {64, 1, 64, 1};
    if (!make_map(&mkt, kt, 4, dims, str, box) || !make_map(&mvt, vt, 4, dims, str, box)) return MEDUSA_ERR_CUDA;
  }
  // 128-row tiles (trees above 64 nodes, GQA groups) split every row over two
  // softmax threads; two-head tiles keep one thread per row.
  constexpr int kSplitPacked = MEDUSA_ATTN_PACKED_SPLIT;
  auto kern = p.packed ? tree_attn_tc_kernel<true, kSplitPacked> : tree_attn_tc_kernel<false, 2>;
  const int threads = tc::threads_for(p.packed ? kSplitPacked : 2);
  const uint32_t smem = tc::smem_bytes(p.packed ? kSplitPacked : 2);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MEDUSA_ERR_CUDA;
  launch_pdl(kern, dim3(plan.grid), dim3(threads), smem, s, mq, mkc, mvc, mkt, mvt, p);
  if (plan.pieces > 1)
    launch_pdl(tree_attn_merge_kernel, dim3((plan.items - plan.full_items) * 16), dim3(256), 0, s, p);
  return launch_status();
}

}  // namespace medusa
