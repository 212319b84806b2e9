// Host-side helpers shared by the entry points of libmedusa_gb300.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "medusa.h"

namespace medusa {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

inline size_t dtype_bytes(medusa_dtype dt) { return dt == MEDUSA_BF16 ? 2 : 4; }
inline bool dtype_ok(int dt) { return dt == MEDUSA_F32 || dt == MEDUSA_BF16; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bump allocator over a caller-provided workspace (256-byte aligned slices).
struct WsCarver {
  char* base;
  size_t used = 0;
  explicit WsCarver(void* p) : base(static_cast<char*>(p)) {}
  template <typename T>
  T* take(size_t count) {
    used = align_up(used, 256);
    T* p = base ? reinterpret_cast<T*>(base + used) : nullptr;
    used += count * sizeof(T);
    return p;
  }
};

// Launches `kern` with programmatic stream serialization (the kernel may be
// scheduled before the previous kernel on the stream has finished; its
// pdl_wait() orders its memory accesses).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

inline medusa_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? MEDUSA_OK : MEDUSA_ERR_CUDA;
}

constexpr int kNumSMsFallback = 152;  // GB300: 2 dies x 76 SMs
int device_sm_count();                 // SMs of the current device (cached per device)

}  // namespace medusa
