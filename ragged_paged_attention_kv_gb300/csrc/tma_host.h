// Host-side tensor-map encoding (cuTensorMapEncodeTiled through the runtime's
// driver entry point, so the library does not link libcuda directly).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <utility>

namespace rpa {

// Encodes a rank-3 tiled map over a row-major array [dim2][dim1][dim0] of
// `elem_bytes`-byte elements (bf16 or raw bytes).  Returns false if the
// driver refuses the map (misaligned base or strides, bad box).
bool encode_map_3d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t dim0,
                   uint64_t dim1, uint64_t dim2, uint32_t box0, uint32_t box1, uint32_t box2,
                   bool swizzle128);
// The same with a chosen swizzle: 0 (none), 64 or 128 bytes.
bool encode_map_3d_swizzle(CUtensorMap* map, const void* base, int elem_bytes, uint64_t dim0,
                           uint64_t dim1, uint64_t dim2, uint32_t box0, uint32_t box1,
                           uint32_t box2, int swizzle_bytes);

// Sets the dynamic shared-memory limit of `func` once per device.
cudaError_t ensure_smem_attr(const void* func, int bytes, std::atomic<unsigned long long>* done_mask);

// Launches `kern` on `stream` as a programmatic dependent of the kernel
// before it (cudaLaunchAttributeProgrammaticStreamSerialization): the launch
// may begin while that kernel still runs, and the kernel must call
// griddep_wait() before it touches anything the earlier kernel writes.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), int grid, int threads, int smem_bytes,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace rpa
