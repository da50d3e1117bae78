// Host-side tensor-map encoding (cuTensorMapEncodeTiled through the runtime's
// driver entry point, so the library does not link libcuda directly).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace rpa {

// Encodes a rank-3 tiled map over a row-major array [dim2][dim1][dim0] of
// `elem_bytes`-byte elements (bf16 or raw bytes).  Returns false if the
// driver refuses the map (misaligned base or strides, bad box).
bool encode_map_3d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t dim0,
                   uint64_t dim1, uint64_t dim2, uint32_t box0, uint32_t box1, uint32_t box2,
                   bool swizzle128);

// Sets the dynamic shared-memory limit of `func` once per device.
cudaError_t ensure_smem_attr(const void* func, int bytes, std::atomic<unsigned long long>* done_mask);

}  // namespace rpa
