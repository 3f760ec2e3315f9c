// Host-side creation of TMA tensor maps (bf16, tiled, 128-byte swizzle).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moda {

// Encodes a rank-`rank` bf16 tensor map over `base` with dims[0] innermost,
// byte strides of dims 1..rank-1 in strides_bytes, and box sizes `box`.
// Out-of-range elements of a box read as zero. Returns CUDA_SUCCESS or the
// driver's error.
// l2_promotion_bytes: 256 (the default) or 128, the granule L2 fetches for a
// box row; 128 when a box row is 128 bytes whose neighbours are not read
// together with it.
CUresult encode_bf16_sw128(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box,
                           int l2_promotion_bytes = 256);

// Same, without swizzle: boxes land in shared memory as plain row-major
// arrays (the inner box extent must be a multiple of 16 bytes).
CUresult encode_bf16_plain(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace moda
