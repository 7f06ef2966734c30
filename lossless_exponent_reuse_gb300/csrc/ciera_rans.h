// ciera_rans.h -- sizes of the RANS kernels' buffers and their launchers
// (ciera_rans.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>

#include "ciera_internal.h"

namespace ciera {

// uint16 words per lane region of a block's coding scratch: the final state
// and at most one renormalisation word per symbol, rounded to 16 bytes.
__host__ __device__ inline int64_t rans_lane_words(int64_t B) {
  return (2 + (B + kRansLanes - 1) / kRansLanes + 7) & ~int64_t(7);
}
// Bytes of one block's coding scratch / record buffer: 32 uint16 lane
// counts, then 32 lane regions (the record is compacted in place).
__host__ __device__ inline int64_t rans_block_bytes(int64_t B) {
  return 2 * (kRansLanes + kRansLanes * rans_lane_words(B));
}

// Dynamic shared memory of the RANS kernels for tiles of T blocks of B.
constexpr int64_t kRansMetaBytes = 8192;  // tables, counters (see ciera_rans.cu)
__host__ __device__ inline int64_t rans_compress_smem(int64_t T, int64_t B) {
  return kRansMetaBytes + 3 * T * B + T * rans_block_bytes(B);
}
__host__ __device__ inline int64_t rans_decompress_smem(int64_t T, int64_t B) {
  return kRansMetaBytes + 4 * T * B + T * rans_block_bytes(B);
}

// Launchers (ciera_rans.cu), returning a cudaError_t value: the RANS sender
// (hist_prev/hist_out: 256 uint32 per rank of the range) and the RANS part
// of the receiver.
int launch_compress_rans(const CompressParams& p, const uint32_t* hist_prev, uint32_t* hist_out,
                         void* stream);
int launch_decompress_rans(const DecompressParams& p, void* stream);

}  // namespace ciera
