// ciera_rans.h -- sizes of the RANS kernels' buffers and their launchers
// (ciera_rans.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>

#include "ciera_internal.h"

namespace ciera {

// uint16 words per lane region of a block's coding scratch: the final state
// and at most one renormalisation word per symbol, rounded up to 2 mod 4 so
// that the lanes' regions start in 32 different shared-memory banks.
__host__ __device__ inline int64_t rans_lane_words(int64_t B) {
  const int64_t need = 2 + (B + kRansLanes - 1) / kRansLanes;
  return need + ((2 - need) & 3);
}
// Bytes of one block's coding buffer: 32 uint16 lane word counts, their
// 33 uint16 exclusive prefixes (padded to 80 bytes), then 32 lane regions
// of rans_lane_words(B) uint16 each.
constexpr int64_t kRansBufHead = 64 + 80;
__host__ __device__ inline int64_t rans_block_bytes(int64_t B) {
  return kRansBufHead + 2 * kRansLanes * rans_lane_words(B);
}

// Per-rank coder tables in the workspace.
//   encoder: 256 entries of 4 uint32 (division constants, renormalisation
//            bound, complement, cumulative frequency), then the 256 uint16
//            frequencies
//   decoder: 4096 uint32 slot entries (symbol, frequency, slot bias)
constexpr int64_t kRansEncTableBytes = 256 * 16 + 256 * 2;
constexpr int64_t kRansDecTableBytes = 4096 * 4;

// Dynamic shared memory of the RANS tile kernels for tiles of T blocks of B.
//   sender:   meta, the tile's exponents (T*B), one coding buffer per block
//   receiver: meta, the tile's sign+mantissa bytes (T*B), its records when
//             they fit in T*B/2 bytes (about 0.4 bytes per value at
//             B = 4096; larger ones are decoded from global memory), and the
//             rank's 16 KB slot table.  Raw tiles stream from global memory
//             and stage nothing.
constexpr int64_t kRansEncMeta = 6144;  // coder table, histogram, sizes (ciera_rans.cu)
constexpr int64_t kRansDecMeta = 1024;  // offsets
__host__ __device__ inline int64_t rans_compress_smem(int64_t T, int64_t B) {
  return kRansEncMeta + T * B + T * rans_block_bytes(B);
}
__host__ __device__ inline int64_t rans_record_stage(int64_t T, int64_t B) { return T * B / 2; }
__host__ __device__ inline int64_t rans_decompress_smem(int64_t T, int64_t B) {
  return kRansDecMeta + T * B + ((rans_record_stage(T, B) + 15) & ~int64_t(15)) +
         kRansDecTableBytes;
}
// Threads of a receiver CTA: four warps, each decoding one changed block at
// a time.
__host__ __device__ inline int rans_decompress_threads(int64_t) { return 128; }
// Blocks per receiver tile for sender tiles of T blocks.  A payload
// addresses its records per block, so the receiver may cut the shard into
// tiles of its own: twice the sender's (at most 32) keeps all four warps
// decoding on shards whose blocks all changed and loads the 16 KB slot
// table once per four blocks instead of two.
__host__ __device__ inline int64_t rans_receiver_blocks(int64_t T) {
  return 2 * T > 32 ? 32 : 2 * T;
}

// Launchers (ciera_rans.cu), returning a cudaError_t value.
//   launch_compress_rans: the RANS sender; hist_prev/hist_out hold 256
//     uint32 per rank of the range (hist_out zeroed by the caller),
//     enc_tables kRansEncTableBytes per rank of the range.
//   launch_decompress_rans: the RANS part of the receiver, after the bitmap
//     scan; dec_tables kRansDecTableBytes per rank.  p.geo is the plan's
//     (the sender's) geometry; the launch re-tiles it to
//     rans_receiver_blocks(p.geo.T) blocks per tile.
int launch_compress_rans(const CompressParams& p, const uint32_t* hist_prev, uint32_t* hist_out,
                         uint8_t* enc_tables, void* stream);
int launch_decompress_rans(const DecompressParams& p, uint32_t* dec_tables, void* stream);

}  // namespace ciera
