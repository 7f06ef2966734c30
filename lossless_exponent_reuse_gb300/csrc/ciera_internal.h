// ciera_internal.h -- launch parameters shared by the host API and the kernels
// of libciera.  Not part of the public ABI.
#pragma once

#include <cstdint>

#include "ciera.h"

namespace ciera {

constexpr int kThreads = 128;             // threads per CTA of the tile kernels
constexpr int kScanThreads = 256;         // threads per CTA of the bitmap scan
#ifndef CIERA_TILE_ELEMS
#define CIERA_TILE_ELEMS 8192
#endif
constexpr int64_t kTileElems = CIERA_TILE_ELEMS;  // target values per tile (T*B)
constexpr int kMaxTileBlocks = static_cast<int>(kTileElems);  // T <= kTileElems (B = 1)
constexpr int kMaxTileWords = kMaxTileBlocks / 32;
constexpr int64_t kFastMinBlock = 256;    // fast path: T <= 32 blocks per tile
constexpr int64_t kFastMaxBlock = 16384;  // fast path: <= 64 KB of staging per CTA
constexpr int64_t kMaxNumel = int64_t(1) << 40;
constexpr int64_t kMaxShardBlocks = int64_t(1) << 30;  // fits the 30-bit prefix field

// Workspace control block at offset 0.
struct Control {
  // compress: (launch number << 32) | tickets drawn in the current launch;
  // the last ticket resets the count and advances the launch number
  unsigned long long ticket;
  uint32_t status;   // kStatus* bits, read and cleared by ciera_status
  uint32_t pad[61];
};
enum : uint32_t {
  kStatusCorrupt = 1u,
  kStatusTimeout = 2u,
  kStatusInternal = 4u,
  kStatusBounds = 8u,  // checked builds: an access outside its buffer was skipped
};

// Decoupled look-back status word of one tile (and, beside it, an
// epoch-tagged word with the tile's flag bits):
//   bits 63..32 the launch's tag (launch number + 1, never 0), bits 31..30
//   state, bits 29..0 count of
//   changed blocks (aggregate of the tile, or inclusive prefix in its shard).
enum : uint32_t { kStateAggregate = 1u, kStateInclusive = 2u };

// Per-shard outcome of a compress launch (result word: launch tag << 32 |
// these bits), read by k_repack after the launch.
enum : uint32_t {
  kResultRepack = 1u,  // raw-ahead shard that is not raw: rewrite it compacted
  kResultRaw = 2u,     // the shard's payload is RAW (the next call predicts raw)
};

// Receiver per-rank state written by the bitmap scan.
enum : uint32_t { kRankSkip = 0u, kRankCompressed = 1u, kRankRaw = 2u, kRankRans = 3u };

// ---- RANS payloads: rANS-coded exponents of changed blocks --------------
constexpr uint32_t kModeRans = 2u;   // descriptor mode (CIERA_MODE_RANS)
constexpr int kRansLanes = 32;

// Payload sections of a shard of len values and nb blocks.
struct RansLayout {
  int64_t A;  // bitmap
  int64_t C;  // frequency table (256 uint16)
  int64_t O;  // nb + 1 uint32 record-byte prefixes
  int64_t D;  // records
};
__host__ __device__ inline RansLayout rans_layout(int64_t len, int64_t nb) {
  RansLayout r;
  r.A = (len + 15) & ~int64_t(15);
  r.C = (r.A + (nb + 7) / 8 + 15) & ~int64_t(15);
  r.O = r.C + 512;
  r.D = (r.O + 4 * (nb + 1) + 15) & ~int64_t(15);
  return r;
}

// Shard/tile geometry of a contiguous rank range.  Inside any range the
// full shards come first, then at most one partial shard, then empty ones.
struct Geometry {
  int64_t S;           // shard size ceil(N/R)
  int64_t B;           // block size
  int64_t T;           // blocks per tile
  int64_t tiles_full;  // tiles of a full shard
  int64_t len_part;    // values of the partial shard in range (0 if none)
  int64_t tiles_part;  // its tiles
  int64_t total_tiles;
  int32_t nfull;       // full shards in range
  int32_t has_part;    // partial shard present (range-local index nfull)
  int32_t rank_count;  // ranks in range, empty ones included
  int32_t pad;
};

struct CompressParams {
  Geometry geo;
  const uint16_t* w;            // first value of the range's first shard
  uint8_t* scache;              // sender exponent cache, same origin
  uint8_t* payloads;            // slot i at payloads + i*stride
  int64_t stride;
  ciera_desc* descs;
  uint8_t* flagbytes;           // per-rank rows of flag_stride bytes
  int64_t flag_stride;
  unsigned long long* tile_status;
  unsigned long long* tile_flags;  // per tile: epoch << 32 | flag bits (tiles of <= 32 blocks)
  unsigned long long* hash_cache;  // hashed change test: 2 words per block
  int64_t hash_stride;             // blocks per rank in hash_cache
  Control* ctl;
  uint64_t timeout_ns;
  uint32_t flags;
  int32_t raw_ahead;            // 1: shards predicted raw skip the look-back
  int32_t fast;                 // staged path allowed for whole-16 tiles
  int32_t hashed;               // 1: hashed change test (k_compress<true>)
  uint32_t* pred;               // per range rank: 1 if its last payload was RAW
                                // (read by k_compress, rewritten by k_repack)
  unsigned long long* result;   // per range rank: launch tag << 32 | kResult* bits
};

struct DecompressParams {
  Geometry geo;                 // the receiver's rank range
  const uint8_t* payloads;      // contiguous layout: range rank r at payloads + r*stride
  const uint8_t* const* payload_ptrs;  // or (non-null) range rank r at payload_ptrs[r]
  int64_t stride;               // slot stride, or with payload_ptrs each buffer's capacity
  const ciera_desc* descs;
  uint8_t* rcache;              // N exponent bytes
  uint16_t* out;                // N values
  uint32_t* bm_words;           // per rank: nw_stride aligned bitmap words
  uint32_t* bm_prefix;          // per rank: exclusive popcount prefix per word
  int64_t nw_stride;
  uint32_t* rank_state;         // per rank: kRank*
  Control* ctl;
  uint64_t timeout_ns;
  int32_t fast;
  int32_t rans;                 // 1: RANS payloads accepted (k_decompress_rans)
};

// Launchers (ciera_kernels.cu).  Return a cudaError_t value.
// smem_bytes: dynamic shared memory of one CTA.
// With p.raw_ahead, also launches k_repack (repack_smem bytes of dynamic
// shared memory per CTA).
int launch_compress(const CompressParams& p, int64_t smem_bytes, int raw_fixup,
                    int64_t repack_smem, void* stream);
int launch_decompress(const DecompressParams& p, int64_t smem_bytes, void* stream);

}  // namespace ciera
