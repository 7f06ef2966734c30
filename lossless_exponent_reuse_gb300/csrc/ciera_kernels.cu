// ciera_kernels.cu -- sm_103a kernels of libciera.
//
// Method: "CIERA: Cross-Iteration Exponent Reuse for Lossless Allgather in
// Sharded MoE Training", Section 3.1 (Exponent Reuse) and Appendix A,
// Algorithm 1.  The paper's sender hashes each block's exponents and ANS-codes
// changed exponents; here a block is compared exactly against the sender's
// cached exponents and a changed block travels as its bf16 values, and the
// receiver merges cached exponents with sign+mantissa bytes.
//
// Kernels (one CTA per tile of T consecutive blocks of one shard):
//   k_compress       split + compare + per-block flags, decoupled look-back
//                    over the count of changed blocks (the paper's "j <- j+1"
//                    over the bitmap, as a single-pass scan), pack, sender
//                    cache refresh, and -- in the shard's last tile -- the
//                    descriptor and the bitmap.
//   k_repack         after k_compress when raw-ahead is on: rewrites, in
//                    compacted layout, the shards predicted raw that were not,
//                    and records every shard's mode as the next prediction.
//   k_raw_fixup      only for plans where a raw payload can still contain
//                    unchanged blocks (tiny B): rewrites such payloads raw.
//   k_bitmap_scan    receiver: validates each descriptor against its bitmap
//                    and writes per-word exclusive popcount prefixes.
//   k_decompress     receiver: fused multi-rank gather + merge + ExpCache
//                    refresh.
// Tiles whose values are all whole 16-value groups use the staged path:
// cp.async.bulk copies into shared memory, completion on an mbarrier, and
// bulk stores back; other tiles use a byte-wise path with the same output.
// Every wait (mbarrier, look-back) is bounded by a timeout that records
// kStatusTimeout and lets the CTA finish.
#include <cuda_runtime.h>

#include <atomic>

#include "ciera_device.cuh"
#include "ciera_internal.h"

namespace ciera {
namespace {

// ------------------------------------------------------------------------
// Hashed change test (Section 3.1, Hash128 / HashCache).  SplitMix64's
// finalizer and increment (Steele, Lea and Flood, 2014); a block hash with
// one seed is fin(L + sum_j fin(word_j ^ key_j)) where word_j packs exponents
// 8j..8j+7 little-endian and key_j is SplitMix64's output j+1 from `seed`;
// the sum is order-free, so threads add their words in any order.

constexpr unsigned long long kGolden = 0x9e3779b97f4a7c15ull;
constexpr unsigned long long kSeed1 = 0x6a09e667f3bcc908ull;
constexpr unsigned long long kSeed2 = 0xbb67ae8584caa73bull;

__device__ __forceinline__ unsigned long long sm64_fin(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

// The keys (SplitMix64's outputs 1 .. kKeyWords from both seeds) of the
// first kKeyWords exponent words of a block, evaluated at compile time.
constexpr int kKeyWords = 2048;  // blocks of up to 16384 values

constexpr unsigned long long sm64_fin_c(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

struct HashKeys {
  unsigned long long k[kKeyWords][2];
};

constexpr HashKeys make_hash_keys() {
  HashKeys h{};
  for (int j = 0; j < kKeyWords; ++j) {
    const unsigned long long step = static_cast<unsigned long long>(j + 1) * kGolden;
    h.k[j][0] = sm64_fin_c(kSeed1 + step);
    h.k[j][1] = sm64_fin_c(kSeed2 + step);
  }
  return h;
}

__device__ const HashKeys g_hash_keys = make_hash_keys();

// Both seeds' terms of exponent word number j (0-based) of a block.
__device__ __forceinline__ void hash_word(unsigned long long word, int64_t j,
                                          unsigned long long& t1, unsigned long long& t2) {
  unsigned long long k1, k2;
  if (j < kKeyWords) {
    const ulonglong2 k = __ldg(reinterpret_cast<const ulonglong2*>(&g_hash_keys.k[j][0]));
    k1 = k.x;
    k2 = k.y;
  } else {
    const unsigned long long step = static_cast<unsigned long long>(j + 1) * kGolden;
    k1 = sm64_fin(kSeed1 + step);
    k2 = sm64_fin(kSeed2 + step);
  }
  t1 = sm64_fin(word ^ k1);
  t2 = sm64_fin(word ^ k2);
}

// ------------------------------------------------------------------------
// Compress: one CTA per tile, tiles in ticket order.
//
//   thread 0   draws the ticket, starts the bulk copies of the tile's
//              values and cached exponents into shared memory
//   warp 0     meanwhile walks the look-back for the tile's exclusive prefix
//   warps 1-3  wait for the copies, flag the tile's blocks, write the flag
//              bytes and publish the tile's aggregate
//   then       warp 0 publishes the inclusive prefix, all warps pack, thread
//              0 issues the bulk stores of the body, and the shard's last
//              tile writes the descriptor and the bitmap.
// A raw-ahead tile (its shard predicted RAW) skips the look-back: thread 0
// stores the values at their raw positions as soon as they land, all four
// warps flag and refresh the cache, and the shard's last tile sums the
// aggregates and checks the prediction (raw_ahead_finish; k_repack rewrites
// the shard if it was wrong).
// Dynamic shared memory: fw[W] flag words | fpre[W] their exclusive
// popcount prefix | (staged tiles) ws[2*TE] values | cs[TE] cached exponents.

struct CompressShared {
  uint32_t ticket;
  uint32_t epoch; // this launch's tag of look-back and flag words (never 0)
  uint32_t X;     // changed blocks before the tile in its shard
  uint32_t agg;   // changed blocks in the tile
  uint32_t bad;   // a bounded wait ran out on this tile
  uint32_t ahead; // raw-ahead tile: values stored at their raw positions, no look-back
  uint32_t red[kThreads / 32];  // per-warp sums of the raw-ahead finish
};

// Named barrier of the nf flagging threads of a compress CTA: warps 1-3
// while warp 0 walks the look-back, all four warps on a raw-ahead tile.
__device__ __forceinline__ void flag_sync(int nf) {
  asm volatile("bar.sync 1, %0;" ::"r"(nf) : "memory");
}

// A compress CTA sends to L2 the values and cached exponents (the hashed
// sender: the HashCache entries) of the tile kPrefetchAhead tickets after its
// own (about a third of the CTAs resident on the GPU), unless that tile's
// shard is predicted raw.  A tile that waits on its look-back holds its
// staging, so fewer loads are in flight; the lines brought in ahead keep DRAM
// busy meanwhile, and the later tile's bulk copies find them in L2.  The
// prefetch is one bulk request per range, from one thread, marked evict_last
// so that the lines outlast the stream of payload and cache writes until
// their tile loads them.  Much further ahead they are evicted before use all
// the same.
constexpr int64_t kPrefetchAhead = 512;
// [a, a + bytes) into L2: a 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void* a, uint32_t bytes) {
  unsigned long long policy;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(a),
               "r"(bytes), "l"(policy)
               : "memory");
}

// Block of 16-value group gi on the staged paths (blocks of G = B/16 >= 16
// groups, gi < 2^16): floor(gi / G) as mulhi(gi, m) with m = ceil(2^32 / G),
// exact there because gi * (m - 2^32/G) / 2^32 < 2^-16 < 1/G.  A runtime
// division per group was the largest item of the loops that use it.
__device__ __forceinline__ uint32_t group_divisor(int64_t B) {
  const uint32_t G = static_cast<uint32_t>(B >> 4);
  return 0xffffffffu / G + 1u;  // = ceil(2^32 / G) for G >= 2
}
__device__ __forceinline__ int block_of_group(int gi, uint32_t m) {
  return static_cast<int>(__umulhi(static_cast<uint32_t>(gi), m));
}

// The flagging threads (ft = 0 .. nf-1), after the flag bits are final: flag
// bytes, popcount prefix, aggregate, and its publication (the inclusive
// prefix directly for a shard's first tile).
__device__ void publish_aggregate(const CompressParams& p, const Tile& x, CompressShared& sh,
                                  uint32_t* fw, uint32_t* fpre, int ft, int nf) {
  const int nw = (x.nblk + 31) >> 5;
  uint8_t* fb = p.flagbytes + static_cast<int64_t>(x.rl) * p.flag_stride + x.k0;
  if (x.nblk > 32) {
    for (int kb = ft; kb < x.nblk; kb += nf) fb[kb] = flag_of(fw, kb) ? 1 : 0;
    if (ft < x.nblk) __threadfence();
    flag_sync(nf);
  }
  if (ft == 0) {
    // with flag bytes, the release of the status below orders these writes
    // (and, through the fences above, those of the other flagging threads)
    if (x.nblk <= 32)
      for (int kb = 0; kb < x.nblk; ++kb) fb[kb] = flag_of(fw, kb) ? 1 : 0;
    if (flags_in_words(p))
      st_relaxed_u64(&p.tile_flags[x.sidx], (static_cast<unsigned long long>(sh.epoch) << 32) | fw[0]);
    uint32_t run = 0;
    for (int i = 0; i < nw; ++i) {
      fpre[i] = run;
      run += __popc(fw[i]);
    }
    sh.agg = run;
    const bool skip = (p.flags & CIERA_DEBUG_SKIP_FIRST_PUBLISH) && x.t == 0;
    // a raw-ahead shard's tiles publish aggregates only; its last tile turns
    // them into prefixes where a rewrite needs them
    const uint32_t state = x.t == 0 && !sh.ahead ? kStateInclusive : kStateAggregate;
    if (!skip) publish(p, x, sh.epoch, state, run);
  }
}

// Body size of a shard (len values, nb blocks) with `total` changed blocks;
// last_changed: its last (possibly partial) block changed.
__device__ __forceinline__ int64_t body_bytes_of(const Tile& x, int64_t B, uint32_t total,
                                                 bool last_changed) {
  const int64_t last_len = x.len - (x.nb - 1) * B;
  const int64_t changed_vals =
      static_cast<int64_t>(total) * B - (last_changed ? (B - last_len) : 0);
  return x.len + changed_vals;
}

// The shard's bitmap (bm bytes) at payload offset `body`, all threads of the
// CTA.  Every tile of the shard wrote its flags during this launch.
__device__ void write_bitmap(const CompressParams& p, const Tile& x, uint32_t epoch,
                             int64_t body, int64_t bm) {
  const int tid = threadIdx.x;
  uint8_t* payload = p.payloads + static_cast<int64_t>(x.rl) * p.stride;
  if (flags_in_words(p)) {
    // each tile stored its flag bits with this launch's tag; wait (bounded)
    // until each word shows it
    const unsigned long long* tf = p.tile_flags + (x.sidx - x.t);
    const int64_t T = p.geo.T;
    bool to = false;
    for (int64_t i = tid; i < bm; i += blockDim.x) {
      uint32_t byte = 0;
      int64_t cur = -1;
      uint32_t bits = 0;
      for (int j = 0; j < 8; ++j) {
        const int64_t k = 8 * i + j;
        if (k >= x.nb) break;
        const int64_t tj = k / T;
        if (tj != cur) {
          cur = tj;
          unsigned long long v = ld_relaxed_u64(tf + tj);
          if ((v >> 32) != epoch) {
            const uint64_t t0 = globaltimer();
            while ((v >> 32) != epoch) {
              if (globaltimer() - t0 > p.timeout_ns) {
                to = true;
                break;
              }
              __nanosleep(32);
              v = ld_relaxed_u64(tf + tj);
            }
          }
          bits = static_cast<uint32_t>(v);
        }
        byte |= ((bits >> (k - tj * T)) & 1u) << j;
      }
      if (in_bounds(p.ctl, body + i, 1, p.stride)) payload[body + i] = static_cast<uint8_t>(byte);
    }
    if (to) record_status(p.ctl, kStatusTimeout);
  } else {
    // every earlier tile wrote its flag bytes before publishing its status;
    // read them from L2 (other CTAs wrote them during this launch)
    const uint8_t* fb = p.flagbytes + static_cast<int64_t>(x.rl) * p.flag_stride;
    for (int64_t i = tid; i < bm; i += blockDim.x) {
      uint32_t byte = 0;
      for (int j = 0; j < 8; ++j) {
        const int64_t k = 8 * i + j;
        if (k < x.nb) byte |= static_cast<uint32_t>(__ldcg(fb + k) & 1u) << j;
      }
      if (in_bounds(p.ctl, body + i, 1, p.stride)) payload[body + i] = static_cast<uint8_t>(byte);
    }
  }
}

// Last tile of a shard: descriptor and bitmap.
__device__ void compress_epilogue(const CompressParams& p, const Tile& x, const CompressShared& sh,
                                  const uint32_t* fw) {
  const int tid = threadIdx.x;
  const uint32_t total = sh.X + sh.agg;  // changed blocks in the shard
  const bool last_changed = flag_of(fw, static_cast<int>(x.nb - 1 - x.k0));
  const int64_t body = body_bytes_of(x, p.geo.B, total, last_changed);
  const int64_t bm = (x.nb + 7) / 8;
  const bool raw = (p.flags & CIERA_COLD) || (body + bm >= 2 * x.len);
  if (tid == 0) {
    ciera_desc d;
    d.mode = raw ? CIERA_MODE_RAW : CIERA_MODE_COMPRESSED;
    d.n_changed_blocks = total;
    d.body_bytes = static_cast<uint64_t>(raw ? 2 * x.len : body);
    d.payload_bytes = static_cast<uint64_t>(raw ? 2 * x.len : body + bm);
    p.descs[x.rl] = d;
    if (p.raw_ahead)
      p.result[x.rl] = (static_cast<unsigned long long>(sh.epoch) << 32) | (raw ? kResultRaw : 0u);
  }
  if (raw) return;
  write_bitmap(p, x, sh.epoch, body, bm);
}

// Last tile of a raw-ahead shard, all threads.  Every tile of the shard
// stored its values at their raw positions and published only its
// aggregate.  Sum the aggregates (each thread a contiguous run of tiles,
// waiting, bounded, for tiles still running) and write the descriptor.  A
// raw shard is then complete.  Otherwise every tile's status word is
// rewritten as its inclusive prefix and the shard is left to k_repack, which
// rewrites the payload compacted and appends the bitmap (the raw stores of
// other tiles may still be in flight, so nothing is compacted here).
__device__ void raw_ahead_finish(const CompressParams& p, const Tile& x, CompressShared& sh,
                                 const uint32_t* fw) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = x.tiles;
  const int64_t chunk = (n + kThreads - 1) / kThreads;
  const int64_t i0 = tid * chunk < n ? tid * chunk : n;
  const int64_t i1 = i0 + chunk < n ? i0 + chunk : n;
  unsigned long long* st = p.tile_status + (x.sidx - x.t);
  const uint32_t epoch = sh.epoch;
  bool to = false;
  uint32_t sum = 0;
  for (int64_t i = i0; i < i1 && !to; ++i) {
    unsigned long long v = ld_relaxed_u64(st + i);
    if ((v >> 32) != epoch || ((v >> 30) & 3ull) == 0) {
      const uint64_t t0 = globaltimer();
      while ((v >> 32) != epoch || ((v >> 30) & 3ull) == 0) {
        if (globaltimer() - t0 > p.timeout_ns) {
          to = true;
          break;
        }
        __nanosleep(256);
        v = ld_relaxed_u64(st + i);
      }
    }
    sum += static_cast<uint32_t>(v & 0x3FFFFFFFull);
  }
  // exclusive prefix of the per-thread sums across the CTA
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sh.red[warp] = incl;
  const bool any_to = __syncthreads_or(to);
  uint32_t base = 0, total = 0;
#pragma unroll
  for (int w2 = 0; w2 < kThreads / 32; ++w2) {
    base += w2 < warp ? sh.red[w2] : 0u;
    total += sh.red[w2];
  }
  if (total > x.nb) total = static_cast<uint32_t>(x.nb);  // only after a timeout
  const bool last_changed = flag_of(fw, static_cast<int>(x.nb - 1 - x.k0));
  const int64_t body = body_bytes_of(x, p.geo.B, total, last_changed);
  const int64_t bm = (x.nb + 7) / 8;
  const bool raw = (p.flags & CIERA_COLD) || (body + bm >= 2 * x.len);
  if (!raw && !any_to) {
    const unsigned long long tag = (static_cast<unsigned long long>(epoch) << 32) |
                                   (static_cast<unsigned long long>(kStateInclusive) << 30);
    uint32_t run = base + incl - sum;
    for (int64_t i = i0; i < i1; ++i) {
      run += static_cast<uint32_t>(ld_relaxed_u64(st + i) & 0x3FFFFFFFull);
      st_relaxed_u64(st + i, tag | run);
    }
  }
  if (tid == 0) {
    if (any_to) record_status(p.ctl, kStatusTimeout);
    ciera_desc d;
    d.mode = raw ? CIERA_MODE_RAW : CIERA_MODE_COMPRESSED;
    d.n_changed_blocks = total;
    d.body_bytes = static_cast<uint64_t>(raw ? 2 * x.len : body);
    d.payload_bytes = static_cast<uint64_t>(raw ? 2 * x.len : body + bm);
    p.descs[x.rl] = d;
    const uint32_t res = any_to ? 0u : raw ? kResultRaw : kResultRepack;
    p.result[x.rl] = (static_cast<unsigned long long>(epoch) << 32) | res;
  }
}

// Thread 0 of a staged tile: bulk stores of the body, one per maximal run of
// equally flagged blocks -- changed runs from the values (ws), unchanged runs
// from their sign+mantissa bytes (cs) -- at offsets that follow from X, the
// changed blocks before the tile in its shard.
__device__ void store_runs(const CompressParams& p, const Tile& x, const uint32_t* fw,
                           const uint32_t* fpre, uint32_t X, const uint8_t* ws, const uint8_t* cs) {
  const int64_t B = p.geo.B;
  uint8_t* payload = p.payloads + static_cast<int64_t>(x.rl) * p.stride;
  int ka = 0;
  while (ka < x.nblk) {
    const bool f = flag_of(fw, ka);
    int kz = ka + 1;
    while (kz < x.nblk && flag_of(fw, kz) == f) ++kz;
    const int64_t ea = static_cast<int64_t>(ka) * B;
    const int64_t ez = static_cast<int64_t>(kz) * B < x.te ? static_cast<int64_t>(kz) * B : x.te;
    const int64_t off = (x.k0 + ka + X + count_before(fw, fpre, ka)) * B;
    const int64_t bytes = (f ? 2 : 1) * (ez - ea);
    if (in_bounds(p.ctl, off, bytes, p.stride))
      bulk_s2g(payload + off, f ? ws + 2 * ea : cs + ea, static_cast<uint32_t>(bytes));
    ka = kz;
  }
  bulk_commit();
}

// kHashed: the change test is the 128-bit block hash against the HashCache
// (16 bytes per block) instead of an exponent compare against the sender's
// exponent cache; then only the values are staged, and cs holds nothing but
// the sign+mantissa bytes of unchanged blocks.  Needs T <= 32.
// Nine CTAs fit an SM by shared memory (24.7 KB each); the bound keeps the
// registers there too (without it the compiler picked 48 and spilled).
template <bool kHashed>
__global__ void __launch_bounds__(kThreads, 9) k_compress(const CompressParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ CompressShared sh;
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t B = p.geo.B;
  const int64_t TE = p.geo.T * B;
  const int W = static_cast<int>((p.geo.T + 31) / 32);
  // flag region: fw[W] | fpre[W] | (kHashed) bsum[2T] hash sums | hs[2T] the
  // tile's HashCache entries, copied in with the values
  const int bsum_off = (8 * W + 15) & ~15;
  const int hs_off = bsum_off + 16 * static_cast<int>(p.geo.T);
  const int FW = kHashed ? ((hs_off + 16 * static_cast<int>(p.geo.T) + 127) & ~127)
                         : ((8 * W + 127) & ~127);
  uint32_t* fw = reinterpret_cast<uint32_t*>(dsm);
  uint32_t* fpre = fw + W;
  unsigned long long* bsum = reinterpret_cast<unsigned long long*>(dsm + bsum_off);
  unsigned long long* hs = reinterpret_cast<unsigned long long*>(dsm + hs_off);
  uint8_t* ws = dsm + FW;
  uint8_t* cs = ws + 2 * TE;

  if (tid == 0) {
    // ticket order = start order: a tile only ever waits on tiles whose
    // CTAs started earlier, so the look-back never waits on an unscheduled CTA
    // The counter word holds (launch number << 32) | tickets drawn.  Every
    // CTA of a launch reads the same launch number with its ticket; the one
    // that draws the last ticket resets the count and advances the number
    // in one exchange, so replays of a captured launch get fresh tags too.
    const unsigned long long v = atomicAdd(&p.ctl->ticket, 1ull);
    const uint32_t t = static_cast<uint32_t>(v);
    const uint32_t launch = static_cast<uint32_t>(v >> 32);
    if (t == gridDim.x - 1) atomicExch(&p.ctl->ticket, static_cast<unsigned long long>(launch + 1u) << 32);
    sh.ticket = t;
    sh.epoch = launch % 0xffffffffu + 1u;  // 1 .. 2^32-1: a zero-filled word never matches
    sh.bad = 0;
    sh.ahead = 0;
  }
  // the launch must provide the flag words (and the staging of staged
  // tiles); if it does not, report it instead of touching memory past it
  const uint32_t need = static_cast<uint32_t>(FW + (p.fast ? 3 * TE : 0));
  if (dynamic_smem_size() < need || (kHashed && p.geo.T > 32)) {
    if (tid == 0) record_status(p.ctl, kStatusInternal);
    return;
  }
  for (int i = tid; i < W; i += blockDim.x) fw[i] = 0;
  if (kHashed)
    for (int i = tid; i < 2 * p.geo.T; i += blockDim.x) bsum[i] = 0;
  __syncthreads();
  const int64_t g = sh.ticket;
  if (g >= p.geo.total_tiles) {
    // the last ticket: descriptors of empty shards in the range
    for (int32_t rl = p.geo.nfull + p.geo.has_part + tid; rl < p.geo.rank_count;
         rl += blockDim.x) {
      ciera_desc d;
      d.mode = CIERA_MODE_RAW;
      d.n_changed_blocks = 0;
      d.body_bytes = 0;
      d.payload_bytes = 0;
      p.descs[rl] = d;
    }
    return;
  }
  const Tile x = decode_ticket(p.geo, g);
  const bool stg = p.fast && (x.te & 15) == 0;
  const uint32_t mG = stg ? group_divisor(B) : 0u;  // block_of_group (staged tiles)
  const bool cold = p.flags & CIERA_COLD;
  const uint16_t* w = p.w + x.shard_off + x.e0;
  uint8_t* c = p.scache + x.shard_off + x.e0;
  const uint32_t te = static_cast<uint32_t>(x.te);
  const unsigned long long* hc_tile =
      kHashed ? p.hash_cache + 2 * (static_cast<int64_t>(x.rl) * p.hash_stride + x.k0) : nullptr;
  if (stg && tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (kHashed) {
      mbar_arrive_expect_tx(&bar, 2u * te + 16u * static_cast<uint32_t>(x.nblk));
      bulk_g2s(ws, w, 2u * te, &bar);
      bulk_g2s(hs, hc_tile, 16u * static_cast<uint32_t>(x.nblk), &bar);
    } else {
      mbar_arrive_expect_tx(&bar, 3u * te);
      bulk_g2s(ws, w, 2u * te, &bar);
      bulk_g2s(cs, c, te, &bar);
    }
    // Raw-ahead: a shard whose last payload was RAW (or any shard of a cold
    // call, which is RAW by definition) is predicted raw again.  Its tiles
    // store their values at their raw positions as soon as they arrive and
    // skip the look-back; the shard's last tile checks the prediction.  Only
    // shards whose every tile is staged take part.
    sh.ahead = p.raw_ahead && (x.len & 15) == 0 && (cold || __ldg(p.pred + x.rl) != 0u);
  }
  __syncthreads();
  if (stg && tid == 0 && g + kPrefetchAhead < p.geo.total_tiles) {
    const Tile y = decode_ticket(p.geo, g + kPrefetchAhead);
    const bool y_ahead =
        p.raw_ahead && (y.len & 15) == 0 && (cold || __ldg(p.pred + y.rl) != 0u);
    // staged plans keep every shard and block start 16-byte aligned; a
    // ragged last tile of a partial shard is left to its own copy
    if (!y_ahead && (y.te & 15) == 0) {
      prefetch_l2_bulk(p.w + y.shard_off + y.e0, static_cast<uint32_t>(2 * y.te));
      if (kHashed)
        prefetch_l2_bulk(p.hash_cache + 2 * (static_cast<int64_t>(y.rl) * p.hash_stride + y.k0),
                         static_cast<uint32_t>(16 * y.nblk));
      else
        prefetch_l2_bulk(p.scache + y.shard_off + y.e0, static_cast<uint32_t>(y.te));
    }
  }

  if (warp == 0 && !sh.ahead) {
    bool to = false;
    const uint32_t X = lookback_exclusive(p, x, sh.epoch, lane, x.k0, &to);
    if (lane == 0) {
      sh.X = X;
      if (to) record_status(p.ctl, kStatusTimeout);
    }
    // with flag bytes, the shard's last tile reads every other tile's flag
    // bytes later on
    if (x.t == x.tiles - 1 && !flags_in_words(p)) __threadfence();
    if (stg) mbar_wait_bounded(&bar, 0, p.timeout_ns);  // this warp reads ws/cs too
  } else {
    // the flagging threads: warps 1-3, or on a raw-ahead tile (no look-back)
    // all four warps, whose thread 0 first stores the values at their raw
    // positions
    const int nf = sh.ahead ? kThreads : kThreads - 32;
    const int ft = sh.ahead ? tid : tid - 32;
    if (stg) {
      if (!mbar_wait_bounded(&bar, 0, p.timeout_ns)) {
        // record it and wait once more, so no copy still writes into this
        // CTA's shared memory when it exits
        record_status(p.ctl, kStatusTimeout);
        sh.bad = 1;
        mbar_wait_bounded(&bar, 0, p.timeout_ns);
      } else if (sh.ahead && tid == 0) {
        int64_t off = 2 * x.e0;
            if (in_bounds(p.ctl, off, 2 * x.te, p.stride))
          bulk_s2g(p.payloads + static_cast<int64_t>(x.rl) * p.stride + off, ws, 2u * te);
        bulk_commit();
      }
    }
    flag_sync(nf);
    if (kHashed) {
      // per-block sums of the two seeds' word terms
      if (stg) {
        const int ngroups = static_cast<int>(te >> 4);
        unsigned long long s1 = 0, s2 = 0;
        // The loop runs whole warps over 32 consecutive groups at a time.  A
        // warp whose groups all lie in one block keeps running sums in
        // registers; when its block changes it reduces them across the warp
        // and lane 0 adds them to the block's sums.  A warp straddling two
        // blocks (blocks of fewer than 512 values) adds lane by lane.
        const int G = static_cast<int>(B / 16);  // groups per block
        int cur = -1;                            // block of the running sums (warp-uniform)
        auto flush = [&]() {
          if (cur < 0) return;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            s2 += __shfl_xor_sync(0xffffffffu, s2, o);
          }
          if (lane == 0) {
            atomicAdd(&bsum[2 * cur], s1);
            atomicAdd(&bsum[2 * cur + 1], s2);
          }
          s1 = s2 = 0;
          cur = -1;
        };
        for (int g0 = ft - lane; g0 < ngroups; g0 += nf) {
          const int gi = g0 + lane;
          const bool in = gi < ngroups;
          int kb = -1;
          unsigned long long t1 = 0, t2 = 0;
          if (in) {
            const uint4 w0 = reinterpret_cast<const uint4*>(ws)[2 * gi];
            const uint4 w1 = reinterpret_cast<const uint4*>(ws)[2 * gi + 1];
            kb = block_of_group(gi, mG);
            const int64_t j0 = 2 * static_cast<int64_t>(gi - kb * G);  // first exponent word
            const unsigned long long lo =
                exp4(w0.x, w0.y) | (static_cast<unsigned long long>(exp4(w0.z, w0.w)) << 32);
            const unsigned long long hi =
                exp4(w1.x, w1.y) | (static_cast<unsigned long long>(exp4(w1.z, w1.w)) << 32);
            unsigned long long a1, a2, b1, b2;
            hash_word(lo, j0, a1, a2);
            hash_word(hi, j0 + 1, b1, b2);
            t1 = a1 + b1;
            t2 = a2 + b2;
          }
          const int kb0 = __shfl_sync(0xffffffffu, kb, 0);  // lane 0 is always in
          const bool uniform = __all_sync(0xffffffffu, !in || kb == kb0);
          if (!(uniform && kb0 == cur)) {
            flush();
            if (!uniform) {
              if (in) {
                atomicAdd(&bsum[2 * kb], t1);
                atomicAdd(&bsum[2 * kb + 1], t2);
              }
              continue;
            }
            cur = kb0;
          }
          s1 += t1;
          s2 += t2;
        }
        flush();
      } else {
        const int64_t wpb = (B + 7) / 8;  // exponent words per block
        const int64_t nwords = static_cast<int64_t>(x.nblk) * wpb;
        for (int64_t q = ft; q < nwords; q += nf) {
          const int kb = static_cast<int>(q / wpb);
          const int64_t j = q - kb * wpb;
          const int64_t first = kb * B + 8 * j;  // tile-relative
          const int64_t blen = (kb + 1) * B < x.te ? B : x.te - kb * B;
          if (8 * j >= blen) continue;
          unsigned long long word = 0;
          for (int i = 0; i < 8 && 8 * j + i < blen; ++i)
            word |= static_cast<unsigned long long>(exp1(w[first + i])) << (8 * i);
          unsigned long long t1, t2;
          hash_word(word, j, t1, t2);
          atomicAdd(&bsum[2 * kb], t1);
          atomicAdd(&bsum[2 * kb + 1], t2);
        }
      }
      flag_sync(nf);
      // one thread per block: finish both hashes, test and refresh the
      // HashCache entry
      for (int kb = ft; kb < x.nblk; kb += nf) {
        const int64_t blen = (kb + 1) * B < x.te ? B : x.te - kb * B;
        const unsigned long long h1 = sm64_fin(static_cast<unsigned long long>(blen) + bsum[2 * kb]);
        const unsigned long long h2 =
            sm64_fin(static_cast<unsigned long long>(blen) + bsum[2 * kb + 1]);
        unsigned long long* hc = const_cast<unsigned long long*>(hc_tile) + 2 * kb;
        const unsigned long long o1 = stg ? hs[2 * kb] : hc[0];
        const unsigned long long o2 = stg ? hs[2 * kb + 1] : hc[1];
        const bool changed = cold || sh.bad || o1 != h1 || o2 != h2;
        if (changed) {
          hc[0] = h1;
          hc[1] = h2;
          atomicOr(&fw[kb >> 5], 1u << (kb & 31));
        }
      }
    } else if (cold || sh.bad) {
      for (int kb = ft; kb < x.nblk; kb += nf) atomicOr(&fw[kb >> 5], 1u << (kb & 31));
    } else if (stg) {
      const int ngroups = static_cast<int>(te >> 4);
      for (int gi = ft; gi < ngroups; gi += nf) {
        const uint4 w0 = reinterpret_cast<const uint4*>(ws)[2 * gi];
        const uint4 w1 = reinterpret_cast<const uint4*>(ws)[2 * gi + 1];
        const uint4 cc = reinterpret_cast<const uint4*>(cs)[gi];
        const uint4 e = make_uint4(exp4(w0.x, w0.y), exp4(w0.z, w0.w), exp4(w1.x, w1.y),
                                   exp4(w1.z, w1.w));
        if ((e.x ^ cc.x) | (e.y ^ cc.y) | (e.z ^ cc.z) | (e.w ^ cc.w)) {
          // a group whose exponents differ lies in a changed block, and these
          // are the only groups of changed blocks whose cache entry moves:
          // refresh it here instead of in a second pass
          reinterpret_cast<uint4*>(c)[gi] = e;
          const int kb = block_of_group(gi, mG);
          atomicOr(&fw[kb >> 5], 1u << (kb & 31));
        }
      }
    } else {
      for (int64_t j = ft; j < x.te; j += nf) {
        if (exp1(w[j]) != c[j]) {
          const int kb = static_cast<int>(j / B);
          atomicOr(&fw[kb >> 5], 1u << (kb & 31));
        }
      }
    }
    flag_sync(nf);
    publish_aggregate(p, x, sh, fw, fpre, ft, nf);
    // Without a compare (cold call, or a timed-out copy) every cache group
    // of the tile is rewritten here; otherwise the compare refreshed them.
    const bool refresh_all = !kHashed && (cold || sh.bad);
    if (stg && (refresh_all || !sh.ahead)) {
      // Pack while warp 0 may still be looking back: nothing here depends
      // on the prefix.  Sign+mantissa bytes of an unchanged block overwrite
      // its own cached exponents in cs, which nothing reads any more.  A
      // raw-ahead tile sends its values as they are and packs nothing.
      const int ngroups = static_cast<int>(te >> 4);
      for (int gi = ft; gi < ngroups; gi += nf) {
        const int kb = block_of_group(gi, mG);
        const bool f = flag_of(fw, kb);
        if (f ? !refresh_all : sh.ahead) continue;
        const uint4 w0 = reinterpret_cast<const uint4*>(ws)[2 * gi];
        const uint4 w1 = reinterpret_cast<const uint4*>(ws)[2 * gi + 1];
        if (f)
          reinterpret_cast<uint4*>(c)[gi] = make_uint4(exp4(w0.x, w0.y), exp4(w0.z, w0.w),
                                                       exp4(w1.x, w1.y), exp4(w1.z, w1.w));
        else
          reinterpret_cast<uint4*>(cs)[gi] =
              make_uint4(sm4(w0.x, w0.y), sm4(w0.z, w0.w), sm4(w1.x, w1.y), sm4(w1.z, w1.w));
      }
      fence_proxy_async_smem();
    }
  }
  __syncthreads();
  if (sh.ahead) {
    if (x.t == x.tiles - 1) raw_ahead_finish(p, x, sh, fw);
    if (tid == 0) bulk_wait_read_all();
    return;
  }
  if (tid == 0 && x.t > 0) publish(p, x, sh.epoch, kStateInclusive, sh.X + sh.agg);

  uint8_t* payload = p.payloads + static_cast<int64_t>(x.rl) * p.stride;
  if (stg) {
    // the bulk stores are the only step that needs the prefix
    if (tid == 0) store_runs(p, x, fw, fpre, sh.X, ws, cs);
  } else {
    for (int64_t j = tid; j < x.te; j += blockDim.x) {
      const int kb = static_cast<int>(j / B);
      const int64_t within = j - kb * B;
      const int64_t kg = x.k0 + kb;
      const int64_t off = (kg + sh.X + count_before(fw, fpre, kb)) * B;
      const uint32_t v = w[j];
      if (flag_of(fw, kb)) {
        if (in_bounds(p.ctl, off + 2 * within, 2, p.stride)) {
          payload[off + 2 * within] = static_cast<uint8_t>(v & 0xFFu);
          payload[off + 2 * within + 1] = static_cast<uint8_t>(v >> 8);
        }
        if (!kHashed) {
          const uint8_t e = static_cast<uint8_t>(exp1(v));
          if (c[j] != e) c[j] = e;
        }
      } else if (in_bounds(p.ctl, off + within, 1, p.stride)) {
        payload[off + within] = static_cast<uint8_t>(sm1(v));
      }
    }
  }
  if (x.t == x.tiles - 1) compress_epilogue(p, x, sh, fw);
  if (stg && tid == 0) bulk_wait_read_all();
}

// A raw payload whose body was written in compressed layout (possible only
// when an unchanged block is not larger than the bitmap): copy the shard.
__global__ void __launch_bounds__(kThreads) k_raw_fixup(const CompressParams p) {
  const Tile x = decode_tile(p.geo, blockIdx.x);
  const ciera_desc d = p.descs[x.rl];
  if (d.mode != CIERA_MODE_RAW || d.n_changed_blocks >= x.nb) return;
  const uint16_t* w = p.w + x.shard_off + x.e0;
  uint8_t* payload = p.payloads + static_cast<int64_t>(x.rl) * p.stride;
  for (int64_t j = threadIdx.x; j < x.te; j += blockDim.x) {
    const uint32_t v = w[j];
    const int64_t o = 2 * (x.e0 + j);
    if (!in_bounds(p.ctl, o, 2, p.stride)) continue;
    payload[o] = static_cast<uint8_t>(v & 0xFFu);
    payload[o + 1] = static_cast<uint8_t>(v >> 8);
  }
}

// After a k_compress launch with raw-ahead on: record each shard's outcome
// as the next call's prediction, and rewrite in compacted layout every
// raw-ahead shard that did not turn out raw.  Such a shard's last tile wrote
// its descriptor and every tile's inclusive prefix; its tiles' flag words
// carry the launch's tag.  CTA b rewrites tiles b, b + gridDim.x, ... of
// each such shard from the values (the payload holds them at their raw
// positions, which the compacted body overwrites), and the shard's last
// tile appends the bitmap.  With nothing to rewrite every CTA exits after
// reading the result words.
// Dynamic shared memory: 128 bytes | ws[2*TE] values | cs[TE] sign+mantissa
// bytes | one bit per shard (shards to rewrite).
__global__ void __launch_bounds__(kThreads) k_repack(const CompressParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ uint32_t s_epoch, s_nfix, s_X, s_bad;
  __shared__ uint32_t s_fw[1], s_fpre[1];
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x;
  const int64_t B = p.geo.B;
  const int64_t TE = p.geo.T * B;
  const int nr = p.geo.nfull + p.geo.has_part;  // shards with tiles
  const int nmw = (nr + 31) / 32;
  uint8_t* ws = dsm + 128;
  uint8_t* cs = ws + 2 * TE;
  uint32_t* mask = reinterpret_cast<uint32_t*>(cs + TE);
  if (dynamic_smem_size() < static_cast<uint32_t>(128 + 3 * TE + 4 * nmw) || p.geo.T > 32) {
    if (tid == 0) record_status(p.ctl, kStatusInternal);
    return;
  }
  // the first result word is loaded alongside the launch counter
  const unsigned long long v0 = tid < nr ? p.result[tid] : 0ull;
  if (tid == 0) {
    // the launch just finished drew its tag from the counter, then advanced it
    const uint32_t launch = static_cast<uint32_t>(ld_relaxed_u64(&p.ctl->ticket) >> 32) - 1u;
    s_epoch = launch % 0xffffffffu + 1u;
    s_nfix = 0;
    s_fpre[0] = 0;
  }
  for (int i = tid; i < nmw; i += kThreads) mask[i] = 0;
  __syncthreads();
  const uint32_t epoch = s_epoch;
  for (int rl = tid; rl < nr; rl += kThreads) {
    const unsigned long long v = rl == tid ? v0 : p.result[rl];
    const bool cur = (v >> 32) == epoch;
    if (blockIdx.x == 0) p.pred[rl] = cur && (v & kResultRaw) ? 1u : 0u;
    if (cur && (v & kResultRepack)) {
      atomicOr(&mask[rl >> 5], 1u << (rl & 31));
      atomicAdd(&s_nfix, 1u);
    }
  }
  __syncthreads();
  if (s_nfix == 0) return;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  uint32_t phase = 0;
  const uint32_t mG = group_divisor(B);
  const unsigned long long ep = static_cast<unsigned long long>(epoch);
  for (int rl = 0; rl < nr; ++rl) {
    if (!((mask[rl >> 5] >> (rl & 31)) & 1u)) continue;
    const int64_t tiles = rl < p.geo.nfull ? p.geo.tiles_full : p.geo.tiles_part;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
      const Tile x = make_tile(p.geo, rl, t);
      const uint32_t te = static_cast<uint32_t>(x.te);
      if (tid == 0) {
        mbar_arrive_expect_tx(&bar, 2u * te);
        bulk_g2s(ws, p.w + x.shard_off + x.e0, 2u * te, &bar);
        const unsigned long long f = ld_relaxed_u64(&p.tile_flags[x.sidx]);
        const unsigned long long q = t > 0 ? ld_relaxed_u64(&p.tile_status[x.sidx - 1])
                                           : (ep << 32) | (uint64_t(kStateInclusive) << 30);
        s_fw[0] = static_cast<uint32_t>(f);
        s_X = static_cast<uint32_t>(q & 0x3FFFFFFFull);
        s_bad = (f >> 32) != ep || (q >> 32) != ep || ((q >> 30) & 3ull) != kStateInclusive ||
                s_X > static_cast<uint32_t>(x.k0);
        if (s_bad) record_status(p.ctl, kStatusInternal);
      }
      __syncthreads();
      const bool ok = mbar_wait_bounded(&bar, phase, p.timeout_ns);
      if (__syncthreads_or(!ok)) {
        // wait once more so that no copy still writes into shared memory
        // when the CTA exits
        if (tid == 0) record_status(p.ctl, kStatusTimeout);
        if (!ok) mbar_wait_bounded(&bar, phase, p.timeout_ns);
        return;
      }
      phase ^= 1u;
      const uint32_t fw0 = s_fw[0];
      if (!s_bad) {
        const int ngroups = static_cast<int>(te >> 4);
        for (int gi = tid; gi < ngroups; gi += kThreads) {
          const int kb = block_of_group(gi, mG);
          if ((fw0 >> kb) & 1u) continue;
          const uint4 w0 = reinterpret_cast<const uint4*>(ws)[2 * gi];
          const uint4 w1 = reinterpret_cast<const uint4*>(ws)[2 * gi + 1];
          reinterpret_cast<uint4*>(cs)[gi] =
              make_uint4(sm4(w0.x, w0.y), sm4(w0.z, w0.w), sm4(w1.x, w1.y), sm4(w1.z, w1.w));
        }
        fence_proxy_async_smem();
      }
      __syncthreads();
      if (!s_bad) {
        if (tid == 0) store_runs(p, x, s_fw, s_fpre, s_X, ws, cs);
        if (x.t == x.tiles - 1) {
          const uint32_t total = s_X + __popc(fw0);
          const bool last_changed = (fw0 >> (x.nb - 1 - x.k0)) & 1u;
          const int64_t body = body_bytes_of(x, B, total, last_changed);
          const int64_t bm = (x.nb + 7) / 8;
          // the shard's last tile found it compressed, so body + bm < 2*len
          if (body + bm < 2 * x.len)
            write_bitmap(p, x, epoch, body, bm);
          else if (tid == 0)
            record_status(p.ctl, kStatusInternal);
        }
      }
      if (tid == 0) bulk_wait_read_all();
      __syncthreads();
    }
  }
}

// ------------------------------------------------------------------------
// Receiver

// One CTA per rank: validate the descriptor, copy the bitmap into aligned
// words and write each word's exclusive popcount prefix.
__global__ void __launch_bounds__(kScanThreads) k_bitmap_scan(const DecompressParams p) {
  __shared__ uint32_t warp_tot[kScanThreads / 32];
  __shared__ uint32_t s_total;
  const int32_t r = blockIdx.x;
  const int tid = threadIdx.x;
  const Geometry& geo = p.geo;
  const int64_t len = shard_len_of(geo, r);
  const int64_t nb = (len + geo.B - 1) / geo.B;
  const int64_t bm = (nb + 7) / 8;
  const int64_t nw = (nb + 31) / 32;
  const ciera_desc d = p.descs[r];
  const uint8_t* payload = payload_of(p, r);
  // a payload from the pointer table must exist, and be 16-byte aligned for
  // the staged path's bulk copies
  const bool ptr_ok =
      !p.payload_ptrs || (payload && !(p.fast && (reinterpret_cast<uintptr_t>(payload) & 15u)));

  // the same decision in every thread of the CTA
  uint32_t state = kRankSkip;
  if (d.mode == CIERA_MODE_RAW) {
    if (d.body_bytes == static_cast<uint64_t>(2 * len) && d.payload_bytes == d.body_bytes &&
        d.n_changed_blocks <= nb)
      state = kRankRaw;
  } else if (d.mode == CIERA_MODE_COMPRESSED && len > 0) {
    if (d.body_bytes >= static_cast<uint64_t>(len) &&
        d.payload_bytes == d.body_bytes + static_cast<uint64_t>(bm) &&
        d.payload_bytes < static_cast<uint64_t>(2 * len) &&
        d.payload_bytes <= static_cast<uint64_t>(p.stride))
      state = kRankCompressed;
  } else if (d.mode == kModeRans && p.rans && len > 0) {
    if (d.body_bytes == static_cast<uint64_t>(rans_layout(len, nb).D) &&
        d.payload_bytes >= d.body_bytes && d.payload_bytes <= static_cast<uint64_t>(p.stride))
      state = kRankRans;
  }
  if (!ptr_ok) state = kRankSkip;
  uint32_t table_bad = 0;
  if (state == kRankRans) {
    // the frequency table: no zero entry, sum 4096 (2 entries per thread)
    const uint8_t* tab = payload + rans_layout(len, nb).C;
    if (tid < 128) {
      const uint32_t f0 = tab[4 * tid] | (static_cast<uint32_t>(tab[4 * tid + 1]) << 8);
      const uint32_t f1 = tab[4 * tid + 2] | (static_cast<uint32_t>(tab[4 * tid + 3]) << 8);
      if (f0 == 0 || f1 == 0) table_bad = 1;
      if (tid == 0) s_total = 0;
      __syncwarp();
    }
    __syncthreads();
    if (tid < 128) {
      const uint32_t f0 = tab[4 * tid] | (static_cast<uint32_t>(tab[4 * tid + 1]) << 8);
      const uint32_t f1 = tab[4 * tid + 2] | (static_cast<uint32_t>(tab[4 * tid + 3]) << 8);
      atomicAdd(&s_total, f0 + f1);
    }
    __syncthreads();
    if (s_total != 4096u) table_bad = 1;
    __syncthreads();
  }
  if (state == kRankCompressed || state == kRankRans) {
    const bool rans = state == kRankRans;
    const uint8_t* bitmap = payload + (rans ? rans_layout(len, nb).A : d.body_bytes);
    uint32_t* words = p.bm_words + static_cast<int64_t>(r) * p.nw_stride;
    uint32_t* pre = p.bm_prefix + static_cast<int64_t>(r) * p.nw_stride;
    const int64_t per = (nw + kScanThreads - 1) / kScanThreads;
    const int64_t lo = tid * per < nw ? tid * per : nw;
    const int64_t hi = lo + per < nw ? lo + per : nw;
    uint32_t local = 0;
    uint32_t pad_bad = 0;
    for (int64_t i = lo; i < hi; ++i) {
      uint32_t word = 0;
      for (int j = 0; j < 4; ++j) {
        const int64_t b = 4 * i + j;
        if (b < bm && in_bounds(p.ctl, (bitmap - payload) + b, 1, p.stride))
          word |= static_cast<uint32_t>(bitmap[b]) << (8 * j);
      }
      if (i == nw - 1 && (nb & 31)) {
        // bits past the last block must be zero
        pad_bad = (word >> (nb & 31)) != 0;
        word &= 0xffffffffu >> (32 - (nb & 31));
      }
      words[i] = word;
      local += __popc(word);
    }
    // block-wide exclusive scan of the per-thread popcounts
    const int lane = tid & 31, wid = tid >> 5;
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    uint32_t wbase = 0;
    for (int i = 0; i < wid; ++i) wbase += warp_tot[i];
    if (tid == kScanThreads - 1) s_total = wbase + incl;
    uint32_t run = wbase + incl - local;
    for (int64_t i = lo; i < hi; ++i) {
      pre[i] = run;
      run += __popc(words[i]);
    }
    const uint32_t any_pad_bad = __syncthreads_or(pad_bad || table_bad);
    if (tid == 0) {
      const uint32_t total = s_total;
      const int64_t last_len = len - (nb - 1) * geo.B;
      const bool last_changed = (words[nw - 1] >> ((nb - 1) & 31)) & 1u;
      const int64_t changed_vals =
          static_cast<int64_t>(total) * geo.B - (last_changed ? geo.B - last_len : 0);
      const bool consistent =
          !any_pad_bad && total == d.n_changed_blocks &&
          (rans || d.body_bytes == static_cast<uint64_t>(len + changed_vals));
      if (!consistent) state = kRankSkip;
    }
  }
  if (tid == 0) {
    if (state == kRankSkip) atomicOr(&p.ctl->status, kStatusCorrupt);
    p.rank_state[r] = state;
  }
}

struct DecompressShared {
  uint32_t X;
  uint32_t bad;
  uint32_t fw[2];  // flag bits of the tile's blocks (staged path: T <= 32)
};

// Byte-wise tile of the receiver.
__device__ void decompress_tile_bytes(const DecompressParams& p, const Tile& x, uint32_t state) {
  const int64_t B = p.geo.B;
  const uint8_t* payload = payload_of(p, x.rl);
  uint8_t* rc = p.rcache + x.shard_off + x.e0;
  uint16_t* out = p.out + x.shard_off + x.e0;
  if (state == kRankRaw) {
    for (int64_t j = threadIdx.x; j < x.te; j += blockDim.x) {
      const int64_t o = 2 * (x.e0 + j);
      if (!in_bounds(p.ctl, o, 2, p.stride)) continue;
      const uint32_t v = payload[o] | (static_cast<uint32_t>(payload[o + 1]) << 8);
      out[j] = static_cast<uint16_t>(v);
      rc[j] = static_cast<uint8_t>(exp1(v));
    }
    return;
  }
  const uint32_t* words = p.bm_words + static_cast<int64_t>(x.rl) * p.nw_stride;
  const uint32_t* pre = p.bm_prefix + static_cast<int64_t>(x.rl) * p.nw_stride;
  for (int64_t j = threadIdx.x; j < x.te; j += blockDim.x) {
    const int64_t kg = x.k0 + j / B;
    const int64_t within = x.e0 + j - kg * B;
    const uint32_t word = words[kg >> 5];
    const uint32_t bit = static_cast<uint32_t>(kg & 31);
    const uint32_t C = pre[kg >> 5] + __popc(word & (bit ? (0xffffffffu >> (32 - bit)) : 0u));
    const int64_t off = (kg + C) * B;
    if ((word >> bit) & 1u) {
      const int64_t o = off + 2 * within;
      if (!in_bounds(p.ctl, o, 2, p.stride)) continue;
      const uint32_t v = payload[o] | (static_cast<uint32_t>(payload[o + 1]) << 8);
      out[j] = static_cast<uint16_t>(v);
      rc[j] = static_cast<uint8_t>(exp1(v));
    } else if (in_bounds(p.ctl, off + within, 1, p.stride)) {
      out[j] = static_cast<uint16_t>(join1(payload[off + within], rc[j]));
    }
  }
}

// Staged tile of the receiver.  Shared memory: ws[2*TE] | ss[TE] | cs[TE].
__device__ void decompress_tile_staged(const DecompressParams& p, const Tile& x, uint32_t state,
                                       DecompressShared& sh, uint8_t* dsm, uint64_t* bar) {
  const int tid = threadIdx.x;
  const int64_t B = p.geo.B;
  const int64_t TE = p.geo.T * B;
  uint8_t* ws = dsm;
  uint8_t* ss = dsm + 2 * TE;
  uint8_t* cs = dsm + 3 * TE;
  const uint8_t* payload = payload_of(p, x.rl);
  uint8_t* rc = p.rcache + x.shard_off + x.e0;
  uint16_t* out = p.out + x.shard_off + x.e0;
  const uint32_t te = static_cast<uint32_t>(x.te);
  const bool raw = state == kRankRaw;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    if (raw) {
      sh.fw[0] = 0xffffffffu;
      sh.X = 0;
      mbar_arrive_expect_tx(bar, 2u * te);
      if (in_bounds(p.ctl, 2 * x.e0, 2 * te, p.stride)) bulk_g2s(ws, payload + 2 * x.e0, 2u * te, bar);
    } else {
      // flag bits of blocks k0 .. k0+nblk-1 (nblk <= 32, may straddle a word)
      const uint32_t* words = p.bm_words + static_cast<int64_t>(x.rl) * p.nw_stride;
      const uint32_t* pre = p.bm_prefix + static_cast<int64_t>(x.rl) * p.nw_stride;
      const int64_t wi = x.k0 >> 5;
      const uint32_t sh0 = static_cast<uint32_t>(x.k0 & 31);
      const uint64_t two = static_cast<uint64_t>(words[wi]) |
                           ((wi + 1 < (x.nb + 31) / 32) ? static_cast<uint64_t>(words[wi + 1]) << 32
                                                        : 0ull);
      const uint32_t fw = static_cast<uint32_t>(two >> sh0) &
                          (x.nblk >= 32 ? 0xffffffffu : ((1u << x.nblk) - 1u));
      const uint32_t X =
          pre[wi] + __popc(words[wi] & (sh0 ? (0xffffffffu >> (32 - sh0)) : 0u));
      sh.fw[0] = fw;
      sh.X = X;
      // a changed value brings 2 payload bytes, a kept one 1 payload byte
      // and 1 cached exponent: 2 bytes of shared memory per value either way
      uint32_t before = 0;
      int ka = 0;
      mbar_arrive_expect_tx(bar, 2u * te);
      while (ka < x.nblk) {
        const bool f = (fw >> ka) & 1u;
        int kz = ka + 1;
        while (kz < x.nblk && (((fw >> kz) & 1u) != 0) == f) ++kz;
        const int64_t ea = static_cast<int64_t>(ka) * B;
        const int64_t ez = static_cast<int64_t>(kz) * B < x.te ? static_cast<int64_t>(kz) * B : x.te;
        const int64_t off = (x.k0 + ka + X + before) * B;
        if (f) {
          if (in_bounds(p.ctl, off, 2 * (ez - ea), p.stride))
            bulk_g2s(ws + 2 * ea, payload + off, static_cast<uint32_t>(2 * (ez - ea)), bar);
          before += static_cast<uint32_t>(kz - ka);
        } else {
          if (in_bounds(p.ctl, off, ez - ea, p.stride))
            bulk_g2s(ss + ea, payload + off, static_cast<uint32_t>(ez - ea), bar);
          bulk_g2s(cs + ea, rc + ea, static_cast<uint32_t>(ez - ea), bar);
        }
        ka = kz;
      }
    }
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(bar, 0, p.timeout_ns);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) record_status(p.ctl, kStatusTimeout);
    mbar_wait_bounded(bar, 0, p.timeout_ns);
    __syncthreads();
    return;
  }
  const uint32_t fw = sh.fw[0];
  const int ngroups = static_cast<int>(te >> 4);
  const uint32_t mG = group_divisor(B);
  for (int gi = tid; gi < ngroups; gi += blockDim.x) {
    const int kb = block_of_group(gi, mG);
    if (raw || ((fw >> kb) & 1u)) {
      const uint4 w0 = reinterpret_cast<const uint4*>(ws)[2 * gi];
      const uint4 w1 = reinterpret_cast<const uint4*>(ws)[2 * gi + 1];
      reinterpret_cast<uint4*>(rc)[gi] = make_uint4(exp4(w0.x, w0.y), exp4(w0.z, w0.w),
                                                    exp4(w1.x, w1.y), exp4(w1.z, w1.w));
    } else {
      const uint4 s = reinterpret_cast<const uint4*>(ss)[gi];
      const uint4 e = reinterpret_cast<const uint4*>(cs)[gi];
      const uint2 v0 = join4(s.x, e.x), v1 = join4(s.y, e.y);
      const uint2 v2 = join4(s.z, e.z), v3 = join4(s.w, e.w);
      reinterpret_cast<uint4*>(ws)[2 * gi] = make_uint4(v0.x, v0.y, v1.x, v1.y);
      reinterpret_cast<uint4*>(ws)[2 * gi + 1] = make_uint4(v2.x, v2.y, v3.x, v3.y);
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {
    bulk_s2g(out, ws, 2u * te);
    bulk_commit();
    bulk_wait_read_all();
  }
}

__global__ void __launch_bounds__(kThreads) k_decompress(const DecompressParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ DecompressShared sh;
  __shared__ __align__(8) uint64_t bar;
  const Tile x = decode_tile(p.geo, blockIdx.x);
  if (p.fast && dynamic_smem_size() < static_cast<uint32_t>(4 * p.geo.T * p.geo.B)) {
    if (threadIdx.x == 0) atomicOr(&p.ctl->status, kStatusInternal);
    return;
  }
  const uint32_t state = p.rank_state[x.rl];
  if (state != kRankRaw && state != kRankCompressed) return;  // RANS ranks: k_decompress_rans
  if (p.fast && (x.te & 15) == 0)
    decompress_tile_staged(p, x, state, sh, dsm, &bar);
  else
    decompress_tile_bytes(p, x, state);
}

// Largest dynamic shared memory already allowed per device and kernel.
constexpr int kMaxDevices = 64;
std::atomic<int64_t> g_compress_smem[kMaxDevices];
std::atomic<int64_t> g_compress_hashed_smem[kMaxDevices];
std::atomic<int64_t> g_decompress_smem[kMaxDevices];
std::atomic<int64_t> g_repack_smem[kMaxDevices];
std::atomic<int> g_sms[kMaxDevices];

// Multiprocessors of the current device (looked up once per device).
cudaError_t sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDevices) {
    const int c = g_sms[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *out = c;
      return cudaSuccess;
    }
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDevices) g_sms[dev].store(n, std::memory_order_relaxed);
  *out = n;
  return cudaSuccess;
}

// Opt the kernel in to `bytes` of dynamic shared memory on the current
// device (the default limit, static + dynamic, is 48 KB).
cudaError_t allow_dynamic_smem(const void* fn, int64_t bytes, std::atomic<int64_t>* done) {
  if (bytes <= 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDevices && done[dev].load(std::memory_order_relaxed) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes));
  if (e == cudaSuccess && dev < kMaxDevices) {
    int64_t cur = done[dev].load(std::memory_order_relaxed);
    while (cur < bytes && !done[dev].compare_exchange_weak(cur, bytes)) {
    }
  }
  return e;
}

}  // namespace

int launch_compress(const CompressParams& p, int64_t smem_bytes, int raw_fixup,
                    int64_t repack_smem, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* fn = p.hashed ? reinterpret_cast<const void*>(k_compress<true>)
                            : reinterpret_cast<const void*>(k_compress<false>);
  cudaError_t e =
      allow_dynamic_smem(fn, smem_bytes, p.hashed ? g_compress_hashed_smem : g_compress_smem);
  if (e != cudaSuccess) return e;
  // one CTA per tile, plus the last ticket (descriptors of empty shards)
  const int64_t grid = p.geo.total_tiles + 1;
  if (p.hashed)
    k_compress<true>
        <<<static_cast<unsigned>(grid), kThreads, static_cast<size_t>(smem_bytes), s>>>(p);
  else
    k_compress<false>
        <<<static_cast<unsigned>(grid), kThreads, static_cast<size_t>(smem_bytes), s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.raw_ahead && p.geo.total_tiles > 0) {
    e = allow_dynamic_smem(reinterpret_cast<const void*>(k_repack), repack_smem, g_repack_smem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = sm_count(&sms);
    if (e != cudaSuccess) return e;
    const int64_t cap = 4 * static_cast<int64_t>(sms);
    const int64_t grid = p.geo.total_tiles < cap ? p.geo.total_tiles : cap;
    k_repack<<<static_cast<unsigned>(grid), kThreads, static_cast<size_t>(repack_smem), s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (raw_fixup && p.geo.total_tiles > 0) {
    k_raw_fixup<<<static_cast<unsigned>(p.geo.total_tiles), kThreads, 0, s>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

int launch_decompress(const DecompressParams& p, int64_t smem_bytes, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(k_decompress), smem_bytes,
                                     g_decompress_smem);
  if (e != cudaSuccess) return e;
  if (p.geo.rank_count > 0) {
    k_bitmap_scan<<<static_cast<unsigned>(p.geo.rank_count), kScanThreads, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.geo.total_tiles > 0) {
    k_decompress<<<static_cast<unsigned>(p.geo.total_tiles), kThreads,
                   static_cast<size_t>(smem_bytes), s>>>(p);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace ciera
