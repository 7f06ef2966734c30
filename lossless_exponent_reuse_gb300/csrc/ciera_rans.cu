// ciera_rans.cu -- RANS payloads: the exponents of changed blocks coded with
// rANS on sm_103a.
//
// Method: "CIERA: Cross-Iteration Exponent Reuse for Lossless Allgather in
// Sharded MoE Training", Section 3.1: the sender sends the sign+mantissa
// bytes of every block and the changed exponents entropy-coded with ANS; the
// receiver decodes them, patches its ExpCache and merges.  The coder is an
// own range variant of ANS (Duda, "Asymmetric numeral systems"): 12-bit
// probabilities, a 32-bit state kept in [2^16, 2^32) and renormalised 16 bits
// at a time, 32 interleaved lanes per block (lane l codes positions l,
// l+32, ...), so one warp codes or decodes one block.
//
// Payload of a shard (len values, nb blocks; rans_layout):
//   [0, len)   sign+mantissa byte of every value, at its own position
//   A          bitmap of changed blocks
//   C          frequency table, 256 uint16 summing to 4096
//   O          nb + 1 uint32: bytes of the records of the blocks before k
//   D          records of the changed blocks: 32 uint16 lane word counts,
//              then the lanes' words in decoding order, padded to 16 bytes
// The table is normalised from the histogram of the shard's exponents one
// iteration earlier, which the previous call accumulated as a by-product.
//
// Kernels:
//   k_compress_rans    one CTA per tile, ticket order: flags (exact test)
//                      and the exponent histogram, cache refresh, sign+
//                      mantissa bytes to their fixed positions, one warp
//                      per changed block codes it, decoupled look-back over
//                      the record sizes places the records.
//   k_rans_raw_fixup   rewrites a shard raw when its RANS payload would not
//                      have been smaller than the raw bytes.
//   k_decompress_rans  one CTA per tile of a RANS rank: bulk copies of the
//                      sign+mantissa bytes, cached exponents, table and
//                      records; one warp per changed block decodes it; merge;
//                      ExpCache refresh.
#include <cuda_runtime.h>

#include <atomic>

#include "ciera_device.cuh"
#include "ciera_internal.h"
#include "ciera_rans.h"

namespace ciera {
namespace {

constexpr int kRansBits = 12;
constexpr uint32_t kRansTotal = 1u << kRansBits;
constexpr uint32_t kRansLow = 1u << 16;

// ---- meta region offsets (bytes) inside the first kRansMetaBytes ----------
// compress
constexpr int kCFw = 0;          // uint32 flag bits of the tile (T <= 32)
constexpr int kCFreq = 16;       // uint16[256]
constexpr int kCCum = 544;       // uint32[257]
constexpr int kCHist = 1584;     // uint32[256] exponent histogram of the tile
constexpr int kCSize = 2624;     // uint32[32] record size of each block, 16-byte units
constexpr int kCPre = 2752;      // uint32[33] exclusive prefix of the sizes
constexpr int kCRed = 2896;      // uint64[8] reductions
// decompress
constexpr int kDFreq = 0;        // uint16[256], bulk-copied from the payload
constexpr int kDCum = 512;       // uint32[257]
constexpr int kDOffs = 1552;     // uint32[33] record-byte prefixes of the tile's blocks
constexpr int kDRed = 1696;      // uint64[8]
constexpr int kDSlot = 2048;     // uint8[4096] slot -> symbol
static_assert(kDSlot + 4096 <= kRansMetaBytes, "meta region");
static_assert(kCRed + 64 <= kRansMetaBytes, "meta region");

// Block-wide sum over all 128 threads (uses red[0..3]; ends with a barrier).
__device__ __forceinline__ unsigned long long block_sum(unsigned long long v,
                                                        unsigned long long* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  const unsigned long long t = red[0] + red[1] + red[2] + red[3];
  __syncthreads();
  return t;
}

__device__ __forceinline__ unsigned long long block_max(unsigned long long v,
                                                        unsigned long long* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = red[0];
  for (int i = 1; i < 4; ++i) t = red[i] > t ? red[i] : t;
  __syncthreads();
  return t;
}

// Exclusive scan of `v` over the 128 threads (uses red[4..7]).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, unsigned long long* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) red[4 + wid] = incl;
  __syncthreads();
  uint32_t base = 0;
  for (int i = 0; i < wid; ++i) base += static_cast<uint32_t>(red[4 + i]);
  __syncthreads();
  return base + incl - v;
}

// Frequency table from a histogram (all 128 threads; symbols 2t, 2t+1 per
// thread): f = 1 + floor(h * 3840 / sum h), the rest of 4096 to the most
// frequent symbol (lowest on a tie), 16 each for an empty histogram.
__device__ void build_table(const uint32_t* h, uint16_t* freq, uint32_t* cum,
                            unsigned long long* red) {
  const int t = threadIdx.x;
  const uint32_t h0 = h[2 * t], h1 = h[2 * t + 1];
  const unsigned long long total = block_sum(static_cast<unsigned long long>(h0) + h1, red);
  uint32_t f0 = 16, f1 = 16;
  if (total) {
    f0 = 1u + static_cast<uint32_t>(static_cast<unsigned long long>(h0) * 3840ull / total);
    f1 = 1u + static_cast<uint32_t>(static_cast<unsigned long long>(h1) * 3840ull / total);
    const unsigned long long sum = block_sum(f0 + f1, red);
    // largest count, lowest symbol on a tie
    const unsigned long long k0 = (static_cast<unsigned long long>(h0) << 8) | (255u - 2 * t);
    const unsigned long long k1 = (static_cast<unsigned long long>(h1) << 8) | (254u - 2 * t);
    const unsigned long long best = block_max(k0 > k1 ? k0 : k1, red);
    const uint32_t bs = 255u - static_cast<uint32_t>(best & 255u);
    const uint32_t rem = kRansTotal - static_cast<uint32_t>(sum);
    if (bs == 2u * t) f0 += rem;
    if (bs == 2u * t + 1) f1 += rem;
  }
  freq[2 * t] = static_cast<uint16_t>(f0);
  freq[2 * t + 1] = static_cast<uint16_t>(f1);
  const uint32_t c = block_exclusive_scan(f0 + f1, red);
  cum[2 * t] = c;
  cum[2 * t + 1] = c + f0;
  if (t == 0) cum[256] = kRansTotal;
  __syncthreads();
}

// One warp codes one block of L values (their exponents) into `rec`: lane
// counts at rec[0..31], lane regions of LW words from rec[32]; then the
// streams are compacted in place behind the counts and padded to 16 bytes.
// Returns the record size in 16-byte units.
__device__ uint32_t rans_encode_block(const uint16_t* vals, int64_t L, const uint16_t* freq,
                                      const uint32_t* cum, uint16_t* rec, int64_t LW, int lane) {
  uint16_t* region = rec + kRansLanes + lane * LW;
  int64_t top = LW;
  uint32_t x = kRansLow;
  if (lane < L) {
    for (int64_t j = lane + ((L - 1 - lane) / kRansLanes) * kRansLanes; j >= 0; j -= kRansLanes) {
      const uint32_t sym = exp1(vals[j]);
      const uint32_t f = freq[sym];
      if (static_cast<unsigned long long>(x) >= (static_cast<unsigned long long>(f) << 20)) {
        region[--top] = static_cast<uint16_t>(x & 0xFFFFu);
        x >>= 16;
      }
      x = ((x / f) << kRansBits) + (x % f) + cum[sym];
    }
  }
  region[--top] = static_cast<uint16_t>(x & 0xFFFFu);
  region[--top] = static_cast<uint16_t>(x >> 16);
  const uint32_t nw = static_cast<uint32_t>(LW - top);
  rec[lane] = static_cast<uint16_t>(nw);
  uint32_t incl = nw;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  const uint32_t pre = incl - nw;
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  __syncwarp();
  // lane l's words move from its region's tail to 32 + prefix(l): never to a
  // higher index, and never over a later lane's words
  for (int l = 0; l < kRansLanes; ++l) {
    const uint32_t n = __shfl_sync(0xffffffffu, nw, l);
    const uint32_t p0 = __shfl_sync(0xffffffffu, pre, l);
    const int64_t src = kRansLanes + l * LW + (LW - n);
    const int64_t dst = kRansLanes + p0;
    for (uint32_t c = 0; c < n; c += 32) {
      const bool ok = c + lane < n;
      uint16_t v = 0;
      if (ok) v = rec[src + c + lane];
      __syncwarp();
      if (ok) rec[dst + c + lane] = v;
      __syncwarp();
    }
  }
  const uint32_t words = kRansLanes + total;
  const uint32_t padded = (words + 7u) & ~7u;
  if (words + lane < padded) rec[words + lane] = 0;
  __syncwarp();
  return padded / 8u;
}

// One warp decodes one record of `rec_words` words into L exponents.
// False (for the whole warp) if the record does not decode cleanly.
__device__ bool rans_decode_block(const uint16_t* rec, uint32_t rec_words, int64_t L,
                                  const uint16_t* freq, const uint32_t* cum,
                                  const uint8_t* slot_sym, uint8_t* exps, int lane) {
  const uint32_t nw = rec_words >= kRansLanes ? rec[lane] : 0u;
  uint32_t incl = nw;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  const uint32_t pre = incl - nw;
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  bool bad = rec_words < kRansLanes || kRansLanes + total > rec_words || nw < 2;
  if (__any_sync(0xffffffffu, bad)) return false;
  const uint16_t* s = rec + kRansLanes + pre;
  uint32_t x = (static_cast<uint32_t>(s[0]) << 16) | s[1];
  uint32_t idx = 2;
  for (int64_t j = lane; j < L; j += kRansLanes) {
    const uint32_t slot = x & (kRansTotal - 1);
    const uint32_t sym = slot_sym[slot];
    exps[j] = static_cast<uint8_t>(sym);
    x = static_cast<uint32_t>(freq[sym]) * (x >> kRansBits) + slot - cum[sym];
    if (x < kRansLow) {
      if (idx >= nw) {
        bad = true;
        break;
      }
      x = (x << 16) | s[idx++];
    }
  }
  bad = bad || idx != nw || x != kRansLow;
  return !__any_sync(0xffffffffu, bad);
}

struct RansShared {
  uint32_t ticket;
  uint32_t epoch;  // this launch's tag of look-back and flag words
  uint32_t X;      // record units (16 bytes) before the tile in its shard
  uint32_t agg;    // record units of the tile
  uint32_t bad;    // a bounded wait ran out on this tile
};

__global__ void __launch_bounds__(kThreads)
    k_compress_rans(const CompressParams p, const uint32_t* __restrict__ hist_prev,
                    uint32_t* __restrict__ hist_out) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ RansShared sh;
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t B = p.geo.B;
  const int64_t T = p.geo.T;
  const int64_t TE = T * B;
  uint32_t* fw = reinterpret_cast<uint32_t*>(dsm + kCFw);
  uint16_t* freq = reinterpret_cast<uint16_t*>(dsm + kCFreq);
  uint32_t* cum = reinterpret_cast<uint32_t*>(dsm + kCCum);
  uint32_t* hist = reinterpret_cast<uint32_t*>(dsm + kCHist);
  uint32_t* rsize = reinterpret_cast<uint32_t*>(dsm + kCSize);
  uint32_t* rpre = reinterpret_cast<uint32_t*>(dsm + kCPre);
  unsigned long long* red = reinterpret_cast<unsigned long long*>(dsm + kCRed);
  uint8_t* ws = dsm + kRansMetaBytes;  // values [2 TE]
  uint8_t* cs = ws + 2 * TE;           // cached exponents, then sign+mantissa bytes [TE]
  uint8_t* scr = cs + TE;              // one record buffer per block [T * BB]
  const int64_t LW = rans_lane_words(B);
  const int64_t BB = rans_block_bytes(B);

  if (tid == 0) {
    const unsigned long long v = atomicAdd(&p.ctl->ticket, 1ull);
    const uint32_t t = static_cast<uint32_t>(v);
    const uint32_t launch = static_cast<uint32_t>(v >> 32);
    if (t == gridDim.x - 1)
      atomicExch(&p.ctl->ticket, static_cast<unsigned long long>(launch + 1u) << 32);
    sh.ticket = t;
    sh.epoch = launch % 0xffffffffu + 1u;
    sh.bad = 0;
    fw[0] = 0;
  }
  if (dynamic_smem_size() < static_cast<uint32_t>(rans_compress_smem(T, B)) || T > 32 ||
      !p.fast) {
    if (tid == 0) record_status(p.ctl, kStatusInternal);
    return;
  }
  for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
  if (tid < 32) rsize[tid] = 0;
  __syncthreads();
  const int64_t g = sh.ticket;
  if (g >= p.geo.total_tiles) {
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
  const bool cold = p.flags & CIERA_COLD;
  const RansLayout Ly = rans_layout(x.len, x.nb);
  // a shard whose sections alone are not smaller than its raw bytes, or a
  // cold one, goes out raw whatever its records would be
  const bool direct_raw = cold || Ly.D >= 2 * x.len;
  const uint16_t* w = p.w + x.shard_off + x.e0;
  uint8_t* c = p.scache + x.shard_off + x.e0;
  const uint32_t te = static_cast<uint32_t>(x.te);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(&bar, 3u * te);
    bulk_g2s(ws, w, 2u * te, &bar);
    bulk_g2s(cs, c, te, &bar);
  }
  __syncthreads();
  // this shard's table, from its exponent histogram one iteration earlier
  build_table(hist_prev + 256 * static_cast<int64_t>(x.rl), freq, cum, red);

  const int ngroups = static_cast<int>(te >> 4);
  if (warp == 0) {
    bool to = false;
    const uint32_t X =
        direct_raw ? 0u : lookback_exclusive(p, x, sh.epoch, lane, x.k0 * (BB / 16), &to);
    if (lane == 0) {
      sh.X = X;
      if (to) record_status(p.ctl, kStatusTimeout);
    }
  } else {
    const int ft = tid - 32;
    if (!mbar_wait_bounded(&bar, 0, p.timeout_ns)) {
      record_status(p.ctl, kStatusTimeout);
      sh.bad = 1;
      mbar_wait_bounded(&bar, 0, p.timeout_ns);
    }
    flaggers_sync();
    const bool all = cold || sh.bad;
    // flags (exact test) and the tile's exponent histogram; the loop runs
    // whole warps so that equal exponents can be merged across lanes
    uint32_t mine = 0;
    for (int g0 = ft - lane; g0 < ngroups; g0 += kThreads - 32) {
      const int gi = g0 + lane;
      const bool in = gi < ngroups;
      uint32_t e[4] = {0x100u, 0x100u, 0x100u, 0x100u};
      if (in) {
        const uint4 w0 = reinterpret_cast<const uint4*>(ws)[2 * gi];
        const uint4 w1 = reinterpret_cast<const uint4*>(ws)[2 * gi + 1];
        const uint4 cc = reinterpret_cast<const uint4*>(cs)[gi];
        e[0] = exp4(w0.x, w0.y);
        e[1] = exp4(w0.z, w0.w);
        e[2] = exp4(w1.x, w1.y);
        e[3] = exp4(w1.z, w1.w);
        const uint32_t d = (e[0] ^ cc.x) | (e[1] ^ cc.y) | (e[2] ^ cc.z) | (e[3] ^ cc.w);
        if (d || all) mine |= 1u << static_cast<int>((static_cast<int64_t>(gi) << 4) / B);
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const uint32_t v = in ? (e[q >> 2] >> (8 * (q & 3))) & 0xFFu : 0x100u + lane;
        const uint32_t same = __match_any_sync(0xffffffffu, v);
        if (in && lane == __ffs(same) - 1) atomicAdd(&hist[v], static_cast<uint32_t>(__popc(same)));
      }
    }
    mine = __reduce_or_sync(0xffffffffu, mine);
    if (lane == 0 && mine) atomicOr(&fw[0], mine);
    flaggers_sync();
    const uint32_t f = fw[0];
    // sender cache of changed blocks; every value's sign+mantissa byte into cs
    for (int gi = ft; gi < ngroups; gi += kThreads - 32) {
      const uint4 w0 = reinterpret_cast<const uint4*>(ws)[2 * gi];
      const uint4 w1 = reinterpret_cast<const uint4*>(ws)[2 * gi + 1];
      const int kb = static_cast<int>((static_cast<int64_t>(gi) << 4) / B);
      if ((f >> kb) & 1u) {
        const uint4 e = make_uint4(exp4(w0.x, w0.y), exp4(w0.z, w0.w), exp4(w1.x, w1.y),
                                   exp4(w1.z, w1.w));
        const uint4 cc = reinterpret_cast<const uint4*>(cs)[gi];
        if (all || ((e.x ^ cc.x) | (e.y ^ cc.y) | (e.z ^ cc.z) | (e.w ^ cc.w)))
          reinterpret_cast<uint4*>(c)[gi] = e;
      }
      if (!direct_raw)
        reinterpret_cast<uint4*>(cs)[gi] =
            make_uint4(sm4(w0.x, w0.y), sm4(w0.z, w0.w), sm4(w1.x, w1.y), sm4(w1.z, w1.w));
    }
    // code the changed blocks: the i-th changed block goes to warp 1 + i % 3
    if (!direct_raw) {
      int i = 0;
      for (int kb = 0; kb < x.nblk; ++kb) {
        if (!((f >> kb) & 1u)) continue;
        if (i % (kThreads / 32 - 1) == warp - 1) {
          const int64_t L = (kb + 1) * B < x.te ? B : x.te - kb * B;
          const uint32_t units =
              rans_encode_block(reinterpret_cast<const uint16_t*>(ws) + kb * B, L, freq, cum,
                                reinterpret_cast<uint16_t*>(scr + kb * BB), LW, lane);
          if (lane == 0) rsize[kb] = units;
        }
        ++i;
      }
    }
    flaggers_sync();
    if (ft == 0) {
      const uint32_t fm = f & (x.nblk >= 32 ? 0xffffffffu : ((1u << x.nblk) - 1u));
      uint8_t* fb = p.flagbytes + static_cast<int64_t>(x.rl) * p.flag_stride + x.k0;
      uint32_t run = 0;
      for (int kb = 0; kb < x.nblk; ++kb) {
        fb[kb] = (fm >> kb) & 1u;
        rpre[kb] = run;
        run += rsize[kb];
      }
      rpre[x.nblk] = run;
      sh.agg = run;
      st_relaxed_u64(&p.tile_flags[x.sidx], (static_cast<unsigned long long>(sh.epoch) << 32) | fm);
      const bool skip = (p.flags & CIERA_DEBUG_SKIP_FIRST_PUBLISH) && x.t == 0;
      if (!direct_raw && !skip)
        publish(p, x, sh.epoch, x.t == 0 ? kStateInclusive : kStateAggregate, run);
    }
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (tid == 0 && x.t > 0 && !direct_raw) publish(p, x, sh.epoch, kStateInclusive, sh.X + sh.agg);

  uint8_t* payload = p.payloads + static_cast<int64_t>(x.rl) * p.stride;
  const int64_t limit = 2 * x.len;  // a payload this large goes out raw instead
  if (tid == 0) {
    if (direct_raw) {
      bulk_s2g(payload + 2 * x.e0, ws, 2u * te);
    } else {
      bulk_s2g(payload + x.e0, cs, te);
      for (int kb = 0; kb < x.nblk; ++kb) {
        const int64_t at = Ly.D + 16 * static_cast<int64_t>(sh.X + rpre[kb]);
        if (rsize[kb] && at + 16 * static_cast<int64_t>(rsize[kb]) <= limit)
          bulk_s2g(payload + at, scr + kb * BB, 16u * rsize[kb]);
      }
    }
    bulk_commit();
  }
  if (!direct_raw) {
    uint32_t* O = reinterpret_cast<uint32_t*>(payload + Ly.O);
    if (tid < x.nblk) O[x.k0 + tid] = 16u * (sh.X + rpre[tid]);
    if (tid == 0 && x.t == x.tiles - 1) O[x.nb] = 16u * (sh.X + sh.agg);
  }
  uint32_t* ho = hist_out + 256 * static_cast<int64_t>(x.rl);
  for (int s = tid; s < 256; s += blockDim.x)
    if (hist[s]) atomicAdd(&ho[s], hist[s]);

  if (x.t == x.tiles - 1) {
    // descriptor, bitmap and table of the shard: the bitmap comes from every
    // tile's epoch-tagged flag word (polled, bounded)
    const int64_t pb = Ly.D + 16 * (static_cast<int64_t>(sh.X) + sh.agg);
    const bool raw = direct_raw || pb >= limit;
    const unsigned long long* tf = p.tile_flags + (x.sidx - x.t);
    const int64_t bm = (x.nb + 7) / 8;
    bool to = false;
    uint32_t nch = 0;
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
          if ((v >> 32) != sh.epoch) {
            const uint64_t t0 = globaltimer();
            while ((v >> 32) != sh.epoch) {
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
      nch += __popc(byte);
      if (!raw) payload[Ly.A + i] = static_cast<uint8_t>(byte);
    }
    if (to) record_status(p.ctl, kStatusTimeout);
    const uint32_t n_changed = static_cast<uint32_t>(block_sum(nch, red));
    if (!raw) {
      for (int s = tid; s < 256; s += blockDim.x)
        reinterpret_cast<uint16_t*>(payload + Ly.C)[s] = freq[s];
      // zero padding before the table and before the records
      for (int64_t i = Ly.A + bm + tid; i < Ly.C; i += blockDim.x) payload[i] = 0;
      for (int64_t i = Ly.O + 4 * (x.nb + 1) + tid; i < Ly.D; i += blockDim.x) payload[i] = 0;
    }
    if (tid == 0) {
      ciera_desc d;
      d.mode = raw ? CIERA_MODE_RAW : kModeRans;
      d.n_changed_blocks = n_changed;
      d.body_bytes = static_cast<uint64_t>(raw ? limit : Ly.D);
      d.payload_bytes = static_cast<uint64_t>(raw ? limit : pb);
      p.descs[x.rl] = d;
    }
  }
  if (tid == 0) bulk_wait_read_all();
}

// A shard that went raw only at the end (its RANS payload would not have
// been smaller than its raw bytes): rewrite it raw.  Shards that went raw
// from the start were written raw by k_compress_rans itself.
__global__ void __launch_bounds__(kThreads) k_rans_raw_fixup(const CompressParams p) {
  const Tile x = decode_tile(p.geo, blockIdx.x);
  if (p.descs[x.rl].mode != CIERA_MODE_RAW) return;
  if (rans_layout(x.len, x.nb).D >= 2 * x.len) return;
  const uint4* w = reinterpret_cast<const uint4*>(p.w + x.shard_off + x.e0);
  uint4* dst = reinterpret_cast<uint4*>(p.payloads + static_cast<int64_t>(x.rl) * p.stride +
                                        2 * x.e0);
  for (int64_t i = threadIdx.x; i < x.te / 8; i += blockDim.x) dst[i] = w[i];
}

__global__ void __launch_bounds__(kThreads) k_decompress_rans(const DecompressParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t s_fw, s_bad;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const Tile x = decode_tile(p.geo, blockIdx.x);
  if (p.rank_state[x.rl] != kRankRans) return;
  const int64_t B = p.geo.B;
  const int64_t T = p.geo.T;
  const int64_t TE = T * B;
  if (dynamic_smem_size() < static_cast<uint32_t>(rans_decompress_smem(T, B)) || T > 32 ||
      !p.fast) {
    if (tid == 0) atomicOr(&p.ctl->status, kStatusInternal);
    return;
  }
  uint16_t* freq = reinterpret_cast<uint16_t*>(dsm + kDFreq);
  uint32_t* cum = reinterpret_cast<uint32_t*>(dsm + kDCum);
  uint32_t* offs = reinterpret_cast<uint32_t*>(dsm + kDOffs);
  unsigned long long* red = reinterpret_cast<unsigned long long*>(dsm + kDRed);
  uint8_t* slot_sym = dsm + kDSlot;
  uint8_t* ss = dsm + kRansMetaBytes;  // sign+mantissa bytes [TE]
  uint8_t* cs = ss + TE;               // exponents: cached, then decoded [TE]
  uint8_t* ws = cs + TE;               // merged values [2 TE]
  uint8_t* recs = ws + 2 * TE;         // records [T * BB]
  const int64_t BB = rans_block_bytes(B);
  const ciera_desc d = p.descs[x.rl];
  const uint8_t* payload = p.payloads + static_cast<int64_t>(x.rl) * p.stride;
  const RansLayout Ly = rans_layout(x.len, x.nb);
  uint8_t* rc = p.rcache + x.shard_off + x.e0;
  const uint32_t te = static_cast<uint32_t>(x.te);
  if (tid <= x.nblk) offs[tid] = reinterpret_cast<const uint32_t*>(payload + Ly.O)[x.k0 + tid];
  __syncthreads();
  if (tid == 0) {
    // the tile's flag bits (from the aligned copy of the bitmap)
    const uint32_t* words = p.bm_words + static_cast<int64_t>(x.rl) * p.nw_stride;
    const int64_t wi = x.k0 >> 5;
    const uint32_t sh0 = static_cast<uint32_t>(x.k0 & 31);
    const uint64_t two = static_cast<uint64_t>(words[wi]) |
                         ((wi + 1 < (x.nb + 31) / 32) ? static_cast<uint64_t>(words[wi + 1]) << 32
                                                      : 0ull);
    uint32_t fw = static_cast<uint32_t>(two >> sh0) &
                  (x.nblk >= 32 ? 0xffffffffu : ((1u << x.nblk) - 1u));
    uint32_t bad = 0;
    uint32_t bytes = 2u * te;
    for (int kb = 0; kb < x.nblk; ++kb) {
      if (!((fw >> kb) & 1u)) continue;
      const uint32_t a = offs[kb], b = offs[kb + 1];
      // a record must be nonempty, lie inside the payload and, for the bulk
      // copy, start and end on 16 bytes and fit its buffer
      if (b <= a || (a & 15u) || (b & 15u) || b - a > BB ||
          static_cast<uint64_t>(Ly.D) + b > d.payload_bytes) {
        bad = 1;
        fw &= ~(1u << kb);
        continue;
      }
      bytes += b - a;
    }
    if (fw) bytes += 512u;
    s_fw = fw;
    s_bad = bad;
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(&bar, bytes);
    bulk_g2s(ss, payload + x.e0, te, &bar);
    bulk_g2s(cs, rc, te, &bar);
    if (fw) {
      bulk_g2s(freq, payload + Ly.C, 512u, &bar);
      for (int kb = 0; kb < x.nblk; ++kb)
        if ((fw >> kb) & 1u)
          bulk_g2s(recs + kb * BB, payload + Ly.D + offs[kb], offs[kb + 1] - offs[kb], &bar);
    }
  }
  __syncthreads();
  if (__syncthreads_or(!mbar_wait_bounded(&bar, 0, p.timeout_ns))) {
    if (tid == 0) atomicOr(&p.ctl->status, kStatusTimeout);
    mbar_wait_bounded(&bar, 0, p.timeout_ns);
    __syncthreads();
    return;
  }
  const uint32_t fw = s_fw;
  bool ok = true;
  if (fw) {
    // cumulative table (validated by the bitmap scan) and slot -> symbol
    // map: thread t fills slots 32t .. 32t+31
    const uint32_t f0 = freq[2 * tid], f1 = freq[2 * tid + 1];
    const uint32_t c0 = block_exclusive_scan(f0 + f1, red);
    cum[2 * tid] = c0;
    cum[2 * tid + 1] = c0 + f0;
    if (tid == kThreads - 1) cum[256] = c0 + f0 + f1;
    __syncthreads();
    const uint32_t j0 = 32u * tid;
    int lo = 0, hi = 255;  // the symbol of slot j0: largest s with cum[s] <= j0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cum[mid] <= j0) lo = mid; else hi = mid - 1;
    }
    uint32_t sym = static_cast<uint32_t>(lo);
    for (int q = 0; q < 8; ++q) {
      uint32_t word = 0;
      for (int b = 0; b < 4; ++b) {
        const uint32_t j = j0 + 4 * q + b;
        while (sym < 255 && cum[sym + 1] <= j) ++sym;
        word |= sym << (8 * b);
      }
      reinterpret_cast<uint32_t*>(slot_sym)[8 * tid + q] = word;
    }
    __syncthreads();
    // decode: the i-th changed block goes to warp i % 4
    int i = 0;
    for (int kb = 0; kb < x.nblk; ++kb) {
      if (!((fw >> kb) & 1u)) continue;
      if (i % (kThreads / 32) == warp) {
        const int64_t L = (kb + 1) * B < x.te ? B : x.te - kb * B;
        ok = rans_decode_block(reinterpret_cast<const uint16_t*>(recs + kb * BB),
                               (offs[kb + 1] - offs[kb]) / 2, L, freq, cum, slot_sym,
                               cs + kb * B, lane) && ok;
      }
      ++i;
    }
  }
  const uint32_t any_bad = __syncthreads_or(!ok);
  if (tid == 0 && (any_bad || s_bad)) atomicOr(&p.ctl->status, kStatusCorrupt);
  // merge; ExpCache refresh of the changed blocks
  const int ngroups = static_cast<int>(te >> 4);
  for (int gi = tid; gi < ngroups; gi += blockDim.x) {
    const int kb = static_cast<int>((static_cast<int64_t>(gi) << 4) / B);
    const uint4 s = reinterpret_cast<const uint4*>(ss)[gi];
    const uint4 e = reinterpret_cast<const uint4*>(cs)[gi];
    reinterpret_cast<uint4*>(ws)[2 * gi] =
        make_uint4(join2(s.x, e.x), join2(s.x >> 16, e.x >> 16), join2(s.y, e.y),
                   join2(s.y >> 16, e.y >> 16));
    reinterpret_cast<uint4*>(ws)[2 * gi + 1] =
        make_uint4(join2(s.z, e.z), join2(s.z >> 16, e.z >> 16), join2(s.w, e.w),
                   join2(s.w >> 16, e.w >> 16));
    if ((fw >> kb) & 1u) reinterpret_cast<uint4*>(rc)[gi] = e;
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {
    bulk_s2g(p.out + x.shard_off + x.e0, ws, 2u * te);
    bulk_commit();
    bulk_wait_read_all();
  }
}

constexpr int kMaxDevices = 64;
std::atomic<int64_t> g_smem_c[kMaxDevices];
std::atomic<int64_t> g_smem_d[kMaxDevices];

cudaError_t allow_smem(const void* fn, int64_t bytes, std::atomic<int64_t>* done) {
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

int launch_compress_rans(const CompressParams& p, const uint32_t* hist_prev, uint32_t* hist_out,
                         void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t smem = rans_compress_smem(p.geo.T, p.geo.B);
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(k_compress_rans), smem, g_smem_c);
  if (e != cudaSuccess) return e;
  const int64_t grid = p.geo.total_tiles + 1;
  k_compress_rans<<<static_cast<unsigned>(grid), kThreads, static_cast<size_t>(smem), s>>>(
      p, hist_prev, hist_out);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (!(p.flags & CIERA_COLD) && p.geo.total_tiles > 0) {
    k_rans_raw_fixup<<<static_cast<unsigned>(p.geo.total_tiles), kThreads, 0, s>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

int launch_decompress_rans(const DecompressParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.geo.total_tiles <= 0) return cudaSuccess;
  const int64_t smem = rans_decompress_smem(p.geo.T, p.geo.B);
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(k_decompress_rans), smem, g_smem_d);
  if (e != cudaSuccess) return e;
  k_decompress_rans<<<static_cast<unsigned>(p.geo.total_tiles), kThreads,
                      static_cast<size_t>(smem), s>>>(p);
  return cudaGetLastError();
}

}  // namespace ciera
