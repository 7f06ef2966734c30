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
// iteration earlier (every 16th value), which the previous call accumulated
// as a by-product.
//
// Kernels:
//   k_rans_enc_tables  one CTA per rank: frequencies from the histogram, and
//                      per symbol the constants of an exact division by its
//                      frequency (Granlund and Montgomery, "Division by
//                      invariant integers using multiplication", 1994), so
//                      that a coding step multiplies instead of dividing.
//   k_compress_rans    one CTA per tile, ticket order: the tile's values and
//                      cached exponents in bulk copies, one streaming pass
//                      (flags by the exact test, cache refresh, sign+mantissa
//                      bytes to their fixed positions, the tile's exponents
//                      into shared memory, the sampled histogram); one warp
//                      per changed block codes it; then a decoupled
//                      look-back over the record sizes places the records,
//                      assembled in shared memory and stored by one bulk
//                      copy per tile (lane by lane when they do not fit).
//   k_rans_raw_fixup   rewrites a shard raw when its RANS payload would not
//                      have been smaller than the raw bytes.
//   k_rans_dec_tables  one CTA per RANS rank: a slot -> (symbol, frequency,
//                      bias) table of 4096 entries from the received
//                      frequencies, so that a decoding step is one lookup.
//   k_decompress_rans  one CTA per receiver tile (rans_receiver_blocks: twice
//                      the sender's blocks).  RAW rank: the values stream from
//                      the payload to out and ExpCache.  RANS rank: bulk copies
//                      of the sign+mantissa bytes and the records; the kept
//                      blocks merge with their cached exponents; one warp per
//                      changed block decodes it (slot table copied into shared
//                      memory) straight into the output and the ExpCache.
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
constexpr int kTableThreads = 256;

// ---- shared-memory meta region of k_compress_rans (bytes) ----------------
constexpr int kCTab = 0;         // uint4[256] coder entries, then uint16[256] frequencies
constexpr int kCFreq = 4096;
constexpr int kCHist = 4608;     // uint32[256] sampled exponent histogram of the tile
constexpr int kCSize = 5632;     // uint32[32] record size of each block, 16-byte units
constexpr int kCPre = 5760;      // uint32[33] exclusive prefix of the sizes
constexpr int kCRed = 5904;      // uint32[8] reductions
constexpr int kCFw = 5936;       // uint32 flag bits of the tile (T <= 32)
static_assert(kCFw + 4 <= kRansEncMeta, "meta region");
static_assert(kRansEncMeta >= 2 * kRansLanes, "the coder's look-ahead reads below the exponents");
static_assert(kCFreq - kCTab + 512 == kRansEncTableBytes, "coder table layout");
// ---- k_decompress_rans ---------------------------------------------------
constexpr int kDOffs = 0;        // uint32[33] record-byte prefixes of the tile's blocks
static_assert(kDOffs + 4 * 33 <= kRansDecMeta, "meta region");

// Hint that the line holding p (global memory) be brought into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Coder entry of a symbol of frequency f and cumulative frequency c, for a
// coding step x -> x + q (4096 - f) + c with q = floor(x / f) (that is,
// q * 4096 + (x - q f) + c):
//   .x, .y  M = ceil(2^64 / f) as low and high words: for a state x < 2^32,
//           q = floor((x M_hi + mulhi(x, M_lo)) / 2^32) exactly, because
//           x (M - 2^64/f) / 2^64 < 2^-32 and x/f is at least 1/f short of
//           the next integer.  For f = 1, M = 2^64 - 1 gives x - 1, and c
//           carries the missing 4095 instead (4095 + c below).
//   .z      f * 2^20, the bound at which the state emits 16 bits first
//   .w      (4096 - f) | c << 16
__device__ __forceinline__ uint4 coder_entry(uint32_t f, uint32_t c) {
  const unsigned long long M = f == 1u ? ~0ull : ~0ull / f + 1ull;
  const uint32_t cc = f == 1u ? c + (kRansTotal - 1u) : c;
  return make_uint4(static_cast<uint32_t>(M), static_cast<uint32_t>(M >> 32), f << 20,
                    (kRansTotal - f) | (cc << 16));
}

// Block-wide reductions over the 256 threads of a table kernel.
__device__ __forceinline__ unsigned long long table_sum(unsigned long long v,
                                                        unsigned long long* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int i = 0; i < kTableThreads / 32; ++i) t += red[i];
  __syncthreads();
  return t;
}

__device__ __forceinline__ unsigned long long table_max(unsigned long long v,
                                                        unsigned long long* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int i = 0; i < kTableThreads / 32; ++i) t = red[i] > t ? red[i] : t;
  __syncthreads();
  return t;
}

// Exclusive prefix sum over the 256 threads.
__device__ __forceinline__ uint32_t table_exclusive_scan(uint32_t v, unsigned long long* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) red[wid] = incl;
  __syncthreads();
  uint32_t base = 0;
  for (int i = 0; i < wid; ++i) base += static_cast<uint32_t>(red[i]);
  __syncthreads();
  return base + incl - v;
}

// One CTA per rank of the range: the shard's frequencies from its exponent
// histogram one iteration earlier, f = 1 + floor(h * 3840 / sum h), the rest
// of 4096 to the most frequent symbol (lowest on a tie), 16 each for an
// empty histogram; then the coder entries.
__global__ void __launch_bounds__(kTableThreads)
    k_rans_enc_tables(const uint32_t* __restrict__ hist_prev, uint8_t* __restrict__ tables) {
  __shared__ unsigned long long red[kTableThreads / 32];
  const int s = threadIdx.x;
  const uint32_t h = hist_prev[256 * static_cast<int64_t>(blockIdx.x) + s];
  const unsigned long long total = table_sum(h, red);
  uint32_t f = 16;
  if (total) {
    f = 1u + static_cast<uint32_t>(static_cast<unsigned long long>(h) * 3840ull / total);
    const unsigned long long sum = table_sum(f, red);
    const unsigned long long best =
        table_max((static_cast<unsigned long long>(h) << 8) | (255u - s), red);
    if (255u - static_cast<uint32_t>(best & 255u) == static_cast<uint32_t>(s))
      f += kRansTotal - static_cast<uint32_t>(sum);
  }
  const uint32_t c = table_exclusive_scan(f, red);
  uint8_t* t = tables + kRansEncTableBytes * static_cast<int64_t>(blockIdx.x);
  reinterpret_cast<uint4*>(t)[s] = coder_entry(f, c);
  reinterpret_cast<uint16_t*>(t + kCFreq)[s] = static_cast<uint16_t>(f);
}

// One warp codes one block of L exponents into its coding buffer `buf`
// (layout: rans_block_bytes): lane l codes positions l, l+32, ... backwards,
// emitting renormalisation words downwards from the end of its region, then
// the final state; the lane word counts and their exclusive prefixes go to
// the buffer's head.  Returns the record's size in 16-byte units (counts,
// streams, zero padding); the record itself is assembled from the buffer
// when it is stored.
__device__ uint32_t rans_encode_block(const uint8_t* exps, int L, const uint4* tab,
                                      uint8_t* buf, int LW, int lane) {
  uint16_t* region = reinterpret_cast<uint16_t*>(buf + kRansBufHead) + lane * LW;
  int top = LW;
  uint32_t x = kRansLow;
  const int n = L > lane ? (L - lane + kRansLanes - 1) / kRansLanes : 0;  // this lane's symbols
  // The next step's entry and the symbol two steps ahead are loaded before
  // this step's store of a word, above which the compiler may not move them
  // (all three live in shared memory).  Near the end the symbol index runs
  // up to 64 bytes below the block's exponents: still inside the CTA's
  // shared memory (the meta region precedes the exponents), and the entry
  // loaded from it is never used.
  const uint8_t* ep = exps + lane;
  uint4 En = tab[ep[kRansLanes * (n - 1)]];
  uint32_t sn = ep[kRansLanes * (n - 2)];
#pragma unroll 16
  for (int m = n - 1; m >= 0; --m) {
    const uint4 E = En;
    En = tab[sn];
    sn = ep[kRansLanes * (m - 2)];
    // x >= f * 2^20: emit the low 16 bits.  The store is unconditional (a
    // word not emitted is overwritten by the next one); only top moves.
    const bool emit = x >= E.z;
    region[top - 1] = static_cast<uint16_t>(x & 0xFFFFu);
    top -= emit ? 1 : 0;
    x = emit ? x >> 16 : x;
    const unsigned long long xm =
        static_cast<unsigned long long>(x) * E.y + __umulhi(x, E.x);
    const uint32_t q = static_cast<uint32_t>(xm >> 32);  // floor(x / f) (x - 1 when f = 1)
    x += q * (E.w & 0xFFFFu) + (E.w >> 16);              // (q << 12) + x - q f + c
  }
  region[--top] = static_cast<uint16_t>(x & 0xFFFFu);
  region[--top] = static_cast<uint16_t>(x >> 16);
  const uint32_t nw = static_cast<uint32_t>(LW - top);
  uint32_t incl = nw;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  uint16_t* head = reinterpret_cast<uint16_t*>(buf);
  head[lane] = static_cast<uint16_t>(nw);
  head[kRansLanes + lane] = static_cast<uint16_t>(incl - nw);
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  if (lane == 31) head[2 * kRansLanes] = static_cast<uint16_t>(total);
  return (kRansLanes + total + 7u) / 8u;
}

// One decoding step of a lane: symbol from the slot table (in shared
// memory), value and
// exponent out, state update, and a renormalisation that reads the word
// loaded one step ahead (branch-free; the index is clamped to the lane's
// last word, an overrun shows in the final check).
__device__ __forceinline__ void decode_step(const uint32_t* tab, const uint16_t* s,
                                            uint32_t last, const uint8_t* sp, uint16_t* op,
                                            uint8_t* rp, uint32_t& x, uint32_t& idx,
                                            uint32_t& nxt) {
  const uint32_t e = tab[x & (kRansTotal - 1)];
  *op = static_cast<uint16_t>(join1(*sp, e >> 12));  // join1 keeps the low 8 bits
  *rp = static_cast<uint8_t>(e >> 12);
  x = (e >> 20) * (x >> kRansBits) + (e & 0xFFFu);  // f (x >> 12) + slot - cum
  const bool renorm = x < kRansLow;
  x = renorm ? (x << 16) | nxt : x;
  idx += renorm ? 1u : 0u;
  nxt = s[idx < last ? idx : last];
}

// One warp decodes one record of `rec_words` words into the block's L
// exponents with the slot table `tab` (entry: (slot - cum) | symbol << 12 |
// f << 20, so that f, on the state's critical path, takes one shift), and
// writes each value (joined with its
// sign+mantissa byte from `ss`) to `out` and its exponent to the ExpCache
// `rc`.  False (for the whole warp) if the record does not decode cleanly.
__device__ bool rans_decode_block(const uint16_t* rec, uint32_t rec_words, int L,
                                  const uint32_t* tab, const uint8_t* ss,
                                  uint16_t* out, uint8_t* rc, int lane) {
  const uint32_t nw = rec_words >= kRansLanes ? rec[lane] : 0u;
  uint32_t incl = nw;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  const uint32_t pre = incl - nw;
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  const bool bad = rec_words < kRansLanes || kRansLanes + total > rec_words || nw < 2;
  if (__any_sync(0xffffffffu, bad)) return false;
  const uint16_t* s = rec + kRansLanes + pre;
  const uint32_t last = nw - 1;
  uint32_t x = (static_cast<uint32_t>(s[0]) << 16) | s[1];
  uint32_t idx = 2;
  uint32_t nxt = s[idx < last ? idx : last];
  const int n = L > lane ? (L - lane + kRansLanes - 1) / kRansLanes : 0;  // this lane's symbols
  const uint8_t* sp = ss + lane;
  uint16_t* op = out + lane;
  uint8_t* rp = rc + lane;
  int m = 0;
  for (; m + 16 <= n; m += 16) {
#pragma unroll
    for (int k = 0; k < 16; ++k)
      decode_step(tab, s, last, sp + 32 * k, op + 32 * k, rp + 32 * k, x, idx, nxt);
    sp += 512;
    op += 512;
    rp += 512;
  }
  for (; m < n; ++m) {
    decode_step(tab, s, last, sp, op, rp, x, idx, nxt);
    sp += 32;
    op += 32;
    rp += 32;
  }
  return !__any_sync(0xffffffffu, idx != nw || x != kRansLow);
}

// One 16-value group of the sender's streaming pass (see k_compress_rans).
__device__ __forceinline__ void stream_group(int gi, bool in, const uint4& w0, const uint4& w1,
                                             const uint4& cc, bool cold, bool direct_raw,
                                             uint32_t mG, uint4* c4, uint8_t* es,
                                             uint8_t* payload, int64_t e0, int64_t stride,
                                             Control* ctl, uint32_t* hist, uint32_t& mine,
                                             int lane) {
  uint32_t sample = 0x100u + lane;
  if (in) {
    const uint4 e = make_uint4(exp4(w0.x, w0.y), exp4(w0.z, w0.w), exp4(w1.x, w1.y),
                               exp4(w1.z, w1.w));
    const uint32_t d = (e.x ^ cc.x) | (e.y ^ cc.y) | (e.z ^ cc.z) | (e.w ^ cc.w);
    if (d || cold) {
      mine |= 1u << __umulhi(static_cast<uint32_t>(gi), mG);
      c4[gi] = e;
    }
    reinterpret_cast<uint4*>(es)[gi] = e;
    if (direct_raw) {
      if (in_bounds(ctl, 2 * e0 + 32 * static_cast<int64_t>(gi), 32, stride)) {
        uint4* dst = reinterpret_cast<uint4*>(payload + 2 * e0) + 2 * gi;
        dst[0] = w0;
        dst[1] = w1;
      }
    } else if (in_bounds(ctl, e0 + 16 * static_cast<int64_t>(gi), 16, stride)) {
      reinterpret_cast<uint4*>(payload + e0)[gi] =
          make_uint4(sm4(w0.x, w0.y), sm4(w0.z, w0.w), sm4(w1.x, w1.y), sm4(w1.z, w1.w));
    }
    sample = e.x & 0xFFu;
  }
  const uint32_t same = __match_any_sync(0xffffffffu, sample);
  if (in && lane == __ffs(same) - 1) atomicAdd(&hist[sample], static_cast<uint32_t>(__popc(same)));
}

// The tile's records, assembled in the exponent region (free once the tile
// is coded) in their payload order and stored by one bulk copy from thread 0:
// one warp per changed block writes its record there (word counts, each
// lane's stream behind them, zero padding), where scattered 2-byte global
// stores would otherwise carry each lane's stream.  Kept out of line so that
// the kernel's own code keeps the layout it has without it.  Every thread of
// the CTA calls it.
__device__ __noinline__ void store_records_bulk(const CompressParams& p, const RansLayout& Ly,
                                                int nblk, uint8_t* es, const uint8_t* scr,
                                                const uint32_t* rsize, const uint32_t* rpre,
                                                uint32_t X, uint32_t agg, uint8_t* payload,
                                                int64_t BB, int64_t LW, int warp, int lane,
                                                int tid) {
  int i = 0;
  for (int kb = 0; kb < nblk; ++kb) {
    if (!rsize[kb]) continue;
    if (i++ % (kThreads / 32) != warp) continue;
    uint16_t* dst = reinterpret_cast<uint16_t*>(es + 16 * rpre[kb]);
    const uint8_t* buf = scr + kb * BB;
    const uint16_t* head = reinterpret_cast<const uint16_t*>(buf);
    const uint32_t n = head[lane];
    const uint32_t pre = head[kRansLanes + lane];
    const uint16_t* src = reinterpret_cast<const uint16_t*>(buf + kRansBufHead) +
                          (lane + 1) * LW - n;
    dst[lane] = static_cast<uint16_t>(n);
    uint16_t* d = dst + kRansLanes + pre;
    for (uint32_t k = 0; k < n; ++k) d[k] = src[k];
    const uint32_t words = kRansLanes + head[2 * kRansLanes];
    if (words + lane < 8u * rsize[kb]) dst[words + lane] = 0;
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0 && agg > 0) {
    const int64_t at = Ly.D + 16 * static_cast<int64_t>(X);
    if (in_bounds(p.ctl, at, 16 * static_cast<int64_t>(agg), p.stride)) {
      bulk_s2g(payload + at, es, 16u * agg);
      bulk_commit();
      bulk_wait_read_all();  // the CTA's shared memory outlives the copy's reads
    }
  }
}

struct RansShared {
  uint32_t ticket;
  uint32_t epoch;  // this launch's tag of look-back and flag words
  uint32_t X;      // record units (16 bytes) before the tile in its shard
  uint32_t agg;    // record units of the tile
  uint32_t coded;  // set once the tile's blocks are coded and its aggregate published
};

__global__ void __launch_bounds__(kThreads)
    k_compress_rans(const CompressParams p, const uint8_t* __restrict__ enc_tables,
                    uint32_t* __restrict__ hist_out) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ RansShared sh;
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t B = p.geo.B;
  const int64_t T = p.geo.T;
  const int64_t TE = T * B;
  const uint4* tab = reinterpret_cast<const uint4*>(dsm + kCTab);
  const uint16_t* freq = reinterpret_cast<const uint16_t*>(dsm + kCFreq);
  uint32_t* hist = reinterpret_cast<uint32_t*>(dsm + kCHist);
  uint32_t* rsize = reinterpret_cast<uint32_t*>(dsm + kCSize);
  uint32_t* rpre = reinterpret_cast<uint32_t*>(dsm + kCPre);
  uint32_t* red = reinterpret_cast<uint32_t*>(dsm + kCRed);
  uint32_t* fw = reinterpret_cast<uint32_t*>(dsm + kCFw);
  uint8_t* es = dsm + kRansEncMeta;  // the tile's exponents [TE]
  uint8_t* scr = es + TE;            // one coding buffer per block [T * BB], at first the
                                     // tile's values (T * BB >= 2 * TE: a lane region
                                     // holds more than two uint16 per value of its lane)
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
    sh.coded = 0;
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
  const uint4* w4 = reinterpret_cast<const uint4*>(p.w + x.shard_off + x.e0);
  uint4* c4 = reinterpret_cast<uint4*>(p.scache + x.shard_off + x.e0);
  uint8_t* payload = p.payloads + static_cast<int64_t>(x.rl) * p.stride;
  const uint32_t te = static_cast<uint32_t>(x.te);
  if (tid == 0) {
    // This shard's coder table (written by k_rans_enc_tables), and the tile's
    // values and cached exponents in two bulk copies.  The values land in the
    // coding buffers and the cached exponents in the exponent region: both are
    // free until the streaming pass has read them (the pass turns each group
    // of cached exponents into the group's new exponents in place).
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(kRansEncTableBytes) + 3u * te);
    bulk_g2s(dsm + kCTab, enc_tables + kRansEncTableBytes * static_cast<int64_t>(x.rl),
             static_cast<uint32_t>(kRansEncTableBytes), &bar);
    bulk_g2s(scr, w4, 2u * te, &bar);
    bulk_g2s(es, c4, te, &bar);
  }
  __syncthreads();

  const int ngroups = static_cast<int>(te >> 4);
  // block of group gi: gi / (B/16), as mulhi(gi, ceil(2^32 / (B/16))), exact for gi < 2^16
  const uint32_t mG = static_cast<uint32_t>(((1ull << 32) + B / 16 - 1) / (B / 16));
  if (warp == 0) {
    bool to = false;
    uint32_t X = 0;
    if (!direct_raw) {
      // The look-back starts once this tile is coded: its predecessors code
      // at the same time, so polling earlier finds nothing and takes issue
      // slots from the coding warps.  The wait is bounded like every other.
      const uint64_t t0 = globaltimer();
      while (!*reinterpret_cast<volatile uint32_t*>(&sh.coded)) {
        if (globaltimer() - t0 > p.timeout_ns) break;
        __nanosleep(256);
      }
      __syncwarp();
      X = lookback_exclusive(p, x, sh.epoch, lane, x.k0 * (BB / 16), &to);
    }
    if (lane == 0) {
      sh.X = X;
      if (to) record_status(p.ctl, kStatusTimeout);
    }
  } else {
    const int ft = tid - 32;
    // One streaming pass over the tile, 16 values per thread and step:
    // flags (exact test), sender-cache refresh of the groups that differ,
    // the payload's bytes (sign+mantissa, or raw values), the exponents for
    // the coder, and the sampled histogram (the first value of each group).
    // The loop runs whole warps so that equal samples merge across lanes.
    if (!mbar_wait_bounded(&bar, 0, p.timeout_ns)) {
      record_status(p.ctl, kStatusTimeout);
      mbar_wait_bounded(&bar, 0, p.timeout_ns);
    }
    uint32_t mine = 0;
    const uint4* ws4 = reinterpret_cast<const uint4*>(scr);
    for (int g0 = ft - lane; g0 < ngroups; g0 += kThreads - 32) {
      const int gi = g0 + lane;
      const bool in = gi < ngroups;
      uint4 w0 = {}, w1 = {}, cc = {};
      if (in) {
        w0 = ws4[2 * gi];
        w1 = ws4[2 * gi + 1];
        cc = reinterpret_cast<const uint4*>(es)[gi];
      }
      stream_group(gi, in, w0, w1, cc, cold, direct_raw, mG, c4, es, payload, x.e0, p.stride,
                   p.ctl, hist, mine, lane);
    }
    mine = __reduce_or_sync(0xffffffffu, mine);
    if (lane == 0 && mine) atomicOr(&fw[0], mine);
    flaggers_sync();
    const uint32_t f = fw[0];
    // code the changed blocks: the i-th changed block goes to warp 1 + i % 3
    if (!direct_raw) {
      int i = 0;
      for (int kb = 0; kb < x.nblk; ++kb) {
        if (!((f >> kb) & 1u)) continue;
        if (i % (kThreads / 32 - 1) == warp - 1) {
          const int L = static_cast<int>((kb + 1) * B < x.te ? B : x.te - kb * B);
          const uint32_t units =
              rans_encode_block(es + kb * B, L, tab, scr + kb * BB, static_cast<int>(LW), lane);
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
      *reinterpret_cast<volatile uint32_t*>(&sh.coded) = 1u;
    }
  }
  __syncthreads();
  if (tid == 0 && x.t > 0 && !direct_raw) publish(p, x, sh.epoch, kStateInclusive, sh.X + sh.agg);

  const int64_t limit = 2 * x.len;  // a payload this large goes out raw instead
  // The tile's records are one contiguous run of 16-byte units at D + 16 X.
  // Records that would end past 2*len are not stored: the shard then goes
  // out raw.  When they fit in the tile's exponent region they are assembled
  // there and stored in one bulk copy; otherwise one warp per changed block
  // stores its record: lane l writes its word count and copies its own
  // stream (the top of its region) to its place behind the counts, and the
  // lanes below the padding write its zeros.
  if (!direct_raw && Ly.D + 16 * (static_cast<int64_t>(sh.X) + sh.agg) <= limit &&
      16 * static_cast<int64_t>(sh.agg) <= static_cast<int64_t>(te)) {
    store_records_bulk(p, Ly, x.nblk, es, scr, rsize, rpre, sh.X, sh.agg, payload, BB, LW, warp,
                       lane, tid);
  } else if (!direct_raw && Ly.D + 16 * (static_cast<int64_t>(sh.X) + sh.agg) <= limit) {
    int i = 0;
    for (int kb = 0; kb < x.nblk; ++kb) {
      if (!rsize[kb]) continue;
      if (i++ % (kThreads / 32) != warp) continue;
      const int64_t at = Ly.D + 16 * (static_cast<int64_t>(sh.X) + rpre[kb]);
      if (!in_bounds(p.ctl, at, 16 * static_cast<int64_t>(rsize[kb]), p.stride)) continue;
      uint16_t* dst = reinterpret_cast<uint16_t*>(payload + at);
      const uint8_t* buf = scr + kb * BB;
      const uint16_t* head = reinterpret_cast<const uint16_t*>(buf);
      const uint32_t n = head[lane];
      const uint32_t pre = head[kRansLanes + lane];
      const uint16_t* src = reinterpret_cast<const uint16_t*>(buf + kRansBufHead) +
                            (lane + 1) * LW - n;
      dst[lane] = static_cast<uint16_t>(n);
      uint16_t* d = dst + kRansLanes + pre;
      for (uint32_t k = 0; k < n; ++k) d[k] = src[k];
      const uint32_t words = kRansLanes + head[2 * kRansLanes];
      if (words + lane < 8u * rsize[kb]) dst[words + lane] = 0;
    }
  }
  if (!direct_raw) {
    uint32_t* O = reinterpret_cast<uint32_t*>(payload + Ly.O);
    if (tid < x.nblk && in_bounds(p.ctl, Ly.O + 4 * (x.k0 + tid), 4, p.stride))
      O[x.k0 + tid] = 16u * (sh.X + rpre[tid]);
    if (tid == 0 && x.t == x.tiles - 1 && in_bounds(p.ctl, Ly.O + 4 * x.nb, 4, p.stride))
      O[x.nb] = 16u * (sh.X + sh.agg);
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
      if (!raw && in_bounds(p.ctl, Ly.A + i, 1, p.stride))
        payload[Ly.A + i] = static_cast<uint8_t>(byte);
    }
    if (to) record_status(p.ctl, kStatusTimeout);
    const uint32_t tot = warp_sum(nch);
    if (lane == 0) red[warp] = tot;
    __syncthreads();
    const uint32_t n_changed = red[0] + red[1] + red[2] + red[3];
    if (!raw && in_bounds(p.ctl, 0, Ly.D, p.stride)) {
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
}

// A shard that went raw only at the end (its RANS payload would not have
// been smaller than its raw bytes): rewrite it raw.  Shards that went raw
// from the start were written raw by k_compress_rans itself.  Every CTA
// walks the ranks (one descriptor read each) and copies its share of the
// tiles of those that need it, so a call with nothing to do costs R reads.
__global__ void __launch_bounds__(kThreads) k_rans_raw_fixup(const CompressParams p) {
  const Geometry& g = p.geo;
  for (int32_t rl = 0; rl < g.nfull + g.has_part; ++rl) {
    if (p.descs[rl].mode != CIERA_MODE_RAW) continue;
    const int64_t tiles = rl < g.nfull ? g.tiles_full : g.tiles_part;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
      const Tile x = make_tile(g, rl, t);
      if (rans_layout(x.len, x.nb).D >= 2 * x.len) break;  // written raw directly
      if (!in_bounds(p.ctl, 2 * x.e0, 2 * x.te, p.stride)) continue;
      const uint4* w = reinterpret_cast<const uint4*>(p.w + x.shard_off + x.e0);
      uint4* dst = reinterpret_cast<uint4*>(p.payloads + static_cast<int64_t>(x.rl) * p.stride +
                                            2 * x.e0);
      for (int64_t i = threadIdx.x; i < x.te / 8; i += blockDim.x) dst[i] = w[i];
    }
  }
}

// One CTA per rank (RANS ranks only, after the bitmap scan has validated the
// frequencies): slot j -> symbol s with cum[s] <= j < cum[s+1], its
// frequency and j - cum[s].
__global__ void __launch_bounds__(kTableThreads)
    k_rans_dec_tables(const DecompressParams p, uint32_t* __restrict__ tables) {
  __shared__ unsigned long long red[kTableThreads / 32];
  __shared__ uint32_t cum[257];
  const int r = blockIdx.x;
  if (p.rank_state[r] != kRankRans) return;
  const int s = threadIdx.x;
  const int64_t len = shard_len_of(p.geo, r);
  const int64_t nb = (len + p.geo.B - 1) / p.geo.B;
  const int64_t C = rans_layout(len, nb).C;
  const uint8_t* tab = payload_of(p, r) + C;
  const uint32_t f = in_bounds(p.ctl, C + 2 * s, 2, p.stride)
                         ? tab[2 * s] | (static_cast<uint32_t>(tab[2 * s + 1]) << 8)
                         : 16u;
  const uint32_t c = table_exclusive_scan(f, red);
  cum[s] = c;
  if (s == kTableThreads - 1) cum[256] = c + f;
  __syncthreads();
  uint32_t* out = tables + 4096 * static_cast<int64_t>(r);
  const uint32_t j0 = 16u * s;  // this thread's slots j0 .. j0+15
  int lo = 0, hi = 255;         // largest symbol with cum <= j0
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cum[mid] <= j0) lo = mid; else hi = mid - 1;
  }
  uint32_t sym = static_cast<uint32_t>(lo);
  for (uint32_t j = j0; j < j0 + 16; ++j) {
    while (sym < 255 && cum[sym + 1] <= j) ++sym;
    out[j] = (j - cum[sym]) | (sym << 12) | ((cum[sym + 1] - cum[sym]) << 20);
  }
}

__global__ void __launch_bounds__(kThreads)
    k_decompress_rans(const DecompressParams p, const uint32_t* __restrict__ dec_tables) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t s_fw, s_bad, s_staged;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const Tile x = decode_tile(p.geo, blockIdx.x);
  const uint32_t state = p.rank_state[x.rl];
  if (state == kRankSkip) return;
  if (state == kRankCompressed) {
    // not a payload of the RANS sender
    if (threadIdx.x == 0 && x.t == 0) atomicOr(&p.ctl->status, kStatusCorrupt);
    return;
  }
  const int64_t B = p.geo.B;
  const int64_t T = p.geo.T;
  const int64_t TE = T * B;
  const int nthreads = static_cast<int>(blockDim.x);  // rans_decompress_threads(T)
  if (dynamic_smem_size() < static_cast<uint32_t>(rans_decompress_smem(T, B)) || T > 32 ||
      !p.fast || nthreads != rans_decompress_threads(T)) {
    if (tid == 0) atomicOr(&p.ctl->status, kStatusInternal);
    return;
  }
  if (state == kRankRaw) {
    // the tile's values streamed from the payload to out, their exponents to
    // the ExpCache (nothing staged)
    if (!in_bounds(p.ctl, 2 * x.e0, 2 * x.te, p.stride)) return;
    const uint4* vs = reinterpret_cast<const uint4*>(payload_of(p, x.rl) + 2 * x.e0);
    uint4* out = reinterpret_cast<uint4*>(p.out + x.shard_off + x.e0);
    uint4* rc = reinterpret_cast<uint4*>(p.rcache + x.shard_off + x.e0);
    for (int gi = tid; gi < static_cast<int>(x.te >> 4); gi += nthreads) {
      const uint4 w0 = __ldcs(vs + 2 * gi);
      const uint4 w1 = __ldcs(vs + 2 * gi + 1);
      out[2 * gi] = w0;
      out[2 * gi + 1] = w1;
      rc[gi] = make_uint4(exp4(w0.x, w0.y), exp4(w0.z, w0.w), exp4(w1.x, w1.y), exp4(w1.z, w1.w));
    }
    return;
  }
  uint32_t* offs = reinterpret_cast<uint32_t*>(dsm + kDOffs);
  uint8_t* ss = dsm + kRansDecMeta;   // sign+mantissa bytes [TE]
  uint8_t* recs = ss + TE;            // the tile's records, when they fit [TE / 2]
  // the rank's slot table, copied in with the tile: a decoding step is one
  // dependent lookup in it, faster from shared memory than through L1
  uint32_t* tabs =
      reinterpret_cast<uint32_t*>(recs + ((rans_record_stage(T, B) + 15) & ~int64_t(15)));
  const ciera_desc d = p.descs[x.rl];
  const uint8_t* payload = payload_of(p, x.rl);
  const RansLayout Ly = rans_layout(x.len, x.nb);
  uint8_t* rc = p.rcache + x.shard_off + x.e0;
  uint16_t* out = p.out + x.shard_off + x.e0;
  const uint32_t te = static_cast<uint32_t>(x.te);
  if (tid <= x.nblk)
    offs[tid] = in_bounds(p.ctl, Ly.O + 4 * (x.k0 + tid), 4, p.stride)
                    ? reinterpret_cast<const uint32_t*>(payload + Ly.O)[x.k0 + tid]
                    : 0u;
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
    uint64_t rec_bytes = 0;
    for (int kb = 0; kb < x.nblk; ++kb) {
      if (!((fw >> kb) & 1u)) continue;
      const uint32_t a = offs[kb], b = offs[kb + 1];
      // a record must be nonempty, lie inside the payload and start and end
      // on 16 bytes (the bulk copy's alignment)
      if (b <= a || (a & 15u) || (b & 15u) ||
          static_cast<uint64_t>(Ly.D) + b > d.payload_bytes) {
        bad = 1;
        fw &= ~(1u << kb);
        continue;
      }
      rec_bytes += b - a;
    }
    // stage the records when they fit; else decode them from global memory
    const bool staged = rec_bytes <= static_cast<uint64_t>(rans_record_stage(T, B));
    s_fw = fw;
    s_bad = bad;
    s_staged = staged;
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(&bar, te + (staged ? static_cast<uint32_t>(rec_bytes) : 0u) +
                                    static_cast<uint32_t>(kRansDecTableBytes));
    bulk_g2s(tabs, dec_tables + 4096 * static_cast<int64_t>(x.rl),
             static_cast<uint32_t>(kRansDecTableBytes), &bar);
    if (in_bounds(p.ctl, x.e0, te, p.stride)) bulk_g2s(ss, payload + x.e0, te, &bar);
    if (staged) {
      uint32_t at = 0;
      for (int kb = 0; kb < x.nblk; ++kb)
        if ((fw >> kb) & 1u) {
          if (in_bounds(p.ctl, Ly.D + offs[kb], offs[kb + 1] - offs[kb], p.stride))
            bulk_g2s(recs + at, payload + Ly.D + offs[kb], offs[kb + 1] - offs[kb], &bar);
          at += offs[kb + 1] - offs[kb];
        }
    }
  }
  __syncthreads();
  const uint32_t fw = s_fw;
  // the kept blocks' cached exponents, read while the bulk copies land
  const uint32_t mG = static_cast<uint32_t>(((1ull << 32) + B / 16 - 1) / (B / 16));
  const int ngroups = static_cast<int>(te >> 4);
  constexpr int kPer = 4;  // groups per thread held in registers before the merge
  uint4 kept[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int gi = tid + q * nthreads;
    if (gi < ngroups && !((fw >> __umulhi(static_cast<uint32_t>(gi), mG)) & 1u))
      kept[q] = reinterpret_cast<const uint4*>(rc)[gi];
  }
  // the kept blocks' cached exponents beyond those groups, 128-byte lines
  // wholly inside the tile, into L2 ahead of the merge (a receiver tile is
  // twice the sender's, so these are half of it)
  for (int li = kPer * nthreads / 8 + tid; li < static_cast<int>(te >> 7); li += nthreads)
    if (!((fw >> __umulhi(static_cast<uint32_t>(8 * li), mG)) & 1u))
      prefetch_l2(rc + 128 * static_cast<int64_t>(li));
  if (__syncthreads_or(!mbar_wait_bounded(&bar, 0, p.timeout_ns))) {
    if (tid == 0) atomicOr(&p.ctl->status, kStatusTimeout);
    mbar_wait_bounded(&bar, 0, p.timeout_ns);
    __syncthreads();
    return;
  }
  // merge of the kept blocks: sign+mantissa bytes with cached exponents
  for (int gi0 = 0; gi0 < ngroups; gi0 += kPer * nthreads) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int gi = gi0 + tid + q * nthreads;
      if (gi >= ngroups || ((fw >> __umulhi(static_cast<uint32_t>(gi), mG)) & 1u)) continue;
      const uint4 e = gi0 == 0 ? kept[q] : reinterpret_cast<const uint4*>(rc)[gi];
      const uint4 s = reinterpret_cast<const uint4*>(ss)[gi];
      uint4* o = reinterpret_cast<uint4*>(out) + 2 * gi;
      const uint2 v0 = join4(s.x, e.x), v1 = join4(s.y, e.y);
      const uint2 v2 = join4(s.z, e.z), v3 = join4(s.w, e.w);
      o[0] = make_uint4(v0.x, v0.y, v1.x, v1.y);
      o[1] = make_uint4(v2.x, v2.y, v3.x, v3.y);
    }
  }
  // decode the changed blocks straight into the output and the ExpCache:
  // the i-th changed block goes to warp i % 4
  const bool staged = s_staged;
  const uint32_t* tab = tabs;
  bool ok = true;
  int i = 0;
  uint32_t at = 0;
  for (int kb = 0; kb < x.nblk; ++kb) {
    if (!((fw >> kb) & 1u)) continue;
    const uint32_t nbytes = offs[kb + 1] - offs[kb];
    if (i % (nthreads / 32) == warp) {
      const int L = static_cast<int>((kb + 1) * B < x.te ? B : x.te - kb * B);
      const uint8_t* rec = staged ? recs + at : payload + Ly.D + offs[kb];
      if (!staged && !in_bounds(p.ctl, Ly.D + offs[kb], nbytes, p.stride)) rec = nullptr;
      ok = rec != nullptr && rans_decode_block(reinterpret_cast<const uint16_t*>(rec), nbytes / 2, L, tab,
                             ss + kb * B, out + kb * B, rc + kb * B, lane) && ok;
    }
    at += nbytes;
    ++i;
  }
  const uint32_t any_bad = __syncthreads_or(!ok);
  if (tid == 0 && (any_bad || s_bad)) atomicOr(&p.ctl->status, kStatusCorrupt);
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
                         uint8_t* enc_tables, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t smem = rans_compress_smem(p.geo.T, p.geo.B);
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(k_compress_rans), smem, g_smem_c);
  if (e != cudaSuccess) return e;
  k_rans_enc_tables<<<static_cast<unsigned>(p.geo.rank_count), kTableThreads, 0, s>>>(
      hist_prev, enc_tables);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t grid = p.geo.total_tiles + 1;
  k_compress_rans<<<static_cast<unsigned>(grid), kThreads, static_cast<size_t>(smem), s>>>(
      p, enc_tables, hist_out);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (!(p.flags & CIERA_COLD) && p.geo.total_tiles > 0) {
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t grid = p.geo.total_tiles < 2 * sms ? p.geo.total_tiles : 2 * sms;
    k_rans_raw_fixup<<<static_cast<unsigned>(grid), kThreads, 0, s>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

// The geometry g with tiles of Tr blocks instead of g.T.
static Geometry retiled(const Geometry& g, int64_t Tr) {
  Geometry r = g;
  r.T = Tr;
  const int64_t nb_full = (g.S + g.B - 1) / g.B;
  r.tiles_full = (nb_full + Tr - 1) / Tr;
  r.tiles_part = g.has_part ? ((g.len_part + g.B - 1) / g.B + Tr - 1) / Tr : 0;
  r.total_tiles = static_cast<int64_t>(g.nfull) * r.tiles_full + r.tiles_part;
  return r;
}

int launch_decompress_rans(const DecompressParams& sender_tiles, uint32_t* dec_tables,
                           void* stream) {
  DecompressParams p = sender_tiles;
  p.geo = retiled(sender_tiles.geo, rans_receiver_blocks(sender_tiles.geo.T));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.geo.total_tiles <= 0) return cudaSuccess;
  const int64_t smem = rans_decompress_smem(p.geo.T, p.geo.B);
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(k_decompress_rans), smem, g_smem_d);
  if (e != cudaSuccess) return e;
  k_rans_dec_tables<<<static_cast<unsigned>(p.geo.rank_count), kTableThreads, 0, s>>>(
      p, dec_tables);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_decompress_rans<<<static_cast<unsigned>(p.geo.total_tiles),
                      static_cast<unsigned>(rans_decompress_threads(p.geo.T)),
                      static_cast<size_t>(smem), s>>>(p, dec_tables);
  return cudaGetLastError();
}

}  // namespace ciera
