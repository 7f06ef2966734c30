// ciera_device.cuh -- device helpers shared by the kernels of libciera:
// PTX wrappers (bulk copies, mbarriers, strong loads and stores), bf16 field
// arithmetic, tile geometry and the decoupled look-back.  Not part of the
// public ABI; every helper lives in an unnamed namespace per translation unit.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "ciera_internal.h"

namespace ciera {
namespace {

// ------------------------------------------------------------------------
// PTX helpers

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes the mbarrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of an mbarrier.  False on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > timeout_ns) return false;
  }
  return true;
}

// Global -> shared bulk copy, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Shared -> global bulk copy in the current bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Bytes of dynamic shared memory this CTA was launched with.
__device__ __forceinline__ uint32_t dynamic_smem_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void record_status(Control* ctl, uint32_t bits) {
  atomicOr(&ctl->status, bits);
}

// Checked builds (-DCIERA_CHECKED): global accesses at computed offsets are
// tested against their buffer first; one that would leave it is skipped and
// kStatusBounds recorded (no trap, no assert).  Other builds compile the
// test away.
#ifdef CIERA_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// True if [off, off + size) lies inside [0, limit); in checked builds a
// false result also records kStatusBounds.
__device__ __forceinline__ bool in_bounds(Control* ctl, int64_t off, int64_t size,
                                          int64_t limit) {
  if (!kChecked) return true;
  if (off >= 0 && size >= 0 && off <= limit - size) return true;
  atomicOr(&ctl->status, kStatusBounds);
  return false;
}

// Received payload of range rank r: its entry of the pointer table when the
// payloads arrived in separate buffers, else its slot of the contiguous
// layout.  p.stride bounds either.
__device__ __forceinline__ const uint8_t* payload_of(const DecompressParams& p, int64_t r) {
  return p.payload_ptrs ? p.payload_ptrs[r] : p.payloads + r * p.stride;
}

// Named barrier of the 96 worker threads (warps 1-3) of a compress CTA.
__device__ __forceinline__ void flaggers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kThreads - 32) : "memory");
}

// ------------------------------------------------------------------------
// bf16 field arithmetic on packed words (two values per 32-bit word).
// exponent e = (w >> 7) & 0xFF; sign+mantissa byte s = sign << 7 | mantissa.

// Exponents of the 4 values in words a (values 0,1) and b (values 2,3), one
// per byte: bits 7..14 of each value are bytes 0 and 2 of the word >> 7.
__device__ __forceinline__ uint32_t exp4(uint32_t a, uint32_t b) {
  return __byte_perm(a >> 7, b >> 7, 0x6420);
}

// Sign+mantissa bytes of the two values of word a in bytes 0 and 2.
__device__ __forceinline__ uint32_t sm_pair(uint32_t a) {
  return ((a >> 8) & 0x00800080u) | (a & 0x007F007Fu);
}

// Sign+mantissa bytes of the two values of word a (low 16 bits).
__device__ __forceinline__ uint32_t sm2(uint32_t a) { return __byte_perm(sm_pair(a), 0u, 0x4420); }

__device__ __forceinline__ uint32_t sm4(uint32_t a, uint32_t b) {
  return __byte_perm(sm_pair(a), sm_pair(b), 0x6420);
}

// Four values from four sign+mantissa bytes s and four exponents e: the high
// byte of a value is sign | exponent >> 1, the low byte exponent bit 0 <<
// 7 | mantissa.  Returns values 0,1 in .x and 2,3 in .y.
__device__ __forceinline__ uint2 join4(uint32_t s, uint32_t e) {
  const uint32_t hi = (s & 0x80808080u) | ((e >> 1) & 0x7F7F7F7Fu);
  const uint32_t lo = ((e << 7) & 0x80808080u) | (s & 0x7F7F7F7Fu);
  return make_uint2(__byte_perm(lo, hi, 0x5140), __byte_perm(lo, hi, 0x7362));
}

// Two values from two sign+mantissa bytes (s, low 16 bits) and two exponents
// (e, low 16 bits).
__device__ __forceinline__ uint32_t join2(uint32_t s, uint32_t e) { return join4(s, e).x; }

__device__ __forceinline__ uint32_t exp1(uint32_t v) { return (v >> 7) & 0xFFu; }
__device__ __forceinline__ uint32_t sm1(uint32_t v) { return ((v >> 8) & 0x80u) | (v & 0x7Fu); }
__device__ __forceinline__ uint32_t join1(uint32_t s, uint32_t e) {
  return ((s & 0x80u) << 8) | ((e & 0xFFu) << 7) | (s & 0x7Fu);
}

// ------------------------------------------------------------------------
// Tile geometry

struct Tile {
  int32_t rl;       // range-local rank
  int64_t t;        // tile index inside the shard
  int64_t sidx;     // shard-major tile index: rl * tiles_full + t
  int64_t len;      // values of the shard
  int64_t nb;       // blocks of the shard
  int64_t tiles;    // tiles of the shard
  int64_t k0;       // first block of the tile
  int32_t nblk;     // blocks in the tile
  int64_t e0;       // first value of the tile, shard-relative
  int64_t te;       // values in the tile
  int64_t shard_off;  // first value of the shard, range-relative
};

__device__ __forceinline__ Tile make_tile(const Geometry& g, int32_t rl, int64_t t) {
  Tile x;
  x.rl = rl;
  x.t = t;
  x.sidx = static_cast<int64_t>(rl) * g.tiles_full + t;
  const bool full = rl < g.nfull;
  x.len = full ? g.S : g.len_part;
  x.tiles = full ? g.tiles_full : g.tiles_part;
  x.nb = (x.len + g.B - 1) / g.B;
  x.k0 = x.t * g.T;
  const int64_t nblk = x.nb - x.k0 < g.T ? x.nb - x.k0 : g.T;
  x.nblk = static_cast<int32_t>(nblk);
  x.e0 = x.k0 * g.B;
  const int64_t te = x.len - x.e0;
  x.te = te < nblk * g.B ? te : nblk * g.B;
  x.shard_off = static_cast<int64_t>(x.rl) * g.S;
  return x;
}

// Shard-major order: tile i of the range (used where tiles are independent).
__device__ __forceinline__ Tile decode_tile(const Geometry& g, int64_t i) {
  const int64_t nf = static_cast<int64_t>(g.nfull) * g.tiles_full;
  if (i < nf) {
    const int32_t rl = static_cast<int32_t>(i / g.tiles_full);
    return make_tile(g, rl, i - static_cast<int64_t>(rl) * g.tiles_full);
  }
  return make_tile(g, g.nfull, i - nf);
}

// Interleaved order of the compress tickets: tile t of every shard, then
// tile t+1 of every shard, ...  Each shard's look-back chain then advances
// by one tile every R tickets instead of every ticket, and tiles of one
// shard still start in order (tile t always before tile t+1).
__device__ __forceinline__ Tile decode_ticket(const Geometry& g, int64_t i) {
  const int64_t P = g.nfull + g.has_part;  // shards with tiles
  const int64_t head = g.tiles_part * P;   // rows in which the partial shard takes part
  if (i < head) return make_tile(g, static_cast<int32_t>(i % P), i / P);
  const int64_t j = i - head;
  return make_tile(g, static_cast<int32_t>(j % g.nfull), g.tiles_part + j / g.nfull);
}

__device__ __forceinline__ int64_t shard_len_of(const Geometry& g, int32_t rl) {
  if (rl < g.nfull) return g.S;
  if (rl == g.nfull && g.has_part) return g.len_part;
  return 0;
}

// Changed blocks before block kb of the tile (kb < nblk), from the tile's
// flag words and their exclusive prefix.
__device__ __forceinline__ uint32_t count_before(const uint32_t* fw, const uint32_t* fpre,
                                                 int kb) {
  const uint32_t mask = (kb & 31) ? (0xffffffffu >> (32 - (kb & 31))) : 0u;
  return fpre[kb >> 5] + __popc(fw[kb >> 5] & mask);
}

__device__ __forceinline__ bool flag_of(const uint32_t* fw, int kb) {
  return (fw[kb >> 5] >> (kb & 31)) & 1u;
}

// ------------------------------------------------------------------------
// Decoupled look-back over the per-tile count of changed blocks.

// Tiles of at most 32 blocks also publish their flag bits in an
// epoch-tagged word (tile_flags), which the shard's last tile polls for the
// bitmap; their status words need no ordering and are stored relaxed.
// Larger tiles (block size below 256) hand their flags over as flag bytes,
// ordered by a release store of the status and read after an acquire.
__device__ __forceinline__ bool flags_in_words(const CompressParams& p) { return p.geo.T <= 32; }

__device__ __forceinline__ void publish(const CompressParams& p, const Tile& x, uint32_t epoch,
                                        uint32_t state, uint32_t value) {
  const unsigned long long v = (static_cast<unsigned long long>(epoch) << 32) |
                               (static_cast<unsigned long long>(state) << 30) | value;
  if (flags_in_words(p))
    st_relaxed_u64(&p.tile_status[x.sidx], v);
  else
    st_release_u64(&p.tile_status[x.sidx], v);
}

// Warp-wide: the number of changed blocks in the tiles before x in its
// shard.  Reads 32 predecessors per round and sums their aggregates until
// one of them carries an inclusive prefix.  It needs nothing of tile x
// itself, so it runs while x's own values are still being copied in.  The
// result is clamped to `cap` (the most the tiles before x can hold) so that
// every offset stays in bounds even after a timeout.
__device__ uint32_t lookback_exclusive(const CompressParams& p, const Tile& x, uint32_t epoch,
                                       uint32_t lane, int64_t cap, bool* timed_out) {
  if (x.t == 0) {
    *timed_out = false;
    return 0;
  }
  const unsigned long long* st = p.tile_status;
  const unsigned long long ep = static_cast<unsigned long long>(epoch) << 32;
  const unsigned long long incl = static_cast<unsigned long long>(kStateInclusive) << 30;
  const int64_t gfirst = x.sidx - x.t;
  int64_t base = x.sidx - 1;
  uint32_t X = 0;
  bool to = false;
  uint64_t t0 = 0;
  bool started = false;
  for (;;) {
    const int64_t idx = base - static_cast<int64_t>(lane);
    unsigned long long v = ep | incl;  // before the shard's first tile: inclusive 0
    if (idx >= gfirst) {
      for (;;) {
        v = flags_in_words(p) ? ld_relaxed_u64(&st[idx]) : ld_acquire_u64(&st[idx]);
        if ((v >> 32) == epoch && ((v >> 30) & 3ull) != 0) break;
        const uint64_t now = globaltimer();
        if (!started) {
          t0 = now;
          started = true;
        } else if (now - t0 > p.timeout_ns) {
          to = true;
          v = ep | incl;
          break;
        }
        // back off: the status word is an L2 round trip away, and a
        // thousand CTAs polling at full rate slow everyone's loads
        // (512 ns measured best among 32 .. 4096 on the OLMoE layer, and
        // again against 128, 256 and 1024 once tiles prefetch ahead)
        __nanosleep(512);
      }
    }
    if (__any_sync(0xffffffffu, to)) {
      X = 0;
      break;
    }
    const uint32_t is_incl = ((v >> 30) & 3ull) == kStateInclusive;
    const uint32_t bal = __ballot_sync(0xffffffffu, is_incl);
    const uint32_t val = static_cast<uint32_t>(v & 0x3FFFFFFFull);
    if (bal) {
      const int first = __ffs(bal) - 1;
      X += warp_sum(static_cast<int>(lane) <= first ? val : 0u);
      break;
    }
    X += warp_sum(val);
    base -= 32;
  }
  if (X > static_cast<uint64_t>(cap)) X = static_cast<uint32_t>(cap);
  *timed_out = __any_sync(0xffffffffu, to);
  return X;
}

}  // namespace
}  // namespace ciera
