// ciera_api.cpp -- host side of the libciera C ABI: plans, argument checks,
// workspace layout, the per-tensor predicate and status reporting.
//
// Method: "CIERA: Cross-Iteration Exponent Reuse for Lossless Allgather in
// Sharded MoE Training", Section 3.1 (block partition of each shard) and
// Section 3.2 (block count, bitmap size, gain of a shard).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "ciera.h"
#include "ciera_internal.h"
#include "ciera_rans.h"

using namespace ciera;

// Flags every compress entry point accepts.
constexpr uint32_t kCompressFlags = CIERA_COLD | CIERA_NO_RAW_AHEAD | CIERA_DEBUG_SKIP_FIRST_PUBLISH;

struct ciera_plan_s {
  int64_t numel;
  int64_t ranks;
  int64_t block;
  int64_t S;           // shard size
  int64_t nb_full;     // blocks of a full shard
  int64_t T;           // blocks per tile
  int64_t tiles_full;
  int64_t r_full;      // shards of exactly S values
  int64_t len_part;    // values of the one partial shard (0 if none)
  int64_t tiles_part;
  int64_t total_tiles;
  int64_t capacity;
  int64_t flag_stride;
  int64_t nw_stride;
  int64_t off_status, off_tflags, off_flags, off_words, off_prefix, off_rstate;
  int64_t off_renc, off_rdec;  // per-rank RANS coder tables (encoder, decoder)
  int64_t off_pred, off_result;  // per-rank raw-ahead prediction and launch result
  int64_t ws_bytes;
  int64_t smem_flags;         // flag words of every compress call (exact test)
  int64_t smem_flags_hashed;  // ... plus the per-block hash sums (hashed test)
  int64_t smem_decompress;
  bool fast;
  bool raw_fixup;
};

namespace {

std::atomic<uint64_t> g_timeout_ns{1000000000ull};
std::mutex g_cost_mu;
ciera_cost_model g_cost = {8e9, 0.22, 20e-6, 8e12, 4096};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t align_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Geometry of ranks [rb, rb+rc).
Geometry range_geometry(const ciera_plan_s* p, int64_t rb, int64_t rc) {
  Geometry g{};
  g.S = p->S;
  g.B = p->block;
  g.T = p->T;
  g.tiles_full = p->tiles_full;
  int64_t nfull = p->r_full - rb;
  if (nfull < 0) nfull = 0;
  if (nfull > rc) nfull = rc;
  const bool has_part = p->len_part > 0 && rb <= p->r_full && p->r_full < rb + rc;
  g.nfull = static_cast<int32_t>(nfull);
  g.has_part = has_part ? 1 : 0;
  g.len_part = has_part ? p->len_part : 0;
  g.tiles_part = has_part ? p->tiles_part : 0;
  g.rank_count = static_cast<int32_t>(rc);
  g.total_tiles = nfull * p->tiles_full + g.tiles_part;
  return g;
}

// Smallest block of a shard of `len` values: a raw payload can hold an
// unchanged block only if some block is not larger than the bitmap.
bool raw_can_hold_unchanged(int64_t len, int64_t B) {
  if (len <= 0) return false;
  const int64_t nb = ceil_div(len, B);
  const int64_t last = len - (nb - 1) * B;
  const int64_t smallest = last < B ? last : B;
  return smallest <= ceil_div(nb, 8);
}

}  // namespace

extern "C" {

const char* ciera_strerror(int status) {
  switch (status) {
    case CIERA_OK: return "ok";
    case CIERA_E_INVAL: return "invalid argument";
    case CIERA_E_CUDA: return "CUDA runtime error";
    case CIERA_E_CORRUPT: return "corrupt descriptor or bitmap";
    case CIERA_E_TIMEOUT: return "bounded device wait timed out";
    case CIERA_E_INTERNAL: return "internal launch configuration error";
    case CIERA_E_BOUNDS: return "out-of-range access skipped (checked build)";
    default: return "unknown status";
  }
}

int ciera_plan(const int64_t* shape, int ndim, int64_t block, int ranks, ciera_plan_t* out) {
  if (!out || ndim < 0 || (ndim > 0 && !shape) || block < 1 || ranks < 1) return CIERA_E_INVAL;
  int64_t n = 1;
  for (int i = 0; i < ndim; ++i) {
    if (shape[i] < 0) return CIERA_E_INVAL;
    if (shape[i] != 0 && n > kMaxNumel / shape[i]) return CIERA_E_INVAL;
    n *= shape[i];
  }
  if (n >= kMaxNumel) return CIERA_E_INVAL;
  ciera_plan_s* p = new (std::nothrow) ciera_plan_s();
  if (!p) return CIERA_E_INVAL;
  p->numel = n;
  p->ranks = ranks;
  p->block = block;
  p->S = n > 0 ? ceil_div(n, ranks) : 0;
  p->nb_full = p->S > 0 ? ceil_div(p->S, block) : 0;
  if (p->nb_full >= kMaxShardBlocks) {
    delete p;
    return CIERA_E_INVAL;
  }
  p->T = block >= kTileElems ? 1 : kTileElems / block;
  p->tiles_full = ceil_div(p->nb_full, p->T);
  p->r_full = p->S > 0 ? n / p->S : 0;
  p->len_part = n - p->r_full * p->S;
  p->tiles_part = p->len_part > 0 ? ceil_div(ceil_div(p->len_part, block), p->T) : 0;
  p->total_tiles = p->r_full * p->tiles_full + p->tiles_part;
  p->capacity = align_up(2 * p->S > 0 ? 2 * p->S : 1, 256);
  p->flag_stride = align_up(p->nb_full > 0 ? p->nb_full : 1, 16);
  p->nw_stride = ceil_div(p->nb_full > 0 ? p->nb_full : 1, 32);
  p->off_status = 256;
  p->off_tflags = align_up(p->off_status + 8 * (p->total_tiles + 1), 256);
  p->off_flags = align_up(p->off_tflags + 8 * (p->total_tiles + 1), 256);
  p->off_words = align_up(p->off_flags + p->flag_stride * ranks, 256);
  p->off_prefix = align_up(p->off_words + 4 * p->nw_stride * ranks, 256);
  p->off_rstate = align_up(p->off_prefix + 4 * p->nw_stride * ranks, 256);
  p->off_renc = align_up(p->off_rstate + 4 * static_cast<int64_t>(ranks), 256);
  p->off_rdec = align_up(p->off_renc + kRansEncTableBytes * ranks, 256);
  p->off_pred = align_up(p->off_rdec + kRansDecTableBytes * ranks, 256);
  p->off_result = align_up(p->off_pred + 4 * static_cast<int64_t>(ranks), 256);
  p->ws_bytes = align_up(p->off_result + 8 * static_cast<int64_t>(ranks), 256);
  p->fast = (block % 16 == 0) && block >= kFastMinBlock && block <= kFastMaxBlock &&
            (p->S % 16 == 0);
  // compress: flag words + their prefix (every call), then 2*TE values and
  // TE exponents (staged calls only)
  p->smem_flags = align_up(8 * ceil_div(p->T, 32), 128);
  p->smem_flags_hashed = align_up(align_up(8 * ceil_div(p->T, 32), 16) + 32 * p->T, 128);
  p->smem_decompress = p->fast ? 4 * p->T * block : 0;
  p->raw_fixup = raw_can_hold_unchanged(p->S, block) ||
                 raw_can_hold_unchanged(p->len_part, block);
  *out = p;
  return CIERA_OK;
}

int ciera_plan_info(ciera_plan_t p, ciera_plan_info_t* info) {
  if (!p || !info) return CIERA_E_INVAL;
  info->numel = p->numel;
  info->ranks = p->ranks;
  info->block = p->block;
  info->shard_len = p->S;
  info->blocks_per_shard = p->nb_full;
  info->tile_blocks = p->T;
  info->total_tiles = p->total_tiles;
  info->payload_capacity = p->capacity;
  info->workspace_bytes = p->ws_bytes;
  info->fast_path = p->fast ? 1 : 0;
  info->raw_fixup = p->raw_fixup ? 1 : 0;
  return CIERA_OK;
}

void ciera_plan_destroy(ciera_plan_t p) { delete p; }

int ciera_workspace_init(ciera_plan_t p, void* workspace_dev, void* stream) {
  if (!p || !workspace_dev) return CIERA_E_INVAL;
  cudaError_t e = cudaMemsetAsync(workspace_dev, 0, static_cast<size_t>(p->ws_bytes),
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CIERA_OK : CIERA_E_CUDA;
}

}  // extern "C"

namespace {

// Shared body of ciera_compress and ciera_compress_hashed.  Exactly one of
// sender_cache_dev / hash_cache_dev is used.
int compress_impl(ciera_plan_t p, int rank_begin, int rank_count, const uint16_t* w_dev,
                  uint8_t* sender_cache_dev, uint64_t* hash_cache_dev, bool hashed,
                  uint8_t* payloads_dev, int64_t payload_stride, ciera_desc* descs_dev,
                  uint8_t* flags_dev, void* workspace_dev, uint32_t flags, void* stream) {
  if (!p || rank_begin < 0 || rank_count < 1 ||
      static_cast<int64_t>(rank_begin) + rank_count > p->ranks)
    return CIERA_E_INVAL;
  if (!payloads_dev || !descs_dev || !workspace_dev || payload_stride < p->capacity)
    return CIERA_E_INVAL;
  if (hashed && p->T > 32) return CIERA_E_INVAL;  // block below 256 values
  const Geometry g = range_geometry(p, rank_begin, rank_count);
  if (g.total_tiles > 0 && (!w_dev || (hashed ? !hash_cache_dev : !sender_cache_dev)))
    return CIERA_E_INVAL;
  if (flags & ~kCompressFlags) return CIERA_E_INVAL;

  uint8_t* ws = static_cast<uint8_t*>(workspace_dev);
  CompressParams kp{};
  kp.geo = g;
  kp.w = w_dev;
  kp.scache = sender_cache_dev;
  kp.hash_cache = reinterpret_cast<unsigned long long*>(hash_cache_dev);
  kp.hash_stride = p->nb_full;
  kp.hashed = hashed ? 1 : 0;
  kp.payloads = payloads_dev;
  kp.stride = payload_stride;
  kp.descs = descs_dev;
  kp.flagbytes = flags_dev ? flags_dev : ws + p->off_flags;
  kp.flag_stride = flags_dev ? p->nb_full : p->flag_stride;
  kp.tile_status = reinterpret_cast<unsigned long long*>(ws + p->off_status);
  kp.tile_flags = reinterpret_cast<unsigned long long*>(ws + p->off_tflags);
  kp.ctl = reinterpret_cast<Control*>(ws);
  kp.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  kp.flags = flags;
  kp.fast = p->fast && aligned16(w_dev) && aligned16(payloads_dev) &&
            (payload_stride % 16 == 0) &&
            (hashed ? aligned16(hash_cache_dev) : aligned16(sender_cache_dev));
  // raw-ahead needs staged tiles of at most 32 blocks (flag bits in one word)
  kp.raw_ahead = kp.fast && p->T <= 32 && !(flags & CIERA_NO_RAW_AHEAD) ? 1 : 0;
  kp.pred = reinterpret_cast<uint32_t*>(ws + p->off_pred) + rank_begin;
  kp.result = reinterpret_cast<unsigned long long*>(ws + p->off_result) + rank_begin;
  const int64_t flag_region = hashed ? p->smem_flags_hashed : p->smem_flags;
  const int64_t smem = flag_region + (kp.fast ? 3 * p->T * p->block : 0);
  const int64_t repack_smem = 128 + 3 * p->T * p->block + 4 * ceil_div(rank_count, 32);
  const int e = launch_compress(kp, smem, p->raw_fixup ? 1 : 0, repack_smem, stream);
  return e == cudaSuccess ? CIERA_OK : CIERA_E_CUDA;
}

}  // namespace

extern "C" {

int ciera_compress(ciera_plan_t p, int rank_begin, int rank_count, const uint16_t* w_dev,
                   uint8_t* sender_cache_dev, uint8_t* payloads_dev, int64_t payload_stride,
                   ciera_desc* descs_dev, uint8_t* flags_dev, void* workspace_dev, uint32_t flags,
                   void* stream) {
  return compress_impl(p, rank_begin, rank_count, w_dev, sender_cache_dev, nullptr, false,
                       payloads_dev, payload_stride, descs_dev, flags_dev, workspace_dev, flags,
                       stream);
}

int ciera_compress_hashed(ciera_plan_t p, int rank_begin, int rank_count, const uint16_t* w_dev,
                          uint64_t* hash_cache_dev, uint8_t* payloads_dev, int64_t payload_stride,
                          ciera_desc* descs_dev, uint8_t* flags_dev, void* workspace_dev,
                          uint32_t flags, void* stream) {
  return compress_impl(p, rank_begin, rank_count, w_dev, nullptr, hash_cache_dev, true,
                       payloads_dev, payload_stride, descs_dev, flags_dev, workspace_dev, flags,
                       stream);
}

int ciera_compress_rans(ciera_plan_t p, int rank_begin, int rank_count, const uint16_t* w_dev,
                        uint8_t* sender_cache_dev, const uint32_t* hist_prev_dev,
                        uint32_t* hist_out_dev, uint8_t* payloads_dev, int64_t payload_stride,
                        ciera_desc* descs_dev, uint8_t* flags_dev, void* workspace_dev,
                        uint32_t flags, void* stream) {
  if (!p || rank_begin < 0 || rank_count < 1 ||
      static_cast<int64_t>(rank_begin) + rank_count > p->ranks)
    return CIERA_E_INVAL;
  if (!payloads_dev || !descs_dev || !workspace_dev || payload_stride < p->capacity ||
      !hist_prev_dev || !hist_out_dev)
    return CIERA_E_INVAL;
  if (flags & ~kCompressFlags) return CIERA_E_INVAL;
  // staged kernel only: every shard a multiple of 16 values, aligned operands
  if (!p->fast || p->numel % 16 != 0 || p->S > (int64_t(1) << 30) || p->T > 32)
    return CIERA_E_INVAL;
  const Geometry g = range_geometry(p, rank_begin, rank_count);
  if (g.total_tiles > 0 && (!w_dev || !sender_cache_dev)) return CIERA_E_INVAL;
  if ((g.total_tiles > 0 && (!aligned16(w_dev) || !aligned16(sender_cache_dev))) ||
      !aligned16(payloads_dev) || payload_stride % 16 != 0 ||
      (reinterpret_cast<uintptr_t>(hist_prev_dev) & 3u) ||
      (reinterpret_cast<uintptr_t>(hist_out_dev) & 3u))
    return CIERA_E_INVAL;
  const size_t hist_bytes = sizeof(uint32_t) * 256 * static_cast<size_t>(rank_count);
  {
    // the histograms must not overlap: the kernel reads one while adding into the other
    const uintptr_t a = reinterpret_cast<uintptr_t>(hist_prev_dev);
    const uintptr_t b = reinterpret_cast<uintptr_t>(hist_out_dev);
    if (a < b + hist_bytes && b < a + hist_bytes) return CIERA_E_INVAL;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(hist_out_dev, 0, hist_bytes, s) != cudaSuccess) return CIERA_E_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace_dev);
  CompressParams kp{};
  kp.geo = g;
  kp.w = w_dev;
  kp.scache = sender_cache_dev;
  kp.payloads = payloads_dev;
  kp.stride = payload_stride;
  kp.descs = descs_dev;
  kp.flagbytes = flags_dev ? flags_dev : ws + p->off_flags;
  kp.flag_stride = flags_dev ? p->nb_full : p->flag_stride;
  kp.tile_status = reinterpret_cast<unsigned long long*>(ws + p->off_status);
  kp.tile_flags = reinterpret_cast<unsigned long long*>(ws + p->off_tflags);
  kp.ctl = reinterpret_cast<Control*>(ws);
  kp.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  kp.flags = flags;
  kp.fast = 1;
  const int e = launch_compress_rans(kp, hist_prev_dev, hist_out_dev, ws + p->off_renc, stream);
  return e == cudaSuccess ? CIERA_OK : CIERA_E_CUDA;
}

}  // extern "C"

namespace {

// Receiver for ranks [rb, rb + rc) (Section 3.1; Algorithm 1, receiver).
// Every array is plan-wide and indexed by absolute rank or value: the
// payloads contiguous (rank r at payloads_dev + r*stride) or given by a
// device table of R pointers (each buffer holding at least `stride` bytes),
// the R descriptors, the N-value ExpCache and output; the workspace regions
// are per absolute rank too, so ranges of one plan may share a workspace.
int decompress_impl(ciera_plan_t p, int rb, int rc, const uint8_t* payloads_dev,
                    const uint8_t* const* payload_ptrs_dev, int64_t stride,
                    const ciera_desc* descs_dev, uint8_t* recv_cache_dev, uint16_t* out_dev,
                    void* workspace_dev, uint32_t flags, void* stream) {
  if (!p || rb < 0 || rc < 1 || static_cast<int64_t>(rb) + rc > p->ranks || !descs_dev ||
      !workspace_dev || (flags & ~CIERA_DECOMPRESS_RANS))
    return CIERA_E_INVAL;
  if (p->numel > 0 && (!recv_cache_dev || !out_dev)) return CIERA_E_INVAL;
  uint8_t* ws = static_cast<uint8_t*>(workspace_dev);
  const int64_t first = static_cast<int64_t>(rb) * p->S;  // first value of the range
  DecompressParams kp{};
  kp.geo = range_geometry(p, rb, rc);
  kp.payloads = payloads_dev ? payloads_dev + rb * stride : nullptr;
  kp.payload_ptrs = payload_ptrs_dev ? payload_ptrs_dev + rb : nullptr;
  kp.stride = stride;
  kp.descs = descs_dev + rb;
  kp.rcache = recv_cache_dev ? recv_cache_dev + first : nullptr;
  kp.out = out_dev ? out_dev + first : nullptr;
  kp.bm_words = reinterpret_cast<uint32_t*>(ws + p->off_words) + rb * p->nw_stride;
  kp.bm_prefix = reinterpret_cast<uint32_t*>(ws + p->off_prefix) + rb * p->nw_stride;
  kp.nw_stride = p->nw_stride;
  kp.rank_state = reinterpret_cast<uint32_t*>(ws + p->off_rstate) + rb;
  kp.ctl = reinterpret_cast<Control*>(ws);
  kp.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  // with a pointer table, each payload's alignment is checked by the bitmap
  // scan (a misaligned one is reported corrupt)
  kp.fast = p->fast && (payload_ptrs_dev || (aligned16(payloads_dev) && stride % 16 == 0)) &&
            aligned16(kp.rcache) && aligned16(kp.out);
  int e;
  if (flags & CIERA_DECOMPRESS_RANS) {
    if (!kp.fast || p->numel % 16 != 0) return CIERA_E_INVAL;
    kp.rans = 1;
    // the bitmap scan alone (no tiles), then the RANS receiver, which takes
    // the RAW ranks too
    DecompressParams scan = kp;
    scan.geo.total_tiles = 0;
    e = launch_decompress(scan, 0, stream);
    if (e == cudaSuccess)
      e = launch_decompress_rans(
          kp, reinterpret_cast<uint32_t*>(ws + p->off_rdec + kRansDecTableBytes * rb), stream);
  } else {
    e = launch_decompress(kp, kp.fast ? p->smem_decompress : 0, stream);
  }
  return e == cudaSuccess ? CIERA_OK : CIERA_E_CUDA;
}

}  // namespace

struct ciera_pipeline_s {
  int max_layers;
  cudaEvent_t fork;
  std::vector<cudaEvent_t> done;  // compress(i) finished
};

extern "C" {

int ciera_pipeline_create(int max_layers, ciera_pipeline_t* out) {
  if (!out || max_layers < 1) return CIERA_E_INVAL;
  ciera_pipeline_s* pp = new (std::nothrow) ciera_pipeline_s();
  if (!pp) return CIERA_E_INVAL;
  pp->max_layers = max_layers;
  pp->done.assign(static_cast<size_t>(max_layers), nullptr);
  bool ok = cudaEventCreateWithFlags(&pp->fork, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < max_layers; ++i)
    ok = cudaEventCreateWithFlags(&pp->done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    ciera_pipeline_destroy(pp);
    return CIERA_E_CUDA;
  }
  *out = pp;
  return CIERA_OK;
}

void ciera_pipeline_destroy(ciera_pipeline_t pp) {
  if (!pp) return;
  if (pp->fork) cudaEventDestroy(pp->fork);
  for (cudaEvent_t e : pp->done)
    if (e) cudaEventDestroy(e);
  delete pp;
}

int ciera_pipeline_step(ciera_pipeline_t pp, const ciera_layer* layers, int n, void* stream,
                        void* side_stream) {
  if (!pp || !layers || n < 1 || n > pp->max_layers || stream == side_stream)
    return CIERA_E_INVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t side = static_cast<cudaStream_t>(side_stream);
  // fork: the side stream starts after what is already queued on `stream`
  if (cudaEventRecord(pp->fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(side, pp->fork, 0) != cudaSuccess)
    return CIERA_E_CUDA;
  for (int i = 0; i < n; ++i) {
    const ciera_layer& L = layers[i];
    if (!L.plan || L.sender > CIERA_SENDER_HASHED) return CIERA_E_INVAL;
    const bool rans = L.sender == CIERA_SENDER_RANS;
    const int ranks = static_cast<int>(L.plan->ranks);
    int rc;
    if (rans)
      rc = ciera_compress_rans(L.plan, 0, ranks, L.w_dev, L.sender_cache_dev, L.hist_prev_dev,
                               L.hist_out_dev, L.payloads_dev, L.payload_stride, L.descs_dev,
                               nullptr, L.workspace_dev, L.flags, side);
    else if (L.sender == CIERA_SENDER_HASHED)
      rc = ciera_compress_hashed(L.plan, 0, ranks, L.w_dev, L.hash_cache_dev, L.payloads_dev,
                                 L.payload_stride, L.descs_dev, nullptr, L.workspace_dev,
                                 L.flags, side);
    else
      rc = ciera_compress(L.plan, 0, ranks, L.w_dev, L.sender_cache_dev, L.payloads_dev,
                          L.payload_stride, L.descs_dev, nullptr, L.workspace_dev, L.flags,
                          side);
    if (rc != CIERA_OK) return rc;
    if (cudaEventRecord(pp->done[i], side) != cudaSuccess ||
        cudaStreamWaitEvent(s, pp->done[i], 0) != cudaSuccess)
      return CIERA_E_CUDA;
    rc = ciera_decompress(L.plan, L.payloads_dev, L.payload_stride, L.descs_dev,
                          L.recv_cache_dev, L.out_dev, L.workspace_dev,
                          rans ? CIERA_DECOMPRESS_RANS : 0u, s);
    if (rc != CIERA_OK) return rc;
  }
  // join: the last decompress already waits for the last compress, and the
  // side stream does nothing after it
  return CIERA_OK;
}

int ciera_decompress(ciera_plan_t p, const uint8_t* payloads_dev, int64_t payload_stride,
                     const ciera_desc* descs_dev, uint8_t* recv_cache_dev, uint16_t* out_dev,
                     void* workspace_dev, uint32_t flags, void* stream) {
  if (!p || !payloads_dev || payload_stride < p->capacity) return CIERA_E_INVAL;
  return decompress_impl(p, 0, static_cast<int>(p->ranks), payloads_dev, nullptr, payload_stride,
                         descs_dev, recv_cache_dev, out_dev, workspace_dev, flags, stream);
}

int ciera_decompress_gather(ciera_plan_t p, const uint8_t* const* payload_ptrs_dev,
                            int64_t payload_capacity, const ciera_desc* descs_dev,
                            uint8_t* recv_cache_dev, uint16_t* out_dev, void* workspace_dev,
                            uint32_t flags, void* stream) {
  if (!p || !payload_ptrs_dev || payload_capacity < p->capacity ||
      (reinterpret_cast<uintptr_t>(payload_ptrs_dev) & 7u))
    return CIERA_E_INVAL;
  return decompress_impl(p, 0, static_cast<int>(p->ranks), nullptr, payload_ptrs_dev,
                         payload_capacity, descs_dev, recv_cache_dev, out_dev, workspace_dev,
                         flags, stream);
}

int ciera_status(void* workspace_dev, void* stream) {
  if (!workspace_dev) return CIERA_E_INVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Control* ctl = static_cast<Control*>(workspace_dev);
  uint32_t status = 0;
  if (cudaMemcpyAsync(&status, &ctl->status, sizeof(status), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return CIERA_E_CUDA;
  if (status != 0) {
    if (cudaMemsetAsync(&ctl->status, 0, sizeof(uint32_t), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return CIERA_E_CUDA;
  }
  if (status & kStatusInternal) return CIERA_E_INTERNAL;
  if (status & kStatusBounds) return CIERA_E_BOUNDS;
  if (status & kStatusTimeout) return CIERA_E_TIMEOUT;
  if (status & kStatusCorrupt) return CIERA_E_CORRUPT;
  return CIERA_OK;
}

int ciera_should_compress(int64_t numel) {
  ciera_cost_model m;
  {
    std::lock_guard<std::mutex> lk(g_cost_mu);
    m = g_cost;
  }
  if (numel <= 0) return 0;
  // Section 3.2: expected payload S_s+m + S_bm + q*S_e for a bf16 tensor
  // (S_s+m = S_e = N bytes); the link time it saves must exceed the
  // receiver's reconstruction time, the one kernel left on the critical path
  // once compression overlaps compute.
  const double n = static_cast<double>(numel);
  const double bitmap = static_cast<double>(ceil_div(ceil_div(numel, m.block), 8));
  const double payload = n + m.q_hat * n + bitmap;
  const double saved_s = (2.0 * n - payload) / m.link_Bps;
  const double decompress_s = m.t_fixed_s + (4.0 + m.q_hat) * n / m.hbm_Bps;
  return saved_s > decompress_s ? 1 : 0;
}

int ciera_bsc_select(const int64_t* numel, const double* q, int n, int world,
                     int64_t cache_budget_bytes, uint8_t* selected, double* gain) {
  if (n < 0 || world < 1 || cache_budget_bytes < 0 ||
      (n > 0 && (!numel || !q || !selected || !gain)))
    return CIERA_E_INVAL;
  for (int i = 0; i < n; ++i)
    if (numel[i] < 0 || !(q[i] >= 0.0) || !(q[i] <= 1.0)) return CIERA_E_INVAL;
  ciera_cost_model m;
  {
    std::lock_guard<std::mutex> lk(g_cost_mu);
    m = g_cost;
  }
  // Section 3.2: g_i = Comm(S_i) - Comm(S_s+m + S_bm + q_i S_e) - T_decmp,
  // with the exponents of the other W-1 ranks' shards as cache footprint.
  std::vector<int> cand;
  std::vector<double> ratio(static_cast<size_t>(n > 0 ? n : 0));
  for (int i = 0; i < n; ++i) {
    const double v = static_cast<double>(numel[i]);
    const double bitmap = static_cast<double>(ceil_div(ceil_div(numel[i], m.block), 8));
    const double saved_s = (2.0 * v - (v + bitmap + q[i] * v)) / m.link_Bps;
    const double decompress_s = m.t_fixed_s + (4.0 + q[i]) * v / m.hbm_Bps;
    gain[i] = saved_s - decompress_s;
    selected[i] = 0;
    const double footprint = static_cast<double>(world - 1) * v;
    ratio[i] = footprint > 0 ? gain[i] / footprint : 0.0;
    if (gain[i] > 0 && footprint > 0) cand.push_back(i);
  }
  // best benefit per cached byte first; equal ratios keep their order
  std::stable_sort(cand.begin(), cand.end(),
                   [&](int a, int b) { return ratio[a] > ratio[b]; });
  int taken = 0;
  int64_t used = 0;
  for (int i : cand) {
    const int64_t footprint = static_cast<int64_t>(world - 1) * numel[i];
    if (footprint <= cache_budget_bytes - used) {
      used += footprint;
      selected[i] = 1;
      ++taken;
    }
  }
  return taken;
}

int ciera_set_cost_model(const ciera_cost_model* model) {
  if (!model || !(model->link_Bps > 0) || !(model->hbm_Bps > 0) || !(model->q_hat >= 0) ||
      !(model->q_hat <= 1) || !(model->t_fixed_s >= 0) || model->block < 1)
    return CIERA_E_INVAL;
  std::lock_guard<std::mutex> lk(g_cost_mu);
  g_cost = *model;
  return CIERA_OK;
}

int ciera_get_cost_model(ciera_cost_model* model) {
  if (!model) return CIERA_E_INVAL;
  std::lock_guard<std::mutex> lk(g_cost_mu);
  *model = g_cost;
  return CIERA_OK;
}

int ciera_set_wait_timeout_ns(uint64_t ns) {
  if (ns == 0) return CIERA_E_INVAL;
  g_timeout_ns.store(ns, std::memory_order_relaxed);
  return CIERA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// One step from host memory and back (Algorithm 1's Send / Recv boundary as a
// single call): upload, sender, receiver and download, in chunks of ranks so
// that the upload of chunk c+1, the kernels of chunk c and the download of
// chunk c-1 run at the same time.

struct ciera_host_session_s {
  int max_chunks = 0;
  cudaStream_t s_in = nullptr, s_out = nullptr;  // upload and download streams
  cudaEvent_t fork = nullptr, join = nullptr;
  std::vector<cudaEvent_t> uploaded, rebuilt;    // per chunk
};

extern "C" {

void ciera_host_session_destroy(ciera_host_session_t h) {
  if (!h) return;
  for (cudaEvent_t e : h->uploaded)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : h->rebuilt)
    if (e) cudaEventDestroy(e);
  if (h->fork) cudaEventDestroy(h->fork);
  if (h->join) cudaEventDestroy(h->join);
  if (h->s_in) cudaStreamDestroy(h->s_in);
  if (h->s_out) cudaStreamDestroy(h->s_out);
  delete h;
}

int ciera_host_session_create(int max_chunks, ciera_host_session_t* out) {
  if (!out || max_chunks < 1) return CIERA_E_INVAL;
  ciera_host_session_s* h = new (std::nothrow) ciera_host_session_s();
  if (!h) return CIERA_E_INVAL;
  h->max_chunks = max_chunks;
  h->uploaded.assign(static_cast<size_t>(max_chunks), nullptr);
  h->rebuilt.assign(static_cast<size_t>(max_chunks), nullptr);
  bool ok = cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->fork, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&h->join, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < max_chunks; ++i)
    ok = cudaEventCreateWithFlags(&h->uploaded[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&h->rebuilt[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    ciera_host_session_destroy(h);
    return CIERA_E_CUDA;
  }
  *out = h;
  return CIERA_OK;
}

int ciera_step_host(ciera_host_session_t h, ciera_plan_t p, const uint16_t* w_host,
                    uint16_t* out_host, uint16_t* w_dev, uint8_t* sender_cache_dev,
                    uint8_t* payloads_dev, int64_t payload_stride, ciera_desc* descs_dev,
                    uint8_t* recv_cache_dev, uint16_t* out_dev, void* workspace_dev,
                    uint32_t flags, int chunks, void* stream) {
  if (!h || !p || chunks < 1 || chunks > h->max_chunks || (flags & ~kCompressFlags))
    return CIERA_E_INVAL;
  if (p->numel > 0 && (!w_host || !out_host || !w_dev || !out_dev)) return CIERA_E_INVAL;
  if (!payloads_dev || !descs_dev || !workspace_dev || payload_stride < p->capacity)
    return CIERA_E_INVAL;
  const int64_t R = p->ranks;
  const int64_t per = ceil_div(R, chunks < R ? chunks : R);  // ranks per chunk
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // fork: the copy streams start after what is already queued on `stream`
  if (cudaEventRecord(h->fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(h->s_in, h->fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(h->s_out, h->fork, 0) != cudaSuccess)
    return CIERA_E_CUDA;
  int c = 0;
  for (int64_t rb = 0; rb < R; rb += per, ++c) {
    const int64_t rc = rb + per < R ? per : R - rb;
    const int64_t v0 = rb * p->S < p->numel ? rb * p->S : p->numel;
    const int64_t v1 = (rb + rc) * p->S < p->numel ? (rb + rc) * p->S : p->numel;
    const size_t bytes = static_cast<size_t>(2 * (v1 - v0));
    if (bytes > 0 && cudaMemcpyAsync(w_dev + v0, w_host + v0, bytes, cudaMemcpyHostToDevice,
                                     h->s_in) != cudaSuccess)
      return CIERA_E_CUDA;
    if (cudaEventRecord(h->uploaded[c], h->s_in) != cudaSuccess ||
        cudaStreamWaitEvent(s, h->uploaded[c], 0) != cudaSuccess)
      return CIERA_E_CUDA;
    int rcode = ciera_compress(p, static_cast<int>(rb), static_cast<int>(rc), w_dev + v0,
                               sender_cache_dev ? sender_cache_dev + v0 : nullptr,
                               payloads_dev ? payloads_dev + rb * payload_stride : nullptr,
                               payload_stride, descs_dev ? descs_dev + rb : nullptr, nullptr,
                               workspace_dev, flags, s);
    if (rcode != CIERA_OK) return rcode;
    rcode = decompress_impl(p, static_cast<int>(rb), static_cast<int>(rc), payloads_dev, nullptr,
                            payload_stride, descs_dev, recv_cache_dev, out_dev, workspace_dev, 0,
                            s);
    if (rcode != CIERA_OK) return rcode;
    if (cudaEventRecord(h->rebuilt[c], s) != cudaSuccess ||
        cudaStreamWaitEvent(h->s_out, h->rebuilt[c], 0) != cudaSuccess)
      return CIERA_E_CUDA;
    if (bytes > 0 && cudaMemcpyAsync(out_host + v0, out_dev + v0, bytes, cudaMemcpyDeviceToHost,
                                     h->s_out) != cudaSuccess)
      return CIERA_E_CUDA;
  }
  // join: every upload precedes a kernel on `stream`; wait for the downloads
  if (cudaEventRecord(h->join, h->s_out) != cudaSuccess ||
      cudaStreamWaitEvent(s, h->join, 0) != cudaSuccess)
    return CIERA_E_CUDA;
  return CIERA_OK;
}

}  // extern "C"
