// ciera_noalloc.cu -- ciera_compress_noalloc: the sender side with its scratch
// memory in a fixed device array instead of a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the point where they
// compress: code running inside a framework's communication hook or an
// allocator callback (where allocating would re-enter the allocator), code
// that must not grow its memory footprint mid-step, or plain C callers that
// have no allocator of their own for a scratch buffer.  They still own and
// pass every input and output; only the scratch (tile look-back words, the
// ticket counter, the status word, per-block flag bytes, the per-rank
// raw-ahead prediction and result words) comes from g_scratch below, which
// every GPU that loads this library holds until the process exits.
//
// Where a plan keeps each piece of scratch (look-back words, flag words, flag
// bytes, predictions) depends on its size, rank count and block size.  A
// call whose plan has another shape than the previous call's on the same
// device would find the previous plan's bytes in its own regions -- for
// instance flag bytes where it expects launch-tagged flag words, which could
// read as a word of its own launch.  So the first call on a device, and
// every call whose plan shape differs from the previous call's there, clears
// the scratch the plan uses (all of it but the launch counter) before its
// kernels run.  Calls of one plan shape reuse the scratch as a workspace is
// reused.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "ciera.h"
#include "ciera_internal.h"

namespace {

// Fixed scratch, shared by every call on a device.  8 MiB covers plans whose
// workspace (ciera_plan_info_t.workspace_bytes) is at most this size, e.g.
// 2.4e9 values over 32 ranks in blocks of 4096.
constexpr size_t kScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

// The plan shape that fixes the scratch layout (every offset of a workspace
// follows from these three numbers).
struct Shape {
  int64_t numel = -1, ranks = -1, block = -1;
  bool operator==(const Shape& o) const {
    return numel == o.numel && ranks == o.ranks && block == o.block;
  }
};

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
Shape g_last_shape[kMaxDevices];  // shape of the last call on each device

// Device address of g_scratch on the current device, and whether `shape`
// differs from the previous call's on that device (recorded as the new last
// shape).  In host code the name g_scratch is only a host-side stand-in, so
// the address comes from cudaGetSymbolAddress, once per device, with that
// device current.
int scratch_address(const Shape& shape, void** out, bool* shape_changed) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CIERA_E_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return CIERA_E_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *shape_changed = !(g_last_shape[dev] == shape);
  g_last_shape[dev] = shape;
  *out = g_scratch_ptr[dev];
  return CIERA_OK;
}

static_assert(offsetof(ciera::Control, ticket) == 0 && sizeof(ciera::Control::ticket) == 8,
              "the launch counter is the first 8 bytes of the scratch");
static_assert(CIERA_STATUS_CORRUPT == ciera::kStatusCorrupt &&
                  CIERA_STATUS_TIMEOUT == ciera::kStatusTimeout &&
                  CIERA_STATUS_INTERNAL == ciera::kStatusInternal &&
                  CIERA_STATUS_BOUNDS == ciera::kStatusBounds,
              "status bits of the public header and of the kernels agree");

}  // namespace

extern "C" int ciera_compress_noalloc(ciera_plan_t plan, int rank_begin, int rank_count,
                                      const uint16_t* w_dev, uint8_t* sender_cache_dev,
                                      uint8_t* payloads_dev, int64_t payload_stride,
                                      ciera_desc* descs_dev, uint8_t* flags_dev,
                                      uint32_t* status_dev, uint32_t flags, void* stream) {
  ciera_plan_info_t info;
  if (ciera_plan_info(plan, &info) != CIERA_OK) return CIERA_E_INVAL;
  if (info.workspace_bytes > static_cast<int64_t>(kScratchBytes)) return CIERA_E_INVAL;
  void* scratch = nullptr;
  bool shape_changed = false;
  const int st =
      scratch_address(Shape{info.numel, info.ranks, info.block}, &scratch, &shape_changed);
  if (st != CIERA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents.  The ticket count (the
  // low half of the counter word) and the status word must start at zero;
  // the launch number in the counter's high half must be kept, because the
  // look-back and flag words are tagged with it.  After a change of plan
  // shape everything past the counter is cleared as well: zero never
  // matches a launch tag, and a zero prediction only sends a shard through
  // the look-back.
  unsigned char* ctl = static_cast<unsigned char*>(scratch);
  if (cudaMemsetAsync(ctl + offsetof(ciera::Control, ticket), 0, sizeof(uint32_t), s) !=
      cudaSuccess)
    return CIERA_E_CUDA;
  const size_t clear_from = offsetof(ciera::Control, status);
  const size_t clear_to =
      shape_changed ? static_cast<size_t>(info.workspace_bytes) : clear_from + sizeof(uint32_t);
  if (cudaMemsetAsync(ctl + clear_from, 0, clear_to - clear_from, s) != cudaSuccess)
    return CIERA_E_CUDA;
  const int rc = ciera_compress(plan, rank_begin, rank_count, w_dev, sender_cache_dev,
                                payloads_dev, payload_stride, descs_dev, flags_dev, scratch,
                                flags, s);
  if (rc != CIERA_OK) return rc;
  if (status_dev) {
    const unsigned char* status_word =
        static_cast<const unsigned char*>(scratch) + offsetof(ciera::Control, status);
    if (cudaMemcpyAsync(status_dev, status_word, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess)
      return CIERA_E_CUDA;
  }
  return CIERA_OK;
}
