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
// every GPU that loads this library holds until the process exits.  Plans
// that share the array share its predictions too; a stale prediction only
// costs the rewrite of a shard, never its bytes.
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
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device.  In host code the name
// g_scratch is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CIERA_E_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return CIERA_E_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return CIERA_OK;
}

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
  const int st = scratch_address(&scratch);
  if (st != CIERA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents.  The ticket count (the
  // low half of the counter word) and the status word must start at zero;
  // the launch number in the counter's high half must be kept, because the
  // look-back and flag words are tagged with it, and the flag bytes are
  // rewritten before they are read.
  unsigned char* ctl = static_cast<unsigned char*>(scratch);
  if (cudaMemsetAsync(ctl + offsetof(ciera::Control, ticket), 0, sizeof(uint32_t), s) !=
          cudaSuccess ||
      cudaMemsetAsync(ctl + offsetof(ciera::Control, status), 0, sizeof(uint32_t), s) !=
          cudaSuccess)
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
