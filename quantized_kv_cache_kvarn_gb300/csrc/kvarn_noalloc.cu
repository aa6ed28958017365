// kvarn_decode_noalloc: kvarn_decode with its split-K scratch taken from a
// fixed array inside the library instead of a caller-supplied workspace.
//
// Some callers can not allocate device memory: a plugin that a host
// framework hands only its input and output tensors, a process whose device
// memory is entirely owned by a pool allocator, or a latency-bound path that
// cannot afford the device-wide synchronisation a cudaMalloc may impose.
// For them this entry point reads and writes its partials in
// kDecodeScratchBytes of static device memory that every GPU loading the
// library holds until the process exits, and allocates nothing.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "../../include/kvarn.h"
#include "kvarn_launch.h"

namespace {

constexpr int64_t kDecodeScratchBytes = KVARN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kDecodeScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lookup;
std::atomic<void*> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device. In host code
// the array's name is only a host-side stand-in, so the address is asked of
// the runtime, with that device current, on the first call that finds none
// cached. Only a successful lookup is kept: a call that failed (during a
// stream capture, say) leaves the next call to try again.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_lookup);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      e = cudaGetSymbolAddress(&p, g_decode_scratch);
      if (e != cudaSuccess) return e;
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" int32_t kvarn_decode_noalloc(const void* q, int32_t num_q_heads, float sm_scale,
                                        const void* cache, const kvarn_layout* layout,
                                        const int32_t* block_table, int32_t bt_stride,
                                        const int32_t* seq_lens, int32_t max_seq_len,
                                        const void* tail_k, const void* tail_v, int32_t num_seqs,
                                        float* out, float* lse, uint32_t* error_flags,
                                        kvarn_stream_t stream) {
  const int64_t need = kvarn_decode_workspace_bytes(layout, num_seqs, num_q_heads, max_seq_len);
  if (need < 0) return KVARN_EINVAL;
  if (need > kDecodeScratchBytes) return KVARN_EWORKSPACE;
  if (num_seqs == 0) return KVARN_OK;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KVARN_ECUDA;
  return kvarn_decode(q, num_q_heads, sm_scale, cache, layout, block_table, bt_stride, seq_lens,
                      max_seq_len, tail_k, tail_v, num_seqs, out, lse, scratch, kDecodeScratchBytes,
                      error_flags, stream);
}
