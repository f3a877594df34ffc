// lora_linear_forward_noalloc: one projection slot for callers that cannot allocate.
//
// The ordinary path asks the caller for a device workspace (segments, work lists and fp32
// scratch, see lora_segments_size).  Some callers have no way to provide one: a plugin whose
// host runtime owns all device memory and hands it only its inputs and outputs, code that
// records into a CUDA graph while stream capture forbids cudaMalloc, or a latency-critical
// loop that must not risk the device-wide synchronisation an allocation can cause.  For
// them this file keeps the scratch in one statically sized device array that exists on
// every GPU that loads the library, and runs the same kernels over it.
//
// Limits: at most kNoAllocMaxTokens tokens per call and a hidden size of at most
// kNoAllocMaxH.  All calls share the array, so calls whose work overlaps on the GPU (two
// streams, or two host threads) race; calls ordered on one stream do not.  Nothing in the
// array has to start at zero: each call rebuilds every value it later reads.
#include <cuda_runtime.h>

#include <mutex>

#include "lora_internal.h"

namespace {

constexpr int32_t kNoAllocMaxTokens = LORA_NOALLOC_MAX_TOKENS;
constexpr int32_t kNoAllocMaxH = LORA_NOALLOC_MAX_H;
// What one call needs at the limits (128 tokens, H = 8192, any number of adapters): the fp32
// LoRA delta, 128 x 8192 x 4 B = 4 MiB; the base GEMM's split-K partial sums, 3 tiles of
// 128 tokens x 8192 features x 4 B = 12 MiB; and under 8 KiB of token ids, segments and work
// units.  The array has 17 MiB; the assertion below recomputes the layout at the limits.
constexpr size_t kScratchBytes = (size_t)LORA_NOALLOC_SCRATCH_BYTES;
static_assert(segments_layout(kNoAllocMaxTokens, kNoAllocMaxH, LORA_MAX_ADAPTERS, 1).total <= kScratchBytes,
              "the static scratch array must hold a workspace at the entry point's limits");

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, resolved once per device.
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return lora_cuda_fail(e, "lora_linear_forward_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return lora_fail(LORA_EINVAL, "lora_linear_forward_noalloc: device ordinal too large");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return lora_cuda_fail(e, "lora_linear_forward_noalloc: cudaGetSymbolAddress");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LORA_OK;
}

}  // namespace

extern "C" int lora_linear_forward_noalloc(lora_pool* pool, const int32_t* token_adapter, int32_t T, int32_t slot,
                                           const void* x, const void* W, void* y, lora_stream_t stream) {
  if (!pool) return lora_fail(LORA_EINVAL, "lora_linear_forward_noalloc: pool is NULL");
  if (T < 0 || T > kNoAllocMaxTokens)
    return lora_fail(LORA_EINVAL, "lora_linear_forward_noalloc: T = " + std::to_string(T) + " exceeds the limit of " +
                                      std::to_string(kNoAllocMaxTokens) + " tokens per call");
  if (pool->H > kNoAllocMaxH)
    return lora_fail(LORA_EINVAL, "lora_linear_forward_noalloc: hidden size " + std::to_string(pool->H) +
                                      " exceeds the limit of " + std::to_string(kNoAllocMaxH));
  const int32_t T_ws = T > 0 ? T : 1;
  const int64_t need = lora_segments_size(pool, T_ws);
  if (need < 0) return (int)need;
  if ((size_t)need > kScratchBytes)
    return lora_fail(LORA_EINVAL, "lora_linear_forward_noalloc: needs " + std::to_string(need) +
                                      " bytes of scratch, the static array holds " + std::to_string(kScratchBytes));
  void* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc != LORA_OK) return rc;
  lora_segments seg;
  rc = lora_segments_init(pool, scratch, (int64_t)kScratchBytes, T_ws, &seg);
  if (rc == LORA_OK) rc = lora_segments_build(pool, token_adapter, T, &seg, stream);
  if (rc == LORA_OK) rc = lora_linear_forward(pool, &seg, slot, x, W, y, nullptr, stream);
  return rc;
}
