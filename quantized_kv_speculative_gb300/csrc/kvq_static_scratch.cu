// Attention for callers that cannot allocate device memory.
//
// kvq_attend needs a caller-provided workspace: split partials, per-(b, kv head)
// ticket counters and a status word.  Some callers cannot make that
// allocation.  Examples: a decode loop that must not allocate after start-up
// (an allocation can synchronize the device or break a pre-reserved memory
// pool), or an integration layer that has no device allocator of its own.
// kvq_attend_static_scratch runs the same attention with its workspace in a
// fixed array compiled into this library.  It allocates nothing.
#include <cstring>
#include <mutex>

#include "kvq_internal.h"

namespace {

// Fixed scratch for kvq_attend_static_scratch.  It lives in every GPU that
// loads this library, for the life of the process.
constexpr size_t kStaticScratchBytes = static_cast<size_t>(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_attend_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The array's name
// in host code is only a host-side stand-in, so its device address is looked
// up once per device with that device current, and remembered.  Under CUDA's
// lazy module loading this first lookup may load the library's module on the
// device, which reserves the array there (and can synchronize), so callers
// make their first call at start-up.
kvq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attend_scratch) != cudaSuccess || p == nullptr) return KVQ_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_attend_static_scratch(const kvq_cache* cache, kvq_mode mode, const void* q,
                                                int32_t num_q_heads, int32_t gamma, const void* pend_k,
                                                const void* pend_v, int32_t n_pend, const int32_t* sel_idx,
                                                const void* sel_k, const void* sel_v, int32_t top_k,
                                                float sm_scale, void* out, float* lse, kvq_stream_t stream) {
  // Every argument is checked, with kvq_attend's own status codes, before
  // anything is enqueued on the shared array.
  size_t need = 0;
  const kvq_status chk = kvq::attend_check(cache, mode, q, num_q_heads, gamma, pend_k, pend_v, n_pend, sel_idx,
                                           sel_k, sel_v, top_k, out, lse, &need);
  if (chk != KVQ_OK) return chk;
  if (need > kStaticScratchBytes) return KVQ_ERR_WORKSPACE;   // this cache needs more than 16 MiB
  void* scratch = nullptr;
  const kvq_status st = scratch_address(&scratch);
  if (st != KVQ_OK) return st;
  // The ticket counters must start at zero.  A finished call leaves them at
  // zero, but an earlier call that gave up on the device might not have.  The
  // status word and the partials need no clearing.
  const size_t units = static_cast<size_t>(cache->desc.batch) * cache->desc.num_kv_heads;
  const size_t counter_bytes = (units * 4 + 255) & ~static_cast<size_t>(255);
  if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + kvq::kStatusBytes, 0, counter_bytes,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return kvq_attend(cache, mode, q, num_q_heads, gamma, pend_k, pend_v, n_pend, sel_idx, sel_k, sel_v,
                    top_k, sm_scale, out, lse, scratch, kStaticScratchBytes, stream);
}
