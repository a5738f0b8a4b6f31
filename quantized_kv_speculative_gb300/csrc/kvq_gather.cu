// Gather of the selected tokens' 16-bit K/V from the full-precision store.
//
// The pages: SpeCache keeps the full 16-bit KV cache in CPU memory and a
// low-bit copy on the GPU, and each step fetches the top-k 16-bit KV pairs
// that the speculative token predicted (SpeCache page, "Approach"); the page's
// limitations note that its sparse CPU-GPU transfer, done with PyTorch
// streams, is several times slower per byte than a full transfer.  MSpecKV
// likewise keeps offloaded KV and reconstructs only the needed subsets on
// demand (MSpecKV page, abstract).
//
// On a Grace-Blackwell node the host memory is reachable from the GPU over
// NVLink-C2C, so the fetch is one kernel that reads the selected rows straight
// out of pinned host memory (or device memory) into the device buffers that
// kvq_attend takes as sel_k / sel_v.  Each warp moves whole rows with 16-byte
// loads, with eight entries' loads in flight per lane before any store, so
// that the link sees thousands of independent 256-byte requests at once.
#include <algorithm>
#include <cstdint>

#include "kvq.h"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherPasses = 8;   // entries' loads in flight per lane

__device__ __forceinline__ uint4 ld_nc16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Entry e = (u, j) with u = b * Hkv + kvh: row idx[e] of unit u's K and V
// (16-byte chunks c of D / 8 per row) to row e of sel_k / sel_v.  A warp pass
// covers 128 / D entries: lanes [0, D/8) the K row, the next D/8 lanes the V
// row, and so on.  An index outside [0, full_tokens) gives a zero row.
template <int D>
__global__ void __launch_bounds__(kGatherThreads) gather_selected_kernel(const uint4* __restrict__ fk,
                                                                        const uint4* __restrict__ fv,
                                                                        long long full_tokens,
                                                                        const int32_t* __restrict__ idx, int top_k,
                                                                        long long n_entries, uint4* __restrict__ sk,
                                                                        uint4* __restrict__ sv) {
  constexpr int LPR = D / 8;              // lanes (16-byte chunks) per row
  constexpr int EPP = 32 / (2 * LPR);     // entries per warp pass
  const int lane = threadIdx.x & 31;
  const int sub = lane / (2 * LPR), is_v = (lane / LPR) & 1, c = lane % LPR;
  const uint4* src_base = is_v ? fv : fk;
  uint4* dst_base = is_v ? sv : sk;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long base = warp0 * EPP * kGatherPasses; base < n_entries; base += nwarps * EPP * kGatherPasses) {
    uint4 v[kGatherPasses];
    long long dst[kGatherPasses];
#pragma unroll
    for (int ps = 0; ps < kGatherPasses; ++ps) {
      const long long e = base + ps * EPP + sub;
      v[ps] = make_uint4(0u, 0u, 0u, 0u);
      dst[ps] = -1;
      if (e < n_entries) {
        const long long u = e / top_k;
        const long long t = idx[e];
        if (t >= 0 && t < full_tokens) v[ps] = ld_nc16(src_base + (u * full_tokens + t) * LPR + c);
        dst[ps] = e * LPR + c;
      }
    }
#pragma unroll
    for (int ps = 0; ps < kGatherPasses; ++ps)
      if (dst[ps] >= 0) dst_base[dst[ps]] = v[ps];
  }
}

// The address a kernel uses for `p`, or nullptr when the device cannot reach
// it (pageable host memory).  Pinned host memory maps to its device alias.
const void* device_view(const void* p, bool allow_host) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return p;
    case cudaMemoryTypeHost:
      return allow_host ? a.devicePointer : nullptr;
    default:
      return nullptr;
  }
}

int sm_count_now() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_gather_selected(const void* full_k, const void* full_v, int64_t full_tokens, int32_t batch,
                                          int32_t num_kv_heads, int32_t head_dim, const int32_t* sel_idx,
                                          int32_t top_k, void* sel_k, void* sel_v, kvq_stream_t stream) {
  if (!full_k || !full_v || !sel_idx || !sel_k || !sel_v) return KVQ_ERR_INVALID_ARG;
  if (batch < 1 || num_kv_heads < 1 || full_tokens < 1 || top_k < 1 || top_k > kMaxTopk) return KVQ_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(full_k) || !aligned16(full_v) || !aligned16(sel_k) || !aligned16(sel_v) ||
      (reinterpret_cast<uintptr_t>(sel_idx) & 3u))
    return KVQ_ERR_INVALID_ARG;
  const void* fk = device_view(full_k, true);
  const void* fv = device_view(full_v, true);
  if (!fk || !fv || !device_view(sel_idx, false) || !device_view(sel_k, false) || !device_view(sel_v, false))
    return KVQ_ERR_INVALID_ARG;
  const long long n = static_cast<long long>(batch) * num_kv_heads * top_k;
  const int epw = (128 / head_dim) * kGatherPasses;             // entries per warp per sweep
  const long long warps = (n + epw - 1) / epw;
  const long long per_cta = kGatherThreads / 32;
  const int sms = sm_count_now();
  const long long cap = sms > 0 ? static_cast<long long>(sms) * 8 : 1216;   // 8 CTAs of 256 threads per SM
  const unsigned grid = static_cast<unsigned>(std::max(1LL, std::min(cap, (warps + per_cta - 1) / per_cta)));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (head_dim == 128)
    gather_selected_kernel<128><<<grid, kGatherThreads, 0, s>>>(
        static_cast<const uint4*>(fk), static_cast<const uint4*>(fv), full_tokens, sel_idx, top_k, n,
        static_cast<uint4*>(sel_k), static_cast<uint4*>(sel_v));
  else
    gather_selected_kernel<64><<<grid, kGatherThreads, 0, s>>>(
        static_cast<const uint4*>(fk), static_cast<const uint4*>(fv), full_tokens, sel_idx, top_k, n,
        static_cast<uint4*>(sel_k), static_cast<uint4*>(sel_v));
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
