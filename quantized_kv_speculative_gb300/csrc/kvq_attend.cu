// Dispatch of the attention kernel over read modes, and the bounded-wait self
// test.  The kernel itself is in kvq_attend_kernel.cuh; each mode's variants
// are compiled in kvq_attend_<mode>.cu.
#include "kvq_modes.cuh"

namespace kvq {
template <int MODE, bool SC> int attend_resident_m(int D, int NJ, int R);
template <int MODE, bool SC> int attend_clusters_m(int D, int NJ, int R, int size);
template <int MODE, bool SC> cudaError_t attend_launch_m(const AttendParams& p, cudaStream_t s);


// The scoring variants exist for the modes that have low-bit keys to rank
// (INT4, INT2, INT1); INT8 has none.
int attend_resident_ctas(int mode, int D, int G, int R, bool score) {
  const int NJ = D / G;
  switch (mode) {
    case KVQ_MODE_INT8: return score ? 0 : attend_resident_m<KVQ_MODE_INT8, false>(D, NJ, R);
    case KVQ_MODE_INT4:
      return score ? attend_resident_m<KVQ_MODE_INT4, true>(D, NJ, R) : attend_resident_m<KVQ_MODE_INT4, false>(D, NJ, R);
    case KVQ_MODE_INT2:
      return score ? attend_resident_m<KVQ_MODE_INT2, true>(D, NJ, R) : attend_resident_m<KVQ_MODE_INT2, false>(D, NJ, R);
    case KVQ_MODE_INT1:
      return score ? attend_resident_m<KVQ_MODE_INT1, true>(D, NJ, R) : attend_resident_m<KVQ_MODE_INT1, false>(D, NJ, R);
    default: return 0;
  }
}

int attend_resident_clusters(int mode, int D, int G, int R, int size, bool score) {
  const int NJ = D / G;
  switch (mode) {
    case KVQ_MODE_INT8: return score ? 0 : attend_clusters_m<KVQ_MODE_INT8, false>(D, NJ, R, size);
    case KVQ_MODE_INT4:
      return score ? attend_clusters_m<KVQ_MODE_INT4, true>(D, NJ, R, size)
                   : attend_clusters_m<KVQ_MODE_INT4, false>(D, NJ, R, size);
    case KVQ_MODE_INT2:
      return score ? attend_clusters_m<KVQ_MODE_INT2, true>(D, NJ, R, size)
                   : attend_clusters_m<KVQ_MODE_INT2, false>(D, NJ, R, size);
    case KVQ_MODE_INT1:
      return score ? attend_clusters_m<KVQ_MODE_INT1, true>(D, NJ, R, size)
                   : attend_clusters_m<KVQ_MODE_INT1, false>(D, NJ, R, size);
    default: return 0;
  }
}

cudaError_t launch_attend(const AttendParams& p, int mode, bool score, cudaStream_t s) {
  switch (mode) {
    case KVQ_MODE_INT8: return score ? cudaErrorInvalidValue : attend_launch_m<KVQ_MODE_INT8, false>(p, s);
    case KVQ_MODE_INT4: return score ? attend_launch_m<KVQ_MODE_INT4, true>(p, s) : attend_launch_m<KVQ_MODE_INT4, false>(p, s);
    case KVQ_MODE_INT2: return score ? attend_launch_m<KVQ_MODE_INT2, true>(p, s) : attend_launch_m<KVQ_MODE_INT2, false>(p, s);
    case KVQ_MODE_INT1: return score ? attend_launch_m<KVQ_MODE_INT1, true>(p, s) : attend_launch_m<KVQ_MODE_INT1, false>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

// Bounded-wait self test: one CTA waits on an mbarrier that nothing arrives at.
__global__ void wait_selftest_kernel(int* status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(&bar, 0, limit)) record_status(status, KVQ_ERR_DEVICE_TIMEOUT);
    // leave the barrier consistent: complete the pending phase before exit
    mbar_arrive(&bar);
  }
}

cudaError_t launch_wait_selftest(int* status, long long limit, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit);
  return cudaGetLastError();
}

}  // namespace kvq
