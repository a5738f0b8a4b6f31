// The attention kernel's INT1 variants (all head dims, group sizes and
// row counts), compiled on their own so that the modes build in parallel.
#include "kvq_attend_kernel.cuh"

namespace kvq {
template int attend_resident_m<KVQ_MODE_INT1, false>(int, int, int);
template int attend_clusters_m<KVQ_MODE_INT1, false>(int, int, int, int);
template cudaError_t attend_launch_m<KVQ_MODE_INT1, false>(const AttendParams&, cudaStream_t);
}  // namespace kvq
