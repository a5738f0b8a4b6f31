// The attention kernel's INT1 variants that also score every quantized
// token for the next step's top-k (kvq_attend_topk), compiled on their own.
#include "kvq_attend_kernel.cuh"

namespace kvq {
template int attend_resident_m<KVQ_MODE_INT1, true>(int, int, int);
template int attend_clusters_m<KVQ_MODE_INT1, true>(int, int, int, int);
template cudaError_t attend_launch_m<KVQ_MODE_INT1, true>(const AttendParams&, cudaStream_t);
}  // namespace kvq
