// Instantiations of the cluster kernel for fp32 storage.
#include "fasa_cluster.cuh"

namespace fasa {

cudaError_t launch_cluster_f32(const Params& p, int head_dim, int C, cudaStream_t s) {
  if (head_dim == 128) return launch_cluster_t<float, 128>(p, C, s);
  if (head_dim == 64) return launch_cluster_t<float, 64>(p, C, s);
  return cudaErrorInvalidValue;
}

int max_active_clusters_f32(int flags, int head_dim, int C, int smem_bytes) {
  if (head_dim == 128) return max_clusters_t<float, 128>(flags, C, smem_bytes);
  if (head_dim == 64) return max_clusters_t<float, 64>(flags, C, smem_bytes);
  return 0;
}

}  // namespace fasa
