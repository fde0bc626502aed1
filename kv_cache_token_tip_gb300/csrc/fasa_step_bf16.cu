// Instantiations and launch of the bf16 fused-step kernel.
#include "fasa_step.cuh"

namespace fasa {

namespace {

// Opts the kernel into the largest dynamic shared memory the device allows
// and into non-portable (up to 16 CTA) clusters; once per process.
template <int D>
cudaError_t prepare_step() {
  static cudaError_t once = [] {
    auto k = fasa_step_kernel<D>;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  }();
  return once;
}

cudaLaunchConfig_t step_config(int C, int units, int smem, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, (unsigned)units, 1);
  cfg.blockDim = dim3(SNT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int D>
cudaError_t launch_d(const StepParams& p, int C, cudaStream_t s) {
  cudaError_t e = prepare_step<D>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = step_config(C, p.B * p.Hkv, p.smem_total, s, attr);
  return cudaLaunchKernelEx(&cfg, fasa_step_kernel<D>, p);
}

template <int D>
int max_clusters_d(int C, int smem) {
  if (prepare_step<D>() != cudaSuccess) return 0;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = step_config(C, 1, smem, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fasa_step_kernel<D>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

cudaError_t launch_step_bf16(const StepParams& p, int head_dim, int C, cudaStream_t s) {
  if (head_dim == 128) return launch_d<128>(p, C, s);
  if (head_dim == 64) return launch_d<64>(p, C, s);
  return cudaErrorInvalidValue;
}

#ifdef FASA_PHASE_TRACE
// Tracing builds: where the step kernel stores its phase timestamps.
extern "C" int fasa_debug_set_trace(void* buf) {
  unsigned long long* p = reinterpret_cast<unsigned long long*>(buf);
  return (int)cudaMemcpyToSymbol(g_step_trace, &p, sizeof(p));
}
#endif

int max_active_clusters_step_bf16(int head_dim, int C, int smem_bytes) {
  if (head_dim == 128) return max_clusters_d<128>(C, smem_bytes);
  if (head_dim == 64) return max_clusters_d<64>(C, smem_bytes);
  return 0;
}

}  // namespace fasa
