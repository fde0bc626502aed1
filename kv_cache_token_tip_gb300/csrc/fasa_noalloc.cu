// fasa_decode_step_noalloc: the fused decode step for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all: plug-ins inside a host runtime
// that owns every device allocation and hands out none, services that forbid
// device allocation after start-up (an allocation synchronises the device
// and can fail under memory pressure at any time), or code that must not
// grow its memory footprint while serving.  fasa_decode_step asks such a
// caller for a score workspace whenever a CTA's share of the cached tokens
// does not fit in shared memory.  This entry point instead uses a fixed
// scratch array that lives in the library image: FASA_NOALLOC_SCRATCH_BYTES
// of device memory, reserved on every GPU that loads the library until the
// process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fasa.h"

namespace {

constexpr size_t kScratchFloats = FASA_NOALLOC_SCRATCH_BYTES / sizeof(float);

// The score workspace of every call of this entry point.  In host code this
// name is only a stand-in for the symbol, never a device address: the device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scores[kScratchFloats];

// Device address of g_noalloc_scores, looked up once per device with that
// device current.
int scratch_address(float** out) {
  static std::mutex mu;
  static float* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return FASA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scores);
    if (e != cudaSuccess) return FASA_ERR_CUDA;
    addr[dev] = static_cast<float*>(p);
  }
  *out = addr[dev];
  return FASA_OK;
}

}  // namespace

extern "C" int fasa_decode_step_noalloc(const void* q, const int32_t* pos, const void* k_cache,
                                        const void* v_cache, const void* k_dom, const int32_t* dom_fc,
                                        const int32_t* seq_lens, int32_t budget, float* out,
                                        int32_t* idx_out, int32_t* count_out, const fasa_dims_t* dims,
                                        fasa_stream_t stream) {
  size_t need = 0;
  int st = fasa_workspace_size(dims, budget, &need);
  if (st != FASA_OK) return st;
  // When the automatic plan's workspace exceeds the scratch array, larger
  // clusters split each unit's tokens finer and need less (none once every
  // CTA's scores fit in shared memory); the first that fits is used.
  fasa_dims_t forced;
  if (need > FASA_NOALLOC_SCRATCH_BYTES && dims->reserved == 0) {
    forced = *dims;
    const int sizes[4] = {2, 4, 8, 16};
    for (int i = 0; i < 4; ++i) {
      forced.reserved = sizes[i];
      size_t n2 = 0;
      if (fasa_workspace_size(&forced, budget, &n2) == FASA_OK && n2 <= FASA_NOALLOC_SCRATCH_BYTES) {
        dims = &forced;
        need = n2;
        break;
      }
    }
  }
  if (need == 0)  // everything fits in shared memory: no scratch at all
    return fasa_decode_step(q, pos, k_cache, v_cache, k_dom, dom_fc, seq_lens, budget, out, idx_out, count_out,
                            nullptr, 0, dims, stream);
  if (need > FASA_NOALLOC_SCRATCH_BYTES) return FASA_ERR_WORKSPACE;
  float* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != FASA_OK) return st;
  // The scores are written before they are read on every call, so the
  // scratch needs no clearing between calls.
  return fasa_decode_step(q, pos, k_cache, v_cache, k_dom, dom_fc, seq_lens, budget, out, idx_out, count_out,
                          scratch, FASA_NOALLOC_SCRATCH_BYTES, dims, stream);
}
