// GPU generator of the seeded synthetic FASA inputs (test and benchmark
// infrastructure, not part of the library).  Same recipe as workload/synth.py:
// SplitMix64 counters -> Box-Muller normals (fp64), x8 outlier FCs, keys
// rotated by their own position (fp64), stored as fp32 or bf16 (RNE).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ double normal_at(uint64_t base, uint64_t i) {
  const uint64_t r1 = splitmix64(base + 2ull * i);
  const uint64_t r2 = splitmix64(base + 2ull * i + 1ull);
  const double u1 = ((double)(r1 >> 11) + 1.0) * 0x1.0p-53;
  const double u2 = (double)(r2 >> 11) * 0x1.0p-53;
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

__device__ __forceinline__ bool is_outlier(const int* outl, int m, int h, int fc) {
  for (int j = 0; j < m; ++j)
    if (outl[h * m + j] == fc) return true;
  return false;
}

template <typename T>
__device__ __forceinline__ T store_as(double x);
template <>
__device__ __forceinline__ float store_as<float>(double x) { return (float)x; }
template <>
__device__ __forceinline__ __nv_bfloat16 store_as<__nv_bfloat16>(double x) { return __float2bfloat16_rn((float)x); }

// One thread per FC pair of K and V: [B, Hkv, T, d/2] pairs.
template <typename T>
__global__ void gen_kv(T* k, T* v, const int* outl, int m, int B, int Hkv, int T_max, int d, double theta,
                       uint64_t base_k, uint64_t base_v) {
  const uint64_t npairs = (uint64_t)B * Hkv * T_max * (d / 2);
  for (uint64_t x = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; x < npairs;
       x += (uint64_t)gridDim.x * blockDim.x) {
    const int i = (int)(x % (d / 2));
    const uint64_t row = x / (d / 2);           // (b*Hkv + h)*T + tau
    const int tau = (int)(row % T_max);
    const int h = (int)((row / T_max) % Hkv);
    const uint64_t e0 = row * d + 2 * i;
    const double s = is_outlier(outl, m, h, i) ? 8.0 : 1.0;
    const double x0 = normal_at(base_k, e0) * s, x1 = normal_at(base_k, e0 + 1) * s;
    const double ang = (double)tau * pow(theta, -2.0 * i / d);
    double sn, cs;
    sincos(ang, &sn, &cs);
    k[e0] = store_as<T>(x0 * cs - x1 * sn);
    k[e0 + 1] = store_as<T>(x0 * sn + x1 * cs);
    v[e0] = store_as<T>(normal_at(base_v, e0));
    v[e0 + 1] = store_as<T>(normal_at(base_v, e0 + 1));
  }
}

template <typename T>
__global__ void gen_q(T* q, const int* outl, int m, int B, int Hq, int Hkv, int d, uint64_t base_q) {
  const int G = Hq / Hkv;
  const int n = B * Hq * d;
  for (int x = blockIdx.x * blockDim.x + threadIdx.x; x < n; x += gridDim.x * blockDim.x) {
    const int dim = x % d;
    const int hq = (x / d) % Hq;
    const double s = is_outlier(outl, m, hq / G, dim / 2) ? 8.0 : 1.0;
    q[x] = store_as<T>(normal_at(base_q, (uint64_t)x) * s);
  }
}

uint64_t stream_base(uint64_t seed, int layer, int tensor) {
  uint64_t key = (seed << 20) ^ ((uint64_t)layer << 4) ^ (uint64_t)tensor;
  uint64_t z = key + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

}  // namespace

extern "C" {

// Fills q [B,Hq,d] (pre-RoPE), k [B,Hkv,T,d] (post-RoPE) and v of one layer.
// outl: device int32 [Hkv, m] outlier FCs.  dtype 0 = fp32, 1 = bf16.
int synth_fill_layer(void* q, void* k, void* v, const int* outl, int m, int B, int Hq, int Hkv, int T_max, int d,
                     double theta, unsigned long long seed, int layer, int dtype, cudaStream_t stream) {
  const uint64_t bq = stream_base(seed, layer, 1), bk = stream_base(seed, layer, 2), bv = stream_base(seed, layer, 3);
  const int threads = 256, blocks = 152 * 16;
  if (dtype == 0) {
    gen_kv<float><<<blocks, threads, 0, stream>>>((float*)k, (float*)v, outl, m, B, Hkv, T_max, d, theta, bk, bv);
    gen_q<float><<<64, threads, 0, stream>>>((float*)q, outl, m, B, Hq, Hkv, d, bq);
  } else {
    gen_kv<__nv_bfloat16><<<blocks, threads, 0, stream>>>((__nv_bfloat16*)k, (__nv_bfloat16*)v, outl, m, B, Hkv,
                                                          T_max, d, theta, bk, bv);
    gen_q<__nv_bfloat16><<<64, threads, 0, stream>>>((__nv_bfloat16*)q, outl, m, B, Hq, Hkv, d, bq);
  }
  return (int)cudaGetLastError();
}

}  // extern "C"
