// Contextual Agreement of the frequency chunks and the choice of dominant FCs
// (the offline calibration of the FASA pages: "The Functional Sparsity
// Hypothesis and the Contextual Agreement (CA) Metric", Eq. 4, and the
// calibration procedure, Algorithm 1).
//
// fc_agreement_kernel: one CTA per (FC i, batch b, KV head h).  Over the
// cached tokens tau < len it scores every token twice -- by the full
// (group-summed) query and by FC i alone -- finds each score vector's exact
// TopK-I set (K' = min(K, len) largest, ties to the smaller token index) with
// a local 12/10/10-bit radix select over order-preserving keys, and writes
// |TopK-I(full) & TopK-I(alpha_i)| / K'.
//
// select_dominant_kernel: per KV head, the n FCs of highest mean CA (equal
// means: smaller FC index first), in ascending order.
#include <cuda_bf16.h>
#include <stdint.h>

#include "fasa_internal.h"
#include "fasa_ptx.cuh"

namespace fasa {
namespace {

constexpr int CA_NT = 256;
constexpr int CA_NW = CA_NT / 32;

struct CaScratch {
  int scan[CA_NW];
  int dstar, cnt_gt;
};

// Exclusive prefix sum over the CTA's threads (thread order); every thread
// calls it.
__device__ int ca_excl_scan(int x, CaScratch* sc, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sc->scan[warp] = incl;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < CA_NW; ++w) {
    const int s = sc->scan[w];
    before += w < warp ? s : 0;
    tot += s;
  }
  __syncthreads();
  total = tot;
  return before + incl - x;
}

// The kk-th largest of keys[0..t) (kk >= 1): its key thr and how many keys
// equal to thr belong to the kk largest (need >= 1).
__device__ void ca_select(const uint32_t* keys, int t, int kk, uint32_t* hist, CaScratch* sc, uint32_t& thr,
                          int& need) {
  uint32_t prefix = 0u;
  int kr = kk;
  for (int pass = 0; pass < 3; ++pass) {
    const int bits = pass == 0 ? 12 : 10;
    const int shift = pass == 0 ? 20 : (pass == 1 ? 10 : 0);
    const int nb = 1 << bits;
    for (int i = threadIdx.x; i < nb; i += CA_NT) hist[i] = 0u;
    __syncthreads();
    for (int tau = threadIdx.x; tau < t; tau += CA_NT) {
      const uint32_t k = keys[tau];
      if (pass == 0 || (k >> (shift + bits)) == prefix) atomicAdd(&hist[(k >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    // thread j owns the nb / CA_NT bins counted from the top
    const int m = nb / CA_NT;
    const int base = nb - ((int)threadIdx.x + 1) * m;
    int sum = 0;
    for (int i = 0; i < m; ++i) sum += (int)hist[base + i];
    int total;
    int run = ca_excl_scan(sum, sc, total);
    for (int i = m - 1; i >= 0; --i) {
      const int c = (int)hist[base + i];
      if (run < kr && kr <= run + c) {
        sc->dstar = base + i;
        sc->cnt_gt = run;
      }
      run += c;
    }
    __syncthreads();
    kr -= sc->cnt_gt;
    prefix = (prefix << bits) | (uint32_t)sc->dstar;
    __syncthreads();
  }
  thr = prefix;
  need = kr;
}

template <typename T, int D>
__global__ void __launch_bounds__(CA_NT) fc_agreement_kernel(const float* __restrict__ q_rot, const T* __restrict__ k,
                                                              const int* __restrict__ seq_lens, int K, float* ca,
                                                              int Hq, int Hkv, int T_max, int* status) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int F = D / 2;
  float* qb = reinterpret_cast<float*>(smem);                       // [D] group-summed query
  CaScratch* sc = reinterpret_cast<CaScratch*>(qb + D);
  uint32_t* hist = reinterpret_cast<uint32_t*>(sc + 1);              // [4096]
  uint32_t* in_full = hist + 4096;                                   // [T_max / 32] membership bits
  uint32_t* keys = in_full + (T_max + 31) / 32;                      // [T_max]
  const int i = blockIdx.x, unit = blockIdx.y;
  const int b = unit / Hkv, h = unit - b * Hkv;
  const int G = Hq / Hkv;
  const int tid = threadIdx.x;

  int len = seq_lens[b];
  if (len < 0 || len > T_max) {
    if (tid == 0 && i == 0) atomicOr(status, 1);
    len = min(max(len, 0), T_max);
  }
  const int kk = min(K, len);
  if (kk == 0) {  // nothing cached: both sets are empty, full agreement
    if (tid == 0) ca[(size_t)unit * F + i] = 1.f;
    return;
  }
  for (int d = tid; d < D; d += CA_NT) {
    float a = 0.f;
    for (int g = 0; g < G; ++g) a += q_rot[((size_t)b * Hq + (size_t)h * G + g) * D + d];
    qb[d] = a;
  }
  for (int w = tid; w < (T_max + 31) / 32; w += CA_NT) in_full[w] = 0u;
  __syncthreads();

  const T* kr = k + (size_t)unit * T_max * D;
  // per-thread contiguous runs of odd length: the scalar shared loads of a
  // warp fall in distinct banks
  const int seg = ((len + CA_NT - 1) / CA_NT) | 1;
  const int s0 = min(len, tid * seg), s1 = min(len, s0 + seg);

  // ---- the full head's TopK-I set, as membership bits
  for (int tau = tid; tau < len; tau += CA_NT) {
    const uint4* row = reinterpret_cast<const uint4*>(kr + (size_t)tau * D);  // 16-byte aligned rows
    float s = 0.f;
    constexpr int EPV = 16 / (int)sizeof(T);  // elements per 16-byte vector
#pragma unroll 4
    for (int v = 0; v < D / EPV; ++v) {
      const uint4 w = row[v];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if constexpr (sizeof(T) == 2) {
          s = fmaf(qb[v * 8 + 2 * c], bf16_lo(u[c]), s);
          s = fmaf(qb[v * 8 + 2 * c + 1], bf16_hi(u[c]), s);
        } else {
          s = fmaf(qb[v * 4 + c], __uint_as_float(u[c]), s);
        }
      }
    }
    keys[tau] = score_key(s);
  }
  __syncthreads();
  uint32_t thr;
  int need;
  ca_select(keys, len, kk, hist, sc, thr, need);
  {
    int ties = 0;
    for (int x = s0; x < s1; ++x) ties += keys[x] == thr;
    int total;
    int r = ca_excl_scan(ties, sc, total);
    for (int x = s0; x < s1; ++x) {
      const uint32_t key = keys[x];
      if (key > thr || (key == thr && r < need)) atomicOr(&in_full[x >> 5], 1u << (x & 31));
      r += key == thr;
    }
  }
  __syncthreads();

  // ---- FC i's TopK-I set and its overlap with the full set
  for (int tau = tid; tau < len; tau += CA_NT) {
    const T* row = kr + (size_t)tau * D;
    const float s = fmaf(qb[2 * i], to_f32<T>(row[2 * i]), qb[2 * i + 1] * to_f32<T>(row[2 * i + 1]));
    keys[tau] = score_key(s);
  }
  __syncthreads();
  ca_select(keys, len, kk, hist, sc, thr, need);
  int ties = 0;
  for (int x = s0; x < s1; ++x) ties += keys[x] == thr;
  int total;
  int r = ca_excl_scan(ties, sc, total);
  int both = 0;
  for (int x = s0; x < s1; ++x) {
    const uint32_t key = keys[x];
    const bool in = key > thr || (key == thr && r < need);
    both += in && ((in_full[x >> 5] >> (x & 31)) & 1u);
    r += key == thr;
  }
  int n_both;
  ca_excl_scan(both, sc, n_both);
  if (tid == 0) ca[(size_t)unit * F + i] = (float)n_both / (float)kk;
}

// One block per KV head, one thread per FC (F <= 64).
__global__ void select_dominant_kernel(const float* ca_mean, int F, int n, int* dom_fc) {
  __shared__ int sel[64];
  const int h = blockIdx.x, i = threadIdx.x;
  const float* c = ca_mean + (size_t)h * F;
  bool keep = false;
  if (i < F) {
    const float v = c[i];
    int rank = 0;
    for (int j = 0; j < F; ++j) rank += c[j] > v || (c[j] == v && j < i);
    keep = rank < n;
  }
  if (i < 64) sel[i] = keep;
  __syncthreads();
  if (keep) {
    int pos = 0;
    for (int j = 0; j < i; ++j) pos += sel[j];
    dom_fc[(size_t)h * n + pos] = i;
  }
}

}  // namespace

size_t fc_agreement_smem(int D, int T_max) {
  return (size_t)D * 4 + sizeof(CaScratch) + 4096 * 4 + (size_t)((T_max + 31) / 32) * 4 + (size_t)T_max * 4;
}

cudaError_t launch_fc_agreement(const float* q_rot, const void* k, const int* lens, int K, float* ca, int B,
                                int Hq, int Hkv, int D, int T_max, bool bf16, int* status, cudaStream_t s) {
  const dim3 grid(D / 2, B * Hkv);
  const size_t smem = fc_agreement_smem(D, T_max);
  cudaError_t e = cudaSuccess;
#define FASA_CA_LAUNCH(TT, DD)                                                                                   \
  do {                                                                                                         \
    e = cudaFuncSetAttribute(fc_agreement_kernel<TT, DD>, cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                             (int)smem);                                                                       \
    if (e == cudaSuccess)                                                                                      \
      fc_agreement_kernel<TT, DD><<<grid, CA_NT, smem, s>>>(q_rot, reinterpret_cast<const TT*>(k), lens, K,   \
                                                             ca, Hq, Hkv, T_max, status);                      \
  } while (0)
  if (bf16) {
    if (D == 128) FASA_CA_LAUNCH(__nv_bfloat16, 128);
    else FASA_CA_LAUNCH(__nv_bfloat16, 64);
  } else {
    if (D == 128) FASA_CA_LAUNCH(float, 128);
    else FASA_CA_LAUNCH(float, 64);
  }
#undef FASA_CA_LAUNCH
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_select_dominant(const float* ca_mean, int Hkv, int F, int n, int* dom_fc, cudaStream_t s) {
  select_dominant_kernel<<<Hkv, 64, 0, s>>>(ca_mean, F, n, dom_fc);
  return cudaGetLastError();
}

}  // namespace fasa
