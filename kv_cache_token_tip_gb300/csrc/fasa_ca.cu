// Contextual Agreement of the frequency chunks and the choice of dominant FCs
// (the offline calibration of the FASA pages: "The Functional Sparsity
// Hypothesis and the Contextual Agreement (CA) Metric", Eq. 4, and the
// calibration procedure, Algorithm 1).
//
// Three launches per call, so that K is read once:
//   ca_scores_kernel   one CTA per (128-token tile, batch b, KV head h): streams
//                      the tile's key rows once and writes, per token, the
//                      full (group-summed) score and the d/2 single-FC scores
//                      as order-preserving keys, FC-major, into the workspace;
//   ca_select_kernel   one CTA per (key row, b, h) -- the d/2 FC rows and the
//                      full row: the row's TopK-I set (K' = min(K, len)
//                      largest, ties to the smaller token index) as a bitmask
//                      over the tokens;
//   ca_count_kernel    one CTA per (FC i, b, h):
//                      CA = popcount(mask_i & mask_full) / K'.
//
// A row's set: a histogram of every 16th key gives a lower bound T0 expected
// to leave about 2K' keys at or above it; one pass appends (key, token) for
// the keys >= T0 to a list in shared memory (one atomic per warp and load).
// When the list holds at least K' entries and did not overflow, the K'-th
// largest key of the row is the list's K'-th largest (a 12/10/10-bit radix
// select over the list) and the members are marked straight from the list.
// Otherwise (a sample that missed, a large K') the radix select runs over the
// whole row and one ordered pass marks the members.  Scores of most FCs crowd
// into a few histogram bins, so a histogram of every key would serialise on
// the shared-memory atomics; the list keeps them to a few thousand per CTA.
//
// select_dominant_kernel: per KV head, the n FCs of highest mean CA (equal
// means: smaller FC index first), in ascending order.
#include <cuda_bf16.h>
#include <stdint.h>

#include "fasa_internal.h"
#include "fasa_ptx.cuh"

namespace fasa {
namespace {

constexpr int CA_NT = 256;            // threads of a select CTA
constexpr int CA_NW = CA_NT / 32;
constexpr int SC_NT = 256;            // threads of a scoring CTA
constexpr int SC_TT = 128;            // tokens per scoring CTA
constexpr int CA_CAP = 2048;          // candidate keys per row held in shared memory
constexpr int CA_STRIDE = 16;         // the threshold sample takes every 16th token
constexpr int CN_NT = 128;            // threads of a counting CTA

struct CaScratch {
  int scan[CA_NW];
  int dstar, cnt_gt, n_eq;
  int n_cand;
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

// The bin of a histogram (nb bins) that holds the kr-th largest key counted
// from the top bin, the count of keys in the bins above it and in the bin
// itself: sc->dstar, sc->cnt_gt, sc->n_eq.  Every thread calls it.
__device__ void find_bin(const uint32_t* hist, int nb, int kr, CaScratch* sc) {
  const int m = nb / CA_NT;  // thread j owns the m bins counted from the top
  const int base = nb - ((int)threadIdx.x + 1) * m;
  // the sum starts at a lane-dependent bin so that a warp's reads spread
  // over the banks (the bins of neighbouring threads are m words apart)
  const int lane = threadIdx.x & 31;
  int sum = 0;
  for (int i = 0; i < m; ++i) sum += (int)hist[base + ((i + lane) & (m - 1))];
  int total;
  int run = ca_excl_scan(sum, sc, total);
  if (run < kr && kr <= run + sum) {  // the one thread whose bins hold it
    for (int i = m - 1; i >= 0; --i) {
      const int c = (int)hist[base + i];
      if (kr <= run + c) {
        sc->dstar = base + i;
        sc->cnt_gt = run;
        sc->n_eq = c;
        break;
      }
      run += c;
    }
  }
  __syncthreads();
}

// A key row in global memory (16-byte aligned), tokens [0, len): visits this
// thread's keys with four 16-byte loads in flight.
struct GlobalRow {
  const uint4* r4;
  int len;
  template <class Fn>
  __device__ void each(Fn&& fn) const {
    const int nv = (len + 3) >> 2;
    for (int v0 = threadIdx.x; v0 < nv; v0 += 4 * CA_NT) {
      uint4 w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + u * CA_NT;
        w[u] = v < nv ? __ldg(r4 + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + u * CA_NT;
        const uint32_t kx[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (4 * v + c < len) fn(kx[c]);
      }
    }
  }
};

// The candidate list in shared memory: (key, token) pairs list[0..n).
struct SharedList {
  const uint2* list;
  int n;
  template <class Fn>
  __device__ void each(Fn&& fn) const {
    for (int j = threadIdx.x; j < n; j += CA_NT) fn(list[j].x);
  }
};

// The kk-th largest key of a key set (1 <= kk <= its size): its key thr, how
// many keys equal to thr belong to the kk largest (need >= 1) and how many
// keys equal thr (n_eq).  Three histogram passes (12, 10, 10 bits).
template <class Src>
__device__ void radix_select(const Src& src, int kk, uint32_t* hist, CaScratch* sc, uint32_t& thr, int& need,
                             int& n_eq) {
  uint32_t prefix = 0u;
  int kr = kk;
  for (int pass = 0; pass < 3; ++pass) {
    const int bits = pass == 0 ? 12 : 10;
    const int shift = pass == 0 ? 20 : (pass == 1 ? 10 : 0);
    const int nb = 1 << bits;
    for (int i = threadIdx.x; i < nb; i += CA_NT) hist[i] = 0u;
    __syncthreads();
    const uint32_t p = prefix;
    src.each([&](uint32_t key) {
      if (pass == 0 || (key >> (shift + bits)) == p) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
    });
    __syncthreads();
    find_bin(hist, nb, kr, sc);
    kr -= sc->cnt_gt;
    prefix = (prefix << bits) | (uint32_t)sc->dstar;
    n_eq = sc->n_eq;
    __syncthreads();
  }
  thr = prefix;
  need = kr;
}

// The TopK-I set of one key row (the kk >= 1 largest of its len keys, equal
// keys to the smaller token) as bits of mask[0 .. ceil(len / 32)): token tau
// is bit tau % 32 of word tau / 32.  The steps are described at the top of
// this file.
__device__ void row_topk_mask(const uint32_t* __restrict__ row, int len, int kk, uint32_t* hist, uint2* list,
                              CaScratch* sc, uint32_t* mask) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int nw = (len + 31) >> 5;
  for (int w = tid; w < nw; w += CA_NT) mask[w] = 0u;
  // 1. histogram of the top 12 key bits of every CA_STRIDE-th token
  const int ns = (len + CA_STRIDE - 1) / CA_STRIDE;
  for (int i = tid; i < 4096; i += CA_NT) hist[i] = 0u;
  if (tid == 0) sc->n_cand = 0;
  __syncthreads();
  for (int j0 = tid; j0 < ns; j0 += 4 * CA_NT) {
    uint32_t key[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u * CA_NT;
      key[u] = j < ns ? __ldg(row + (size_t)j * CA_STRIDE) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (j0 + u * CA_NT < ns) atomicAdd(&hist[key[u] >> 20], 1u);
  }
  __syncthreads();
  // aim at about 2K' keys of the whole row at or above T0
  find_bin(hist, 4096, min(ns, (2 * kk + CA_STRIDE - 1) / CA_STRIDE + 8), sc);
  const uint32_t t0 = (uint32_t)sc->dstar << 20;
  // 2. append (key, token) for every key >= T0; warp-uniform trip count for
  // the shuffles, one shared atomic per warp and 16-byte load
  const int nv = (len + 3) >> 2;
  const uint4* r4 = reinterpret_cast<const uint4*>(row);
  for (int vw = tid - lane; vw < nv; vw += 4 * CA_NT) {
    uint4 w4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = vw + lane + u * CA_NT;
      w4[u] = v < nv ? __ldg(r4 + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = vw + lane + u * CA_NT;
      const uint32_t kx[4] = {w4[u].x, w4[u].y, w4[u].z, w4[u].w};
      // one ballot per key slot: slot c of the warp's lanes lands after the
      // earlier slots, lanes in order (the list order is free)
      uint32_t bal[4];
      int tot = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        bal[c] = __ballot_sync(0xffffffffu, (4 * v + c < len) && kx[c] >= t0);
        tot += __popc(bal[c]);
      }
      if (tot == 0) continue;  // warp-uniform
      int base = 0;
      if (lane == 0) base = atomicAdd(&sc->n_cand, tot);
      base = __shfl_sync(0xffffffffu, base, 0);
      const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if ((bal[c] >> lane) & 1u) {
          const int pos = base + __popc(bal[c] & lt);
          if (pos < CA_CAP) list[pos] = make_uint2(kx[c], (uint32_t)(4 * v + c));
        }
        base += __popc(bal[c]);
      }
    }
  }
  __syncthreads();
  const int n = sc->n_cand;
  __syncthreads();
  uint32_t thr;
  int need, n_eq;
  if (n >= kk && n <= CA_CAP) {
    // 3. the list holds every key >= the kk-th largest: select there and mark
    // the members straight from the list
    radix_select(SharedList{list, n}, kk, hist, sc, thr, need, n_eq);
    for (int j = tid; j < n; j += CA_NT) {
      const uint2 e = list[j];
      bool in = e.x > thr;
      if (e.x == thr) {
        if (need == n_eq) {
          in = true;
        } else {  // rank among the equal keys by token (rare: exact ties)
          int rank = 0;
          for (int q = 0; q < n; ++q) rank += list[q].x == thr && list[q].y < e.y;
          in = rank < need;
        }
      }
      if (in) atomicOr(&mask[e.y >> 5], 1u << (e.y & 31));
    }
  } else {
    // 3'. select over the whole row, then one ordered pass: thread j holds the
    // 16 tokens 16j..16j+15 of each CTA-wide slab (half a mask word), so a
    // thread-order scan of the tie counts ranks the ties by token
    radix_select(GlobalRow{r4, len}, kk, hist, sc, thr, need, n_eq);
    int run = 0;
    for (int v0 = 0; v0 < nv; v0 += 4 * CA_NT) {
      const int v = v0 + 4 * tid;
      uint32_t u[16];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint4 a = v + h < nv ? __ldg(r4 + v + h) : make_uint4(0u, 0u, 0u, 0u);
        u[4 * h] = a.x; u[4 * h + 1] = a.y; u[4 * h + 2] = a.z; u[4 * h + 3] = a.w;
      }
      int ties = 0;
#pragma unroll
      for (int c = 0; c < 16; ++c) ties += (4 * v + c < len) && u[c] == thr;
      int tot;
      int r = run + ca_excl_scan(ties, sc, tot);
      uint32_t bits = 0u;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (4 * v + c < len) {
          const bool in = u[c] > thr || (u[c] == thr && r < need);
          r += u[c] == thr;
          bits |= (uint32_t)in << c;
        }
      }
      if (bits) atomicOr(&mask[(4 * v) >> 5], bits << ((4 * v) & 31));
      run += tot;
    }
  }
}

__device__ int clamp_len(const int* seq_lens, int b, int T_max) {
  const int len = seq_lens[b];
  return min(max(len, 0), T_max);
}

// E consecutive elements of a key row (E * sizeof(T) = 4, 8 or 16 bytes):
// the raw words, then their fp32 values.
template <typename T, int E>
__device__ void load_raw(const T* p, uint32_t (&u)[E * sizeof(T) / 4]) {
  constexpr int BYTES = E * (int)sizeof(T);
  if constexpr (BYTES == 16) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
    u[0] = w.x; u[1] = w.y; u[2] = w.z; u[3] = w.w;
  } else if constexpr (BYTES == 8) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
    u[0] = w.x; u[1] = w.y;
  } else {
    u[0] = __ldg(reinterpret_cast<const uint32_t*>(p));
  }
}

template <typename T, int E>
__device__ void decode_raw(const uint32_t (&u)[E * sizeof(T) / 4], float (&x)[E]) {
#pragma unroll
  for (int j = 0; j < E * (int)sizeof(T) / 4; ++j) {
    if constexpr (sizeof(T) == 2) {
      x[2 * j] = bf16_lo(u[j]);
      x[2 * j + 1] = bf16_hi(u[j]);
    } else {
      x[j] = __uint_as_float(u[j]);
    }
  }
}

// COMPOUND: two rows per unit instead of d/2 + 1 -- the summed scores of the
// chosen FCs dom_fc[h, 0..n_tip) (row 0) and the full scores (row 1).
template <typename T, int D, bool COMPOUND>
__global__ void __launch_bounds__(SC_NT) ca_scores_kernel(const float* __restrict__ q_rot, const T* __restrict__ k,
                                                           const int* __restrict__ seq_lens,
                                                           const int* __restrict__ dom_fc, int n_tip, uint32_t* keys,
                                                           int Hq, int Hkv, int T_max, int* status) {
  constexpr int F = D / 2, E = D / 32, S = SC_TT + 1;
  constexpr int R = COMPOUND ? 2 : F + 1;  // key rows per unit; the full scores are row R - 1
  __shared__ float qs[D];
  __shared__ uint32_t ks[R * S];
  __shared__ unsigned long long dmask;
  const int unit = blockIdx.y, t0 = blockIdx.x * SC_TT;
  const int b = unit / Hkv, h = unit - b * Hkv;
  const int G = Hq / Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int raw = seq_lens[b];
  if ((raw < 0 || raw > T_max) && blockIdx.x == 0 && tid == 0) atomicOr(status, 1);
  const int len = min(max(raw, 0), T_max);
  if (t0 >= len) return;
  // the tile's key rows first, so that their loads overlap the query's:
  // warp w scores the tile's tokens w, w + 8, ... (one row per warp-wide load)
  constexpr int RPW = SC_TT / (SC_NT / 32);
  constexpr int WPL = E * (int)sizeof(T) / 4;  // 32-bit words per lane and row
  const T* kr = k + ((size_t)unit * T_max + t0) * D + lane * E;
  uint32_t u[RPW][WPL];
#pragma unroll
  for (int j = 0; j < RPW; ++j) {
    const int c = warp + j * (SC_NT / 32);
    if (t0 + c < len) load_raw<T, E>(kr + (size_t)c * D, u[j]);
  }
  for (int d = tid; d < D; d += SC_NT) {
    float a = 0.f;
#pragma unroll
    for (int g = 0; g < G_MAX; ++g)
      if (g < G) a += q_rot[((size_t)b * Hq + (size_t)h * G + g) * D + d];
    qs[d] = a;
  }
  if (COMPOUND && tid == 0) {
    unsigned long long m = 0ull;
    for (int j = 0; j < n_tip; ++j) {  // the head's set: the entries before the first negative one
      const int i = dom_fc[(size_t)h * n_tip + j];
      if (i < 0) break;
      if (i < F) m |= 1ull << i;
      else if (blockIdx.x == 0) atomicOr(status, 1);
    }
    dmask = m;
  }
  __syncthreads();
  float qr[E];
#pragma unroll
  for (int e = 0; e < E; ++e) qr[e] = qs[lane * E + e];

#pragma unroll
  for (int j = 0; j < RPW; ++j) {
    const int c = warp + j * (SC_NT / 32);
    if (t0 + c >= len) continue;  // warp-uniform
    float x[E];
    decode_raw<T, E>(u[j], x);
    float full = 0.f, comp = 0.f;
#pragma unroll
    for (int f = 0; f < E / 2; ++f) {
      const float a = fmaf(qr[2 * f], x[2 * f], qr[2 * f + 1] * x[2 * f + 1]);
      if constexpr (COMPOUND) {
        if ((dmask >> (lane * (E / 2) + f)) & 1ull) comp += a;
      } else {
        ks[(lane * (E / 2) + f) * S + c] = score_key(a);
      }
      full += a;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) full += __shfl_xor_sync(0xffffffffu, full, o);
    if constexpr (COMPOUND) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) comp += __shfl_xor_sync(0xffffffffu, comp, o);
      if (lane == 0) ks[c] = score_key(comp);
    }
    if (lane == 0) ks[(R - 1) * S + c] = score_key(full);
  }
  __syncthreads();
  uint32_t* out = keys + (size_t)unit * R * T_max + t0;
  for (int r = warp; r < R; r += SC_NT / 32) {
#pragma unroll
    for (int c = lane; c < SC_TT; c += 32)
      if (t0 + c < len) out[(size_t)r * T_max + c] = ks[r * S + c];
  }
}

// One CTA per (key row r < R, unit).
__global__ void __launch_bounds__(CA_NT, 4) ca_select_kernel(const uint32_t* __restrict__ keys,
                                                           const int* __restrict__ seq_lens, int K, int R, int Hkv,
                                                           int T_max, uint32_t* masks) {
  __shared__ uint32_t hist[4096];
  __shared__ uint2 list[CA_CAP];
  __shared__ CaScratch sc;
  const int r = blockIdx.x, unit = blockIdx.y;
  const int len = clamp_len(seq_lens, unit / Hkv, T_max);
  const int kk = min(K, len);
  if (kk == 0) return;
  const size_t row = (size_t)unit * R + r;
  row_topk_mask(keys + row * T_max, len, kk, hist, list, &sc, masks + row * (T_max / 32));
}

// One CTA per (row i < R - 1, unit): popcount(mask_i & mask_full) / K', the
// full scores being row R - 1; written to ca[unit * (R - 1) + i].
__global__ void __launch_bounds__(CN_NT) ca_count_kernel(const uint32_t* __restrict__ masks,
                                                          const int* __restrict__ seq_lens, int K, int R, int Hkv,
                                                          int T_max, float* ca) {
  const int F = R - 1;
  __shared__ int part[CN_NT / 32];
  const int i = blockIdx.x, unit = blockIdx.y;
  const int len = clamp_len(seq_lens, unit / Hkv, T_max);
  const int kk = min(K, len);
  if (kk == 0) {  // nothing cached: both sets are empty, full agreement
    if (threadIdx.x == 0) ca[(size_t)unit * F + i] = 1.f;
    return;
  }
  const uint32_t* mi = masks + ((size_t)unit * R + i) * (T_max / 32);
  const uint32_t* mf = masks + ((size_t)unit * R + F) * (T_max / 32);
  const int nw = (len + 31) >> 5;
  int both = 0;
  for (int w = threadIdx.x; w < nw; w += CN_NT) both += __popc(__ldg(mi + w) & __ldg(mf + w));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) both += __shfl_xor_sync(0xffffffffu, both, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = both;
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = 0;
    for (int w = 0; w < CN_NT / 32; ++w) n += part[w];
    ca[(size_t)unit * F + i] = (float)n / (float)kk;
  }
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

size_t fc_agreement_workspace(int units, int D, int T_max) {
  return (size_t)units * (D / 2 + 1) * ((size_t)T_max + T_max / 32) * 4;
}

cudaError_t launch_fc_agreement(const float* q_rot, const void* k, const int* lens, const int* dom_fc, int n_tip,
                                int K, float* ca, int B, int Hq, int Hkv, int D, int T_max, bool bf16, void* ws,
                                int* status, cudaStream_t s) {
  const int units = B * Hkv;
  const bool comp = dom_fc != nullptr;
  const int R = comp ? 2 : D / 2 + 1;
  uint32_t* keys = static_cast<uint32_t*>(ws);
  const dim3 grid((T_max + SC_TT - 1) / SC_TT, units);
#define FASA_CA_SCORES(TT, DD, CC)                                                                             \
  ca_scores_kernel<TT, DD, CC><<<grid, SC_NT, 0, s>>>(q_rot, static_cast<const TT*>(k), lens, dom_fc, n_tip, keys, \
                                                      Hq, Hkv, T_max, status)
  if (bf16) {
    if (D == 128) {
      if (comp) FASA_CA_SCORES(__nv_bfloat16, 128, true); else FASA_CA_SCORES(__nv_bfloat16, 128, false);
    } else {
      if (comp) FASA_CA_SCORES(__nv_bfloat16, 64, true); else FASA_CA_SCORES(__nv_bfloat16, 64, false);
    }
  } else {
    if (D == 128) {
      if (comp) FASA_CA_SCORES(float, 128, true); else FASA_CA_SCORES(float, 128, false);
    } else {
      if (comp) FASA_CA_SCORES(float, 64, true); else FASA_CA_SCORES(float, 64, false);
    }
  }
#undef FASA_CA_SCORES
  uint32_t* masks = keys + (size_t)units * R * T_max;
  ca_select_kernel<<<dim3(R, units), CA_NT, 0, s>>>(keys, lens, K, R, Hkv, T_max, masks);
  ca_count_kernel<<<dim3(R - 1, units), CN_NT, 0, s>>>(masks, lens, K, R, Hkv, T_max, ca);
  return cudaGetLastError();
}

cudaError_t launch_select_dominant(const float* ca_mean, int Hkv, int F, int n, int* dom_fc, cudaStream_t s) {
  select_dominant_kernel<<<Hkv, 64, 0, s>>>(ca_mean, F, n, dom_fc);
  return cudaGetLastError();
}

}  // namespace fasa
