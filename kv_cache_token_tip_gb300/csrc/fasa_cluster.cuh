// The cluster kernel of the FASA decode step.
//
// One thread-block cluster of C CTAs owns one (batch, KV head) unit and runs
// the whole path on it without leaving the chip:
//
//   1. RoPE of the G query heads of the group and the GQA-summed query
//      restricted to the dominant FCs.  Angles come from fixed-point turns
//      (pos * theta_i / 2pi in 64-bit integer arithmetic), so no fp64 is used.
//   2. TIP: each CTA streams its contiguous token range of the FC-major
//      dominant key copy with 1-D bulk (TMA) copies into a shared-memory ring
//      and forms S_tau = sum_j qbar^[j] . k_dom[j, tau] in fp32.  The scores
//      stay in shared memory; the first 12-bit histogram of their
//      order-preserving keys is built on the way.
//   3. Top-k: a radix select over 32-bit keys with digits of 12, 10 and 10
//      bits.  Each CTA adds its non-zero histogram bins into the leader CTA
//      with distributed-shared-memory reductions; after one cluster barrier
//      every CTA reads the totals and finds the same threshold digit.  When
//      the keys at or above the threshold bucket fit the candidate buffer,
//      each CTA lists its own candidates (token order) and every CTA pulls the
//      concatenated list, finishes the selection locally and compacts the
//      chosen tokens in ascending order.
//   4. FAC: the selected rows are split evenly over the cluster; each CTA
//      gathers its K and V rows with cp.async into a padded ring, forms the
//      logits and an online softmax in fp32 (exp2 of log2(e)/sqrt(d)-scaled
//      logits), and pushes its partial (m, l, o) per head to the CTA that
//      combines that head.
//
// The same kernel serves the separate stages (flags select the phases):
// TIP only, top-k on given scores, FAC on given indices, and dense
// attention over all rows.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "../../include/fasa.h"
#include "fasa_internal.h"
#include "fasa_ptx.cuh"

namespace fasa {


enum : int { MODE_NONE = 0, MODE_FILL = 1, MODE_TIES = 2, MODE_CAND = 3, MODE_BX = 4 };
// Largest threshold bucket resolved by exchanging its entries (see the
// bucket exchange after the first radix digit).
constexpr int BX_MAX = 512;

struct Misc {
  int dstar, cnt_gt, bucket, my_count;
  int ncand, my_above, my_ties, pad0;
  int cntR[C_MAX];
  int offR[C_MAX];
  int tiesR[C_MAX];
  int scan[NW];
  int scan2[NW];
  int tip_fail;          // a TIP stage wait ran out
  int big_unsafe;        // a TIP copy did not land in time: `big` is not reused
  int bx_n;              // bucket entries received from the cluster (remote atomics)
  int bx_fail;           // set remotely by a CTA without a candidate list
  int bx_loc;            // this CTA's bucket entries
  int bx_off[C_MAX];     // where this CTA's entries go in each CTA
  uint32_t tip_done[4];  // per TIP stage: warps done with it so far (monotonic)
  int tip_last[4];       // per TIP stage: last tile issued into it (-1: none)
  int nfc;               // this head's dominant-FC count (its leading valid entries)
  uint8_t fac_pair[64];  // F_KSPLIT: the FC of each pair position of a FAC key row
};
static_assert(sizeof(Misc) <= MISC_BYTES, "misc scratch too small");

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sums eight per-lane values over the 32 lanes of a warp with 9 shuffles
// (instead of 8 x 5): each halving step exchanges the half of the values the
// partner keeps.  On return lane L holds the total of value index
// ((L >> 2) & 7) in bit order (bit 4 of L selects the upper four values,
// bit 3 the upper two of those, bit 2 the odd one).
__device__ __forceinline__ float warp_sum8(const float (&a)[8], int lane) {
  float b[4], c[2];
  const bool u4 = lane & 16, u2 = lane & 8, u1 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = u4 ? a[i] : a[i + 4];
    const float keep = u4 ? a[i + 4] : a[i];
    b[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = u2 ? b[i] : b[i + 2];
    const float keep = u2 ? b[i + 2] : b[i];
    c[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  const float send = u1 ? c[0] : c[1];
  const float keep = u1 ? c[1] : c[0];
  float v = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v;
}

// Exclusive prefix sum over the NT threads of the CTA (thread order).
// Every thread must call it.  `scratch` holds NW ints.
__device__ __forceinline__ int block_excl_scan(int x, int* scratch, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const int s = scratch[w];
    before += (w < warp) ? s : 0;
    tot += s;
  }
  __syncthreads();
  total = tot;
  return before + incl - x;
}

// Four consecutive scores starting at p[tl] (tl multiple of 4); entries at or
// past n are marked invalid.
__device__ __forceinline__ void load4(const float* p, int tl, int n, float (&v)[4], bool (&ok)[4]) {
  if (tl + 4 <= n) {
    const float4 x = *reinterpret_cast<const float4*>(p + tl);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    ok[0] = ok[1] = ok[2] = ok[3] = true;
  } else {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      ok[t] = tl + t < n;
      v[t] = ok[t] ? p[tl + t] : 0.f;
    }
  }
}

// cos / sin of the RoPE angle m * theta_i.  `turns` = theta_i / (2 pi) * 2^64;
// the wrapped 64-bit product is the angle in turns, exact up to the rounding
// of `turns`.  Its top 32 bits as a signed fraction x in [-1, 1) give the
// angle pi * x, evaluated with sincospif.
__device__ __forceinline__ float2 rope_cos_sin(unsigned long long turns, int m) {
  const unsigned long long t = (unsigned long long)(long long)m * turns;
  const float x = (float)(int)(t >> 32) * 4.656612873077393e-10f;  // 2^-31
  float s, c;
  sincospif(x, &s, &c);
  return make_float2(c, s);
}

// FASA-M split keys ("FASA: Frequency-aware Sparse Attention", "Hardware-
// Aware Variants": the dominant key dims stay in device memory, the others
// sit with V in host memory).  A key's FAC row is laid out as its
// non-dominant FC pairs in FC order (the k_nondom row, ndp = d/2 - n pairs),
// then its n dominant pairs in the order of the head's FC table (from
// K_dom); the query is laid out alike, so q . k is unchanged.  One warp
// fills fac_pair[p] = the FC whose pair sits at position p of that row.
// Returns (every lane) whether the table holds n distinct FCs in range --
// the only tables the split layout can represent.
__device__ __forceinline__ bool split_pairs(const int* dom, int n, int npairs, uint8_t* fac_pair) {
  const int lane = threadIdx.x & 31;
  uint32_t m0 = 0u, m1 = 0u;
  bool ok = true;
  for (int j = lane; j < n; j += 32) {
    const int i = dom[j];
    if (i < 0 || i >= npairs) {
      ok = false;
    } else if (i < 32) {
      m0 |= 1u << i;
    } else {
      m1 |= 1u << (i - 32);
    }
  }
  m0 = __reduce_or_sync(0xffffffffu, m0);
  m1 = __reduce_or_sync(0xffffffffu, m1);
  ok = __all_sync(0xffffffffu, ok) && __popc(m0) + __popc(m1) == n;
  const int ndp = npairs - n;
  for (int f = lane; f < npairs; f += 32) {
    const bool dominant = f < 32 ? ((m0 >> f) & 1u) != 0u : ((m1 >> (f - 32)) & 1u) != 0u;
    if (!dominant) {
      const int rank = f < 32 ? __popc(~m0 & ((1u << f) - 1u))
                              : __popc(~m0) + __popc(~m1 & ((1u << (f - 32)) - 1u));
      if (rank < ndp) fac_pair[rank] = (uint8_t)f;
    }
  }
  for (int j = lane; j < n; j += 32) fac_pair[ndp + j] = (uint8_t)min(max(dom[j], 0), npairs - 1);
  return ok;
}

// 16-byte chunk ch of the split FAC row of token t (bf16): chunks below
// ndp / 4 from the token's k_nondom row (ndp pairs, a multiple of four),
// the others four dominant pairs from the unit's K_dom.  Zero-filled when
// the row is not real (t must still lie in the unit).
__device__ __forceinline__ void split_key_chunk(uint32_t dst, const __nv_bfloat16* knd_unit,
                                                const __nv_bfloat16* kd_unit, int ndp, int n, int t, int ch,
                                                bool real) {
  if (4 * ch < ndp) {
    cp_async16_zfill(dst, knd_unit + (size_t)t * 2 * ndp + ch * 8, real ? 16u : 0u);
  } else {
    const __nv_bfloat16* src =
        kd_unit + ((size_t)(t / KDOM_BLOCK) * n + (4 * ch - ndp)) * KDOM_BLOCK * 2 + (t % KDOM_BLOCK) * 2;
#pragma unroll
    for (int u = 0; u < 4; ++u) cp_async4_zfill(dst + 4u * u, src + u * KDOM_BLOCK * 2, real ? 4u : 0u);
  }
}

// Loads EPL consecutive elements of a K or V row from shared memory as fp32.
template <typename T, int EPL>
__device__ __forceinline__ void load_row(const unsigned char* p, float (&x)[EPL]) {
  if constexpr (sizeof(T) == 2) {
    if constexpr (EPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      x[0] = bf16_lo(w); x[1] = bf16_hi(w);
    }
  } else {
    if constexpr (EPL == 4) {
      const float4 w = *reinterpret_cast<const float4*>(p);
      x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
    } else {
      const float2 w = *reinterpret_cast<const float2*>(p);
      x[0] = w.x; x[1] = w.y;
    }
  }
}

// Radix digits of the keys: 12, 10, 10 bits, from the top.
__device__ __forceinline__ int dig_bits(int p) { return p == 0 ? 12 : 10; }
__device__ __forceinline__ int dig_shift(int p) { return p == 0 ? 20 : (p == 1 ? 10 : 0); }
__device__ __forceinline__ int lead_off(int p) { return p == 0 ? 0 : (p == 1 ? 4096 : 5120); }

// Finds the digit holding the k_rem-th largest key in a histogram of NB bins
// in this CTA's shared memory.  Thread t owns the NB/NT consecutive bins
// counted from the top.  Writes dstar / cnt_gt (keys in larger digits) /
// bucket into `ms`.  Every thread must call it.
template <int NB>
__device__ __forceinline__ void radix_find(const uint32_t* hist, int k_rem, Misc* ms) {
  constexpr int M = NB / NT;
  static_assert(M >= 1 && NB % NT == 0, "bins per thread");
  const int tid = threadIdx.x;
  const int base = NB - (tid + 1) * M;
  uint32_t c[M];
  if constexpr (M % 4 == 0) {
#pragma unroll
    for (int q = 0; q < M / 4; ++q) {
      const uint4 v = reinterpret_cast<const uint4*>(hist + base)[q];
      c[4 * q] = v.x; c[4 * q + 1] = v.y; c[4 * q + 2] = v.z; c[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < M; ++i) c[i] = hist[base + i];
  }
  int tsum = 0;
#pragma unroll
  for (int i = 0; i < M; ++i) tsum += (int)c[i];
  int total;
  int run = block_excl_scan(tsum, ms->scan, total);
#pragma unroll
  for (int i = M - 1; i >= 0; --i) {
    const int ci = (int)c[i];
    if (run < k_rem && k_rem <= run + ci) {
      ms->dstar = base + i;
      ms->cnt_gt = run;
      ms->bucket = ci;
    }
    run += ci;
  }
  __syncthreads();
}

// TIP scores of one staged k_dom tile (ntok tokens from the tile start, in
// blocks of KDOM_BLOCK tokens, FC-major inside a block).  Thread t takes four
// consecutive tokens at a time over all n FCs: one 16-byte (bf16) or two
// (fp32) shared-memory loads per FC give the four tokens' (re, im) pairs.
// NFC > 0 fixes n at compile time; NFC == 0 reads it from nfc_rt.  Scores go
// to sc[0..ntok); with `hist`, each key's top 12 bits are counted in hloc.
template <typename T, int NFC>
__device__ __forceinline__ void tip_tile(const unsigned char* st, int ntok, int nfc_rt, const float* qbar, float* sc,
                                         uint32_t* hloc, bool hist) {
  constexpr int ES = sizeof(T);
  const int nfc = NFC > 0 ? NFC : nfc_rt;
  constexpr uint32_t fc_row_bytes = KDOM_BLOCK * 2 * ES;
  const uint32_t blk_bytes = (uint32_t)nfc * fc_row_bytes;
  for (int tl = threadIdx.x * 4; tl < ntok; tl += NT * 4) {
    const unsigned char* row = st + (tl / KDOM_BLOCK) * blk_bytes + (tl % KDOM_BLOCK) * 2 * ES;
    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
    // adds FC j's term q_re * k_re + q_im * k_im of the four tokens into a
    auto fc_add = [&](int j, float (&a)[4]) {
      const float2 qq = *reinterpret_cast<const float2*>(&qbar[2 * j]);
      if constexpr (ES == 2) {
        const uint4 w = *reinterpret_cast<const uint4*>(row + j * fc_row_bytes);
        a[0] = fmaf(qq.x, bf16_lo(w.x), fmaf(qq.y, bf16_hi(w.x), a[0]));
        a[1] = fmaf(qq.x, bf16_lo(w.y), fmaf(qq.y, bf16_hi(w.y), a[1]));
        a[2] = fmaf(qq.x, bf16_lo(w.z), fmaf(qq.y, bf16_hi(w.z), a[2]));
        a[3] = fmaf(qq.x, bf16_lo(w.w), fmaf(qq.y, bf16_hi(w.w), a[3]));
      } else {
        const float4 w0 = *reinterpret_cast<const float4*>(row + j * fc_row_bytes);
        const float4 w1 = *reinterpret_cast<const float4*>(row + j * fc_row_bytes + 16);
        a[0] = fmaf(qq.x, w0.x, fmaf(qq.y, w0.y, a[0]));
        a[1] = fmaf(qq.x, w0.z, fmaf(qq.y, w0.w, a[1]));
        a[2] = fmaf(qq.x, w1.x, fmaf(qq.y, w1.y, a[2]));
        a[3] = fmaf(qq.x, w1.z, fmaf(qq.y, w1.w, a[3]));
      }
    };
    if constexpr (NFC > 0) {
#pragma unroll
      for (int j = 0; j + 2 <= NFC; j += 2) {
        fc_add(j, a0);
        fc_add(j + 1, a1);
      }
      if constexpr ((NFC & 1) != 0) fc_add(NFC - 1, a0);
    } else {
      int j = 0;
#pragma unroll 2
      for (; j + 2 <= nfc; j += 2) {
        fc_add(j, a0);
        fc_add(j + 1, a1);
      }
      if (j < nfc) fc_add(j, a0);
    }
    float acc[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[t] = a0[t] + a1[t];
    if (tl + 4 <= ntok) {
      *reinterpret_cast<float4*>(sc + tl) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    } else {
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (tl + t < ntok) sc[tl + t] = acc[t];
    }
    if (hist) {
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (tl + t < ntok) atomicAdd(&hloc[score_key(acc[t]) >> 20], 1u);
    }
  }
}

// KIND names the launch in profiles and lets the compiler drop unused phases:
// KIND_STEP = fused decode step, KIND_DENSE = dense attention, KIND_STAGE =
// the separate stage entry points (phases chosen by p.flags).
enum : int { KIND_STEP = 0, KIND_DENSE = 1, KIND_STAGE = 2 };

__host__ __device__ constexpr int kind_flags(int kind, int flags) {
  return kind == KIND_STEP ? (flags & (F_ROPE | F_TIP | F_SELECT | F_FAC | F_IDX_OUT | F_APPEND | F_KSPLIT))
         : kind == KIND_DENSE ? F_DENSE
                              : flags;
}

template <typename T, int D, int KIND>
__global__ void __launch_bounds__(NT, 1) fasa_cluster_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int ES = sizeof(T);
  constexpr int EPL = D / 32;           // FAC elements per lane
  constexpr int KB = KDOM_BLOCK;        // k_dom tokens per block
  constexpr int ROWB = D * ES;          // bytes of one K/V row
  constexpr int ROWS = ROWB + 16;       // padded row stride in shared memory
  constexpr int CPR = ROWB / 16;        // 16-byte chunks per row

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank();
  const int C = (int)cluster_size();
  const int unit = blockIdx.y;
  const int b = unit / p.Hkv, h = unit - (unit / p.Hkv) * p.Hkv;
  const int G = p.G;
  const int flags = kind_flags(KIND, p.flags);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  Misc* ms = reinterpret_cast<Misc*>(smem + p.off_misc);
  float* qrot = reinterpret_cast<float*>(smem + p.off_qrot);
  float* qbar = reinterpret_cast<float*>(smem + p.off_qbar);
  float* stile = reinterpret_cast<float*>(smem + p.off_stile);
  uint32_t* hloc = reinterpret_cast<uint32_t*>(smem + p.off_hloc);
  uint32_t* hlead = reinterpret_cast<uint32_t*>(smem + p.off_hlead);
  float* sc_s = reinterpret_cast<float*>(smem + p.off_sc);
  int* idx_s = reinterpret_cast<int*>(smem + p.off_idx);
  uint2* own2 = reinterpret_cast<uint2*>(smem + p.off_own);
  float* part = reinterpret_cast<float*>(smem + p.off_part);
  unsigned char* big = smem + p.off_big;

  // Shared-memory set-up first: the release below then has no outstanding
  // global loads to wait for.
  // nfc_max: the dominant-FC table's row length and K_dom's plane count; nfc:
  // this head's count, the entries before the first negative one
  const int nfc_max = p.n_tip, tt = p.tip_tile, ns = p.tip_stages;
  int nfc = nfc_max;
  if (tid == 0) {
    for (int s = 0; s < ns; ++s) mbar_init(smem_u32(&bars[s]), 1);
    if (flags & F_SELECT) mbar_init(smem_u32(&bars[7]), 1);  // score reload
    fence_mbar_init();
    ms->tip_fail = 0;
    ms->big_unsafe = 0;
    ms->bx_n = 0;
    ms->bx_fail = 0;
    ms->bx_loc = 0;
    for (int s = 0; s < 4; ++s) {
      ms->tip_done[s] = 0u;
      ms->tip_last[s] = -1;
    }
  }
  if (flags & F_SELECT) {
    uint4* z = reinterpret_cast<uint4*>(hloc);
    for (int i = tid; i < HLOC_BINS / 4; i += NT) z[i] = make_uint4(0u, 0u, 0u, 0u);
    z = reinterpret_cast<uint4*>(hlead);
    for (int i = tid; i < HLEAD_BINS / 4; i += NT) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  // release: the zeroed histograms are visible before any CTA adds into them;
  // completed by cluster_wait() before the first DSMEM access
  cluster_arrive();
  __syncthreads();

  // every small input is loaded up front so the loads overlap each other
  // (and go out before the bulk TIP traffic)
  bool bad = false;
  int len = p.seq_lens[b];
  // with F_APPEND the query sits at the new token's position, len
  const int m_pos = (flags & F_ROPE) ? ((flags & F_APPEND) ? len : p.pos[b]) : 0;
  const int dom_i = (tid < nfc_max && (flags & F_TIP)) ? p.dom_fc[h * nfc_max + tid] : 0;
  if ((flags & F_TIP) && warp == 0) {  // this head's count, from two ballots
    const int d1 = lane + 32 < nfc_max ? p.dom_fc[h * nfc_max + lane + 32] : 0;
    const unsigned b0 = __ballot_sync(0xffffffffu, lane < nfc_max && dom_i < 0);
    const unsigned b1 = __ballot_sync(0xffffffffu, lane + 32 < nfc_max && d1 < 0);
    nfc = b0 ? __ffs(b0) - 1 : (b1 ? 31 + __ffs(b1) : nfc_max);
    nfc = max(nfc, 1);  // an empty set: slot 0 is used (and reported by the check below)
    if (lane == 0) ms->nfc = nfc;
  }
  // F_APPEND: the new token's key and value pairs (thread i < D/2: pair i),
  // loaded here with the other small inputs whichever CTA turns out to own it
  T kn0 = T(0.f), kn1 = T(0.f), vn0 = T(0.f), vn1 = T(0.f);
  if ((flags & F_APPEND) && tid < D / 2) {
    const T* kn = reinterpret_cast<const T*>(p.k_new) + (size_t)unit * D;
    const T* vn = reinterpret_cast<const T*>(p.v_new) + (size_t)unit * D;
    kn0 = kn[2 * tid];
    kn1 = kn[2 * tid + 1];
    vn0 = vn[2 * tid];
    vn1 = vn[2 * tid + 1];
  }
  constexpr int QPAIRS = (G_MAX * D / 2 + NT - 1) / NT;  // query pairs per thread
  float2 qv[QPAIRS];
#pragma unroll
  for (int k = 0; k < QPAIRS; ++k) {
    const int x = tid + k * NT;
    qv[k] = make_float2(0.f, 0.f);
    if (x < G * (D / 2)) {
      const int g = x / (D / 2), i = x - g * (D / 2);
      const size_t off = ((size_t)b * p.Hq + (size_t)h * G + g) * D + 2 * i;
      if (flags & F_ROPE) {
        const T* qg = reinterpret_cast<const T*>(p.q) + off;
        qv[k] = make_float2(to_f32<T>(qg[0]), to_f32<T>(qg[1]));
      } else if (flags & (F_TIP | F_FAC | F_DENSE)) {
        qv[k] = *reinterpret_cast<const float2*>(p.q_rot + off);
      }
    }
  }
  if (len < 0 || len > p.T_max) {
    bad = true;
    len = min(max(len, 0), p.T_max);
  }

  // F_APPEND: the step's own token goes to index t_new = len and is attended
  // with the others (a full cache cannot take it: reported, not appended)
  int t_new = -1;
  if (flags & F_APPEND) {
    if (len < p.T_max) {
      t_new = len;
      len += 1;
    } else {
      bad = true;
    }
  }

  const int k_eff = min(p.budget, len);
  const bool sel_flag = (flags & F_SELECT) != 0;
  const bool need_select = sel_flag && len > p.budget;
  const bool do_tip = (flags & F_TIP) && (!sel_flag || need_select);
  const bool read_sc = (flags & F_SC_IN) && need_select;

  // contiguous token range of this CTA (start aligned to a k_dom block)
  const int chunk = ((len + C - 1) / C + KB - 1) / KB * KB;
  const int t0 = min(len, (int)crank * chunk);
  const int t1 = min(len, t0 + chunk);
  const int nloc = t1 - t0;
  // K_dom is streamed up to the new token, which this CTA (if it owns it)
  // scores from registers
  const bool own_new = t_new >= t0 && t_new < t1;
  const int t1s = own_new ? t_new : t1;
  const int nloc_s = t1s - t0;

  // ---------------------------------------------------------------- TIP loads
  const int ntiles = do_tip ? (nloc_s + tt - 1) / tt : 0;
  // k_dom is [.., T_max/KB, n_tip, KB, 2]: a tile of whole blocks is one
  // contiguous range, moved by a single bulk copy
  // (a head using fewer than nfc_max planes takes the leading nfc planes of
  // each block: one copy per block, packed in the stage)
  const uint32_t fc_row_bytes = (uint32_t)KB * 2 * ES;
  const uint32_t stage_bytes = (uint32_t)(tt / KB) * nfc_max * fc_row_bytes;
  const T* kd_unit = reinterpret_cast<const T*>(p.k_dom) + (size_t)unit * nfc_max * p.T_max * 2;
  auto tip_issue = [&](int it) {  // one thread of warp 0 (its nfc is this head's)
    const int s = it % ns;
    const int tau0 = t0 + it * tt;
    const int nblk = (min(tt, t1s - tau0) + KB - 1) / KB;
    const uint32_t blk_bytes = (uint32_t)nfc * fc_row_bytes;
    const uint32_t bar = smem_u32(&bars[s]);
    mbar_arrive_expect_tx(bar, (uint32_t)nblk * blk_bytes);
    const T* src = kd_unit + (size_t)(tau0 / KB) * nfc_max * KB * 2;
    if (it != p.drop_stage) {  // (test hook: one tile's copy left unissued)
      if (nfc == nfc_max) {
        bulk_g2s(smem_u32(big + s * stage_bytes), src, (uint32_t)nblk * blk_bytes, bar);
      } else {
        for (int bi = 0; bi < nblk; ++bi)
          bulk_g2s(smem_u32(big + s * stage_bytes + bi * blk_bytes), src + (size_t)bi * nfc_max * KB * 2, blk_bytes,
                   bar);
      }
    }
    ms->tip_last[s] = it;
  };
  if (tid == 0)
    for (int it = 0; it < min(ns, ntiles); ++it) tip_issue(it);
  // F_KSPLIT: the FAC key rows' pair order (the last warp; read after the
  // barriers that follow)
  if (ES == 2 && (flags & F_KSPLIT) && warp == NW - 1)
    bad = !split_pairs(p.dom_fc + h * nfc_max, nfc_max, D / 2, ms->fac_pair) || bad;

  // ------------------------------------------------------------ query prep
#pragma unroll
  for (int k = 0; k < QPAIRS; ++k) {
    const int x = tid + k * NT;
    if (x < G * (D / 2)) {
      const int g = x / (D / 2), i = x - g * (D / 2);
      float2 r = qv[k];
      if (flags & F_ROPE) {
        const float2 c = rope_cos_sin(p.rope_turns[i], m_pos);
        r = make_float2(qv[k].x * c.x - qv[k].y * c.y, qv[k].x * c.y + qv[k].y * c.x);
      }
      *reinterpret_cast<float2*>(&qrot[g * D + 2 * i]) = r;
    }
  }
  __syncthreads();
  if (flags & F_TIP) nfc = ms->nfc;
  if (do_tip) {
    for (int j = tid; j < nfc; j += NT) {
      int i = (j == tid) ? dom_i : p.dom_fc[h * nfc_max + j];
      if (i < 0 || i >= D / 2) {
        bad = true;
        i = min(max(i, 0), D / 2 - 1);
      }
      float a0 = 0.f, a1 = 0.f;
      for (int g = 0; g < G; ++g) {
        a0 += qrot[g * D + 2 * i];
        a1 += qrot[g * D + 2 * i + 1];
      }
      qbar[2 * j] = a0;
      qbar[2 * j + 1] = a1;
    }
  }
  __syncthreads();

  // F_APPEND, in the CTA that owns the new token: rotate its key by its
  // position, store key and value at index t_new of the cache and the key's
  // dominant FCs in K_dom, and score it exactly as the TIP loop scores a
  // streamed token (same FC order, same accumulation; stored precision).
  // With F_KSPLIT the key row is the token's k_nondom row: its non-dominant
  // pairs in FC order (fac_pair positions below ndp).
  float s_new = 0.f;
  if (own_new) {
    float2* knew = reinterpret_cast<float2*>(stile);  // rotated key pairs, as stored
    const bool ksplit_w = ES == 2 && (flags & F_KSPLIT) != 0;
    const int ndp_w = D / 2 - nfc_max;
    T* Kw = const_cast<T*>(reinterpret_cast<const T*>(p.k_cache)) +
            ((size_t)unit * p.T_max + t_new) * (ksplit_w ? 2 * ndp_w : D);
    T* Vw = const_cast<T*>(reinterpret_cast<const T*>(p.v_cache)) + ((size_t)unit * p.T_max + t_new) * D;
    if (tid < D / 2) {  // D / 2 <= NT
      const int i = tid;
      const float x0 = to_f32<T>(kn0), x1 = to_f32<T>(kn1);
      const float2 c = rope_cos_sin(p.rope_turns[i], t_new);
      const T r0 = from_f32<T>(x0 * c.x - x1 * c.y), r1 = from_f32<T>(x0 * c.y + x1 * c.x);
      if (!ksplit_w) {
        Kw[2 * i] = r0;
        Kw[2 * i + 1] = r1;
      }
      Vw[2 * i] = vn0;
      Vw[2 * i + 1] = vn1;
      knew[i] = make_float2(to_f32<T>(r0), to_f32<T>(r1));
    }
    __syncthreads();
    if (ksplit_w && tid < ndp_w) {
      const float2 kp = knew[ms->fac_pair[tid]];
      Kw[2 * tid] = from_f32<T>(kp.x);
      Kw[2 * tid + 1] = from_f32<T>(kp.y);
    }
    T* kdw = const_cast<T*>(kd_unit) + ((size_t)(t_new / KB) * nfc_max * KB + (t_new % KB)) * 2;
    auto dom_at = [&](int j) { return min(max(p.dom_fc[h * nfc_max + j], 0), D / 2 - 1); };
    for (int j = tid; j < nfc; j += NT) {
      const float2 kp = knew[dom_at(j)];
      kdw[(size_t)j * KB * 2] = from_f32<T>(kp.x);
      kdw[(size_t)j * KB * 2 + 1] = from_f32<T>(kp.y);
    }
    if (tid == 0 && do_tip) {
      float a0 = 0.f, a1 = 0.f;
      auto fc_add = [&](int j, float& a) {
        const float2 kp = knew[dom_at(j)];
        a = fmaf(qbar[2 * j], kp.x, fmaf(qbar[2 * j + 1], kp.y, a));
      };
      int j = 0;
      for (; j + 2 <= nfc; j += 2) {
        fc_add(j, a0);
        fc_add(j + 1, a1);
      }
      if (j < nfc) fc_add(j, a0);
      s_new = a0 + a1;
    }
    __syncthreads();
  }
  cluster_wait();

  // ---------------------------------------------------------------- TIP scan
  // No CTA barrier per tile: each warp counts itself done with a stage in
  // ms->tip_done[s], and the warp whose count completes the stage refills it
  // (every warp's reads of the stage completed before its count).  A wait
  // that runs out stops the warp and, through ms->tip_fail, the others at
  // their next tile.
  float* scw = (p.s_cap > 0) ? sc_s : (p.scores + (size_t)unit * p.T_max + t0);
  if (own_new && do_tip && tid == 0) {  // the appended token's score, as TIP would
    scw[t_new - t0] = s_new;
    if (need_select) atomicAdd(&hloc[score_key(s_new) >> 20], 1u);
  }
  int tip_fail = 0;
  for (int it = 0; it < ntiles; ++it) {
    const int s = it % ns;
    const uint32_t parity = (uint32_t)(it / ns) & 1u;
    int stop = lane == 0 ? *reinterpret_cast<volatile int*>(&ms->tip_fail) : 0;
    if (__shfl_sync(0xffffffffu, stop, 0)) break;
    const bool ok = mbar_wait_bounded(smem_u32(&bars[s]), parity, p.wait_ns);
    if (!__all_sync(0xffffffffu, ok)) {
      tip_fail = 1;
      if (lane == 0) atomicOr(&ms->tip_fail, 1);
      break;
    }
    const int tau_base = it * tt;
    const int ntok = min(tt, nloc_s - tau_base);
    const unsigned char* st = big + s * stage_bytes;
    switch (nfc) {  // the common dominant-FC counts get fully unrolled loops
      case 8: tip_tile<T, 8>(st, ntok, nfc, qbar, scw + tau_base, hloc, need_select); break;
      case 12: tip_tile<T, 12>(st, ntok, nfc, qbar, scw + tau_base, hloc, need_select); break;
      case 16: tip_tile<T, 16>(st, ntok, nfc, qbar, scw + tau_base, hloc, need_select); break;
      default: tip_tile<T, 0>(st, ntok, nfc, qbar, scw + tau_base, hloc, need_select); break;
    }
    // every lane's reads of the stage have returned (their values fed the
    // FMAs above), so no fence is needed before the count: a fence here would
    // also wait for this warp's global score stores
    __syncwarp();
    if (lane == 0) {
      const uint32_t prev = atomicAdd(&ms->tip_done[s], 1u);
      if ((prev + 1u) % NW == 0u && it + ns < ntiles) tip_issue(it + ns);
    }
  }
  if (__syncthreads_or(tip_fail | (ntiles > 0 ? ms->tip_fail : 0))) {
    if (tid == 0) {
      atomicOr(p.status, FASA_DEV_TIMEOUT);
      // let copies still in flight land before the shared memory is reused;
      // one that does not within one more bound (all stages together) is
      // reported, and `big` is left alone for the rest of the launch
      bool drained = true;
      const uint64_t start = global_timer_ns();
      for (int s = 0; s < ns; ++s)
        if (ms->tip_last[s] >= 0) {
          const uint64_t spent = global_timer_ns() - start;
          const uint64_t left = spent < p.wait_ns ? p.wait_ns - spent : 1ull;
          drained &= mbar_wait_bounded(smem_u32(&bars[s]), (uint32_t)(ms->tip_last[s] / ns) & 1u, left);
        }
      if (!drained) {
        atomicOr(p.status, FASA_DEV_UNDRAINED);
        ms->big_unsafe = 1;
      }
    }
    __syncthreads();
  }
  const bool big_ok = ms->big_unsafe == 0;

  // ----------------------------------------------------- FAC row source
  // The attention rows of this CTA: fr_n rows, either contiguous tokens
  // fr_r0.. or a token list -- fr_list (int) or fr_pairs ((key, token)
  // pairs); a set high bit in a list entry masks the row.  K/V rows are
  // staged with cp.async in a FAC_STAGES-deep ring at the start of `big`
  // (the TIP ring is no longer needed once they are issued).
  unsigned char* fac_stage = big;
  constexpr uint32_t FAC_STAGE_B = 2u * RT * ROWS;
  const int* fr_list = nullptr;
  const uint2* fr_pairs = nullptr;
  int fr_n = 0, fr_r0 = 0;
  bool fr_contig = true, fac_started = false;
  // F_KSPLIT (bf16): k_cache holds the keys' non-dominant pairs (ndp per token)
  const bool ksplit = ES == 2 && (flags & F_KSPLIT) != 0;
  const int ndp = D / 2 - p.n_tip;
  const T* Kb = reinterpret_cast<const T*>(p.k_cache) + (size_t)unit * p.T_max * (ksplit ? 2 * ndp : D);
  const T* Vb = reinterpret_cast<const T*>(p.v_cache) + (size_t)unit * p.T_max * D;
  const __nv_bfloat16* kd16 = reinterpret_cast<const __nv_bfloat16*>(p.k_dom) + (size_t)unit * p.n_tip * p.T_max * 2;
  // one 16-byte chunk of row i (token tok) into dst: V, or K whole or split
  auto kv_chunk = [&](uint32_t dst, int which, int ch, int tok, bool real) {
    if (ksplit && !which)
      split_key_chunk(dst, reinterpret_cast<const __nv_bfloat16*>(Kb), kd16, ndp, p.n_tip, tok, ch, real);
    else
      cp_async16_zfill(dst, (which ? Vb : Kb) + (size_t)tok * D + ch * (16 / ES), real ? 16u : 0u);
  };
  auto row_token = [&](int i) -> int {
    if (fr_contig) return fr_r0 + i;
    if (fr_pairs) return (int)(fr_pairs[i].y & 0x7FFFFFFFu);
    return fr_list[i] & 0x7FFFFFFF;
  };
  auto row_masked = [&](int i) -> bool {
    if (fr_contig) return false;
    if (fr_pairs) return (fr_pairs[i].y >> 31) != 0u;
    return fr_list[i] < 0;
  };
  auto fac_issue = [&](int t) {
    const int ntile = (fr_n + RT - 1) / RT;
    if (t < ntile) {
      const int s = t % FAC_STAGES;
      const int rows_t = min(RT, fr_n - t * RT);
      const uint32_t st0 = smem_u32(fac_stage) + s * FAC_STAGE_B;
      // one warp per row: lanes take the 16-byte chunks of its K then V row;
      // rows past the end of the tile are zero-filled (the tensor-core path
      // multiplies them by zero weights, which must not meet stale NaNs)
      for (int rr = warp; rr < RT; rr += NW) {
        const bool real = rr < rows_t;
        const size_t row_off = real ? (size_t)row_token(t * RT + rr) * D : 0;
        for (int c = lane; c < 2 * CPR; c += 32) {
          const int which = c >= CPR;
          const int ch = c - which * CPR;
          cp_async16_zfill(st0 + which * RT * ROWS + rr * ROWS + ch * 16, (which ? Vb : Kb) + row_off + ch * (16 / ES),
                           real ? 16u : 0u);
        }
      }
    }
    cp_async_commit();
  };
  // bf16: warp w gathers and attends the GR-row groups w, w + NW, ...; slot
  // s of its p.fac_wst private slots holds one group's K rows then V rows.
  // Rows past fr_n are zero-filled.  Every call commits one cp.async group.
  // Rows are ROWB bytes apart; 16-byte chunk c of row r sits at chunk
  // position c ^ (r & 7), so the eight rows an ldmatrix reads fall in
  // distinct banks.  Rows past fr_n are zero-filled (the tensor cores
  // multiply them by zero weights, which must not meet stale NaNs).  Every
  // call commits one cp.async group.
  constexpr uint32_t GSLOT_B = 2u * GR * ROWB;
  auto grp_issue = [&](int g, int s) {
    if (g * GR < fr_n) {
      const uint32_t st0 = smem_u32(big) + (uint32_t)(warp * p.fac_wst + s) * GSLOT_B;
      for (int c = lane; c < GR * 2 * CPR; c += 32) {
        const int rr = c / (2 * CPR), rem = c - rr * (2 * CPR);
        const int which = rem >= CPR, ch = rem - which * CPR;
        const int i = g * GR + rr;
        const bool real = i < fr_n;
        kv_chunk(st0 + which * GR * ROWB + rr * ROWB + ((ch ^ (rr & 7)) * 16), which, ch, real ? row_token(i) : 0,
                 real);
      }
    }
    cp_async_commit();
  };
  auto fac_start = [&]() {
    if (!big_ok) {  // nothing is gathered into unsafe staging: an empty record
      fr_n = 0;
      fac_started = true;
      return;
    }
    if constexpr (ES == 2) {
      // the first p.fac_wst groups of every warp are issued by the whole CTA
      // (a few rows per thread instead of up to 32 per warp); the FAC loop
      // waits for them once, CTA-wide, before it starts
      const int nfirst = min((fr_n + GR - 1) / GR * GR, p.fac_wst * NW * GR);
      for (int c = tid; c < nfirst * 2 * CPR; c += NT) {
        const int i = c / (2 * CPR), rem = c - i * (2 * CPR);
        const int which = rem >= CPR, ch = rem - which * CPR;
        const int g = i / GR, rr = i - g * GR;  // group g: warp g % NW, slot g / NW
        const uint32_t st0 = smem_u32(big) + (uint32_t)((g % NW) * p.fac_wst + g / NW) * GSLOT_B;
        const bool real = i < fr_n;
        kv_chunk(st0 + which * GR * ROWB + rr * ROWB + ((ch ^ (rr & 7)) * 16), which, ch, real ? row_token(i) : 0,
                 real);
      }
      cp_async_commit();
    } else {
#pragma unroll
      for (int s = 0; s < FAC_STAGES - 1; ++s) fac_issue(s);
    }
    fac_started = true;
  };

  // ---------------------------------------------------------------- top-k
  // Cluster radix select with digits of 12, 10 and 10 bits.  After the first
  // digit every CTA lists its own candidates (keys at or above the threshold
  // bucket) in token order and starts gathering their K/V rows; the later
  // digits are resolved on those short lists.  The selection ends either with
  // an exactly filled bucket (every key >= a bound) or, after all 32 bits,
  // with ties on one key K*, shared out in token order.
  int own_n = 0;        // entries of own2
  bool own_list = false;  // own2 lists every candidate of this CTA (else: scan the scores)
  if (need_select) {
    // Scores in global memory (the CTA's range did not fit in shared memory
    // next to the TIP ring, or they are an input) are copied back into `big`
    // when they fit there -- it is idle until the FAC gather -- so the list
    // sweeps below read shared memory.  Warp w moves its own share.
    const float* scr_g = read_sc ? (p.scores_in + (size_t)unit * p.T_max + t0) : scw;
    const int nv = (nloc + 3) >> 2;  // score vectors (rows are padded to whole vectors)
    const int per_w = (nv + NW - 1) / NW;
    const int v0 = min(nv, warp * per_w), v1 = min(nv, v0 + per_w);
    const bool reload = big_ok && (read_sc || p.s_cap == 0) && nv > 0 && nv * 16 <= p.smem_total - p.off_big;
    const uint32_t rbar = smem_u32(&bars[7]);
    if (reload) {
      if (!read_sc) fence_proxy_async_global();  // this thread's score stores, before the copy reads them
      __syncthreads();
      if (lane == 0) {
        if (warp == 0) mbar_arrive_expect_tx(rbar, (uint32_t)nv * 16u);
        if (v1 > v0) bulk_g2s(smem_u32(big) + v0 * 16, scr_g + v0 * 4, (uint32_t)(v1 - v0) * 16u, rbar);
      }
    }
    bool reload_wait = reload;
    auto reload_done = [&]() {
      if (reload_wait && !mbar_wait_bounded(rbar, 0u, p.wait_ns)) atomicOr(p.status, 2);
      reload_wait = false;
    };
    const float* scr = reload ? reinterpret_cast<const float*>(big) : scr_g;
    if (read_sc) {
      reload_done();
      for (int tl = tid * 4; tl < nloc; tl += NT * 4) {
        float v[4];
        bool ok[4];
        load4(scr, tl, nloc, v, ok);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          if (ok[t]) atomicAdd(&hloc[score_key(v[t]) >> 20], 1u);
      }
    }
    __syncthreads();

    const uint32_t hglob_l = smem_u32(hlead);
    int k_rem = k_eff, mode = MODE_NONE, shift = 20;
    uint32_t prefix = 0u;
    for (int pass = 0; pass < 3; ++pass) {
      const int bits = dig_bits(pass);
      const int nb = 1 << bits;
      shift = dig_shift(pass);
      int lo_bin = 0;
      if (pass == 0) {
        // Bins below this CTA's own k-th largest key cannot hold the global
        // threshold (the global k-th key is at least every CTA's local k-th
        // key), so only the bins from there up are sent.
        if (nloc >= k_eff) {
          radix_find<4096>(hloc, k_eff, ms);
          lo_bin = ms->dstar;
        }
      } else {
        // local histogram of the keys inside the current prefix
        for (int i = tid; i < nb; i += NT) hloc[i] = 0u;
        __syncthreads();
        if (own_list) {
          for (int e = tid; e < own_n; e += NT) {
            const uint32_t key = own2[e].x;
            if ((key >> (shift + bits)) == prefix) atomicAdd(&hloc[(key >> shift) & (nb - 1)], 1u);
          }
        } else {
          for (int tl = tid * 4; tl < nloc; tl += NT * 4) {
            float v[4];
            bool ok[4];
            load4(scr, tl, nloc, v, ok);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const uint32_t key = score_key(v[t]);
              if (ok[t] && (key >> (shift + bits)) == prefix) atomicAdd(&hloc[(key >> shift) & (nb - 1)], 1u);
            }
          }
        }
        __syncthreads();
      }
      // add the non-zero bins into every CTA's copy of the cluster totals
      const uint32_t dst = hglob_l + lead_off(pass) * 4;
      for (int i = lo_bin + tid; i < nb; i += NT) {
        const uint32_t c = hloc[i];
        if (c)
          for (int r = 0; r < C; ++r) dsmem_red_add_u32(dsmem_map(dst + i * 4, (uint32_t)r), c);
      }
      cluster_sync();
      if (pass == 0) radix_find<4096>(hlead + lead_off(0), k_rem, ms);
      else radix_find<1024>(hlead + lead_off(pass), k_rem, ms);
      const int cnt_gt = ms->cnt_gt, bucket = ms->bucket;
      k_rem -= cnt_gt;
      prefix = (prefix << bits) | (uint32_t)ms->dstar;
      if (bucket == k_rem) mode = MODE_FILL;
      else if (pass == 2) mode = MODE_TIES;
      __syncthreads();

      if (pass == 0) {
        // this CTA's candidates (top 12 bits >= prefix), token order, into
        // own2 when they fit.  Thread t takes a contiguous run of tokens (odd
        // length: the scalar shared-memory loads of a warp fall in distinct
        // banks); it counts, one block scan places the runs, and it writes.
        reload_done();
        const int seg = ((nloc + NT - 1) / NT) | 1;
        const int s0 = min(nloc, tid * seg), s1 = min(nloc, s0 + seg);
        // A score is a candidate iff its key is at least the smallest key of
        // the threshold bin, i.e. iff the score is at least that key's float
        // (keys order floats, with -0 = +0); bins below 8 start at -inf or
        // at NaN patterns, where -inf is the bound.
        const uint32_t kmin = prefix << 20;
        const float fmin = prefix >= 8u ? __uint_as_float((kmin & 0x80000000u) ? (kmin & 0x7FFFFFFFu) : ~kmin)
                                        : -CUDART_INF_F;
        // eight loads ahead of the tests, both sweeps
        auto scores8 = [&](int i0, float (&x)[8]) {
#pragma unroll
          for (int j = 0; j < 8; ++j) x[j] = i0 + j < s1 ? scr[i0 + j] : -CUDART_INF_F;
        };
        int cnt = 0;
        for (int i0 = s0; i0 < s1; i0 += 8) {
          float x[8];
          scores8(i0, x);
#pragma unroll
          for (int j = 0; j < 8; ++j) cnt += (i0 + j < s1) && x[j] >= fmin;
        }
        int total;
        const int before = block_excl_scan(cnt, ms->scan, total);
        own_list = total <= p.cand_cap;
        if (own_list) {
          // no early exit: the loads of a batch do not wait for the stores
          // of the one before
          int pos = before;
          for (int i0 = s0; i0 < s1; i0 += 8) {
            float x[8];
            scores8(i0, x);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if ((i0 + j < s1) && x[j] >= fmin) own2[pos++] = make_uint2(score_key(x[j]), (uint32_t)(t0 + i0 + j));
          }
          own_n = total;
          __syncthreads();
          if (flags & F_FAC) {
            fr_pairs = own2;
            fr_n = own_n;
            fr_contig = false;
            fac_start();  // gather now; the later digits only mask rows out
          }
        }
      }
      if (pass == 0 && mode == MODE_NONE && bucket <= BX_MAX) {
        // Bucket exchange: instead of more radix digits, every CTA sends the
        // entries (key, token) of the threshold bucket to every CTA -- into
        // hloc, idle until a later digit would zero it -- at offsets reserved
        // with remote atomics.  After one cluster barrier each CTA ranks its
        // own bucket entries in the whole bucket (key descending, token
        // ascending: the stable order) and keeps those ranked below k_rem.
        // A CTA without a candidate list vetoes it; the radix digits follow.
        // entries travel as key << 32 | ~token: larger = earlier in the stable order
        unsigned long long* bx_in = reinterpret_cast<unsigned long long*>(hloc);  // [bucket]
        int* bx_own = reinterpret_cast<int*>(hloc) + 2 * BX_MAX;  // own2 indices of the own entries
        uint32_t* bx_h = hloc + 3 * BX_MAX;                        // 1024-bin digit histogram
        if (own_list)
          for (int e = tid; e < own_n; e += NT)
            if ((own2[e].x >> 20) == prefix) {
              const int j = atomicAdd(&ms->bx_loc, 1);
              if (j < BX_MAX) bx_own[j] = e;
            }
        __syncthreads();
        const int nbo = min(ms->bx_loc, BX_MAX);
        if (tid < C) {
          if (!own_list) dsmem_st_u32(dsmem_map(smem_u32(&ms->bx_fail), (uint32_t)tid), 1u);
          else if (nbo > 0)
            ms->bx_off[tid] = (int)dsmem_atom_add_u32(dsmem_map(smem_u32(&ms->bx_n), (uint32_t)tid), (uint32_t)nbo);
        }
        __syncthreads();
        if (own_list)
          for (int x = tid; x < nbo * C; x += NT) {
            const int j = x / C, r = x - j * C;
            const int off = ms->bx_off[r] + j;
            if (off < BX_MAX) {
              const uint2 en = own2[bx_own[j]];
              dsmem_st_v2u32(dsmem_map(smem_u32(bx_in + off), (uint32_t)r), ~en.y, en.x);
            }
          }
        cluster_sync();
        if (ms->bx_fail == 0 && ms->bx_n == bucket) {
          auto packed = [&](int j) {
            const uint2 en = own2[bx_own[j]];
            return ((unsigned long long)en.x << 32) | (unsigned long long)(~en.y);
          };
          if (nbo * bucket <= 32 * NT) {
            // few comparisons: rank each own entry in the bucket, one warp per
            // entry, the lanes splitting the bucket
            for (int j = warp; j < nbo; j += NW) {
              const unsigned long long me = packed(j);
              uint32_t rank = 0u;
              for (int f0 = 0; f0 < bucket; f0 += 4 * 32) {
                unsigned long long o[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int f = f0 + u * 32 + lane;
                  o[u] = f < bucket ? bx_in[f] : 0ull;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) rank += o[u] > me;
              }
              rank = __reduce_add_sync(0xffffffffu, rank);
              if (lane == 0 && rank >= (uint32_t)k_rem) own2[bx_own[j]].y |= 0x80000000u;
            }
          } else {
            // the k_rem-th largest key of the bucket from its two lower 10-bit
            // digits (local histograms), then ties on that key by token
            uint32_t kpre = prefix;  // key bits fixed so far (from the top)
            int kr = k_rem, nfix = 12;
            bool fill = false;
            for (int dgt = 0; dgt < 2 && !fill; ++dgt) {
              const int sh = 10 - 10 * dgt;
              for (int i = tid; i < 1024; i += NT) bx_h[i] = 0u;
              __syncthreads();
              for (int f = tid; f < bucket; f += NT) {
                const uint32_t key = (uint32_t)(bx_in[f] >> 32);
                if ((key >> (32 - nfix)) == kpre) atomicAdd(&bx_h[(key >> sh) & 1023u], 1u);
              }
              __syncthreads();
              radix_find<1024>(bx_h, kr, ms);
              kr -= ms->cnt_gt;
              kpre = (kpre << 10) | (uint32_t)ms->dstar;
              nfix += 10;
              fill = ms->bucket == kr;
            }
            // selected: key above the fixed bits, or equal on them and (when the
            // last digit did not fill) among the first kr by token
            for (int j = warp; j < nbo; j += NW) {
              const unsigned long long me = packed(j);
              const uint32_t kme = (uint32_t)(me >> 32) >> (32 - nfix);
              bool keep = kme > kpre;
              if (kme == kpre) {
                if (fill) {
                  keep = true;
                } else {
                  uint32_t before = 0u;  // entries with the same key, earlier tokens
                  for (int f = lane; f < bucket; f += 32) {
                    const unsigned long long o = bx_in[f];
                    before += ((uint32_t)(o >> 32) == (uint32_t)(me >> 32)) && o > me;
                  }
                  keep = __reduce_add_sync(0xffffffffu, before) < (uint32_t)kr;
                }
              }
              if (lane == 0 && !keep) own2[bx_own[j]].y |= 0x80000000u;
            }
          }
          mode = MODE_BX;
        }
        __syncthreads();
      }
      if (mode != MODE_NONE) break;
    }

    // TIES: the threshold key K* (= prefix) has more copies than needed.  The
    // CTAs exchange their tie counts; CTA r keeps the first ties in token
    // order after those of CTAs 0..r-1.
    int my_need = 0;
    if (mode == MODE_TIES) {
      int ties = 0;
      if (own_list) {
        for (int e = tid; e < own_n; e += NT) ties += own2[e].x == prefix;
      } else {
        for (int tl = tid * 4; tl < nloc; tl += NT * 4) {
          float v[4];
          bool ok[4];
          load4(scr, tl, nloc, v, ok);
#pragma unroll
          for (int t = 0; t < 4; ++t) ties += (ok[t] && score_key(v[t]) == prefix);
        }
      }
      int tot;
      block_excl_scan(ties, ms->scan, tot);
      if (tid == 0) ms->my_ties = tot;
      cluster_sync();
      if (tid < C) ms->tiesR[tid] = (int)dsmem_ld_u32(dsmem_map(smem_u32(&ms->my_ties), (uint32_t)tid));
      __syncthreads();
      int before = 0;
      for (int r = 0; r < (int)crank; ++r) before += ms->tiesR[r];
      my_need = min(max(k_rem - before, 0), ms->tiesR[crank]);
    }

    // Final selection of this CTA's tokens.  List mode: mask the candidates
    // that are not selected.  Scan mode: list the selected tokens now.
    // Either way each selected entry of own2 ends up holding its rank among
    // this CTA's selections in .x (its key is not needed any more).
    const bool ties_mode = mode == MODE_TIES;
    // (the bucket exchange already masked the list entries it drops)
    auto selected = [&](uint32_t key, int tie_rank, uint32_t y) -> bool {
      if (mode == MODE_BX) return (y >> 31) == 0u;
      if (ties_mode) return key > prefix || (key == prefix && tie_rank < my_need);
      return (key >> shift) >= prefix;
    };
    // After the bucket exchange the list is already masked, and after a
    // bucket filled at the first digit every list entry is selected: the
    // sweeps below then only rank the selections for idx_out.
    const bool list_final = mode == MODE_BX || (mode == MODE_FILL && shift == dig_shift(0));
    if (own_list && list_final && !(flags & F_IDX_OUT)) {
      // nothing to do
    } else if (own_list) {
      // warp w takes a contiguous share of the list; ranks within a warp
      // come from ballots, across warps from per-warp totals
      const uint32_t lt = (1u << lane) - 1u;
      const int per_w = (own_n + NW - 1) / NW;
      const int e0 = min(own_n, warp * per_w), e1 = min(own_n, e0 + per_w);
      int tie_base = 0;
      if (ties_mode) {
        int c = 0;
        for (int e = e0 + lane; e < e1; e += 32) c += own2[e].x == prefix;
        c = __reduce_add_sync(0xffffffffu, c);
        if (lane == 0) ms->scan2[warp] = c;
        __syncthreads();
        for (int w = 0; w < warp; ++w) tie_base += ms->scan2[w];
      }
      int nsel = 0;
      for (int eb = e0; eb < e1; eb += 32) {
        const int e = eb + lane;
        const bool valid = e < e1;
        const uint32_t key = valid ? own2[e].x : 0u;
        const uint32_t tb = __ballot_sync(0xffffffffu, valid && ties_mode && key == prefix);
        const bool sel = valid && selected(key, tie_base + __popc(tb & lt), own2[e].y);
        if (valid && !sel) own2[e].y |= 0x80000000u;
        nsel += __popc(__ballot_sync(0xffffffffu, sel));
        tie_base += __popc(tb);
      }
      if (lane == 0) ms->scan[warp] = nsel;
      __syncthreads();
      int ps = 0, tot_s = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const int c = ms->scan[w];
        ps += w < warp ? c : 0;
        tot_s += c;
      }
      // the rank of each selected entry among this CTA's selections replaces
      // its key (no longer needed)
      for (int eb = e0; eb < e1; eb += 32) {
        const int e = eb + lane;
        const uint32_t y = e < e1 ? own2[e].y : 0x80000000u;
        const bool sel = (y >> 31) == 0u;
        const uint32_t sb = __ballot_sync(0xffffffffu, sel);
        if (sel) own2[e].x = (uint32_t)(ps + __popc(sb & lt));
        ps += __popc(sb);
      }
      if (tid == 0) ms->my_count = tot_s;
    } else {
      const int seg = ((nloc + NT - 1) / NT) | 1;
      const int s0 = min(nloc, tid * seg), s1 = min(nloc, s0 + seg);
      int ct = 0;
      if (ties_mode)
        for (int i = s0; i < s1; ++i) ct += score_key(scr[i]) == prefix;
      int tot_t = 0;
      int tr = ties_mode ? block_excl_scan(ct, ms->scan, tot_t) : 0;
      int cs = 0;
      {
        int trr = tr;
        for (int i = s0; i < s1; ++i) {
          const uint32_t key = score_key(scr[i]);
          cs += selected(key, trr, 0u);
          trr += ties_mode && key == prefix;
        }
      }
      int tot_s;
      int ps = block_excl_scan(cs, ms->scan, tot_s);
      for (int i = s0; i < s1; ++i) {
        const uint32_t key = score_key(scr[i]);
        if (selected(key, tr, 0u) && ps < p.cand_cap) {
          own2[ps] = make_uint2((uint32_t)ps, (uint32_t)(t0 + i));
          ++ps;
        }
        tr += ties_mode && key == prefix;
      }
      own_n = min(tot_s, p.cand_cap);
      if (tid == 0) ms->my_count = own_n;
      __syncthreads();
      if (flags & F_FAC) {
        fr_pairs = own2;
        fr_n = own_n;
        fr_contig = false;
        fac_start();
      }
    }
    __syncthreads();
  }

  // idx_out / count_out: the selected tokens of every CTA, concatenated in
  // cluster-rank (= token) order.  Every CTA has pushed its count into every
  // CTA's cntR (push_count) before a cluster barrier; each CTA then writes its
  // own run at the offset the lower ranks' counts give.
  auto push_count = [&]() {
    if (tid < C) dsmem_st_u32(dsmem_map(smem_u32(&ms->cntR[crank]), (uint32_t)tid), (uint32_t)ms->my_count);
  };
  auto write_idx_out = [&]() {
    if (crank == 0 && p.count_out && tid == 0) p.count_out[unit] = k_eff;
    if (!p.idx_out) return;
    int* io = p.idx_out + (size_t)unit * p.budget;
    if (!need_select) {
      if (crank == 0)
        for (int i = tid; i < p.budget; i += NT) io[i] = (i < k_eff) ? i : -1;
      return;
    }
    int off = 0, total = 0;
    for (int r = 0; r < C; ++r) {
      const int c = ms->cntR[r];
      off += r < (int)crank ? c : 0;
      total += c;
    }
    for (int e = tid; e < own_n; e += NT) {
      const uint2 en = own2[e];
      const int at = off + (int)en.x;
      if ((en.y >> 31) == 0u && at < p.budget) io[at] = (int)en.y;
    }
    if (crank == (uint32_t)C - 1)
      for (int i = total + tid; i < p.budget; i += NT) io[i] = -1;
  };

  // ---------------------------------------------------------------- FAC
  if (flags & (F_FAC | F_DENSE)) {
    if (!fac_started) {
      // an appended row may be gathered by another CTA of the cluster: the
      // barrier orders its owner's stores before the gathers
      if (t_new >= 0) cluster_sync();
      int n_total;
      if (flags & F_DENSE) {
        n_total = len;
        fr_contig = true;
      } else if (flags & F_IDX_IN) {
        n_total = p.count_in[unit];
        if (n_total < 0 || n_total > k_eff) {
          bad = true;
          n_total = min(max(n_total, 0), k_eff);
        }
        fr_contig = false;
      } else {
        n_total = k_eff;  // every cached token is selected
        fr_contig = true;
      }
      const int r0 = (n_total * (int)crank) / C;
      const int r1 = (n_total * ((int)crank + 1)) / C;
      fr_n = r1 - r0;
      fr_r0 = r0;
      if (flags & F_IDX_IN) {
        const int* gi = p.idx_in + (size_t)unit * p.budget + r0;
        for (int i = tid; i < fr_n; i += NT) {
          int t = gi[i];
          if (t < 0 || t >= len) {
            bad = true;
            t = min(max(t, 0), len - 1);
          }
          idx_s[i] = t;
        }
        fr_list = idx_s;
        __syncthreads();
      }
      fac_start();
    }

    constexpr int PSTRIDE = D + 4;
    const int ntile = (fr_n + RT - 1) / RT;
    // Merges nrec partial records (o[0..D), m, l) per head, stored at
    // mst[(g * nrec + r) * (D + 2)], into this CTA's record part[g].
    // (the FAC scratch stile is idle here: wts holds each head's maximum and
    // record weights, computed once instead of once per element)
    auto merge_records = [&](const float* mst, int nrec) {
      float* wts = stile;  // [G][nrec] weights exp2(m_r - M), then [G] maxima
      if (tid < G) {
        const int g = tid;
        float M = -CUDART_INF_F;
        for (int r = 0; r < nrec; ++r) M = fmaxf(M, mst[(g * nrec + r) * (D + 2) + D]);
        for (int r = 0; r < nrec; ++r) {
          const float m_r = mst[(g * nrec + r) * (D + 2) + D];
          wts[g * nrec + r] = m_r != -CUDART_INF_F ? exp2f(m_r - M) : 0.f;
        }
        wts[G * nrec + g] = M;
      }
      __syncthreads();
      for (int x = tid; x < G * (D + 2); x += NT) {
        const int g = x / (D + 2), e = x - g * (D + 2);
        float val = wts[G * nrec + g];
        if (e != D) {
          float acc = 0.f;
          for (int r = 0; r < nrec; ++r) {
            const float w = wts[g * nrec + r];
            if (w != 0.f) acc += w * mst[(g * nrec + r) * (D + 2) + e];
          }
          val = acc;
        }
        part[g * PSTRIDE + e] = val;
      }
    };
    if (!big_ok) {
      // the staging may still receive a late TIP copy: an empty record
      for (int x = tid; x < G * PSTRIDE; x += NT) {
        const int e = x % PSTRIDE;
        part[x] = e == D ? -CUDART_INF_F : 0.f;
      }
    } else if constexpr (ES == 2) {
      // Tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate), one
      // flash-decoding pass per warp over its own 16-row groups, no block
      // barriers: QK as S^T = K Q^T (16 rows x 8 heads), PV as O^T = V^T P^T
      // (16 head dims x 8 heads per MMA).  q and the softmax weights P are
      // split into bf16 hi + lo parts, so the products keep ~16 mantissa bits.
      // Lane (gq, tq) = (lane / 4, lane % 4) holds rows gq, gq + 8 of S^T and
      // head dims gq, gq + 8 of O^T, for heads 2tq and 2tq + 1.
      constexpr int KS = D / 16;
      const float qs = 1.4426950408889634f * rsqrtf((float)D);
      const int gq = lane >> 2, tq = lane & 3;
      uint32_t qb[KS][2][2];  // [k-step][b0 / b1][hi / lo]
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int d0 = ks * 16 + 2 * tq + hb * 8;
          const int ds = ksplit ? 2 * ms->fac_pair[d0 >> 1] : d0;  // the key rows' pair order
          const float x0 = gq < G ? qrot[gq * D + ds] * qs : 0.f;
          const float x1 = gq < G ? qrot[gq * D + ds + 1] * qs : 0.f;
          split_bf16(x0, x1, qb[ks][hb][0], qb[ks][hb][1]);
        }
      float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F;  // running max (log2 units), heads 2tq, 2tq + 1
      float l0 = 0.f, l1 = 0.f;                      // this lane's share of the running sums
      float oc[KS][4];
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) oc[mt][0] = oc[mt][1] = oc[mt][2] = oc[mt][3] = 0.f;
      float* pt = stile + warp * (G_MAX * PTS);  // this warp's P tile [head][row]
      // ldmatrix row addresses (swizzled chunks): K as the A operand of QK --
      // rows (lane & 7) + 8 (mi & 1), chunk 2 ks + (mi >> 1); V^T via .trans --
      // rows (lane & 7) + 8 (mi >> 1), chunk 2 mt + (mi & 1)
      const int mi = lane >> 3;
      const int kr = (lane & 7) + 8 * (mi & 1), vr = (lane & 7) + 8 * (mi >> 1);
      const uint32_t k_row = kr * ROWB, v_row = vr * ROWB;
      const int k_c = mi >> 1, v_c = mi & 1, sw = lane & 7;
      const int wst = p.fac_wst;
      const int ngrp = (fr_n + GR - 1) / GR;
      cp_async_wait<0>();  // the CTA-wide first groups (fac_start)
      __syncthreads();
      int it = 0;
      for (int g = warp; g < ngrp; g += NW, ++it) {
        const int s = wst == 2 ? (it & 1) : 0;
        if (wst == 2) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncwarp();
        const uint32_t Ks = smem_u32(big) + (uint32_t)(warp * wst + s) * GSLOT_B;
        const uint32_t Vs = Ks + GR * ROWB;
        float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(Ks + k_row + (((2 * ks + k_c) ^ sw) << 4), a0, a1, a2, a3);
          mma_bf16_16816(sh, a0, a1, a2, a3, qb[ks][0][0], qb[ks][1][0]);
          mma_bf16_16816(sl, a0, a1, a2, a3, qb[ks][0][1], qb[ks][1][1]);
        }
        const int r0 = g * GR + gq, r1 = r0 + 8;
        const bool v0 = r0 < fr_n && !row_masked(r0);
        const bool v1 = r1 < fr_n && !row_masked(r1);
        const float s0 = v0 ? sh[0] + sl[0] : -CUDART_INF_F, s1 = v0 ? sh[1] + sl[1] : -CUDART_INF_F;
        const float s2 = v1 ? sh[2] + sl[2] : -CUDART_INF_F, s3 = v1 ? sh[3] + sl[3] : -CUDART_INF_F;
        float x0 = fmaxf(s0, s2), x1 = fmaxf(s1, s3);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o));
          x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o));
        }
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        // every row so far may be masked: then nothing is rescaled or added
        const float c0 = n0 == -CUDART_INF_F ? 1.f : exp2f(m0 - n0);
        const float c1 = n1 == -CUDART_INF_F ? 1.f : exp2f(m1 - n1);
        const float p0 = n0 == -CUDART_INF_F ? 0.f : exp2f(s0 - n0);
        const float p2 = n0 == -CUDART_INF_F ? 0.f : exp2f(s2 - n0);
        const float p1 = n1 == -CUDART_INF_F ? 0.f : exp2f(s1 - n1);
        const float p3 = n1 == -CUDART_INF_F ? 0.f : exp2f(s3 - n1);
        l0 = l0 * c0 + p0 + p2;
        l1 = l1 * c1 + p1 + p3;
        m0 = n0;
        m1 = n1;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          oc[mt][0] *= c0;
          oc[mt][1] *= c1;
          oc[mt][2] *= c0;
          oc[mt][3] *= c1;
        }
        // P^T as the B operand: lane (gq, tq) needs head gq, rows 2tq.. --
        // transposed through the warp's tile
        pt[(2 * tq) * PTS + gq] = p0;
        pt[(2 * tq + 1) * PTS + gq] = p1;
        pt[(2 * tq) * PTS + gq + 8] = p2;
        pt[(2 * tq + 1) * PTS + gq + 8] = p3;
        __syncwarp();
        const float2 pa = *reinterpret_cast<const float2*>(pt + gq * PTS + 2 * tq);
        const float2 pb = *reinterpret_cast<const float2*>(pt + gq * PTS + 2 * tq + 8);
        uint32_t b0h, b0l, b1h, b1l;
        split_bf16(pa.x, pa.y, b0h, b0l);
        split_bf16(pb.x, pb.y, b1h, b1l);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(Vs + v_row + (((2 * mt + v_c) ^ sw) << 4), a0, a1, a2, a3);
          mma_bf16_16816(oc[mt], a0, a1, a2, a3, b0h, b1h);
          mma_bf16_16816(oc[mt], a0, a1, a2, a3, b0l, b1l);
        }
        __syncwarp();  // the slot and the P tile are free again
        grp_issue(g + wst * NW, s);
      }
      cp_async_wait<0>();
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
      }
      __syncthreads();  // every warp is done with its slots: `big` takes the warp records
      float* rec = reinterpret_cast<float*>(big);
      const int h0 = 2 * tq, h1 = 2 * tq + 1;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int dd = mt * 16 + gq;
        if (h0 < G) {
          rec[(h0 * NW + warp) * (D + 2) + dd] = oc[mt][0];
          rec[(h0 * NW + warp) * (D + 2) + dd + 8] = oc[mt][2];
        }
        if (h1 < G) {
          rec[(h1 * NW + warp) * (D + 2) + dd] = oc[mt][1];
          rec[(h1 * NW + warp) * (D + 2) + dd + 8] = oc[mt][3];
        }
      }
      if (gq == 0) {
        if (h0 < G) {
          rec[(h0 * NW + warp) * (D + 2) + D] = m0;
          rec[(h0 * NW + warp) * (D + 2) + D + 1] = l0;
        }
        if (h1 < G) {
          rec[(h1 * NW + warp) * (D + 2) + D] = m1;
          rec[(h1 * NW + warp) * (D + 2) + D + 1] = l1;
        }
      }
      __syncthreads();
      merge_records(rec, NW);
    } else {
    const float qs = 1.4426950408889634f * rsqrtf((float)D);
    float qreg[G_MAX][EPL];
#pragma unroll
    for (int g = 0; g < G_MAX; ++g)
#pragma unroll
      for (int e = 0; e < EPL; ++e) qreg[g][e] = (g < G) ? qrot[g * D + lane * EPL + e] * qs : 0.f;
    const int nparts = max(1, NW / G);
    const int my_g = warp % G, my_part = warp / G;
    const bool pv_warp = warp < G * nparts;
    float m_run = -CUDART_INF_F, l_run = 0.f;
    float o_run[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o_run[e] = 0.f;

    for (int t = 0; t < ntile; ++t) {
      cp_async_wait<FAC_STAGES - 2>();
      __syncthreads();
      fac_issue(t + FAC_STAGES - 1);
      const int s = t % FAC_STAGES;
      const unsigned char* Ks = fac_stage + s * FAC_STAGE_B;
      const unsigned char* Vs = Ks + RT * ROWS;
      const int rows_t = min(RT, fr_n - t * RT);
      for (int rr = warp; rr < rows_t; rr += NW) {
        float kv[EPL];
        load_row<T, EPL>(Ks + rr * ROWS + lane * EPL * ES, kv);
        float a[G_MAX];
#pragma unroll
        for (int g = 0; g < G_MAX; ++g) {
          a[g] = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) a[g] = fmaf(qreg[g][e], kv[e], a[g]);
        }
        float v = warp_sum8(a, lane);
        if (row_masked(t * RT + rr)) v = -CUDART_INF_F;
        const int g = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
        if ((lane & 3) == 0 && g < G) stile[g * RT + rr] = v;
      }
      __syncthreads();
      if (pv_warp) {
        const int nr = (rows_t - my_part + nparts - 1) / nparts;
        if (nr > 0) {
          const float sv = (lane < nr) ? stile[my_g * RT + my_part + lane * nparts] : -CUDART_INF_F;
          const float m_new = fmaxf(m_run, warp_max(sv));
          if (m_new != -CUDART_INF_F) {  // every row of this part may be masked
            const float scale = exp2f(m_run - m_new);
            const float pe = (lane < nr) ? exp2f(sv - m_new) : 0.f;
            l_run = l_run * scale + warp_sum(pe);
#pragma unroll
            for (int e = 0; e < EPL; ++e) o_run[e] *= scale;
            for (int i = 0; i < nr; ++i) {
              const float pi = __shfl_sync(0xffffffffu, pe, i);
              if (pi != 0.f) {
                float vv[EPL];
                load_row<T, EPL>(Vs + (my_part + i * nparts) * ROWS + lane * EPL * ES, vv);
#pragma unroll
                for (int e = 0; e < EPL; ++e) o_run[e] = fmaf(pi, vv[e], o_run[e]);
              }
            }
            m_run = m_new;
          }
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();

    // merge the row-parts of each head into this CTA's partial record
    // part[g] = (o[0..D), m, l) with m in log2 units; other CTAs pull it
    float* mst = reinterpret_cast<float*>(fac_stage);
    if (pv_warp) {
      float* dst = mst + (my_g * nparts + my_part) * (D + 2);
#pragma unroll
      for (int e = 0; e < EPL; ++e) dst[lane * EPL + e] = o_run[e];
      if (lane == 0) {
        dst[D] = m_run;
        dst[D + 1] = l_run;
      }
    }
    __syncthreads();
    merge_records(mst, nparts);
    }
    __syncthreads();  // part[] is complete

    // Combine by push: each CTA cuts its record into the C output slices (runs
    // of 4-element groups of the G*D outputs) and stores each slice, with
    // (m, l) of every head and its selected count, into the shared memory of
    // the CTA that finishes that slice.  One cluster barrier makes the stores
    // visible; after it no CTA touches another's shared memory.
    const int ngrp = G * (D / 4);
    const int sl = (ngrp + C - 1) / C;
    float4* recv_o = reinterpret_cast<float4*>(smem + p.off_recv);  // [C][sl]
    float2* recv_ml = reinterpret_cast<float2*>(recv_o + C * sl);    // [C][G]
    const uint32_t recv_o_l = smem_u32(recv_o), recv_ml_l = smem_u32(recv_ml);
    for (int q = tid; q < ngrp; q += NT) {
      const int r = ((q + 1) * C - 1) / ngrp;  // the CTA whose slice holds group q
      const int q0r = (ngrp * r) / C;
      const int g = q / (D / 4), e4 = q - g * (D / 4);
      const float4 v = *reinterpret_cast<const float4*>(part + g * PSTRIDE + e4 * 4);
      dsmem_st_v4f(dsmem_map(recv_o_l + ((int)crank * sl + q - q0r) * 16, (uint32_t)r), v.x, v.y, v.z, v.w);
    }
    for (int x = tid; x < C * G; x += NT) {
      const int r = x / G, g = x - r * G;
      dsmem_st_v2f(dsmem_map(recv_ml_l + ((int)crank * G + g) * 8, (uint32_t)r), part[g * PSTRIDE + D],
                   part[g * PSTRIDE + D + 1]);
    }
    if ((flags & F_IDX_OUT) && need_select) push_count();
    cluster_sync();

    // Finish this CTA's slice: lpg lanes per output group (the power of two
    // >= C), lane r taking CTA r's record, reduced with width-lpg shuffles; a
    // warp takes 32 / lpg groups per pass, so every shuffle runs with all 32
    // lanes.
    const int q0 = (ngrp * (int)crank) / C, q1 = (ngrp * ((int)crank + 1)) / C;
    const int lpg = C <= 1 ? 1 : 1 << (32 - __clz(C - 1));
    const int gpw = 32 / lpg;  // groups per warp and pass
    for (int qw = q0 + gpw * warp; qw < q1; qw += gpw * NW) {  // warp-uniform bound
      const int q = qw + lane / lpg, r = lane & (lpg - 1);
      const bool ok = q < q1 && r < C;
      const int g = ok ? q / (D / 4) : 0, e4 = ok ? q - g * (D / 4) : 0;
      const float2 ml = ok ? recv_ml[r * G + g] : make_float2(-CUDART_INF_F, 0.f);
      float M = ml.x;
      for (int o = lpg >> 1; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o, lpg));
      const float w = (ml.x != -CUDART_INF_F) ? exp2f(ml.x - M) : 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (w != 0.f) {
        const float4 v = recv_o[r * sl + q - q0];
        acc = make_float4(w * v.x, w * v.y, w * v.z, w * v.w);
      }
      float L = w * ml.y;
      for (int o = lpg >> 1; o >= 1; o >>= 1) {
        L += __shfl_xor_sync(0xffffffffu, L, o, lpg);
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o, lpg);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o, lpg);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o, lpg);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o, lpg);
      }
      if (r == 0 && q < q1) {
        if (L > 0.f) {
          const float inv = 1.f / L;
          acc.x *= inv;
          acc.y *= inv;
          acc.z *= inv;
          acc.w *= inv;
        }
        *reinterpret_cast<float4*>(p.out + ((size_t)b * p.Hq + (size_t)h * G + g) * D + e4 * 4) = acc;
      }
    }
    if (flags & F_IDX_OUT) write_idx_out();
  } else if (need_select) {
    if (flags & F_IDX_OUT) push_count();
    cluster_sync();  // the counts are in; no CTA reads another's shared memory after this
    if (flags & F_IDX_OUT) write_idx_out();
  } else if (flags & F_IDX_OUT) {
    write_idx_out();
  }
  if (bad) atomicOr(p.status, 1);
}

// Opts the kernel into the largest dynamic shared memory the device allows
// and into non-portable (up to 16 CTA) clusters; once per process.
template <typename T, int D, int KIND>
cudaError_t prepare_kernel() {
  static cudaError_t once = [] {
    auto k = fasa_cluster_kernel<T, D, KIND>;
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

inline int kind_of(int flags) {
  if ((flags & (F_TIP | F_SELECT | F_FAC | F_ROPE)) == (F_TIP | F_SELECT | F_FAC | F_ROPE)) return KIND_STEP;
  if (flags == F_DENSE) return KIND_DENSE;
  return KIND_STAGE;
}

template <int KIND>
inline cudaLaunchConfig_t cluster_config(int C, int units, int smem, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, (unsigned)units, 1);
  cfg.blockDim = dim3(NT, 1, 1);
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

template <typename T, int D, int KIND>
cudaError_t launch_kind(const Params& p, int C, cudaStream_t s) {
  cudaError_t e = prepare_kernel<T, D, KIND>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config<KIND>(C, p.B * p.Hkv, p.smem_total, s, attr);
  return cudaLaunchKernelEx(&cfg, fasa_cluster_kernel<T, D, KIND>, p);
}

template <typename T, int D>
cudaError_t launch_cluster_t(const Params& p, int C, cudaStream_t s) {
  switch (kind_of(p.flags)) {
    case KIND_STEP: return launch_kind<T, D, KIND_STEP>(p, C, s);
    case KIND_DENSE: return launch_kind<T, D, KIND_DENSE>(p, C, s);
    default: return launch_kind<T, D, KIND_STAGE>(p, C, s);
  }
}

template <typename T, int D, int KIND>
int max_clusters_kind(int C, int smem_bytes) {
  if (prepare_kernel<T, D, KIND>() != cudaSuccess) return 0;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config<KIND>(C, 1, smem_bytes, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fasa_cluster_kernel<T, D, KIND>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <typename T, int D>
int max_clusters_t(int flags, int C, int smem_bytes) {
  switch (kind_of(flags)) {
    case KIND_STEP: return max_clusters_kind<T, D, KIND_STEP>(C, smem_bytes);
    case KIND_DENSE: return max_clusters_kind<T, D, KIND_DENSE>(C, smem_bytes);
    default: return max_clusters_kind<T, D, KIND_STAGE>(C, smem_bytes);
  }
}

}  // namespace fasa
