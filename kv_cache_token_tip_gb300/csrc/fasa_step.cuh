// The fused FASA decode step for bf16 caches, laid out for the shortest chain
// of dependent phases at small batch.
//
// One thread-block cluster of C CTAs owns one (batch, KV head) unit:
//
//   1. RoPE of the G query heads of the group, the GQA-summed query
//      restricted to the dominant FCs (q-bar), and TIP: each CTA streams its
//      contiguous token range of the FC-major dominant-key copy into shared
//      memory with 1-D bulk copies and forms S_tau = sum_j qbar^[j] . k^[j]
//      in fp32 ("FASA: Frequency-aware Sparse Attention", "Online Stage 1:
//      Token Importance Predictor").  When the range fits in shared memory
//      every copy is issued at once and nothing is refilled.  A 12-bit
//      histogram of the scores' order-preserving keys is built on the way.
//   2. Top-k in one exchange.  Each CTA lists its own top-rho tokens in the
//      stable order (score descending, token ascending) -- rho is about k/C
//      plus four standard deviations of a random share -- and sends the list
//      to every CTA of the cluster.  Every CTA then finds the k-th largest
//      entry theta of the union.  The entries >= theta are the exact TopK-I
//      of the unit unless some CTA that cut its list (and sent fewer than k)
//      had every entry it sent selected: only then could a token it left out
//      belong to the top k.  In that case the CTAs exchange their exact local
//      top-k lists, whose union always holds the top k, and select again.
//   3. FAC ("Online Stage 2: Focused Attention Computation"): each CTA
//      gathers its own selected K/V rows with cp.async -- when they fit, the
//      whole first-round list is gathered while the exchange is in flight and
//      the rows that lose are masked -- and runs softmax(q K^T / sqrt(d)) V
//      on tensor cores (mma.sync, bf16 hi/lo-split q and P, fp32
//      accumulation).  The per-head partial records (o, m, l) are cut into
//      output slices and pushed to the CTAs that finish those slices.
//
// Exchanges are distributed-shared-memory stores followed by one
// release-arrive per destination on that CTA's mbarrier: a CTA waits only
// for the data it needs, every wait is bounded, and one cluster barrier at
// the end keeps each CTA's shared memory alive until no peer can touch it.
#pragma once

#include <limits.h>

#include "fasa_cluster.cuh"

namespace fasa {

constexpr int SB_X1 = 12;          // first selection exchange (C arrivals)
constexpr int SB_X2 = 13;          // second selection exchange (C arrivals)
constexpr int SB_COMB = 14;        // partial records for the combine (C arrivals)
constexpr int SB_RELOAD = 15;      // score reload from the workspace


struct StepMisc {
  int dig, gt, bucket, pad0;  // radix digit search result
  int scan[NW];
  int scan2[NW];
  int tip_fail;
  int big_unsafe;       // a TIP copy did not land in time: shared staging is not reused
  int nfc;              // this head's dominant-FC count
  int hist_clobbered;   // the digit-0 histogram was overwritten by later digits
  uint32_t tip_done[ST_MAX_STAGES];
  int tip_last[ST_MAX_STAGES];
  int4 hdr1[C_MAX];     // per source CTA: (listed, cut short, shared staging unusable, -)
  int4 hdr2[C_MAX];
  int sel[C_MAX];       // per source CTA: its entries >= theta
  int n_rows;
};
static_assert(sizeof(StepMisc) <= ST_MISC_BYTES, "step scratch too small");

// Selected: key > thr, or key == thr and the token's rank among this CTA's
// keys equal to thr (token order) is below `need`.
struct SelRule {
  uint32_t thr;
  int need;
};

#ifdef FASA_PHASE_TRACE
#define STEP_TRACE(i)                                                                   \
  do {                                                                                  \
    if (threadIdx.x == 0 && p.trace)                                                    \
      p.trace[((size_t)blockIdx.y * gridDim.x + blockIdx.x) * 16 + (i)] = global_timer_ns(); \
  } while (0)
#else
#define STEP_TRACE(i) \
  do {                \
  } while (0)
#endif

__device__ __forceinline__ int warp_sum_i(int v) { return __reduce_add_sync(0xffffffffu, v); }

// Exclusive prefix over the lanes of a warp.
__device__ __forceinline__ int warp_excl_scan(int v, int lane) {
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  return incl - v;
}

// Finds the digit holding the k_rem-th largest key in a histogram of NB bins
// (bins counted from the top).  out[0] = digit, out[1] = keys in larger
// digits, out[2] = keys in the digit.  Every thread must call it.
template <int NB>
__device__ __forceinline__ void find_digit(const uint32_t* hist, int k_rem, int* scan, int* out) {
  constexpr int M = NB / NT;
  static_assert(M >= 1 && NB % NT == 0 && M % 4 == 0, "bins per thread");
  const int tid = threadIdx.x;
  const int base = NB - (tid + 1) * M;
  uint32_t c[M];
#pragma unroll
  for (int q = 0; q < M / 4; ++q) {
    const uint4 v = reinterpret_cast<const uint4*>(hist + base)[q];
    c[4 * q] = v.x;
    c[4 * q + 1] = v.y;
    c[4 * q + 2] = v.z;
    c[4 * q + 3] = v.w;
  }
  int tsum = 0;
#pragma unroll
  for (int i = 0; i < M; ++i) tsum += (int)c[i];
  int total;
  int run = block_excl_scan(tsum, scan, total);
#pragma unroll
  for (int i = M - 1; i >= 0; --i) {
    const int ci = (int)c[i];
    if (run < k_rem && k_rem <= run + ci) {
      out[0] = base + i;
      out[1] = run;
      out[2] = ci;
    }
    run += ci;
  }
  __syncthreads();
}

// TIP score of four consecutive tokens over NFC dominant FCs (NFC == 0: nfc
// at run time).  `row` points at the lane's 16 bytes of FC 0 in a staged
// block (FC j is fc_row_bytes further on); two accumulators per token keep
// the FMA chains short.
template <int NFC>
__device__ __forceinline__ void tip4(const unsigned char* row, int nfc_rt, const float* qbar, float (&acc)[4]) {
  constexpr uint32_t FCB = KDOM_BLOCK * 2 * 2;  // bf16 FC row of a block
  const int nfc = NFC > 0 ? NFC : nfc_rt;
  float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
  auto fc_add = [&](int j, float (&a)[4]) {
    const float2 qq = *reinterpret_cast<const float2*>(&qbar[2 * j]);
    const uint4 w = *reinterpret_cast<const uint4*>(row + j * FCB);
    a[0] = fmaf(qq.x, bf16_lo(w.x), fmaf(qq.y, bf16_hi(w.x), a[0]));
    a[1] = fmaf(qq.x, bf16_lo(w.y), fmaf(qq.y, bf16_hi(w.y), a[1]));
    a[2] = fmaf(qq.x, bf16_lo(w.z), fmaf(qq.y, bf16_hi(w.z), a[2]));
    a[3] = fmaf(qq.x, bf16_lo(w.w), fmaf(qq.y, bf16_hi(w.w), a[3]));
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
#pragma unroll
  for (int t = 0; t < 4; ++t) acc[t] = a0[t] + a1[t];
}

// Up to four scores at scr[tl..tl+4) below `end`, as keys; ok marks the valid ones.
__device__ __forceinline__ void keys4(const float* scr, int tl, int end, uint32_t (&key)[4], bool (&ok)[4]) {
  if (tl + 4 <= end) {
    const float4 x = *reinterpret_cast<const float4*>(scr + tl);
    key[0] = score_key(x.x);
    key[1] = score_key(x.y);
    key[2] = score_key(x.z);
    key[3] = score_key(x.w);
    ok[0] = ok[1] = ok[2] = ok[3] = true;
  } else {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      ok[t] = tl + t < end;
      key[t] = ok[t] ? score_key(scr[tl + t]) : 0u;
    }
  }
}

// The rule that selects this CTA's top r scores (stable order) -- or, when
// the digit-0 bucket leaves at most `cap` keys at or above it, all of those
// (a longer prefix of the same order).  scr holds the CTA's nloc scores;
// hist the digit-0 histogram of their keys (rebuilt first unless hist_ok).
// Later digits (10 + 10 bits) overwrite the histogram.  Every thread calls it.
__device__ SelRule local_rule(int r, int cap, bool hist_ok, const float* scr, int nloc, uint32_t* hist,
                              StepMisc* ms) {
  const int tid = threadIdx.x;
  if (r >= nloc) return SelRule{0u, INT_MAX};  // every key is >= 0
  if (!hist_ok) {
    uint4* z = reinterpret_cast<uint4*>(hist);
    for (int i = tid; i < HLOC_BINS / 4; i += NT) z[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    for (int tl = tid * 4; tl < nloc; tl += NT * 4) {
      uint32_t key[4];
      bool ok[4];
      keys4(scr, tl, nloc, key, ok);
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (ok[t]) atomicAdd(&hist[key[t] >> 20], 1u);
    }
    __syncthreads();
  }
  int* res = &ms->dig;
  find_digit<HLOC_BINS>(hist, r, ms->scan, res);
  const int d0 = res[0], gt0 = res[1], b0 = res[2];
  if (gt0 + b0 <= cap) return SelRule{(uint32_t)d0 << 20, INT_MAX};
  // digits 1 and 2 (10 bits each) over the keys still in the running prefix
  if (tid == 0) ms->hist_clobbered = 1;
  int k_rem = r - gt0;
  uint32_t prefix = (uint32_t)d0;
  for (int dg = 1; dg <= 2; ++dg) {
    const int shift = dg == 1 ? 10 : 0;
    for (int i = tid; i < 1024; i += NT) hist[i] = 0u;
    __syncthreads();
    for (int tl = tid * 4; tl < nloc; tl += NT * 4) {
      uint32_t key[4];
      bool ok[4];
      keys4(scr, tl, nloc, key, ok);
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (ok[t] && (key[t] >> (shift + 10)) == prefix) atomicAdd(&hist[(key[t] >> shift) & 1023u], 1u);
    }
    __syncthreads();
    find_digit<1024>(hist, k_rem, ms->scan, res);
    k_rem -= res[1];
    prefix = (prefix << 10) | (uint32_t)res[0];
    if (res[2] == k_rem) return SelRule{prefix << shift, INT_MAX};
  }
  return SelRule{prefix, k_rem};  // ties on the full key, taken in token order
}

// Lists the entries of this CTA's nloc scores (tokens t0..) that rule R
// selects, in token order, into dst as packed (key << 32 | ~token): a
// larger value comes earlier in the stable order.  Warp w sweeps its own
// contiguous share of the tokens, four per lane per step.  Returns the count
// (at most cap entries are written).  Every thread calls it.
__device__ int list_rule(SelRule R, const float* scr, int nloc, int t0, unsigned long long* dst, int cap,
                         StepMisc* ms) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool ties = R.need != INT_MAX;
  const int wlen = (((nloc + NW - 1) / NW) + 3) & ~3;
  const int w0 = min(nloc, warp * wlen), w1 = min(nloc, w0 + wlen);
  int tie_base = 0;
  if (ties) {
    int c = 0;
    for (int tl = w0 + lane * 4; tl < w1; tl += 128) {
      uint32_t key[4];
      bool ok[4];
      keys4(scr, tl, w1, key, ok);
#pragma unroll
      for (int t = 0; t < 4; ++t) c += ok[t] && key[t] == R.thr;
    }
    c = warp_sum_i(c);
    if (lane == 0) ms->scan2[warp] = c;
    __syncthreads();
    for (int w = 0; w < warp; ++w) tie_base += ms->scan2[w];
  }
  // selection flags of a lane's four tokens; tb = ties before this step (CTA)
  auto flags4 = [&](int tl, int tb, uint32_t (&key)[4], bool (&sel)[4], int& nties) {
    bool ok[4];
    keys4(scr, tl, w1, key, ok);
    int lt = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) lt += ok[t] && key[t] == R.thr;
    int before = 0;
    nties = 0;
    if (ties) {
      before = warp_excl_scan(lt, lane);
      nties = __shfl_sync(0xffffffffu, before + lt, 31);
    }
    int rank = tb + before;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const bool tie = ok[t] && key[t] == R.thr;
      sel[t] = ok[t] && (key[t] > R.thr || (tie && rank < R.need));
      rank += tie;
    }
  };
  int cnt = 0;
  {
    int tb = tie_base;
    for (int tl0 = w0; tl0 < w1; tl0 += 128) {
      uint32_t key[4];
      bool sel[4];
      int nt;
      flags4(tl0 + lane * 4, tb, key, sel, nt);
      tb += nt;
#pragma unroll
      for (int t = 0; t < 4; ++t) cnt += sel[t];
    }
  }
  cnt = warp_sum_i(cnt);
  if (lane == 0) ms->scan[warp] = cnt;
  __syncthreads();
  int base = 0, total = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const int c = ms->scan[w];
    base += w < warp ? c : 0;
    total += c;
  }
  int tb = tie_base;
  for (int tl0 = w0; tl0 < w1; tl0 += 128) {
    uint32_t key[4];
    bool sel[4];
    int nt;
    const int tl = tl0 + lane * 4;
    flags4(tl, tb, key, sel, nt);
    tb += nt;
    const int mine = (int)sel[0] + (int)sel[1] + (int)sel[2] + (int)sel[3];
    const int bef = warp_excl_scan(mine, lane);
    int at = base + bef;
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (sel[t]) {
        if (at < cap)
          dst[at] = ((unsigned long long)key[t] << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)(t0 + tl + t));
        ++at;
      }
    base += __shfl_sync(0xffffffffu, bef + mine, 31);
  }
  __syncthreads();
  return min(total, cap);
}

// Sends this CTA's list (slot crank of `recv`, n entries, already in place
// locally) and its header to every other CTA of the cluster, then arrives on
// every CTA's exchange barrier `bar_off`.  Every thread calls it.
__device__ __forceinline__ void push_list(unsigned long long* recv, int cap, int n, int4 hdr, int4* hdrs,
                                          uint32_t bar_local, uint32_t crank, int C) {
  const int tid = threadIdx.x;
  const int nvec = (n + 1) >> 1;  // 16-byte vectors of two entries
  const uint32_t slot = smem_u32(recv + (size_t)crank * cap);
  const uint4* src = reinterpret_cast<const uint4*>(recv + (size_t)crank * cap);
  for (int x = tid; x < (C - 1) * nvec; x += NT) {
    const int rr = x / nvec, v = x - rr * nvec;
    const uint32_t r = (uint32_t)(rr + (rr >= (int)crank));
    dsmem_st_v4u32(dsmem_map(slot + v * 16, r), src[v]);
  }
  if (tid < C)
    dsmem_st_v4u32(dsmem_map(smem_u32(&hdrs[crank]), (uint32_t)tid),
                   make_uint4((uint32_t)hdr.x, (uint32_t)hdr.y, (uint32_t)hdr.z, (uint32_t)hdr.w));
  __syncthreads();
  if (tid < C) mbar_arrive_remote(dsmem_map(bar_local, (uint32_t)tid));
}

// The k-th largest value theta of the union of the C received lists (slot r
// holds hdrs[r].x entries; values are distinct), by 8-bit most-significant
// digits: exactly k entries are >= theta (the caller guarantees the union
// holds at least k).  Also stores per source the count of its entries >=
// theta in ms->sel.  Every thread calls it.
__device__ unsigned long long union_kth(const unsigned long long* recv, const int4* hdrs, int cap, int C, int k,
                                        uint32_t* uh, StepMisc* ms) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  static_assert(NT == UH_BINS, "one digit bin per thread");
  unsigned long long prefix = 0ull;
  int shift = 64, k_rem = k;
  const int nslots = C * cap;
  while (true) {
    shift -= 8;
    uh[tid] = 0u;
    __syncthreads();
    for (int f = tid; f < nslots; f += NT) {
      const int r = f / cap, i = f - r * cap;
      if (i < hdrs[r].x) {
        const unsigned long long x = recv[f];
        if (shift == 56 || (x >> (shift + 8)) == prefix) atomicAdd(&uh[(uint32_t)(x >> shift) & 255u], 1u);
      }
    }
    __syncthreads();
    if (warp == 0) {
      // lane L owns bins 255 - 8L - j, j = 0..7, counted from the top
      uint32_t c[8];
      int s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = uh[255 - 8 * lane - j];
        s += (int)c[j];
      }
      int run = warp_excl_scan(s, lane);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run < k_rem && k_rem <= run + (int)c[j]) {
          ms->dig = 255 - 8 * lane - j;
          ms->gt = run;
          ms->bucket = (int)c[j];
        }
        run += (int)c[j];
      }
    }
    __syncthreads();
    const int d = ms->dig, gt = ms->gt, bucket = ms->bucket;
    k_rem -= gt;
    prefix = (prefix << 8) | (unsigned long long)d;
    if (bucket == k_rem || shift == 0) break;
  }
  const unsigned long long theta = prefix << shift;
  for (int r = warp; r < C; r += NW) {
    int c = 0;
    for (int i = lane; i < hdrs[r].x; i += 32) c += recv[(size_t)r * cap + i] >= theta;
    c = warp_sum_i(c);
    if (lane == 0) ms->sel[r] = c;
  }
  __syncthreads();
  return theta;
}

template <int D>
__global__ void __launch_bounds__(NT, 1) fasa_step_kernel(const __grid_constant__ StepParams p) {
  using T = __nv_bfloat16;
  constexpr int ES = 2;
  constexpr int KB = KDOM_BLOCK;  // k_dom tokens per block
  constexpr int ROWB = D * ES;    // bytes of one K/V row
  constexpr int CPR = ROWB / 16;  // 16-byte chunks per row
  constexpr uint32_t FCB = KB * 2 * ES;  // one FC of one k_dom block
  extern __shared__ __align__(1024) unsigned char smem[];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank();
  const int C = (int)cluster_size();
  const int unit = blockIdx.y;
  const int b = unit / p.Hkv, h = unit - (unit / p.Hkv) * p.Hkv;
  const int G = p.G;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  StepMisc* ms = reinterpret_cast<StepMisc*>(smem + p.off_misc);
  float* qrot = reinterpret_cast<float*>(smem + p.off_qrot);
  float* qbar = reinterpret_cast<float*>(smem + p.off_qbar);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + p.off_hist);
  uint32_t* uh = reinterpret_cast<uint32_t*>(smem + p.off_uh);
  float* sc_s = reinterpret_cast<float*>(smem + p.off_sc);
  unsigned long long* recv1 = reinterpret_cast<unsigned long long*>(smem + p.off_recv1);
  int* rows = reinterpret_cast<int*>(smem + p.off_rows);
  unsigned char* big = smem + p.off_big;
  unsigned long long* recv2 = reinterpret_cast<unsigned long long*>(smem + p.off_recv2);

  STEP_TRACE(0);
  // ---------------------------------------------------------------- set-up
  const int nfc_max = p.n_tip, tt = p.tip_tile, ns = p.tip_stages;
  if (tid == 0) {
    for (int s = 0; s < ns; ++s) mbar_init(smem_u32(&bars[s]), 1);
    mbar_init(smem_u32(&bars[SB_X1]), (uint32_t)C);
    mbar_init(smem_u32(&bars[SB_X2]), (uint32_t)C);
    mbar_init(smem_u32(&bars[SB_COMB]), (uint32_t)C);
    mbar_init(smem_u32(&bars[SB_RELOAD]), 1);
    fence_mbar_init();
    ms->tip_fail = 0;
    ms->big_unsafe = 0;
    ms->hist_clobbered = 0;
    ms->n_rows = 0;
    for (int r = 0; r < C_MAX; ++r) ms->sel[r] = 0;
    for (int s = 0; s < ST_MAX_STAGES; ++s) {
      ms->tip_done[s] = 0u;
      ms->tip_last[s] = -1;
    }
  }
  {
    uint4* z = reinterpret_cast<uint4*>(hist);
    for (int i = tid; i < HLOC_BINS / 4; i += NT) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  // release: the initialised barriers are visible to every peer before its
  // first remote arrive (the matching wait comes after TIP)
  cluster_arrive();
  __syncthreads();

  // small inputs, all loads in flight together
  const bool append = (p.flags & F_APPEND) != 0;
  bool bad = false;
  int len = p.seq_lens[b];
  int m_pos = append ? 0 : p.pos[b];
  const int dom_i = tid < nfc_max ? p.dom_fc[h * nfc_max + tid] : 0;
  int nfc = nfc_max;
  if (warp == 0) {  // this head's count: the entries before the first negative one
    const int d1 = lane + 32 < nfc_max ? p.dom_fc[h * nfc_max + lane + 32] : 0;
    const unsigned b0 = __ballot_sync(0xffffffffu, lane < nfc_max && dom_i < 0);
    const unsigned b1 = __ballot_sync(0xffffffffu, lane + 32 < nfc_max && d1 < 0);
    nfc = b0 ? __ffs(b0) - 1 : (b1 ? 31 + __ffs(b1) : nfc_max);
    nfc = max(nfc, 1);  // an empty set uses slot 0 (reported below)
    if (lane == 0) ms->nfc = nfc;
  }
  // F_APPEND: the new token's key and value pairs (thread i < D/2: pair i),
  // loaded whichever CTA turns out to own the token
  T kn0 = T(0.f), kn1 = T(0.f), vn0 = T(0.f), vn1 = T(0.f);
  if (append && tid < D / 2) {
    const T* kn = reinterpret_cast<const T*>(p.k_new) + (size_t)unit * D;
    const T* vn = reinterpret_cast<const T*>(p.v_new) + (size_t)unit * D;
    kn0 = kn[2 * tid];
    kn1 = kn[2 * tid + 1];
    vn0 = vn[2 * tid];
    vn1 = vn[2 * tid + 1];
  }
  constexpr int QPAIRS = (G_MAX * D / 2 + NT - 1) / NT;
  float2 qv[QPAIRS];
#pragma unroll
  for (int k = 0; k < QPAIRS; ++k) {
    const int x = tid + k * NT;
    qv[k] = make_float2(0.f, 0.f);
    if (x < G * (D / 2)) {
      const int g = x / (D / 2), i = x - g * (D / 2);
      const T* qg = reinterpret_cast<const T*>(p.q) + ((size_t)b * p.Hq + (size_t)h * G + g) * D + 2 * i;
      qv[k] = make_float2(to_f32<T>(qg[0]), to_f32<T>(qg[1]));
    }
  }
  if (len < 0 || len > p.T_max) {
    bad = true;
    len = min(max(len, 0), p.T_max);
  }
  // F_APPEND: the step's own token goes to index t_new = len, the query sits
  // at that position, and the step attends len + 1 tokens (a full cache
  // cannot take the token: reported, not appended)
  int t_new = -1;
  if (append) {
    m_pos = len;
    if (len < p.T_max) {
      t_new = len;
      len += 1;
    } else {
      bad = true;
    }
  }
  const int k_eff = min(p.budget, len);
  const bool need_select = len > p.budget;
  // contiguous token range of this CTA, its start aligned to a k_dom block
  const int chunk = ((len + C - 1) / C + KB - 1) / KB * KB;
  const int t0 = min(len, (int)crank * chunk);
  const int t1 = min(len, t0 + chunk);
  const int nloc = t1 - t0;
  // K_dom is streamed up to the new token, which its CTA scores from registers
  const bool own_new = t_new >= t0 && t_new < t1;
  const int nloc_s = own_new ? t_new - t0 : nloc;
  const int t1s = t0 + nloc_s;

  // ---------------------------------------------------------------- TIP loads
  // k_dom is [.., T_max/KB, n_tip, KB, 2]: a tile of whole blocks is one
  // contiguous range (one bulk copy); a head using fewer planes takes the
  // leading nfc planes of each block, packed in the stage
  const int ntiles = need_select ? (nloc_s + tt - 1) / tt : 0;
  const uint32_t stage_bytes = (uint32_t)(tt / KB) * nfc_max * FCB;
  const T* kd_unit = reinterpret_cast<const T*>(p.k_dom) + (size_t)unit * nfc_max * p.T_max * 2;
  auto tip_issue = [&](int it) {  // one thread; nfc is this head's count
    const int s = it % ns;
    const int tau0 = t0 + it * tt;
    const int nblk = (min(tt, t1s - tau0) + KB - 1) / KB;
    const uint32_t blk_bytes = (uint32_t)nfc * FCB;
    const uint32_t bar = smem_u32(&bars[s]);
    mbar_arrive_expect_tx(bar, (uint32_t)nblk * blk_bytes);
    const T* src = kd_unit + (size_t)(tau0 / KB) * nfc_max * KB * 2;
    if (it != p.drop_stage) {
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

  // ------------------------------------------------------------ query prep
#pragma unroll
  for (int k = 0; k < QPAIRS; ++k) {
    const int x = tid + k * NT;
    if (x < G * (D / 2)) {
      const int g = x / (D / 2), i = x - g * (D / 2);
      const float2 c = rope_cos_sin(p.rope_turns[i], m_pos);
      *reinterpret_cast<float2*>(&qrot[g * D + 2 * i]) =
          make_float2(qv[k].x * c.x - qv[k].y * c.y, qv[k].x * c.y + qv[k].y * c.x);
    }
  }
  __syncthreads();
  nfc = ms->nfc;
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
  __syncthreads();

  // F_APPEND, in the CTA that owns the new token: rotate its key by its
  // position, store key and value at index t_new of the cache and the key's
  // dominant FCs in K_dom, and score it exactly as the TIP loop scores a
  // streamed token (same FC order and accumulation, stored precision).
  float s_new = 0.f;
  if (own_new) {
    float2* knew = reinterpret_cast<float2*>(uh);  // rotated key pairs, as stored (D/2 <= UH_BINS/2)
    T* Kw = const_cast<T*>(reinterpret_cast<const T*>(p.k_cache)) + ((size_t)unit * p.T_max + t_new) * D;
    T* Vw = const_cast<T*>(reinterpret_cast<const T*>(p.v_cache)) + ((size_t)unit * p.T_max + t_new) * D;
    if (tid < D / 2) {
      const int i = tid;
      const float x0 = to_f32<T>(kn0), x1 = to_f32<T>(kn1);
      const float2 c = rope_cos_sin(p.rope_turns[i], t_new);
      const T r0 = from_f32<T>(x0 * c.x - x1 * c.y), r1 = from_f32<T>(x0 * c.y + x1 * c.x);
      Kw[2 * i] = r0;
      Kw[2 * i + 1] = r1;
      Vw[2 * i] = vn0;
      Vw[2 * i + 1] = vn1;
      knew[i] = make_float2(to_f32<T>(r0), to_f32<T>(r1));
    }
    __syncthreads();
    T* kdw = const_cast<T*>(kd_unit) + ((size_t)(t_new / KB) * nfc_max * KB + (t_new % KB)) * 2;
    auto dom_at = [&](int j) { return min(max(p.dom_fc[h * nfc_max + j], 0), D / 2 - 1); };
    for (int j = tid; j < nfc; j += NT) {
      const float2 kp = knew[dom_at(j)];
      kdw[(size_t)j * KB * 2] = from_f32<T>(kp.x);
      kdw[(size_t)j * KB * 2 + 1] = from_f32<T>(kp.y);
    }
    if (tid == 0 && need_select) {
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
  STEP_TRACE(1);

  // ---------------------------------------------------------------- TIP scan
  // Warp w scores the 128-token units w, w + NW, ...; a unit lies in one
  // stage.  In a refilled ring each unit's warp counts itself done with the
  // stage, and the warp that completes the stage refills it.  A wait that
  // runs out stops the warp and, through ms->tip_fail, the others.
  float* scw = p.s_cap > 0 ? sc_s : p.scores + (size_t)unit * p.T_max + t0;
  if (own_new && need_select && tid == 0) {  // the appended token's score, as TIP would
    scw[nloc_s] = s_new;
    atomicAdd(&hist[score_key(s_new) >> 20], 1u);
  }
  const int upt = tt / TIP_UNIT;
  const int nunits = ntiles > 0 ? (nloc_s + TIP_UNIT - 1) / TIP_UNIT : 0;
  const bool ring = ntiles > ns;
  const uint32_t blk_bytes = (uint32_t)nfc * FCB;
  int tip_fail = 0;
  for (int u = warp; u < nunits; u += NW) {
    const int it = u / upt, s = it % ns;
    const uint32_t parity = (uint32_t)(it / ns) & 1u;
    int stop = lane == 0 ? *reinterpret_cast<volatile int*>(&ms->tip_fail) : 0;
    if (__shfl_sync(0xffffffffu, stop, 0)) break;
    const bool ok = mbar_wait_bounded(smem_u32(&bars[s]), parity, p.wait_ns);
    if (!__all_sync(0xffffffffu, ok)) {
      tip_fail = 1;
      if (lane == 0) atomicOr(&ms->tip_fail, 1);
      break;
    }
    const unsigned char* row =
        big + s * stage_bytes + ((u - it * upt) * 2 + (lane >> 4)) * blk_bytes + (lane & 15) * 16;
    float acc[4];
    switch (nfc) {  // the common counts get fully unrolled loops
      case 8: tip4<8>(row, nfc, qbar, acc); break;
      case 12: tip4<12>(row, nfc, qbar, acc); break;
      case 16: tip4<16>(row, nfc, qbar, acc); break;
      default: tip4<0>(row, nfc, qbar, acc); break;
    }
    const int tl = u * TIP_UNIT + lane * 4;
    if (tl + 4 <= nloc_s) {
      *reinterpret_cast<float4*>(scw + tl) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    } else {
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (tl + t < nloc_s) scw[tl + t] = acc[t];
    }
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (tl + t < nloc_s) atomicAdd(&hist[score_key(acc[t]) >> 20], 1u);
    if (ring) {
      // every lane's reads of the stage returned (they fed the FMAs above)
      __syncwarp();
      if (lane == 0) {
        const uint32_t prev = atomicAdd(&ms->tip_done[s], 1u);
        const int n_in = min(upt, nunits - it * upt);
        if ((int)prev + 1 == n_in) {
          ms->tip_done[s] = 0u;
          if (it + ns < ntiles) tip_issue(it + ns);
        }
      }
    }
  }
  if (__syncthreads_or(tip_fail | (nunits > 0 ? ms->tip_fail : 0))) {
    if (tid == 0) {
      atomicOr(p.status, 2);
      // copies still in flight must land before the staging is reused; one
      // that does not within one more wait bound (for all stages together)
      // is reported and the staging is left alone
      bool drained = true;
      const uint64_t start = global_timer_ns();
      for (int s = 0; s < ns; ++s)
        if (ms->tip_last[s] >= 0) {
          const uint64_t spent = global_timer_ns() - start;
          const uint64_t left = spent < p.wait_ns ? p.wait_ns - spent : 1ull;
          drained &= mbar_wait_bounded(smem_u32(&bars[s]), (uint32_t)(ms->tip_last[s] / ns) & 1u, left);
        }
      if (!drained) {
        atomicOr(p.status, 4);
        ms->big_unsafe = 1;
      }
    }
    __syncthreads();
  }
  const bool big_ok = ms->big_unsafe == 0;
  // Waits on peer CTAs get 8x the copy bound: a peer reaches each exchange
  // after at most three copy-bound waits of its own (TIP, drain, reload), so
  // a peer's timeout never makes this CTA give up on it, and every CTA sees
  // the same exchanged data and takes the same branches around the cluster
  // barriers.
  const uint64_t xwait = p.wait_ns * 8ull;
  // the peers' barriers are initialised (paired with the arrive at set-up)
  cluster_wait();
  STEP_TRACE(2);

  // ---------------------------------------------------------------- top-k
  unsigned long long theta = 0ull;
  int n1 = 0;
  bool second = false;         // the second exchange decided the selection
  int sel_before = 0;          // selected tokens of the lower-ranked CTAs
  const bool spec = p.spec != 0 && big_ok;
  const T* Kb = reinterpret_cast<const T*>(p.k_cache) + (size_t)unit * p.T_max * D;
  const T* Vb = reinterpret_cast<const T*>(p.v_cache) + (size_t)unit * p.T_max * D;
  constexpr uint32_t GSLOT_B = 2u * GR * ROWB;
  // FAC rows: fr_n rows, contiguous tokens fr_r0.. or a list -- the
  // first-round list itself (masked by theta) or the compact own selection
  const unsigned long long* fslot = nullptr;
  bool contig = true;
  int fr_n = 0, fr_r0 = 0;
  auto row_token = [&](int i) -> int {
    if (contig) return fr_r0 + i;
    if (fslot) return (int)(0xFFFFFFFFu - (uint32_t)fslot[i]);
    return rows[i];
  };
  // The first fac_wst groups of every warp, issued by the whole CTA (group g
  // belongs to warp g % NW, slot g / NW).  Rows past fr_n are zero-filled:
  // the tensor cores multiply them by zero weights, which must not meet
  // stale NaNs.  Row chunk c sits at chunk position c ^ (row & 7) so the
  // eight rows an ldmatrix reads fall in distinct banks.
  auto fac_start = [&]() {
    const int nfirst = min((fr_n + GR - 1) / GR * GR, p.fac_wst * NW * GR);
    for (int c = tid; c < nfirst * 2 * CPR; c += NT) {
      const int i = c / (2 * CPR), rem = c - i * (2 * CPR);
      const int which = rem >= CPR, ch = rem - which * CPR;
      const int g = i / GR, rr = i - g * GR;
      const uint32_t st0 = smem_u32(big) + (uint32_t)((g % NW) * p.fac_wst + g / NW) * GSLOT_B;
      const bool real = i < fr_n;
      const size_t row_off = real ? (size_t)row_token(i) * D : 0;
      cp_async16_zfill(st0 + which * GR * ROWB + rr * ROWB + ((ch ^ (rr & 7)) * 16),
                       (which ? Vb : Kb) + row_off + ch * (16 / ES), real ? 16u : 0u);
    }
    cp_async_commit();
  };

  if (need_select) {
    // the sweeps read shared memory: scores kept there, or workspace scores
    // copied back into the idle staging (warp w moves its share)
    const float* scr = p.s_cap > 0 ? sc_s : scw;
    if (p.reload && big_ok) {
      const int nv = (nloc + 3) >> 2;
      const int per_w = (nv + NW - 1) / NW;
      const int v0 = min(nv, warp * per_w), v1 = min(nv, v0 + per_w);
      const uint32_t rbar = smem_u32(&bars[SB_RELOAD]);
      fence_proxy_async_global();  // this thread's score stores, before the copy reads them
      __syncthreads();
      if (lane == 0) {
        if (warp == 0) mbar_arrive_expect_tx(rbar, (uint32_t)nv * 16u);
        if (v1 > v0) bulk_g2s(smem_u32(big) + v0 * 16, scw + v0 * 4, (uint32_t)(v1 - v0) * 16u, rbar);
      }
      if (!mbar_wait_bounded(rbar, 0u, p.wait_ns)) {
        if (tid == 0) atomicOr(p.status, 2);
      } else {
        scr = reinterpret_cast<const float*>(big);
      }
    }
    // first round: the own top-rho list, sent to every CTA
    const SelRule R1 = local_rule(min(p.rho, nloc), p.cap1, true, scr, nloc, hist, ms);
    n1 = list_rule(R1, scr, nloc, t0, recv1 + (size_t)crank * p.cap1, p.cap1, ms);
    STEP_TRACE(3);
    if (spec) {  // gather the listed rows now; the selection only masks them
      fslot = recv1 + (size_t)crank * p.cap1;
      contig = false;
      fr_n = n1;
      fac_start();
    }
    push_list(recv1, p.cap1, n1, make_int4(n1, nloc > n1 ? 1 : 0, big_ok ? 0 : 1, 0), ms->hdr1,
              smem_u32(&bars[SB_X1]), crank, C);
    if (!mbar_wait_cluster_bounded(smem_u32(&bars[SB_X1]), 0u, xwait) && tid == 0) atomicOr(p.status, 2);
    STEP_TRACE(4);
    if (tid < C) ms->hdr1[tid].x = min(max(ms->hdr1[tid].x, 0), p.cap1);  // (only a timed-out wait leaves stale ones)
    __syncthreads();
    int total = 0;
    bool any_unsafe = false;
    for (int r = 0; r < C; ++r) {
      total += ms->hdr1[r].x;
      any_unsafe |= ms->hdr1[r].z != 0;
    }
    bool valid = total >= k_eff;
    if (valid) {
      theta = union_kth(recv1, ms->hdr1, p.cap1, C, k_eff, uh, ms);
      for (int r = 0; r < C; ++r) {
        const int4 hd = ms->hdr1[r];
        if (hd.y && hd.x < k_eff && ms->sel[r] == hd.x) valid = false;
      }
    }
    STEP_TRACE(5);
    if (!valid && !any_unsafe) {
      // Second round: every CTA sends its exact local top-k.  The staging
      // that receives them must be idle in every CTA first.
      second = true;
      cp_async_wait<0>();
      __syncthreads();
      cluster_sync();
      const float* scr2 = p.s_cap > 0 ? sc_s : scw;
      const SelRule R2 = local_rule(min(k_eff, nloc), p.cap2, ms->hist_clobbered == 0, scr2, nloc, hist, ms);
      const int n2 = list_rule(R2, scr2, nloc, t0, recv2 + (size_t)crank * p.cap2, p.cap2, ms);
      push_list(recv2, p.cap2, n2, make_int4(n2, nloc > n2 ? 1 : 0, 0, 0), ms->hdr2, smem_u32(&bars[SB_X2]),
                crank, C);
      if (!mbar_wait_cluster_bounded(smem_u32(&bars[SB_X2]), 0u, xwait) && tid == 0) atomicOr(p.status, 2);
      if (tid < C) ms->hdr2[tid].x = min(max(ms->hdr2[tid].x, 0), p.cap2);
      __syncthreads();
      int total2 = 0;
      for (int r = 0; r < C; ++r) total2 += ms->hdr2[r].x;
      if (total2 >= k_eff) theta = union_kth(recv2, ms->hdr2, p.cap2, C, k_eff, uh, ms);
      STEP_TRACE(6);
    }
    for (int r = 0; r < (int)crank; ++r) sel_before += ms->sel[r];
    // the own selection, compact and in token order (the own list is in
    // token order): warp w takes a contiguous share of the list
    {
      const unsigned long long* own = second ? recv2 + (size_t)crank * p.cap2 : recv1 + (size_t)crank * p.cap1;
      const int n_own = second ? ms->hdr2[crank].x : n1;
      const int per_w = (n_own + NW - 1) / NW;
      const int e0 = min(n_own, warp * per_w), e1 = min(n_own, e0 + per_w);
      int c = 0;
      for (int e = e0 + lane; e < e1; e += 32) c += own[e] >= theta;
      c = warp_sum_i(c);
      if (lane == 0) ms->scan2[warp] = c;
      __syncthreads();
      int at = 0, n_sel = 0;
      for (int w = 0; w < NW; ++w) {
        at += w < warp ? ms->scan2[w] : 0;
        n_sel += ms->scan2[w];
      }
      for (int e0b = e0; e0b < e1; e0b += 32) {
        const int e = e0b + lane;
        const bool s = e < e1 && own[e] >= theta;
        const unsigned bal = __ballot_sync(0xffffffffu, s);
        const int pos = at + __popc(bal & ((1u << lane) - 1u));
        if (s && pos < p.rows_cap) rows[pos] = (int)(0xFFFFFFFFu - (uint32_t)own[e]);
        at += __popc(bal);
      }
      if (tid == 0) ms->n_rows = min(n_sel, p.rows_cap);
      __syncthreads();
    }
    if (!spec || second) {
      fslot = nullptr;
      contig = false;
      fr_n = ms->n_rows;
      if (big_ok) fac_start();
    }
  } else {
    // every cached token is attended: rows split evenly over the cluster.
    // An appended row may be gathered by another CTA: the barrier orders its
    // owner's stores before the gathers.
    if (t_new >= 0) cluster_sync();
    fr_r0 = (k_eff * (int)crank) / C;
    fr_n = (k_eff * ((int)crank + 1)) / C - fr_r0;
    contig = true;
    if (big_ok) fac_start();
  }
  if (!big_ok) fr_n = 0;  // nothing was gathered: an empty record
  STEP_TRACE(7);

  // ---------------------------------------------------------------- FAC
  // Tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate), one
  // flash-decoding pass per warp over its own 16-row groups: QK as
  // S^T = K Q^T (16 rows x 8 heads), PV as O^T = V^T P^T (16 head dims x 8
  // heads per MMA).  q and the softmax weights P are split into bf16 hi + lo
  // parts, so the products keep ~16 mantissa bits.  Lane (gq, tq) holds rows
  // gq, gq + 8 of S^T and head dims gq, gq + 8 of O^T, heads 2tq, 2tq + 1.
  constexpr int PSTRIDE = D + 4;
  constexpr int KS = D / 16;
  float* rec = reinterpret_cast<float*>(big);                         // [G][NW][D + 2]
  float* part = rec + G_MAX * NW * (D + 2);                           // [G][D + 4]
  float* wts = part + G_MAX * PSTRIDE;                                // [G][NW] + [G]
  {
    const float qs = 1.4426950408889634f * rsqrtf((float)D);
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t qb[KS][2][2];  // [k-step][b0 / b1][hi / lo]
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int d0 = ks * 16 + 2 * tq + hb * 8;
        const float x0 = gq < G ? qrot[gq * D + d0] * qs : 0.f;
        const float x1 = gq < G ? qrot[gq * D + d0 + 1] * qs : 0.f;
        split_bf16(x0, x1, qb[ks][hb][0], qb[ks][hb][1]);
      }
    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F;  // running max (log2 units), heads 2tq, 2tq + 1
    float l0 = 0.f, l1 = 0.f;
    float oc[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) oc[mt][0] = oc[mt][1] = oc[mt][2] = oc[mt][3] = 0.f;
    float* pt = reinterpret_cast<float*>(smem + p.off_pt) + warp * (G_MAX * PTS);
    const int mi = lane >> 3;
    const int kr = (lane & 7) + 8 * (mi & 1), vr = (lane & 7) + 8 * (mi >> 1);
    const uint32_t k_row = kr * ROWB, v_row = vr * ROWB;
    const int k_c = mi >> 1, v_c = mi & 1, sw = lane & 7;
    const int wst = p.fac_wst;
    const int ngrp = (fr_n + GR - 1) / GR;
    auto grp_issue = [&](int g, int s) {
      if (g * GR < fr_n) {
        const uint32_t st0 = smem_u32(big) + (uint32_t)(warp * wst + s) * GSLOT_B;
        for (int c = lane; c < GR * 2 * CPR; c += 32) {
          const int rr = c / (2 * CPR), rem = c - rr * (2 * CPR);
          const int which = rem >= CPR, ch = rem - which * CPR;
          const int i = g * GR + rr;
          const bool real = i < fr_n;
          const size_t row_off = real ? (size_t)row_token(i) * D : 0;
          cp_async16_zfill(st0 + which * GR * ROWB + rr * ROWB + ((ch ^ (rr & 7)) * 16),
                           (which ? Vb : Kb) + row_off + ch * (16 / ES), real ? 16u : 0u);
        }
      }
      cp_async_commit();
    };
    cp_async_wait<0>();  // the CTA-wide first groups
    __syncthreads();
    int it = 0;
    for (int g = warp; g < ngrp; g += NW, ++it) {
      const int s = wst == 2 ? (it & 1) : 0;
      if (it > 0) {
        if (wst == 2) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncwarp();
      }
      const uint32_t Ks = smem_u32(big) + (uint32_t)(warp * wst + s) * GSLOT_B;
      const uint32_t Vs = Ks + GR * ROWB;
      float sh[4] = {0.f, 0.f, 0.f, 0.f}, slo[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(Ks + k_row + (((2 * ks + k_c) ^ sw) << 4), a0, a1, a2, a3);
        mma_bf16_16816(sh, a0, a1, a2, a3, qb[ks][0][0], qb[ks][1][0]);
        mma_bf16_16816(slo, a0, a1, a2, a3, qb[ks][0][1], qb[ks][1][1]);
      }
      const int r0 = g * GR + gq, r1 = r0 + 8;
      const bool v0 = r0 < fr_n && !(fslot && fslot[r0] < theta);
      const bool v1 = r1 < fr_n && !(fslot && fslot[r1] < theta);
      const float s0 = v0 ? sh[0] + slo[0] : -CUDART_INF_F, s1 = v0 ? sh[1] + slo[1] : -CUDART_INF_F;
      const float s2 = v1 ? sh[2] + slo[2] : -CUDART_INF_F, s3 = v1 ? sh[3] + slo[3] : -CUDART_INF_F;
      float x0 = fmaxf(s0, s2), x1 = fmaxf(s1, s3);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o));
      }
      const float n0 = fmaxf(m0, x0), n1m = fmaxf(m1, x1);
      // every row so far may be masked: then nothing is rescaled or added
      const float c0 = n0 == -CUDART_INF_F ? 1.f : exp2f(m0 - n0);
      const float c1 = n1m == -CUDART_INF_F ? 1.f : exp2f(m1 - n1m);
      const float p0 = n0 == -CUDART_INF_F ? 0.f : exp2f(s0 - n0);
      const float p2 = n0 == -CUDART_INF_F ? 0.f : exp2f(s2 - n0);
      const float p1 = n1m == -CUDART_INF_F ? 0.f : exp2f(s1 - n1m);
      const float p3 = n1m == -CUDART_INF_F ? 0.f : exp2f(s3 - n1m);
      l0 = l0 * c0 + p0 + p2;
      l1 = l1 * c1 + p1 + p3;
      m0 = n0;
      m1 = n1m;
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
      grp_issue(g + wst * NW, s);  // commits a group even when empty: the waits count groups
    }
    cp_async_wait<0>();
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    __syncthreads();  // every warp is done with its slots: `big` takes the warp records
    STEP_TRACE(8);
    if (big_ok) {
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
    }
    __syncthreads();
  }
  // merge the warps' records per head into this CTA's record part[g] =
  // (o[0..D), m, l): the head's maximum and the warp weights exp2(m_w - M)
  // once, then one multiply-add per warp and element
  if (big_ok) {
    if (tid < G) {
      const int g = tid;
      float M = -CUDART_INF_F;
      for (int r = 0; r < NW; ++r) M = fmaxf(M, rec[(g * NW + r) * (D + 2) + D]);
      for (int r = 0; r < NW; ++r) {
        const float m_r = rec[(g * NW + r) * (D + 2) + D];
        wts[g * NW + r] = m_r != -CUDART_INF_F ? exp2f(m_r - M) : 0.f;
      }
      wts[G * NW + g] = M;
    }
    __syncthreads();
    for (int x = tid; x < G * (D + 2); x += NT) {
      const int g = x / (D + 2), e = x - g * (D + 2);
      float val = wts[G * NW + g];
      if (e != D) {
        float acc = 0.f;
        for (int r = 0; r < NW; ++r) {
          const float w = wts[g * NW + r];
          if (w != 0.f) acc += w * rec[(g * NW + r) * (D + 2) + e];
        }
        val = acc;
      }
      part[g * PSTRIDE + e] = val;
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------- combine
  // Each CTA cuts its record into the C output slices (runs of 4-element
  // groups of the G*D outputs) and stores each slice, with (m, l) of every
  // head, into the shared memory of the CTA that finishes it, then arrives on
  // that CTA's barrier.
  const int ngrp4 = G * (D / 4);
  const int sl = (ngrp4 + C - 1) / C;
  float4* recv_o = reinterpret_cast<float4*>(smem + p.off_comb);  // [C][sl]
  float2* recv_ml = reinterpret_cast<float2*>(recv_o + C * sl);    // [C][G]
  const uint32_t recv_o_l = smem_u32(recv_o), recv_ml_l = smem_u32(recv_ml);
  for (int q = tid; q < ngrp4; q += NT) {
    const int r = ((q + 1) * C - 1) / ngrp4;  // the CTA whose slice holds group q
    const int q0r = (ngrp4 * r) / C;
    const int g = q / (D / 4), e4 = q - g * (D / 4);
    const float4 v = big_ok ? *reinterpret_cast<const float4*>(part + g * PSTRIDE + e4 * 4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    dsmem_st_v4f(dsmem_map(recv_o_l + ((int)crank * sl + q - q0r) * 16, (uint32_t)r), v.x, v.y, v.z, v.w);
  }
  for (int x = tid; x < C * G; x += NT) {
    const int r = x / G, g = x - r * G;
    const float mm = big_ok ? part[g * PSTRIDE + D] : -CUDART_INF_F;
    const float ll = big_ok ? part[g * PSTRIDE + D + 1] : 0.f;
    dsmem_st_v2f(dsmem_map(recv_ml_l + ((int)crank * G + g) * 8, (uint32_t)r), mm, ll);
  }
  __syncthreads();
  if (tid < C) mbar_arrive_remote(dsmem_map(smem_u32(&bars[SB_COMB]), (uint32_t)tid));
  // first half of the final cluster barrier: this CTA touches no peer's
  // shared memory after this point
  cluster_arrive();
  STEP_TRACE(9);
  if (!mbar_wait_cluster_bounded(smem_u32(&bars[SB_COMB]), 0u, xwait) && tid == 0) atomicOr(p.status, 2);
  STEP_TRACE(10);

  // Finish this CTA's slice: lpg lanes per output group (the power of two
  // >= C), lane r taking CTA r's record, reduced with width-lpg shuffles.
  const int q0 = (ngrp4 * (int)crank) / C, q1 = (ngrp4 * ((int)crank + 1)) / C;
  const int lpg = C <= 1 ? 1 : 1 << (32 - __clz(C - 1));
  const int gpw = 32 / lpg;
  for (int qw = q0 + gpw * warp; qw < q1; qw += gpw * NW) {  // warp-uniform bound
    const int q = qw + lane / lpg, r = lane & (lpg - 1);
    const bool okq = q < q1 && r < C;
    const int g = okq ? q / (D / 4) : 0, e4 = okq ? q - g * (D / 4) : 0;
    const float2 ml = okq ? recv_ml[r * G + g] : make_float2(-CUDART_INF_F, 0.f);
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

  // idx_out / count_out: the selected tokens of every CTA, concatenated in
  // cluster-rank (= token) order
  if (p.idx_out) {
    int* io = p.idx_out + (size_t)unit * p.budget;
    if (!need_select) {
      if (crank == 0)
        for (int i = tid; i < p.budget; i += NT) io[i] = i < k_eff ? i : -1;
    } else {
      const int n_own = ms->n_rows;
      for (int i = tid; i < n_own; i += NT)
        if (sel_before + i < p.budget) io[sel_before + i] = rows[i];
    }
  }
  if (p.count_out && crank == 0 && tid == 0) p.count_out[unit] = k_eff;
  if (bad) atomicOr(p.status, 1);
  STEP_TRACE(11);
  cluster_wait();
}

}  // namespace fasa
