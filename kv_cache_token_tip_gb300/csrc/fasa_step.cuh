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
// The exchange and the combine move each CTA's list or record slice to the
// other CTAs as one bulk copy per destination (shared memory to shared
// memory), completing on the destination's mbarrier: a CTA waits only for
// the data it needs, every wait is bounded, and one cluster barrier at the
// end keeps each CTA's shared memory alive until no copy or peer can touch
// it.
#pragma once

#include <limits.h>

#include "../../include/fasa.h"
#include "fasa_cluster.cuh"

namespace fasa {

constexpr int SB_X1 = 12;          // first selection exchange (the peers' bulk copies)
constexpr int SB_X2 = 13;          // second selection exchange (C arrivals)
constexpr int SB_COMB = 14;        // partial records for the combine (the peers' bulk copies)
constexpr int SB_RELOAD = 15;      // score reload from the workspace


// The unit's length and this CTA's token range, planned by the issuing warp
// and read by every thread after the set-up barrier.
struct StepHdr {
  int len, m_pos, t_new, bad;  // tokens attended, query position, appended index (-1: none), bad input
  int t0, nloc, nloc_s, ntiles;  // range start and size, tokens streamed, TIP tiles
  int nfc, pad[3];               // this head's dominant-FC count
};

struct StepMisc {
  StepHdr hdr;
  int dig, gt, bucket, pad0;  // radix digit search result
  int scan[SNW];
  int scan2[SNW];
  int tip_fail;
  int big_unsafe;       // a TIP copy did not land in time: shared staging is not reused
  int hist_clobbered;   // the digit-0 histogram was overwritten by later digits
  uint32_t tip_done[ST_MAX_STAGES];
  int tip_last[ST_MAX_STAGES];
  int sel[C_MAX];       // per source CTA: its entries >= theta
  int n_rows;
  uint32_t list_max;    // largest key listed
  int bkt_n;            // entries gathered from the union's threshold bucket
  unsigned long long theta;
  uint32_t chist[64];   // coarse histogram of the score keys (key >> 26)
  uint8_t fac_pair[64];  // F_KSPLIT: the FC of each pair position of a FAC key row
  unsigned long long bkt[32];
  int bkt_src[32];
};
static_assert(sizeof(StepMisc) <= ST_MISC_BYTES, "step scratch too small");

// Selected: key > thr, or key == thr and the token's rank among this CTA's
// keys equal to thr (token order) is below `need`.
struct SelRule {
  uint32_t thr;
  int need;
};

#ifdef FASA_PHASE_TRACE
// Tracing builds: lane 0 of every warp stores globaltimer (ns) in slot i and
// clock64 in slot 64 + i of its 128-slot record; 64 slots per warp.
__device__ unsigned long long* g_step_trace;
#define STEP_TRACE(i)                                                                                  \
  do {                                                                                                 \
    if ((threadIdx.x & 31) == 0 && g_step_trace) {                                                     \
      unsigned long long* tr_ =                                                                        \
          g_step_trace + (((size_t)blockIdx.y * gridDim.x + blockIdx.x) * SNW + (threadIdx.x >> 5)) * 128; \
      tr_[(i)] = global_timer_ns();                                                                    \
      tr_[64 + (i)] = clock64();                                                                       \
    }                                                                                                  \
  } while (0)
#define STEP_TRACE_VAL(i, v)                                                                           \
  do {                                                                                                 \
    if ((threadIdx.x & 31) == 0 && g_step_trace)                                                       \
      g_step_trace[(((size_t)blockIdx.y * gridDim.x + blockIdx.x) * SNW + (threadIdx.x >> 5)) * 128 + (i)] = \
          (unsigned long long)(v);                                                                     \
  } while (0)
#else
#define STEP_TRACE(i) \
  do {                \
  } while (0)
#define STEP_TRACE_VAL(i, v) \
  do {                       \
  } while (0)
#endif

__device__ __forceinline__ int warp_sum_i(int v) { return __reduce_add_sync(0xffffffffu, v); }

// n / d for 0 <= n < 2^31 with m = floor(2^32 / d) (0xffffffff for d = 1):
// the multiply-high is n / d or one less.
__device__ __forceinline__ int div_magic(int n, int d, uint32_t m) {
  int q = (int)__umulhi((uint32_t)n, m);
  return q + (n - q * d >= d ? 1 : 0);
}

// 2^x by the hardware approximation (relative error ~2^-22; -inf -> +0):
// the softmax weights need far less than that.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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

// Exclusive prefix sum over the SNT threads of the CTA (thread order); every
// thread calls it.  `scratch` holds SNW ints.
__device__ __forceinline__ int block_scan_s(int x, int* scratch, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  const int cw = lane < SNW ? scratch[lane] : 0;  // lane w: warp w's sum
  const int tot = __reduce_add_sync(0xffffffffu, cw);
  const int before = __reduce_add_sync(0xffffffffu, lane < warp ? cw : 0);
  __syncthreads();
  total = tot;
  return before + incl - x;
}

// Finds the digit holding the k_rem-th largest key in a histogram of NB bins
// (bins counted from the top).  out[0] = digit, out[1] = keys in larger
// digits, out[2] = keys in the digit.  Every thread must call it.
template <int NB>
__device__ __forceinline__ void find_digit(const uint32_t* hist, int k_rem, int* scan, int* out) {
  constexpr int M = NB / SNT;
  static_assert(M >= 1 && NB % SNT == 0, "bins per thread");
  const int tid = threadIdx.x;
  const int base = NB - (tid + 1) * M;
  int tsum = 0;
  if constexpr (M % 4 == 0) {
    const uint4* h4 = reinterpret_cast<const uint4*>(hist + base);
#pragma unroll 1
    for (int q = 0; q < M / 4; ++q) {
      const uint4 v = h4[q];
      tsum += (int)(v.x + v.y + v.z + v.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < M; ++i) tsum += (int)hist[base + i];
  }
  int total;
  int run = block_scan_s(tsum, scan, total);
  if (run < k_rem && k_rem <= run + tsum) {  // the digit is among this thread's bins
#pragma unroll 1
    for (int i = M - 1; i >= 0; --i) {
      const int ci = (int)hist[base + i];
      if (k_rem <= run + ci) {
        out[0] = base + i;
        out[1] = run;
        out[2] = ci;
        break;
      }
      run += ci;
    }
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

// The four scores at scr[tl..tl+4) as keys; ok marks those below `end`.
// tl is a multiple of 4; a group starting at or past `end` is not read (a
// sweep's last lanes would otherwise read past the CTA's scores, past the
// workspace for the last unit), and one starting below it stays inside the
// score buffer, which extends to a multiple of 4 (shared memory: the CTA's
// whole token chunk; workspace: T_max, a multiple of 64).
__device__ __forceinline__ void keys4(const float* scr, int tl, int end, uint32_t (&key)[4], bool (&ok)[4]) {
  const float4 x = tl < end ? *reinterpret_cast<const float4*>(scr + tl) : make_float4(0.f, 0.f, 0.f, 0.f);
  key[0] = score_key(x.x);
  key[1] = score_key(x.y);
  key[2] = score_key(x.z);
  key[3] = score_key(x.w);
#pragma unroll
  for (int t = 0; t < 4; ++t) ok[t] = tl + t < end;
}

// The rule that selects this CTA's top r scores (stable order) -- or, when
// the digit-0 bucket leaves at most `cap` keys at or above it, all of those
// (a longer prefix of the same order).  scr holds the CTA's nloc scores;
// hist the digit-0 histogram of their keys (rebuilt first unless hist_ok).
// Later digits (10 + 10 bits) overwrite the histogram.  Every thread calls it.
__device__ __noinline__ SelRule local_rule(int r, int cap, bool hist_ok, const float* scr, int nloc,
                                           uint32_t* hist, StepMisc* ms) {
  const int tid = threadIdx.x;
  if (r >= nloc) return SelRule{0u, INT_MAX};  // every key is >= 0
  if (!hist_ok) {
    uint4* z = reinterpret_cast<uint4*>(hist);
#pragma unroll 1
    for (int i = tid; i < HLOC_BINS / 4; i += SNT) z[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
#pragma unroll 1
    for (int tl = tid * 4; tl < nloc; tl += SNT * 4) {
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
#pragma unroll 1
  for (int dg = 1; dg <= 2; ++dg) {
    const int shift = dg == 1 ? 10 : 0;
#pragma unroll 1
    for (int i = tid; i < 1024; i += SNT) hist[i] = 0u;
    __syncthreads();
#pragma unroll 1
    for (int tl = tid * 4; tl < nloc; tl += SNT * 4) {
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
// contiguous share of the tokens, four per lane per step (lane-major token
// order, so a lane's place follows from ballots).  Returns the count (at
// most cap entries are written).  Every thread calls it.
template <bool TIES>
__device__ __forceinline__ int list_rule_t(SelRule R, const float* scr, int nloc, int t0, unsigned long long* dst,
                                           int cap, StepMisc* ms) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt = (1u << lane) - 1u;
  constexpr bool ties = TIES;
  const int wlen = (((nloc + SNW - 1) / SNW) + 3) & ~3;
  const int w0 = min(nloc, warp * wlen), w1 = min(nloc, w0 + wlen);
  int tie_base = 0;
  if constexpr (ties) {
    int c = 0;
#pragma unroll 1
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
#pragma unroll 1
    for (int w = 0; w < warp; ++w) tie_base += ms->scan2[w];
  }
  // selection flags of a lane's four tokens; tb = this CTA's ties before the
  // step, returned advanced past it
  auto flags4 = [&](int tl, int& tb, uint32_t (&key)[4], bool (&sel)[4]) {
    bool ok[4];
    keys4(scr, tl, w1, key, ok);
    if constexpr (!ties) {
#pragma unroll
      for (int t = 0; t < 4; ++t) sel[t] = ok[t] && key[t] >= R.thr;
      return;
    }
    bool tie[4];
    int rank = tb;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      tie[t] = ok[t] && key[t] == R.thr;
      const unsigned bt = __ballot_sync(0xffffffffu, tie[t]);
      rank += __popc(bt & lt);
      tb += __popc(bt);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      sel[t] = ok[t] && (key[t] > R.thr || (tie[t] && rank < R.need));
      rank += tie[t];
    }
  };
  int cnt = 0;
  {
    int tb = tie_base;
#pragma unroll 1
    for (int tl0 = w0; tl0 < w1; tl0 += 128) {
      uint32_t key[4];
      bool sel[4];
      flags4(tl0 + lane * 4, tb, key, sel);
#pragma unroll
      for (int t = 0; t < 4; ++t) cnt += sel[t];
    }
  }
  STEP_TRACE(46);
  cnt = warp_sum_i(cnt);
  if (lane == 0) ms->scan[warp] = cnt;
  __syncthreads();
  STEP_TRACE(26);
  const int cw = lane < SNW ? ms->scan[lane] : 0;  // lane w: warp w's count
  const int total = __reduce_add_sync(0xffffffffu, cw);
  int base = __reduce_add_sync(0xffffffffu, lane < warp ? cw : 0);
  STEP_TRACE(47);
  int tb = tie_base;
  uint32_t kmax = 0u;
#pragma unroll 1
  for (int tl0 = w0; tl0 < w1; tl0 += 128) {
    uint32_t key[4];
    bool sel[4];
    const int tl = tl0 + lane * 4;
    flags4(tl, tb, key, sel);
    int at = base;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const unsigned bs = __ballot_sync(0xffffffffu, sel[t]);
      at += __popc(bs & lt);
      base += __popc(bs);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (sel[t]) {
        if (at < cap)
          dst[at] = ((unsigned long long)key[t] << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)(t0 + tl + t));
        ++at;
        kmax = max(kmax, key[t]);
      }
  }
  STEP_TRACE(48);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0 && kmax) atomicMax(&ms->list_max, kmax);
  __syncthreads();
  return min(total, cap);
}

// list_rule_t<false> in one sweep: each warp writes its selected entries,
// in token order, to its own segment of `stage` (scap entries per warp),
// then copies them to dst at its offset.  Returns -1 (every thread) when a
// warp selected more than scap entries: the caller then runs the two-pass
// listing.  Every thread calls it.
__device__ __forceinline__ int list_rule_1p(SelRule R, const float* scr, int nloc, int t0, unsigned long long* dst,
                                            int cap, StepMisc* ms, unsigned long long* stage, int scap) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const int wlen = (((nloc + SNW - 1) / SNW) + 3) & ~3;
  const int w0 = min(nloc, warp * wlen), w1 = min(nloc, w0 + wlen);
  unsigned long long* seg = stage + (size_t)warp * scap;
  int wc = 0;  // the warp's entries so far
  uint32_t kmax = 0u;
#pragma unroll 1
  for (int tl0 = w0; tl0 < w1; tl0 += 128) {
    const int tl = tl0 + lane * 4;
    uint32_t key[4];
    bool ok[4];
    keys4(scr, tl, w1, key, ok);
    bool sel[4];
    int at = wc, n = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      sel[t] = ok[t] && key[t] >= R.thr;
      const unsigned bs = __ballot_sync(0xffffffffu, sel[t]);
      at += __popc(bs & lt);
      n += __popc(bs);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (sel[t]) {
        if (at < scap)
          seg[at] = ((unsigned long long)key[t] << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)(t0 + tl + t));
        ++at;
        kmax = max(kmax, key[t]);
      }
    wc += n;
  }
  STEP_TRACE(46);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    ms->scan[warp] = wc;
    if (kmax) atomicMax(&ms->list_max, kmax);
  }
  if (__syncthreads_or(wc > scap)) return -1;
  STEP_TRACE(26);
  const int cw = lane < SNW ? ms->scan[lane] : 0;  // lane w: warp w's count
  const int total = __reduce_add_sync(0xffffffffu, cw);
  const int base = __reduce_add_sync(0xffffffffu, lane < warp ? cw : 0);
#pragma unroll 1
  for (int i = lane; i < wc && base + i < cap; i += 32) dst[base + i] = seg[i];
  STEP_TRACE(48);
  __syncthreads();
  return min(total, cap);
}

// list_rule_t for any rule, out of line (ties on the threshold key, second round).
__device__ __noinline__ int list_rule_any(SelRule R, const float* scr, int nloc, int t0, unsigned long long* dst,
                                          int cap, StepMisc* ms) {
  return R.need == INT_MAX ? list_rule_t<false>(R, scr, nloc, t0, dst, cap, ms)
                           : list_rule_t<true>(R, scr, nloc, t0, dst, cap, ms);
}

// Exchange slots: slot r of a receive region holds source CTA r's list --
// a 16-byte header (int4: entries, cut short, staging unusable, -) and then
// the entries (packed u64), `stride` u64 per slot in all.
__device__ __forceinline__ int4* slot_hdr(unsigned long long* recv, int stride, int r) {
  return reinterpret_cast<int4*>(recv + (size_t)r * stride);
}
__device__ __forceinline__ const int4* slot_hdr(const unsigned long long* recv, int stride, int r) {
  return reinterpret_cast<const int4*>(recv + (size_t)r * stride);
}

// Sends this CTA's slot (header and n entries, in place locally) to every
// other CTA of the cluster with distributed-shared-memory stores, then
// arrives on every CTA's barrier (count C).  Every thread calls it.
__device__ __forceinline__ void push_list(unsigned long long* recv, int stride, int n, uint32_t bar_local,
                                          uint32_t crank, int C) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = (n + 3) >> 1;  // 16-byte vectors: the header, then two entries each
  const uint32_t slot = smem_u32(recv + (size_t)crank * stride);
  const uint4* src = reinterpret_cast<const uint4*>(recv + (size_t)crank * stride);
#pragma unroll 1
  for (int rr = warp; rr < C - 1; rr += SNW) {  // warp per destination, lanes over the vectors
    const uint32_t r = (uint32_t)(rr + (rr >= (int)crank));
#pragma unroll 1
    for (int v = lane; v < nvec; v += 32) dsmem_st_v4u32(dsmem_map(slot + v * 16, r), src[v]);
  }
  __syncthreads();
  if (tid < C) mbar_arrive_remote(dsmem_map(bar_local, (uint32_t)tid));
}

// The k-th largest value theta of the union of the C received lists (exchange
// slots of `stride` u64, slot r holding its header's count of entries, at
// most cap; values are distinct): exactly k entries are >=
// theta (the caller guarantees the union holds at least k).  The bits above
// the highest one where the union's maximum and minimum differ are common to
// every entry; the rest is resolved by 11-bit digits, most significant
// first, each a histogram in `hb` (2048 bins).  Also stores per source the
// count of its entries >= theta in ms->sel.  Every thread calls it.
__device__ __noinline__ unsigned long long union_kth(const unsigned long long* recv, int stride, int cap, int C,
                                                     int k, uint32_t* hb, StepMisc* ms) {
  constexpr int NB = 2048, DB = 11;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nslots = C * cap;
  const float inv_cap = 1.f / (float)cap;
  // slot f = r * cap + i of the flattened lists; (f + 0.5) / cap stays at
  // least 0.5 / cap away from an integer, far above the fp32 rounding error
  auto entry = [&](int f, unsigned long long& x) -> bool {
    const int r = __float2int_rz(((float)f + 0.5f) * inv_cap);
    const int i = f - r * cap;
    if (i >= slot_hdr(recv, stride, r)->x) return false;
    x = recv[(size_t)r * stride + 2 + i];
    return true;
  };
  unsigned long long mx = 0ull, mn = ~0ull;
#pragma unroll 1
  for (int f = tid; f < nslots; f += SNT) {
    unsigned long long x;
    if (entry(f, x)) {
      mx = max(mx, x);
      mn = min(mn, x);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  unsigned long long* red = reinterpret_cast<unsigned long long*>(hb);  // [SNW] maxima, [SNW] minima
  if (lane == 0) {
    red[warp] = mx;
    red[SNW + warp] = mn;
  }
  __syncthreads();
  mx = red[0];
  mn = red[SNW];
#pragma unroll
  for (int w = 1; w < SNW; ++w) {
    mx = max(mx, red[w]);
    mn = min(mn, red[SNW + w]);
  }
  __syncthreads();
  const unsigned long long diff = mx ^ mn;
  int shift = diff ? 64 - __clzll((long long)diff) : 0;  // bits below `shift` are still open
  unsigned long long prefix = shift == 64 ? 0ull : (mx >> shift);
  int k_rem = k;
  int* res = &ms->dig;
  int pass = 0;
  while (shift > 0) {
    const int nb = min(DB, shift);
    shift -= nb;
    {
      uint4* z = reinterpret_cast<uint4*>(hb);
#pragma unroll 1
      for (int i = tid; i < NB / 4; i += SNT) z[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
#pragma unroll 1
    for (int f = tid; f < nslots; f += SNT) {
      unsigned long long x;
      if (entry(f, x) && (shift + nb == 64 || (x >> (shift + nb)) == prefix))
        atomicAdd(&hb[(uint32_t)(x >> shift) & ((1u << nb) - 1u)], 1u);
    }
    __syncthreads();
    find_digit<NB>(hb, k_rem, ms->scan, res);
    ++pass;
    k_rem -= res[1];
    prefix = (prefix << nb) | (unsigned long long)res[0];
    if (res[2] == k_rem) break;
  }
  const unsigned long long theta = shift == 64 ? 0ull : (prefix << shift);
#pragma unroll 1
  for (int r = warp; r < C; r += SNW) {
    int c = 0;
#pragma unroll 1
    for (int i = lane; i < slot_hdr(recv, stride, r)->x; i += 32) c += recv[(size_t)r * stride + 2 + i] >= theta;
    c = warp_sum_i(c);
    if (lane == 0) ms->sel[r] = c;
  }
  __syncthreads();
  return theta;
}

// One warp: the bin of a 4096-bin histogram (hist; fine bin f lies in coarse
// bin f >> 6 of chist) holding the r-th largest entry, read from the 64
// coarse bins and then the 64 fine bins of the coarse bin found, one warp
// scan each.  Writes ms->dig / gt (entries in larger bins) / bucket.
// 1 <= r <= the histogram's total.
__device__ __forceinline__ void warp_find_d0(const uint32_t* hist, const uint32_t* chist, int r, StepMisc* ms) {
  const int lane = threadIdx.x & 31;
  int base = 0, above = 0;
  const uint32_t* h = chist;
#pragma unroll 1
  for (int level = 0; level < 2; ++level) {
    // lane L holds bins 63 - 2L and 62 - 2L of this level (counted from the top)
    const int ca = (int)h[63 - 2 * lane], cb = (int)h[62 - 2 * lane];
    const int sum = ca + cb;
    const int before = above + warp_excl_scan(sum, lane);
    const bool mine = before < r && r <= before + sum;
    const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    int bin = 63 - 2 * lane, gt = before, cnt = ca;
    if (r > before + ca) {
      bin -= 1;
      gt += ca;
      cnt = cb;
    }
    bin = __shfl_sync(0xffffffffu, bin, src);
    gt = __shfl_sync(0xffffffffu, gt, src);
    cnt = __shfl_sync(0xffffffffu, cnt, src);
    base = base * 64 + bin;
    above = gt;
    if (level == 1 && lane == 0) {
      ms->dig = base;
      ms->gt = gt;
      ms->bucket = cnt;
    }
    h = hist + base * 64;
  }
}

// The k-th largest value theta of the union of the C received lists
// (exchange slots of `stride` u64; a slot's header carries its count and the
// smallest and largest key it listed; values are distinct): exactly k
// entries are >= theta (the caller guarantees the union holds at least k).
// One pass bins every entry by its key's offset from the smallest key,
// shifted to at most 4096 fine bins (hb) and 64 coarse bins of 64 fine ones
// (ch); warp 0 finds the bin holding the k-th entry, coarse level first; a
// second pass counts each source's entries in higher bins and gathers that
// bin's entries, which one warp ranks; theta goes to ms->theta.  A bin of
// more than 32 entries (dense or tied keys; ms->bucket > 32 on return) is
// left to the caller's radix search.  hb, ch, ms->sel and ms->bkt_n arrive
// cleared.  Stores per source the count of its entries >= theta in ms->sel.
// Warps 0..nuw-1 call it (named barrier 4).
__device__ __forceinline__ void union_select(const unsigned long long* recv, int stride, int cap, int C, int k,
                                             uint32_t* hb, uint32_t* ch, StepMisc* ms, int nuw, int wps,
                                             float inv_wps) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;  // lane r reads source r's header
  if (lane < C) {
    const int4 hd = *slot_hdr(recv, stride, lane);
    if (hd.x > 0) {
      lo = (uint32_t)hd.z;
      hi = (uint32_t)hd.w;
    }
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  STEP_TRACE(40);
  const uint32_t span = hi - lo;  // keys lie in [lo, hi]
  const int shift = max(0, (32 - __clz((int)(span | 1u))) - 12);
  // wps warps per source (at least one): a source's entries are split over
  // its warps' lanes; warp / wps by the rounded reciprocal (exact: both
  // are at most 16)
  const int sw = __float2int_rz(((float)warp + 0.5f) * inv_wps);
  const int sl_ = (warp - sw * wps) * 32 + lane, sstride = wps * 32;
  const int sources_step = wps == 1 ? nuw : __float2int_rz(((float)nuw + 0.5f) * inv_wps);  // nuw / wps
#pragma unroll 1
  for (int r = sw; r < C; r += sources_step) {
    const unsigned long long* e = recv + (size_t)r * stride + 2;
    const int n = min(slot_hdr(recv, stride, r)->x, cap);
#pragma unroll 1
    for (int i = sl_; i < n; i += sstride) {
      const uint32_t bin = ((uint32_t)(e[i] >> 32) - lo) >> shift;
      atomicAdd(&hb[bin], 1u);
      atomicAdd(&ch[bin >> 6], 1u);
    }
  }
  STEP_TRACE(42);
  named_bar_sync(4, nuw * 32);
  STEP_TRACE(25);
  if (warp == 0) warp_find_d0(hb, ch, k, ms);
  STEP_TRACE(43);
  named_bar_sync(4, nuw * 32);
  STEP_TRACE(31);
  const uint32_t bs = (uint32_t)ms->dig;
  const int k_rem = k - ms->gt, nbk = ms->bucket;
  if (nbk > 32) return;  // (uniform) the caller runs the radix search
#pragma unroll 1
  for (int r = sw; r < C; r += sources_step) {
    const unsigned long long* e = recv + (size_t)r * stride + 2;
    const int n = min(slot_hdr(recv, stride, r)->x, cap);
    int above = 0;
#pragma unroll 1
    for (int i = sl_; i < n; i += sstride) {
      const unsigned long long x = e[i];
      const uint32_t b = ((uint32_t)(x >> 32) - lo) >> shift;
      above += b > bs;
      if (b == bs) {
        const int j = atomicAdd(&ms->bkt_n, 1);
        ms->bkt[j] = x;
        ms->bkt_src[j] = r;
      }
    }
    above = warp_sum_i(above);
    if (lane == 0 && above) atomicAdd(&ms->sel[r], above);
  }
  STEP_TRACE(44);
  named_bar_sync(4, nuw * 32);
  STEP_TRACE(6);
  if (warp == 0) {
    const unsigned long long x = lane < nbk ? ms->bkt[lane] : 0ull;  // (lanes >= nbk hold 0: never larger)
    int rank = 0;  // entries of the bin larger than x
#pragma unroll 8
    for (int i = 0; i < nbk; ++i) rank += ms->bkt[i] > x;
    if (lane < nbk) {
      if (rank == k_rem - 1) ms->theta = x;
      if (rank < k_rem) atomicAdd(&ms->sel[ms->bkt_src[lane]], 1);
    }
  }
  STEP_TRACE(45);
  named_bar_sync(4, nuw * 32);
}

// ----------------------------------------------------------- rare paths
// Out of line so that the common path's code stays short (instruction fetch,
// not arithmetic, bounds most phases of a launch this size).

// A TIP stage wait ran out: report it, and let the copies still in flight
// land before the staging is reused -- one that does not within one more
// wait bound (all stages together) is reported, and the staging is left
// alone.  One thread.
__device__ __noinline__ void tip_fail_drain(uint64_t* bars, StepMisc* ms, int ns, uint64_t wait_ns, int* status) {
  atomicOr(status, FASA_DEV_TIMEOUT);
  bool drained = true;
  const uint64_t start = global_timer_ns();
#pragma unroll 1
  for (int s = 0; s < ns; ++s)
    if (ms->tip_last[s] >= 0) {
      const uint64_t spent = global_timer_ns() - start;
      const uint64_t left = spent < wait_ns ? wait_ns - spent : 1ull;
      drained &= mbar_wait_bounded(smem_u32(&bars[s]), (uint32_t)(ms->tip_last[s] / ns) & 1u, left);
    }
  if (!drained) {
    atomicOr(status, FASA_DEV_UNDRAINED);
    ms->big_unsafe = 1;
  }
}

// Copies this CTA's nloc workspace scores (scw, written by its own threads)
// back into shared memory at dst with bulk copies, one share per warp.
// Returns false when the copy did not land in time.  Every thread calls it.
__device__ __noinline__ bool reload_scores(const float* scw, int nloc, unsigned char* dst, uint32_t rbar,
                                           uint64_t wait_ns) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nv = (nloc + 3) >> 2;
  const int per_w = (nv + SNW - 1) / SNW;
  const int v0 = min(nv, warp * per_w), v1 = min(nv, v0 + per_w);
  fence_proxy_async_global();  // this thread's score stores, before the copy reads them
  __syncthreads();
  if (lane == 0) {
    if (warp == 0) mbar_arrive_expect_tx(rbar, (uint32_t)nv * 16u);
    if (v1 > v0) bulk_g2s(smem_u32(dst) + v0 * 16, scw + v0 * 4, (uint32_t)(v1 - v0) * 16u, rbar);
  }
  return __syncthreads_and(mbar_wait_bounded(rbar, 0u, wait_ns)) != 0;
}

// F_APPEND, in the CTA that owns the new token: rotate its key (pairs kn,
// stored dtype) by position t_new, store key and value vn at index t_new of
// the caches and the key's dominant FCs in K_dom (slot row kdw), and return
// (thread 0) the token's TIP score computed exactly as the TIP loop scores a
// streamed token: same FC order and accumulation, stored precision.  With a
// split key layout (fac_pair non-null) Kw is the token's k_nondom row and
// takes only the ndp non-dominant pairs, in FC order (fac_pair[0, ndp)).
// `scratch` holds D/2 float2.  Every thread calls it.
template <int D>
__device__ __noinline__ float append_own_token(const unsigned long long* turns, __nv_bfloat162 kn, __nv_bfloat162 vn,
                                               int t_new, __nv_bfloat16* Kw, __nv_bfloat16* Vw, __nv_bfloat16* kdw,
                                               const int* dom, int nfc, const float* qbar, bool score,
                                               float2* scratch, const uint8_t* fac_pair, int ndp) {
  using T = __nv_bfloat16;
  const int tid = threadIdx.x;
  if (tid < D / 2) {
    const int i = tid;
    const float x0 = __low2float(kn), x1 = __high2float(kn);
    const float2 c = rope_cos_sin(turns[i], t_new);
    const T r0 = __float2bfloat16_rn(x0 * c.x - x1 * c.y), r1 = __float2bfloat16_rn(x0 * c.y + x1 * c.x);
    if (!fac_pair) {
      Kw[2 * i] = r0;
      Kw[2 * i + 1] = r1;
    }
    Vw[2 * i] = __low2bfloat16(vn);
    Vw[2 * i + 1] = __high2bfloat16(vn);
    scratch[i] = make_float2(__bfloat162float(r0), __bfloat162float(r1));
  }
  __syncthreads();
  if (fac_pair && tid < ndp) {
    const float2 kp = scratch[fac_pair[tid]];
    Kw[2 * tid] = __float2bfloat16_rn(kp.x);
    Kw[2 * tid + 1] = __float2bfloat16_rn(kp.y);
  }
  auto dom_at = [&](int j) { return min(max(dom[j], 0), D / 2 - 1); };
#pragma unroll 1
  for (int j = tid; j < nfc; j += SNT) {
    const float2 kp = scratch[dom_at(j)];
    kdw[(size_t)j * KDOM_BLOCK * 2] = __float2bfloat16_rn(kp.x);
    kdw[(size_t)j * KDOM_BLOCK * 2 + 1] = __float2bfloat16_rn(kp.y);
  }
  float s_new = 0.f;
  if (tid == 0 && score) {
    float a0 = 0.f, a1 = 0.f;
    auto fc_add = [&](int j, float& a) {
      const float2 kp = scratch[dom_at(j)];
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
  return s_new;
}

// The second round of the selection: every CTA sends its exact local top-k
// (their union always holds the unit's top k) and the k-th entry of the
// union is found again.  The staging that receives the lists must be idle
// in every CTA first: the gathers still in flight are drained and the
// cluster synchronises.  Returns theta; ms->sel holds the per-source counts.
// Every thread of every CTA of the cluster calls it (the decision to run it
// is taken on the same exchanged data everywhere).
__device__ __noinline__ unsigned long long second_round(int k_eff, int nloc, int t0, int cap2, const float* scr,
                                                        uint32_t* hist, unsigned long long* recv2, StepMisc* ms,
                                                        uint32_t bar_x2, uint32_t crank, int C, uint64_t xwait,
                                                        int* status) {
  const int tid = threadIdx.x;
  cp_async_wait<0>();
  __syncthreads();
  cluster_sync();
  const int stride = cap2 + 2;
  const SelRule R2 = local_rule(min(k_eff, nloc), cap2, ms->hist_clobbered == 0, scr, nloc, hist, ms);
  const int n2 = list_rule_any(R2, scr, nloc, t0, recv2 + (size_t)crank * stride + 2, cap2, ms);
  if (tid == 0) *slot_hdr(recv2, stride, crank) = make_int4(n2, nloc > n2 ? 1 : 0, 0, 0);
  __syncthreads();
  push_list(recv2, stride, n2, bar_x2, crank, C);
  if (!mbar_wait_cluster_bounded(bar_x2, 0u, xwait) && tid == 0) atomicOr(status, FASA_DEV_TIMEOUT);
  if (tid < C) slot_hdr(recv2, stride, tid)->x = min(max(slot_hdr(recv2, stride, tid)->x, 0), cap2);
  __syncthreads();
  const int total = __reduce_add_sync(0xffffffffu, (threadIdx.x & 31) < C ? slot_hdr(recv2, stride, threadIdx.x & 31)->x : 0);
  return total >= k_eff ? union_kth(recv2, stride, cap2, C, k_eff, hist, ms) : 0ull;
}

template <int D>
__global__ void __launch_bounds__(SNT, 1) fasa_step_kernel(const __grid_constant__ StepParams p) {
  using T = __nv_bfloat16;
  constexpr int ES = 2;
  constexpr int KB = KDOM_BLOCK;         // k_dom tokens per block
  constexpr int ROWB = D * ES;           // bytes of one K/V row
  constexpr int CPR = ROWB / 16;         // 16-byte chunks per row
  constexpr uint32_t FCB = KB * 2 * ES;  // one FC of one k_dom block
  constexpr uint32_t GSLOT_B = 2u * GR * ROWB;
  extern __shared__ __align__(1024) unsigned char smem[];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank();
  const int C = (int)cluster_size();
  const int unit = blockIdx.y;
  const int b = unit / p.Hkv, h = unit - b * p.Hkv;
  const int G = p.G;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  // FAC slot s of attending warp c: full (32 producer-lane arrivals, each
  // once its copies have landed) and empty (one arrival by the attending warp)
  uint64_t* fbars = reinterpret_cast<uint64_t*>(smem + p.off_fbar);
  auto fbar_full = [&](int c, int s) { return smem_u32(fbars + c * FAC_WST_MAX + s); };
  auto fbar_empty = [&](int c, int s) { return smem_u32(fbars + (FNW + c) * FAC_WST_MAX + s); };
  StepMisc* ms = reinterpret_cast<StepMisc*>(smem + p.off_misc);
  float* qrot = reinterpret_cast<float*>(smem + p.off_qrot);
  float* qbar = reinterpret_cast<float*>(smem + p.off_qbar);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + p.off_hist);
  uint32_t* uh = reinterpret_cast<uint32_t*>(smem + p.off_uh);
  float* sc_s = reinterpret_cast<float*>(smem + p.off_sc);
  unsigned long long* recv1 = reinterpret_cast<unsigned long long*>(smem + p.off_recv1);
  int* rows = reinterpret_cast<int*>(smem + p.off_rows);
  unsigned char* big = smem + p.off_big;
  const uint32_t fbase = smem_u32(smem + p.off_fac);  // the FAC group slots

  STEP_TRACE(0);
  constexpr int QW = 8;  // query warps
  constexpr int QPAIRS = (G_MAX * D / 2 + QW * 32 - 1) / (QW * 32);
  const int nfc_max = p.n_tip, tt = p.tip_tile, ns = p.tip_stages;
  const bool append = (p.flags & F_APPEND) != 0;
  // k_dom is [.., T_max/KB, n_tip, KB, 2]: a tile of whole blocks is one
  // contiguous range (one bulk copy); a head using fewer planes takes the
  // leading nfc planes of each block, packed in the stage
  const uint32_t stage_bytes = (uint32_t)(tt / KB) * nfc_max * FCB;
  const T* kd_unit = reinterpret_cast<const T*>(p.k_dom) + (size_t)unit * nfc_max * p.T_max * 2;
  // the unit's length and this CTA's range (warp 1 plans them; every thread
  // reads them after the set-up barrier)
  int len = 0, m_pos = 0, t_new = -1, t0 = 0, nloc = 0, nloc_s = 0, ntiles = 0, nfc = 1;
  bool bad = false;
  auto tip_issue = [&](int it) {  // one thread per tile; nfc is this head's count
    const int s = it < ns ? it : it % ns;
    const int tau0 = t0 + it * tt;
    const int nblk = (min(tt, t0 + nloc_s - tau0) + KB - 1) / KB;
    const uint32_t blk_bytes = (uint32_t)nfc * FCB;
    const uint32_t bar = smem_u32(&bars[s]);
    mbar_arrive_expect_tx(bar, (uint32_t)nblk * blk_bytes);
    const T* src = kd_unit + (size_t)(tau0 / KB) * nfc_max * KB * 2;
    if (it != p.drop_stage) {
      if (nfc == nfc_max) {
        bulk_g2s(smem_u32(big + s * stage_bytes), src, (uint32_t)nblk * blk_bytes, bar);
      } else {
#pragma unroll 1
        for (int bi = 0; bi < nblk; ++bi)
          bulk_g2s(smem_u32(big + s * stage_bytes + bi * blk_bytes), src + (size_t)bi * nfc_max * KB * 2, blk_bytes,
                   bar);
      }
    }
    ms->tip_last[s] = it;
  };

  // ---------------------------------------------------------------- set-up
  // Split so that the TIP copies go out as soon as the unit's length and FC
  // table are in: warp 1 loads them, plans this CTA's token range and issues
  // the copies; meanwhile warp 0 initialises the barriers and the scratch
  // (a release fence waits for its thread's loads, so warp 0 loads nothing
  // before it) and the other warps load the query and clear the histogram.
  if (warp == 0) {
    if (lane < ST_BARS && (lane < ns || lane >= ST_MAX_STAGES)) {
      // X1 and COMB complete when the C - 1 peers' bulk copies have landed
      // (their bytes are expected here, with the one local arrival); X2
      // takes one arrival per CTA
      mbar_init(smem_u32(&bars[lane]), lane == SB_X2 ? (uint32_t)C : 1u);
      fence_mbar_init();
      if (lane == SB_X1) mbar_arrive_expect_tx(smem_u32(&bars[lane]), (uint32_t)((C - 1) * (p.cap1 + 2) * 8));
      if (lane == SB_COMB) mbar_arrive_expect_tx(smem_u32(&bars[lane]), (uint32_t)((C - 1) * p.comb_slot));
    }
    if (lane < ST_MAX_STAGES) {
      ms->tip_done[lane] = 0u;
      ms->tip_last[lane] = -1;
    }
    if (lane < C_MAX) ms->sel[lane] = 0;
    ms->chist[lane] = 0u;
    ms->chist[lane + 32] = 0u;
    if (lane == 0) {
      ms->tip_fail = 0;
      ms->big_unsafe = 0;
      ms->hist_clobbered = 0;
      ms->n_rows = 0;
      ms->list_max = 0u;
    }
    STEP_TRACE(16);
    named_bar_arrive(2, 64);  // barriers and stage records ready for warp 1
  } else if (warp == 1) {
    len = p.seq_lens[b];
    m_pos = append ? 0 : p.pos[b];
    const int d0 = lane < nfc_max ? p.dom_fc[h * nfc_max + lane] : 0;
    const int d1 = lane + 32 < nfc_max ? p.dom_fc[h * nfc_max + lane + 32] : 0;
    // this head's count: the entries before the first negative one (an
    // empty set uses slot 0, reported below)
    const unsigned b0 = __ballot_sync(0xffffffffu, lane < nfc_max && d0 < 0);
    const unsigned b1 = __ballot_sync(0xffffffffu, lane + 32 < nfc_max && d1 < 0);
    nfc = max(b0 ? __ffs(b0) - 1 : (b1 ? 31 + __ffs(b1) : nfc_max), 1);
    if (len < 0 || len > p.T_max) {
      bad = true;
      len = min(max(len, 0), p.T_max);
    }
    // F_APPEND: the step's own token goes to index t_new = len, the query
    // sits at that position, and the step attends len + 1 tokens (a full
    // cache cannot take the token: reported, not appended)
    if (append) {
      m_pos = len;
      if (len < p.T_max) {
        t_new = len;
        len += 1;
      } else {
        bad = true;
      }
    }
    // contiguous token range of this CTA, its start aligned to a k_dom
    // block; K_dom is streamed up to the new token, which its CTA scores
    // from registers
    const int chunk = (div_magic(len + C - 1, C, p.c_magic) + KB - 1) / KB * KB;
    t0 = min(len, (int)crank * chunk);
    nloc = min(len, t0 + chunk) - t0;
    nloc_s = t_new >= t0 && t_new < t0 + nloc ? t_new - t0 : nloc;
    ntiles = len > p.budget ? div_magic(nloc_s + tt - 1, tt, p.tt_magic) : 0;
    STEP_TRACE(20);
    if (lane == 0) {
      StepHdr& hd = ms->hdr;
      hd.len = len;
      hd.m_pos = m_pos;
      hd.t_new = t_new;
      hd.bad = bad;
      hd.t0 = t0;
      hd.nloc = nloc;
      hd.nloc_s = nloc_s;
      hd.ntiles = ntiles;
      hd.nfc = nfc;
    }
    named_bar_sync(2, 64);
    STEP_TRACE(21);
    if (lane < min(ns, ntiles)) tip_issue(lane);  // one stage per lane
    STEP_TRACE(13);
  }
  // Warps 2..9 (the query warps) rotate the G query heads and form q-bar
  // while warp 1 waits for the length and issues the copies: that code runs
  // before the TIP data streams into the SM (instruction fetches compete
  // with it).  Each query warp copies its share of the RoPE table to shared
  // memory first (per-thread indices into kernel parameters serialize
  // within a warp).
  unsigned long long* turns = reinterpret_cast<unsigned long long*>(uh);  // [D/2]
  if (warp >= 2 && warp < 2 + QW) {
    const int qt = tid - 64;
    const int l0 = p.seq_lens[b];
    const int mp = append ? min(max(l0, 0), p.T_max) : p.pos[b];
    T qv0[QPAIRS], qv1[QPAIRS];
#pragma unroll
    for (int k = 0; k < QPAIRS; ++k) {
      const int x = qt + k * QW * 32;
      qv0[k] = qv1[k] = T(0.f);
      if (x < G * (D / 2)) {
        const T* qg = reinterpret_cast<const T*>(p.q) + ((size_t)b * p.Hq + (size_t)h * G) * D + 2 * x;
        qv0[k] = qg[0];
        qv1[k] = qg[1];
      }
    }
    // q-bar threads: entry qt of the FC table, and (warps 2, 3) the count
    const int dq = qt < nfc_max ? p.dom_fc[h * nfc_max + qt] : 0;
    constexpr int TPQ = D / 2 / QW;
    static_assert(TPQ >= 1 && TPQ * QW == D / 2, "RoPE table share per query warp");
    if (lane < TPQ) turns[(warp - 2) * TPQ + lane] = p.rope_turns[(warp - 2) * TPQ + lane];
    // F_KSPLIT: the FAC key rows' pair order, needed for the query fragments
    if ((p.flags & F_KSPLIT) && warp == 2)
      bad = !split_pairs(p.dom_fc + h * nfc_max, nfc_max, D / 2, ms->fac_pair) || bad;
    named_bar_sync(3, QW * 32);  // the table is complete
#pragma unroll 1
    for (int k = 0; k < QPAIRS; ++k) {
      const int x = qt + k * QW * 32;
      if (x < G * (D / 2)) {
        const int i = x & (D / 2 - 1);
        const float2 c = rope_cos_sin(turns[i], mp);
        const float x0 = __bfloat162float(qv0[k]), x1 = __bfloat162float(qv1[k]);
        *reinterpret_cast<float2*>(&qrot[2 * x]) = make_float2(x0 * c.x - x1 * c.y, x0 * c.y + x1 * c.x);
      }
    }
    STEP_TRACE(22);
    named_bar_sync(3, QW * 32);  // the rotated query is complete
    if (warp < 4) {  // q-bar: the group sum of the rotated query on the dominant FCs
      const int e0 = lane < nfc_max ? p.dom_fc[h * nfc_max + lane] : 0;
      const int e1 = lane + 32 < nfc_max ? p.dom_fc[h * nfc_max + lane + 32] : 0;
      const unsigned b0 = __ballot_sync(0xffffffffu, lane < nfc_max && e0 < 0);
      const unsigned b1 = __ballot_sync(0xffffffffu, lane + 32 < nfc_max && e1 < 0);
      const int nq = max(b0 ? __ffs(b0) - 1 : (b1 ? 31 + __ffs(b1) : nfc_max), 1);
      if (qt < nq) {
        int i = dq;
        if (i < 0 || i >= D / 2) {
          bad = true;
          i = min(max(i, 0), D / 2 - 1);
        }
        float a0 = 0.f, a1 = 0.f;
        for (int g = 0; g < G; ++g) {
          a0 += qrot[g * D + 2 * i];
          a1 += qrot[g * D + 2 * i + 1];
        }
        qbar[2 * qt] = a0;
        qbar[2 * qt + 1] = a1;
      }
    }
    // The FAC's query operand, built here once and stored over the rotated
    // query (the same 4 KB): lane (gq, tq) of an attending warp needs, per
    // 16-column k-step ks, the log2(e)/sqrt(d)-scaled pairs at columns 2tq
    // and 2tq + 8 (in the key rows' pair order) of head gq, each split into
    // bf16 hi + lo.  Item (ks, lane) is one uint4 at [ks][lane].
    {
      constexpr int KSQ = D / 16;
      static_assert(KSQ <= QW && KSQ * 32 * 16 <= G_MAX * D * 4, "query fragments: one item per query thread, "
                                                                   "within the rotated query's bytes");
      const float qs = 1.4426950408889634f * rsqrtf((float)D);
      const int ks = qt >> 5, ln = qt & 31, gq = ln >> 2, tq = ln & 3;
      uint32_t v[4] = {0u, 0u, 0u, 0u};
      if (ks < KSQ) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int d0 = ks * 16 + 2 * tq + hb * 8;
          const int ds = (p.flags & F_KSPLIT) ? 2 * ms->fac_pair[d0 >> 1] : d0;
          const float x0 = gq < G ? qrot[gq * D + ds] * qs : 0.f;
          const float x1 = gq < G ? qrot[gq * D + ds + 1] * qs : 0.f;
          split_bf16(x0, x1, v[2 * hb], v[2 * hb + 1]);
        }
      }
      named_bar_sync(3, QW * 32);  // every read of the rotated query is done
      if (ks < KSQ) reinterpret_cast<uint4*>(qrot)[ks * 32 + ln] = make_uint4(v[0], v[1], v[2], v[3]);
    }
    STEP_TRACE(17);
  }
  __nv_bfloat162 kn = __float2bfloat162_rn(0.f), vn = kn;
  if (append && tid < D / 2) {  // (element-aligned inputs: two 2-byte loads each)
    const T* knp = reinterpret_cast<const T*>(p.k_new) + (size_t)unit * D + 2 * tid;
    const T* vnp = reinterpret_cast<const T*>(p.v_new) + (size_t)unit * D + 2 * tid;
    kn = __halves2bfloat162(knp[0], knp[1]);
    vn = __halves2bfloat162(vnp[0], vnp[1]);
  }
  if (warp == SNW - 1) {  // (idle in the set-up) the FAC slots' barriers
#pragma unroll 1
    for (int i = lane; i < 2 * FNW * FAC_WST_MAX; i += 32) mbar_init(smem_u32(fbars + i), i < FNW * FAC_WST_MAX ? 32u : 1u);
    fence_mbar_init();
  }
  {
    uint4* z = reinterpret_cast<uint4*>(hist);
    for (int i = tid; i < HLOC_BINS / 4; i += SNT) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  STEP_TRACE(19);
  // The barrier inits were fenced at cluster scope above; the matching wait
  // (after TIP) comes before any peer touches this CTA's shared memory.  A
  // relaxed arrive does not wait for this thread's loads still in flight.
  cluster_arrive_relaxed();
  __syncthreads();
  STEP_TRACE(12);
  {
    const StepHdr& hd = ms->hdr;
    len = hd.len;
    m_pos = hd.m_pos;
    t_new = hd.t_new;
    bad = bad || hd.bad != 0;
    t0 = hd.t0;
    nloc = hd.nloc;
    nloc_s = hd.nloc_s;
    ntiles = hd.ntiles;
    nfc = hd.nfc;
  }
  const int k_eff = min(p.budget, len);
  const bool need_select = len > p.budget;
  const int t1 = t0 + nloc;
  const bool own_new = t_new >= t0 && t_new < t1;

  float s_new = 0.f;
  if (own_new) {  // (uh: the RoPE table, then this scratch)
    // a split key layout keeps ndp = D/2 - nfc_max pairs per k_nondom row
    const bool ksplit_w = (p.flags & F_KSPLIT) != 0;
    const int krow = ksplit_w ? D - 2 * nfc_max : D;
    s_new = append_own_token<D>(turns, kn, vn, t_new,
                                const_cast<T*>(reinterpret_cast<const T*>(p.k_cache)) + ((size_t)unit * p.T_max + t_new) * krow,
                                const_cast<T*>(reinterpret_cast<const T*>(p.v_cache)) + ((size_t)unit * p.T_max + t_new) * D,
                                const_cast<T*>(kd_unit) + ((size_t)(t_new / KB) * nfc_max * KB + (t_new % KB)) * 2,
                                p.dom_fc + h * nfc_max, nfc, qbar, need_select,
                                reinterpret_cast<float2*>(uh) + D / 2, ksplit_w ? ms->fac_pair : nullptr,
                                D / 2 - nfc_max);
  }
  STEP_TRACE(1);

  // ---------------------------------------------------------------- TIP scan
  // Warp w scores the 128-token units w, w + W, ... (W = p.tip_warps); a unit lies in one
  // stage.  In a refilled ring each unit's warp counts itself done with the
  // stage, and the warp that completes the stage refills it.  A wait that
  // runs out stops the warp and, through ms->tip_fail, the others.
  float* scw = p.s_cap > 0 ? sc_s : p.scores + (size_t)unit * p.T_max + t0;
  if (own_new && need_select && tid == 0) {  // the appended token's score, as TIP would
    scw[nloc_s] = s_new;
    const uint32_t key = score_key(s_new);
    atomicAdd(&hist[key >> 20], 1u);
    atomicAdd(&ms->chist[key >> 26], 1u);
  }
  const int upt = tt / TIP_UNIT;
  const int nunits = ntiles > 0 ? (nloc_s + TIP_UNIT - 1) / TIP_UNIT : 0;
  const bool ring = ntiles > ns;
  const uint32_t blk_bytes = (uint32_t)nfc * FCB;
  int tip_fail = 0;
  const int tip_stride = p.tip_warps;
  for (int u = warp; warp < tip_stride && u < nunits; u += tip_stride) {  // (warps >= tip_warps score nothing)
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
      if (tl + t < nloc_s) {
        const uint32_t key = score_key(acc[t]);
        atomicAdd(&hist[key >> 20], 1u);
        atomicAdd(&ms->chist[key >> 26], 1u);
      }
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
    if (tid == 0) tip_fail_drain(bars, ms, ns, p.wait_ns, p.status);
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
  bool second = false;  // the second exchange decided the selection
  int sel_before = 0;   // selected tokens of the lower-ranked CTAs
  const bool spec = p.spec != 0 && big_ok;
  // F_KSPLIT: k_cache holds the keys' non-dominant pairs (ndp per token)
  const bool ksplit = (p.flags & F_KSPLIT) != 0;
  const int ndp = D / 2 - nfc_max;
  const T* Kb = reinterpret_cast<const T*>(p.k_cache) + (size_t)unit * p.T_max * (ksplit ? 2 * ndp : D);
  const T* Vb = reinterpret_cast<const T*>(p.v_cache) + (size_t)unit * p.T_max * D;
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
  // Row gathers: a warp copies RPI rows per instruction, lane l the 16-byte
  // chunk l % (2 CPR) of its row's K (the first CPR) then V, into the row's
  // group slot: group g belongs to warp g % FNW, its slot (g / FNW) mod
  // fac_wst (the slots are reused in turn); chunk c of a row sits at chunk
  // position c ^ (row & 7) so the eight rows an ldmatrix reads fall in
  // distinct banks.  Rows past fr_n are zero-filled: the tensor cores
  // multiply them by zero weights, which must not meet stale NaNs.
  constexpr int LPR = 2 * CPR;   // lanes per row
  constexpr int RPI = 32 / LPR;  // rows per warp instruction
  static_assert(RPI >= 1 && RPI * LPR == 32 && GR % RPI == 0, "row gather lanes");
  const int g_sub = lane / LPR, g_cc = lane - g_sub * LPR;
  const int g_kv = g_cc >= CPR ? 1 : 0, g_ch = g_cc - g_kv * CPR;
  auto row_copy = [&](int i) {  // this lane's chunk of row i
    const int g = i / GR, rr = i & (GR - 1);
    const uint32_t dst = fbase + (uint32_t)((g % FNW) * p.fac_wst + (g / FNW) % p.fac_wst) * GSLOT_B +
                         (uint32_t)(g_kv * GR + rr) * ROWB + (uint32_t)((g_ch ^ (rr & 7)) << 4);
    const bool real = i < fr_n;
    const int tok = real ? row_token(i) : 0;
    if (ksplit && !g_kv)
      split_key_chunk(dst, Kb, kd_unit, ndp, nfc_max, tok, g_ch, real);
    else
      cp_async16_zfill(dst, (g_kv ? Vb : Kb) + (size_t)tok * D + g_ch * (16 / ES), real ? 16u : 0u);
  };
  // the first fac_wst groups of every FAC warp, by warps w, w + 1, .. (nw
  // of them), RPI rows per warp and step
  auto fac_start = [&](int w, int nw) {
    const int nfirst = min((fr_n + GR - 1) / GR * GR, p.fac_wst * FNW * GR);
#pragma unroll 1
    for (int i0 = w * RPI; i0 < nfirst; i0 += nw * RPI) row_copy(i0 + g_sub);
    cp_async_commit();
  };
  // Resident FAC (p.rfac): the scores of resident group g (its slot as
  // row_copy places it; every group of the list is resident at once) on the
  // tensor cores, S^T = K Q^T as in the FAC below, stored unmasked (log2
  // units) as s_rows[head][row], row stride srs.  One warp.
  float* s_rows = reinterpret_cast<float*>(smem + p.off_pt);
  const int srs = p.cap1 + 8;
  auto qk_group = [&](int g) {
    constexpr int KSG = D / 16;
    const int gq = lane >> 2, tq = lane & 3, mi = lane >> 3;
    const uint32_t k_row = ((lane & 7) + 8 * (mi & 1)) * ROWB;
    const int k_c = mi >> 1, sw = lane & 7;
    const uint32_t Ks = fbase + (uint32_t)((g % FNW) * p.fac_wst + g / FNW) * GSLOT_B;
    float sh[4] = {0.f, 0.f, 0.f, 0.f}, slo[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KSG; ++ks) {
      const uint4 f = reinterpret_cast<const uint4*>(qrot)[ks * 32 + lane];
      uint32_t a0, a1, a2, a3;
      ldsm_x4(Ks + k_row + (((2 * ks + k_c) ^ sw) << 4), a0, a1, a2, a3);
      mma_bf16_16816(sh, a0, a1, a2, a3, f.x, f.z);
      mma_bf16_16816(slo, a0, a1, a2, a3, f.y, f.w);
    }
    const int r = g * GR + gq;
    s_rows[(2 * tq) * srs + r] = sh[0] + slo[0];
    s_rows[(2 * tq + 1) * srs + r] = sh[1] + slo[1];
    s_rows[(2 * tq) * srs + r + 8] = sh[2] + slo[2];
    s_rows[(2 * tq + 1) * srs + r + 8] = sh[3] + slo[3];
  };

  if (need_select) {
    // the sweeps read shared memory: scores kept there, or workspace scores
    // copied back into the idle staging
    const float* scr = p.s_cap > 0 ? sc_s : scw;
    if (p.reload && big_ok) {
      if (reload_scores(scw, nloc, big, smem_u32(&bars[SB_RELOAD]), p.wait_ns)) scr = reinterpret_cast<const float*>(big);
      else if (tid == 0) atomicOr(p.status, FASA_DEV_TIMEOUT);
    }
    // First round: the own top-rho list (or the whole digit-0 bucket at the
    // threshold when that fits), sent to every CTA
    const int r1 = min(p.rho, nloc);
    const int stride1 = p.cap1 + 2;
    unsigned long long* own1 = recv1 + (size_t)crank * stride1;
    SelRule R1{0u, INT_MAX};
    if (r1 < nloc) {
      if (warp == 0) warp_find_d0(hist, ms->chist, r1, ms);
      __syncthreads();
      STEP_TRACE(23);
      R1.thr = (uint32_t)ms->dig << 20;
      if (ms->gt + ms->bucket > p.cap1) R1 = local_rule(r1, p.cap1, true, scr, nloc, hist, ms);
    }
    STEP_TRACE(14);
    // one sweep into per-warp segments of the idle staging when it is free
    // (scores not reloaded there) and a segment holds at least twice a
    // warp's share of the list, else (or when a warp's entries overflow its
    // segment) the two-pass listing
    n1 = -1;
    const int scap = min(p.cap1, (p.smem_total - p.off_big) / (SNW * 8));
    if (R1.need == INT_MAX && !p.reload && big_ok && scap >= max(64, 2 * p.cap1 / SNW))
      n1 = list_rule_1p(R1, scr, nloc, t0, own1 + 2, p.cap1, ms, reinterpret_cast<unsigned long long*>(big), scap);
    if (n1 < 0)
      n1 = R1.need == INT_MAX ? list_rule_t<false>(R1, scr, nloc, t0, own1 + 2, p.cap1, ms)
                              : list_rule_any(R1, scr, nloc, t0, own1 + 2, p.cap1, ms);
    STEP_TRACE(3);
    // the own slot goes to every peer as one bulk copy, completing on the
    // peer's first-exchange barrier
    // header: count, cut short, staging unusable, smallest and largest key
    // listed (every listed key is >= the rule's threshold)
    if (tid == 0)
      *slot_hdr(recv1, stride1, crank) =
          make_int4(n1, (nloc > n1 ? 1 : 0) | (big_ok ? 0 : 2), (int)R1.thr, (int)ms->list_max);
    fence_proxy_async();  // the slot's generic writes, before the async proxy reads them
    __syncthreads();
    if (lane == 0 && warp < C && warp != (int)crank)  // warp r sends to CTA r
      bulk_s2cluster(dsmem_map(smem_u32(own1), (uint32_t)warp), smem_u32(own1), (uint32_t)stride1 * 8u,
                     dsmem_map(smem_u32(&bars[SB_X1]), (uint32_t)warp));
    STEP_TRACE(24);
    // While the lists travel, the listed rows are gathered (the selection
    // only masks them): by the warps past the first C when at least four
    // are left over -- the union select then runs on warps 0..C-1 alone --
    // else by every warp before the wait.
    if (spec) {
      fslot = own1 + 2;
      contig = false;
      fr_n = n1;
    }
    const int nuw = p.u_nuw;  // warps of the union select
    if (spec && nuw == SNW) fac_start(warp, SNW);
    if (warp < nuw) {
      // clear the union's histograms (the local one is spent; a second
      // round rebuilds it)
      uint4* z = reinterpret_cast<uint4*>(hist);
      for (int i = tid; i < HLOC_BINS / 4; i += nuw * 32) z[i] = make_uint4(0u, 0u, 0u, 0u);
      if (warp == 0) {
        ms->chist[lane] = 0u;
        ms->chist[lane + 32] = 0u;
        if (lane < C_MAX) ms->sel[lane] = 0;
        if (lane == 0) {
          ms->bkt_n = 0;
          ms->hist_clobbered = 1;
        }
      }
      STEP_TRACE(27);
      if (!mbar_wait_cluster_bounded(smem_u32(&bars[SB_X1]), 0u, xwait) && tid == 0)
        atomicOr(p.status, FASA_DEV_TIMEOUT);
      STEP_TRACE(4);
      // (only a timed-out wait leaves a stale count; the own slot may still
      // be read by the outgoing copies and is left alone)
      if (tid < C && tid != (int)crank)
        slot_hdr(recv1, stride1, tid)->x = min(max(slot_hdr(recv1, stride1, tid)->x, 0), p.cap1);
      named_bar_sync(4, nuw * 32);
      STEP_TRACE(30);
      const int total = __reduce_add_sync(0xffffffffu, lane < C ? slot_hdr(recv1, stride1, lane)->x : 0);
      if (total >= k_eff) union_select(recv1, stride1, p.cap1, C, k_eff, hist, ms->chist, ms, nuw, p.u_wps, p.u_inv_wps);
    } else {
      fac_start(warp - nuw, SNW - nuw);
      if (spec && p.rfac) {  // the listed rows' scores, once these warps' copies have landed
        cp_async_wait<0>();
        named_bar_sync(5, (SNW - nuw) * 32);
        STEP_TRACE(32);
#pragma unroll 1
        for (int g = warp - nuw; g < (fr_n + GR - 1) / GR; g += SNW - nuw) qk_group(g);
        STEP_TRACE(33);
      }
    }
    __syncthreads();
    // lane r reads source r's header (every warp, so the result is everywhere)
    const int4 hd = lane < C ? *slot_hdr(recv1, stride1, lane) : make_int4(0, 0, 0, 0);
    const int total = __reduce_add_sync(0xffffffffu, hd.x);
    const bool any_unsafe = __any_sync(0xffffffffu, (hd.y & 2) != 0);
    bool valid = total >= k_eff;
    if (valid) {
      // a threshold bin of more than 32 entries (dense or tied keys): the
      // radix search over the union, by every warp
      theta = ms->bucket > 32 ? union_kth(recv1, stride1, p.cap1, C, k_eff, hist, ms) : ms->theta;
      // a source that cut its list short (and sent fewer than k) with every
      // entry selected could have left out a selected token
      const int selr = lane < C ? ms->sel[lane] : 0;
      valid = !__any_sync(0xffffffffu, (hd.y & 1) && hd.x < k_eff && selr == hd.x);
    }
    STEP_TRACE(5);
    if (!valid && !any_unsafe) {
      second = true;
      theta = second_round(k_eff, nloc, t0, p.cap2, p.s_cap > 0 ? sc_s : scw, hist,
                           reinterpret_cast<unsigned long long*>(smem + p.off_recv2), ms, smem_u32(&bars[SB_X2]),
                           crank, C, xwait, p.status);
      STEP_TRACE(6);
    }
    sel_before = __reduce_add_sync(0xffffffffu, lane < (int)crank ? ms->sel[lane] : 0);
    // The own selection, compact and in token order (the own list is in
    // token order), for the gather when the first round's rows were not
    // gathered already and for the index output: warp w takes a contiguous
    // share of the list.
    if (!spec || second || p.idx_out) {
      const unsigned long long* recv2 = reinterpret_cast<const unsigned long long*>(smem + p.off_recv2);
      const unsigned long long* own = second ? recv2 + (size_t)crank * (p.cap2 + 2) + 2 : own1 + 2;
      const int n_own = second ? slot_hdr(recv2, p.cap2 + 2, crank)->x : n1;
      const int per_w = (n_own + SNW - 1) / SNW;
      const int e0 = min(n_own, warp * per_w), e1 = min(n_own, e0 + per_w);
      int c = 0;
#pragma unroll 1
      for (int e = e0 + lane; e < e1; e += 32) c += own[e] >= theta;
      c = warp_sum_i(c);
      if (lane == 0) ms->scan2[warp] = c;
      __syncthreads();
      const int cw = lane < SNW ? ms->scan2[lane] : 0;  // lane w: warp w's count
      const int n_sel = __reduce_add_sync(0xffffffffu, cw);
      int at = __reduce_add_sync(0xffffffffu, lane < warp ? cw : 0);
#pragma unroll 1
      for (int e0b = e0; e0b < e1; e0b += 32) {
        const int e = e0b + lane;
        const bool sl = e < e1 && own[e] >= theta;
        const unsigned bal = __ballot_sync(0xffffffffu, sl);
        const int pos = at + __popc(bal & ((1u << lane) - 1u));
        if (sl && pos < p.rows_cap) rows[pos] = (int)(0xFFFFFFFFu - (uint32_t)own[e]);
        at += __popc(bal);
      }
      if (tid == 0) ms->n_rows = min(n_sel, p.rows_cap);
      __syncthreads();
    }
    if (!spec || second) {
      fslot = nullptr;
      contig = false;
      fr_n = ms->n_rows;
      if (big_ok) fac_start(warp, SNW);
    }
  } else {
    // every cached token is attended: rows split evenly over the cluster.
    // An appended row may be gathered by another CTA: the barrier orders its
    // owner's stores before the gathers.
    if (t_new >= 0) cluster_sync();
    fr_r0 = (k_eff * (int)crank) / C;
    fr_n = (k_eff * ((int)crank + 1)) / C - fr_r0;
    contig = true;
    if (big_ok) fac_start(warp, SNW);
  }
  if (!big_ok) fr_n = 0;  // nothing was gathered: an empty record
  STEP_TRACE(7);

  // ---------------------------------------------------------------- FAC
  // The combine staging: the G*D outputs are cut into C slices of sl float4
  // groups (the last one shorter); slice r with (m, l) of every head goes to
  // slot r of the staging (CTA r's share; this CTA's own share into its
  // receive slot), each slot then one bulk copy to CTA r, which finishes
  // slice r.
  const int ngrp4 = G * (D / 4);
  const int sl = p.comb_sl;  // ceil(ngrp4 / C)
  const int cs = p.comb_slot;  // bytes: sl float4, then G (m, l) float2 (padded)
  const float inv_sl = p.comb_inv_sl;
  unsigned char* crcv = smem + p.off_comb;      // [C][cs], slot r from CTA r
  unsigned char* csnd = smem + p.off_comb_snd;  // [C][cs], slot r for CTA r
  auto stage_out = [&](int g, int e, float val) {  // output element (head g, dim e)
    const int q = g * (D / 4) + (e >> 2);
    const int r = __float2int_rz(((float)q + 0.5f) * inv_sl);  // q / sl, exact for these sizes
    unsigned char* dst = (r == (int)crank ? crcv : csnd) + r * cs;
    *reinterpret_cast<float*>(dst + (q - r * sl) * 16 + (e & 3) * 4) = val;
  };
  if (spec && p.rfac && need_select && !second) {
    // Resident FAC: every row of the own first-round list sits in its slot
    // and its scores are in s_rows (taken by the gather warps during the
    // selection, or now).  Warp w < D/16 takes head dims 16w..16w+15 of
    // every head: it compacts the list's entries at or above theta, takes
    // each head's maximum M over them, and attends those rows only, 16 per
    // step -- lane (gq, tq) reads the scores of head gq at the step's rows
    // 2tq, 2tq+1, 2tq+8, 2tq+9 and forms P = exp2(s - M), and the warp
    // computes O^T = V^T P^T on the tensor cores (ldmatrix rows gathered by
    // index, P split into bf16 hi + lo).  M and L = sum P come out the same
    // in every warp.  The warp's slice of the CTA's (M, L, acc) record goes
    // straight into the combine slots: no per-warp records to merge.
    constexpr int KS = D / 16;
    const int ngrp = (fr_n + GR - 1) / GR;
    if (p.u_nuw == SNW) {  // (uniform) every warp gathered: the scores now
      cp_async_wait<0>();
      __syncthreads();
#pragma unroll 1
      for (int g = warp; g < ngrp; g += SNW) qk_group(g);
      __syncthreads();
    }
    if (warp < KS) {
      // Every attending warp compacts the selected entries of the list (key
      // >= theta, in list order) into its own index array sp and takes each
      // head's maximum M over them (each warp on its own: one warp doing it
      // for all and a barrier measured slower).
      uint16_t* sp = reinterpret_cast<uint16_t*>(s_rows + G_MAX * srs) + warp * p.cap1;
      const int gq = lane >> 2, tq = lane & 3, mt = warp;
      float mx[G_MAX];
#pragma unroll
      for (int h = 0; h < G_MAX; ++h) mx[h] = -CUDART_INF_F;
      int n_sel = 0;
#pragma unroll 1
      for (int e0 = 0; e0 < fr_n; e0 += 32) {
        const int e = e0 + lane;
        const bool v = e < fr_n && fslot[e] >= theta;
        const unsigned bal = __ballot_sync(0xffffffffu, v);
        if (v) {
#pragma unroll
          for (int h = 0; h < G_MAX; ++h)
            if (h < G) mx[h] = fmaxf(mx[h], s_rows[h * srs + e]);
          sp[n_sel + __popc(bal & ((1u << lane) - 1u))] = (uint16_t)e;
        }
        n_sel += __popc(bal);
      }
      // head gq's maximum over the warp (order-preserving unsigned keys)
      float M = 0.f;
#pragma unroll
      for (int h = 0; h < G_MAX; ++h) {
        uint32_t u = __float_as_uint(mx[h]);
        u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
        u = __reduce_max_sync(0xffffffffu, u);
        if (gq == h && h < G) M = __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
      }
      __syncwarp();
      const float* Sh = s_rows + gq * srs;
      auto row_at = [&](int ci) { return (int)sp[ci < n_sel ? ci : 0]; };
      // ldmatrix (transposed) of V: lane gives row vr of matrix (lane >> 3),
      // chunk 2 mt + v_c; the row's chunk sits at c ^ (slot row & 7).
      // Selected rows past n_sel: a real row with weight 0.
      const int vr = (lane & 7) + 8 * ((lane >> 3) >> 1), v_c = (lane >> 3) & 1;
      const int ngs = (n_sel + GR - 1) / GR;
      float L = 0.f, oc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int vg = 0; vg < ngs; ++vg) {
        const int c0 = vg * GR + 2 * tq;
        const float p0 = c0 < n_sel ? ex2_approx(Sh[row_at(c0)] - M) : 0.f;
        const float p1 = c0 + 1 < n_sel ? ex2_approx(Sh[row_at(c0 + 1)] - M) : 0.f;
        const float p2 = c0 + 8 < n_sel ? ex2_approx(Sh[row_at(c0 + 8)] - M) : 0.f;
        const float p3 = c0 + 9 < n_sel ? ex2_approx(Sh[row_at(c0 + 9)] - M) : 0.f;
        L += (p0 + p1) + (p2 + p3);
        uint32_t b0h, b0l, b1h, b1l;
        split_bf16(p0, p1, b0h, b0l);
        split_bf16(p2, p3, b1h, b1l);
        const int pr = row_at(vg * GR + vr);
        const int pg = pr / GR, rr = pr & (GR - 1);
        const uint32_t va = fbase + (uint32_t)((pg % FNW) * p.fac_wst + pg / FNW) * GSLOT_B +
                            (uint32_t)(GR + rr) * ROWB + (uint32_t)(((2 * mt + v_c) ^ (rr & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(va, a0, a1, a2, a3);
        mma_bf16_16816(oc, a0, a1, a2, a3, b0h, b1h);
        mma_bf16_16816(oc, a0, a1, a2, a3, b0l, b1l);
      }
      L += __shfl_xor_sync(0xffffffffu, L, 1);
      L += __shfl_xor_sync(0xffffffffu, L, 2);
      STEP_TRACE(36);
      // oc: head dims 16 mt + gq (+ 8) x heads 2tq, 2tq + 1
      if (2 * tq < G) {
        stage_out(2 * tq, mt * 16 + gq, oc[0]);
        stage_out(2 * tq, mt * 16 + gq + 8, oc[2]);
      }
      if (2 * tq + 1 < G) {
        stage_out(2 * tq + 1, mt * 16 + gq, oc[1]);
        stage_out(2 * tq + 1, mt * 16 + gq + 8, oc[3]);
      }
      // every head's (M, L) into each slot: warp w the slots w, w + D/16, ..
      if (tq == 0 && gq < G)
#pragma unroll 1
        for (int r = warp; r < C; r += KS)
          *reinterpret_cast<float2*>((r == (int)crank ? crcv : csnd) + r * cs + sl * 16 + gq * 8) = make_float2(M, L);
    }
    STEP_TRACE(8);
  } else {
    // Tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate), one
    // flash-decoding pass per warp over its own 16-row groups: QK as
    // S^T = K Q^T (16 rows x 8 heads), PV as O^T = V^T P^T (16 head dims x 8
    // heads per MMA).  q and the softmax weights P are split into bf16 hi + lo
    // parts, so the products keep ~16 mantissa bits.  Lane (gq, tq) holds rows
    // gq, gq + 8 of S^T and head dims gq, gq + 8 of O^T, heads 2tq, 2tq + 1.
    //
    // The first fac_wst groups of every attending warp come from the CTA-wide
    // first issue.  Rows gathered after the selection (no first-round list in
    // the slots): warp FNW + c is the producer of attending warp c's later
    // groups -- it refills c's slots in turn, each once c has released it
    // (empty), and arms the slot's full barrier with its lanes' completion
    // arrivals.  Otherwise (the listed rows) each attending warp refills its
    // own slots.
    constexpr int KS = D / 16;
    const int ngrp = (fr_n + GR - 1) / GR;
    const int nrec = min(FNW, ngrp);  // warps that attend rows
    const bool pc = fslot == nullptr;  // (uniform)
    float* rec = reinterpret_cast<float*>(big);  // [G][FNW][D + 2]
    cp_async_wait<0>();  // the CTA-wide first groups
    __syncthreads();
    if (pc && warp >= FNW) {
      const int c = warp - FNW, wst = p.fac_wst;
      int it = wst;
#pragma unroll 1
      for (int g = c + wst * FNW; g < ngrp; g += FNW, ++it) {
        const int s = it % wst, n = it / wst;  // use n >= 1 of slot s
        if (!mbar_wait_bounded(fbar_empty(c, s), (uint32_t)(n - 1) & 1u, p.wait_ns)) {
          atomicOr(p.status, FASA_DEV_TIMEOUT);
          break;
        }
#pragma unroll 4
        for (int r = 0; r < GR; r += RPI) row_copy(g * GR + r + g_sub);
        if (c != 0 || it - wst != p.drop_refill)  // (test hook: a withheld completion report)
          cp_async_mbar_arrive(fbar_full(c, s));
      }
      cp_async_wait<0>();
    } else if (warp < nrec) {
      const int gq = lane >> 2, tq = lane & 3;
      uint32_t qb[KS][2][2];  // [k-step][b0 / b1][hi / lo], built in the set-up
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint4 f = reinterpret_cast<const uint4*>(qrot)[ks * 32 + lane];
        qb[ks][0][0] = f.x;
        qb[ks][0][1] = f.y;
        qb[ks][1][0] = f.z;
        qb[ks][1][1] = f.w;
      }
      float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F;  // running max (log2 units), heads 2tq, 2tq + 1
      float l0 = 0.f, l1 = 0.f;
      float oc[KS][4];
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) oc[mt][0] = oc[mt][1] = oc[mt][2] = oc[mt][3] = 0.f;
      float* pt = reinterpret_cast<float*>(smem + p.off_pt) + warp * (G * PTS);  // [head < G][PTS]
      const int mi = lane >> 3;
      const int kr = (lane & 7) + 8 * (mi & 1), vr = (lane & 7) + 8 * (mi >> 1);
      const uint32_t k_row = kr * ROWB, v_row = vr * ROWB;
      const int k_c = mi >> 1, v_c = mi & 1, sw = lane & 7;
      const int wst = p.fac_wst;
      int it = 0;
      for (int g = warp; g < ngrp; g += FNW, ++it) {
        const int s = it % wst;
        if (pc) {  // a refill: the producer's copies into this slot have landed
          if (it >= wst && !mbar_wait_bounded(fbar_full(warp, s), (uint32_t)(it / wst - 1) & 1u, p.wait_ns))
            atomicOr(p.status, FASA_DEV_TIMEOUT);
          __syncwarp();
        } else if (it > 0) {  // at most wst - 1 of this thread's later groups may still be in flight
          if (wst >= 4) cp_async_wait<3>();
          else if (wst == 3) cp_async_wait<2>();
          else if (wst == 2) cp_async_wait<1>();
          else cp_async_wait<0>();
          __syncwarp();
        }
        const uint32_t Ks = fbase + (uint32_t)(warp * wst + s) * GSLOT_B;
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
        const float c0 = n0 == -CUDART_INF_F ? 1.f : ex2_approx(m0 - n0);
        const float c1 = n1m == -CUDART_INF_F ? 1.f : ex2_approx(m1 - n1m);
        const float p0 = n0 == -CUDART_INF_F ? 0.f : ex2_approx(s0 - n0);
        const float p2 = n0 == -CUDART_INF_F ? 0.f : ex2_approx(s2 - n0);
        const float p1 = n1m == -CUDART_INF_F ? 0.f : ex2_approx(s1 - n1m);
        const float p3 = n1m == -CUDART_INF_F ? 0.f : ex2_approx(s3 - n1m);
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
        if (2 * tq < G) {
          pt[(2 * tq) * PTS + gq] = p0;
          pt[(2 * tq) * PTS + gq + 8] = p2;
        }
        if (2 * tq + 1 < G) {
          pt[(2 * tq + 1) * PTS + gq] = p1;
          pt[(2 * tq + 1) * PTS + gq + 8] = p3;
        }
        __syncwarp();
        const float2 pa = gq < G ? *reinterpret_cast<const float2*>(pt + gq * PTS + 2 * tq) : make_float2(0.f, 0.f);
        const float2 pb = gq < G ? *reinterpret_cast<const float2*>(pt + gq * PTS + 2 * tq + 8) : make_float2(0.f, 0.f);
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
        if (pc) {
          if (lane == 0) mbar_arrive(fbar_empty(warp, s));
        } else {
          // the warp's next group after the ones in flight (commits a group
          // even when empty: the waits count groups)
          const int gn = g + wst * FNW;
          if (gn < ngrp) {
#pragma unroll 4
            for (int r = 0; r < GR; r += RPI) row_copy(gn * GR + r + g_sub);
          }
          cp_async_commit();
        }
      }
      cp_async_wait<0>();
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
      }
      __syncwarp();
      // the warp's record, once every warp is done with its slots
      asm volatile("bar.sync 1, %0;" ::"r"(nrec * 32) : "memory");
      if (big_ok) {
        const int h0 = 2 * tq, h1 = 2 * tq + 1;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int dd = mt * 16 + gq;
          if (h0 < G) {
            rec[(h0 * FNW + warp) * (D + 2) + dd] = oc[mt][0];
            rec[(h0 * FNW + warp) * (D + 2) + dd + 8] = oc[mt][2];
          }
          if (h1 < G) {
            rec[(h1 * FNW + warp) * (D + 2) + dd] = oc[mt][1];
            rec[(h1 * FNW + warp) * (D + 2) + dd + 8] = oc[mt][3];
          }
        }
        if (gq == 0) {
          if (h0 < G) {
            rec[(h0 * FNW + warp) * (D + 2) + D] = m0;
            rec[(h0 * FNW + warp) * (D + 2) + D + 1] = l0;
          }
          if (h1 < G) {
            rec[(h1 * FNW + warp) * (D + 2) + D] = m1;
            rec[(h1 * FNW + warp) * (D + 2) + D + 1] = l1;
          }
        }
      }
    }
    __syncthreads();
    STEP_TRACE(8);
    // ---------------------------------------------------------------- combine
    // The G*D outputs are cut into C slices of sl float4 groups (the last one
    // shorter).  The records of the warps that attended rows are merged per
    // head -- each thread takes the head's maximum M over the records and the
    // weights exp2(m_w - M) itself, then one multiply-add per warp; no rows:
    // m = -inf, l = 0 -- and written straight into the combine slots: slice r
    // with (m, l) of every head goes to slot r of the staging (CTA r's share;
    // this CTA's own share into its receive slot), each slot then one bulk
    // copy to CTA r (issued by warp r), which finishes slice r.
#pragma unroll 1
    for (int x = tid; x < G * (D + 2); x += SNT) {
      const int g = x / (D + 2), e = x - g * (D + 2);
      float val = e == D ? -CUDART_INF_F : 0.f;
      if (big_ok && nrec > 0) {
        // (unrolled over the at most FNW records, so the loads overlap)
        const float* rg = rec + g * FNW * (D + 2);
        float mr[FNW], M = -CUDART_INF_F;
#pragma unroll
        for (int r = 0; r < FNW; ++r) {
          mr[r] = r < nrec ? rg[r * (D + 2) + D] : -CUDART_INF_F;
          M = fmaxf(M, mr[r]);
        }
        if (e == D) {
          val = M;
        } else {  // (e == D + 1: the record's l)
          float acc = 0.f;
#pragma unroll
          for (int r = 0; r < FNW; ++r)
            if (r < nrec) {
              const float w = mr[r] != -CUDART_INF_F ? ex2_approx(mr[r] - M) : 0.f;
              acc = fmaf(w, rg[r * (D + 2) + e], acc);
            }
          val = acc;
        }
      }
      if (e < D) {
        const int q = g * (D / 4) + (e >> 2);
        const int r = __float2int_rz(((float)q + 0.5f) * inv_sl);  // q / sl, exact for these sizes
        unsigned char* dst = (r == (int)crank ? crcv : csnd) + r * cs;
        *reinterpret_cast<float*>(dst + (q - r * sl) * 16 + (e & 3) * 4) = val;
      } else {
#pragma unroll 1
        for (int r = 0; r < C; ++r)
          *reinterpret_cast<float*>((r == (int)crank ? crcv : csnd) + r * cs + sl * 16 + g * 8 + (e - D) * 4) = val;
      }
    }
  }
  fence_proxy_async();  // the staging's generic writes, before the async proxy reads them
  __syncthreads();
  STEP_TRACE(28);
  if (lane == 0 && warp < C && warp != (int)crank)
    bulk_s2cluster(dsmem_map(smem_u32(crcv + crank * cs), (uint32_t)warp), smem_u32(csnd + warp * cs), (uint32_t)cs,
                   dsmem_map(smem_u32(&bars[SB_COMB]), (uint32_t)warp));
  STEP_TRACE(29);
  if (!mbar_wait_cluster_bounded(smem_u32(&bars[SB_COMB]), 0u, xwait) && tid == 0) atomicOr(p.status, FASA_DEV_TIMEOUT);
  STEP_TRACE(10);
  // First half of the final cluster barrier, once every copy into this CTA
  // has landed: when the barrier completes, every CTA's outgoing copies have
  // finished reading its shared memory, and no peer touches it any more.
  cluster_arrive_relaxed();
  STEP_TRACE(9);

  // Finish this CTA's slice: one thread per output element (4 per float4
  // group), each merging the C CTA records of its head with the loads of
  // all records in flight at once.
  const int q0 = min(ngrp4, (int)crank * sl), q1 = min(ngrp4, q0 + sl);
#pragma unroll 1
  for (int t = tid; t < 4 * (q1 - q0); t += SNT) {
    const int q = q0 + (t >> 2), c4 = t & 3;
    const int g = q / (D / 4), e = (q - g * (D / 4)) * 4 + c4;
    float mr[C_MAX], M = -CUDART_INF_F;
#pragma unroll
    for (int r = 0; r < C_MAX; ++r) {
      mr[r] = r < C ? *reinterpret_cast<const float*>(crcv + r * cs + sl * 16 + g * 8) : -CUDART_INF_F;
      M = fmaxf(M, mr[r]);
    }
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int r = 0; r < C_MAX; ++r)
      if (r < C && mr[r] != -CUDART_INF_F) {
        const float w = ex2_approx(mr[r] - M);
        L = fmaf(w, *reinterpret_cast<const float*>(crcv + r * cs + sl * 16 + g * 8 + 4), L);
        acc = fmaf(w, *reinterpret_cast<const float*>(crcv + r * cs + (q - q0) * 16 + c4 * 4), acc);
      }
    p.out[((size_t)b * p.Hq + (size_t)h * G + g) * D + e] = L > 0.f ? acc / L : 0.f;
  }

  // idx_out / count_out: the selected tokens of every CTA, concatenated in
  // cluster-rank (= token) order
  if (p.idx_out) {
    int* io = p.idx_out + (size_t)unit * p.budget;
    if (!need_select) {
      if (crank == 0)
#pragma unroll 1
        for (int i = tid; i < p.budget; i += SNT) io[i] = i < k_eff ? i : -1;
    } else {
      const int n_own = ms->n_rows;  // in token order
#pragma unroll 1
      for (int i = tid; i < n_own; i += SNT)
        if (sel_before + i < p.budget) io[sel_before + i] = rows[i];
    }
  }
  if (p.count_out && crank == 0 && tid == 0) p.count_out[unit] = k_eff;
  if (bad) atomicOr(p.status, FASA_DEV_BAD_INPUT);
  STEP_TRACE(11);
  cluster_wait();
}

}  // namespace fasa
