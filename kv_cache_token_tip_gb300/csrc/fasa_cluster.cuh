// The cluster kernel of the FASA decode step.
//
// One thread-block cluster of C CTAs owns one (batch, KV head) unit and runs
// the whole path on it without leaving the chip:
//
//   1. RoPE of the G query heads of the group (angles in fp64), and the
//      GQA-summed query restricted to the dominant FCs.
//   2. TIP: each CTA streams its contiguous token range of the FC-major
//      dominant key copy with 1-D bulk (TMA) copies into a shared-memory ring
//      and forms S_tau = sum_j qbar^[j] . k_dom[j, tau] (fp32).  Scores stay in
//      shared memory.
//   3. Top-k: a radix select over order-preserving 32-bit keys, distributed
//      over the cluster.  Each CTA histograms its scores (8-bit digits); the
//      CTAs read each other's histograms through distributed shared memory
//      and all reach the same digit.  Once the threshold bucket is small the
//      CTAs push their candidate (key, token) pairs, in token order, into
//      every CTA's shared memory; each CTA then finishes the selection
//      locally and compacts the selected tokens in ascending order.
//   4. FAC: the selected rows are split evenly over the cluster; each CTA
//      gathers its K and V rows with cp.async into a padded ring, computes the
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

#include "fasa_internal.h"
#include "fasa_ptx.cuh"

namespace fasa {

constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;  // 1 s for one bulk-copy wait

enum : int { MODE_NONE = 0, MODE_FILL = 1, MODE_TIES = 2, MODE_CAND = 3 };

struct Misc {
  int dstar, cnt_gt, bucket, failed;
  int ncand, pad0, pad1, pad2;
  int aboveR[C_MAX];
  int bucketR[C_MAX];
  int needR[C_MAX];
  int offR[C_MAX];
  int wsum[NW][C_MAX];
  int scan[NW];
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

// Warp-aggregated histogram increment; all 32 lanes must call it.
__device__ __forceinline__ void hist_add(uint32_t* H, uint32_t bin, bool valid, int lane) {
  const unsigned m = __ballot_sync(0xffffffffu, valid);
  if (valid) {
    const unsigned peers = __match_any_sync(m, bin);
    if (lane == __ffs(peers) - 1) atomicAdd(&H[bin], (uint32_t)__popc(peers));
  }
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

// RoPE angle of FC i at position m: theta_i = B^(-2i/d), a = m theta_i formed
// and reduced modulo 2 pi in fp64; cos/sin of the reduced angle in fp32.
__device__ __forceinline__ float2 rope_cos_sin(double base, int i, int d, int m) {
  const double th = exp2(-(2.0 * i / d) * log2(base));
  const double a = (double)m * th;
  const double k = rint(a * 0.15915494309189535);  // a / (2 pi)
  const double r = fma(-k, 6.283185307179586, a);
  float s, c;
  sincosf((float)r, &s, &c);
  return make_float2(c, s);
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

template <typename T, int D>
__global__ void __launch_bounds__(NT, 1) fasa_cluster_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int ES = sizeof(T);
  constexpr int EPL = D / 32;           // FAC elements per lane
  constexpr int TPV = 16 / (2 * ES);    // k_dom tokens per 16 bytes
  constexpr int ROWB = D * ES;          // bytes of one K/V row
  constexpr int ROWS = ROWB + 16;       // padded row stride in shared memory
  constexpr int CPR = ROWB / 16;        // 16-byte chunks per row

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank();
  const int C = (int)cluster_size();
  const int unit = blockIdx.y;
  const int b = unit / p.Hkv, h = unit - (unit / p.Hkv) * p.Hkv;
  const int G = p.G;
  const int flags = p.flags;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  Misc* ms = reinterpret_cast<Misc*>(smem + p.off_misc);
  float* qrot = reinterpret_cast<float*>(smem + p.off_qrot);
  float* qbar = reinterpret_cast<float*>(smem + p.off_qbar);
  float* stile = reinterpret_cast<float*>(smem + p.off_stile);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + p.off_hist);
  float* sc_s = reinterpret_cast<float*>(smem + p.off_sc);
  int* idx_s = reinterpret_cast<int*>(smem + p.off_idx);
  float* part = reinterpret_cast<float*>(smem + p.off_part);
  unsigned char* big = smem + p.off_big;

  bool bad = false;
  int len = p.seq_lens[b];
  if (len < 0 || len > p.T_max) {
    bad = true;
    len = min(max(len, 0), p.T_max);
  }
  const int k_eff = min(p.budget, len);
  const bool sel_flag = (flags & F_SELECT) != 0;
  const bool need_select = sel_flag && len > p.budget;
  const bool do_tip = (flags & F_TIP) && (!sel_flag || need_select);
  const bool read_sc = (flags & F_SC_IN) && need_select;

  // contiguous token range of this CTA (start aligned to 16 tokens)
  const int chunk = ((len + C - 1) / C + 15) & ~15;
  const int t0 = min(len, (int)crank * chunk);
  const int t1 = min(len, t0 + chunk);
  const int nloc = t1 - t0;

  const int nfc = p.n_tip, tt = p.tip_tile, ns = p.tip_stages;
  if (tid == 0) {
    for (int s = 0; s < ns; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
    ms->failed = 0;
  }
  for (int i = tid; i < 512; i += NT) hist[i] = 0u;
  cluster_arrive_relaxed();  // completed by cluster_wait() before any DSMEM access
  __syncthreads();

  // ---------------------------------------------------------------- TIP loads
  const int ntiles = do_tip ? (nloc + tt - 1) / tt : 0;
  const uint32_t fc_bytes_tile = (uint32_t)tt * 2 * ES;
  const uint32_t stage_bytes = (uint32_t)nfc * fc_bytes_tile;
  const T* kd_unit = reinterpret_cast<const T*>(p.k_dom) + (size_t)unit * nfc * p.T_max * 2;
  auto tip_issue = [&](int it) {  // warp 0
    const int s = it % ns;
    const int tau0 = t0 + it * tt;
    const int ntok = min(tt, t1 - tau0);
    const int ntokp = (ntok + TPV - 1) / TPV * TPV;
    const uint32_t bytes = (uint32_t)ntokp * 2 * ES;
    const uint32_t bar = smem_u32(&bars[s]);
    if (lane == 0) mbar_arrive_expect_tx(bar, bytes * nfc);
    __syncwarp();
    for (int j = lane; j < nfc; j += 32)
      bulk_g2s(smem_u32(big + s * stage_bytes + j * fc_bytes_tile),
               kd_unit + ((size_t)j * p.T_max + tau0) * 2, bytes, bar);
  };
  if (warp == 0)
    for (int it = 0; it < min(ns, ntiles); ++it) tip_issue(it);

  // ------------------------------------------------------------ query prep
  if (flags & F_ROPE) {
    float2* cs = reinterpret_cast<float2*>(stile);
    const int m = p.pos[b];
    for (int i = tid; i < D / 2; i += NT) cs[i] = rope_cos_sin(p.rope_theta, i, D, m);
    __syncthreads();
    const T* qg = reinterpret_cast<const T*>(p.q) + ((size_t)b * p.Hq + (size_t)h * G) * D;
    for (int x = tid; x < G * (D / 2); x += NT) {
      const int g = x / (D / 2), i = x - g * (D / 2);
      const float x0 = to_f32<T>(qg[g * D + 2 * i]);
      const float x1 = to_f32<T>(qg[g * D + 2 * i + 1]);
      const float2 c = cs[i];
      qrot[g * D + 2 * i] = x0 * c.x - x1 * c.y;
      qrot[g * D + 2 * i + 1] = x0 * c.y + x1 * c.x;
    }
  } else if (flags & (F_TIP | F_FAC | F_DENSE)) {
    const float* qg = p.q_rot + ((size_t)b * p.Hq + (size_t)h * G) * D;
    for (int x = tid; x < G * D; x += NT) qrot[x] = qg[x];
  }
  __syncthreads();
  if (do_tip) {
    for (int j = tid; j < nfc; j += NT) {
      int i = p.dom_fc[h * nfc + j];
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
  cluster_wait();

  // ---------------------------------------------------------------- TIP scan
  float* scw = (p.s_cap > 0) ? sc_s : (p.scores + (size_t)unit * p.T_max + t0);
  for (int it = 0; it < ntiles; ++it) {
    const int s = it % ns;
    const uint32_t parity = (uint32_t)(it / ns) & 1u;
    int fail = 0;
    if (!mbar_wait_bounded(smem_u32(&bars[s]), parity, WAIT_LIMIT_NS)) fail = 1;
    const int tau_base = it * tt;
    const int ntok = min(tt, nloc - tau_base);
    const unsigned char* st = big + s * stage_bytes;
    for (int gb = warp * 32; gb * 4 < ntok; gb += NT) {  // warp-uniform
      const int tl = (gb + lane) * 4;
      const bool act = tl < ntok;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (act) {
        for (int j = 0; j < nfc; ++j) {
          const float2 qq = *reinterpret_cast<const float2*>(&qbar[2 * j]);
          const unsigned char* row = st + j * fc_bytes_tile + tl * 2 * ES;
          if constexpr (ES == 2) {
            const uint4 w = *reinterpret_cast<const uint4*>(row);
            acc[0] = fmaf(qq.x, bf16_lo(w.x), fmaf(qq.y, bf16_hi(w.x), acc[0]));
            acc[1] = fmaf(qq.x, bf16_lo(w.y), fmaf(qq.y, bf16_hi(w.y), acc[1]));
            acc[2] = fmaf(qq.x, bf16_lo(w.z), fmaf(qq.y, bf16_hi(w.z), acc[2]));
            acc[3] = fmaf(qq.x, bf16_lo(w.w), fmaf(qq.y, bf16_hi(w.w), acc[3]));
          } else {
            const float4 w0 = *reinterpret_cast<const float4*>(row);
            const float4 w1 = *reinterpret_cast<const float4*>(row + 16);
            acc[0] = fmaf(qq.x, w0.x, fmaf(qq.y, w0.y, acc[0]));
            acc[1] = fmaf(qq.x, w0.z, fmaf(qq.y, w0.w, acc[1]));
            acc[2] = fmaf(qq.x, w1.x, fmaf(qq.y, w1.y, acc[2]));
            acc[3] = fmaf(qq.x, w1.z, fmaf(qq.y, w1.w, acc[3]));
          }
        }
        const int tloc = tau_base + tl;
        if (tl + 4 <= ntok) {
          *reinterpret_cast<float4*>(scw + tloc) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        } else {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (tl + t < ntok) scw[tloc + t] = acc[t];
        }
      }
      if (need_select) {
#pragma unroll
        for (int t = 0; t < 4; ++t) hist_add(hist, score_key(acc[t]) >> 24, act && (tl + t < ntok), lane);
      }
    }
    const int anyfail = __syncthreads_or(fail);
    if (anyfail) {
      if (tid == 0) {
        atomicOr(p.status, 2);
        // let copies still in flight land before the shared memory is released
        for (int it2 = it + 1; it2 < min(ntiles, it + ns); ++it2)
          mbar_wait_bounded(smem_u32(&bars[it2 % ns]), (uint32_t)(it2 / ns) & 1u, WAIT_LIMIT_NS);
      }
      __syncthreads();
      break;
    }
    if (warp == 0 && it + ns < ntiles) {
      fence_proxy_async();
      tip_issue(it + ns);
    }
  }

  // ---------------------------------------------------------------- top-k
  if (need_select) {
    const float* scr = read_sc ? (p.scores_in + (size_t)unit * p.T_max + t0) : scw;
    if (read_sc) {
      for (int c0 = 0; c0 < nloc; c0 += NT * 4) {
        float v[4];
        bool ok[4];
        load4(scr, c0 + 4 * tid, nloc, v, ok);
#pragma unroll
        for (int t = 0; t < 4; ++t) hist_add(hist, score_key(v[t]) >> 24, ok[t], lane);
      }
    }
    if (tid < C_MAX) ms->aboveR[tid] = 0;
    __syncthreads();

    int k_rem = k_eff, above_total = 0, mode = MODE_NONE, shift = 24, last_pass = 0;
    uint32_t prefix = 0u;
    for (int pass = 0; pass < 4; ++pass) {
      shift = 24 - 8 * pass;
      last_pass = pass;
      uint32_t* H = hist + (pass & 1) * 256;
      if (pass > 0) {
        // H was last read by the other CTAs two passes ago, before the
        // previous cluster barrier.
        for (int i = tid; i < 256; i += NT) H[i] = 0u;
        __syncthreads();
        for (int c0 = 0; c0 < nloc; c0 += NT * 4) {
          float v[4];
          bool ok[4];
          load4(scr, c0 + 4 * tid, nloc, v, ok);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint32_t key = score_key(v[t]);
            hist_add(H, (key >> shift) & 255u, ok[t] && (key >> (shift + 8)) == prefix, lane);
          }
        }
      }
      __syncthreads();
      cluster_sync();
      // thread tid holds digit 255 - tid: an exclusive scan counts larger digits
      const int bin = 255 - tid;
      const uint32_t la = smem_u32(&H[bin]);
      uint32_t v[C_MAX];
      uint32_t tot = 0u;
#pragma unroll
      for (int r = 0; r < C_MAX; ++r) {
        v[r] = (r < C) ? dsmem_ld_u32(dsmem_map(la, (uint32_t)r)) : 0u;
        tot += v[r];
      }
      int total;
      const int excl = block_excl_scan((int)tot, ms->scan, total);
      if (excl < k_rem && k_rem <= excl + (int)tot) {
        ms->dstar = bin;
        ms->cnt_gt = excl;
        ms->bucket = (int)tot;
#pragma unroll
        for (int r = 0; r < C_MAX; ++r)
          if (r < C) ms->bucketR[r] = (int)v[r];
      }
      __syncthreads();
      const int dstar = ms->dstar, cnt_gt = ms->cnt_gt, bucket = ms->bucket;
      const bool above = bin > dstar;
#pragma unroll
      for (int r = 0; r < C_MAX; ++r) {
        const unsigned x = __reduce_add_sync(0xffffffffu, above ? v[r] : 0u);
        if (lane == 0) ms->wsum[warp][r] = (int)x;
      }
      __syncthreads();
      if (tid < C) {
        int s = 0;
        for (int w = 0; w < NW; ++w) s += ms->wsum[w][tid];
        ms->aboveR[tid] += s;
      }
      k_rem -= cnt_gt;
      above_total += cnt_gt;
      prefix = (prefix << 8) | (uint32_t)dstar;
      if (bucket == k_rem) mode = MODE_FILL;
      else if (pass == 3) mode = MODE_TIES;
      else if (above_total + bucket <= p.cand_cap) mode = MODE_CAND;
      __syncthreads();
      if (mode != MODE_NONE) break;
    }

    // per-CTA candidate counts and offsets (identical in every CTA)
    if (tid == 0) {
      int run = 0, ties_before = 0;
      for (int r = 0; r < C; ++r) {
        int need = ms->bucketR[r];
        if (mode == MODE_TIES) {
          need = min(max(k_rem - ties_before, 0), ms->bucketR[r]);
          ties_before += ms->bucketR[r];
        }
        ms->needR[r] = need;
        ms->offR[r] = run;
        run += ms->aboveR[r] + need;
      }
      ms->ncand = run;
    }
    __syncthreads();
    const int my_off = ms->offR[crank], my_need = ms->needR[crank], ncand = ms->ncand;
    uint32_t* ckey = reinterpret_cast<uint32_t*>(big);
    int* ctau = reinterpret_cast<int*>(big + (size_t)p.cand_cap * 4);
    const uint32_t ckey_l = smem_u32(ckey), ctau_l = smem_u32(ctau);

    // push this CTA's candidates, in token order, to every CTA of the cluster
    int run_s = 0, run_t = 0;
    for (int c0 = 0; c0 < nloc; c0 += NT * 4) {
      float v[4];
      bool ok[4];
      load4(scr, c0 + 4 * tid, nloc, v, ok);
      uint32_t key[4];
      bool strict[4], tie[4];
      int cs_ = 0, ct_ = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        key[t] = score_key(v[t]);
        if (mode == MODE_TIES) {
          strict[t] = ok[t] && key[t] > prefix;
          tie[t] = ok[t] && key[t] == prefix;
        } else {
          strict[t] = ok[t] && (key[t] >> shift) >= prefix;
          tie[t] = false;
        }
        cs_ += strict[t];
        ct_ += tie[t];
      }
      int tot;
      const int ex = block_excl_scan(cs_ | (ct_ << 16), ms->scan, tot);
      int s_before = run_s + (ex & 0xFFFF), t_before = run_t + (ex >> 16);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const bool take = strict[t] || (tie[t] && t_before < my_need);
        if (take) {
          const int pos = my_off + s_before + min(t_before, my_need);
          const uint32_t tau = (uint32_t)(t0 + c0 + 4 * tid + t);
          for (int r = 0; r < C; ++r) {
            dsmem_st_u32(dsmem_map(ckey_l + pos * 4, (uint32_t)r), key[t]);
            dsmem_st_u32(dsmem_map(ctau_l + pos * 4, (uint32_t)r), tau);
          }
        }
        s_before += strict[t];
        t_before += tie[t];
      }
      run_s += tot & 0xFFFF;
      run_t += tot >> 16;
    }
    cluster_sync();

    // finish the selection locally on the (identical) candidate list
    long long kthr = -1;
    int ties_take = 0;
    if (mode == MODE_CAND) {
      uint32_t pre = prefix;
      int kr = k_rem;
      for (int qp = last_pass + 1; qp < 4; ++qp) {
        const int s2 = 24 - 8 * qp;
        for (int i = tid; i < 256; i += NT) hist[i] = 0u;
        __syncthreads();
        for (int e0 = 0; e0 < ncand; e0 += NT) {
          const int e = e0 + tid;
          const uint32_t key = (e < ncand) ? ckey[e] : 0u;
          hist_add(hist, (key >> s2) & 255u, e < ncand && (key >> (s2 + 8)) == pre, lane);
        }
        __syncthreads();
        const int bin = 255 - tid;
        const int cnt = (int)hist[bin];
        int total;
        const int excl = block_excl_scan(cnt, ms->scan, total);
        if (excl < kr && kr <= excl + cnt) {
          ms->dstar = bin;
          ms->cnt_gt = excl;
          ms->bucket = cnt;
        }
        __syncthreads();
        kr -= ms->cnt_gt;
        pre = (pre << 8) | (uint32_t)ms->dstar;
        const int bucket = ms->bucket;
        __syncthreads();
        if (bucket == kr) {
          kthr = ((long long)pre << s2) - 1;
          ties_take = 0;
          break;
        }
        if (qp == 3) {
          kthr = (long long)pre;
          ties_take = kr;
        }
      }
    }
    int run = 0, runq = 0;
    for (int e0 = 0; e0 < ncand; e0 += NT) {
      const int e = e0 + tid;
      const bool valid = e < ncand;
      const long long key = valid ? (long long)ckey[e] : -1;
      const bool gt = valid && key > kthr;
      const bool eq = valid && key == kthr && ties_take > 0;
      int tot;
      const int ex = block_excl_scan((int)gt | ((int)eq << 16), ms->scan, tot);
      const int tb = runq + (ex >> 16);
      if (gt || (eq && tb < ties_take)) idx_s[run + (ex & 0xFFFF) + min(tb, ties_take)] = ctau[e];
      run += tot & 0xFFFF;
      runq += tot >> 16;
    }
    __syncthreads();
  }

  if ((flags & F_IDX_OUT) && crank == 0) {
    if (p.idx_out) {
      int* io = p.idx_out + (size_t)unit * p.budget;
      for (int i = tid; i < p.budget; i += NT) io[i] = (i < k_eff) ? (need_select ? idx_s[i] : i) : -1;
    }
    if (p.count_out && tid == 0) p.count_out[unit] = k_eff;
  }

  // ---------------------------------------------------------------- FAC
  if (flags & (F_FAC | F_DENSE)) {
    int n_total;
    bool contiguous;
    int lofs = 0;
    if (flags & F_DENSE) {
      n_total = len;
      contiguous = true;
    } else if (flags & F_IDX_IN) {
      n_total = p.count_in[unit];
      if (n_total < 0 || n_total > k_eff) {
        bad = true;
        n_total = min(max(n_total, 0), k_eff);
      }
      contiguous = false;
    } else if (need_select) {
      n_total = k_eff;
      contiguous = false;
    } else {
      n_total = k_eff;
      contiguous = true;
    }
    const int r0 = (int)(((long long)n_total * crank) / C);
    const int r1 = (int)(((long long)n_total * (crank + 1)) / C);
    const int nrows = r1 - r0;
    if (flags & F_IDX_IN) {
      const int* gi = p.idx_in + (size_t)unit * p.budget + r0;
      for (int i = tid; i < nrows; i += NT) {
        int t = gi[i];
        if (t < 0 || t >= len) {
          bad = true;
          t = min(max(t, 0), len - 1);
        }
        idx_s[i] = t;
      }
      __syncthreads();
    } else if (!contiguous) {
      lofs = r0;
    }

    const T* Kb = reinterpret_cast<const T*>(p.k_cache) + (size_t)unit * p.T_max * D;
    const T* Vb = reinterpret_cast<const T*>(p.v_cache) + (size_t)unit * p.T_max * D;
    const int ntile = (nrows + RT - 1) / RT;
    constexpr uint32_t STAGE_B = 2u * RT * ROWS;
    const uint32_t fac_l = smem_u32(big);
    auto fac_issue = [&](int t) {
      if (t < ntile) {
        const int s = t % FAC_STAGES;
        for (int c = tid; c < 2 * RT * CPR; c += NT) {
          const int which = c / (RT * CPR);
          const int rr = (c / CPR) % RT;
          const int ch = c % CPR;
          const int i = t * RT + rr;
          if (i < nrows) {
            const int tau = contiguous ? (r0 + i) : idx_s[lofs + i];
            const T* src = (which ? Vb : Kb) + (size_t)tau * D + ch * (16 / ES);
            cp_async16(fac_l + s * STAGE_B + which * RT * ROWS + rr * ROWS + ch * 16, src);
          }
        }
      }
      cp_async_commit();
    };

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

#pragma unroll
    for (int s = 0; s < FAC_STAGES - 1; ++s) fac_issue(s);
    for (int t = 0; t < ntile; ++t) {
      cp_async_wait<FAC_STAGES - 2>();
      __syncthreads();
      fac_issue(t + FAC_STAGES - 1);
      const int s = t % FAC_STAGES;
      const unsigned char* Ks = big + s * STAGE_B;
      const unsigned char* Vs = Ks + RT * ROWS;
      const int rows_t = min(RT, nrows - t * RT);
      for (int rr = warp; rr < rows_t; rr += NW) {
        float kv[EPL];
        load_row<T, EPL>(Ks + rr * ROWS + lane * EPL * ES, kv);
#pragma unroll
        for (int g = 0; g < G_MAX; ++g) {
          if (g < G) {
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) a = fmaf(qreg[g][e], kv[e], a);
            a = warp_sum(a);
            if (lane == g) stile[g * RT + rr] = a;
          }
        }
      }
      __syncthreads();
      if (pv_warp) {
        const int nr = (rows_t - my_part + nparts - 1) / nparts;
        if (nr > 0) {
          const float sv = (lane < nr) ? stile[my_g * RT + my_part + lane * nparts] : -CUDART_INF_F;
          const float m_new = fmaxf(m_run, warp_max(sv));
          const float scale = exp2f(m_run - m_new);
          const float pe = (lane < nr) ? exp2f(sv - m_new) : 0.f;
          l_run = l_run * scale + warp_sum(pe);
#pragma unroll
          for (int e = 0; e < EPL; ++e) o_run[e] *= scale;
          for (int i = 0; i < nr; ++i) {
            const float pi = __shfl_sync(0xffffffffu, pe, i);
            float vv[EPL];
            load_row<T, EPL>(Vs + (my_part + i * nparts) * ROWS + lane * EPL * ES, vv);
#pragma unroll
            for (int e = 0; e < EPL; ++e) o_run[e] = fmaf(pi, vv[e], o_run[e]);
          }
          m_run = m_new;
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();

    // merge the row-parts of each head, then push the CTA partial
    float* mst = reinterpret_cast<float*>(big);
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
    for (int x = tid; x < G * (D + 2); x += NT) {
      const int g = x / (D + 2), e = x - g * (D + 2);
      float M = -CUDART_INF_F;
      for (int pp = 0; pp < nparts; ++pp) M = fmaxf(M, mst[(g * nparts + pp) * (D + 2) + D]);
      float val = M;
      if (e != D) {
        float acc = 0.f;
        for (int pp = 0; pp < nparts; ++pp) {
          const float* sp = mst + (g * nparts + pp) * (D + 2);
          if (sp[D] != -CUDART_INF_F) acc += exp2f(sp[D] - M) * sp[e];
        }
        val = acc;
      }
      const uint32_t dst = smem_u32(part + ((g / C) * C + (int)crank) * (D + 2) + e);
      dsmem_st_f32(dsmem_map(dst, (uint32_t)(g % C)), val);
    }
    cluster_sync();
    for (int x = tid; x < p.hpc * D; x += NT) {
      const int hs = x / D, e = x - hs * D;
      const int g = hs * C + (int)crank;
      if (g < G) {
        const float* base = part + hs * C * (D + 2);
        float M = -CUDART_INF_F;
        for (int r = 0; r < C; ++r) M = fmaxf(M, base[r * (D + 2) + D]);
        float L = 0.f, O = 0.f;
        if (M != -CUDART_INF_F) {
          for (int r = 0; r < C; ++r) {
            const float* sp = base + r * (D + 2);
            if (sp[D] != -CUDART_INF_F) {
              const float w = exp2f(sp[D] - M);
              L += w * sp[D + 1];
              O += w * sp[e];
            }
          }
        }
        p.out[((size_t)b * p.Hq + (size_t)h * G + g) * D + e] = (L > 0.f) ? O / L : 0.f;
      }
    }
  }
  if (bad) atomicOr(p.status, 1);
}

template <typename T, int D>
cudaError_t prepare_kernel() {
  static cudaError_t once = [] {
    auto k = fasa_cluster_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  }();
  return once;
}

template <typename T, int D>
cudaError_t launch_cluster_t(const Params& p, int C, cudaStream_t s) {
  cudaError_t e = prepare_kernel<T, D>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, (unsigned)(p.B * p.Hkv), 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)p.smem_total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fasa_cluster_kernel<T, D>, p);
}

template <typename T, int D>
int max_clusters_t(int C, int smem_bytes) {
  if (prepare_kernel<T, D>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fasa_cluster_kernel<T, D>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace fasa
